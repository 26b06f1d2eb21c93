"""Seeded synthetic inputs for the tree verify / expand step.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no attention, no argmax, no tree walk).  Both the CUDA
path (through the tests and ``bench.py``) and the fp64 oracle (through the
tests) are fed from here, so the two see the same bytes.

Recipe (shared by every workload):

* Q, K, V: fp32 draws from N(0, 1), rounded to bfloat16 (round to nearest
  even) and kept as raw ``uint16`` bit patterns.
* Logits: fp32 N(0, 1) of shape ``[num_req][n_tree_max][vocab]``.  One entry
  per row, at a uniformly drawn token (the *planted peak*), is set to
  ``PLANTED_PEAK`` so that the draft-token rule below can be applied without
  computing an argmax here.  A standard normal exceeds 8 with probability
  about 6e-16 per draw, so the planted token is the row's argmax for every
  workload in this file.
* Draft tokens: node 0 (the root, i.e. the last verified token) is uniform in
  ``[0, vocab)``; node ``i >= 1`` takes the planted peak of its parent's row
  with probability ``p_accept`` and a uniform token otherwise, and siblings
  carry distinct tokens (a drafter expands a node into distinct tokens; a
  repeat is redrawn).  This is the greedy acceptance model of the NVIDIA
  draft-length article (each draft token is accepted independently with a
  fixed probability).
* Tree shapes: ``parent[0] = -1`` and ``parent[i]`` uniform over earlier
  nodes (optionally only over nodes whose depth is below a cap), so
  ``parent[i] < i`` always holds (leaves are appended, SwiftSpec summary
  §3.1.3, Figure 3).
* Prefix lengths: fixed or uniform over the stated range.
* Paged KV: a pool of 16-row blocks; every request's logical blocks are
  mapped through a block table that is a random permutation of the pool.

Random streams come from ``numpy.random.SeedSequence(seed).spawn(8)`` in a
fixed order (see ``_streams``), seed 0 for every named workload.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PLANTED_PEAK = np.float32(8.0)
PAGE_SIZE = 16


# --------------------------------------------------------------------------
# raw draws
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); return bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = (b + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 24
    for s in range(0, n, step):  # chunked to bound the fp32 temporary
        e = min(n, s + step)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def _streams(seed: int):
    ss = np.random.SeedSequence(seed)
    names = ["lengths", "shape", "logits", "tokens", "q", "k", "v", "blocks", "draft"]
    return {nm: np.random.default_rng(s) for nm, s in zip(names, ss.spawn(len(names)))}


# --------------------------------------------------------------------------
# trees and tokens
# --------------------------------------------------------------------------
def random_parents(rng: np.random.Generator, n: int, depth_cap: Optional[int] = None) -> np.ndarray:
    """parent[0] = -1; parent[i] uniform over earlier nodes of depth < depth_cap."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int64)
    for i in range(1, n):
        while True:
            p = int(rng.integers(0, i))
            if depth_cap is None or depth[p] < depth_cap:
                break
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def grow_parents(rng: np.random.Generator, parent: np.ndarray, extra: int) -> np.ndarray:
    """Append ``extra`` nodes whose parents are uniform over all earlier nodes."""
    n0 = len(parent)
    out = np.concatenate([parent.astype(np.int32), np.full(extra, -1, np.int32)])
    for i in range(n0, n0 + extra):
        out[i] = int(rng.integers(0, i))
    return out


def chain_parents(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def planted_logits(rng: np.random.Generator, rows: int, vocab: int):
    """N(0,1) logits with one planted peak per row; returns (logits, peak_token)."""
    logits = rng.standard_normal((rows, vocab), dtype=np.float32)
    peak = rng.integers(0, vocab, size=rows).astype(np.int32)
    logits[np.arange(rows), peak] = PLANTED_PEAK
    return logits, peak


def draft_tokens(rng: np.random.Generator, parent: np.ndarray, peak: np.ndarray,
                 vocab: int, p_accept: float, peak_rows: Optional[int] = None,
                 distinct_siblings: bool = True) -> np.ndarray:
    """token[0] uniform; token[i] = peak[parent[i]] w.p. p_accept, else uniform.

    Nodes whose parent index is >= ``peak_rows`` (nodes the target never
    scored) always draw a uniform token.  With ``distinct_siblings`` (the
    default) no two children of one node carry the same token, as when a
    drafter expands a node into its top tokens: a draw that repeats a
    sibling's token is replaced by a fresh uniform draw among unused tokens.
    """
    n = len(parent)
    if peak_rows is None:
        peak_rows = n
    tok = np.zeros(n, dtype=np.int32)
    tok[0] = rng.integers(0, vocab)
    used = {-1: {int(tok[0])}}
    for i in range(1, n):
        u = rng.random()
        t = int(rng.integers(0, vocab))
        p = int(parent[i])
        sib = used.setdefault(p, set())
        if p >= 0 and p < peak_rows and u < p_accept and (not distinct_siblings or int(peak[p]) not in sib):
            t = int(peak[p])
        elif distinct_siblings and len(sib) < vocab:
            while t in sib:
                t = int(rng.integers(0, vocab))
        tok[i] = t
        sib.add(t)
    return tok


# --------------------------------------------------------------------------
# containers
# --------------------------------------------------------------------------
@dataclasses.dataclass
class AttnCase:
    num_req: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    n_tree_max: int
    n_query: int
    max_kv_len: int          # contiguous: rows per request; paged: blocks_per_req * PAGE_SIZE
    paged: bool
    prefix_len: np.ndarray   # [num_req] int32
    n_tree: np.ndarray       # [num_req] int32
    parent: np.ndarray       # [num_req][n_tree_max] int32
    q: np.ndarray            # [num_req][n_query][Hq][d] uint16 (bf16 bits)
    k: np.ndarray            # contiguous [num_req][max_kv_len][Hkv][d] or pool [blocks][16][Hkv][d]
    v: np.ndarray
    block_table: Optional[np.ndarray] = None   # [num_req][max_blocks] int32 (paged only)
    softmax_scale: float = 0.0                  # 0 -> 1/sqrt(head_dim)
    rope_theta: float = 0.0                     # > 0: queries rotated at their tree positions

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale > 0 else 1.0 / math.sqrt(self.head_dim)


@dataclasses.dataclass
class AcceptCase:
    num_req: int
    n_tree_max: int
    vocab: int
    n_tree: np.ndarray       # [num_req] int32
    parent: np.ndarray       # [num_req][n_tree_max] int32
    tokens: np.ndarray       # [num_req][n_tree_max] int32
    logits: np.ndarray       # [num_req][n_tree_max][vocab] float32
    planted: np.ndarray      # [num_req][n_tree_max] int32 (generator's intended argmax)


@dataclasses.dataclass
class CompactCase:
    """A re-root + compaction call: tree metadata and the verified tokens."""
    num_req: int
    n_tree_max: int
    prefix_len: np.ndarray   # [num_req]
    n_tree: np.ndarray       # [num_req]
    parent: np.ndarray       # [num_req][n_tree_max]
    tokens: np.ndarray       # [num_req][n_tree_max]
    verified: Optional[np.ndarray] = None   # [num_req][m_max] (filled from acceptance when None)
    m: Optional[np.ndarray] = None          # [num_req]


@dataclasses.dataclass
class DraftState:
    """Draft-side expansion inputs: a tree whose nodes already carry their
    candidate children (tokens and decreasing log-probabilities, as a draft
    model would have produced them), and the draft logits of the nodes that
    expansions 2..d query (expansion 1 draws on the existing candidates)."""
    num_req: int
    w: int                   # nodes added per expansion (= attention queries)
    k: int                   # candidates per node
    bs: int                  # nodes of the subtree selected at the end
    vocab: int
    n0: int                  # nodes before the first expansion
    parent: np.ndarray       # [num_req][n_tree_max] int32
    tokens: np.ndarray       # [num_req][n_tree_max] int32
    weight: np.ndarray       # [num_req][n_tree_max] float32, non-increasing from parent to child
    cand_tok: np.ndarray     # [num_req][n_tree_max][k] int32 (distinct per node)
    cand_lp: np.ndarray      # [num_req][n_tree_max][k] float32, decreasing, < 0
    cand_taken: np.ndarray   # [num_req][n_tree_max] int32 (children already in the tree, capped at k)
    logits: list             # per expansion 2..d: float32 [num_req][w][vocab]


@dataclasses.dataclass
class Workload:
    name: str
    description: str
    attn: list                       # list[AttnCase]; config 2 has one per expansion
    accept: Optional[AcceptCase] = None
    compact: Optional[CompactCase] = None          # target side: same tree as acceptance
    compact_draft: Optional[CompactCase] = None    # draft side (long-context workload)
    num_layers: int = 1
    draft: Optional[DraftState] = None             # draft-side expansion loop (config 2)


# --------------------------------------------------------------------------
# KV generation helpers
# --------------------------------------------------------------------------
def _contiguous_kv(rs, num_req, max_kv_len, hkv, d):
    k = normal_bf16(rs["k"], (num_req, max_kv_len, hkv, d))
    v = normal_bf16(rs["v"], (num_req, max_kv_len, hkv, d))
    return k, v


def _paged_kv(rs, rows_needed, hkv, d, extra_blocks=0):
    """Pool of 16-row blocks and a shuffled block table covering rows_needed[b]."""
    nblk = [(int(r) + PAGE_SIZE - 1) // PAGE_SIZE for r in rows_needed]
    total = sum(nblk) + extra_blocks
    perm = rs["blocks"].permutation(total).astype(np.int32)
    max_blocks = max(nblk)
    table = np.full((len(nblk), max_blocks), -1, dtype=np.int32)
    off = 0
    for b, nb in enumerate(nblk):
        table[b, :nb] = perm[off:off + nb]
        off += nb
    k = normal_bf16(rs["k"], (total, PAGE_SIZE, hkv, d))
    v = normal_bf16(rs["v"], (total, PAGE_SIZE, hkv, d))
    return k, v, table, max_blocks * PAGE_SIZE


def _trees(rs, num_req, n, depth_cap=None, chain=False):
    par = np.stack([chain_parents(n) if chain else random_parents(rs["shape"], n, depth_cap)
                    for _ in range(num_req)]).astype(np.int32)
    return par


def _accept(rs, parent, n_tree, vocab, p_accept, distinct_siblings=True):
    num_req, n_max = parent.shape
    logits = np.empty((num_req, n_max, vocab), dtype=np.float32)
    planted = np.zeros((num_req, n_max), dtype=np.int32)
    tokens = np.zeros((num_req, n_max), dtype=np.int32)
    for b in range(num_req):
        lg, pk = planted_logits(rs["logits"], n_max, vocab)
        logits[b] = lg
        planted[b] = pk
        n = int(n_tree[b])
        tokens[b, :n] = draft_tokens(rs["tokens"], parent[b, :n], pk, vocab, p_accept,
                                     distinct_siblings=distinct_siblings)
    return AcceptCase(num_req, n_max, vocab, n_tree.astype(np.int32).copy(), parent.copy(),
                      tokens, logits, planted)


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------
def tree16_prefix128(seed: int = 0) -> Workload:
    """1 request, 8 q / 2 kv heads, d 64, prefix 128, 16-node tree, vocab 1024, p 0.7."""
    rs = _streams(seed)
    num_req, hq, hkv, d, P, n, V = 1, 8, 2, 64, 128, 16, 1024
    parent = _trees(rs, num_req, n)
    n_tree = np.full(num_req, n, np.int32)
    prefix = np.full(num_req, P, np.int32)
    k, v = _contiguous_kv(rs, num_req, P + n, hkv, d)
    q = normal_bf16(rs["q"], (num_req, n, hq, d))
    attn = AttnCase(num_req, hq, hkv, d, n, n, P + n, False, prefix, n_tree, parent, q, k, v)
    acc = _accept(rs, parent, n_tree, V, 0.7)
    comp = CompactCase(num_req, n, prefix.copy(), n_tree.copy(), parent.copy(), acc.tokens.copy())
    return Workload("tree16_prefix128_g4_d64", "1 req, Hq 8 / Hkv 2, d 64, prefix 128, "
                    "16-node tree, 16x144 keys, vocab 1024, p 0.7", [attn], acc, comp)


def expand_w8_prefix2048(seed: int = 0) -> Workload:
    """SwiftSpec-style draft expansion: 64-node tree (depth <= 8) + 4 expansions of 8 leaves."""
    rs = _streams(seed)
    num_req, hq, hkv, d, P, n0, w, steps = 1, 32, 8, 128, 2048, 64, 8, 4
    base = random_parents(rs["shape"], n0, depth_cap=8)
    full = grow_parents(rs["shape"], base, w * steps)
    n_max = n0 + w * steps
    parent = full[None, :].astype(np.int32)
    prefix = np.full(num_req, P, np.int32)
    k, v = _contiguous_kv(rs, num_req, P + n_max, hkv, d)
    cases = []
    for e in range(steps):
        n = n0 + w * (e + 1)
        q = normal_bf16(rs["q"], (num_req, w, hq, d))
        cases.append(AttnCase(num_req, hq, hkv, d, n_max, w, P + n_max, False, prefix,
                              np.full(num_req, n, np.int32), parent, q, k, v))
    # the draft side of the same iteration: the 64-node tree with candidate
    # children on every node, draft logits (vocab 128256, a 32/8/128-head
    # model's) for the nodes expansions 2..4 query, a 32-node subtree at the end
    k, bs, vocab = 8, 32, 128256
    g = rs["draft"]
    weight = np.zeros((num_req, n_max), np.float32)
    for i in range(1, n0):
        weight[0, i] = weight[0, base[i]] - np.float32(g.exponential(1.0))
    cand_tok = np.stack([[g.choice(vocab, size=k, replace=False) for _ in range(n_max)]]).astype(np.int32)
    cand_lp = (-np.cumsum(g.exponential(0.7, size=(num_req, n_max, k)), axis=2)).astype(np.float32)
    children = np.bincount(base[1:], minlength=n_max)[:n_max]
    taken = np.minimum(children, k).astype(np.int32)[None, :]
    tokens = g.integers(0, vocab, size=(num_req, n_max)).astype(np.int32)
    dparent = np.full((num_req, n_max), -1, np.int32)
    dparent[0, :n0] = base
    logits = [(g.normal(size=(num_req, w, vocab)) * 2.0).astype(np.float32) for _ in range(steps - 1)]
    draft = DraftState(num_req, w, k, bs, vocab, n0, dparent, tokens, weight, cand_tok, cand_lp, taken, logits)
    return Workload("expand_w8_prefix2048", "1 req, Hq 32 / Hkv 8, d 128, prefix 2048, "
                    "tree 64 (depth<=8) + 4 expansions of w=8 new leaves (8x2120..8x2144)", cases, draft=draft)


def verify_b8_tree16(seed: int = 0) -> Workload:
    """Llama-70B-shaped target verify: 8 requests, 64/8 heads, 16-node trees, prefix U{1024..4096}."""
    rs = _streams(seed)
    num_req, hq, hkv, d, n, V = 8, 64, 8, 128, 16, 128256
    prefix = rs["lengths"].integers(1024, 4097, size=num_req).astype(np.int32)
    parent = _trees(rs, num_req, n)
    n_tree = np.full(num_req, n, np.int32)
    max_kv = 4096 + n
    k, v = _contiguous_kv(rs, num_req, max_kv, hkv, d)
    q = normal_bf16(rs["q"], (num_req, n, hq, d))
    attn = AttnCase(num_req, hq, hkv, d, n, n, max_kv, False, prefix, n_tree, parent, q, k, v)
    acc = _accept(rs, parent, n_tree, V, 0.7)
    comp = CompactCase(num_req, n, prefix.copy(), n_tree.copy(), parent.copy(), acc.tokens.copy())
    return Workload("verify_b8_tree16_g8", "8 req, Hq 64 / Hkv 8, d 128, prefix U{1024..4096}, "
                    "16-node trees (D=15, G(1+D)=128), vocab 128256, p 0.7", [attn], acc, comp)


def chain_verify_b16_paged(seed: int = 0) -> Workload:
    """MineDraft-style batched chain verify over paged KV (block 16, shuffled table)."""
    rs = _streams(seed)
    num_req, hq, hkv, d, n = 16, 64, 8, 128, 5
    ctx = rs["lengths"].integers(512, 8193, size=num_req).astype(np.int32)
    parent = _trees(rs, num_req, n, chain=True)
    n_tree = np.full(num_req, n, np.int32)
    k, v, table, max_kv = _paged_kv(rs, ctx + n, hkv, d)
    q = normal_bf16(rs["q"], (num_req, n, hq, d))
    attn = AttnCase(num_req, hq, hkv, d, n, n, max_kv, True, ctx, n_tree, parent, q, k, v, table)
    return Workload("chain_verify_b16_paged", "16 req, Hq 64 / Hkv 8, d 128, chain k=4 + 1, "
                    "context U{512..8192}, paged KV block 16 with shuffled block table", [attn])


def longctx_verify_b4_p32k(seed: int = 0, num_layers: int = 64, with_kv: bool = True) -> Workload:
    """Long-context verify + evolving-tree-cache update: 4 req, 32/8 heads, prefix 32768, 32-node trees.

    The draft-side tree has 64 nodes: its first 32 are the verified tree and
    nodes 32..63 were grown while the target verified (SwiftSpec summary
    §3.1.2, Figure 2), with the draft-token rule applied against the target's
    planted peak when the parent is one of the first 32 nodes.
    """
    rs = _streams(seed)
    num_req, hq, hkv, d, P, n, nd, V = 4, 32, 8, 128, 32768, 32, 64, 152064
    prefix = np.full(num_req, P, np.int32)
    parent = _trees(rs, num_req, n)
    n_tree = np.full(num_req, n, np.int32)
    max_kv = P + n
    if with_kv:
        k, v = _contiguous_kv(rs, num_req, max_kv, hkv, d)
        q = normal_bf16(rs["q"], (num_req, n, hq, d))
    else:
        k = v = q = None
    attn = AttnCase(num_req, hq, hkv, d, n, n, max_kv, False, prefix, n_tree, parent, q, k, v)
    acc = _accept(rs, parent, n_tree, V, 0.8)
    comp = CompactCase(num_req, n, prefix.copy(), n_tree.copy(), parent.copy(), acc.tokens.copy())
    dpar = np.zeros((num_req, nd), np.int32)
    dtok = np.zeros((num_req, nd), np.int32)
    for b in range(num_req):
        dpar[b] = grow_parents(rs["shape"], parent[b], nd - n)
        grown = draft_tokens(rs["tokens"], dpar[b], acc.planted[b], V, 0.8, peak_rows=n)
        dtok[b, :n] = acc.tokens[b]
        dtok[b, n:] = grown[n:]
    draft = CompactCase(num_req, nd, prefix.copy(), np.full(num_req, nd, np.int32), dpar, dtok)
    return Workload("longctx_verify_b4_p32k", "4 req, Hq 32 / Hkv 8, d 128, prefix 32768, "
                    "32-node trees (D=31, G(1+D)=128), vocab 152064, p 0.8, compaction over "
                    f"{num_layers} layers (target side 32-node, draft side 64-node trees)",
                    [attn], acc, comp, draft, num_layers)


WORKLOADS = {
    1: tree16_prefix128,
    2: expand_w8_prefix2048,
    3: verify_b8_tree16,
    4: chain_verify_b16_paged,
    5: longctx_verify_b4_p32k,
}


# --------------------------------------------------------------------------
# small random cases for parity tests
# --------------------------------------------------------------------------
def random_attn_case(seed: int, num_req=2, hq=8, hkv=2, d=64, n_tree_max=16, n_query=None,
                     prefix_range=(0, 200), paged=False, chain=False, depth_cap=None,
                     ragged_tree=False, scale=0.0, extra_blocks=3) -> AttnCase:
    """A small attention case with ragged prefixes (and optionally ragged trees)."""
    rs = _streams(seed)
    nq = n_query if n_query is not None else n_tree_max
    lo, hi = prefix_range
    prefix = rs["lengths"].integers(lo, hi + 1, size=num_req).astype(np.int32)
    if ragged_tree:
        n_tree = rs["lengths"].integers(nq, n_tree_max + 1, size=num_req).astype(np.int32)
    else:
        n_tree = np.full(num_req, n_tree_max, np.int32)
    parent = np.full((num_req, n_tree_max), -1, np.int32)
    for b in range(num_req):
        nb = int(n_tree[b])
        parent[b, :nb] = chain_parents(nb) if chain else random_parents(rs["shape"], nb, depth_cap)
    q = normal_bf16(rs["q"], (num_req, nq, hq, d))
    if paged:
        k, v, table, max_kv = _paged_kv(rs, prefix + n_tree, hkv, d, extra_blocks)
    else:
        max_kv = int((prefix + n_tree).max()) + 5
        k, v = _contiguous_kv(rs, num_req, max_kv, hkv, d)
        table = None
    return AttnCase(num_req, hq, hkv, d, n_tree_max, nq, max_kv, paged, prefix, n_tree, parent,
                    q, k, v, table, scale)


def random_accept_case(seed: int, num_req=3, n_tree_max=16, vocab=1000, p_accept=0.7,
                       chain=False, ragged_tree=True, distinct_siblings=True) -> AcceptCase:
    rs = _streams(seed)
    if ragged_tree:
        n_tree = rs["lengths"].integers(1, n_tree_max + 1, size=num_req).astype(np.int32)
    else:
        n_tree = np.full(num_req, n_tree_max, np.int32)
    parent = np.full((num_req, n_tree_max), -1, np.int32)
    for b in range(num_req):
        nb = int(n_tree[b])
        parent[b, :nb] = chain_parents(nb) if chain else random_parents(rs["shape"], nb)
    return _accept(rs, parent, n_tree, vocab, p_accept, distinct_siblings)


def random_compact_case(seed: int, num_req=3, n_tree_max=24, vocab=50, p_follow=0.8,
                        prefix_range=(0, 40), max_verified=None, forest=False) -> CompactCase:
    """Tree metadata plus a verified-token sequence that walks part of the tree.

    The verified sequence follows a random root path of the tree for a random
    number of steps and then (with probability 1/2) appends a token that may
    or may not label a child, so every outcome of the walk occurs: full match
    with survivors, mismatch part-way, empty sequence.
    """
    rs = _streams(seed)
    prefix = rs["lengths"].integers(prefix_range[0], prefix_range[1] + 1, size=num_req).astype(np.int32)
    n_tree = rs["lengths"].integers(0, n_tree_max + 1, size=num_req).astype(np.int32)
    parent = np.full((num_req, n_tree_max), -1, np.int32)
    tokens = np.zeros((num_req, n_tree_max), np.int32)
    m_max = max_verified or (n_tree_max + 1)
    verified = np.zeros((num_req, m_max), np.int32)
    m = np.zeros(num_req, np.int32)
    g = rs["shape"]
    for b in range(num_req):
        nb = int(n_tree[b])
        if nb == 0:
            mm = int(g.integers(0, 2))
            verified[b, :mm] = g.integers(0, vocab, size=mm)
            m[b] = mm
            continue
        par = random_parents(g, nb)
        if forest:
            for i in range(1, nb):
                if g.random() < 0.2:
                    par[i] = -1
        parent[b, :nb] = par
        tokens[b, :nb] = g.integers(0, vocab, size=nb)
        # walk: choose random children (by the generator's own children lists)
        children = {c: [] for c in range(-1, nb)}
        for i in range(nb):
            children[int(par[i])].append(i)
        seq = []
        cur = -1
        while children[cur] and g.random() < p_follow and len(seq) < m_max - 1:
            cur = children[cur][int(g.integers(0, len(children[cur])))]
            seq.append(int(tokens[b, cur]))
        if g.random() < 0.5 and len(seq) < m_max:
            seq.append(int(g.integers(0, vocab)))
        verified[b, :len(seq)] = seq
        m[b] = len(seq)
    return CompactCase(num_req, n_tree_max, prefix, n_tree, parent, tokens, verified, m)


# --------------------------------------------------------------------------
# device copies (torch is imported only when one of these is called)
# --------------------------------------------------------------------------
def bf16_dev(a: np.ndarray):
    """bfloat16 bit patterns (uint16) -> a bfloat16 tensor on the current CUDA device."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def i32_dev(a):
    """Integers -> an int32 tensor on the current CUDA device."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).cuda()


def attn_inputs(case: AttnCase) -> dict:
    """The device tensors of one attention case: q, k_cache, v_cache, prefix_len, n_tree, parent
    (and block_table for paged K/V)."""
    d = {
        "q": bf16_dev(case.q), "k_cache": bf16_dev(case.k), "v_cache": bf16_dev(case.v),
        "prefix_len": i32_dev(case.prefix_len), "n_tree": i32_dev(case.n_tree), "parent": i32_dev(case.parent),
    }
    if case.paged:
        d["block_table"] = i32_dev(case.block_table)
    return d
