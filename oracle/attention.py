"""Tree-masked grouped-query attention, fp64, explicit mask, no tiling.

SwiftSpec summary, §3.1.3 and Figure 3 (non-square mask: rows are the new
leaves, columns the prefix plus the whole tree; each leaf sees its ancestors
and itself) and §3.3 (the masked attention kernel).  The NVIDIA draft-length
article defines G as query heads per KV head.

Readings where the pages are silent:
* softmax scale = 1/sqrt(head_dim) unless the caller gives one;
* query head h reads KV head h // G (contiguous groups);
* inputs are finite bf16 values; the softmax is written as its definition,
  exp(s_j) / sum_j exp(s_j), which fp64 evaluates without overflow for
  |s| < 700 (asserted).
"""
from __future__ import annotations

import math

import numpy as np

from .tree import tree_mask

PAGE_SIZE = 16


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> fp64 (a bf16 value is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def logical_rows(cache: np.ndarray, b: int, nrows: int, block_table=None) -> np.ndarray:
    """Rows [0, nrows) of request b.

    Contiguous cache: ``[num_req][max_kv_len][...]``.  Paged cache (MineDraft
    summary, §5.3: vLLM KV blocks): a pool ``[num_blocks][16][...]`` where
    logical row r of request b is row r % 16 of block block_table[b][r // 16].
    """
    if block_table is None:
        return cache[b, :nrows]
    nblk = (nrows + PAGE_SIZE - 1) // PAGE_SIZE
    blocks = [cache[int(block_table[b][j])] for j in range(nblk)]
    if not blocks:
        return cache[:0, 0]
    return np.concatenate(blocks, axis=0)[:nrows]


def tree_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, prefix_len: int, n: int,
                   parent, n_query: int, scale: float, heads=None):
    """One request's tree attention.

    q: [n_query][Hq][d] fp64; k, v: [prefix_len + n][Hkv][d] fp64 (logical rows).
    Returns (out [n_query][Hq][d], lse [Hq][n_query]) with lse the natural-log
    sum of exponentials of the visible scores.  ``heads`` restricts the
    computation to some query heads (others stay zero).
    """
    nq, hq, d = q.shape
    hkv = k.shape[1]
    assert hq % hkv == 0
    g = hq // hkv
    keys = prefix_len + n
    assert k.shape[0] >= keys and v.shape[0] >= keys
    assert np.isfinite(q).all() and np.isfinite(k[:keys]).all() and np.isfinite(v[:keys]).all()
    mask = tree_mask(parent, prefix_len, n, n_query)
    out = np.zeros((nq, hq, d))
    lse = np.zeros((hq, nq))
    for h in (range(hq) if heads is None else heads):
        kvh = h // g
        s = (q[:, h, :] @ k[:keys, kvh, :].T) * scale          # [nq][keys]
        assert np.abs(s).max(initial=0.0) < 700.0
        e = np.where(mask, np.exp(s), 0.0)
        den = e.sum(axis=1)
        out[:, h, :] = (e @ v[:keys, kvh, :]) / den[:, None]
        lse[h] = np.log(den)
    return out, lse


def tree_positions(parent, n: int, prefix_len: int) -> np.ndarray:
    """Position id of each tree node: the prefix length plus the node's depth
    (the root, parent -1, sits at position prefix_len).  Nodes on one root
    path get consecutive positions, siblings share one: the tree positions
    that RoPE inside the verify attention uses (SwiftSpec summary §3.3)."""
    pos = np.zeros(n, dtype=np.int64)
    for i in range(n):
        p = int(parent[i])
        pos[i] = prefix_len if p < 0 else pos[p] + 1
    return pos


def rope(x: np.ndarray, positions, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half convention, fp64: for j < d/2,
    angle = position * theta^(-2j/d), and the pair (x_j, x_{j+d/2}) turns by
    that angle.  x: [rows][heads][d], positions: [rows]."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-2.0 * np.arange(half) / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]      # [rows][half]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (through float32, round to nearest even on the 16
    dropped bits); the attention's operands are bf16."""
    bits = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    rounded = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).astype(np.float64)


def default_scale(head_dim: int, softmax_scale: float = 0.0) -> float:
    return softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(head_dim)


def attention_case(case, requests=None, heads=None, round_rotated_q=True):
    """Oracle outputs for an ``AttnCase``-shaped object (tests only).

    Returns {b: (out [nq][Hq][d], lse [Hq][nq])} for the chosen requests.
    With RoPE, the rotated queries enter the attention as bf16 (the
    attention's operand precision); ``round_rotated_q=False`` keeps the fp64
    rotation instead, to show how much that reading changes the result.
    """
    res = {}
    scale = default_scale(case.head_dim, case.softmax_scale)
    table = case.block_table if case.paged else None
    for b in (range(case.num_req) if requests is None else requests):
        P = int(case.prefix_len[b])
        n = int(case.n_tree[b])
        keys = P + n
        kb = bf16_bits_to_f64(logical_rows(case.k, b, keys, table))
        vb = bf16_bits_to_f64(logical_rows(case.v, b, keys, table))
        qb = bf16_bits_to_f64(case.q[b])
        theta = getattr(case, "rope_theta", 0.0)
        if theta > 0:   # queries at their tree positions, as bf16 operands; K rows are stored rotated
            pos = tree_positions(case.parent[b], n, P)[n - case.n_query:]
            qb = rope(qb, pos, theta)
            if round_rotated_q:
                qb = round_bf16(qb)
        res[b] = tree_attention(qb, kb, vb, P, n, case.parent[b][:n], case.n_query, scale, heads)
    return res
