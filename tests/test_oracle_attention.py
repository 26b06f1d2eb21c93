"""Pins for the oracle's tree attention.

The oracle is checked against: torch's scaled_dot_product_attention with a
causal mask (a chain-shaped tree is ordinary causal decoding with a prefix,
MineDraft summary / NVIDIA draft-length article: chain verify is standard
speculative decoding); brute force that runs every root path as its own
causal sequence (SwiftSpec summary, Figure 3: a leaf sees its ancestors);
closed forms (V constant per KV head, Q = 0 gives lse = log #visible keys);
invariance to masked keys; and the definition of paged KV blocks.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A


def _f64(case, b):
    P, n = int(case.prefix_len[b]), int(case.n_tree[b])
    table = case.block_table if case.paged else None
    k = A.bf16_bits_to_f64(A.logical_rows(case.k, b, P + n, table))
    v = A.bf16_bits_to_f64(A.logical_rows(case.v, b, P + n, table))
    return A.bf16_bits_to_f64(case.q[b]), k, v, P, n


def test_bf16_widening_known_values():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F7F], np.uint16)
    vals = A.bf16_bits_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[3] == 0.0
    assert vals[2] == 3.140625
    assert vals[5] == (2 - 2 ** -7) * 2.0 ** 127


def test_generator_rounds_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    back = A.bf16_bits_to_f64(W.f32_to_bf16_bits(x))
    assert list(back) == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0]


@pytest.mark.parametrize("seed", range(3))
def test_chain_tree_equals_causal_sdpa(seed):
    case = W.random_attn_case(seed, num_req=2, hq=6, hkv=2, d=32, n_tree_max=9,
                              prefix_range=(0, 30), chain=True)
    G = case.num_q_heads // case.num_kv_heads
    for b in range(case.num_req):
        q, k, v, P, n = _f64(case, b)
        out, _ = A.tree_attention(q, k, v, P, n, case.parent[b], n, case.scale)
        qt = torch.from_numpy(q).permute(1, 0, 2)                      # [Hq][n][d]
        kt = torch.from_numpy(k[:P + n]).permute(1, 0, 2).repeat_interleave(G, 0)
        vt = torch.from_numpy(v[:P + n]).permute(1, 0, 2).repeat_interleave(G, 0)
        causal = torch.ones(n, P + n, dtype=torch.bool).tril(diagonal=P)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=causal,
                                                               scale=case.scale)
        np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_every_root_path_as_its_own_causal_sequence(seed):
    case = W.random_attn_case(seed, num_req=2, hq=4, hkv=2, d=16, n_tree_max=12,
                              prefix_range=(0, 20), ragged_tree=True, n_query=5)
    G = case.num_q_heads // case.num_kv_heads
    for b in range(case.num_req):
        q, k, v, P, n = _f64(case, b)
        nq = case.n_query
        out, lse = A.tree_attention(q, k, v, P, n, case.parent[b][:n], nq, case.scale)
        for r in range(nq):
            u = n - nq + r
            path = []
            x = u
            while x != -1:
                path.append(x)
                x = int(case.parent[b][x])
            seq = list(range(P)) + [P + a for a in reversed(path)]   # the sequence ending at u
            for h in range(case.num_q_heads):
                ks, vs = k[seq, h // G], v[seq, h // G]
                s = ks @ q[r, h] * case.scale
                w = np.exp(s - s.max())
                ref = (w / w.sum()) @ vs
                np.testing.assert_allclose(out[r, h], ref, rtol=0, atol=1e-12)
                assert abs(lse[h, r] - (s.max() + math.log(w.sum()))) < 1e-12


def test_group_mapping_constant_values_per_kv_head():
    case = W.random_attn_case(7, num_req=1, hq=12, hkv=3, d=8, n_tree_max=6, prefix_range=(4, 9))
    q, k, v, P, n = _f64(case, 0)
    for j in range(3):
        v[:, j, :] = 10.0 * (j + 1)
    out, _ = A.tree_attention(q, k, v, P, n, case.parent[0], n, case.scale)
    for h in range(12):
        np.testing.assert_allclose(out[:, h, :], 10.0 * (h // 4 + 1), rtol=1e-14)


def test_value_ones_gives_ones():
    case = W.random_attn_case(1, num_req=1, hq=4, hkv=1, d=8, n_tree_max=7, prefix_range=(0, 5))
    q, k, v, P, n = _f64(case, 0)
    out, _ = A.tree_attention(q, k, np.ones_like(v), P, n, case.parent[0], n, case.scale)
    np.testing.assert_allclose(out, 1.0, rtol=1e-14)


def test_zero_query_lse_counts_visible_keys():
    case = W.random_attn_case(2, num_req=1, hq=2, hkv=1, d=8, n_tree_max=10, prefix_range=(3, 3))
    q, k, v, P, n = _f64(case, 0)
    _, lse = A.tree_attention(np.zeros_like(q), k, v, P, n, case.parent[0], n, case.scale)
    for u in range(n):
        depth = 0
        x = int(case.parent[0][u])
        while x != -1:
            depth += 1
            x = int(case.parent[0][x])
        assert abs(lse[0, u] - math.log(P + depth + 1)) < 1e-12


def test_masked_keys_do_not_change_output():
    case = W.random_attn_case(3, num_req=1, hq=4, hkv=2, d=16, n_tree_max=10, prefix_range=(2, 6))
    q, k, v, P, n = _f64(case, 0)
    par = case.parent[0]
    out, lse = A.tree_attention(q, k, v, P, n, par, n, case.scale)
    u = n - 1
    anc = set()
    x = u
    while x != -1:
        anc.add(x)
        x = int(par[x])
    k2, v2 = k.copy(), v.copy()
    for j in range(n):
        if j not in anc:
            k2[P + j] = 37.0
            v2[P + j] = -1e6
    out2, lse2 = A.tree_attention(q, k2, v2, P, n, par, n, case.scale)
    assert (out2[u] == out[u]).all() and (lse2[:, u] == lse[:, u]).all()


def test_single_key_returns_its_value():
    case = W.random_attn_case(4, num_req=1, hq=2, hkv=2, d=8, n_tree_max=1, prefix_range=(0, 0))
    q, k, v, P, n = _f64(case, 0)
    out, _ = A.tree_attention(q, k, v, 0, 1, [-1], 1, case.scale)
    np.testing.assert_allclose(out[0], v[0], rtol=1e-15)


def test_paged_rows_follow_block_table():
    """Scatter a contiguous cache into a shuffled pool; the oracle must read it back."""
    case = W.random_attn_case(5, num_req=3, hq=4, hkv=2, d=16, n_tree_max=8, prefix_range=(10, 60))
    rng = np.random.default_rng(99)
    rows = case.prefix_len + case.n_tree
    nblk = [(int(r) + 15) // 16 for r in rows]
    perm = rng.permutation(sum(nblk) + 2)
    pool_k = np.zeros((len(perm), 16) + case.k.shape[2:], np.uint16)
    pool_v = np.zeros_like(pool_k)
    table = np.full((3, max(nblk)), -1, np.int32)
    off = 0
    for b in range(3):
        for j in range(nblk[b]):
            blk = perm[off]
            off += 1
            table[b, j] = blk
            lo, hi = 16 * j, min(16 * (j + 1), case.k.shape[1])
            pool_k[blk, : hi - lo] = case.k[b, lo:hi]
            pool_v[blk, : hi - lo] = case.v[b, lo:hi]
    ref = A.attention_case(case)
    case.k, case.v, case.block_table, case.paged = pool_k, pool_v, table, True
    got = A.attention_case(case)
    for b in range(3):
        assert (got[b][0] == ref[b][0]).all() and (got[b][1] == ref[b][1]).all()


def test_named_workloads_have_stated_shapes():
    w = W.tree16_prefix128()
    a = w.attn[0]
    assert a.q.shape == (1, 16, 8, 64) and a.k.shape == (1, 144, 2, 64)
    assert w.accept.logits.shape == (1, 16, 1024)
    w2 = W.expand_w8_prefix2048()
    assert [int(c.prefix_len[0] + c.n_tree[0]) for c in w2.attn] == [2120, 2128, 2136, 2144]
    assert all(c.n_query == 8 for c in w2.attn)
    depths = []
    par = w2.attn[0].parent[0]
    for u in range(64):
        d, x = 0, int(par[u])
        while x != -1:
            d, x = d + 1, int(par[x])
        depths.append(d)
    assert max(depths) <= 8
    # determinism
    w1b = W.tree16_prefix128()
    assert (w1b.attn[0].k == a.k).all() and (w1b.accept.tokens == w.accept.tokens).all()
