"""The seeded input generators follow the stated recipe: the same seed gives
the same bytes; trees are topological with the stated depth caps; draft
tokens follow the target's planted argmax with the stated probability and
siblings carry distinct tokens; paged pools cover each request with distinct
blocks.  (Host logic only; these generators hold none of the method's
arithmetic.)"""
import numpy as np
import pytest

import workloads as W
from oracle import tree as T


def _depths(parent):
    return [T.depth(list(parent), i) for i in range(len(parent))]


def test_same_seed_same_bytes():
    a, b = W.tree16_prefix128(0), W.tree16_prefix128(0)
    for x, y in ((a.attn[0].q, b.attn[0].q), (a.attn[0].k, b.attn[0].k), (a.attn[0].parent, b.attn[0].parent),
                 (a.accept.logits, b.accept.logits), (a.accept.tokens, b.accept.tokens)):
        assert np.array_equal(x, y)
    c = W.tree16_prefix128(1)
    assert not np.array_equal(a.attn[0].q, c.attn[0].q)
    x, y = W.random_attn_case(7, paged=True), W.random_attn_case(7, paged=True)
    assert np.array_equal(x.k, y.k) and np.array_equal(x.block_table, y.block_table)


@pytest.mark.parametrize("seed", range(5))
def test_random_parents_are_topological_and_respect_the_depth_cap(seed):
    rng = np.random.default_rng(seed)
    for cap in (None, 1, 3, 8):
        par = W.random_parents(rng, 64, cap)
        assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, 64))
        if cap is not None:
            assert max(_depths(par)) <= cap


def test_chain_parents():
    assert list(W.chain_parents(5)) == [-1, 0, 1, 2, 3]


@pytest.mark.parametrize("p_accept", [0.0, 0.7, 1.0])
def test_draft_tokens_follow_the_planted_argmax_and_siblings_differ(p_accept):
    rng = np.random.default_rng(3)
    n, V = 120, 5000
    par = W.random_parents(rng, n)
    _, peak = W.planted_logits(rng, n, V)
    hits, trials = 0, 0
    for rep in range(20):
        tok = W.draft_tokens(rng, par, peak, V, p_accept)
        for u in range(n):
            kids = [i for i in range(1, n) if par[i] == u]
            assert len({int(tok[i]) for i in kids}) == len(kids)   # distinct siblings
            if kids:
                # the first child of a node is never blocked by a sibling, so it follows the peak w.p. p
                trials += 1
                hits += int(tok[kids[0]] == peak[u])
    rate = hits / trials
    if p_accept == 1.0:
        assert rate == 1.0
    elif p_accept == 0.0:
        assert rate < 0.01                                          # only a chance draw (1/V) matches
    else:
        sigma = np.sqrt(p_accept * (1 - p_accept) / trials)
        assert abs(rate - p_accept) < 5 * sigma + 1.0 / V


def test_planted_peak_is_each_rows_unique_argmax():
    rng = np.random.default_rng(4)
    lg, peak = W.planted_logits(rng, 64, 128256)
    assert np.array_equal(lg.argmax(axis=1), peak)
    srt = np.sort(lg, axis=1)
    assert (srt[:, -1] > srt[:, -2]).all()


def test_paged_pool_covers_every_request_with_distinct_blocks():
    a = W.random_attn_case(8, num_req=6, paged=True, chain=True, n_tree_max=5, prefix_range=(0, 300))
    used = []
    for b in range(a.num_req):
        need = (int(a.prefix_len[b]) + int(a.n_tree[b]) + W.PAGE_SIZE - 1) // W.PAGE_SIZE
        row = a.block_table[b]
        assert (row[:need] >= 0).all() and (row[need:] == -1).all()
        used += list(row[:need])
    assert len(used) == len(set(used)) and max(used) < a.k.shape[0]
    # a chain verify: every tree is a chain of n_query nodes
    assert all(list(a.parent[b]) == list(W.chain_parents(a.n_tree_max)) for b in range(a.num_req))


def test_expansion_workload_trees_have_depth_at_most_eight():
    wl = W.expand_w8_prefix2048(0)
    par = wl.attn[0].parent[0]
    n0 = 64
    assert max(_depths(par[:n0])) <= 8
