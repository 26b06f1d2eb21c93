"""Pins for the oracle's tree bookkeeping: mask, greedy acceptance, re-root.

Each test pins ``oracle.tree`` to something other than itself: the worked
figures of the SwiftSpec summary (fixtures under tests/golden/), closed forms
(E[AL] of a chain, the AL range of the NVIDIA draft-length article) and brute
force over every root path.
"""
import json
import os

import numpy as np
import pytest

import workloads as W
from oracle import tree as T

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# mask (SwiftSpec summary, Figure 3)
# --------------------------------------------------------------------------
def test_fig3_mask_row_t7():
    g = _load("fig3_mask.json")
    names = g["tokens"]
    mask = T.tree_mask(g["parent"], g["prefix_len"], len(names), g["n_query"])
    assert list(mask.shape) == g["mask_shape"]
    first_query = len(names) - g["n_query"]
    row = mask[names.index(g["query"]) - first_query]
    assert [names[j] for j in np.nonzero(row)[0]] == g["visible"]


def test_mask_chain_is_causal_and_prefix_always_visible():
    n, P = 9, 5
    mask = T.tree_mask(W.chain_parents(n), P, n, n)
    expect = np.zeros((n, P + n), bool)
    for r in range(n):
        expect[r, : P + r + 1] = True      # key j visible iff j <= P + r
    assert (mask == expect).all()


def test_mask_star_sees_root_and_self_only():
    n = 7
    parent = np.array([-1] + [0] * (n - 1))
    mask = T.tree_mask(parent, 0, n, n)
    for r in range(1, n):
        assert set(np.nonzero(mask[r])[0]) == {0, r}


def test_mask_rejects_non_topological_parent():
    with pytest.raises(AssertionError):
        T.tree_mask([-1, 2, 0], 0, 3, 3)


# --------------------------------------------------------------------------
# greedy acceptance
# --------------------------------------------------------------------------
def _logits_with_argmax(argmax, vocab):
    lg = np.zeros((len(argmax), vocab), np.float32)
    for i, a in enumerate(argmax):
        lg[i, a] = 1.0
    return lg


def test_fig2_target_verify():
    g = _load("fig2_walkthrough.json")["target_verify"]
    lg = _logits_with_argmax(g["argmax"], g["vocab"])
    r = T.greedy_accept(lg, g["tokens"], g["parent"], len(g["tokens"]))
    e = g["expect"]
    assert r.path == e["path"] and r.accept_len == e["accept_len"]
    assert r.bonus == e["bonus"] and r.verified == e["verified"]


def _brute_force_accept(logits, tokens, parent, n):
    """Every node's root path checked edge by edge; keep the longest (lowest index on ties)."""
    best = None
    for u in range(n):
        path = []
        x = u
        while x != -1:
            path.append(x)
            x = int(parent[x])
        path.reverse()
        if path[0] != 0:
            continue
        ok = all(int(tokens[c]) == int(np.argmax(logits[a])) for a, c in zip(path, path[1:]))
        if ok and (best is None or len(path) > len(best)):
            best = path
    return best


@pytest.mark.parametrize("seed", range(12))
def test_accept_matches_brute_force_and_al_range(seed):
    case = W.random_accept_case(seed, num_req=4, n_tree_max=12, vocab=6, p_accept=0.6,
                                distinct_siblings=bool(seed % 2))
    for b in range(case.num_req):
        n = int(case.n_tree[b])
        par, tok, lg = case.parent[b][:n], case.tokens[b][:n], case.logits[b][:n]
        r = T.greedy_accept(lg, tok, par, n)
        assert r.path == _brute_force_accept(lg, tok, par, n)
        maxdepth = max(T.depth(par, u) for u in range(n))
        assert 1 <= r.accept_len <= 1 + maxdepth <= n
        assert r.bonus == int(np.argmax(lg[r.path[-1]]))
        assert len(r.verified) == r.accept_len + 1


def test_accept_chain_all_match_gives_full_length():
    case = W.random_accept_case(3, num_req=3, n_tree_max=9, vocab=500, p_accept=1.0,
                                chain=True, ragged_tree=False)
    for b in range(case.num_req):
        r = T.greedy_accept(case.logits[b], case.tokens[b], case.parent[b], 9)
        assert r.accept_len == 9 and r.path == list(range(9))


def test_accept_forced_mismatch_gives_al_one():
    case = W.random_accept_case(5, num_req=3, n_tree_max=10, vocab=300)
    for b in range(case.num_req):
        n = int(case.n_tree[b])
        tok = case.tokens[b][:n].copy()
        for i in range(1, n):
            tok[i] = (case.planted[b][case.parent[b][i]] + 1) % case.vocab
        r = T.greedy_accept(case.logits[b][:n], tok, case.parent[b][:n], n)
        assert r.accept_len == 1 and r.path == [0]
        assert r.bonus == case.planted[b][0]


def test_accept_argmax_tie_goes_to_lowest_token():
    lg = np.zeros((2, 8), np.float32)
    lg[0, [2, 5]] = 3.0
    r = T.greedy_accept(lg, [7, 5], [-1, 0], 2)
    assert r.argmax[0] == 2 and r.accept_len == 1
    r = T.greedy_accept(lg, [7, 2], [-1, 0], 2)
    assert r.accept_len == 2


def test_accept_equal_length_paths_prefer_lowest_last_index():
    # node 0 has two children carrying the argmax token: both accepted, same depth
    lg = np.zeros((3, 4), np.float32)
    lg[0, 1] = 1.0
    r = T.greedy_accept(lg, [0, 1, 1], [-1, 0, 0], 3)
    assert r.path == [0, 1]


def test_accept_expected_length_closed_form_on_chains():
    """E[AL] = sum_{j=0..D} q^j, q = p + (1-p)/V (independent per-token acceptance).

    NVIDIA draft-length article: AL counts accepted drafts plus the target's
    token; with each draft accepted independently with probability q the
    prefix of matches is geometric, truncated at D.
    """
    D, V, p = 7, 64, 0.7
    case = W.random_accept_case(11, num_req=3000, n_tree_max=D + 1, vocab=V, p_accept=p,
                                chain=True, ragged_tree=False)
    al = np.array([T.greedy_accept(case.logits[b], case.tokens[b], case.parent[b], D + 1).accept_len
                   for b in range(case.num_req)], dtype=np.float64)
    q = p + (1 - p) / V
    expect = sum(q ** j for j in range(D + 1))
    sem = al.std(ddof=1) / np.sqrt(len(al))
    assert abs(al.mean() - expect) < 5 * sem, (al.mean(), expect, sem)
    assert al.min() >= 1 and al.max() <= D + 1


def test_planted_peak_is_the_argmax():
    case = W.random_accept_case(2, num_req=4, n_tree_max=8, vocab=2000)
    am = case.logits.argmax(axis=2)
    assert (am == case.planted).all()


def test_empty_tree_accept():
    r = T.greedy_accept(np.zeros((0, 4), np.float32), [], [], 0)
    assert r.accept_len == 0 and r.bonus == -1 and r.path == []


# --------------------------------------------------------------------------
# re-root + compaction (SwiftSpec summary, §3.2, Figures 2 and 4)
# --------------------------------------------------------------------------
def test_fig4_compaction():
    g = _load("fig4_compaction.json")
    e = g["expect"]
    P = len(g["prefix_tokens"])
    toks = g["tokens"]
    r = T.reroot(g["parent"], toks, len(toks), P, g["verified"])
    assert [toks[u] for u in r.path] == e["promoted"]
    assert r.new_tokens == e["tree_after"] and r.new_parent == e["tree_parent_after"]
    kept = {toks[u] for u in r.src}
    assert sorted(set(toks) - kept) == e["dropped"]
    assert r.new_prefix_len == e["new_prefix_len"] and r.new_n_tree == e["new_n_tree"]
    # KV rows: tag every row with its own index and apply the move
    rows = np.arange(P + len(toks))[:, None].repeat(3, axis=1)
    moved = T.compact_rows(rows, P, r.src)
    for old, new in e["row_moves"]:
        assert (moved[new] == old).all()
    assert (moved[:P] == rows[:P]).all()
    # the tokens now in the prefix region, in order
    full = g["prefix_tokens"] + toks
    assert [full[int(moved[i, 0])] for i in range(r.new_prefix_len)] == g["prefix_tokens"] + e["promoted"]


def test_fig2_draft_reroots():
    g = _load("fig2_walkthrough.json")
    for key in ("draft_iter1", "draft_iter2"):
        c = g[key]
        e = c["expect"]
        r = T.reroot(c["parent"], c["tokens"], len(c["tokens"]), c["prefix_len"], c["verified"])
        assert [c["tokens"][u] for u in r.path] == e["promoted"]
        assert r.new_tokens == e["tree_after"]
        if "tree_parent_after" in e:
            assert r.new_parent == e["tree_parent_after"]
        assert r.new_prefix_len == e["new_prefix_len"] and r.new_n_tree == e["new_n_tree"]
        assert len(r.survivors) == e["reused"]
    # iteration 2 continues from iteration 1's result
    c1 = g["draft_iter1"]
    r1 = T.reroot(c1["parent"], c1["tokens"], 12, c1["prefix_len"], c1["verified"])
    c2 = g["draft_iter2"]
    assert r1.new_tokens == c2["tokens"] and r1.new_parent == c2["parent"]
    assert r1.new_prefix_len == c2["prefix_len"]


def test_reroot_empty_verified_is_identity():
    case = W.random_compact_case(4, num_req=5)
    for b in range(case.num_req):
        n = int(case.n_tree[b])
        r = T.reroot(case.parent[b][:n], case.tokens[b][:n], n, int(case.prefix_len[b]), [])
        assert r.src == list(range(n)) and r.path == []
        assert r.new_parent == [int(x) for x in case.parent[b][:n]]
        assert r.new_prefix_len == int(case.prefix_len[b])


def _root_path_tokens(parent, tokens, u, stop=-1):
    seq = []
    while u != stop:
        seq.append(int(tokens[u]))
        u = int(parent[u])
    return tuple(reversed(seq))


@pytest.mark.parametrize("seed", range(10))
def test_reroot_invariants(seed):
    case = W.random_compact_case(seed, num_req=6, n_tree_max=20, vocab=4, forest=bool(seed % 2))
    for b in range(case.num_req):
        n = int(case.n_tree[b])
        P = int(case.prefix_len[b])
        par, tok = case.parent[b][:n], case.tokens[b][:n]
        v = case.verified[b][: int(case.m[b])]
        r = T.reroot(par, tok, n, P, v)
        # valid tree, sizes, strictly increasing source list (so dst <= src)
        T.check_tree(r.new_parent, r.new_n_tree)
        assert r.new_prefix_len + r.new_n_tree == P + len(r.src)
        assert all(a < b2 for a, b2 in zip(r.src, r.src[1:]))
        # promoted tokens are a prefix of the verified sequence
        assert [int(tok[u]) for u in r.path] == [int(x) for x in v[: len(r.path)]]
        # survivors: same token sequences below the new root as below the last matched node
        cur = r.path[-1] if r.path else -1
        old = sorted(_root_path_tokens(par, tok, u, cur) for u in r.survivors)
        new = sorted(_root_path_tokens(r.new_parent, r.new_tokens, j) for j in range(r.new_n_tree))
        assert old == new
        if len(r.path) < len(v):
            assert r.survivors == []
        # rows below P are untouched and moved rows carry their source
        rows = np.arange(P + n + 2)
        moved = T.compact_rows(rows, P, r.src)
        assert (moved[:P] == rows[:P]).all()
        assert [int(x) for x in moved[P:P + len(r.src)]] == [P + s for s in r.src]


def test_target_side_verified_tokens_leave_no_survivors():
    """Under greedy acceptance the bonus never labels a child of the last accepted node.

    Holds for trees whose siblings carry distinct tokens (a drafter expands a
    node into distinct tokens); then the token walk retraces the accepted path.
    """
    case = W.random_accept_case(8, num_req=20, n_tree_max=14, vocab=5, p_accept=0.8)
    for b in range(case.num_req):
        n = int(case.n_tree[b])
        a = T.greedy_accept(case.logits[b][:n], case.tokens[b][:n], case.parent[b][:n], n)
        r = T.reroot(case.parent[b][:n], case.tokens[b][:n], n, 100, a.verified)
        assert r.path == a.path and r.survivors == []
        assert r.new_prefix_len == 100 + a.accept_len
