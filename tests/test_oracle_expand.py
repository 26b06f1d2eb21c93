"""Pins for oracle.expand (maximum-likelihood expansion and subtree selection,
SwiftSpec summary §3.1.1 and §3.1.3, Figure 2): closed forms of the
log-softmax candidates, weights against products of softmax probabilities,
the step's picks against a brute-force sort of every available candidate,
the subtree against exhaustive search over all subtrees of bs nodes."""
import itertools
import math

import numpy as np
import pytest

from oracle import expand as E


# ---------------------------------------------------------------- candidates
def test_candidates_of_a_uniform_distribution():
    c = E.draft_candidates(np.zeros(50), 4)
    assert [t for t, _ in c] == [0, 1, 2, 3]   # ties: lower token id
    for _, lp in c:
        assert lp == pytest.approx(-math.log(50), abs=1e-12)


def test_candidates_of_two_tokens():
    a, b = 1.25, -0.5
    c = E.draft_candidates(np.array([b, a]), 2)
    assert [t for t, _ in c] == [1, 0]
    assert c[0][1] == pytest.approx(-math.log1p(math.exp(b - a)), abs=1e-12)
    assert c[1][1] == pytest.approx(-math.log1p(math.exp(a - b)), abs=1e-12)


def test_candidates_cover_the_distribution_and_ignore_shifts():
    rng = np.random.default_rng(0)
    x = rng.normal(size=37) * 3
    c = E.draft_candidates(x, 37)
    assert sum(math.exp(lp) for _, lp in c) == pytest.approx(1.0, abs=1e-12)
    assert all(c[i][1] >= c[i + 1][1] for i in range(36))
    assert sorted(t for t, _ in c) == list(range(37))
    c2 = E.draft_candidates(x + 123.5, 5)
    for (t1, l1), (t2, l2) in zip(c[:5], c2):
        assert t1 == t2 and l1 == pytest.approx(l2, abs=1e-9)


# ---------------------------------------------------------------- expansion
def _grow(seed, vocab, w, k, steps, capacity, root_weight=0.0):
    """Grow a tree from a root; logits of every node drawn when it is queried."""
    rng = np.random.default_rng(seed)
    tree = E.DraftTree([-1], [int(rng.integers(vocab))], [root_weight], [[]], [0])
    node_logits = {}
    rows = [0]
    history = []
    for _ in range(steps):
        lg = rng.normal(size=(len(rows), vocab)) * 2.0
        for r, u in enumerate(rows):
            node_logits[u] = lg[r]
        before = _available(tree, rows, lg, k)
        added = E.expand_step(tree, rows, lg, w, k, capacity)
        history.append((before, added))
        rows = added
    return tree, node_logits, history


def _available(tree, rows, lg, k):
    """Every candidate available to the coming step, found independently:
    (weight, node, rank, token) over all ranks not yet taken."""
    cand = {u: list(tree.cand[u]) for u in range(tree.n)}
    taken = dict(enumerate(tree.taken))
    for r, u in enumerate(rows):
        p = np.exp(lg[r] - lg[r].max())
        p /= p.sum()
        order = sorted(range(lg.shape[1]), key=lambda v: (-lg[r][v], v))[:k]
        cand[u] = [(v, math.log(p[v])) for v in order]
        taken[u] = 0
    out = []
    for u, cs in cand.items():
        for j in range(taken[u], len(cs)):
            out.append((tree.weight[u] + cs[j][1], u, j, cs[j][0]))
    return out


@pytest.mark.parametrize("seed,vocab,w,k,steps", [(1, 6, 2, 2, 3), (2, 5, 3, 3, 4), (3, 9, 4, 2, 3), (4, 4, 2, 4, 5)])
def test_each_step_takes_the_best_available_candidates(seed, vocab, w, k, steps):
    tree, _, history = _grow(seed, vocab, w, k, steps, capacity=200)
    for before, added in history:
        best = sorted(before, key=lambda c: (-c[0], c[1], c[2]))[:w]
        assert len(added) == len(best)
        for node, (wt, u, _, tok) in zip(added, best):
            assert tree.parent[node] == u and tree.tokens[node] == tok
            assert tree.weight[node] == pytest.approx(wt, abs=1e-12)


def test_weights_are_log_products_of_softmax_probabilities():
    tree, node_logits, _ = _grow(5, 7, 3, 3, 4, capacity=200, root_weight=-0.25)
    for i in range(1, tree.n):
        prob, u = 1.0, i
        while tree.parent[u] >= 0:
            lg = node_logits[tree.parent[u]]
            e = np.exp(lg - lg.max())
            prob *= e[tree.tokens[u]] / e.sum()
            u = tree.parent[u]
        assert tree.weight[i] == pytest.approx(-0.25 + math.log(prob), abs=1e-10)
        assert tree.weight[i] <= tree.weight[tree.parent[i]] + 1e-15


def test_figure2_counts_two_nodes_per_expansion():
    tree, _, history = _grow(6, 50, 2, 2, 3, capacity=200)
    assert [len(a) for _, a in history] == [2, 2, 2] and tree.n == 1 + 6


def test_growth_stops_at_capacity_and_when_candidates_run_out():
    tree, _, history = _grow(7, 10, 4, 4, 3, capacity=6)
    assert tree.n == 6 and [len(a) for _, a in history] == [4, 1, 0]
    tree, _, history = _grow(8, 10, 3, 1, 1, capacity=50)   # one candidate per node
    assert [len(a) for _, a in history] == [1]


# ---------------------------------------------------------------- selection
def _closed(subset, parent):
    s = set(subset)
    return all(parent[i] < 0 or parent[i] in s for i in subset)


@pytest.mark.parametrize("seed", range(6))
def test_selected_subtree_maximises_expected_accepted_nodes(seed):
    tree, _, _ = _grow(10 + seed, 6, 2, 3, 3, capacity=9)
    n = tree.n
    for bs in range(1, n + 1):
        r = E.select_subtree(tree.parent, tree.tokens, tree.weight, n, bs)
        assert len(r.keep) == bs and r.keep[0] == 0 and _closed(r.keep, tree.parent)
        got = sum(math.exp(tree.weight[i]) for i in r.keep)
        best = max(sum(math.exp(tree.weight[i]) for i in c)
                   for c in itertools.combinations(range(n), bs) if _closed(c, tree.parent))
        assert got == pytest.approx(best, rel=1e-12)
        for j, i in enumerate(r.keep):   # remapped parents point at the same nodes
            p = tree.parent[i]
            assert (r.parent[j] == -1) if p < 0 else (r.keep[r.parent[j]] == p)
            assert r.tokens[j] == tree.tokens[i]


def test_selecting_everything_is_the_identity():
    tree, _, _ = _grow(20, 5, 2, 2, 2, capacity=50)
    r = E.select_subtree(tree.parent, tree.tokens, tree.weight, tree.n, tree.n + 3)
    assert r.keep == list(range(tree.n)) and r.parent == tree.parent and r.tokens == tree.tokens
