"""Pins for oracle.stochastic (stochastic tree acceptance; MineDraft summary's
residual norm(max(0, p - q)), generalised to trees): the emitted token
follows the target distribution when the children are draws from the draft
(Monte Carlo against p), a near-zero temperature reproduces greedy
acceptance, and the acceptance length stays within [1, 1 + depth]."""
import numpy as np
import pytest

import workloads as W
from oracle import stochastic as S
from oracle import tree as T


def _first_token_law(seed, V, m, trials, T_=1.0):
    """Root with m children whose tokens are drawn from q_root: returns the
    empirical law of the first emitted token and p_root."""
    rng = np.random.default_rng(seed)
    tl = rng.normal(size=(m + 1, V)) * 1.5
    dl = rng.normal(size=(m + 1, V)) * 1.5
    p = S.softmax_t(tl[0], T_)
    q = S.softmax_t(dl[0], T_)
    parent = [-1] + [0] * m
    counts = np.zeros(V)
    for _ in range(trials):
        tokens = [0] + list(rng.choice(V, size=m, p=q))
        r = S.stochastic_accept(tl, dl, tokens, parent, m + 1, T_, rng.random(m + 1), rng.random(m + 1))
        first = tokens[r.path[1]] if len(r.path) > 1 else r.bonus
        counts[first] += 1
    return counts / trials, p


@pytest.mark.parametrize("seed,V,m", [(0, 5, 1), (1, 5, 3), (2, 7, 4), (3, 3, 6)])
def test_emitted_token_follows_the_target_distribution(seed, V, m):
    trials = 20000
    emp, p = _first_token_law(seed, V, m, trials)
    sigma = np.sqrt(p * (1 - p) / trials)
    assert np.all(np.abs(emp - p) <= 4.5 * sigma + 1e-12), (emp, p)


def test_the_law_is_not_the_draft_law():
    # the same test has power: the draft's own law is far from the target's here
    emp, p = _first_token_law(4, 5, 2, 4000)
    rng = np.random.default_rng(4)
    rng.normal(size=(3, 5))                       # the target rows of _first_token_law
    q = S.softmax_t(rng.normal(size=(3, 5))[0] * 1.5, 1.0)
    assert np.abs(q - p).max() > 0.1 and np.abs(emp - p).max() < np.abs(q - p).max()


@pytest.mark.parametrize("seed", range(5))
def test_near_zero_temperature_is_greedy_acceptance(seed):
    case = W.random_accept_case(seed, num_req=3, n_tree_max=24, vocab=300, p_accept=0.8)
    rng = np.random.default_rng(100 + seed)
    for b in range(3):
        n = int(case.n_tree[b])
        if n == 0:
            continue
        tl = case.logits[b][:n].astype(np.float64)
        dl = rng.normal(size=tl.shape)
        g = T.greedy_accept(case.logits[b], case.tokens[b], case.parent[b], n)
        r = S.stochastic_accept(tl, dl, case.tokens[b], case.parent[b], n, 1e-4, rng.random(n), rng.random(n))
        assert r.path == g.path and r.bonus == g.bonus


def test_acceptance_length_bounds_and_sure_acceptance():
    rng = np.random.default_rng(9)
    for trial in range(30):
        n = int(rng.integers(1, 20))
        par = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        depth = max(T.depth(par, i) for i in range(n))
        V = 6
        tl, dl = rng.normal(size=(n, V)), rng.normal(size=(n, V))
        tokens = list(rng.integers(0, V, size=n))
        r = S.stochastic_accept(tl, dl, tokens, par, n, 1.0, rng.random(n), rng.random(n))
        assert 1 <= r.accept_len <= 1 + depth and 0 <= r.bonus < V
        assert all(par[r.path[i]] == r.path[i - 1] for i in range(1, len(r.path)))
        # U_acc = 0: the first child is always taken (its target probability is > 0)
        r0 = S.stochastic_accept(tl, dl, tokens, par, n, 1.0, np.zeros(n), rng.random(n))
        u, walk = 0, [0]
        while True:
            kids = [i for i in range(n) if par[i] == u]
            if not kids:
                break
            u = kids[0]
            walk.append(u)
        assert r0.path == walk


def test_inverse_transform_sampling():
    r = np.array([0.1, 0.0, 0.6, 0.3])
    assert [S.sample_inverse(r, u) for u in (0.0, 0.0999, 0.1, 0.69, 0.7, 0.9999)] == [0, 0, 2, 2, 3, 3]
    assert S.sample_inverse(r * 7.0, 0.5) == 2    # unnormalised weights
