"""GPU parity: tree_accept_sample (stochastic tree acceptance, through the C
ABI) against oracle.stochastic (MineDraft summary's residual
norm(max(0, p - q)) per child, the bonus by inverse transform).

Accept tests and the bonus draw are decisions on fp32 probabilities (the
GPU) and fp64 ones (the oracle).  The path is compared exactly when every
accept test of the oracle's walk clears MARGIN (relative); the bonus must
fall in the oracle's CDF interval up to fp32 rounding of the prefix sums,
and equal the oracle's when that interval is wide.  Every GPU walk is also
checked to be a valid one, and the law of the emitted token is checked on
the GPU itself by Monte Carlo."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import stochastic as S
from oracle import tree as T

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():   # on a GPU machine a missing library is an error, not a skip
    import speculative_decoding_tree_forward_gb300 as ts
else:
    ts = None
from gpu_util import i32_dev  # noqa: E402

MARGIN = 1e-4


def _walk(tl, dl, tokens, parent, n, temp, u_acc, u_bonus):
    """The oracle's walk, replayed to expose its decisions: the path, the
    smallest relative margin of its accept tests, the final r and the
    bonus target U * sum(r)."""
    children = [[] for _ in range(n)]
    for i in range(1, n):
        if parent[i] >= 0:
            children[parent[i]].append(i)
    u, path, m = 0, [0], math.inf
    while True:
        r, q = S.softmax_t(tl[u], temp), S.softmax_t(dl[u], temp)
        nxt = -1
        for c in children[u]:
            t = int(tokens[c])
            if q[t] > 0:
                ratio = r[t] / q[t]
                m = min(m, abs(float(u_acc[c]) - ratio) / max(1.0, ratio))
                if float(u_acc[c]) < ratio:
                    nxt = c
                    break
            res = np.maximum(0.0, r - q)
            if res.sum() > 0:
                r = res / res.sum()
        if nxt < 0:
            return path, m, r, float(u_bonus[u]) * r.sum()
        path.append(nxt)
        u = nxt


BONUS_EPS = 1e-5   # fp32 prefix sums over up to ~1.5e5 probabilities


def _case(seed, B, n_max, vocab, noise, plain=False):
    acc = W.random_accept_case(seed, num_req=B, n_tree_max=n_max, vocab=vocab, p_accept=0.8)
    rng = np.random.default_rng(seed + 1000)
    if plain:   # N(0, 1) logits with no planted peak; draft tokens follow the oracle's argmax at rate 0.8
        acc.logits[:] = rng.standard_normal(acc.logits.shape, dtype=np.float32)
        for b in range(B):
            n = int(acc.n_tree[b])
            if n == 0:
                continue
            am = T.greedy_accept(acc.logits[b][:n], np.zeros(n, np.int32), acc.parent[b][:n], n).argmax
            acc.tokens[b, :n] = W.draft_tokens(rng, acc.parent[b][:n], np.array(am, np.int32), vocab, 0.8)
    tl = acc.logits.astype(np.float32)
    dl = (tl + rng.normal(size=tl.shape) * noise).astype(np.float32)
    u_acc = rng.random((B, n_max)).astype(np.float32)
    u_bonus = rng.random((B, n_max)).astype(np.float32)
    return acc, tl, dl, u_acc, u_bonus


def _run_gpu(acc, tl, dl, u_acc, u_bonus, temp):
    dev = "cuda"
    out = ts.tree_accept_sample(torch.from_numpy(tl).to(dev), torch.from_numpy(dl).to(dev), i32_dev(acc.tokens),
                                i32_dev(acc.parent), i32_dev(acc.n_tree), torch.from_numpy(u_acc).to(dev),
                                torch.from_numpy(u_bonus).to(dev), temp)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("seed,B,n_max,vocab,noise,temp,plain", [
    (0, 6, 16, 1000, 0.3, 1.0, False),
    (1, 4, 32, 152064, 0.5, 1.0, False),      # several vocab slices, 16-byte rows
    (2, 5, 24, 1001, 0.2, 0.7, False),        # odd vocab (4-byte loads)
    (3, 3, 64, 50000, 1.0, 1.5, False),       # a draft far from the target: many rejections
    (4, 8, 8, 300, 0.05, 1.0, False),         # a draft close to the target: long paths
    (5, 4, 16, 128256, 0.3, 1.0, True),       # plain N(0, 1) logits, no planted peak
    (6, 2, 32, 152064, 0.5, 0.8, True),
])
def test_stochastic_acceptance_matches_oracle(seed, B, n_max, vocab, noise, temp, plain):
    acc, tl, dl, u_acc, u_bonus = _case(seed, B, n_max, vocab, noise, plain)
    got = _run_gpu(acc, tl, dl, u_acc, u_bonus, temp)
    compared = 0
    for b in range(B):
        n = int(acc.n_tree[b])
        if n == 0:
            assert got["accept_len"][b] == 0 and got["bonus"][b] == -1
            continue
        args = (tl[b][:n].astype(np.float64), dl[b][:n].astype(np.float64), acc.tokens[b], acc.parent[b], n, temp,
                u_acc[b], u_bonus[b])
        al = int(got["accept_len"][b])
        path = list(got["path"][b][:al])
        assert all(x == -1 for x in got["path"][b][al:])
        assert path[0] == 0 and all(acc.parent[b][path[i]] == path[i - 1] for i in range(1, al))
        assert 0 <= got["bonus"][b] < vocab
        assert list(got["verified"][b][:al]) == [int(acc.tokens[b][x]) for x in path]
        assert got["verified"][b][al] == got["bonus"][b] and got["verified_len"][b] == al + 1
        opath, margin, r, target = _walk(*args)
        if margin > MARGIN:
            ref = S.stochastic_accept(*args)
            assert path == ref.path == opath, f"request {b}"
            # the bonus: in the oracle's CDF interval, up to fp32 rounding of the prefix sums;
            # exact when that interval is wide
            c = np.cumsum(r)
            v = int(got["bonus"][b])
            lo = c[v - 1] if v > 0 else 0.0
            assert lo - BONUS_EPS * c[-1] <= target <= c[v] + BONUS_EPS * c[-1], f"request {b} bonus {v}"
            olo = c[ref.bonus - 1] if ref.bonus > 0 else 0.0
            if min(target - olo, c[ref.bonus] - target) > BONUS_EPS * c[-1]:
                assert v == ref.bonus
            compared += 1
    assert compared >= B // 2


def test_one_workspace_over_many_calls():
    """The walk's command words are not reset between calls (their numbering
    carries on): six calls of one shape on one workspace, each checked
    against the oracle, the last two on the inputs of the first two."""
    B, n_max, vocab = 4, 24, 20000
    cases = [_case(40 + k, B, n_max, vocab, 0.6, plain=(k % 2 == 1)) for k in range(4)]
    cases += cases[:2]
    ws = None
    for acc, tl, dl, u_acc, u_bonus in cases:
        dev = "cuda"
        a = [torch.from_numpy(tl).to(dev), torch.from_numpy(dl).to(dev), i32_dev(acc.tokens), i32_dev(acc.parent),
             i32_dev(acc.n_tree), torch.from_numpy(u_acc).to(dev), torch.from_numpy(u_bonus).to(dev)]
        if ws is None:
            dummy = {k: torch.empty(1, dtype=torch.int32, device=dev)
                     for k in ("path", "accept_len", "bonus", "verified", "verified_len")}
            probe = ts.sample_args(*a, 1.0, dummy)
            ws = ts.new_workspace(ts.tree_accept_sample_workspace_size(probe), dev)
        got = ts.tree_accept_sample(*a, 1.0, workspace=ws)
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in got.items()}
        assert ts.read_device_error(ws) == 0
        for b in range(B):
            n = int(acc.n_tree[b])
            if n == 0:
                assert got["accept_len"][b] == 0
                continue
            args = (tl[b][:n].astype(np.float64), dl[b][:n].astype(np.float64), acc.tokens[b], acc.parent[b], n, 1.0,
                    u_acc[b], u_bonus[b])
            opath, margin, r, target = _walk(*args)
            al = int(got["accept_len"][b])
            if margin > MARGIN:
                assert list(got["path"][b][:al]) == opath


def test_a_walk_wait_that_runs_out_returns_and_the_next_call_is_right():
    """With the walk's hand-off waits bounded by 1 ns, a helper CTA that polls
    for the first command before the leader has posted it gives up
    (TS_DEVERR_TIMEOUT) and returns, and the leader's wait for that helper's
    answer runs out in turn: the call's outputs are void and the context stays
    usable.  On the workspace zeroed again, a call with the default bound
    matches the oracle."""
    B, n_max, vocab = 4, 24, 20000
    acc, tl, dl, u_acc, u_bonus = _case(60, B, n_max, vocab, 0.6)
    dev = "cuda"
    a = [torch.from_numpy(tl).to(dev), torch.from_numpy(dl).to(dev), i32_dev(acc.tokens), i32_dev(acc.parent),
         i32_dev(acc.n_tree), torch.from_numpy(u_acc).to(dev), torch.from_numpy(u_bonus).to(dev)]
    dummy = {k: torch.empty(1, dtype=torch.int32, device=dev) for k in ("path", "accept_len", "bonus", "verified",
                                                                        "verified_len")}
    ws = ts.new_workspace(ts.tree_accept_sample_workspace_size(ts.sample_args(*a, 1.0, dummy)), dev)
    ts.tree_accept_sample(*a, 1.0, workspace=ws, wait_limit_ns=1)
    torch.cuda.synchronize()
    assert ts.read_device_error(ws) & ts.TS_DEVERR_TIMEOUT
    ws.zero_()
    got = ts.tree_accept_sample(*a, 1.0, workspace=ws)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in got.items()}
    assert ts.read_device_error(ws) == 0
    for b in range(B):
        n = int(acc.n_tree[b])
        if n == 0:
            continue
        args = (tl[b][:n].astype(np.float64), dl[b][:n].astype(np.float64), acc.tokens[b], acc.parent[b], n, 1.0,
                u_acc[b], u_bonus[b])
        opath, margin, r, target = _walk(*args)
        if margin > MARGIN:
            assert list(got["path"][b][:int(got["accept_len"][b])]) == opath


@pytest.mark.parametrize("u_value", [0.0, float(np.float32(1.0) - np.float32(2.0 ** -24))])
def test_bonus_at_either_end_of_the_distribution(u_value):
    """Bonus uniforms of 0 (the first token with r > 0: in the leader's own
    vocab slice) and of the largest float below 1 (the last tokens with
    r > 0: the last slice, where fp32 rounding can put the target past the
    slice sums and the slice's last token with r > 0 is taken), checked
    against the oracle's CDF interval like every bonus."""
    B, n_max, vocab = 4, 16, 30000
    acc, tl, dl, u_acc, u_bonus = _case(70, B, n_max, vocab, 0.8)
    u_bonus = np.full_like(u_bonus, u_value)
    got = _run_gpu(acc, tl, dl, u_acc, u_bonus, 1.0)
    for b in range(B):
        n = int(acc.n_tree[b])
        if n == 0:
            continue
        args = (tl[b][:n].astype(np.float64), dl[b][:n].astype(np.float64), acc.tokens[b], acc.parent[b], n, 1.0,
                u_acc[b], u_bonus[b])
        opath, margin, r, target = _walk(*args)
        if margin <= MARGIN:
            continue
        al = int(got["accept_len"][b])
        assert list(got["path"][b][:al]) == opath
        c = np.cumsum(r)
        v = int(got["bonus"][b])
        assert 0 <= v < vocab
        lo = c[v - 1] if v > 0 else 0.0
        assert lo - BONUS_EPS * c[-1] <= target <= c[v] + BONUS_EPS * c[-1], f"request {b} bonus {v}"
        assert got["verified"][b][al] == v and got["verified_len"][b] == al + 1


def test_near_zero_temperature_is_greedy_acceptance_on_gpu():
    acc, tl, dl, u_acc, u_bonus = _case(7, 6, 24, 2000, 1.0)
    got = _run_gpu(acc, tl, dl, u_acc, u_bonus, 1e-3)
    g = ts.tree_accept_greedy(torch.from_numpy(acc.logits).cuda(), i32_dev(acc.tokens), i32_dev(acc.parent),
                              i32_dev(acc.n_tree))
    torch.cuda.synchronize()
    assert np.array_equal(got["accept_len"], g["accept_len"].cpu().numpy())
    assert np.array_equal(got["bonus"], g["bonus"].cpu().numpy())
    assert np.array_equal(got["path"], g["path"].cpu().numpy())


def test_sure_acceptance_follows_first_children():
    acc, tl, dl, u_acc, u_bonus = _case(8, 4, 20, 700, 2.0)
    got = _run_gpu(acc, tl, dl, np.zeros_like(u_acc), u_bonus, 1.0)
    for b in range(4):
        n = int(acc.n_tree[b])
        if n == 0:
            continue
        u, walk = 0, [0]
        while True:
            kids = [i for i in range(n) if acc.parent[b][i] == u]
            if not kids:
                break
            u = kids[0]
            walk.append(u)
        assert list(got["path"][b][:len(walk)]) == walk and got["accept_len"][b] == len(walk)


def test_emitted_token_follows_the_target_law_on_gpu():
    """4096 requests, each a root with three children drawn from the draft:
    the first emitted token's histogram against the target distribution."""
    B, V, m = 4096, 5, 3
    rng = np.random.default_rng(9)
    row_t = rng.normal(size=V) * 1.5
    row_d = rng.normal(size=V) * 1.5
    p, q = S.softmax_t(row_t, 1.0), S.softmax_t(row_d, 1.0)
    tl = np.tile(row_t.astype(np.float32), (B, m + 1, 1))
    dl = np.tile(row_d.astype(np.float32), (B, m + 1, 1))
    tokens = np.concatenate([np.zeros((B, 1), np.int32), rng.choice(V, size=(B, m), p=q).astype(np.int32)], axis=1)
    parent = np.tile(np.array([-1] + [0] * m, np.int32), (B, 1))
    acc = W.AcceptCase(B, m + 1, V, np.full(B, m + 1, np.int32), parent, tokens, tl, np.zeros((B, m + 1), np.int32))
    got = _run_gpu(acc, tl, dl, rng.random((B, m + 1)).astype(np.float32),
                   rng.random((B, m + 1)).astype(np.float32), 1.0)
    first = np.where(got["accept_len"] > 1, tokens[np.arange(B), np.maximum(got["path"][:, 1], 0)], got["bonus"])
    emp = np.bincount(first, minlength=V) / B
    sigma = np.sqrt(p * (1 - p) / B)
    assert np.all(np.abs(emp - p) <= 4.5 * sigma + 1e-12), (emp, p)
    assert np.abs(q - p).max() > 0.1   # the draft's law is far from the target's


def test_bad_temperature_is_rejected():
    acc, tl, dl, u_acc, u_bonus = _case(10, 2, 8, 100, 0.3)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(ts.TreeSpecError):
            _run_gpu(acc, tl, dl, u_acc, u_bonus, bad)
