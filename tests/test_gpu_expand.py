"""GPU parity: tree_expand and tree_select_subtree (through the C ABI) against
oracle.expand (SwiftSpec summary §3.1.1, §3.1.3, Figure 2).

Candidate tokens are decided on the input logits alone, so they are compared
exactly (ties: lower token id).  Log-probabilities and weights carry the
fp32 log-sum-exp of the row: within LP_TOL of the fp64 oracle.  A pick or a
selection is compared exactly when the oracle's margin at that decision is
above WEIGHT_EPS; inside the margin any tied choice is valid, so there the
test checks validity and continues from the GPU's state."""
import math

import numpy as np
import pytest
import torch

from oracle import expand as E

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():   # on a GPU machine a missing library is an error, not a skip
    import speculative_decoding_tree_forward_gb300 as ts
else:
    ts = None

LP_TOL = 2e-5          # fp32 log-softmax of one row (|lse| < 20) vs fp64
WEIGHT_EPS = 5e-4      # LP_TOL plus fp32 rounding, accumulated over up to a dozen levels


def _gpu_state(tree, b):
    """One request's GPU tree as an oracle DraftTree (candidates with token -1 dropped)."""
    n = int(tree.n_tree[b])
    ct = tree.cand_tok[b, :n].tolist()
    cl = tree.cand_lp[b, :n].double().tolist()
    cand = [[(t, l) for t, l in zip(ct[i], cl[i]) if t >= 0] for i in range(n)]
    taken = [min(t, len(c)) for t, c in zip(tree.cand_taken[b, :n].tolist(), cand)]
    return E.DraftTree(tree.parent[b, :n].tolist(), tree.tokens[b, :n].tolist(),
                       tree.weight[b, :n].double().tolist(), cand, taken)


def _available(otree):
    out = []
    for u in range(otree.n):
        for j in range(otree.taken[u], len(otree.cand[u])):
            out.append((otree.weight[u] + otree.cand[u][j][1], u, j, otree.cand[u][j][0]))
    return sorted(out, key=lambda c: (-c[0], c[1], c[2]))


def _margin(avail, w):
    top = [c[0] for c in avail[: w + 1]]
    return min((top[i] - top[i + 1] for i in range(len(top) - 1)), default=math.inf)


def _run(seed, B, n_max, vocab, w, k, steps, root_w=None, plant_ties=False, logits="normal"):
    rng = np.random.default_rng(seed)
    dev = "cuda"
    tree = ts.DraftTree(B, n_max, k)
    otrees = []
    for b in range(B):
        tok = int(rng.integers(vocab))
        rw = 0.0 if root_w is None else float(root_w[b])
        tree.tokens[b, 0] = tok
        tree.weight[b, 0] = rw
        tree.n_tree[b] = 1
        otrees.append(E.DraftTree([-1], [tok], [float(np.float32(rw))], [[]], [0]))
    rows = torch.full((B, w), -1, dtype=torch.int32, device=dev)
    rows[:, 0] = 0
    ws = None
    for step in range(steps):
        if logits == "int":      # a few distinct values: hundreds of ties at the top of every slice
            lg = rng.integers(-1, 2, size=(B, w, vocab)).astype(np.float32)
        elif logits == "const":  # every logit equal: the k lowest tokens, log-prob -log(vocab)
            lg = np.full((B, w, vocab), 0.25, dtype=np.float32)
        else:
            lg = (rng.normal(size=(B, w, vocab)) * 2.0).astype(np.float32)
        if plant_ties:
            lg[:, :, 5 % vocab] = lg[:, :, 3 % vocab] = lg.max() + 1.0   # equal top logits: lower token first
        logits = torch.from_numpy(lg).to(dev)
        rows_h = rows.cpu().numpy()
        a_args = ts.expand_args(tree, logits, rows, torch.empty_like(rows))
        if ws is None:
            ws = ts.new_workspace(ts.tree_expand_workspace_size(a_args))
        added = ts.tree_expand(tree, logits, rows, workspace=ws)
        torch.cuda.synchronize()
        assert ts.read_device_error(ws) == 0
        added_h = added.cpu().numpy()
        for b in range(B):
            ot = otrees[b]
            # the oracle's state before the picks: candidates of the queried rows
            for r, u in enumerate(rows_h[b]):
                if u >= 0:
                    ot.cand[u] = E.draft_candidates(lg[b, r], k)
                    ot.taken[u] = 0
                    got_t = tree.cand_tok[b, u].tolist()
                    got_l = tree.cand_lp[b, u].double().tolist()
                    exp_t = [t for t, _ in ot.cand[u]] + [-1] * (k - len(ot.cand[u]))
                    assert got_t == exp_t, f"step {step} request {b} node {u}: candidate tokens"
                    for (t, l), gl in zip(ot.cand[u], got_l):
                        assert abs(gl - l) <= LP_TOL, f"candidate log-prob {gl} vs {l}"
            avail = _available(ot)
            margin = _margin(avail, w)
            n_before = ot.n
            exp_added = E.expand_step(ot, [-1] * w, lg[b], w, k, n_max)   # candidates already set above
            got_added = [int(x) for x in added_h[b] if x >= 0]
            n_now = int(tree.n_tree[b])
            assert n_now == n_before + len(got_added) and len(got_added) == len(exp_added)
            assert list(added_h[b][len(got_added):]) == [-1] * (w - len(got_added))
            gs = _gpu_state(tree, b)
            if margin > WEIGHT_EPS:
                assert got_added == exp_added
                assert gs.parent[n_before:] == ot.parent[n_before:] and gs.tokens[n_before:] == ot.tokens[n_before:]
                assert gs.taken == ot.taken
                for node in got_added:
                    assert abs(gs.weight[node] - ot.weight[node]) <= WEIGHT_EPS
            else:
                # near-tie: every GPU pick is among the oracle's best within the margin
                last = avail[len(got_added) - 1][0] if got_added else math.inf
                best = [c for c in avail if c[0] >= last - WEIGHT_EPS]
                for x in got_added:
                    assert any(c[1] == gs.parent[x] and c[3] == gs.tokens[x] for c in best)
                otrees[b] = gs
        rows = added.clone()
    return tree, otrees


@pytest.mark.parametrize("seed,B,n_max,vocab,w,k,steps", [
    (0, 3, 64, 1000, 4, 4, 5),
    (1, 2, 128, 152064, 8, 8, 4),        # several vocab slices, 16-byte path
    (2, 4, 40, 3, 3, 5, 4),              # vocab smaller than k: token -1 past the vocabulary
    (9, 2, 40, 1001, 3, 5, 4),           # odd vocab (4-byte loads)
    (3, 1, 128, 50000, 16, 16, 6),       # the largest w and k
    (4, 5, 20, 4096, 2, 2, 12),          # growth stops at capacity
    (5, 2, 96, 128256, 8, 3, 5),
    (10, 9, 128, 152064, 16, 16, 2),     # 144 rows: 8 slices, three batches of loads per thread
])
def test_expansion_matches_oracle(seed, B, n_max, vocab, w, k, steps):
    _run(seed, B, n_max, vocab, w, k, steps)


def test_expansion_ties_go_to_the_lower_token_and_node():
    _run(6, 2, 64, 300, 4, 4, 3, plant_ties=True)
    # two identical rows under equal weights: equal keys, the lower node gives first
    tree = ts.DraftTree(1, 16, 2)
    tree.n_tree[0] = 3
    tree.parent[0, :3] = torch.tensor([-1, 0, 0], dtype=torch.int32)
    tree.weight[0, :3] = torch.tensor([0.0, -0.5, -0.5])
    row = torch.randn(200)
    logits = torch.stack([row, row]).unsqueeze(0).cuda().float().contiguous()
    rows = torch.tensor([[2, 1]], dtype=torch.int32, device="cuda")
    added = ts.tree_expand(tree, logits, rows)
    torch.cuda.synchronize()
    assert tree.parent[0, 3:5].tolist() == [1, 2] and added[0].tolist() == [3, 4]


@pytest.mark.parametrize("kind,vocab,k", [("int", 20000, 8), ("int", 152064, 16), ("const", 5000, 5),
                                           ("const", 128256, 16), ("int", 1001, 3)])
def test_expansion_with_heavy_ties_matches_oracle(kind, vocab, k):
    """Logits with hundreds or thousands of equal values at the top of each
    vocab slice: the candidates are still the k largest with the lower token
    first."""
    _run(11, 2, 64, vocab, 4, k, 3, logits=kind)


def test_figure2_two_nodes_per_expansion_on_gpu():
    tree, _ = _run(7, 1, 32, 50, 2, 2, 3)
    assert int(tree.n_tree[0]) == 1 + 6


def test_select_subtree_matches_oracle():
    tree, _ = _run(8, 3, 128, 20000, 8, 6, 8)
    B = 3
    for bs in (1, 4, 16, 31, 57, 64, 200):
        out = ts.tree_select_subtree(tree.n_tree, tree.parent, tree.tokens, tree.weight, bs)
        torch.cuda.synchronize()
        for b in range(B):
            gs = _gpu_state(tree, b)
            n = gs.n
            r = E.select_subtree(gs.parent, gs.tokens, gs.weight, n, bs)   # the oracle on the GPU's tree
            ns = int(out["n_sel"][b])
            assert ns == min(bs, n)
            assert out["keep"][b, :ns].tolist() == r.keep
            assert out["new_parent"][b, :ns].tolist() == r.parent
            assert out["new_tokens"][b, :ns].tolist() == r.tokens
            assert out["keep"][b, ns:].tolist() == [-1] * (bs - ns)


def test_select_reports_a_parent_that_is_not_kept():
    dev = "cuda"
    parent = torch.tensor([[-1, 0, 1, 0]], dtype=torch.int32, device=dev)
    weight = torch.tensor([[0.0, -3.0, -0.5, -1.0]], device=dev)      # node 2 outweighs its parent 1
    ws = ts.new_workspace(256)
    out = ts.tree_select_subtree(torch.tensor([4], dtype=torch.int32, device=dev), parent,
                                 torch.arange(4, dtype=torch.int32, device=dev).view(1, 4), weight, 2, workspace=ws)
    torch.cuda.synchronize()
    assert out["keep"][0].tolist() == [0, 2] and out["new_parent"][0].tolist() == [-1, -1]
    assert ts.read_device_error(ws) & ts.TS_DEVERR_BAD_PARENT


def test_expansion_then_attention_on_the_grown_tree():
    """The draft loop on one stream: each expansion appends w nodes, then the
    tree attention queries exactly those nodes, reading the parents and tree
    size the expansion wrote (SwiftSpec summary §3.1.1 and Figure 3: the new
    leaves attend to their ancestors and the prefix)."""
    import dataclasses

    import workloads as W
    from oracle import attention as A
    from gpu_util import attn_inputs, check_attention

    B, w, k, n_max, steps, vocab = 2, 4, 4, 40, 3, 3000
    case = W.random_attn_case(90, num_req=B, hq=16, hkv=4, d=128, n_tree_max=n_max, n_query=w,
                              prefix_range=(100, 400))
    d = attn_inputs(case)
    rng = np.random.default_rng(91)
    tree = ts.DraftTree(B, n_max, k)
    n0 = 12
    for b in range(B):   # a chain of n0 nodes whose last node has candidates
        tree.parent[b, :n0] = torch.arange(-1, n0 - 1, dtype=torch.int32)
        tree.weight[b, :n0] = -torch.arange(n0, dtype=torch.float32) * 0.3
        tree.cand_tok[b, n0 - 1] = torch.from_numpy(rng.choice(vocab, size=k, replace=False).astype(np.int32))
        tree.cand_lp[b, n0 - 1] = torch.tensor([-0.1, -0.5, -1.2, -2.0])
        tree.cand_taken[b, n0 - 1] = 0
    tree.n_tree.fill_(n0)
    out = torch.empty_like(d["q"])
    lse = torch.empty((B, case.num_q_heads, w), dtype=torch.float32, device="cuda")
    a = ts.attn_args(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], tree.n_tree, tree.parent, out, lse,
                     None, case.softmax_scale, 2)
    aws = ts.new_workspace(ts.tree_attn_workspace_size(a))
    rows = torch.full((B, w), -1, dtype=torch.int32, device="cuda")
    for step in range(steps):
        logits = torch.randn((B, w, vocab), device="cuda")
        added = ts.tree_expand(tree, logits, rows)
        ts.tree_attn_forward_args(a, aws)
        torch.cuda.synchronize()
        assert (added >= 0).all()
        n = tree.n_tree.cpu().numpy()
        assert (n == n0 + w * (step + 1)).all()
        grown = dataclasses.replace(case, n_tree=n.astype(np.int32), parent=tree.parent.cpu().numpy())
        check_attention(grown, out, lse, A.attention_case(grown, heads=[0, 5, 11]), heads=[0, 5, 11])
        rows = added
