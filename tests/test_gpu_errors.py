"""GPU: the kernels' handling of malformed inputs and of a bounded wait that
runs out.  Every fault here is made on the host (a corrupted block-table
entry, a length beyond its bound, a token outside the vocab, a wait bound of
one nanosecond); none traps or hangs the GPU.  Each case checks the
TS_DEVERR_* bit of the workspace's error word and the stated behaviour
(rows of a bad block read as zeros and are not moved, lengths clamped,
tokens never accepted, an aborted call returns and the next call is right)
against the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import tree as T

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():   # on a GPU machine a missing library is an error, not a skip
    import speculative_decoding_tree_forward_gb300 as ts
else:
    ts = None
from gpu_util import attn_inputs, check_attention, i32_dev  # noqa: E402

PAGE = W.PAGE_SIZE


def _attn(case, d, path, ws=None, **kw):
    a_out = torch.empty_like(d["q"])
    lse = torch.empty((case.num_req, case.num_q_heads, case.n_query), dtype=torch.float32, device="cuda")
    a = ts.attn_args(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"], a_out, lse,
                     d.get("block_table"), case.softmax_scale, path, kw.get("num_ctas", 0), 0.0,
                     kw.get("wait_limit_ns", 0))
    if ws is None:
        ws = ts.new_workspace(ts.tree_attn_workspace_size(a))
    ts.tree_attn_forward_args(a, ws)
    torch.cuda.synchronize()
    return a_out, lse, ts.read_device_error(ws)


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("path", [1, 2])
def test_attention_reads_a_bad_block_as_zero_rows(path):
    """A block-table entry outside [0, num_blocks): its 16 rows read as zeros
    (they still take part in the softmax with score 0 and value 0), and
    TS_DEVERR_BAD_BLOCK is set."""
    kw = (dict(num_req=3, hq=64, hkv=8, d=128, n_tree_max=5, chain=True) if path == 2
          else dict(num_req=3, hq=8, hkv=2, d=64, n_tree_max=12))
    case = W.random_attn_case(700 + path, prefix_range=(100, 300), paged=True, **kw)
    b, page = 1, 3   # a prefix page of request 1 (P >= 100 keys, so page 3 holds keys 48..63)
    table = case.block_table.copy()
    blk = int(table[b, page])
    table[b, page] = case.k.shape[0] + 5
    # the oracle sees the same cache with that block's rows zero (the block
    # belongs to request 1 only: the table is a permutation of the pool)
    k0, v0 = case.k.copy(), case.v.copy()
    k0[blk] = 0
    v0[blk] = 0
    ref = A.attention_case(dataclasses.replace(case, k=k0, v=v0))
    d = attn_inputs(case)
    d["block_table"] = i32_dev(table)
    out, lse, err = _attn(case, d, path)
    assert err & ts.TS_DEVERR_BAD_BLOCK
    check_attention(case, out, lse, ref)


@pytest.mark.parametrize("path", [1, 2])
def test_attention_clamps_lengths_beyond_their_bounds(path):
    """n_tree above n_tree_max and a prefix running past the cache are clamped
    (to n_tree_max, and to max_kv_len - n) and TS_DEVERR_BAD_LENGTH is set."""
    kw = (dict(num_req=3, hq=64, hkv=8, d=128, n_tree_max=16) if path == 2
          else dict(num_req=3, hq=8, hkv=2, d=64, n_tree_max=16))
    case = W.random_attn_case(710 + path, prefix_range=(50, 400), **kw)
    bad_n, bad_p = case.n_tree.copy(), case.prefix_len.copy()
    bad_n[0] = case.n_tree_max + 7
    bad_p[2] = case.max_kv_len + 100
    clamped = dataclasses.replace(case, n_tree=case.n_tree.copy(), prefix_len=case.prefix_len.copy())
    clamped.n_tree[0] = case.n_tree_max
    clamped.prefix_len[2] = case.max_kv_len - int(case.n_tree[2])
    d = attn_inputs(case)
    d["n_tree"], d["prefix_len"] = i32_dev(bad_n), i32_dev(bad_p)
    out, lse, err = _attn(case, d, path)
    assert err & ts.TS_DEVERR_BAD_LENGTH
    check_attention(case, out, lse, A.attention_case(clamped))


@pytest.mark.parametrize("path", [1, 2])
def test_a_wait_that_runs_out_returns_and_the_next_call_is_right(path):
    """With every pipeline wait bounded by 1 ns, the first wait that does not
    find its data already there runs out: the kernel sets TS_DEVERR_TIMEOUT,
    waits (with the default bound) for its own copies in flight, frees its
    tensor memory and returns.  The call's outputs are void; the context stays
    usable, and a call with the default bound on a fresh workspace is right.
    Eight CTAs share the keys, so each one streams many more tiles than its
    ring holds and its loader has to wait for free slots."""
    kw = (dict(num_req=4, hq=64, hkv=8, d=128, n_tree_max=16) if path == 2
          else dict(num_req=4, hq=8, hkv=2, d=64, n_tree_max=16))
    case = W.random_attn_case(720 + path, prefix_range=(3000, 6000), **kw)
    d = attn_inputs(case)
    _, _, err = _attn(case, d, path, wait_limit_ns=1, num_ctas=8)
    assert err & ts.TS_DEVERR_TIMEOUT
    out, lse, err2 = _attn(case, d, path)
    assert err2 == 0
    check_attention(case, out, lse, A.attention_case(case, heads=[0, case.num_q_heads - 1]),
                    heads=[0, case.num_q_heads - 1])


# ------------------------------------------------------------------ acceptance
def _accept_case():
    case = W.random_accept_case(730, num_req=3, n_tree_max=16, vocab=5000, p_accept=0.9, ragged_tree=False)
    bad = case.tokens.copy()
    bad[0, 1] = case.vocab + 3     # a child of the root
    bad[1, 5] = -2
    bad[2, 0] = case.vocab + 11    # the root's own token: not tested, not reported
    return case, bad


def test_greedy_acceptance_never_accepts_a_token_outside_the_vocab():
    case, bad = _accept_case()
    ws = ts.new_workspace(1 << 20)
    res = ts.tree_accept_greedy(torch.from_numpy(case.logits).cuda(), i32_dev(bad), i32_dev(case.parent),
                                i32_dev(case.n_tree), workspace=ws)
    torch.cuda.synchronize()
    assert ts.read_device_error(ws) & ts.TS_DEVERR_BAD_TOKEN
    for b in range(case.num_req):
        r = T.greedy_accept(case.logits[b], bad[b], case.parent[b], 16)
        assert res["accept_len"][b].item() == r.accept_len and res["path"][b, :r.accept_len].tolist() == r.path
        assert res["bonus"][b].item() == r.bonus
        bad_nodes = [i for i in range(1, 16) if not 0 <= bad[b, i] < case.vocab]
        assert not set(bad_nodes) & set(r.path)


def test_stochastic_acceptance_never_accepts_a_token_outside_the_vocab():
    case, bad = _accept_case()
    rng = np.random.default_rng(731)
    tl = torch.from_numpy(case.logits).cuda()
    dl = tl + 0.3 * torch.from_numpy(rng.standard_normal(case.logits.shape).astype(np.float32)).cuda()
    u_acc = torch.zeros((3, 16), device="cuda")   # every test passes unless the token is invalid
    u_bon = torch.full((3, 16), 0.5, device="cuda")
    ws = ts.new_workspace(64 << 20)
    res = ts.tree_accept_sample(tl, dl, i32_dev(bad), i32_dev(case.parent), i32_dev(case.n_tree), u_acc, u_bon,
                                1.0, workspace=ws)
    torch.cuda.synchronize()
    assert ts.read_device_error(ws) & ts.TS_DEVERR_BAD_TOKEN
    for b in range(case.num_req):
        al = res["accept_len"][b].item()
        path = res["path"][b, :al].tolist()
        assert all(0 <= bad[b, i] < case.vocab for i in path[1:])
        # with uniforms of 0 the walk takes the first valid child at every level
        u, expect = 0, [0]
        while True:
            kids = [c for c in range(1, 16) if case.parent[b, c] == u and 0 <= bad[b, c] < case.vocab]
            if not kids:
                break
            u = kids[0]
            expect.append(u)
        assert path == expect


# ------------------------------------------------------------------ compaction
def test_compaction_does_not_move_rows_of_a_bad_block():
    """A bad block on a page holding moved rows: those moves are skipped (the
    destination keeps its row), every other move happens, the new metadata is
    the oracle's, and TS_DEVERR_BAD_BLOCK is set."""
    rng = np.random.default_rng(740)
    n, P = 40, 5 * PAGE + 3
    tokens = rng.integers(0, 1000, size=n).astype(np.int32)
    parent = W.random_parents(rng, n)
    # verified: the tokens of a three-node root path (always the last child),
    # so that path becomes prefix and the last node's subtree moves up
    walk, cur = [], -1
    for _ in range(3):
        kids = [i for i in range(n) if parent[i] == cur]
        if not kids:
            break
        cur = kids[-1]
        walk.append(cur)
    verified = [int(tokens[u]) for u in walk]
    r = T.reroot(parent, tokens, n, P, verified)
    moved = [(P + int(s), P + j) for j, s in enumerate(r.src) if int(s) != j]
    assert moved, "the case must move rows"
    nrows = P + n
    nblk = (nrows + PAGE - 1) // PAGE
    table = rng.permutation(nblk + 2)[:nblk].astype(np.int32)[None, :]
    hkv, dd = 2, 64
    pool = rng.integers(0, 65535, size=(nblk + 2, PAGE, hkv, dd), dtype=np.uint16)
    bad_page = moved[0][1] // PAGE   # the page of the first moved destination
    bad_table = table.copy()
    bad_table[0, bad_page] = nblk + 9
    old = A.logical_rows(pool, 0, nrows, table)
    expect = old.copy()
    for s, dst in moved:
        if s // PAGE != bad_page and dst // PAGE != bad_page:
            expect[dst] = old[s]
    kd = torch.from_numpy(pool.view(np.int16)).cuda()
    vd = torch.from_numpy(pool.copy().view(np.int16)).cuda()
    ws = ts.new_workspace(1 << 16)
    res = ts.tree_cache_compact([kd], [vd], i32_dev([P]), i32_dev([n]), i32_dev(parent[None, :]),
                                i32_dev(tokens[None, :]), i32_dev([verified + [0] * (n + 1 - len(verified))]),
                                i32_dev([len(verified)]), block_table=i32_dev(bad_table), workspace=ws)
    torch.cuda.synchronize()
    assert ts.read_device_error(ws) & ts.TS_DEVERR_BAD_BLOCK
    assert res["new_prefix_len"][0].item() == r.new_prefix_len and res["new_n_tree"][0].item() == r.new_n_tree
    got = A.logical_rows(kd.cpu().numpy().view(np.uint16), 0, nrows, table)
    keep = [x for x in range(nrows) if x // PAGE != bad_page]
    assert np.array_equal(got[keep], expect[keep])
