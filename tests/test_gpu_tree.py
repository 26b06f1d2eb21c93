"""GPU parity: tree metadata, greedy acceptance and re-root/compaction against the oracle (bit-exact)."""
import json
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import tree as T

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import speculative_decoding_tree_forward_gb300 as ts
else:
    ts = None
from gpu_util import i32_dev  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ metadata
@pytest.mark.parametrize("seed", range(4))
def test_tree_masks_match_oracle(seed):
    case = W.random_accept_case(seed, num_req=5, n_tree_max=128 if seed == 0 else 37)
    depth, anc = ts.tree_build_mask(i32_dev(case.parent), i32_dev(case.n_tree))
    depth, anc = depth.cpu().numpy(), anc.cpu().numpy().view(np.uint32)
    for b in range(case.num_req):
        n = int(case.n_tree[b])
        for u in range(n):
            expect = set(T.ancestors_or_self(case.parent[b], u))
            bits = {j for j in range(128) if (int(anc[b, u, j >> 5]) >> (j & 31)) & 1}
            assert bits == expect
            assert depth[b, u] == T.depth(case.parent[b], u)
        assert (depth[b, n:] == -1).all() and (anc[b, n:] == 0).all()


def test_fig3_mask_on_gpu():
    with open(os.path.join(GOLDEN, "fig3_mask.json")) as f:
        g = json.load(f)
    depth, anc = ts.tree_build_mask(i32_dev([g["parent"]]), i32_dev([10]))
    a = int(anc.cpu().numpy().view(np.uint32)[0, g["tokens"].index("t7"), 0])
    assert [g["tokens"][j] for j in range(10) if (a >> j) & 1] == g["visible"]


# ------------------------------------------------------------------ acceptance
def check_accept(case, res):
    got = {k: v.cpu().numpy() for k, v in res.items()}
    for b in range(case.num_req):
        n = int(case.n_tree[b])
        r = T.greedy_accept(case.logits[b][:n], case.tokens[b][:n], case.parent[b][:n], n)
        assert list(got["argmax"][b][:n]) == r.argmax
        assert (got["argmax"][b][n:] == -1).all()
        assert got["accept_len"][b] == r.accept_len and got["bonus"][b] == r.bonus
        assert list(got["path"][b][: r.accept_len]) == r.path and (got["path"][b][r.accept_len:] == -1).all()
        assert got["verified_len"][b] == len(r.verified)
        assert list(got["verified"][b][: len(r.verified)]) == r.verified


def run_accept(case):
    res = ts.tree_accept_greedy(torch.from_numpy(case.logits).cuda(), i32_dev(case.tokens), i32_dev(case.parent),
                                i32_dev(case.n_tree))
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("seed", range(6))
def test_accept_random_trees(seed):
    kw = [dict(vocab=1000), dict(vocab=7, distinct_siblings=False), dict(vocab=50000, n_tree_max=128),
          dict(vocab=8193, chain=True, p_accept=0.9), dict(vocab=4097, p_accept=1.0), dict(vocab=3)][seed]
    case = W.random_accept_case(seed, num_req=6, **kw)
    check_accept(case, run_accept(case))


def test_accept_argmax_ties_take_lowest_index():
    case = W.random_accept_case(1, num_req=2, n_tree_max=8, vocab=20000)
    case.logits[:, :, 17] = 9.0
    case.logits[:, :, 12345] = 9.0
    case.logits[:, :, 19999] = 9.0
    check_accept(case, run_accept(case))


@pytest.mark.parametrize("vocab,B,n,p_acc", [(128256, 8, 16, 0.7), (152064, 4, 32, 0.8)])
def test_accept_plain_normal_logits(vocab, B, n, p_acc):
    """Logits drawn plainly from N(0, 1) at the workloads' vocab sizes, with no
    planted peak: each row's maximum stands only a few tenths above the
    runner-up.  Draft tokens follow the oracle's own argmax at rate p_acc."""
    rng = np.random.default_rng(vocab + n)
    logits = rng.standard_normal((B, n, vocab), dtype=np.float32)
    parent = np.stack([W.random_parents(rng, n) for _ in range(B)]).astype(np.int32)
    am = np.array([T.greedy_accept(logits[b], np.zeros(n, np.int32), parent[b], n).argmax for b in range(B)],
                  np.int32)
    tokens = np.stack([W.draft_tokens(rng, parent[b], am[b], vocab, p_acc) for b in range(B)]).astype(np.int32)
    case = W.AcceptCase(B, n, vocab, np.full(B, n, np.int32), parent, tokens, logits, am)
    check_accept(case, run_accept(case))


def _normal_case(seed, B, n_max, vocab, n_tree=None, p_acc=0.7):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((B, n_max, vocab), dtype=np.float32)
    parent = np.stack([W.random_parents(rng, n_max) for _ in range(B)]).astype(np.int32)
    nt = np.full(B, n_max, np.int32) if n_tree is None else np.asarray(n_tree, np.int32)
    am = np.array([T.greedy_accept(logits[b], np.zeros(n_max, np.int32), parent[b], n_max).argmax for b in range(B)],
                  np.int32)
    tokens = np.stack([W.draft_tokens(rng, parent[b], am[b], vocab, p_acc) for b in range(B)]).astype(np.int32)
    return W.AcceptCase(B, n_max, vocab, nt, parent, tokens, logits, am)


@pytest.mark.parametrize("B,n_max,vocab,n_tree", [
    (5, 48, 32768, [48, 0, 17, 1, 30]),          # ragged and empty trees
    (10, 30, 8192, None),                        # 300 rows, one vocab slice each
    (8, 32, 152064, [0, 0, 0, 1, 0, 0, 0, 0]),   # one valid row among 256
    (3, 40, 65536, [40, 39, 2]),
])
def test_accept_large_ragged_shapes(B, n_max, vocab, n_tree):
    """Tens of MB of N(0, 1) logits with ragged, empty and single-node trees:
    only rows below each request's tree size are read and reduced."""
    case = _normal_case(B * 1000 + vocab, B, n_max, vocab, n_tree)
    check_accept(case, run_accept(case))


def test_accept_ties_across_vocab_slices():
    """Equal maxima planted in each row on both sides of a boundary between
    the vocab slices of a 152-SM launch (rows x slices = eight CTAs per SM,
    slices rounded up to 1024 floats): on even rows the lowest lies in the
    earlier slice, on odd rows at the start of the later one; the lowest index
    wins."""
    B, n_max, vocab = 4, 32, 152064
    case = _normal_case(11, B, n_max, vocab)
    slices = max(1, 152 * 8 // (B * n_max))
    chunk = (vocab + slices - 1) // slices
    chunk = (chunk + 1023) // 1024 * 1024
    for b in range(B):
        for i in range(n_max):
            g = b * n_max + i
            start = chunk * (1 + g % max(1, vocab // chunk - 1))    # a slice boundary inside the row
            spots = [start, vocab - 4, vocab - 1] + ([start - 4] if g % 2 == 0 else [])
            case.logits[b, i, spots] = 7.5
    rng = np.random.default_rng(12)
    am = [T.greedy_accept(case.logits[b], np.zeros(n_max, np.int32), case.parent[b], n_max).argmax for b in range(B)]
    case.tokens = np.stack([W.draft_tokens(rng, case.parent[b], np.asarray(am[b], np.int32), vocab, 0.7)
                            for b in range(B)]).astype(np.int32)
    check_accept(case, run_accept(case))


def test_accept_fig2_target_verify():
    with open(os.path.join(GOLDEN, "fig2_walkthrough.json")) as f:
        g = json.load(f)["target_verify"]
    lg = np.zeros((1, 4, g["vocab"]), np.float32)
    for i, a in enumerate(g["argmax"]):
        lg[0, i, a] = 1.0
    res = ts.tree_accept_greedy(torch.from_numpy(lg).cuda(), i32_dev([g["tokens"]]), i32_dev([g["parent"]]),
                                i32_dev([4]))
    e = g["expect"]
    assert res["accept_len"].item() == e["accept_len"] and res["bonus"].item() == e["bonus"]
    assert res["path"][0, :2].tolist() == e["path"] and res["verified"][0, :3].tolist() == e["verified"]


def test_accept_empty_tree():
    case = W.random_accept_case(2, num_req=2, n_tree_max=4, vocab=64)
    case.n_tree[1] = 0
    check_accept(case, run_accept(case))


@pytest.mark.slow
@pytest.mark.parametrize("wl", ["verify_b8_tree16", "longctx_verify_b4_p32k", "tree16_prefix128"])
def test_accept_named_workloads(wl):
    w = getattr(W, wl)(**({"with_kv": False} if wl.startswith("longctx") else {}))
    check_accept(w.accept, run_accept(w.accept))


# ------------------------------------------------------------------ compaction
def _logical(cache, b, nrows, table):
    return A.logical_rows(cache, b, nrows, table)


def run_compact_case(case, layers=3, hkv=2, d=64, paged=False, seed=0, max_rows=None, workspace=None):
    """Random KV for `layers` layers; compaction on GPU vs oracle (metadata + bytes)."""
    rng = np.random.default_rng(seed)
    B = case.num_req
    rows = case.prefix_len + case.n_tree
    if paged:
        nblk = [(int(r) + 15) // 16 for r in rows]
        perm = rng.permutation(sum(nblk) + 2)
        table = np.full((B, max(max(nblk), 1)), -1, np.int32)
        off = 0
        for b in range(B):
            table[b, :nblk[b]] = perm[off:off + nblk[b]]
            off += nblk[b]
        shape = (len(perm), 16, hkv, d)
    else:
        table = None
        shape = (B, int(rows.max()) + 3, hkv, d)
    ks = [rng.integers(0, 65535, size=shape, dtype=np.uint16) for _ in range(layers)]
    vs = [rng.integers(0, 65535, size=shape, dtype=np.uint16) for _ in range(layers)]
    kd = [torch.from_numpy(x.view(np.int16)).cuda() for x in ks]
    vd = [torch.from_numpy(x.view(np.int16)).cuda() for x in vs]
    res = ts.tree_cache_compact(kd, vd, i32_dev(case.prefix_len), i32_dev(case.n_tree), i32_dev(case.parent),
                                i32_dev(case.tokens), i32_dev(case.verified), i32_dev(case.m),
                                block_table=None if table is None else i32_dev(table), workspace=workspace)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in res.items() if not k.startswith("_")}
    for b in range(B):
        n, P = int(case.n_tree[b]), int(case.prefix_len[b])
        r = T.reroot(case.parent[b][:n], case.tokens[b][:n], n, P, case.verified[b][: int(case.m[b])])
        assert got["new_prefix_len"][b] == r.new_prefix_len and got["new_n_tree"][b] == r.new_n_tree
        assert list(got["new_parent"][b][: r.new_n_tree]) == r.new_parent
        assert list(got["new_tokens"][b][: r.new_n_tree]) == r.new_tokens
        assert list(got["src_rows"][b][: len(r.src)]) == r.src
        keep = P + len(r.src)
        for li in range(layers):
            for host, dev in ((ks[li], kd[li]), (vs[li], vd[li])):
                before = _logical(host, b, P + n, table)
                expect = T.compact_rows(before, P, r.src)[:keep]
                after = _logical(dev.cpu().numpy().view(np.uint16), b, keep, table)
                assert np.array_equal(after, expect), f"request {b} layer {li}"


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("paged", [False, True])
def test_compact_random(seed, paged):
    case = W.random_compact_case(seed, num_req=5, n_tree_max=24 if seed else 128, forest=bool(seed % 2))
    run_compact_case(case, layers=2 + seed % 3, hkv=2 if seed % 2 else 8, d=64 if seed < 3 else 128,
                     paged=paged, seed=seed)


@pytest.mark.parametrize("paged", [False, True])
def test_compact_many_layers_and_requests(paged):
    """Sixteen requests x 24 layers of 1 KB rows on 128-node trees: several
    (layer, K|V) items per CTA and row moves staged in several batches."""
    case = W.random_compact_case(40, num_req=16, n_tree_max=128, max_verified=129)
    run_compact_case(case, layers=24, hkv=8, d=64, paged=paged, seed=40)


def test_compact_one_workspace_serves_repeated_calls():
    """The per-request tickets are left at zero: one workspace serves
    successive calls of different shapes."""
    ws = ts.new_workspace(1 << 16)
    for seed, nreq, nmax in ((50, 6, 24), (51, 3, 128), (52, 9, 40), (53, 6, 24)):
        case = W.random_compact_case(seed, num_req=nreq, n_tree_max=nmax)
        run_compact_case(case, layers=3, hkv=4, d=64, paged=bool(seed % 2), seed=seed, workspace=ws)
        assert int(ws[256:256 + 4 * nreq].view(torch.int32).abs().sum()) == 0
        assert int(ws[:4].view(torch.int32)[0]) == 0


def _compact_inputs(case, layers, hkv, d, paged, seed):
    """Random KV of `layers` layers for a compaction case, the C arguments of
    its call and their device buffers (kept alive by the returned dict)."""
    rng = np.random.default_rng(seed)
    B = case.num_req
    rows = case.prefix_len + case.n_tree
    if paged:
        nblk = [(int(r) + 15) // 16 for r in rows]
        perm = rng.permutation(sum(nblk) + 2)
        table = np.full((B, max(max(nblk), 1)), -1, np.int32)
        off = 0
        for b in range(B):
            table[b, :nblk[b]] = perm[off:off + nblk[b]]
            off += nblk[b]
        shape = (len(perm), 16, hkv, d)
    else:
        table = None
        shape = (B, int(rows.max()) + 3, hkv, d)
    ks = [rng.integers(0, 65535, size=shape, dtype=np.uint16) for _ in range(layers)]
    vs = [rng.integers(0, 65535, size=shape, dtype=np.uint16) for _ in range(layers)]
    dev = {"kd": [torch.from_numpy(x.view(np.int16)).cuda() for x in ks],
           "vd": [torch.from_numpy(x.view(np.int16)).cuda() for x in vs]}
    dev["kp"], dev["vp"] = ts.layer_pointer_table(dev["kd"]), ts.layer_pointer_table(dev["vd"])
    meta = {k: i32_dev(getattr(case, k)) for k in ("prefix_len", "n_tree", "parent", "tokens", "verified", "m")}
    out = {"new_prefix_len": torch.empty(B, dtype=torch.int32, device="cuda"),
           "new_n_tree": torch.empty(B, dtype=torch.int32, device="cuda"),
           "new_parent": torch.empty_like(meta["parent"]), "new_tokens": torch.empty_like(meta["tokens"]),
           "src_rows": torch.empty_like(meta["parent"])}
    bt = None if table is None else i32_dev(table)
    args = ts.compact_args(dev["kp"], dev["vp"], layers, hkv, d, meta["prefix_len"], meta["n_tree"], meta["parent"],
                           meta["tokens"], meta["verified"], meta["m"], out["new_prefix_len"], out["new_n_tree"],
                           out["new_parent"], out["new_tokens"], out["src_rows"],
                           shape[1] if table is None else 0, bt, 16 if paged else 0, shape[0] if paged else 0)
    return {"args": args, "ks": ks, "vs": vs, "table": table, "dev": dev, "meta": meta, "out": out, "bt": bt,
            "layers": layers}


def _check_compact(case, x):
    got = {k: v.cpu().numpy() for k, v in x["out"].items()}
    table = x["table"]
    for b in range(case.num_req):
        n, P = int(case.n_tree[b]), int(case.prefix_len[b])
        r = T.reroot(case.parent[b][:n], case.tokens[b][:n], n, P, case.verified[b][: int(case.m[b])])
        assert got["new_prefix_len"][b] == r.new_prefix_len and got["new_n_tree"][b] == r.new_n_tree
        assert list(got["new_parent"][b][: r.new_n_tree]) == r.new_parent
        assert list(got["new_tokens"][b][: r.new_n_tree]) == r.new_tokens
        assert list(got["src_rows"][b][: len(r.src)]) == r.src
        keep = P + len(r.src)
        for li in range(x["layers"]):
            for host, dv in ((x["ks"][li], x["dev"]["kd"][li]), (x["vs"][li], x["dev"]["vd"][li])):
                expect = T.compact_rows(_logical(host, b, P + n, table), P, r.src)[:keep]
                after = _logical(dv.cpu().numpy().view(np.uint16), b, keep, table)
                assert np.array_equal(after, expect), f"request {b} layer {li}"


@pytest.mark.parametrize("count", [1, 2, 4])
def test_compact_batch_matches_oracle(count):
    """tree_cache_compact_batch: up to four independent caches of different
    shapes and layouts (a target-side and a draft-side cache, say) in one
    launch, each compared with the oracle as if compacted alone."""
    shapes = [(61, 4, 32, 3, 8, 128, False), (62, 6, 64, 2, 2, 64, True), (63, 3, 128, 5, 4, 64, False),
              (64, 7, 24, 1, 8, 128, True)]
    cases, xs = [], []
    for seed, nreq, nmax, layers, hkv, d, paged in shapes[:count]:
        case = W.random_compact_case(seed, num_req=nreq, n_tree_max=nmax, forest=bool(seed % 2))
        cases.append(case)
        xs.append(_compact_inputs(case, layers, hkv, d, paged, seed))
    wss = [ts.new_workspace(ts.tree_compact_workspace_size(x["args"])) for x in xs]
    ts.tree_cache_compact_batch_args([x["args"] for x in xs], wss)
    torch.cuda.synchronize()
    for case, x, ws in zip(cases, xs, wss):
        _check_compact(case, x)
        assert ts.read_device_error(ws) == 0
        assert int(ws[256:256 + 4 * case.num_req].view(torch.int32).abs().sum()) == 0   # tickets left at zero


def test_compact_batch_rejects_bad_calls():
    case = W.random_compact_case(65, num_req=2, n_tree_max=16)
    x = _compact_inputs(case, 1, 2, 64, False, 65)
    ws = ts.new_workspace(ts.tree_compact_workspace_size(x["args"]))
    for bad in ([], [x["args"]] * 5):
        with pytest.raises(ts.TreeSpecError):
            ts.tree_cache_compact_batch_args(bad, [ws] * len(bad))
    small = ts.new_workspace(256)
    with pytest.raises(ts.TreeSpecError):   # the second call's workspace is too small: nothing runs
        ts.tree_cache_compact_batch_args([x["args"], x["args"]], [ws, small])


def test_compact_fig4_on_gpu():
    with open(os.path.join(GOLDEN, "fig4_compaction.json")) as f:
        g = json.load(f)
    case = W.CompactCase(1, 8, np.array([4], np.int32), np.array([8], np.int32), np.array([g["parent"]], np.int32),
                         np.array([g["tokens"]], np.int32), np.array([g["verified"]], np.int32),
                         np.array([2], np.int32))
    run_compact_case(case, layers=2)


def test_compact_target_side_after_accept():
    """accept -> compact chained on the device: the accepted path becomes prefix, nothing survives."""
    acc = W.random_accept_case(9, num_req=4, n_tree_max=16, vocab=300, p_accept=0.8)
    res = run_accept(acc)
    case = W.CompactCase(4, 16, np.full(4, 50, np.int32), acc.n_tree, acc.parent, acc.tokens,
                         res["verified"].cpu().numpy(), res["verified_len"].cpu().numpy())
    run_compact_case(case, layers=2)


def test_compact_in_place_metadata():
    case = W.random_compact_case(3, num_req=4, n_tree_max=20)
    par, tok = i32_dev(case.parent), i32_dev(case.tokens)
    k = [torch.zeros((4, 80, 2, 64), dtype=torch.int16, device="cuda")]
    res = ts.tree_cache_compact(k, [torch.zeros_like(k[0])], i32_dev(case.prefix_len), i32_dev(case.n_tree), par,
                                tok, i32_dev(case.verified), i32_dev(case.m), in_place_metadata=True)
    torch.cuda.synchronize()
    for b in range(4):
        n = int(case.n_tree[b])
        r = T.reroot(case.parent[b][:n], case.tokens[b][:n], n, int(case.prefix_len[b]),
                     case.verified[b][: int(case.m[b])])
        assert par[b, : r.new_n_tree].tolist() == r.new_parent and tok[b, : r.new_n_tree].tolist() == r.new_tokens
    assert res["new_parent"].data_ptr() == par.data_ptr()
