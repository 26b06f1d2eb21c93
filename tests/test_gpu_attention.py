"""GPU parity: tree_attn_forward (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():   # on a GPU machine a missing library is an error, not a skip
    import speculative_decoding_tree_forward_gb300 as ts
else:
    ts = None
from gpu_util import ATOL, RTOL, attn_inputs, bf16_dev, bf16_host_f64, check_attention  # noqa: E402


def run(case, **kw):
    d = attn_inputs(case)
    out, lse = ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"],
                                    block_table=d.get("block_table"), softmax_scale=case.softmax_scale, **kw)
    torch.cuda.synchronize()
    return out, lse


SMALL = [
    dict(num_req=2, hq=8, hkv=2, d=64, n_tree_max=16, prefix_range=(0, 200)),
    dict(num_req=3, hq=8, hkv=2, d=128, n_tree_max=16, prefix_range=(50, 300)),
    dict(num_req=2, hq=32, hkv=8, d=128, n_tree_max=40, n_query=8, prefix_range=(100, 400)),   # expansion
    dict(num_req=4, hq=64, hkv=8, d=128, n_tree_max=5, prefix_range=(60, 300), chain=True),   # R = 40
    dict(num_req=2, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(0, 500)),              # R = 128
    dict(num_req=2, hq=32, hkv=8, d=128, n_tree_max=32, prefix_range=(0, 300)),              # R = 128
    dict(num_req=2, hq=16, hkv=2, d=64, n_tree_max=40, n_query=32, prefix_range=(0, 100)),    # R = 256, 2 row groups
    dict(num_req=3, hq=12, hkv=4, d=64, n_tree_max=20, n_query=7, ragged_tree=True, prefix_range=(0, 150)),  # G=3
    dict(num_req=2, hq=4, hkv=4, d=128, n_tree_max=128, prefix_range=(0, 70)),                # max tree, G=1
    dict(num_req=2, hq=8, hkv=1, d=64, n_tree_max=24, prefix_range=(0, 0)),                   # no prefix
]


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("cfg", range(len(SMALL)))
def test_small_cases_match_oracle(cfg, paged):
    case = W.random_attn_case(100 + cfg, paged=paged, **SMALL[cfg])
    out, lse = run(case, force_path=1)
    check_attention(case, out, lse, A.attention_case(case))


# packed rows R = G * n_query = 128 with head_dim 128: the tcgen05 / TMEM kernel
TC = [
    dict(num_req=2, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(0, 500)),
    dict(num_req=2, hq=32, hkv=8, d=128, n_tree_max=32, prefix_range=(0, 300)),
    dict(num_req=3, hq=16, hkv=1, d=128, n_tree_max=24, n_query=8, ragged_tree=True, prefix_range=(10, 400)),
    dict(num_req=2, hq=128, hkv=1, d=128, n_tree_max=3, n_query=1, prefix_range=(0, 200)),
    dict(num_req=1, hq=2, hkv=2, d=128, n_tree_max=128, prefix_range=(0, 150)),
    dict(num_req=2, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(0, 0)),
]


# R < 128: the tcgen05 kernel pads the packed rows to one 128-row tile; with
# R <= 64 and an even KV-head count two adjacent heads share the tile
TC_SMALL_R = [
    dict(num_req=4, hq=64, hkv=8, d=128, n_tree_max=5, prefix_range=(60, 700), chain=True),          # R = 40
    dict(num_req=2, hq=32, hkv=8, d=128, n_tree_max=40, n_query=8, prefix_range=(100, 400)),         # R = 32
    dict(num_req=3, hq=4, hkv=4, d=128, n_tree_max=20, n_query=8, ragged_tree=True, prefix_range=(0, 300)),  # R = 8
    dict(num_req=2, hq=2, hkv=2, d=128, n_tree_max=6, n_query=1, prefix_range=(0, 260)),             # R = 1
    dict(num_req=2, hq=16, hkv=4, d=128, n_tree_max=30, n_query=25, prefix_range=(0, 200)),          # R = 100
    dict(num_req=1, hq=127, hkv=1, d=128, n_tree_max=9, n_query=1, prefix_range=(30, 90)),           # R = 127
    dict(num_req=2, hq=3, hkv=3, d=128, n_tree_max=12, n_query=8, prefix_range=(0, 300)),            # R = 8, odd Hkv
    dict(num_req=2, hq=32, hkv=16, d=128, n_tree_max=40, n_query=32, ragged_tree=True,
         prefix_range=(0, 400)),                                                                   # R = 64
]


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("cfg", range(len(TC_SMALL_R)))
def test_tcgen05_fewer_rows_match_oracle(cfg, paged):
    case = W.random_attn_case(250 + cfg, paged=paged, **TC_SMALL_R[cfg])
    out, lse = run(case, force_path=2)
    check_attention(case, out, lse, A.attention_case(case))


@pytest.mark.parametrize("num_ctas", [1, 5, 64, 700])
def test_tcgen05_fewer_rows_split_counts(num_ctas):
    case = W.random_attn_case(260, num_req=3, hq=64, hkv=8, d=128, n_tree_max=5, prefix_range=(10, 900), chain=True)
    out, lse = run(case, force_path=2, num_ctas=num_ctas)
    check_attention(case, out, lse, A.attention_case(case))


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("cfg", range(len(TC)))
def test_tcgen05_cases_match_oracle(cfg, paged):
    case = W.random_attn_case(200 + cfg, paged=paged, **TC[cfg])
    out, lse = run(case, force_path=2)
    check_attention(case, out, lse, A.attention_case(case))


@pytest.mark.parametrize("num_ctas", [1, 3, 64, 130, 1000])   # 12 units: merge share groups 1, 1, 2, 4, 8
def test_tcgen05_split_counts_match_oracle(num_ctas):
    case = W.random_attn_case(8, num_req=3, hq=16, hkv=4, d=128, n_tree_max=40, n_query=32, prefix_range=(10, 700),
                              ragged_tree=True)
    out, lse = run(case, force_path=2, num_ctas=num_ctas)
    check_attention(case, out, lse, A.attention_case(case))


def _scaled_bf16(bits, exp2):
    """bf16 bit patterns times 2^exp2 (exact: only the exponent changes)."""
    f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** exp2)
    return W.f32_to_bf16_bits(f)


@pytest.mark.parametrize("path,num_ctas,shape", [
    (2, 64, "r128"), (2, 0, "r128"), (2, 64, "two_heads"), (1, 64, "r128"), (1, 7, "d64")])
def test_large_magnitude_values_scale_exactly(path, num_ctas, shape):
    """V scaled by 2^17 (entries up to about 2^19, split-KV partials and
    outputs far beyond fp16's range): every fp32 step scales exactly, so the
    output must be 2^17 times the unscaled one bit for bit, with the same
    lse; the unscaled output is checked against the oracle.  Both kernels,
    split and unsplit."""
    import dataclasses
    kw = {"r128": dict(num_req=3, hq=64, hkv=8, d=128, n_tree_max=16),
          "two_heads": dict(num_req=3, hq=64, hkv=8, d=128, n_tree_max=5, chain=True),
          "d64": dict(num_req=2, hq=8, hkv=2, d=64, n_tree_max=16)}[shape]
    case = W.random_attn_case(860, prefix_range=(300, 900), **kw)
    big = dataclasses.replace(case, v=_scaled_bf16(case.v, 17))
    out, lse = run(case, force_path=path, num_ctas=num_ctas)
    out_big, lse_big = run(big, force_path=path, num_ctas=num_ctas)
    assert torch.isfinite(out_big.float()).all()
    assert torch.equal(out_big.float(), out.float() * 2.0 ** 17)
    assert torch.equal(lse_big, lse)
    check_attention(case, out, lse, A.attention_case(case))


@pytest.mark.parametrize("num_ctas", [190, 300, 400])
def test_tcgen05_first_call_many_short_splits(num_ctas):
    """A fresh workspace and two to four tiles per CTA: every unit is combined from many partials."""
    case = W.random_attn_case(21, num_req=8, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(300, 1200))
    out, lse = run(case, force_path=2, num_ctas=num_ctas)
    check_attention(case, out, lse, A.attention_case(case))


@pytest.mark.parametrize("which", ["tc_r128", "tc_two_heads", "mma_r16"])
def test_merge_of_many_split_units(which):
    """More split rows than one resident wave of warp-per-row merge CTAs
    holds, so the merge takes one row per half-warp: 80 units of 128 rows,
    160 two-head units, and 624 units of 16 rows at head_dim 64 (one float4
    per lane)."""
    if which == "tc_r128":
        case = W.random_attn_case(32, num_req=10, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(100, 700))
        path = 2
    elif which == "tc_two_heads":
        case = W.random_attn_case(33, num_req=40, hq=32, hkv=8, d=128, n_tree_max=16, n_query=8,
                                  prefix_range=(100, 500), ragged_tree=True)
        path = 2
    else:
        case = W.random_attn_case(31, num_req=78, hq=16, hkv=8, d=64, n_tree_max=8, prefix_range=(10, 150))
        path = 1
    out, lse = run(case, force_path=path)
    check_attention(case, out, lse, A.attention_case(case))


@pytest.mark.parametrize("path", [1, 2])
def test_large_scores_rescale_running_max(path):
    """Scale 2.0 makes scores grow by far more than 2^8 across tiles: the running max is raised many times."""
    case = W.random_attn_case(9, num_req=2, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(300, 900),
                              scale=2.0)
    out, lse = run(case, force_path=path)
    check_attention(case, out, lse, A.attention_case(case))


def test_tcgen05_rows_past_the_last_key_may_hold_nan():
    case = W.random_attn_case(15, num_req=2, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(20, 100))
    d = attn_inputs(case)
    ref = A.attention_case(case)
    for b in range(case.num_req):
        end = int(case.prefix_len[b] + case.n_tree[b])
        d["k_cache"][b, end:] = float("nan")
        d["v_cache"][b, end:] = float("inf")
    out, lse = ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"],
                                    force_path=2)
    torch.cuda.synchronize()
    check_attention(case, out, lse, ref)


def test_automatic_path_choice():
    case = W.random_attn_case(16, num_req=1, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(5, 5))
    d = attn_inputs(case)
    a = ts.attn_args(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"],
                     torch.empty_like(d["q"]))
    assert ts.tree_attn_selected_path(a) == "tcgen05"
    # R = 40 (chain verify, G = 8): one padded 128-row tile on the tcgen05 path
    case2 = W.random_attn_case(16, num_req=1, hq=64, hkv=8, d=128, n_tree_max=5, prefix_range=(5, 5))
    d2 = attn_inputs(case2)
    a2 = ts.attn_args(d2["q"], d2["k_cache"], d2["v_cache"], d2["prefix_len"], d2["n_tree"], d2["parent"],
                      torch.empty_like(d2["q"]))
    assert ts.tree_attn_selected_path(a2) == "tcgen05"
    # head_dim 64 and R > 128 stay on the warp-MMA kernel
    case3 = W.random_attn_case(16, num_req=1, hq=8, hkv=2, d=64, n_tree_max=16, prefix_range=(5, 5))
    d3 = attn_inputs(case3)
    a3 = ts.attn_args(d3["q"], d3["k_cache"], d3["v_cache"], d3["prefix_len"], d3["n_tree"], d3["parent"],
                      torch.empty_like(d3["q"]))
    assert ts.tree_attn_selected_path(a3) == "mma"
    case4 = W.random_attn_case(16, num_req=1, hq=16, hkv=1, d=128, n_tree_max=16, prefix_range=(5, 5))
    d4 = attn_inputs(case4)
    a4 = ts.attn_args(d4["q"], d4["k_cache"], d4["v_cache"], d4["prefix_len"], d4["n_tree"], d4["parent"],
                      torch.empty_like(d4["q"]))
    assert ts.tree_attn_selected_path(a4) == "mma"   # R = 256


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 1000])
def test_split_counts_match_oracle(num_ctas):
    """Every split of the key range (one CTA for everything up to one tile per CTA) merges to the same result."""
    case = W.random_attn_case(7, num_req=3, hq=16, hkv=4, d=128, n_tree_max=12, prefix_range=(10, 400),
                              ragged_tree=True, n_query=6)
    out, lse = run(case, force_path=1, num_ctas=num_ctas)
    check_attention(case, out, lse, A.attention_case(case))


def test_single_node_single_key():
    case = W.random_attn_case(3, num_req=1, hq=2, hkv=2, d=64, n_tree_max=1, prefix_range=(0, 0))
    out, lse = run(case)
    np.testing.assert_array_equal(bf16_host_f64(out)[0, 0], A.bf16_bits_to_f64(case.v[0, 0]))


def test_masked_tree_rows_do_not_leak():
    """Non-ancestor tree K/V replaced by large finite garbage: outputs stay bit-identical."""
    case = W.random_attn_case(11, num_req=2, hq=8, hkv=2, d=128, n_tree_max=16, prefix_range=(30, 90))
    out1, lse1 = run(case)
    u = 15
    for b in range(case.num_req):
        P = int(case.prefix_len[b])
        anc = set()
        x = u
        while x != -1:
            anc.add(x)
            x = int(case.parent[b][x])
        for j in range(16):
            if j not in anc:
                case.k[b, P + j] = W.f32_to_bf16_bits(np.full(case.k.shape[2:], 300.0, np.float32))
                case.v[b, P + j] = W.f32_to_bf16_bits(np.full(case.v.shape[2:], -3e4, np.float32))
    out2, lse2 = run(case)
    assert torch.equal(out1[:, u], out2[:, u]) and torch.equal(lse1[:, :, u], lse2[:, :, u])


def test_rows_past_the_last_key_may_hold_nan():
    """Memory after P + n (next request, unwritten rows) never reaches the output, even as NaN/Inf."""
    case = W.random_attn_case(12, num_req=2, hq=8, hkv=2, d=64, n_tree_max=10, prefix_range=(20, 40))
    d = attn_inputs(case)
    ref = A.attention_case(case)
    for b in range(case.num_req):
        end = int(case.prefix_len[b] + case.n_tree[b])
        d["k_cache"][b, end:] = float("nan")
        d["v_cache"][b, end:] = float("inf")
    out, lse = ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"])
    torch.cuda.synchronize()
    check_attention(case, out, lse, ref)


def test_bad_parent_is_reported_not_trapped():
    case = W.random_attn_case(13, num_req=1, hq=4, hkv=1, d=64, n_tree_max=6, prefix_range=(5, 5))
    case.parent[0, 3] = 5   # not an earlier node
    d = attn_inputs(case)
    ws = ts.new_workspace(ts.tree_attn_workspace_size(ts.attn_args(
        d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"], torch.empty_like(d["q"]))))
    ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"], workspace=ws)
    code = ts.read_device_error(ws)
    assert code & ts.TS_DEVERR_BAD_PARENT
    assert ts.read_device_error(ws) == 0


def test_invalid_arguments_are_rejected():
    case = W.random_attn_case(14, num_req=1, hq=6, hkv=4, d=64, n_tree_max=4, prefix_range=(3, 3))
    d = attn_inputs(case)
    with pytest.raises(ts.TreeSpecError):   # Hq % Hkv != 0
        ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"])


# ------------------------------------------------------------------ named workloads
def _sampled(case, requests, heads, **kw):
    out, lse = run(case, **kw)
    ref = A.attention_case(case, requests=requests, heads=heads)
    check_attention(case, out, lse, ref, heads=heads)


def test_tcgen05_one_workspace_serves_repeated_calls():
    """One workspace serves repeated calls, also of other shapes and CTA
    counts, with identical results and a clean error word."""
    cases = [
        (W.random_attn_case(31, num_req=3, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(200, 1500))),  # R = 128
        (W.random_attn_case(32, num_req=5, hq=64, hkv=8, d=128, n_tree_max=5, prefix_range=(100, 2000),
                            chain=True, paged=True)),                                                      # R = 40
    ]
    ws = ts.new_workspace(1 << 24)
    for num_ctas in (40, 0, 96):
        for case in cases:
            d = attn_inputs(case)
            outs = []
            for _ in range(2):
                out = torch.empty_like(d["q"])
                lse = torch.empty((case.num_req, case.num_q_heads, case.n_query), dtype=torch.float32, device="cuda")
                a = ts.attn_args(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"], out,
                                 lse, d.get("block_table"), case.softmax_scale, 2, num_ctas)
                assert ts.tree_attn_workspace_size(a) <= ws.numel()
                ts.tree_attn_forward_args(a, ws)
                torch.cuda.synchronize()
                assert int(ws[:4].view(torch.int32)[0]) == 0
                outs.append((out.clone(), lse.clone()))
            assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
            check_attention(case, outs[0][0], outs[0][1], A.attention_case(case))


ROPE = [  # (case, forced path)
    (dict(num_req=2, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(0, 3000)), 2),                  # R = 128
    (dict(num_req=3, hq=64, hkv=8, d=128, n_tree_max=5, prefix_range=(60, 900), chain=True, paged=True), 2),  # R = 40
    (dict(num_req=2, hq=32, hkv=8, d=128, n_tree_max=40, n_query=8, prefix_range=(100, 400)), 2),      # expansion
    (dict(num_req=2, hq=8, hkv=2, d=64, n_tree_max=24, prefix_range=(0, 300), ragged_tree=True), 1),   # warp MMA
    (dict(num_req=1, hq=32, hkv=8, d=128, n_tree_max=32, prefix_range=(32000, 32768)), 2),             # far positions
    (dict(num_req=2, hq=32, hkv=2, d=128, n_tree_max=8, prefix_range=(100, 900)), 2),                  # G = 16
    (dict(num_req=2, hq=32, hkv=1, d=128, n_tree_max=4, prefix_range=(10, 700)), 2),                   # G = 32
    (dict(num_req=2, hq=16, hkv=8, d=128, n_tree_max=20, prefix_range=(50, 500), ragged_tree=True), 2),  # G = 2
]


@pytest.mark.parametrize("theta", [10000.0, 500000.0])
@pytest.mark.parametrize("cfg", range(len(ROPE)))
def test_rope_at_tree_positions_matches_oracle(cfg, theta):
    """Queries rotated at position prefix_len + depth inside the attention call."""
    import dataclasses
    kw, path = ROPE[cfg]
    case = dataclasses.replace(W.random_attn_case(300 + cfg, **kw), rope_theta=theta)
    d = attn_inputs(case)
    q_before = d["q"].clone()
    out, lse = ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"],
                                    block_table=d.get("block_table"), force_path=path, rope_theta=theta)
    torch.cuda.synchronize()
    assert torch.equal(d["q"], q_before)   # the rotation goes to workspace scratch
    heads = list(range(0, case.num_q_heads, max(1, case.num_q_heads // 6)))
    check_attention(case, out, lse, A.attention_case(case, heads=heads), heads=heads)


@pytest.mark.parametrize("cfg", [0, 4])
def test_rope_error_against_the_unrounded_rotation(cfg, record_property):
    """The effect of reading the rotated queries as bf16 operands: the GPU
    output against the oracle with bf16-rounded rotated queries (the stated
    reading) and against the oracle that keeps the fp64 rotation.  Both errors
    are reported (as multiples of the tolerance) and both stay within it."""
    import dataclasses
    kw, path = ROPE[cfg]
    case = dataclasses.replace(W.random_attn_case(300 + cfg, **kw), rope_theta=500000.0)
    d = attn_inputs(case)
    out, _ = ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"],
                                  block_table=d.get("block_table"), force_path=path, rope_theta=500000.0)
    torch.cuda.synchronize()
    got = bf16_host_f64(out)
    heads = list(range(0, case.num_q_heads, max(1, case.num_q_heads // 6)))
    worst = {}
    for name, rnd in (("rounded", True), ("unrounded", False)):
        ref = A.attention_case(case, heads=heads, round_rotated_q=rnd)
        w = 0.0
        for b, (ro, _) in ref.items():
            for h in heads:
                e = np.abs(got[b][:, h, :] - ro[:, h, :]) / (ATOL + RTOL * np.abs(ro[:, h, :]))
                w = max(w, float(e.max()))
        worst[name] = w
    record_property("tolerance_used_rounded", worst["rounded"])
    record_property("tolerance_used_unrounded", worst["unrounded"])
    print(f"rope cfg {cfg}: max error / tolerance = {worst['rounded']:.3f} (bf16-rounded rotated queries), "
          f"{worst['unrounded']:.3f} (fp64 rotation)")
    assert worst["rounded"] <= 1.0 and worst["unrounded"] <= 1.0


def test_rope_changes_the_result_and_rejects_bad_bases():
    import dataclasses
    case = W.random_attn_case(320, num_req=1, hq=32, hkv=8, d=128, n_tree_max=32, prefix_range=(500, 600))
    plain, _ = run(case, force_path=2)
    rotated, _ = run(case, force_path=2, rope_theta=10000.0)
    assert not torch.equal(plain, rotated)
    d = attn_inputs(case)
    for bad in (float("nan"), 0.5, float("inf"), -1.0):
        with pytest.raises(ts.TreeSpecError):
            ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"],
                                 rope_theta=bad)


def test_workload_tree16_prefix128():
    w = W.tree16_prefix128()
    _sampled(w.attn[0], None, None)


def test_workload_expand_w8_prefix2048():
    w = W.expand_w8_prefix2048()
    for case in w.attn:
        _sampled(case, None, None)


@pytest.mark.slow
def test_workload_verify_b8_tree16():
    w = W.verify_b8_tree16()
    _sampled(w.attn[0], [0, 3, 7], [0, 9, 63])


@pytest.mark.slow
def test_workload_verify_b8_tree16_mma_path():
    w = W.verify_b8_tree16()
    _sampled(w.attn[0], [1, 6], [5, 40], force_path=1)


@pytest.mark.slow
def test_workload_chain_verify_b16_paged():
    w = W.chain_verify_b16_paged()
    _sampled(w.attn[0], [0, 5, 15], [0, 17, 63])


@pytest.mark.slow
def test_workload_longctx_verify_b4_p32k():
    w = W.longctx_verify_b4_p32k(num_layers=1)
    _sampled(w.attn[0], [0, 3], [0, 31])
