"""The allocation-free attention entry point agrees with the workspace entry point.

tree_attn_forward_noalloc serves callers that cannot allocate device memory
(a host framework that owns all device memory through its own pool, or a
latency-critical loop where cudaMalloc would synchronize the device): the
library keeps the split-KV scratch in its own device array.  This file is
collected last, and its test passes alone in a fresh process as well as after
the rest of the suite.
"""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import speculative_decoding_tree_forward_gb300 as ts
else:
    ts = None
from gpu_util import ATOL, LSE_ATOL, LSE_RTOL, RTOL, attn_inputs, check_attention  # noqa: E402
from oracle import attention as A  # noqa: E402


def _close(a, b, atol, rtol):
    a, b = a.double(), b.double()
    return bool(((a - b).abs() <= atol + rtol * b.abs()).all())


CASES = {  # (case arguments, forced path, RoPE base)
    "tcgen05": (dict(num_req=8, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(300, 1200)), 0, 0.0),
    "paged": (dict(num_req=5, hq=64, hkv=8, d=128, n_tree_max=5, chain=True, paged=True, prefix_range=(60, 900)), 0,
              0.0),
    "warp_mma_d64": (dict(num_req=3, hq=8, hkv=2, d=64, n_tree_max=16, prefix_range=(100, 600)), 0, 0.0),
    "forced_warp_mma": (dict(num_req=4, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(200, 700)), 1, 0.0),
    "rope": (dict(num_req=2, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(500, 3000)), 0, 500000.0),
}


@pytest.mark.parametrize("num_ctas", [0, 1000])
@pytest.mark.parametrize("name", list(CASES))
def test_no_alloc_matches_workspace_entry_point_twice(name, num_ctas):
    """Two calls in a row through the C ABI; the second sees the first call's leftovers in the scratch.

    The shapes cover both kernels (tcgen05, warp MMA), paged K/V and queries
    rotated at their tree positions.  num_ctas=1000 asks for more split-KV CTAs
    than the scratch can hold partials for, so the entry point has to shrink
    the split to fit.  The first call is also checked against the oracle.
    """
    kw, path, theta = CASES[name]
    case = W.random_attn_case(21, **kw)
    if theta > 0:
        import dataclasses
        case = dataclasses.replace(case, rope_theta=theta)
    d = attn_inputs(case)
    bt = d.get("block_table")
    ref_out, ref_lse = ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"],
                                            d["parent"], block_table=bt, force_path=path, rope_theta=theta)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        ts.tree_attn_forward_noalloc(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"],
                                     out, lse, block_table=bt, force_path=path, num_ctas=num_ctas, rope_theta=theta)
        torch.cuda.synchronize()
        assert _close(out, ref_out, ATOL, RTOL)
        assert _close(lse, ref_lse, LSE_ATOL, LSE_RTOL)
        if call == 0 and num_ctas == 0:
            heads = [0, case.num_q_heads - 1]
            check_attention(case, out, lse, A.attention_case(case, heads=heads), heads=heads)
