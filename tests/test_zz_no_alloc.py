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
from gpu_util import ATOL, LSE_ATOL, LSE_RTOL, RTOL, attn_inputs  # noqa: E402


def _close(a, b, atol, rtol):
    a, b = a.double(), b.double()
    return bool(((a - b).abs() <= atol + rtol * b.abs()).all())


@pytest.mark.parametrize("num_ctas", [0, 1000])
def test_no_alloc_matches_workspace_entry_point_twice(num_ctas):
    """Two calls in a row through the C ABI; the second sees the first call's leftovers in the scratch.

    num_ctas=1000 asks for more split-KV CTAs than the scratch can hold partials
    for, so the entry point has to shrink the split to fit.
    """
    case = W.random_attn_case(21, num_req=8, hq=64, hkv=8, d=128, n_tree_max=16, prefix_range=(300, 1200),
                              paged=False)
    d = attn_inputs(case)
    ref_out, ref_lse = ts.tree_attn_forward(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"],
                                            d["parent"])
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        ts.tree_attn_forward_noalloc(d["q"], d["k_cache"], d["v_cache"], d["prefix_len"], d["n_tree"], d["parent"],
                                     out, lse, num_ctas=num_ctas)
        torch.cuda.synchronize()
        assert _close(out, ref_out, ATOL, RTOL)
        assert _close(lse, ref_lse, LSE_ATOL, LSE_RTOL)
