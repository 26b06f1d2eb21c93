"""Helpers shared by the GPU parity tests: host arrays -> device tensors, oracle comparison."""
import numpy as np
import torch

from workloads import attn_inputs, bf16_dev, i32_dev  # noqa: F401  (device copies of the seeded inputs)

# Attention tolerance (bf16 inputs, fp32 accumulation, bf16 output):
# |gpu - oracle| <= ATOL + RTOL * |oracle| elementwise.
ATOL, RTOL = 2e-3, 1e-2
# log-sum-exp is accumulated in fp32 from exact bf16 products; its error is
# the fp32 rounding of a few thousand exp2 terms and of the scaled score.
LSE_ATOL, LSE_RTOL = 1e-4, 1e-4


def bf16_host_f64(t: torch.Tensor) -> np.ndarray:
    bits = t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def check_attention(case, out, lse, ref, requests=None, heads=None):
    """Compare GPU (out bf16 [B][nq][Hq][d], lse [B][Hq][nq]) with oracle results for chosen rows."""
    o = bf16_host_f64(out)
    l = lse.cpu().numpy().astype(np.float64) if lse is not None else None
    worst = 0.0
    for b, (ro, rl) in ref.items():
        hs = range(case.num_q_heads) if heads is None else heads
        for h in hs:
            got, exp = o[b][:, h, :], ro[:, h, :]
            err = np.abs(got - exp) - (ATOL + RTOL * np.abs(exp))
            worst = max(worst, float(err.max()))
            assert (err <= 0).all(), f"request {b} head {h}: max excess {err.max():.3e}"
            if l is not None:
                e2 = np.abs(l[b][h] - rl[h]) - (LSE_ATOL + LSE_RTOL * np.abs(rl[h]))
                assert (e2 <= 0).all(), f"lse request {b} head {h}: max excess {e2.max():.3e}"
    return worst
