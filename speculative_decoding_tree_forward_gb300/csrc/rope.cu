// Rotary position embedding of the verify / expand queries at their tree
// positions, run by the attention call before the attention kernel (SwiftSpec
// summary §3.3: RoPE inside the tree attention; a tree node's position is the
// prefix length plus its depth, the root at depth 0, so siblings share a
// position and a root path counts up like ordinary decoding).
//
// One CTA per (request, query node): thread 0 walks the node's parent chain
// for its depth; threads j < d/2 compute the pair angle position *
// theta^(-2j/d) in fp64 (positions reach 10^5 and more, where an fp32 angle
// would be off by several 1e-3 rad) and its cosine and sine; then every
// (head, pair) of the node's G x Hkv heads turns (x_j, x_{j+d/2}) in fp32 and
// stores bf16 into the workspace copy of Q that the attention kernel reads.
#include "attn_common.cuh"

namespace ts {
namespace {

constexpr int kRopeThreads = 128;

__global__ void __launch_bounds__(kRopeThreads) rope_q_kernel(const AttnParams p, const __nv_bfloat16* q_in,
                                                              __nv_bfloat16* q_out, double theta) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x / p.n_query;
  const int r = blockIdx.x % p.n_query;
  const int half = p.head_dim / 2;
  __shared__ int pos_s;
  __shared__ float cs[64], sn[64];
  if (threadIdx.x == 0) {
    int P, n;
    attn_lengths(p, b, P, n, false);  // clamped exactly as the attention kernels clamp
    int u = n - p.n_query + r, depth = 0;
    const int32_t* par = p.parent + static_cast<int64_t>(b) * p.n_tree_max;
    for (int guard = 0; guard < TS_MAX_TREE; ++guard) {  // parent[i] < i: at most n steps
      int q = par[u];
      if (q < -1 || q >= u) q = -1;  // reported by the attention kernel
      if (q < 0) break;
      u = q;
      ++depth;
    }
    pos_s = P + depth;
  }
  __syncthreads();
  if (threadIdx.x < half) {
    const double a = static_cast<double>(pos_s) * pow(theta, -2.0 * threadIdx.x / p.head_dim);
    double c, s;
    sincos(a, &s, &c);
    cs[threadIdx.x] = static_cast<float>(c);
    sn[threadIdx.x] = static_cast<float>(s);
  }
  __syncthreads();
  const int64_t row = (static_cast<int64_t>(b) * p.n_query + r) * p.hq * p.head_dim;
  for (int x = threadIdx.x; x < p.hq * half; x += kRopeThreads) {
    const int h = x / half, j = x % half;
    const int64_t i0 = row + static_cast<int64_t>(h) * p.head_dim + j;
    const float a0 = __bfloat162float(q_in[i0]), a1 = __bfloat162float(q_in[i0 + half]);
    q_out[i0] = __float2bfloat16_rn(a0 * cs[j] - a1 * sn[j]);
    q_out[i0 + half] = __float2bfloat16_rn(a0 * sn[j] + a1 * cs[j]);
  }
}

}  // namespace

cudaError_t launch_rope_q(const AttnParams& p, const void* q_in, void* q_out, float theta, cudaStream_t stream) {
  return launch_pdl(rope_q_kernel, dim3(p.num_req * p.n_query), dim3(kRopeThreads), 0, stream, p,
                    static_cast<const __nv_bfloat16*>(q_in), static_cast<__nv_bfloat16*>(q_out),
                    static_cast<double>(theta));
}

}  // namespace ts
