// Rotary position embedding of the verify / expand queries at their tree
// positions, run by the attention call before the attention kernel (SwiftSpec
// summary §3.3: RoPE inside the tree attention; a tree node's position is the
// prefix length plus its depth, the root at depth 0, so siblings share a
// position and a root path counts up like ordinary decoding).
//
// One CTA per (request, query node): the request's parents are staged in
// shared memory and thread 0 walks the node's chain there for its depth.
// Thread j < d/2 forms the pair angle position * inv_freq[j] in fp64 (the
// host computed inv_freq[j] = theta^(-2j/d) in fp64: positions reach 10^5,
// where an fp32 product would be off by several 1e-3 rad), reduces it modulo
// 2 pi in fp64 and takes sincosf of the reduced angle.  Then every (head,
// 8 pairs) item of the node turns (x_j, x_{j+d/2}) in fp32 with 16-byte loads
// and stores, into the workspace copy of Q that the attention kernel reads.
#include "attn_common.cuh"

namespace ts {
namespace {

constexpr int kRopeThreads = 128;

__global__ void __launch_bounds__(kRopeThreads) rope_q_kernel(const AttnParams p, const RopeFreqs f,
                                                              const __nv_bfloat16* __restrict__ q_in,
                                                              __nv_bfloat16* __restrict__ q_out) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x / p.n_query;
  const int r = blockIdx.x % p.n_query;
  const int half = p.head_dim / 2;
  __shared__ int pos_s;
  __shared__ int par_s[TS_MAX_TREE];
  __shared__ float cs[64], sn[64];
  int P, n;
  attn_lengths(p, b, P, n, false);  // clamped exactly as the attention kernels clamp
  for (int i = threadIdx.x; i < n; i += kRopeThreads) {  // the request's parents, one coalesced load
    const int q = p.parent[static_cast<int64_t>(b) * p.n_tree_max + i];
    par_s[i] = (q < -1 || q >= i) ? -1 : q;  // a bad parent is reported by the attention kernel
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int u = n - p.n_query + r, depth = 0;
    while (par_s[u] >= 0) {  // parent[i] < i: at most n steps
      u = par_s[u];
      ++depth;
    }
    pos_s = P + depth;
  }
  __syncthreads();
  if (threadIdx.x < half) {
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    const double a = static_cast<double>(pos_s) * f.inv_freq[threadIdx.x];
    const float red = static_cast<float>(a - kTwoPi * rint(a / kTwoPi));  // in [-pi, pi]
    float s, c;
    sincosf(red, &s, &c);
    cs[threadIdx.x] = c;
    sn[threadIdx.x] = s;
  }
  __syncthreads();
  const int64_t row = (static_cast<int64_t>(b) * p.n_query + r) * p.hq * p.head_dim;
  const int per_head = half / 8;  // 8-pair items per head
  for (int x = threadIdx.x; x < p.hq * per_head; x += kRopeThreads) {
    const int h = x / per_head, j0 = (x % per_head) * 8;
    const int64_t i0 = row + static_cast<int64_t>(h) * p.head_dim + j0;
    const uint4 va = *reinterpret_cast<const uint4*>(q_in + i0);
    const uint4 vb = *reinterpret_cast<const uint4*>(q_in + i0 + half);
    const __nv_bfloat16* a8 = reinterpret_cast<const __nv_bfloat16*>(&va);
    const __nv_bfloat16* b8 = reinterpret_cast<const __nv_bfloat16*>(&vb);
    uint4 oa, ob;
    __nv_bfloat16* oa8 = reinterpret_cast<__nv_bfloat16*>(&oa);
    __nv_bfloat16* ob8 = reinterpret_cast<__nv_bfloat16*>(&ob);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x0 = __bfloat162float(a8[e]), x1 = __bfloat162float(b8[e]);
      const float c = cs[j0 + e], s = sn[j0 + e];
      oa8[e] = __float2bfloat16_rn(x0 * c - x1 * s);
      ob8[e] = __float2bfloat16_rn(x0 * s + x1 * c);
    }
    *reinterpret_cast<uint4*>(q_out + i0) = oa;
    *reinterpret_cast<uint4*>(q_out + i0 + half) = ob;
  }
}

}  // namespace

cudaError_t launch_rope_q(const AttnParams& p, const RopeFreqs& f, const void* q_in, void* q_out,
                          cudaStream_t stream) {
  return launch_pdl(rope_q_kernel, dim3(p.num_req * p.n_query), dim3(kRopeThreads), 0, stream, p, f,
                    static_cast<const __nv_bfloat16*>(q_in), static_cast<__nv_bfloat16*>(q_out));
}

}  // namespace ts
