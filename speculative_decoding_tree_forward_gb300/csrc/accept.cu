// Greedy tree acceptance: vocab argmax at every node, then the longest
// accepted root path.
//
// NVIDIA draft-length article (Acceptance Length: accepted drafts up to the
// first mismatch plus the target's own token, 1 <= AL <= 1 + D) and the
// SwiftSpec summary, Figure 2 (the target picks one path of the tree).
//
// Kernel 1 streams the fp32 logits once (16-byte loads, a slice of the vocab
// per CTA, sized on the host so that all CTAs are resident at once) and keeps
// (max, lowest index) per slice.  Kernel 2 runs one CTA
// per request: it reduces the chunk partials to argmax[i], builds the
// ancestor bitmasks, marks node i "ok" when token[i] equals the argmax at its
// parent, accepts i iff every node on its root path is ok, and picks the
// deepest accepted node (smallest index on ties).  Because parent[i] < i,
// the path in root-to-leaf order is the ancestor set in increasing index
// order, so it is written straight from the winner's bitmask.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kArgmaxThreads = 256;

__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

// At most 32 registers: eight CTAs per SM, the residency the host's slice
// sizing assumes (rows x slices = about eight CTAs per SM, one wave).
__global__ void __launch_bounds__(kArgmaxThreads, 8) argmax_chunk_kernel(const AcceptParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x;  // b * n_tree_max + i
  const int b = row / p.n_tree_max, i = row % p.n_tree_max;
  int n = p.n_tree[b];
  n = min(max(n, 0), p.n_tree_max);
  if (i >= n) return;
  const int64_t v0 = static_cast<int64_t>(blockIdx.y) * p.chunk;
  const int64_t v1 = min(static_cast<int64_t>(p.vocab), v0 + p.chunk);
  const float* lg = p.logits + static_cast<int64_t>(row) * p.vocab;
  float bv = -INFINITY;
  int bi = INT32_MAX;
  // vector body when the row start is 16-byte aligned (vocab % 4 == 0)
  if ((p.vocab & 3) == 0) {
    const float4* lg4 = reinterpret_cast<const float4*>(lg);
    const int a = static_cast<int>(v0 / 4), e = static_cast<int>(v1 / 4);  // vocab < 2^31
#pragma unroll 8
    for (int x = a + static_cast<int>(threadIdx.x); x < e; x += kArgmaxThreads) {
      const float4 f = __ldcs(lg4 + x);
      const int base = x * 4;
      better(bv, bi, f.x, base);
      better(bv, bi, f.y, base + 1);
      better(bv, bi, f.z, base + 2);
      better(bv, bi, f.w, base + 3);
    }
  } else {
    for (int64_t x = v0 + threadIdx.x; x < v1; x += kArgmaxThreads) better(bv, bi, __ldcs(lg + x), static_cast<int>(x));
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bv, bi, ov, oi);
  }
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ int si[kArgmaxThreads / 32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kArgmaxThreads / 32; ++w) better(bv, bi, sv[w], si[w]);
    p.part_val[static_cast<int64_t>(row) * p.num_chunks + blockIdx.y] = bv;
    p.part_idx[static_cast<int64_t>(row) * p.num_chunks + blockIdx.y] = bi;
  }
}

__device__ __forceinline__ void block_sync() { __syncthreads(); }

__global__ void __launch_bounds__(TS_MAX_TREE) accept_scan_kernel(const AcceptParams p) {
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  __shared__ uint32_t anc[TS_MAX_TREE][4];
  __shared__ int jmp[TS_MAX_TREE];
  __shared__ int am_s[TS_MAX_TREE];
  __shared__ uint32_t ok_mask[4];
  __shared__ int best_key[TS_MAX_TREE / 32];

  // The tree (sizes, parents, tokens) is an input of the call, final before
  // the argmax kernel passed its own wait, which precedes this grid's launch:
  // read it and build the ancestor masks before waiting for the argmax.
  int n = p.n_tree[b];
  if (n < 0 || n > p.n_tree_max) {
    if (i == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);
    n = min(max(n, 0), p.n_tree_max);
  }
  const int64_t rowbase = static_cast<int64_t>(b) * p.n_tree_max;
  int par = -1, tok = 0;
  if (i < n) {
    par = p.parent[rowbase + i];
    if (par < -1 || par >= i) par = -1;  // reported by build_ancestor_masks
    tok = p.tokens[rowbase + i];
    // a draft token outside the vocab never equals an argmax: never accepted
    // (the root's own token is not tested)
    if (i > 0 && (tok < 0 || tok >= p.vocab)) report_error(p.err, TS_DEVERR_BAD_TOKEN);
  }
  if (n > 0) build_ancestor_masks(p.parent + rowbase, n, anc, jmp, i, blockDim.x, p.err, block_sync);
  pdl_wait();
  pdl_launch_dependents();
  // argmax per node from the chunk partials
  int am = -1;
  if (i < n) {  // sixteen chunks' partials requested together: one round trip for up to 16 chunks
    float bv = -INFINITY;
    int bi = INT32_MAX;
    const float* pv = p.part_val + (rowbase + i) * p.num_chunks;
    const int* pi = p.part_idx + (rowbase + i) * p.num_chunks;
    for (int c0 = 0; c0 < p.num_chunks; c0 += 16) {
      float v[16];
      int x[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const bool in = c0 + q < p.num_chunks;
        v[q] = in ? pv[c0 + q] : -INFINITY;
        x[q] = in ? pi[c0 + q] : INT32_MAX;
      }
#pragma unroll
      for (int q = 0; q < 16; ++q) better(bv, bi, v[q], x[q]);
    }
    am = bi;
  }
  if (i < p.n_tree_max) p.argmax[rowbase + i] = (i < n) ? am : -1;
  am_s[i] = am;
  if (n == 0) {
    if (i < p.n_tree_max) p.path[rowbase + i] = -1;
    if (i == 0) {
      p.accept_len[b] = 0;
      p.bonus[b] = -1;
      if (p.verified_len) p.verified_len[b] = 0;
    }
    if (p.verified)
      for (int x = i; x <= p.n_tree_max; x += blockDim.x) p.verified[static_cast<int64_t>(b) * (p.n_tree_max + 1) + x] = -1;
    return;
  }
  __syncthreads();  // am_s complete
  // ok[i]: the root, or a child whose token is the target argmax at its parent
  bool ok = false;
  if (i < n) ok = (i == 0) || (par >= 0 && tok == am_s[par]);
  const unsigned bal = __ballot_sync(0xffffffffu, ok);
  if ((i & 31) == 0) ok_mask[i >> 5] = bal;
  __syncthreads();
  int key = -1;
  if (i < n) {
    bool acc = true;
#pragma unroll
    for (int w = 0; w < 4; ++w) acc = acc && ((anc[i][w] & ~ok_mask[w]) == 0u);
    if (acc) {
      const int depth = __popc(anc[i][0]) + __popc(anc[i][1]) + __popc(anc[i][2]) + __popc(anc[i][3]) - 1;
      key = (depth << 8) | (255 - i);  // deeper wins, then the smaller index
    }
  }
  for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
  if ((i & 31) == 0) best_key[i >> 5] = key;
  __syncthreads();
  int best = best_key[0];
  for (int w = 1; w < TS_MAX_TREE / 32; ++w) best = max(best, best_key[w]);
  const int last = 255 - (best & 255);  // node 0 is always accepted, so best >= 0
  uint32_t pm[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) pm[w] = anc[last][w];
  const int al = __popc(pm[0]) + __popc(pm[1]) + __popc(pm[2]) + __popc(pm[3]);
  // position of node i on the path = number of path nodes with a smaller index
  if (i < p.n_tree_max) {
    const bool on = i < n && ((pm[i >> 5] >> (i & 31)) & 1u);
    if (on) {
      int pos = 0;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if (w < (i >> 5)) pos += __popc(pm[w]);
        else if (w == (i >> 5)) pos += __popc(pm[w] & ((1u << (i & 31)) - 1u));
      }
      p.path[rowbase + pos] = i;
      if (p.verified) p.verified[static_cast<int64_t>(b) * (p.n_tree_max + 1) + pos] = tok;
    }
    if (i >= al) p.path[rowbase + i] = -1;
  }
  if (p.verified) {
    int32_t* vrow = p.verified + static_cast<int64_t>(b) * (p.n_tree_max + 1);
    for (int x = i; x <= p.n_tree_max; x += blockDim.x)
      if (x > al) vrow[x] = -1;
    if (i == 0) vrow[al] = am_s[last];
  }
  if (i == 0) {
    p.accept_len[b] = al;
    p.bonus[b] = am_s[last];
    if (p.verified_len) p.verified_len[b] = al + 1;
  }
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream) {
  dim3 grid(p.num_req * p.n_tree_max, p.num_chunks);
  cudaError_t e = launch_pdl(argmax_chunk_kernel, grid, dim3(kArgmaxThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(accept_scan_kernel, dim3(p.num_req), dim3(TS_MAX_TREE), 0, stream, p);
}

}  // namespace ts
