// Tree metadata: depth and ancestor-or-self bitmask of every node.
//
// SwiftSpec summary, §3.1.3 / Figure 3: the attention mask row of a node is
// its ancestor set plus itself (t7 -> t1, t2, t4, t7).  One CTA per request
// builds the 128-bit masks by pointer jumping (common.cuh); depth is the
// mask's population count minus one.  The attention and acceptance kernels
// build the same masks in shared memory themselves; this entry point exposes
// them for callers and tests.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

__device__ __forceinline__ void block_sync() { __syncthreads(); }

__global__ void __launch_bounds__(TS_MAX_TREE) tree_meta_kernel(const int32_t* parent, const int32_t* n_tree,
                                                               int n_tree_max, int32_t* depth, uint32_t* anc_out,
                                                               unsigned* err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ uint32_t anc[TS_MAX_TREE][4];
  __shared__ int jmp[TS_MAX_TREE];
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  int n = n_tree[b];
  if (n < 0 || n > n_tree_max) {
    if (i == 0) report_error(err, TS_DEVERR_BAD_LENGTH);
    n = min(max(n, 0), n_tree_max);
  }
  const int64_t rowbase = static_cast<int64_t>(b) * n_tree_max;
  build_ancestor_masks(parent + rowbase, n, anc, jmp, i, blockDim.x, err, block_sync);
  if (i < n_tree_max) {
    uint32_t a[4] = {0, 0, 0, 0};
    int d = -1;
    if (i < n) {
#pragma unroll
      for (int w = 0; w < 4; ++w) a[w] = anc[i][w];
      d = __popc(a[0]) + __popc(a[1]) + __popc(a[2]) + __popc(a[3]) - 1;
    }
    depth[rowbase + i] = d;
    reinterpret_cast<uint4*>(anc_out)[rowbase + i] = make_uint4(a[0], a[1], a[2], a[3]);
  }
}

}  // namespace

cudaError_t launch_tree_meta(const int32_t* parent, const int32_t* n_tree, int num_req, int n_tree_max,
                             int32_t* depth, uint32_t* anc, unsigned* err, cudaStream_t stream) {
  return launch_pdl(tree_meta_kernel, dim3(num_req), dim3(TS_MAX_TREE), 0, stream, parent, n_tree, n_tree_max, depth,
                    anc, err);
}

}  // namespace ts
