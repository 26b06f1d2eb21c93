// Evolving tree cache: re-root walk and in-place KV-row compaction.
//
// SwiftSpec summary, §3.2 (the prefix-cache / tree-cache invariant and its
// update procedure), Figure 4 (t12, t15 promoted, t17, t18 moved to the front
// of the tree cache, the rest dropped) and Figure 2 with its walkthrough
// (re-rooting at t6 reuses its subtree; an out-of-tree token reuses nothing).
//
// Kernel 1 (one CTA per request) walks the verified tokens down the tree,
// taking at each step the lowest-index child that carries the token, and
// writes the source-row list src = path ++ survivors into the workspace plan,
// plus the new prefix length, tree size, parents and tokens.
//
// Kernel 2 moves the rows: one CTA per (chunk of the row bytes, K|V, layer,
// request).  The source list is strictly increasing (parent[i] < i, and
// survivors descend from the last matched node), so every destination row
// P + j is at or below its source row P + src[j]; a CTA first loads its byte
// chunk of every source row into shared memory and only then stores, so no
// row is overwritten before it is read.  Rows whose source equals their
// destination are skipped.  Transfers are 16-byte vectors.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kWalkThreads = TS_MAX_TREE;
constexpr int kGatherThreads = 256;

__device__ __forceinline__ void block_sync() { __syncthreads(); }

__global__ void __launch_bounds__(kWalkThreads) reroot_walk_kernel(const CompactParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  __shared__ int par_s[TS_MAX_TREE];
  __shared__ int tok_s[TS_MAX_TREE];
  __shared__ uint32_t anc[TS_MAX_TREE][4];
  __shared__ int jmp[TS_MAX_TREE];
  __shared__ int path_s[TS_MAX_TREE + 1];
  __shared__ int red[2 * (kWalkThreads / 32)];
  __shared__ int cnt[kWalkThreads / 32];
  __shared__ int ver_s[TS_MAX_TREE + 1];

  const int64_t rowbase = static_cast<int64_t>(b) * p.n_tree_max;
  int n = p.n_tree[b];
  int m = p.m[b];
  int P = p.prefix_len[b];
  bool bad = false;
  if (n < 0 || n > p.n_tree_max) { n = min(max(n, 0), p.n_tree_max); bad = true; }
  if (m < 0 || m > p.m_max) { m = min(max(m, 0), p.m_max); bad = true; }
  const int cap = p.paged ? p.max_blocks * p.page_size : p.max_kv_len;
  if (P < 0 || P + n > cap) { P = min(max(P, 0), max(cap - n, 0)); bad = true; }
  if (bad && i == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);

  // the verified tokens, loaded once (the walk below reads one per step).
  // A walk step matches at most one node, so with n <= TS_MAX_TREE nodes the
  // walk has always ended by step TS_MAX_TREE + 1: later tokens are never read.
  const int mw = min(m, TS_MAX_TREE + 1);
  for (int j = i; j < mw; j += kWalkThreads) ver_s[j] = p.verified[static_cast<int64_t>(b) * p.m_max + j];
  int my_par = -1, my_tok = 0;
  if (i < n) {
    my_par = p.parent[rowbase + i];
    if (my_par < -1 || my_par >= i) {
      report_error(p.err, TS_DEVERR_BAD_PARENT);
      my_par = -1;
    }
    my_tok = p.tokens[rowbase + i];
    par_s[i] = my_par;
    tok_s[i] = my_tok;
  }
  __syncthreads();  // every read of parent/tokens happens before any write (aliasing allowed)

  // ---- walk the verified tokens from the prefix tail
  int cur = -1, plen = 0;
  bool matched_all = true;
  for (int j = 0; j < mw; ++j) {
    const int v = ver_s[j];
    int cand = (i < n && my_par == cur && my_tok == v) ? i : INT32_MAX;
    for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    // two slot sets: set j % 2 is rewritten at step j + 2, after every
    // thread has passed the barrier of step j + 1 and so finished reading it
    if ((i & 31) == 0) red[(j & 1) * (kWalkThreads / 32) + (i >> 5)] = cand;
    __syncthreads();
    int c = red[(j & 1) * (kWalkThreads / 32)];
    for (int w = 1; w < kWalkThreads / 32; ++w) c = min(c, red[(j & 1) * (kWalkThreads / 32) + w]);
    if (c == INT32_MAX) {
      matched_all = false;
      break;
    }
    if (i == 0) path_s[plen] = c;
    ++plen;
    cur = c;
  }
  // ---- survivors: proper descendants of cur (everything when cur = -1)
  build_ancestor_masks(par_s, n, anc, jmp, i, kWalkThreads, nullptr, block_sync);
  bool surv = false;
  if (matched_all && i < n && i != cur) surv = (cur < 0) || ((anc[i][cur >> 5] >> (cur & 31)) & 1u);
  const unsigned bal = __ballot_sync(0xffffffffu, surv);
  if ((i & 31) == 0) cnt[i >> 5] = __popc(bal);
  __syncthreads();
  int before = 0, total = 0;
  for (int w = 0; w < kWalkThreads / 32; ++w) {
    if (w < (i >> 5)) before += cnt[w];
    total += cnt[w];
  }
  const int rank = before + __popc(bal & ((1u << (i & 31)) - 1u));  // new index if surv
  // ranks of all nodes for the parent remap
  __shared__ int newidx[TS_MAX_TREE];
  if (i < n) newidx[i] = surv ? rank : -1;
  __syncthreads();

  int32_t* plan = p.plan + static_cast<int64_t>(b) * kPlanStride;
  if (i == 0) {
    plan[0] = P;
    plan[1] = plen + total;
    p.new_prefix_len[b] = P + plen;
    p.new_n_tree[b] = total;
  }
  if (i < plen) plan[2 + i] = path_s[i];
  if (surv) {
    plan[2 + plen + rank] = i;
    const int np = (my_par == cur) ? -1 : newidx[my_par];
    p.new_parent[rowbase + rank] = np;
    p.new_tokens[rowbase + rank] = my_tok;
  }
  if (p.src_rows != nullptr && i < p.n_tree_max) {
    int v = -1;
    if (i < plen) v = path_s[i];
    p.src_rows[rowbase + i] = v;  // survivors overwrite their slots below
  }
  __syncthreads();
  if (p.src_rows != nullptr && surv) p.src_rows[rowbase + plen + rank] = i;
  // entries of the new tree beyond its size
  if (i >= total && i < p.n_tree_max) {
    p.new_parent[rowbase + i] = -1;
    p.new_tokens[rowbase + i] = 0;
  }
}

__device__ __forceinline__ uint8_t* row_ptr(const CompactParams& p, void* layer, int b, int row) {
  uint8_t* base = static_cast<uint8_t*>(layer);
  if (!p.paged) return base + (static_cast<int64_t>(b) * p.max_kv_len + row) * p.row_bytes;
  const int blk = p.block_table[static_cast<int64_t>(b) * p.max_blocks + row / p.page_size];
  if (blk < 0 || blk >= p.num_blocks) return nullptr;
  return base + (static_cast<int64_t>(blk) * p.page_size + row % p.page_size) * p.row_bytes;
}

__global__ void __launch_bounds__(kGatherThreads) compact_gather_kernel(const CompactParams p) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ uint4 buf[];  // [rows][chunk_bytes / 16]
  __shared__ int plan_s[kPlanStride];
  const int group = blockIdx.z;
  const int kv = blockIdx.y;  // 0 = K, 1 = V
  const int layer = blockIdx.x / p.num_req;
  const int b = blockIdx.x % p.num_req;
  const int32_t* plan = p.plan + static_cast<int64_t>(b) * kPlanStride;
  for (int x = threadIdx.x; x < kPlanStride; x += blockDim.x) plan_s[x] = plan[x];
  __syncthreads();
  const int P = plan_s[0];
  const int L = min(max(plan_s[1], 0), TS_MAX_TREE);
  void* base = kv == 0 ? p.k_layers[layer] : p.v_layers[layer];
  const int vecs = p.chunk_bytes / 16;
  const int c0 = group * p.chunk_bytes;
  const int nvec = min(vecs, (p.row_bytes - c0) / 16);
  if (nvec <= 0) return;
  const int total = L * nvec;
  // load phase: four independent 16-byte loads in flight per thread
  for (int x0 = threadIdx.x; x0 < total; x0 += 4 * kGatherThreads) {
    uint4 v[4];
    int slot[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int x = x0 + q * kGatherThreads;
      slot[q] = -1;
      if (x < total) {
        const int j = x / nvec, e = x % nvec;
        const int src = plan_s[2 + j];
        if (src != j) {
          const uint8_t* sp = row_ptr(p, base, b, P + src);
          if (sp == nullptr) {
            report_error(p.err, TS_DEVERR_BAD_BLOCK);
          } else {
            v[q] = *reinterpret_cast<const uint4*>(sp + c0 + 16 * e);
            slot[q] = j * vecs + e;
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (slot[q] >= 0) buf[slot[q]] = v[q];
  }
  __syncthreads();
  // store phase
  for (int x = threadIdx.x; x < total; x += kGatherThreads) {
    const int j = x / nvec, e = x % nvec;
    const int src = plan_s[2 + j];
    if (src == j) continue;
    uint8_t* d = row_ptr(p, base, b, P + j);
    const uint8_t* sp = row_ptr(p, base, b, P + src);
    if (d == nullptr || sp == nullptr) continue;
    *reinterpret_cast<uint4*>(d + c0 + 16 * e) = buf[j * vecs + e];
  }
}

}  // namespace

cudaError_t launch_compact(const CompactParams& p, cudaStream_t stream) {
  cudaError_t e = launch_pdl(reroot_walk_kernel, dim3(p.num_req), dim3(kWalkThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(p.n_tree_max) * p.chunk_bytes;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(compact_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  dim3 grid(p.num_layers * p.num_req, 2, p.num_chunk_groups);
  return launch_pdl(compact_gather_kernel, grid, dim3(kGatherThreads), smem, stream, p);
}

}  // namespace ts
