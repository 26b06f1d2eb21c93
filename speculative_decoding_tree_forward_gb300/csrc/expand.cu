// Draft-side tree growth: maximum-likelihood expansion and the selection of
// the most promising subtree.
//
// SwiftSpec summary, §3.1.1 (Algorithm 1: Expand the w most probable leaves d
// times, Select a subtree of size bs) and §3.1.3 (a node's value is the
// log-softmax probability of its token under the draft model, its weight the
// sum of the values from the root; the leaves to expand come from a priority
// queue); Figure 2 (w nodes per expansion).
//
// Kernel 1 (candidates) streams the draft logits of the queried nodes once:
// each CTA takes a vocab slice of one row with 16-byte loads and keeps, per
// thread, an online log-sum-exp and a sorted list of its largest logits
// (ties: lower token; 8 or 16 long, the smallest that holds k); the block
// merges the lists (one warp arg-max over list heads per entry) and writes
// one partial per (row, slice).  Per batch of eight 16-byte loads the
// log-sum-exp takes the batch max first, so its exponentials are independent.
// Kernel 2 (step) runs one CTA per request: it merges a row's partials into
// the node's k candidates (value = logit - log-sum-exp), then makes the w
// picks of the step, each a block-wide arg-max over the nodes' next
// candidates.  Kernel 3 (select) ranks the nodes by weight and keeps the top
// bs in index order.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kCandThreads = 256;
constexpr int K = TS_MAX_EXPAND;  // candidate slots stored per (row, slice) and per node

// (value, index) order of the candidate lists: larger value first, then the
// lower index
__device__ __forceinline__ bool ahead(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// Inserts (x, i) into a list sorted by `ahead`; x arrives with the largest
// index seen so far, so an equal value stays behind the entries present.
template <int KL>
__device__ __forceinline__ void list_insert(float (&val)[KL], int (&idx)[KL], float x, int i) {
  if (!(x > val[KL - 1])) return;
  float cv = x;
  int ci = i;
#pragma unroll
  for (int j = 0; j < KL; ++j) {
    if (cv > val[j]) {
      const float tv = val[j];
      const int ti = idx[j];
      val[j] = cv;
      idx[j] = ci;
      cv = tv;
      ci = ti;
    }
  }
}

// Drops the head of a sorted list (the next entry becomes the head).
template <int KL>
__device__ __forceinline__ void list_pop(float (&val)[KL], int (&idx)[KL]) {
#pragma unroll
  for (int j = 0; j < KL - 1; ++j) {
    val[j] = val[j + 1];
    idx[j] = idx[j + 1];
  }
  val[KL - 1] = -INFINITY;
  idx[KL - 1] = INT32_MAX;
}

// Merges the lanes' sorted lists: round j's winner (the best head over the
// warp) goes to (out_v[j], out_i[j]) on every lane, and its lane pops it.
template <int KL>
__device__ __forceinline__ void warp_merge(float (&val)[KL], int (&idx)[KL], float (&out_v)[KL], int (&out_i)[KL]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < KL; ++j) {
    float bv = val[0];
    int bi = idx[0], bl = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
      if (ahead(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
        bl = ol;
      }
    }
    out_v[j] = bv;
    out_i[j] = bi;
    if (lane == bl) list_pop(val, idx);
  }
}

// (max, sum of exp(x - max)) pairs; __expf's error is a few ulp here (its
// argument is <= 0 and above -100 for finite logits of one distribution)
__device__ __forceinline__ void lse_combine(float& m, float& s, float om, float os) {
  if (om > m) {
    s = s * __expf(m - om) + os;
    m = om;
  } else if (om != -INFINITY) {
    s += os * __expf(om - m);
  }
}

__device__ __forceinline__ int clamp_n(const ExpandParams& p, int b) {
  return min(max(p.n_tree[b], 0), p.n_tree_max);
}

template <int KL>  // list length: the smallest of 8, 16 that holds k
__global__ void __launch_bounds__(kCandThreads) cand_partial_kernel(const ExpandParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x;  // b * w + r
  const int b = row / p.w;
  const int u = p.rows[row];
  if (u < 0 || u >= clamp_n(p, b)) return;  // not a queried node: the step kernel skips the row too
  const int64_t v0 = static_cast<int64_t>(blockIdx.y) * p.slice;
  const int64_t v1 = min(static_cast<int64_t>(p.vocab), v0 + p.slice);
  const float* lg = p.logits + static_cast<int64_t>(row) * p.vocab;
  float m = -INFINITY, s = 0.f;
  float val[KL];
  int idx[KL];
#pragma unroll
  for (int j = 0; j < KL; ++j) {
    val[j] = -INFINITY;
    idx[j] = INT32_MAX;
  }
  auto push = [&](float x, int i) {
    if (x > m) {
      s = s * __expf(m - x) + 1.f;
      m = x;
    } else {
      s += __expf(x - m);
    }
    list_insert<KL>(val, idx, x, i);
  };
  if ((p.vocab & 3) == 0) {  // 16-byte rows: slices are multiples of 1024 floats
    // eight 16-byte loads in flight per thread, issued before any of them is
    // consumed (the insertions branch)
    constexpr int kLoads = 8;
    const float4* lg4 = reinterpret_cast<const float4*>(lg);
    const int64_t e4 = v1 / 4;
    for (int64_t x0 = v0 / 4 + threadIdx.x; x0 < e4; x0 += kLoads * kCandThreads) {
      float4 f[kLoads];
#pragma unroll
      for (int q = 0; q < kLoads; ++q)
        f[q] = x0 + q * kCandThreads < e4 ? __ldcs(lg4 + x0 + q * kCandThreads)
                                          : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      // log-sum-exp of the batch: its max first, then independent exponentials
      float bm = m;
#pragma unroll
      for (int q = 0; q < kLoads; ++q) bm = fmaxf(bm, fmaxf(fmaxf(f[q].x, f[q].y), fmaxf(f[q].z, f[q].w)));
      if (bm > m) {
        s *= __expf(m - bm);
        m = bm;
      }
      float es[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kLoads; ++q) {
        es[0] += __expf(f[q].x - m);   // -inf (past the slice) gives 0
        es[1] += __expf(f[q].y - m);
        es[2] += __expf(f[q].z - m);
        es[3] += __expf(f[q].w - m);
      }
      s += (es[0] + es[1]) + (es[2] + es[3]);
#pragma unroll
      for (int q = 0; q < kLoads; ++q) {
        if (x0 + q * kCandThreads >= e4) break;
        const int i = static_cast<int>((x0 + q * kCandThreads) * 4);
        list_insert<KL>(val, idx, f[q].x, i);
        list_insert<KL>(val, idx, f[q].y, i + 1);
        list_insert<KL>(val, idx, f[q].z, i + 2);
        list_insert<KL>(val, idx, f[q].w, i + 3);
      }
    }
  } else {
    for (int64_t x = v0 + threadIdx.x; x < v1; x += kCandThreads) push(__ldcs(lg + x), static_cast<int>(x));
  }
  // block: (m, s) by shuffles + shared memory; lists warp by warp, then warp 0
  __shared__ float wm[kCandThreads / 32], wsum[kCandThreads / 32];
  __shared__ float wv[kCandThreads / 32][KL];
  __shared__ int wi[kCandThreads / 32][KL];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lse_combine(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
  float tv[KL];
  int ti[KL];
  warp_merge<KL>(val, idx, tv, ti);
  if (lane == 0) {
    wm[warp] = m;
    wsum[warp] = s;
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      wv[warp][j] = tv[j];
      wi[warp][j] = ti[j];
    }
  }
  __syncthreads();
  if (warp == 0) {
    float bm = -INFINITY, bs = 0.f;
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      val[j] = -INFINITY;
      idx[j] = INT32_MAX;
    }
    if (lane < kCandThreads / 32) {
      bm = wm[lane];
      bs = wsum[lane];
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        val[j] = wv[lane][j];
        idx[j] = wi[lane][j];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      lse_combine(bm, bs, __shfl_xor_sync(0xffffffffu, bm, o), __shfl_xor_sync(0xffffffffu, bs, o));
    warp_merge<KL>(val, idx, tv, ti);
    if (lane == 0) {
      CandPartial* out = p.part + static_cast<int64_t>(row) * p.num_slices + blockIdx.y;
      out->m = bm;
      out->s = bs;
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        out->val[j] = tv[j];
        out->idx[j] = ti[j];
      }
    }
  }
}

constexpr int kStepThreads = 2 * TS_MAX_TREE;  // thread i < n owns node i; warp r merges row r

template <int KL>
__global__ void __launch_bounds__(kStepThreads) expand_step_kernel(const ExpandParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nb = static_cast<int64_t>(b) * p.n_tree_max;
  __shared__ float c_lp[TS_MAX_TREE][KL];
  __shared__ int c_tok[TS_MAX_TREE][KL];
  __shared__ int rows_s[K];
  __shared__ float red_v[kStepThreads / 32];
  __shared__ int red_i[kStepThreads / 32];
  int n = p.n_tree[b];
  if (n < 0 || n > p.n_tree_max) {
    if (tid == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);
    n = min(max(n, 0), p.n_tree_max);
  }
  if (tid < p.w) rows_s[tid] = p.rows[static_cast<int64_t>(b) * p.w + tid];
  // each node's candidates as they stand (rows queried now are replaced below)
  int taken = p.k;
  const float my_w = tid < n ? p.weight[nb + tid] : 0.f;
  if (tid < n) {
    taken = min(max(p.cand_taken[nb + tid], 0), p.k);
    float lp[KL];
    int tk[KL];
#pragma unroll
    for (int j = 0; j < KL; ++j) {  // issued together
      lp[j] = j < p.k ? p.cand_lp[(nb + tid) * p.k + j] : -INFINITY;
      tk[j] = j < p.k ? p.cand_tok[(nb + tid) * p.k + j] : -1;
    }
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      c_lp[tid][j] = lp[j];
      c_tok[tid][j] = tk[j];
    }
  }
  __syncthreads();
  // ---- 1. the queried rows: merge the slices into k candidates (warp per row)
  for (int r = warp; r < p.w; r += kStepThreads / 32) {
    const int u = rows_s[r];
    if (u < 0) continue;
    if (u >= n) {
      if (lane == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);
      continue;
    }
    const CandPartial* part = p.part + (static_cast<int64_t>(b) * p.w + r) * p.num_slices;
    float val[KL];
    int idx[KL];
    float m = -INFINITY, s = 0.f;
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      val[j] = -INFINITY;
      idx[j] = INT32_MAX;
    }
    if (lane < p.num_slices) {  // num_slices <= 32
      m = part[lane].m;
      s = part[lane].s;
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        val[j] = part[lane].val[j];
        idx[j] = part[lane].idx[j];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lse_combine(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    const float lse = m + logf(s);
    float tv[KL];
    int ti[KL];
    warp_merge<KL>(val, idx, tv, ti);
    if (lane < p.k) {
      float v = -INFINITY;
      int t = -1;
#pragma unroll
      for (int j = 0; j < KL; ++j)
        if (j == lane) {
          v = tv[j];
          t = ti[j];
        }
      const bool real = t != INT32_MAX && v != -INFINITY;
      c_lp[u][lane] = real ? v - lse : -INFINITY;
      c_tok[u][lane] = real ? t : -1;
    }
  }
  __syncthreads();
  for (int r = 0; r < p.w; ++r)
    if (rows_s[r] == tid && tid < n) taken = 0;
  // ---- 2. the picks: each node offers its next candidate
  float key = (tid < n && taken < p.k && c_tok[tid][taken] >= 0) ? my_w + c_lp[tid][taken] : -INFINITY;
  int added = 0;
  for (int j = 0; j < p.w; ++j) {
    if (n >= p.n_tree_max) break;  // uniform: n is the same in every thread
    float bv = key;
    int bi = tid;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ahead(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      red_v[warp] = bv;
      red_i[warp] = bi;
    }
    __syncthreads();
    bv = red_v[0];
    bi = red_i[0];
#pragma unroll
    for (int q = 1; q < kStepThreads / 32; ++q)
      if (ahead(red_v[q], red_i[q], bv, bi)) {
        bv = red_v[q];
        bi = red_i[q];
      }
    __syncthreads();  // red_* is rewritten next round
    if (bv == -INFINITY) break;
    const int nn = n;  // the new node
    if (tid == bi) {
      p.parent[nb + nn] = bi;
      p.tokens[nb + nn] = c_tok[bi][taken];
      p.weight[nb + nn] = bv;
      p.cand_taken[nb + nn] = p.k;
      p.added[static_cast<int64_t>(b) * p.w + j] = nn;
      ++taken;
      key = (taken < p.k && c_tok[tid][taken] >= 0) ? my_w + c_lp[tid][taken] : -INFINITY;
    }
    if (tid == nn) {  // no candidates until its logits come
      taken = p.k;
      key = -INFINITY;
    }
    ++n;
    ++added;
  }
  if (tid < p.w && tid >= added) p.added[static_cast<int64_t>(b) * p.w + tid] = -1;
  // write back the candidates of the queried rows and every node's taken count
  if (tid < n) {
    bool queried = false;
    for (int r = 0; r < p.w; ++r) queried = queried || rows_s[r] == tid;
    if (queried)
      for (int j = 0; j < p.k; ++j) {
        p.cand_lp[(nb + tid) * p.k + j] = c_lp[tid][j];
        p.cand_tok[(nb + tid) * p.k + j] = c_tok[tid][j];
      }
    if (tid < n - added) p.cand_taken[nb + tid] = taken;
  }
  if (tid == 0) p.n_tree[b] = n;
}

__global__ void __launch_bounds__(TS_MAX_TREE) select_subtree_kernel(const SelectParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nb = static_cast<int64_t>(b) * p.n_tree_max;
  const int64_t ob = static_cast<int64_t>(b) * p.bs;
  __shared__ float w_s[TS_MAX_TREE];
  __shared__ int newidx[TS_MAX_TREE];
  __shared__ int cnt[TS_MAX_TREE / 32];
  int n = p.n_tree[b];
  if (n < 0 || n > p.n_tree_max) {
    if (tid == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);
    n = min(max(n, 0), p.n_tree_max);
  }
  const float wi = tid < n ? p.weight[nb + tid] : -INFINITY;
  w_s[tid] = wi;
  __syncthreads();
  // rank of node tid in (weight descending, index ascending) order
  int rank = 0;
  if (tid < n)
    for (int j = 0; j < n; ++j) rank += ahead(w_s[j], j, wi, tid) ? 1 : 0;
  const bool keep = tid < n && rank < p.bs;
  const unsigned bal = __ballot_sync(0xffffffffu, keep);
  if (lane == 0) cnt[warp] = __popc(bal);
  __syncthreads();
  int before = 0;
  for (int q = 0; q < warp; ++q) before += cnt[q];
  const int ni = before + __popc(bal & ((1u << lane) - 1u));
  newidx[tid] = keep ? ni : -1;
  __syncthreads();
  const int n_sel = min(p.bs, n);
  if (keep) {
    const int par = p.parent[nb + tid];
    int np = -1;
    if (par >= 0 && par < n) {
      np = newidx[par];
      if (np < 0) report_error(p.err, TS_DEVERR_BAD_PARENT);
    } else if (par != -1) {
      report_error(p.err, TS_DEVERR_BAD_PARENT);
    }
    p.keep[ob + ni] = tid;
    p.new_parent[ob + ni] = np;
    p.new_tokens[ob + ni] = p.tokens[nb + tid];
    p.new_weight[ob + ni] = wi;
  }
  for (int j = n_sel + tid; j < p.bs; j += TS_MAX_TREE) {
    p.keep[ob + j] = -1;
    p.new_parent[ob + j] = -1;
    p.new_tokens[ob + j] = 0;
    p.new_weight[ob + j] = -INFINITY;
  }
  if (tid == 0) p.n_sel[b] = n_sel;
}

}  // namespace

cudaError_t launch_expand(const ExpandParams& p, cudaStream_t stream) {
  const dim3 grid(p.num_req * p.w, p.num_slices);
  cudaError_t e = p.k <= 8 ? launch_pdl(cand_partial_kernel<8>, grid, dim3(kCandThreads), 0, stream, p)
                           : launch_pdl(cand_partial_kernel<16>, grid, dim3(kCandThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return p.k <= 8 ? launch_pdl(expand_step_kernel<8>, dim3(p.num_req), dim3(kStepThreads), 0, stream, p)
                  : launch_pdl(expand_step_kernel<16>, dim3(p.num_req), dim3(kStepThreads), 0, stream, p);
}

cudaError_t launch_select(const SelectParams& p, cudaStream_t stream) {
  return launch_pdl(select_subtree_kernel, dim3(p.num_req), dim3(TS_MAX_TREE), 0, stream, p);
}

}  // namespace ts
