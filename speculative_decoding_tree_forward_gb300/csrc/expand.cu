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
// each CTA takes a vocab slice of one row in batches of 16 values per thread
// (four 16-byte loads issued together), keeps an online log-sum-exp, and
// selects the slice's k largest logits (ties: lower token) without sorted
// lists: per batch, the k-th largest of a warp's 32 per-thread maxima bounds
// the warp's k-th largest value from below; the warps publish their bounds
// in shared memory and filter with the largest, so only values at or above
// it go to a shared-memory list.  The entries at or above the final bound
// are gathered and ranked (the count of entries ahead of each); the k best
// are those of rank below k.  A CTA whose list overflows (heavy ties) takes
// its k best in k rounds of block arg-max.
// Kernel 2 (step) runs one CTA per request.  It loads the tree state before
// waiting for kernel 1; then each warp merges one queried row (lower bounds
// of the row's k-th largest: any slice's k-th entry and the k-th largest
// slice head; the entries at or above them are ranked; the row's
// log-sum-exp comes from the slices' pairs).  Warp 0 then makes the step's w
// picks: every node offers its untaken candidates with keys weight +
// log-prob that never increase, so the picks are the w largest keys overall
// (ties: lower node, then earlier slot); a bound from the nodes' heads and
// from any node's w-th key limits the slots that are ranked.  Many equal
// keys fall back to w rounds of warp arg-max.  Kernel 3 (select) ranks the
// nodes by weight and keeps the top bs in index order.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kCandThreads = 512;
constexpr int kCandWarps = kCandThreads / 32;
constexpr int kBatch = 16;        // values per thread per batch
constexpr int kCandCap = 512;     // listed candidates per CTA
constexpr int kMergeWarps = 8;    // warps that merge the queried rows
constexpr int kMaxSlices = 16;    // candidate slices per row
constexpr int kPickCap = 256;     // listed pick candidates
constexpr int K = TS_MAX_EXPAND;  // candidate slots stored per (row, slice) and per node

// (value, index) order of the candidate lists: larger value first, then the
// lower index
__device__ __forceinline__ bool ahead(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }
__device__ __forceinline__ bool ahead(int2 a, int2 b) { return ahead(__int_as_float(a.x), a.y, __int_as_float(b.x), b.y); }

// Floats as ints in the same order (for atomicMax on shared memory).
__device__ __forceinline__ int float_order(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float order_float(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

// The warp's 32 values in decreasing order (lane j holds the (j+1)-th
// largest): a bitonic sorting network over shuffles.
__device__ __forceinline__ float warp_sort_desc(float v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, j);
      v = (((lane & j) == 0) == ((lane & k) == 0)) ? fmaxf(v, o) : fminf(v, o);
    }
  return v;
}

// Inclusive prefix sum over the warp.
__device__ __forceinline__ int warp_incl_scan(int c, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, c, o);
    if (lane >= o) c += t;
  }
  return c;
}

// Warp arg-max in `ahead` order; every lane gets the winner.
__device__ __forceinline__ void warp_best(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ahead(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
}

// Log-sum-exp is kept as (max, sum of exp(x - max)) pairs and combined by a
// max reduction, then a sum of the pairs' sums rescaled to that max.
// __expf's error is a few ulp here: its argument is <= 0 and above -100 for
// finite logits of one distribution.

__device__ __forceinline__ int clamp_n(const ExpandParams& p, int b) {
  return min(max(p.n_tree[b], 0), p.n_tree_max);
}

// Phase 1 of a CTA: the k largest logits of its vocab slice of one queried
// row (ties: lower token) and the slice's (max, sum of exp), into `out`.
template <int KL>
__device__ __forceinline__ void slice_candidates(const ExpandParams& p, const float* lg, int v0, int v1,
                                                 CandPartial* out, int2* sbuf) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int2* cand = sbuf;              // [kCandCap]: (value bits, token)
  int2* elig = sbuf + kCandCap;   // [kCandCap]: the listed entries at or above the CTA's bound
  __shared__ int cnt_s, n_elig_s, bound_s;
  __shared__ float wm[kCandWarps], wsum[kCandWarps];
  __shared__ float red_v[kCandWarps];
  __shared__ int red_i[kCandWarps];
  if (tid == 0) {
    cnt_s = 0;
    n_elig_s = 0;
    bound_s = float_order(-INFINITY);
  }
  if (tid < KL) {  // slots the ranks below do not fill (a slice shorter than k)
    out->val[tid] = -INFINITY;
    out->idx[tid] = INT32_MAX;
  }
  __syncthreads();
  float m = -INFINITY, s = 0.f;
  float own = -INFINITY;  // warp-uniform: at most the warp's k-th largest value so far
  const bool vec = (p.vocab & 3) == 0;  // 16-byte rows; slices are multiples of 1024 floats
  for (int base = v0; base < v1; base += kBatch * kCandThreads) {
    float x[kBatch];
    int xi[kBatch];  // token, -1 past the slice
    if (vec) {
#pragma unroll
      for (int q = 0; q < kBatch / 4; ++q) {
        const int t = base + 4 * (q * kCandThreads + tid);
        const float4 f = t < v1 ? __ldcs(reinterpret_cast<const float4*>(lg + t))
                                : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        x[4 * q] = f.x;
        x[4 * q + 1] = f.y;
        x[4 * q + 2] = f.z;
        x[4 * q + 3] = f.w;
#pragma unroll
        for (int e = 0; e < 4; ++e) xi[4 * q + e] = t < v1 ? t + e : -1;
      }
    } else {
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int t = base + q * kCandThreads + tid;
        x[q] = t < v1 ? __ldcs(lg + t) : -INFINITY;
        xi[q] = t < v1 ? t : -1;
      }
    }
    // log-sum-exp: the batch max first, then independent exponentials
    float bm = -INFINITY;
#pragma unroll
    for (int q = 0; q < kBatch; ++q) bm = fmaxf(bm, x[q]);
    const float lane_max = bm;
    if (bm > m) {
      s *= __expf(m - bm);
      m = bm;
    }
    if (m > -INFINITY) {
      float es[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < kBatch; ++q) es[q & 3] += __expf(x[q] - m);  // -inf (past the slice) gives 0
      s += (es[0] + es[1]) + (es[2] + es[3]);
    }
    // the k-th largest lane maximum: k lanes hold a value at least that
    // large.  The warp publishes its own bound and filters with the largest
    // any warp has published (each bounds the CTA's k-th largest from below).
    own = fmaxf(own, __shfl_sync(0xffffffffu, warp_sort_desc(lane_max, lane), p.k - 1));
    int pub = 0;
    if (lane == 0) pub = atomicMax(&bound_s, float_order(own));
    const float bound = fmaxf(own, order_float(__shfl_sync(0xffffffffu, pub, 0)));
    int c = 0;
#pragma unroll
    for (int q = 0; q < kBatch; ++q) c += (xi[q] >= 0 && x[q] >= bound) ? 1 : 0;
    if (__any_sync(0xffffffffu, c > 0)) {
      const int incl = warp_incl_scan(c, lane);
      int pos = 0;
      if (lane == 31) pos = atomicAdd(&cnt_s, incl);
      pos = __shfl_sync(0xffffffffu, pos, 31) + incl - c;
#pragma unroll
      for (int q = 0; q < kBatch; ++q)
        if (xi[q] >= 0 && x[q] >= bound) {
          if (pos < kCandCap) cand[pos] = make_int2(__float_as_int(x[q]), xi[q]);
          ++pos;
        }
    }
  }
  {  // the warp's pair: the lanes' max, then their sums rescaled to it
    float mx = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sm = m != -INFINITY ? s * __expf(m - mx) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    if (lane == 0) {
      wm[warp] = mx;
      wsum[warp] = sm;
    }
  }
  __syncthreads();
  if (warp == 0) {  // the warps' pairs: their max, then the sums rescaled to it
    const float wmx = lane < kCandWarps ? wm[lane] : -INFINITY;
    float mx = wmx;
#pragma unroll
    for (int o = kCandWarps / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sm = (lane < kCandWarps && wmx != -INFINITY) ? wsum[lane] * __expf(wmx - mx) : 0.f;
#pragma unroll
    for (int o = kCandWarps / 2; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    if (lane == 0) {
      out->m = mx;
      out->s = sm;
    }
  }
  const int n_c = cnt_s;
  if (n_c <= kCandCap) {
    // Every value at or above the largest published bound B is listed (no
    // filter ever used more than B), and at least k are: an entry below B is
    // not among the k best.  Those at or above B are gathered, and the rank
    // of each among them (the number ahead of it) is its slot.
    const float bb = order_float(bound_s);
    for (int e0 = 0; e0 < n_c; e0 += kCandThreads) {  // uniform trip count
      const int e = e0 + tid;
      const int2 me = e < n_c ? cand[e] : make_int2(0, 0);
      const bool in = e < n_c && __int_as_float(me.x) >= bb;
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      int pos = 0;
      if (lane == 0 && bal != 0u) pos = atomicAdd(&n_elig_s, __popc(bal));
      pos = __shfl_sync(0xffffffffu, pos, 0) + __popc(bal & ((1u << lane) - 1u));
      if (in) elig[pos] = me;
    }
    __syncthreads();
    const int n_e = n_elig_s;
    // the rank of each entry is counted by g adjacent lanes (g a power of two
    // up to 32, as many as the CTA's threads allow), each over every g-th
    // entry, and summed by shuffles within the group
    int lg = 0;  // g = 1 << lg
    while (lg < 5 && (2 << lg) * n_e <= kCandThreads) ++lg;
    const int g = 1 << lg;
    for (int x0 = 0; x0 < n_e * g; x0 += kCandThreads) {  // uniform trip count
      const int x = x0 + tid, e = x >> lg, part = x & (g - 1);
      int2 me = make_int2(0, 0);
      int rank = 0;
      if (e < n_e) {
        me = elig[e];
        for (int j = part; j < n_e; j += g) rank += ahead(elig[j], me) ? 1 : 0;
      }
      for (int o = g >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
      if (e < n_e && part == 0 && rank < p.k) {
        out->val[rank] = __int_as_float(me.x);
        out->idx[rank] = me.y;
      }
    }
  } else {
    // heavy ties: k rounds, each the best value behind the previous winner
    float pv = INFINITY;
    int pi = -1;
    for (int r = 0; r < p.k; ++r) {
      float bv = -INFINITY;
      int bi = INT32_MAX;
      for (int t = v0 + tid; t < v1; t += kCandThreads) {
        const float x = lg[t];
        if (ahead(pv, pi, x, t) && ahead(x, t, bv, bi)) {
          bv = x;
          bi = t;
        }
      }
      warp_best(bv, bi);
      if (lane == 0) {
        red_v[warp] = bv;
        red_i[warp] = bi;
      }
      __syncthreads();
      bv = red_v[0];
      bi = red_i[0];
#pragma unroll
      for (int q = 1; q < kCandWarps; ++q)
        if (ahead(red_v[q], red_i[q], bv, bi)) {
          bv = red_v[q];
          bi = red_i[q];
        }
      __syncthreads();  // red_* is rewritten next round
      if (bi == INT32_MAX) break;
      if (tid == 0) {
        out->val[r] = bv;
        out->idx[r] = bi;
      }
      pv = bv;
      pi = bi;
    }
  }
}

// One queried row's slices, as one lane's share of a warp's merge: slice
// `lane`'s (max, sum) pair and its first k entries.
template <int KL>
struct RowSlices {
  float m, s;
  float val[KL];
  int idx[KL];
  __device__ __forceinline__ void load(const ExpandParams& p, int b, int r, int lane) {
    m = -INFINITY;
    s = 0.f;
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      val[j] = -INFINITY;
      idx[j] = INT32_MAX;
    }
    if (r < p.w && lane < p.num_slices) {
      const CandPartial* part = p.part + (static_cast<int64_t>(b) * p.w + r) * p.num_slices + lane;
      m = __ldcg(&part->m);
      s = __ldcg(&part->s);
#pragma unroll
      for (int j = 0; j < KL; ++j)
        if (j < p.k) {
          val[j] = __ldcg(&part->val[j]);
          idx[j] = __ldcg(&part->idx[j]);
        }
    }
  }
};

constexpr int kStepThreads = 256;  // one CTA per request: 8 warps merge rows; warp 0 picks

// Warp helpers of the step kernel, not inlined: the merge and the picks run
// the same copy, so the picks find it in the instruction cache (the step's
// code runs once per call, on one SM).
__device__ __noinline__ float step_sort_desc(float v, int lane) { return warp_sort_desc(v, lane); }
__device__ __noinline__ int step_scan(int c, int lane) { return warp_incl_scan(c, lane); }
__device__ __noinline__ int step_rank(const int2* list, int total, int2 me) {
  int rank = 0;
  for (int j = 0; j < total; ++j) rank += ahead(list[j], me) ? 1 : 0;
  return rank;
}

// The step, one CTA per request b: each queried node's k candidates from its
// row's slices (warp per row), then the step's w picks (warp 0), then the
// write-backs.  The tree state is requested before the wait for the
// candidate pass.
template <int KL>
__global__ void __launch_bounds__(kStepThreads) expand_step_kernel(const ExpandParams p) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nb = static_cast<int64_t>(b) * p.n_tree_max;
  __shared__ float c_lp[TS_MAX_TREE][KL];
  __shared__ int c_tok[TS_MAX_TREE][KL];
  __shared__ float key_s[TS_MAX_TREE][KL];
  __shared__ float w_s[TS_MAX_TREE];
  __shared__ int taken_s[TS_MAX_TREE];
  __shared__ int queried_s[TS_MAX_TREE];
  __shared__ int rows_s[K];
  __shared__ int2 mbuf[kMergeWarps][kMaxSlices * K];
  __shared__ int2 plist[kPickCap];
  __shared__ int4 pick_s[K];  // the step's new nodes: parent, token, weight bits
  __shared__ int n_out;
  // The tree state is final before this kernel starts: only step kernels
  // write it, and the candidate pass between them triggers this kernel only
  // after its own wait for the kernel before it.  Loads bypass L1; none
  // waits for n.
  int n = __ldcg(p.n_tree + b);
  if (tid < p.w) rows_s[tid] = __ldcg(p.rows + static_cast<int64_t>(b) * p.w + tid);
  if (tid < TS_MAX_TREE) {
    const int u = tid;
    float wv = -INFINITY;
    int tk = p.k;
    float lp[KL];
#pragma unroll
    for (int j = 0; j < KL; ++j) lp[j] = -INFINITY;
    if (u < p.n_tree_max) {
      wv = __ldcg(p.weight + nb + u);
      tk = __ldcg(p.cand_taken + nb + u);
#pragma unroll
      for (int j = 0; j < KL; ++j)
        if (j < p.k) lp[j] = __ldcg(p.cand_lp + (nb + u) * p.k + j);
    }
    if (n < 0 || n > p.n_tree_max) {
      if (tid == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);
      n = min(max(n, 0), p.n_tree_max);
    }
    queried_s[u] = 0;
    w_s[u] = u < n ? wv : -INFINITY;
    taken_s[u] = u < n ? min(max(tk, 0), p.k) : p.k;
#pragma unroll
    for (int j = 0; j < KL; ++j) c_lp[u][j] = lp[j];
  } else if (tid < 2 * TS_MAX_TREE) {
    const int u = tid - TS_MAX_TREE;
    int tk[KL];
#pragma unroll
    for (int j = 0; j < KL; ++j) tk[j] = -1;
    if (u < p.n_tree_max) {
#pragma unroll
      for (int j = 0; j < KL; ++j)
        if (j < p.k) tk[j] = __ldcg(p.cand_tok + (nb + u) * p.k + j);
    }
#pragma unroll
    for (int j = 0; j < KL; ++j) c_tok[u][j] = tk[j];
  }
  n = min(max(n, 0), p.n_tree_max);
  pdl_launch_dependents();
  pdl_wait();  // the candidate partials
  RowSlices<KL> rs;
  if (warp < kMergeWarps) rs.load(p, b, warp, lane);
  __syncthreads();
  // ---- 1. the queried rows: merge the slices into k candidates (warp per row)
  if (warp < kMergeWarps) {
    for (int r = warp; r < p.w; r += kMergeWarps) {
      if (r != warp) rs.load(p, b, r, lane);
      const int u = rows_s[r];
      if (u < 0) continue;
      if (u >= n) {
        if (lane == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);
        continue;
      }
      if (lane < p.k) {
        c_lp[u][lane] = -INFINITY;
        c_tok[u][lane] = -1;
      }
      // the row's log-sum-exp from the slices' pairs: their max, then the
      // sums rescaled to it
      float m = rs.m;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float s = rs.m != -INFINITY ? rs.s * __expf(rs.m - m) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const float lse = m + logf(s);
      // Lower bounds of the row's k-th largest: any slice's k-th entry (the
      // least of its first k), and the k-th largest of the slices' heads.
      // Only a slice's first k entries can be among the row's k best.
      float kth = INFINITY;
#pragma unroll
      for (int j = 0; j < KL; ++j)
        if (j < p.k) kth = fminf(kth, rs.val[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) kth = fmaxf(kth, __shfl_xor_sync(0xffffffffu, kth, o));
      kth = fmaxf(kth, __shfl_sync(0xffffffffu, step_sort_desc(rs.val[0], lane), p.k - 1));
      int c = 0;
#pragma unroll
      for (int j = 0; j < KL; ++j) c += (j < p.k && rs.idx[j] != INT32_MAX && rs.val[j] >= kth) ? 1 : 0;
      const int incl = step_scan(c, lane);
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      int pos = incl - c;
#pragma unroll
      for (int j = 0; j < KL; ++j)
        if (j < p.k && rs.idx[j] != INT32_MAX && rs.val[j] >= kth)
          mbuf[warp][pos++] = make_int2(__float_as_int(rs.val[j]), rs.idx[j]);
      __syncwarp();
      for (int e = lane; e < total; e += 32) {
        const int2 me = mbuf[warp][e];
        const float v = __int_as_float(me.x);
        const int rank = step_rank(mbuf[warp], total, me);
        if (rank < p.k && v != -INFINITY) {
          c_lp[u][rank] = v - lse;
          c_tok[u][rank] = me.y;
        }
      }
      if (lane == 0) {
        taken_s[u] = 0;
        queried_s[u] = 1;
      }
      __syncwarp();  // mbuf is reused by the warp's next row
    }
  }
  __syncthreads();
  // keys of every node's slots: weight + log-prob, -inf where no candidate
  for (int i = tid; i < TS_MAX_TREE * KL; i += kStepThreads) {
    const int v = i / KL, t = i % KL;
    key_s[v][t] = (v < n && t < p.k && c_tok[v][t] >= 0) ? w_s[v] + c_lp[v][t] : -INFINITY;
  }
  __syncthreads();
  // ---- 2. the picks (warp 0).  Each node offers its untaken candidates in
  // order, with keys weight + log-prob that never increase, so the w picks
  // are the w largest keys over all offered slots (ties: lower node, then
  // earlier slot).  Lane l holds nodes l, l + 32, l + 64, l + 96.
  if (warp == 0) {
    constexpr int kPer = TS_MAX_TREE / 32;
    int t0[kPer];
    float lane_head = -INFINITY, wth = -INFINITY;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int v = lane + 32 * q;
      t0[q] = taken_s[v];
      if (t0[q] < KL) lane_head = fmaxf(lane_head, key_s[v][t0[q]]);
      if (t0[q] + p.w - 1 < KL) wth = fmaxf(wth, key_s[v][t0[q] + p.w - 1]);
    }
    // B: w offered slots have a key at least B (w lanes' best heads, or one
    // node's first w); every slot at or above B is listed
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wth = fmaxf(wth, __shfl_xor_sync(0xffffffffu, wth, o));
    const float bb = fmaxf(wth, __shfl_sync(0xffffffffu, step_sort_desc(lane_head, lane), p.w - 1));
    int cq[kPer], c = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int v = lane + 32 * q;
      int t = t0[q];
      while (t < KL && key_s[v][t] >= bb && key_s[v][t] > -INFINITY) ++t;
      cq[q] = t - t0[q];
      c += cq[q];
    }
    const int incl = step_scan(c, lane);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int nn = n;
    if (total <= kPickCap) {
      int pos = incl - c;
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int v = lane + 32 * q;
        for (int i = 0; i < cq[q]; ++i) plist[pos++] = make_int2(__float_as_int(key_s[v][t0[q] + i]), v * K + t0[q] + i);
      }
      __syncwarp();
      const int npick = min(min(p.w, p.n_tree_max - n), total);
      for (int e = lane; e < total; e += 32) {
        const int2 me = plist[e];
        const int rank = step_rank(plist, total, me);
        if (rank < npick) {
          const int v = me.y / K, t = me.y % K;
          pick_s[rank] = make_int4(v, c_tok[v][t], me.x, 0);
          atomicMax(&taken_s[v], t + 1);
        }
      }
      nn = n + npick;
    } else {
      // many equal keys: the picks one at a time, each a warp arg-max over
      // the nodes' next candidates
      float key[kPer];
      int tk[kPer];
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        tk[q] = t0[q];
        key[q] = tk[q] < KL ? key_s[lane + 32 * q][tk[q]] : -INFINITY;
      }
      int j = 0;
      for (; j < p.w && nn < p.n_tree_max; ++j) {
        float bv = key[0];
        int bi = lane;
#pragma unroll
        for (int q = 1; q < kPer; ++q)
          if (key[q] > bv) {  // a tie keeps the lower node
            bv = key[q];
            bi = lane + 32 * q;
          }
        warp_best(bv, bi);
        if (bv == -INFINITY) break;
#pragma unroll
        for (int q = 0; q < kPer; ++q)
          if (lane + 32 * q == bi) {
            const int t = tk[q];
            pick_s[j] = make_int4(bi, c_tok[bi][t], __float_as_int(bv), 0);
            tk[q] = t + 1;
            key[q] = t + 1 < KL ? key_s[bi][t + 1] : -INFINITY;
          }
        ++nn;  // the new node: no candidates until its logits come (its key stays -inf)
      }
#pragma unroll
      for (int q = 0; q < kPer; ++q) taken_s[lane + 32 * q] = tk[q];
    }
    if (lane == 0) n_out = nn;
  }
  __syncthreads();
  // ---- 3. write back the new nodes, the queried rows' candidates and the
  // old nodes' taken counts
  const int n_new = n_out - n;
  if (tid < p.w) {
    p.added[static_cast<int64_t>(b) * p.w + tid] = tid < n_new ? n + tid : -1;
    if (tid < n_new) {
      const int4 pk = pick_s[tid];
      p.parent[nb + n + tid] = pk.x;
      p.tokens[nb + n + tid] = pk.y;
      p.weight[nb + n + tid] = __int_as_float(pk.z);
      p.cand_taken[nb + n + tid] = p.k;
    }
  }
  if (tid < n) {
    p.cand_taken[nb + tid] = taken_s[tid];
    if (queried_s[tid])
      for (int j = 0; j < p.k; ++j) {
        p.cand_lp[(nb + tid) * p.k + j] = c_lp[tid][j];
        p.cand_tok[(nb + tid) * p.k + j] = c_tok[tid][j];
      }
  }
  if (tid == 0) p.n_tree[b] = n_out;
}

// The candidate pass: CTA (b * w + r, slice) takes its slice of row r
// (nothing if the row queries no node; the step kernel skips it too).
template <int KL>  // slots written per partial: the smallest of 8, 16 that holds k
__global__ void __launch_bounds__(kCandThreads, 1) cand_partial_kernel(const ExpandParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x;  // b * w + r
  const int b = row / p.w;
  const int u = p.rows[row];
  if (u < 0 || u >= clamp_n(p, b)) return;
  __shared__ int2 sbuf[2 * kCandCap];
  const int v0 = blockIdx.y * p.slice;
  slice_candidates<KL>(p, p.logits + static_cast<int64_t>(row) * p.vocab, v0, min(p.vocab, v0 + p.slice),
                       p.part + static_cast<int64_t>(row) * p.num_slices + blockIdx.y, sbuf);
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
