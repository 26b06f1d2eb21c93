// Pieces shared by the two tree-attention kernels and their merge.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace ts {

// Per-request lengths, clamped to the stated bounds (violations reported).
// Every kernel of one call clamps the same way, so they agree on the schedule.
__device__ __forceinline__ void attn_lengths(const AttnParams& p, int b, int& P, int& n, bool report) {
  P = p.prefix_len[b];
  n = p.n_tree[b];
  bool bad = false;
  if (n < p.n_query) { n = p.n_query; bad = true; }
  if (n > p.n_tree_max) { n = p.n_tree_max; bad = true; }
  const int cap = p.paged ? p.max_blocks * p.page_size : p.max_kv_len;
  if (P < 0) { P = 0; bad = true; }
  if (P > cap - n) { P = max(cap - n, 0); bad = true; }
  if (bad && report) report_error(p.err, TS_DEVERR_BAD_LENGTH);
}

// Ancestor-or-self set of node u (bit j = node j) by walking a validated
// parent array (parent[i] in [-1, i)) held in shared memory.
__device__ __forceinline__ void ancestor_walk(const int* par, int u, uint32_t a[4]) {
  uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  while (u >= 0) {
    const uint32_t bit = 1u << (u & 31);
    const int w = u >> 5;
    a0 |= (w == 0) ? bit : 0u;
    a1 |= (w == 1) ? bit : 0u;
    a2 |= (w == 2) ? bit : 0u;
    a3 |= (w == 3) ? bit : 0u;
    u = par[u];
  }
  a[0] = a0;
  a[1] = a1;
  a[2] = a2;
  a[3] = a3;
}

__device__ __forceinline__ int attn_tiles(int keys) { return (keys + kBlockN - 1) / kBlockN; }

// Visibility of the 64 keys [P + off, P + off + 64) for a query whose
// ancestor-or-self set is `a` (bit j = tree node j): prefix keys (negative
// offsets) are visible; tree key j is visible iff bit j is set; keys at or
// beyond P + n are never visible (their bits are zero in `a`).
__device__ __forceinline__ uint64_t tile_visibility(const uint32_t a[4], int off) {
  const uint64_t lo = static_cast<uint64_t>(a[0]) | (static_cast<uint64_t>(a[1]) << 32);
  const uint64_t hi = static_cast<uint64_t>(a[2]) | (static_cast<uint64_t>(a[3]) << 32);
  uint64_t tree;
  if (off >= 128 || off <= -64) tree = 0;
  else if (off >= 64) tree = hi >> (off - 64);
  else if (off > 0) tree = (lo >> off) | (hi << (64 - off));
  else if (off == 0) tree = lo;
  else tree = lo << (-off);
  uint64_t pre = 0;
  if (off < 0) pre = (off <= -64) ? ~0ull : ((1ull << (-off)) - 1ull);
  return tree | pre;
}

// ---------------------------------------------------------------- split-KV combine
// A unit whose tiles several CTAs share is combined by the CTA that finishes
// its share last (SwiftSpec summary §3.3: the partial results of a head split
// across thread blocks are combined without a second pass).  Every CTA with
// a partial of the unit fences its partial stores and increments the unit's
// counter; the one that brings it to the number of contributing CTAs merges
// all partials and resets the counter to zero for the next call.

// Number of CTAs with a non-empty tile range in [c_lo, c_hi].
__device__ __forceinline__ int split_contributors(int64_t T, int NC, int c_lo, int c_hi) {
  int k = 0;
  for (int c = c_lo; c <= c_hi; ++c) k += sched_begin(c, T, NC) < sched_begin(c + 1, T, NC) ? 1 : 0;
  return k;
}

// Called by all `nthr` threads of the group that wrote this CTA's partial of
// `unit` (tiles [first, first + tiles) of the global sequence), after a
// barrier over that group; returns true in every thread of the group when
// this CTA is the last contributor.  `flag` is one int of shared memory.
template <class Sync>
__device__ __forceinline__ bool split_arrive(const AttnParams& p, int64_t unit, int64_t T, int64_t first, int tiles,
                                             int tid, volatile int* flag, Sync sync) {
  sync();
  if (tid == 0) {
    const int c_lo = sched_cta_of(first, T, p.num_ctas);
    const int c_hi = sched_cta_of(first + tiles - 1, T, p.num_ctas);
    const int expected = split_contributors(T, p.num_ctas, c_lo, c_hi);
    __threadfence();
    const int old = atomicAdd(&p.counters[unit], 1);
    const bool last = (old == expected - 1);
    if (last) p.counters[unit] = 0;
    *flag = last ? 1 : 0;
  }
  sync();
  const bool last = *flag != 0;
  if (last) __threadfence();
  return last;
}

// Merge every partial of `unit` (rows [0, rows_here) of row group rg) and
// write the bf16 output and the natural-log lse:
//   O = sum_s w_s O_s,  w_s = 2^(lse_s - lse),  lse = log2 sum_s 2^lse_s
// over the CTAs with a non-empty range in [c_lo, c_hi].  `nthr` threads of
// the calling group take part (tid in [0, nthr), nthr >= rows_here, whole
// warps); `sync` is a barrier over them.  `wbuf` is free shared memory of
// `wbuf_floats` floats: the slot list and the weights w_s per row.  Phase 1
// gives each row to one thread (independent loads of the partial lse's);
// phase 2 gives each row to one warp, whose lanes stream the partial rows
// with 16-byte loads.  Units split over more CTAs than `wbuf` holds weights
// for fall back to a row-at-a-time loop.
template <class Sync>
__device__ __forceinline__ void merge_unit_rows(const AttnParams& p, int64_t unit, int b, int kvh, int rg, int64_t T,
                                                int64_t first, int tiles, int tid, int nthr, float* wbuf,
                                                int wbuf_floats, Sync sync) {
  const int c_lo = sched_cta_of(first, T, p.num_ctas);
  const int c_hi = sched_cta_of(first + tiles - 1, T, p.num_ctas);
  const int D = p.head_dim;
  const int rows_here = min(kMaxRowsPerUnit, p.rows - rg * kMaxRowsPerUnit);
  constexpr int kMaxList = 32;
  int* slots = reinterpret_cast<int*>(wbuf);        // [kMaxList] contributing CTAs, then their count
  float* w = wbuf + kMaxList + 4;                   // [slot][kMaxRowsPerUnit] weights
  const int cap = min(kMaxList, (wbuf_floats - kMaxList - 4) / kMaxRowsPerUnit);
  if (tid == 0) {
    int k = 0;
    for (int c = c_lo; c <= c_hi; ++c)
      if (sched_begin(c, T, p.num_ctas) < sched_begin(c + 1, T, p.num_ctas)) {
        if (k < cap) slots[k] = c;
        ++k;
      }
    slots[kMaxList] = k;
  }
  sync();
  const int ns = slots[kMaxList];
  const int warp = tid / 32, lane = tid % 32, nwarps = nthr / 32;
  const float ln2 = 0.69314718055994530942f;
  if (ns <= cap) {
    // phase 1: weights of every slot for row tid
    if (tid < rows_here) {
      float mx = -INFINITY;
      for (int k = 0; k < ns; ++k) {
        const float v = __ldcg(p.part_lse + (slots[k] + unit) * p.rows_pad + tid);
        w[k * kMaxRowsPerUnit + tid] = v;
        mx = fmaxf(mx, v);
      }
      const float base = (mx == -INFINITY) ? 0.f : mx;
      float sum = 0.f;
      for (int k = 0; k < ns; ++k) {
        const float e = exp2f(w[k * kMaxRowsPerUnit + tid] - base);
        w[k * kMaxRowsPerUnit + tid] = e;
        sum += e;
      }
      const float inv = sum > 0.f ? __frcp_rn(sum) : 0.f;
      for (int k = 0; k < ns; ++k) w[k * kMaxRowsPerUnit + tid] *= inv;
      if (p.lse != nullptr) {
        const int r = rg * kMaxRowsPerUnit + tid;
        const int i = r / p.group, h = kvh * p.group + r % p.group;
        p.lse[(static_cast<int64_t>(b) * p.hq + h) * p.n_query + i] = (base + log2f(sum)) * ln2;
      }
    }
    sync();
    // phase 2: one row per warp, lanes over the head dim in float4s
    const int nvec = D / 4;
    for (int rl = warp; rl < rows_here; rl += nwarps) {
      if (lane < nvec) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < ns; ++k) {
          const float wk = w[k * kMaxRowsPerUnit + rl];
          const float4 v = __ldcg(reinterpret_cast<const float4*>(
                                      p.part_o + ((slots[k] + unit) * p.rows_pad + rl) * D) + lane);
          acc.x += wk * v.x;
          acc.y += wk * v.y;
          acc.z += wk * v.z;
          acc.w += wk * v.w;
        }
        const int r = rg * kMaxRowsPerUnit + rl;
        const int i = r / p.group, h = kvh * p.group + r % p.group;
        __nv_bfloat16* orow = p.out + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * D;
        *reinterpret_cast<uint2*>(orow + 4 * lane) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
      }
    }
  } else {
    for (int rl = warp; rl < rows_here; rl += nwarps) {
      float mx = -INFINITY;
      for (int c = c_lo; c <= c_hi; ++c)
        if (sched_begin(c, T, p.num_ctas) < sched_begin(c + 1, T, p.num_ctas))
          mx = fmaxf(mx, __ldcg(p.part_lse + (c + unit) * p.rows_pad + rl));
      const float base = (mx == -INFINITY) ? 0.f : mx;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      float wsum = 0.f;
      for (int c = c_lo; c <= c_hi; ++c) {
        if (sched_begin(c, T, p.num_ctas) == sched_begin(c + 1, T, p.num_ctas)) continue;
        const int64_t slot = c + unit;
        const float wk = exp2f(__ldcg(p.part_lse + slot * p.rows_pad + rl) - base);
        wsum += wk;
        const float* po = p.part_o + (slot * p.rows_pad + rl) * D;
        for (int j = 0; j < D / 32; ++j) acc[j] += wk * __ldcg(po + lane + 32 * j);
      }
      const float inv = wsum > 0.f ? __frcp_rn(wsum) : 0.f;
      const int r = rg * kMaxRowsPerUnit + rl;
      const int i = r / p.group, h = kvh * p.group + r % p.group;
      __nv_bfloat16* orow = p.out + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * D;
      for (int j = 0; j < D / 32; ++j) orow[lane + 32 * j] = __float2bfloat16_rn(acc[j] * inv);
      if (p.lse != nullptr && lane == 0)
        p.lse[(static_cast<int64_t>(b) * p.hq + h) * p.n_query + i] = (base + log2f(wsum)) * ln2;
    }
  }
  sync();  // wbuf is free again
}

}  // namespace ts
