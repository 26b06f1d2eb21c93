// Pieces shared by the two tree-attention kernels and their merge.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace ts {

// A pipeline wait: the default bound, or (the bounded-wait variant, when the
// call gives its own bound) that bound; waits that drain copies in flight
// after an abort always take the default bound.  Most pipeline waits find
// their phase already complete, so the default instance first tests it once
// without blocking: entering the try_wait loop costs the issuing warps even
// then (the long-context call: 99.2 -> 95.1 us warm on one GB300).
template <bool kBounded>
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if constexpr (kBounded) return mbar_wait_bounded(bar, parity, limit_ns);
  else return mbar_test(bar, parity) || mbar_wait(bar, parity);
}

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

// RoPE at a tree position (SwiftSpec summary §3.3: RoPE inside the verify
// attention, position = prefix length + depth).  Pair j of a query at
// position pos turns by pos * theta^(-2j/d) rad.  The host gives each
// frequency as a 64-bit fraction of a turn (theta^(-2j/d) / 2 pi * 2^64), so
// pos times it modulo 2^64 is the angle's fractional turn, exact up to that
// fraction's rounding (far below 1e-9 rad at any int32 position).  Its top 32
// bits read as a signed fraction give the angle in [-pi, pi), where the fast
// sine and cosine are accurate to about 2^-21, well below the bf16 rounding
// of the rotated query.
__device__ __forceinline__ void rope_cos_sin(int pos, uint64_t turn_frac, float& c, float& s) {
  const uint64_t t = static_cast<uint64_t>(static_cast<uint32_t>(pos)) * turn_frac;  // modulo 2^64
  const float a = static_cast<float>(static_cast<int32_t>(t >> 32)) * 1.4629180792671596e-09f;  // 2 pi / 2^32
  __sincosf(a, &s, &c);
}

// Rotate-half RoPE of 8 pairs held as two 16-byte chunks of bf16: x_j (chunk
// a, column j of the first half) and x_{j + d/2} (chunk b); pair e of the
// chunks is frequency j0 + e (turn_frac in shared or parameter memory).
__device__ __forceinline__ void rope_rotate8(uint4& a, uint4& b, int pos, const uint64_t* turn_frac, int j0) {
  __nv_bfloat16* a8 = reinterpret_cast<__nv_bfloat16*>(&a);
  __nv_bfloat16* b8 = reinterpret_cast<__nv_bfloat16*>(&b);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float c, s;
    rope_cos_sin(pos, turn_frac[j0 + e], c, s);
    const float x0 = __bfloat162float(a8[e]), x1 = __bfloat162float(b8[e]);
    a8[e] = __float2bfloat16_rn(x0 * c - x1 * s);
    b8[e] = __float2bfloat16_rn(x0 * s + x1 * c);
  }
}

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

// The CTAs holding tiles of one unit under the split of the tile sequence
// (plain when E = 0, cost-weighted with a first-tile weight of 1 + E
// otherwise): CTA c left a share of the unit iff c_lo <= c <= c_hi and
// holds(c).  before = tiles of earlier requests, T = all tiles, tiles = tiles
// of every unit of request b, upr = units per request, nc = CTAs.
struct UnitSplit {
  int64_t T, W, pf;
  int E, tiles, nc, c_lo, c_hi;
  __device__ __forceinline__ void init(int64_t before, int64_t T_, int tiles_, int b, int uir, int upr, int num_req,
                                       int E_, int nc_) {
    T = T_;
    tiles = tiles_;
    E = E_;
    nc = nc_;
    W = T + static_cast<int64_t>(E) * upr * num_req;
    pf = before + static_cast<int64_t>(E) * upr * b + static_cast<int64_t>(uir) * (tiles + E);
    const int64_t first = before + static_cast<int64_t>(uir) * tiles;
    c_lo = E > 0 ? wsched_cta_of_pos(pf, W, nc) : sched_cta_of(first, T, nc);
    c_hi = E > 0 ? wsched_cta_of_pos(pf + (tiles >= 2 ? E + tiles - 1 : 0), W, nc)
                 : sched_cta_of(first + tiles - 1, T, nc);
  }
  __device__ __forceinline__ bool holds(int c) const {
    if (E == 0) return sched_begin(c, T, nc) < sched_begin(c + 1, T, nc);
    if (c == c_lo) return true;
    const int j = wsched_tile_in_unit(wsched_x(c, W, nc) - pf, E, tiles);
    return j < tiles && wsched_cta_of_pos(pf + E + j, W, nc) == c;
  }
};

}  // namespace ts
