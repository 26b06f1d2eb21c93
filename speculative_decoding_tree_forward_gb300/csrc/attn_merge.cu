// Split-KV combine: SwiftSpec summary §3.3 (a head is split across thread
// blocks and their partial results are combined).
//
// A unit (request, KV head, row group) whose tiles several CTAs shared left
// one normalised fp32 partial O_s and its log2-sum-exp lse_s per CTA.  This
// kernel combines them,
//   O = sum_s 2^(lse_s - lse) O_s,   lse = log2 sum_s 2^lse_s,
// skipping CTAs whose tile range was empty, and writes the bf16 output and
// the natural-log lse.  Units held by one CTA were written directly by the
// attention kernel and are skipped here.  The split (which CTAs hold tiles
// of the unit) follows from the request lengths alone, so it is worked out
// before the kernel waits for the attention kernel's results.  After the
// wait the lse of a row's first shares (one per lane) and its first few
// partial rows (coalesced reads) are all requested before the weights are
// known, so a row with up to that many shares costs one round trip to L2;
// shares of CTAs that hold no tile of the unit get weight 0.
//
// The warp-MMA kernel's partials are row-major ([slot][row][head_dim]); two
// shapes, picked by the host, merge them: one warp per row with eight shares
// prefetched (when that grid fits one resident wave of CTAs: many shares per
// row, few rows), or one half-warp per row with four prefetched (twice the
// rows in flight for the same registers, so a grid of many rows lands in
// one wave instead of two).  The tcgen05 kernel's partials are column-blocked
// (float4 j of row r at (slot * 32 + j) * 128 + r) and merged with one thread
// per (row, 16 columns, group of shares).
#include "attn_common.cuh"

namespace ts {
namespace {

constexpr int kMergeWarps = 8;
constexpr int kPrefetchWarp = 8;              // warp per row: partial rows loaded before the weights are known
constexpr int kRowsPerCtaHalf = 2 * kMergeWarps;  // half-warp per row
constexpr int kPrefetchHalf = 4;              // half-warp per row: partial rows loaded before the weights are known
constexpr int kMaxVec = 2;                    // half-warp per row: float4 per lane of one partial row (head_dim 128)

// The split as the attention kernel laid it out, from the request lengths it
// read (clamped the same way).  They were final before the attention kernel
// passed its own wait, which precedes the merge grid's launch, so warp 0 of a
// merge CTA works the split out for the CTA's unit before the wait for the
// attention kernel's results: the CTAs holding tiles of the unit and, for the
// first 32 of them, which hold a share (bit i of *hold: CTA c_lo + i).
__device__ __forceinline__ void merge_split(const AttnParams& p, int b, int uir, int units_per_req, int lane,
                                            UnitSplit* sp, unsigned* hold) {
  int64_t before = 0, total = 0;
  int mine = 0;
  for (int r = lane; r < p.num_req; r += 32) {
    int P, n;
    attn_lengths(p, r, P, n, false);
    const int t = attn_tiles(P + n);
    total += static_cast<int64_t>(t) * units_per_req;
    if (r < b) before += static_cast<int64_t>(t) * units_per_req;
    if (r == b) mine = t;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
    mine = max(mine, __shfl_xor_sync(0xffffffffu, mine, o));
  }
  if (lane == 0) sp->init(before, total, mine, b, uir, units_per_req, p.num_req, p.seg_cost, p.num_ctas);
  __syncwarp();
  const int c = sp->c_lo + lane;
  const unsigned h = __ballot_sync(0xffffffffu, c <= sp->c_hi && sp->c_lo != sp->c_hi && sp->holds(c));
  if (lane == 0) *hold = h;
}

// One warp per output row, eight rows per CTA, each lane owning four
// columns; the first kPrefetchWarp shares of a row are prefetched.  At most
// 64 registers: four CTAs (32 warps) per SM.
__global__ void __launch_bounds__(kMergeWarps * 32, 4) merge_row_per_warp_kernel(const AttnParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t unit = blockIdx.x;
  // a unit is (request, group of hp KV heads, row group); with hp = 2 the
  // unit's rows are two heads' R <= 64 rows at 0 and 64
  const int units_per_req = (p.hkv / p.hp) * p.row_groups;
  const int b = static_cast<int>(blockIdx.x) / units_per_req;
  const int uir = static_cast<int>(blockIdx.x) % units_per_req;
  const int kvh = uir / p.row_groups;  // head group
  const int rg = uir % p.row_groups;
  const int rl = blockIdx.y * kMergeWarps + warp;
  const int hj = p.hp == 2 ? rl >> 6 : 0, loc = p.hp == 2 ? rl & 63 : rl;
  const bool row_valid = p.hp == 2 ? loc < p.rows : rl < min(kMaxRowsPerUnit, p.rows - rg * kMaxRowsPerUnit);
  __shared__ UnitSplit s_sp;
  __shared__ unsigned s_hold;
  if (warp == 0) merge_split(p, b, uir, units_per_req, lane, &s_sp, &s_hold);
  __syncthreads();
  const int c_lo = s_sp.c_lo, c_hi = s_sp.c_hi;
  const bool valid_l = (s_hold >> lane) & 1u;
  pdl_wait();
  pdl_launch_dependents();
  if (!row_valid || c_lo == c_hi) return;  // padding row, or one CTA held the whole unit and wrote it
  auto holds = [&](int c) -> bool { return s_sp.holds(c); };

  // slot of CTA c: c + unit; its lse at part_lse[slot * rows_pad + row]
  const float* lse_col = p.part_lse + unit * p.rows_pad + rl;
  const int D = p.head_dim;
  const bool active = lane * 4 < D;
  auto part_row = [&](int c) {
    return reinterpret_cast<const float4*>(p.part_o + ((static_cast<int64_t>(c) + unit) * p.rows_pad + rl) * D +
                                           lane * 4);
  };
  // one round trip: the lse of the first 32 slots (one per lane) and the
  // partial rows of the first kPrefetchWarp slots, all issued before the
  // weights are known (slots of CTAs without a share get weight 0)
  const unsigned hold = s_hold;
  float lse_l = -INFINITY;
  if (valid_l) lse_l = __ldcg(lse_col + static_cast<int64_t>(c_lo + lane) * p.rows_pad);
  float4 x[kPrefetchWarp];
#pragma unroll
  for (int q = 0; q < kPrefetchWarp; ++q) {
    x[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (((hold >> q) & 1u) && active) x[q] = __ldcg(part_row(c_lo + q));
  }
  float mx = valid_l ? lse_l : -INFINITY;
  for (int c0 = c_lo + 32; c0 <= c_hi; c0 += 32) {  // more than 32 shares: rare
    const int c = c0 + lane;
    if (c <= c_hi && holds(c)) mx = fmaxf(mx, __ldcg(lse_col + static_cast<int64_t>(c) * p.rows_pad));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float mbase = (mx == -INFINITY) ? 0.f : mx;

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wl = valid_l ? exp2f(lse_l - mbase) : 0.f;
  float wsum = wl;
#pragma unroll
  for (int q = 0; q < kPrefetchWarp; ++q) {
    const float wq = __shfl_sync(0xffffffffu, wl, q);
    acc.x += wq * x[q].x;
    acc.y += wq * x[q].y;
    acc.z += wq * x[q].z;
    acc.w += wq * x[q].w;
  }
  // slots kPrefetchWarp .. 31 of the first chunk, then further chunks of 32
  for (int c0 = c_lo; c0 <= c_hi; c0 += 32) {
    float wc = wl;
    if (c0 != c_lo) {
      const int c = c0 + lane;
      const bool v = c <= c_hi && holds(c);
      wc = v ? exp2f(__ldcg(lse_col + static_cast<int64_t>(c) * p.rows_pad) - mbase) : 0.f;
      wsum += wc;
    }
    const int q0 = c0 == c_lo ? kPrefetchWarp : 0;
    for (int q = q0; q < 32 && c0 + q <= c_hi; q += 4) {  // warp-uniform bounds
      float w4[4];
      float4 y[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool in = q + u < 32 && c0 + q + u <= c_hi;
        w4[u] = __shfl_sync(0xffffffffu, wc, in ? q + u : 0);
        if (!in) w4[u] = 0.f;
        y[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in && w4[u] != 0.f && active) y[u] = __ldcg(part_row(c0 + q + u));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc.x += w4[u] * y[u].x;
        acc.y += w4[u] * y[u].y;
        acc.z += w4[u] * y[u].z;
        acc.w += w4[u] * y[u].w;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  const float inv = wsum > 0.f ? __frcp_rn(wsum) : 0.f;
  const int r = rg * kMaxRowsPerUnit + loc;
  const int i = r / p.group, h = (p.hp * kvh + hj) * p.group + r % p.group;
  if (active) {
    uint2* dst = reinterpret_cast<uint2*>(p.out + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * D + lane * 4);
    *dst = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  }
  if (p.lse != nullptr && lane == 0)
    p.lse[(static_cast<int64_t>(b) * p.hq + h) * p.n_query + i] = (mbase + log2f(wsum)) * 0.69314718055994530942f;
}

// One half-warp per output row, 16 rows per CTA, each of its 16 lanes
// owning head_dim / 16 columns; the first kPrefetchHalf shares of a row are
// prefetched.  At most 64 registers: four CTAs (32 warps, 64 rows) per SM.
__global__ void __launch_bounds__(kMergeWarps * 32, 4) merge_row_per_half_warp_kernel(const AttnParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;  // the row of this half-warp, the lane within it
  const int64_t unit = blockIdx.x;
  // a unit is (request, group of hp KV heads, row group); with hp = 2 the
  // unit's rows are two heads' R <= 64 rows at 0 and 64
  const int units_per_req = (p.hkv / p.hp) * p.row_groups;
  const int b = static_cast<int>(blockIdx.x) / units_per_req;
  const int uir = static_cast<int>(blockIdx.x) % units_per_req;
  const int kvh = uir / p.row_groups;  // head group
  const int rg = uir % p.row_groups;
  const int rl = blockIdx.y * kRowsPerCtaHalf + warp * 2 + half;
  const int hj = p.hp == 2 ? rl >> 6 : 0, loc = p.hp == 2 ? rl & 63 : rl;
  const bool row_valid = p.hp == 2 ? loc < p.rows : rl < min(kMaxRowsPerUnit, p.rows - rg * kMaxRowsPerUnit);
  __shared__ UnitSplit s_sp;
  __shared__ unsigned s_hold;
  if (warp == 0) merge_split(p, b, uir, units_per_req, lane, &s_sp, &s_hold);
  __syncthreads();
  const int c_lo = s_sp.c_lo, c_hi = s_sp.c_hi;
  const unsigned hold = s_hold;
  const bool valid_l = row_valid && ((hold >> hl) & 1u);  // this lane's share of the first 16
  pdl_wait();
  pdl_launch_dependents();
  // padding rows (both halves), or one CTA held the whole unit and wrote it
  if (!__any_sync(0xffffffffu, row_valid) || c_lo == c_hi) return;
  auto holds = [&](int c) -> bool { return s_sp.holds(c); };
  const int D = p.head_dim;
  const int nv = D >> 6;  // float4 per lane: 1 (head_dim 64) or 2 (128)
  const int col = hl * (D >> 4);
  // slot of CTA c: c + unit; its lse at part_lse[slot * rows_pad + row]
  const float* lse_col = p.part_lse + unit * p.rows_pad + rl;
  auto part_row = [&](int c) {
    return reinterpret_cast<const float4*>(p.part_o + ((static_cast<int64_t>(c) + unit) * p.rows_pad + rl) * D + col);
  };
  const int hbase = half * 16;

  // one round trip: the lse of the first 16 slots (one per lane of the half)
  // and the partial rows of the first kPrefetchHalf slots, all issued before the
  // weights are known (slots of CTAs without a share get weight 0)
  float lse_l = -INFINITY;
  if (valid_l) lse_l = __ldcg(lse_col + static_cast<int64_t>(c_lo + hl) * p.rows_pad);
  float4 x[kPrefetchHalf][kMaxVec];
#pragma unroll
  for (int q = 0; q < kPrefetchHalf; ++q)
#pragma unroll
    for (int v = 0; v < kMaxVec; ++v) {
      x[q][v] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row_valid && ((hold >> q) & 1u) && v < nv) x[q][v] = __ldcg(part_row(c_lo + q) + v);
    }
  float mx = lse_l;
  for (int c0 = c_lo + 16; c0 <= c_hi; c0 += 16) {  // more than 16 shares: rare
    const int c = c0 + hl;
    if (row_valid && c <= c_hi && holds(c)) mx = fmaxf(mx, __ldcg(lse_col + static_cast<int64_t>(c) * p.rows_pad));
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));  // within the half
  const float mbase = (mx == -INFINITY) ? 0.f : mx;

  float4 acc[kMaxVec];
#pragma unroll
  for (int v = 0; v < kMaxVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float wl = valid_l ? exp2f(lse_l - mbase) : 0.f;
  float wsum = wl;
#pragma unroll
  for (int q = 0; q < kPrefetchHalf; ++q) {
    const float wq = __shfl_sync(0xffffffffu, wl, hbase + q);
#pragma unroll
    for (int v = 0; v < kMaxVec; ++v) {
      acc[v].x += wq * x[q][v].x;
      acc[v].y += wq * x[q][v].y;
      acc[v].z += wq * x[q][v].z;
      acc[v].w += wq * x[q][v].w;
    }
  }
  // slots kPrefetchHalf .. 15 of the first chunk, then further chunks of 16
  // (the unit, hence every bound, is the same for both halves)
  for (int c0 = c_lo; c0 <= c_hi; c0 += 16) {
    float wc = wl;
    if (c0 != c_lo) {
      const int c = c0 + hl;
      const bool v = row_valid && c <= c_hi && holds(c);
      wc = v ? exp2f(__ldcg(lse_col + static_cast<int64_t>(c) * p.rows_pad) - mbase) : 0.f;
      wsum += wc;
    }
    const int q0 = c0 == c_lo ? kPrefetchHalf : 0;
    for (int q = q0; q < 16 && c0 + q <= c_hi; q += 2) {  // warp-uniform bounds
      float w2[2];
      float4 y[2][kMaxVec];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const bool in = q + u < 16 && c0 + q + u <= c_hi;
        w2[u] = __shfl_sync(0xffffffffu, wc, hbase + (in ? q + u : 0));
        if (!in) w2[u] = 0.f;
#pragma unroll
        for (int v = 0; v < kMaxVec; ++v) {
          y[u][v] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (in && w2[u] != 0.f && v < nv) y[u][v] = __ldcg(part_row(c0 + q + u) + v);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int v = 0; v < kMaxVec; ++v) {
          acc[v].x += w2[u] * y[u][v].x;
          acc[v].y += w2[u] * y[u][v].y;
          acc[v].z += w2[u] * y[u][v].z;
          acc[v].w += w2[u] * y[u][v].w;
        }
    }
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);  // within the half
  if (!row_valid) return;
  const float inv = wsum > 0.f ? __frcp_rn(wsum) : 0.f;
  const int r = rg * kMaxRowsPerUnit + loc;
  const int i = r / p.group, h = (p.hp * kvh + hj) * p.group + r % p.group;
  __nv_bfloat16* orow = p.out + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * D + col;
  if (nv == 2) {
    *reinterpret_cast<uint4*>(orow) =
        make_uint4(pack_bf16x2(acc[0].x * inv, acc[0].y * inv), pack_bf16x2(acc[0].z * inv, acc[0].w * inv),
                   pack_bf16x2(acc[1].x * inv, acc[1].y * inv), pack_bf16x2(acc[1].z * inv, acc[1].w * inv));
  } else {
    *reinterpret_cast<uint2*>(orow) =
        make_uint2(pack_bf16x2(acc[0].x * inv, acc[0].y * inv), pack_bf16x2(acc[0].z * inv, acc[0].w * inv));
  }
  if (p.lse != nullptr && hl == 0)
    p.lse[(static_cast<int64_t>(b) * p.hq + h) * p.n_query + i] = (mbase + log2f(wsum)) * 0.69314718055994530942f;
}


// tcgen05 layout: float4 j of row r of slot s at (s * 32 + j) * 128 + r, so
// a warp's 32 consecutive rows read 512 contiguous bytes.  A warp takes a
// block of 32 rows x 16 columns of a unit and one of S share groups (the
// unit's shares g, g + S, g + 2 S, ...): it requests the lse and partial
// columns of kPrefetchTc of its shares at a time, before their weights are
// known, and folds each batch in with a running max.  With S > 1 the S warps
// of a block combine their sums through shared memory.  S grows with the
// shares a unit has on average, so a unit split across many CTAs costs about
// as many round trips to L2 as one split across a few.  Grid (units, 4 S),
// 256 threads: 8 / S blocks per CTA.
constexpr int kPrefetchTc = 4;
constexpr int kMaxShareGroups = 8;
static_assert(kPrefetchTc * kMaxShareGroups == kMergeSharesPerRound, "the host caps a unit's shares at one round");

__global__ void __launch_bounds__(256, 2) merge_tc_kernel(const AttnParams p) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int S = static_cast<int>(gridDim.y) / 4;  // share groups: 1, 2, 4 or 8
  const int64_t unit = blockIdx.x;
  const int units_per_req = p.hkv / p.hp;  // one row group per unit on this path
  const int b = static_cast<int>(blockIdx.x) / units_per_req;
  const int uir = static_cast<int>(blockIdx.x) % units_per_req;
  const int blk = static_cast<int>(blockIdx.y) * (8 / S) + warp / S;  // 0..31
  const int g = warp % S;
  const int cb = blk >> 2;                 // 16 columns: float4 4 cb .. 4 cb + 3
  const int r = (blk & 3) * 32 + lane;     // row of the 128-row tile
  const int hj = p.hp == 2 ? r >> 6 : 0, loc = p.hp == 2 ? r & 63 : r;
  __shared__ UnitSplit s_sp;
  __shared__ unsigned s_hold;
  __shared__ float xch[8][18][32];  // per warp: max, sum, 16 columns; lane-minor
  if (warp == 0) merge_split(p, b, uir, units_per_req, lane, &s_sp, &s_hold);
  __syncthreads();
  const int c_lo = s_sp.c_lo, c_hi = s_sp.c_hi;
  const unsigned hold = s_hold;
  pdl_wait();
  // No early trigger: the next kernel's CTAs are placed as these exit, so
  // they spread over every SM instead of piling onto the SMs that hold no
  // merge CTA (a streaming kernel after this one is bound by its busiest SM).
  if (c_lo == c_hi) return;  // one CTA held the whole unit and wrote it
  const bool row_ok = loc < p.rows;  // else a padding row of the tile
  auto held = [&](int c) -> bool { return c - c_lo < 32 ? ((hold >> (c - c_lo)) & 1u) != 0 : s_sp.holds(c); };
  const float* lse_col = p.part_lse + unit * kMaxRowsPerUnit + r;
  const float4* o_col = reinterpret_cast<const float4*>(p.part_o) + unit * (32 * kMaxRowsPerUnit) +
                        (4 * cb) * kMaxRowsPerUnit + r;
  auto lse_of = [&](int c) { return __ldcg(lse_col + static_cast<int64_t>(c) * kMaxRowsPerUnit); };
  auto o_of = [&](int c, int j) { return __ldcg(o_col + (static_cast<int64_t>(c) * 32 + j) * kMaxRowsPerUnit); };

  float m = -INFINITY, ws = 0.f;
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (row_ok) {
    for (int c0 = c_lo + g; c0 <= c_hi; c0 += kPrefetchTc * S) {
      float lx[kPrefetchTc];
      float4 x[kPrefetchTc][4];
#pragma unroll
      for (int q = 0; q < kPrefetchTc; ++q) {
        const int c = c0 + q * S;
        lx[q] = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) x[q][j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c <= c_hi && held(c)) {
          lx[q] = lse_of(c);
#pragma unroll
          for (int j = 0; j < 4; ++j) x[q][j] = o_of(c, j);
        }
      }
      float rm = lx[0];
#pragma unroll
      for (int q = 1; q < kPrefetchTc; ++q) rm = fmaxf(rm, lx[q]);
      if (rm > m) {  // rescale what is summed so far (nothing yet: m = -inf gives 0)
        const float sc = exp2f(m - rm);
        ws *= sc;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[j].x *= sc;
          acc[j].y *= sc;
          acc[j].z *= sc;
          acc[j].w *= sc;
        }
        m = rm;
      }
      const float mb = m == -INFINITY ? 0.f : m;
#pragma unroll
      for (int q = 0; q < kPrefetchTc; ++q) {
        const float w = exp2f(lx[q] - mb);  // 0 for shares that are not held (lse -inf)
        ws += w;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[j].x += w * x[q][j].x;
          acc[j].y += w * x[q][j].y;
          acc[j].z += w * x[q][j].z;
          acc[j].w += w * x[q][j].w;
        }
      }
    }
  }
  if (S > 1) {  // CTA-uniform
    xch[warp][0][lane] = m;
    xch[warp][1][lane] = ws;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      xch[warp][2 + 4 * j][lane] = acc[j].x;
      xch[warp][3 + 4 * j][lane] = acc[j].y;
      xch[warp][4 + 4 * j][lane] = acc[j].z;
      xch[warp][5 + 4 * j][lane] = acc[j].w;
    }
    __syncthreads();
    if (g != 0) return;
    for (int o = 1; o < S; ++o) {
      const float om = xch[warp + o][0][lane], ow = xch[warp + o][1][lane];
      float sa, sb;  // scales of this warp's sums and of the other's
      if (om > m) {
        sa = exp2f(m - om);
        sb = 1.f;
        m = om;
      } else if (om != -INFINITY) {
        sa = 1.f;
        sb = exp2f(om - m);
      } else {
        continue;
      }
      ws = ws * sa + ow * sb;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[j].x = acc[j].x * sa + xch[warp + o][2 + 4 * j][lane] * sb;
        acc[j].y = acc[j].y * sa + xch[warp + o][3 + 4 * j][lane] * sb;
        acc[j].z = acc[j].z * sa + xch[warp + o][4 + 4 * j][lane] * sb;
        acc[j].w = acc[j].w * sa + xch[warp + o][5 + 4 * j][lane] * sb;
      }
    }
  }
  if (!row_ok) return;
  const float inv = ws > 0.f ? __frcp_rn(ws) : 0.f;
  const int i = loc / p.group, h = (p.hp * uir + hj) * p.group + loc % p.group;
  uint4* dst = reinterpret_cast<uint4*>(p.out + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * 128 + 16 * cb);
  dst[0] = make_uint4(pack_bf16x2(acc[0].x * inv, acc[0].y * inv), pack_bf16x2(acc[0].z * inv, acc[0].w * inv),
                      pack_bf16x2(acc[1].x * inv, acc[1].y * inv), pack_bf16x2(acc[1].z * inv, acc[1].w * inv));
  dst[1] = make_uint4(pack_bf16x2(acc[2].x * inv, acc[2].y * inv), pack_bf16x2(acc[2].z * inv, acc[2].w * inv),
                      pack_bf16x2(acc[3].x * inv, acc[3].y * inv), pack_bf16x2(acc[3].z * inv, acc[3].w * inv));
  if (p.lse != nullptr && cb == 0)
    p.lse[(static_cast<int64_t>(b) * p.hq + h) * p.n_query + i] = (m + log2f(ws)) * 0.69314718055994530942f;
}

}  // namespace

cudaError_t launch_attn_merge(const AttnParams& p, bool tc_layout, cudaStream_t stream) {
  if (tc_layout) {
    // share groups: enough that kPrefetchTc shares per warp cover a unit's
    // average share count (its CTAs plus one at a boundary)
    const int64_t shares = (p.num_ctas + p.num_units - 1) / p.num_units + 1;
    int groups = 1;
    while (groups < kMaxShareGroups && static_cast<int64_t>(groups) * kPrefetchTc < shares) groups *= 2;
    return launch_pdl(merge_tc_kernel, dim3(static_cast<unsigned>(p.num_units), 4 * groups), dim3(256), 0, stream,
                      p);
  }
  if (p.merge_half_warp) {
    const int row_blocks = (p.rows_pad + kRowsPerCtaHalf - 1) / kRowsPerCtaHalf;
    return launch_pdl(merge_row_per_half_warp_kernel, dim3(static_cast<unsigned>(p.num_units), row_blocks),
                      dim3(kMergeWarps * 32), 0, stream, p);
  }
  const int row_blocks = (p.rows_pad + kMergeWarps - 1) / kMergeWarps;
  return launch_pdl(merge_row_per_warp_kernel, dim3(static_cast<unsigned>(p.num_units), row_blocks),
                    dim3(kMergeWarps * 32), 0, stream, p);
}

}  // namespace ts
