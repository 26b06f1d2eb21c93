// Split-KV combine: SwiftSpec summary §3.3 (a head is split across thread
// blocks and their partial results are combined).
//
// A unit (request, KV head, row group) whose tiles several CTAs shared left
// one normalised fp32 partial O_s and its log2-sum-exp lse_s per CTA.  This
// kernel combines them,
//   O = sum_s 2^(lse_s - lse) O_s,   lse = log2 sum_s 2^lse_s,
// skipping CTAs whose tile range was empty, and writes the bf16 output and
// the natural-log lse.  Units held by one CTA were written directly by the
// attention kernel and are skipped here.  One warp per output row, eight rows
// per CTA, each lane owning four columns.  The split (which CTAs hold tiles
// of the unit) follows from the request lengths alone, so it is worked out
// before the kernel waits for the attention kernel's results.  After the wait
// the lse of the row's first 32 shares (one per lane) and its first eight
// partial rows (coalesced 512-byte reads) are all requested before the
// weights are known, so a row with up to eight shares costs one round trip
// to L2; shares of CTAs that hold no tile of the unit get weight 0.
#include "attn_common.cuh"

namespace ts {
namespace {

constexpr int kMergeWarps = 8;  // rows per CTA
constexpr int kPrefetchSlots = 8;  // partial rows loaded before the weights are known

// at most 64 registers: four CTAs (32 warps) per SM, so the grid lands in one wave
__global__ void __launch_bounds__(kMergeWarps * 32, 4) attn_merge_kernel(const AttnParams p) {
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
  // The split as the attention kernel laid it out, from the request lengths
  // it read (clamped the same way).  They were final before the attention
  // kernel passed its own wait, which precedes this grid's launch, so warp 0
  // works the split out for the CTA's unit before the wait for the attention
  // kernel's results: the CTAs holding tiles of the unit and, for the first
  // 32 of them, which hold a share.
  __shared__ UnitSplit s_sp;
  __shared__ unsigned s_hold;
  if (warp == 0) {
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
    if (lane == 0) s_sp.init(before, total, mine, b, uir, units_per_req, p.num_req, p.seg_cost, p.num_ctas);
    __syncwarp();
    const int c = s_sp.c_lo + lane;
    const unsigned hold = __ballot_sync(0xffffffffu, c <= s_sp.c_hi && s_sp.c_lo != s_sp.c_hi && s_sp.holds(c));
    if (lane == 0) s_hold = hold;
  }
  __syncthreads();
  const int c_lo = s_sp.c_lo, c_hi = s_sp.c_hi;
  const bool valid_l = (s_hold >> lane) & 1u;
  pdl_wait();
  pdl_launch_dependents();
  if (!row_valid || c_lo == c_hi) return;  // padding row, or one CTA held the whole unit and wrote it
  auto holds = [&](int c) -> bool { return s_sp.holds(c); };
  const int ncs = c_hi - c_lo + 1;

  // slot of CTA c: c + unit; its lse at part_lse[slot * rows_pad + row]
  const float* lse_col = p.part_lse + unit * p.rows_pad + rl;
  const int D = p.head_dim;
  const bool active = lane * 4 < D;
  auto part_row = [&](int c) {
    return reinterpret_cast<const float4*>(p.part_o + ((static_cast<int64_t>(c) + unit) * p.rows_pad + rl) * D +
                                           lane * 4);
  };
  // one round trip: the lse of the first 32 slots (one per lane) and the
  // partial rows of the first kPrefetchSlots slots, all issued before the
  // weights are known (slots of CTAs without a share get weight 0)
  const unsigned hold = s_hold;
  float lse_l = -INFINITY;
  if (valid_l) lse_l = __ldcg(lse_col + static_cast<int64_t>(c_lo + lane) * p.rows_pad);
  float4 x[kPrefetchSlots];
#pragma unroll
  for (int q = 0; q < kPrefetchSlots; ++q) {
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
  for (int q = 0; q < kPrefetchSlots; ++q) {
    const float wq = __shfl_sync(0xffffffffu, wl, q);
    acc.x += wq * x[q].x;
    acc.y += wq * x[q].y;
    acc.z += wq * x[q].z;
    acc.w += wq * x[q].w;
  }
  // slots kPrefetchSlots .. 31 of the first chunk, then further chunks of 32
  for (int c0 = c_lo; c0 <= c_hi; c0 += 32) {
    float wc = wl;
    if (c0 != c_lo) {
      const int c = c0 + lane;
      const bool v = c <= c_hi && holds(c);
      wc = v ? exp2f(__ldcg(lse_col + static_cast<int64_t>(c) * p.rows_pad) - mbase) : 0.f;
      wsum += wc;
    }
    const int q0 = c0 == c_lo ? kPrefetchSlots : 0;
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

}  // namespace

cudaError_t launch_attn_merge(const AttnParams& p, cudaStream_t stream) {
  const int row_blocks = (p.rows_pad + kMergeWarps - 1) / kMergeWarps;
  return launch_pdl(attn_merge_kernel, dim3(static_cast<unsigned>(p.num_units), row_blocks), dim3(kMergeWarps * 32), 0,
                    stream, p);
}

}  // namespace ts
