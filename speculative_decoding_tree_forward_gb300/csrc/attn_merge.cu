// Split-KV combine: SwiftSpec summary §3.3 (a head is split across thread
// blocks and their partial results are combined).
//
// A unit (request, KV head, row group) whose tiles several CTAs shared left
// one normalised fp32 partial O_s and its log2-sum-exp lse_s per CTA.  This
// kernel combines them,
//   O = sum_s 2^(lse_s - lse) O_s,   lse = log2 sum_s 2^lse_s,
// skipping CTAs whose tile range was empty, and writes the bf16 output and
// the natural-log lse.  Units held by one CTA were written directly by the
// attention kernel and are skipped here.  One warp per output row: the lanes
// find the row's non-empty slots with a ballot and each lane owns four
// columns, so a slot's partial row is one coalesced 512-byte read and up to
// four slots are in flight per lane; no block-wide synchronisation.
#include "attn_common.cuh"

namespace ts {
namespace {

constexpr int kMergeWarps = 4;  // rows per CTA

__device__ __forceinline__ bool slot_nonempty(int c, int64_t T, int nc) {
  return sched_begin(c, T, nc) < sched_begin(c + 1, T, nc);
}

__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const AttnParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t unit = blockIdx.x;
  // a unit is (request, group of hp KV heads, row group); with hp = 2 the
  // unit's rows are two heads' R <= 64 rows at 0 and 64
  const int units_per_req = (p.hkv / p.hp) * p.row_groups;
  const int b = static_cast<int>(unit / units_per_req);
  const int uir = static_cast<int>(unit % units_per_req);
  const int kvh = uir / p.row_groups;  // head group
  const int rg = uir % p.row_groups;
  const int rl = blockIdx.y * kMergeWarps + warp;
  const int hj = p.hp == 2 ? rl >> 6 : 0, loc = p.hp == 2 ? rl & 63 : rl;
  if (p.hp == 2 ? loc >= p.rows : rl >= min(kMaxRowsPerUnit, p.rows - rg * kMaxRowsPerUnit)) return;
  // tiles before this unit and in total (same clamped lengths as the attention kernels)
  long long before = 0, total = 0;
  for (int bb = lane; bb < p.num_req; bb += 32) {
    int P, n;
    attn_lengths(p, bb, P, n, false);
    const long long tl = static_cast<long long>(attn_tiles(P + n)) * units_per_req;
    total += tl;
    if (bb < b) before += tl;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  const int64_t T = total;
  int P, n;
  attn_lengths(p, b, P, n, false);
  const int tiles = attn_tiles(P + n);
  const int64_t first = before + static_cast<int64_t>(uir) * tiles;
  // CTAs holding the unit's first and last tile (plain or cost-weighted split)
  const int E = p.seg_cost;
  const int64_t W = T + static_cast<int64_t>(E) * units_per_req * p.num_req;
  const int64_t pf = before + static_cast<int64_t>(E) * units_per_req * b + static_cast<int64_t>(uir) * (tiles + E);
  const int c_lo = E > 0 ? wsched_cta_of_pos(pf, W, p.num_ctas) : sched_cta_of(first, T, p.num_ctas);
  const int c_hi = E > 0 ? wsched_cta_of_pos(pf + (tiles >= 2 ? E + tiles - 1 : 0), W, p.num_ctas)
                         : sched_cta_of(first + tiles - 1, T, p.num_ctas);
  if (c_lo == c_hi) return;  // one CTA held the whole unit and wrote it
  // does CTA c (c_lo <= c <= c_hi) hold a tile of this unit, i.e. a partial?
  auto holds = [&](int c) -> bool {
    if (E == 0) return slot_nonempty(c, T, p.num_ctas);
    if (c == c_lo) return true;
    const int j = wsched_tile_in_unit(wsched_x(c, W, p.num_ctas) - pf, E, tiles);
    return j < tiles && wsched_cta_of_pos(pf + E + j, W, p.num_ctas) == c;
  };

  // slot of CTA c: c + unit; its lse at part_lse[slot * rows_pad + row]
  const float* lse_col = p.part_lse + unit * p.rows_pad + rl;
  float mx = -INFINITY;
  for (int c0 = c_lo; c0 <= c_hi; c0 += 32) {
    const int c = c0 + lane;
    if (c <= c_hi && holds(c))
      mx = fmaxf(mx, __ldcg(lse_col + static_cast<int64_t>(c) * p.rows_pad));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float mbase = (mx == -INFINITY) ? 0.f : mx;

  const int D = p.head_dim;
  const bool active = lane * 4 < D;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  for (int c0 = c_lo; c0 <= c_hi; c0 += 32) {
    const int c = c0 + lane;
    const bool valid = c <= c_hi && holds(c);
    const float wl = valid ? exp2f(__ldcg(lse_col + static_cast<int64_t>(c) * p.rows_pad) - mbase) : 0.f;
    wsum += wl;
    unsigned mask = __ballot_sync(0xffffffffu, valid);
    while (mask != 0u) {  // warp-uniform
      int j[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        j[q] = mask != 0u ? __ffs(mask) - 1 : -1;
        if (mask != 0u) mask &= mask - 1u;
      }
      float w[4];
      float4 x[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        w[q] = __shfl_sync(0xffffffffu, wl, j[q] < 0 ? 0 : j[q]);
        x[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j[q] >= 0 && active)
          x[q] = __ldcg(reinterpret_cast<const float4*>(
              p.part_o + ((static_cast<int64_t>(c0 + j[q]) + unit) * p.rows_pad + rl) * D + lane * 4));
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float wq = j[q] >= 0 ? w[q] : 0.f;
        acc.x += wq * x[q].x;
        acc.y += wq * x[q].y;
        acc.z += wq * x[q].z;
        acc.w += wq * x[q].w;
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
