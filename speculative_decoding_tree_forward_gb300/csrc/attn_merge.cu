// Split-KV combine: SwiftSpec summary §3.3 (a head is split across thread
// blocks and their partial results are combined).
//
// A unit (request, KV head, row group) whose tiles several CTAs shared left
// one normalised fp32 partial O_s and its log2-sum-exp lse_s per CTA.  This
// kernel combines them,
//   O = sum_s 2^(lse_s - lse) O_s,   lse = log2 sum_s 2^lse_s,
// skipping CTAs whose tile range was empty, and writes the bf16 output and
// the natural-log lse.  Units held by one CTA were written directly by the
// attention kernel and are skipped here.  One CTA per (unit, 32 rows); a
// thread owns one (row, 32-column segment), so every partial row is streamed
// with independent 16-byte loads and the whole GPU shares the combine.
#include "attn_common.cuh"

namespace ts {
namespace {

constexpr int kMergeRows = 32;
constexpr int kMergeThreads = 128;
constexpr int kMaxSlots = 64;

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnParams p) {
  const int64_t unit = blockIdx.x;
  const int units_per_req = p.hkv * p.row_groups;
  const int b = static_cast<int>(unit / units_per_req);
  const int uir = static_cast<int>(unit % units_per_req);
  const int kvh = uir / p.row_groups;
  const int rg = uir % p.row_groups;
  __shared__ long long red[kMergeThreads];
  __shared__ int slots[kMaxSlots];
  __shared__ int n_slots;
  // tiles before this unit and in total (same clamped lengths as the attention kernels)
  long long before = 0, total = 0;
  for (int bb = threadIdx.x; bb < p.num_req; bb += blockDim.x) {
    int P, n;
    attn_lengths(p, bb, P, n, false);
    const long long tl = static_cast<long long>(attn_tiles(P + n)) * units_per_req;
    total += tl;
    if (bb < b) before += tl;
  }
  red[threadIdx.x] = before;
  __syncthreads();
  for (int s = kMergeThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  const long long base = red[0];
  __syncthreads();
  red[threadIdx.x] = total;
  __syncthreads();
  for (int s = kMergeThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  const int64_t T = red[0];
  int P, n;
  attn_lengths(p, b, P, n, false);
  const int tiles = attn_tiles(P + n);
  const int64_t first = base + static_cast<int64_t>(uir) * tiles;
  const int c_lo = sched_cta_of(first, T, p.num_ctas);
  const int c_hi = sched_cta_of(first + tiles - 1, T, p.num_ctas);
  if (c_lo == c_hi) return;  // one CTA held the whole unit and wrote it
  if (threadIdx.x == 0) {
    int k = 0;
    for (int c = c_lo; c <= c_hi; ++c)
      if (sched_begin(c, T, p.num_ctas) < sched_begin(c + 1, T, p.num_ctas)) {
        if (k < kMaxSlots) slots[k] = c;
        ++k;
      }
    n_slots = k;
  }
  __syncthreads();
  const int ns = n_slots;
  const int D = p.head_dim;
  const int nseg = D / 32;
  const int rows_here = min(kMaxRowsPerUnit, p.rows - rg * kMaxRowsPerUnit);
  const int row0 = blockIdx.y * kMergeRows;
  for (int item = threadIdx.x; item < kMergeRows * nseg; item += blockDim.x) {
    const int rl = row0 + item / nseg, sg = item % nseg;
    if (rl >= rows_here) continue;
    // weights 2^(lse_s - max) of this row
    float mx = -INFINITY;
    for (int k = 0; k < ns; ++k) {
      const int c = k < kMaxSlots ? slots[k] : 0;
      if (k < kMaxSlots) mx = fmaxf(mx, __ldcg(p.part_lse + (c + unit) * p.rows_pad + rl));
    }
    if (ns > kMaxSlots)  // very many splits: walk the CTA range instead of the list
      for (int c = c_lo; c <= c_hi; ++c)
        if (sched_begin(c, T, p.num_ctas) < sched_begin(c + 1, T, p.num_ctas))
          mx = fmaxf(mx, __ldcg(p.part_lse + (c + unit) * p.rows_pad + rl));
    const float mbase = (mx == -INFINITY) ? 0.f : mx;
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    auto add_slot = [&](int c) {
      const float w = exp2f(__ldcg(p.part_lse + (c + unit) * p.rows_pad + rl) - mbase);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(p.part_o + ((c + unit) * p.rows_pad + rl) * D + sg * 32);
      float4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = __ldcg(src + q);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        acc[4 * q + 0] += w * v[q].x;
        acc[4 * q + 1] += w * v[q].y;
        acc[4 * q + 2] += w * v[q].z;
        acc[4 * q + 3] += w * v[q].w;
      }
    };
    if (ns <= kMaxSlots) {
#pragma unroll 2
      for (int k = 0; k < ns; ++k) add_slot(slots[k]);
    } else {
      for (int c = c_lo; c <= c_hi; ++c)
        if (sched_begin(c, T, p.num_ctas) < sched_begin(c + 1, T, p.num_ctas)) add_slot(c);
    }
    const float inv = wsum > 0.f ? __frcp_rn(wsum) : 0.f;
    const int r = rg * kMaxRowsPerUnit + rl;
    const int i = r / p.group, h = kvh * p.group + r % p.group;
    uint4* dst = reinterpret_cast<uint4*>(p.out + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * D + sg * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      dst[q] = make_uint4(pack_bf16x2(acc[8 * q + 0] * inv, acc[8 * q + 1] * inv),
                          pack_bf16x2(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv),
                          pack_bf16x2(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv),
                          pack_bf16x2(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv));
    if (p.lse != nullptr && sg == 0)
      p.lse[(static_cast<int64_t>(b) * p.hq + h) * p.n_query + i] = (mbase + log2f(wsum)) * 0.69314718055994530942f;
  }
}

}  // namespace

cudaError_t launch_attn_merge(const AttnParams& p, cudaStream_t stream) {
  const int row_blocks = (p.rows_pad + kMergeRows - 1) / kMergeRows;
  dim3 grid(static_cast<unsigned>(p.num_units), row_blocks);
  attn_merge_kernel<<<grid, kMergeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ts
