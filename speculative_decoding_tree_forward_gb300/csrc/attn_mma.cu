// Tree-masked GQA attention on warp-level bf16 MMA (m16n8k16, fp32 accumulate).
//
// SwiftSpec summary, §3.1.3 / Figure 3 (non-square ancestor mask) and §3.3
// (a head split across thread blocks, partials combined).  Used whenever the
// packed query rows of a KV head (R = G * n_query, NVIDIA draft-length
// article) do not fill a 128-row tensor-core tile.
//
// CTA layout: warp 0 is the producer (one lane issues TMA loads of 64-key K
// and V tiles into a ring of shared-memory stages, 128-byte swizzled);
// warps 1..RB each own 16 packed query rows and stream every tile of the
// CTA's key range through QK^T, an online softmax in the exp2 domain and PV.
// Keys are split across CTAs by the stream-K schedule in common.cuh; a CTA
// that holds a whole unit writes the bf16 output directly, otherwise it
// writes a normalised fp32 partial and its log2-sum-exp, which the combine
// kernel (attn_merge.cu) merges.
#include "attn_common.cuh"

namespace ts {
namespace {

constexpr int kThreadsPerWarp = 32;

struct SmemLayout {
  uint32_t stage_bytes, kv_bytes, qs, bars, par, cum, flag, total;
};

// [stages x (K tile, V tile)] [Q: 16 rows per consumer warp] [barriers]
// [parent copy per consumer warp] [schedule]
__host__ __device__ inline SmemLayout mma_layout(int head_dim, int stages, int num_req, int rows_pad) {
  SmemLayout L;
  L.kv_bytes = static_cast<uint32_t>(head_dim) * kBlockN * 2;     // one of K or V
  L.stage_bytes = 2 * L.kv_bytes;
  L.qs = static_cast<uint32_t>(stages) * L.stage_bytes;            // 1024-aligned
  L.bars = L.qs + static_cast<uint32_t>(rows_pad) * head_dim * 2;  // 1024-aligned
  L.par = L.bars + 2 * 8 * stages;
  L.cum = L.par + static_cast<uint32_t>(rows_pad / 16) * TS_MAX_TREE * 4;
  L.cum = (L.cum + 7) & ~7u;
  L.flag = L.cum + 8 * (kMaxRequestsAttn + 1);  // fixed: launch shape independent of the batch
  (void)num_req;
  L.total = L.flag + 16;
  return L;
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <int D, bool kBounded>
__global__ void __launch_bounds__(288) attn_mma_kernel(const __grid_constant__ CUtensorMap kmap,
                                                       const __grid_constant__ CUtensorMap vmap,
                                                       const AttnParams p) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemLayout L = mma_layout(D, p.stages, p.num_req, p.rows_pad);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty_bar = full_bar + p.stages;
  int64_t* cum = reinterpret_cast<int64_t*>(smem + L.cum);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flag);

  const int tid = threadIdx.x;
  const int warp = tid / kThreadsPerWarp;
  const int lane = tid % kThreadsPerWarp;
  const int RB = p.rows_pad / 16;
  const int n_consumers = RB * kThreadsPerWarp;
  const int units_per_req = p.hkv * p.row_groups;

  // ---- schedule: tiles per request, prefix sums (request-major units)
  for (int b = tid; b < p.num_req; b += blockDim.x) {
    int P, n;
    attn_lengths(p, b, P, n, blockIdx.x == 0);
    cum[b + 1] = static_cast<int64_t>(attn_tiles(P + n)) * units_per_req;
  }
  if (tid == 0) {
    cum[0] = 0;
    *abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], RB);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int b = 0; b < p.num_req; ++b) cum[b + 1] += cum[b];
  }
  __syncthreads();
  const int64_t T = cum[p.num_req];
  const int64_t t_begin = sched_begin(blockIdx.x, T, p.num_ctas);
  const int64_t t_end = sched_begin(blockIdx.x + 1, T, p.num_ctas);
  if (t_begin >= t_end) return;

  // locate the request holding tile t_begin
  int b0 = 0;
  {
    int lo = 0, hi = p.num_req - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (cum[mid] <= t_begin) lo = mid; else hi = mid - 1;
    }
    b0 = lo;
  }

  if (warp == 0) {
    // ================= producer =================
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      int b = b0;
      int P = 0, n = 0, tiles = 1;
      attn_lengths(p, b, P, n, false);
      tiles = attn_tiles(P + n);
      int64_t local = t_begin - cum[b];
      int uir = static_cast<int>(local / tiles);
      int tile = static_cast<int>(local % tiles);
      const int halves = D / 64;
      const uint32_t kv_half = kBlockN * 128;
      const int n_tiles = static_cast<int>(t_end - t_begin);
      int s = 0;
      uint32_t phase = 0;  // completed passes over the ring
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        if (it >= p.stages) {
          if (!pipe_wait<kBounded>(&empty_bar[s], (phase - 1) & 1, p.wait_ns)) {
            report_error(p.err, TS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
        uint8_t* ks = smem + static_cast<size_t>(s) * L.stage_bytes;
        uint8_t* vs = ks + L.kv_bytes;
        const int kvh = (uir / p.row_groups);
        const int key0 = tile * kBlockN;
        mbar_arrive_expect_tx(&full_bar[s], L.stage_bytes);
        if (!p.paged) {
          const int row = b * p.max_kv_len + key0;
          for (int h = 0; h < halves; ++h) {
            tma_load_3d(ks + h * kv_half, &kmap, h * 64, kvh, row, &full_bar[s]);
            tma_load_3d(vs + h * kv_half, &vmap, h * 64, kvh, row, &full_bar[s]);
          }
        } else {
          const int pages = kBlockN / p.page_size;
          const int keys = P + n;
          for (int pg = 0; pg < pages; ++pg) {
            const int lb = key0 / p.page_size + pg;
            int row = p.num_blocks * p.page_size;  // past the pool: TMA fills zeros
            if (lb * p.page_size < keys) {
              const int blk = p.block_table[static_cast<int64_t>(b) * p.max_blocks + lb];
              if (blk >= 0 && blk < p.num_blocks) row = blk * p.page_size;
              else report_error(p.err, TS_DEVERR_BAD_BLOCK);
            }
            const uint32_t off = static_cast<uint32_t>(pg * p.page_size) * 128u;
            for (int h = 0; h < halves; ++h) {
              tma_load_3d(ks + h * kv_half + off, &kmap, h * 64, kvh, row, &full_bar[s]);
              tma_load_3d(vs + h * kv_half + off, &vmap, h * 64, kvh, row, &full_bar[s]);
            }
          }
        }
        ++issued;
        if (++s == p.stages) {
          s = 0;
          ++phase;
        }
        // advance
        if (++tile == tiles) {
          tile = 0;
          if (++uir == units_per_req) {
            uir = 0;
            ++b;
            if (b < p.num_req) {
              attn_lengths(p, b, P, n, false);
              tiles = attn_tiles(P + n);
            }
          }
        }
      }
      // Do not leave while copies issued into this CTA's shared memory are
      // still in flight (possible only after an abort): drain, bounded.
      if (*abort_flag) {
        for (int st = 0; st < p.stages && st < issued; ++st) {
          const int last = issued - 1 - ((issued - 1 - st) % p.stages);
          mbar_wait(&full_bar[st], static_cast<uint32_t>((last / p.stages) & 1));
        }
      }
    }
    return;
  }

  // ================= consumers =================
  const int ctid = tid - kThreadsPerWarp;
  const int rb = warp - 1;
  const int g = lane >> 2;  // row within the 8-row half of the fragment
  const int t4 = lane & 3;  // column pair
  constexpr int NB_O = D / 8;     // n8 blocks of the output
  const uint32_t kv_half = kBlockN * 128;
  const uint32_t smem_base = smem_u32(smem);

  float o[NB_O][4];
  int* par_w = reinterpret_cast<int*>(smem + L.par) + rb * TS_MAX_TREE;
  const uint32_t qs_warp = smem_u32(smem + L.qs) + static_cast<uint32_t>(rb) * 16 * D * 2;
  // Per-lane pieces of the 128-byte-swizzled ldmatrix addresses (the rest are
  // compile-time offsets): within a 1024-byte block, row r and 16-byte chunk c
  // sit at r*128 + ((c ^ (r & 7)) << 4), and every row index below is
  // (lane & 7) plus a multiple of 8.
  const uint32_t l7 = lane & 7;
  const uint32_t q_row_off = (l7 + ((lane >> 3) & 1) * 8) * 128;
  const uint32_t kv_row_off = l7 * 128;
  const uint32_t v_row_off = (l7 + ((lane >> 3) & 1) * 8) * 128;
  uint32_t q_sw[4], k_sw[2], v_sw[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) q_sw[j] = (((2 * j + (lane >> 4)) ^ l7) & 7) << 4;
#pragma unroll
  for (int j = 0; j < 2; ++j) k_sw[j] = (((4 * j + (lane >> 3)) ^ l7) & 7) << 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) v_sw[j] = (((2 * j + (lane >> 4)) ^ l7) & 7) << 4;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  uint32_t anc0[4] = {0, 0, 0, 0}, anc1[4] = {0, 0, 0, 0};

  int b = b0;
  int P = 0, n = 0, tiles = 1;
  attn_lengths(p, b, P, n, false);
  tiles = attn_tiles(P + n);
  int64_t local = t_begin - cum[b];
  int uir = static_cast<int>(local / tiles);
  int tile = static_cast<int>(local % tiles);
  int seg_first = tile;
  int anc_req = -1;
  bool need_setup = true;

  const int n_tiles = static_cast<int>(t_end - t_begin);
  int s = 0;
  uint32_t phase = 0;
  for (int it = 0; it < n_tiles; ++it) {
    if (need_setup) {
      // ---- start of a unit: ancestor masks (once per request), Q fragments, state
      need_setup = false;
      const int kvh = uir / p.row_groups;
      const int rg = uir % p.row_groups;
      if (anc_req != b) {
        // this warp's copy of the request's parent array (validated)
        __syncwarp();
        for (int i = lane; i < n; i += kThreadsPerWarp) {
          int q = p.parent[static_cast<int64_t>(b) * p.n_tree_max + i];
          if (q < -1 || q >= i) {
            if (blockIdx.x == 0) report_error(p.err, TS_DEVERR_BAD_PARENT);
            q = -1;
          }
          par_w[i] = q;
        }
        __syncwarp();
        anc_req = b;
      }
      const int r0 = rg * kMaxRowsPerUnit + rb * 16 + g;
      const int r1 = r0 + 8;
      ancestor_walk(par_w, n - p.n_query + min(r0, p.rows - 1) / p.group, anc0);
      ancestor_walk(par_w, n - p.n_query + min(r1, p.rows - 1) / p.group, anc1);
      // this warp's 16 query rows -> shared memory, 128-byte swizzled rows;
      // with RoPE each (row, 8 pairs) item is rotated on the way, at position
      // P + depth of the row's node (SwiftSpec summary §3.3): chunk c16 of the
      // first half pairs with chunk c16 + D / 16 of the second
      {
        uint8_t* qw = smem + L.qs + static_cast<uint32_t>(rb) * 16 * D * 2;
        const int per_row = p.rope ? D / 16 : D / 8;  // items per row
        for (int x = lane; x < 16 * per_row; x += kThreadsPerWarp) {
          const int rr = x / per_row, c16 = x % per_row;
          const int r = rg * kMaxRowsPerUnit + rb * 16 + rr;
          uint4 v = make_uint4(0, 0, 0, 0), w = make_uint4(0, 0, 0, 0);
          if (r < p.rows) {
            const int i = r / p.group, h = kvh * p.group + r % p.group;
            const __nv_bfloat16* qrow = p.q + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * D;
            v = __ldg(reinterpret_cast<const uint4*>(qrow + c16 * 8));
            if (p.rope) {
              w = __ldg(reinterpret_cast<const uint4*>(qrow + D / 2 + c16 * 8));
              int u = n - p.n_query + i, depth = 0;
              while (par_w[u] >= 0) {  // parent[u] < u: at most n steps
                u = par_w[u];
                ++depth;
              }
              rope_rotate8(v, w, P + depth, p.rope_turn, 8 * c16);
            }
          }
          *reinterpret_cast<uint4*>(qw + (c16 >> 3) * (16 * 128) + sw128(rr, c16 & 7)) = v;
          if (p.rope) {
            const int c2 = c16 + D / 16;
            *reinterpret_cast<uint4*>(qw + (c2 >> 3) * (16 * 128) + sw128(rr, c2 & 7)) = w;
          }
        }
        __syncwarp();
      }
#pragma unroll
      for (int nb = 0; nb < NB_O; ++nb) o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
    }
    if (*abort_flag || !pipe_wait<kBounded>(&full_bar[s], phase & 1, p.wait_ns)) {
      report_error(p.err, TS_DEVERR_TIMEOUT);
      *abort_flag = 1;
      break;
    }
    const uint32_t ks = smem_base + static_cast<uint32_t>(s) * L.stage_bytes;
    const uint32_t vs = ks + L.kv_bytes;
    const int key0 = tile * kBlockN;
    const int keys = P + n;
    if (key0 + kBlockN > keys) {
      // Rows past the last key may hold anything (another request's rows,
      // unwritten memory).  Their probability is 0, but 0 * NaN is NaN, so
      // each warp zeroes them before its own PV (all warps write the same
      // zeros, so no cross-warp barrier is needed).
      uint8_t* vgen = smem + static_cast<size_t>(s) * L.stage_bytes + L.kv_bytes;
      const int first = keys - key0;
      const int nvec = (kBlockN - first) * 8;  // 16-byte vectors per half
      for (int h = 0; h < D / 64; ++h)
        for (int x = lane; x < nvec; x += kThreadsPerWarp)
          reinterpret_cast<uint4*>(vgen + h * kv_half + first * 128)[x] = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
      __syncwarp();
    }
    // visibility of this thread's 16 columns (nb*8 + 2*t4 + e) as bit nb*2+e
    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
    const bool tree_tile = key0 + kBlockN > P;
    if (tree_tile) {
      const uint64_t w0 = tile_visibility(anc0, key0 - P) >> (2 * t4);
      const uint64_t w1 = tile_visibility(anc1, key0 - P) >> (2 * t4);
      vm0 = 0;
      vm1 = 0;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
        vm0 |= static_cast<uint32_t>((w0 >> (nb * 8)) & 3ull) << (2 * nb);
        vm1 |= static_cast<uint32_t>((w1 >> (nb * 8)) & 3ull) << (2 * nb);
      }
    }

    // The 64-key tile is consumed as two 32-key halves, each a full
    // QK^T -> masked online softmax -> PV step, which keeps the live score
    // and probability registers small next to the 16 x D accumulator.
#pragma unroll
    for (int hk = 0; hk < 2; ++hk) {
      // ---- S = Q K^T (16 rows x 32 keys per warp)
      float sc[4][4];
#pragma unroll
      for (int nb = 0; nb < 4; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
#pragma unroll
      for (int kk2 = 0; kk2 < D / 32; ++kk2) {
        uint32_t qf[2][4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          // A fragment: lanes 0-7 / 8-15 give rows 0-7 / 8-15 of the low 8 columns, lanes 16-31 the high 8
          const int c16 = (2 * kk2 + h2) * 2;  // + (lane >> 4)
          ldsm_x4(qs_warp + (c16 >> 3) * (16 * 128) + q_row_off + q_sw[(c16 & 7) >> 1], qf[h2][0], qf[h2][1],
                  qf[h2][2], qf[h2][3]);
        }
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
          // B fragments of 8 keys: lane -> key (hk*4+nb)*8 + (lane & 7), 16-byte chunk kk2*4 + (lane >> 3)
          const int c16 = kk2 * 4;
          const uint32_t addr = ks + (c16 >> 3) * kv_half + (hk * 4 + nb) * 1024 + kv_row_off + k_sw[(c16 & 7) >> 2];
          uint32_t b0r, b1r, b2r, b3r;
          ldsm_x4(addr, b0r, b1r, b2r, b3r);
          mma_16816(sc[nb], qf[0], b0r, b1r);
          mma_16816(sc[nb], qf[1], b2r, b3r);
        }
      }

      // ---- mask + online softmax (exp2 domain)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int bit = 2 * (hk * 4 + nb) + e;
          float x0 = sc[nb][e] * p.scale_log2;
          float x1 = sc[nb][2 + e] * p.scale_log2;
          x0 = ((vm0 >> bit) & 1u) ? x0 : -INFINITY;
          x1 = ((vm1 >> bit) & 1u) ? x1 : -INFINITY;
          sc[nb][e] = x0;
          sc[nb][2 + e] = x1;
          mx0 = fmaxf(mx0, x0);
          mx1 = fmaxf(mx1, x1);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float alpha0 = exp2f(m0 - base0), alpha1 = exp2f(m1 - base1);
      m0 = mn0;
      m1 = mn1;
      // probabilities -> bf16 A fragments of P (the m16n8 C layout of two
      // adjacent n8 blocks is the m16k16 A layout)
      // On tiles that hold tree keys a query may see only a few keys, whose V
      // rows can cancel; there the bf16 rounding residual of P is carried by
      // a second PV product (P = hi + lo), so rows with few keys keep fp32-like
      // accuracy.  Prefix-only tiles use P rounded once.
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pa[2][4], pl[2][4];
#pragma unroll
      for (int kc = 0; kc < 2; ++kc) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int nb = 2 * kc + hb;
          const float e0 = exp2f(sc[nb][0] - base0), e1 = exp2f(sc[nb][1] - base0);
          const float e2 = exp2f(sc[nb][2] - base1), e3 = exp2f(sc[nb][3] - base1);
          rs0 += e0 + e1;
          rs1 += e2 + e3;
          pa[kc][2 * hb + 0] = pack_bf16x2(e0, e1);
          pa[kc][2 * hb + 1] = pack_bf16x2(e2, e3);
          pl[kc][2 * hb + 0] = bf16x2_residual(pa[kc][2 * hb + 0], e0, e1);
          pl[kc][2 * hb + 1] = bf16x2_residual(pa[kc][2 * hb + 1], e2, e3);
        }
      }
      l0 = l0 * alpha0 + rs0;
      l1 = l1 * alpha1 + rs1;
#pragma unroll
      for (int nb = 0; nb < NB_O; ++nb) {
        o[nb][0] *= alpha0;
        o[nb][1] *= alpha0;
        o[nb][2] *= alpha1;
        o[nb][3] *= alpha1;
      }

      // ---- O += P V
#pragma unroll
      for (int kc = 0; kc < 2; ++kc) {
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          // transposed B fragments: lane -> key (hk*2+kc)*16 + ((lane >> 3) & 1) * 8 + (lane & 7),
          // 16-byte chunk dp*2 + (lane >> 4)
          const int c16 = dp * 2;
          const uint32_t addr = vs + (c16 >> 3) * kv_half + (hk * 2 + kc) * 2048 + v_row_off + v_sw[(c16 & 7) >> 1];
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(addr, r0, r1, r2, r3);
          mma_16816(o[2 * dp], pa[kc], r0, r1);
          mma_16816(o[2 * dp + 1], pa[kc], r2, r3);
          if (tree_tile) {
            mma_16816(o[2 * dp], pl[kc], r0, r1);
            mma_16816(o[2 * dp + 1], pl[kc], r2, r3);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
    if (++s == p.stages) {
      s = 0;
      ++phase;
    }

    // ---- end of a unit segment: direct bf16 output or a partial for the merge
    const bool last_of_cta = (it + 1 == n_tiles);
    if (tile == tiles - 1 || last_of_cta) {
      const int kvh = uir / p.row_groups;
      const int rg = uir % p.row_groups;
      float L0 = l0, L1 = l1;
      L0 += __shfl_xor_sync(0xffffffffu, L0, 1);
      L0 += __shfl_xor_sync(0xffffffffu, L0, 2);
      L1 += __shfl_xor_sync(0xffffffffu, L1, 1);
      L1 += __shfl_xor_sync(0xffffffffu, L1, 2);
      const float inv0 = L0 > 0.f ? __frcp_rn(L0) : 0.f;
      const float inv1 = L1 > 0.f ? __frcp_rn(L1) : 0.f;
      const int rl0 = rb * 16 + g, rl1 = rl0 + 8;
      const int r0 = rg * kMaxRowsPerUnit + rl0, r1 = r0 + 8;
      const bool complete = (seg_first == 0) && (tile == tiles - 1);
      if (complete) {
        const float ln2 = 0.69314718055994530942f;
        if (r0 < p.rows) {
          const int i = r0 / p.group, h = kvh * p.group + r0 % p.group;
          __nv_bfloat16* orow = p.out + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * D;
#pragma unroll
          for (int nb = 0; nb < NB_O; ++nb)
            *reinterpret_cast<uint32_t*>(orow + nb * 8 + 2 * t4) = pack_bf16x2(o[nb][0] * inv0, o[nb][1] * inv0);
          if (p.lse != nullptr && t4 == 0) p.lse[(static_cast<int64_t>(b) * p.hq + h) * p.n_query + i] = (m0 + log2f(L0)) * ln2;
        }
        if (r1 < p.rows) {
          const int i = r1 / p.group, h = kvh * p.group + r1 % p.group;
          __nv_bfloat16* orow = p.out + ((static_cast<int64_t>(b) * p.n_query + i) * p.hq + h) * D;
#pragma unroll
          for (int nb = 0; nb < NB_O; ++nb)
            *reinterpret_cast<uint32_t*>(orow + nb * 8 + 2 * t4) = pack_bf16x2(o[nb][2] * inv1, o[nb][3] * inv1);
          if (p.lse != nullptr && t4 == 0) p.lse[(static_cast<int64_t>(b) * p.hq + h) * p.n_query + i] = (m1 + log2f(L1)) * ln2;
        }
      } else {
        const int64_t unit = static_cast<int64_t>(b) * units_per_req + uir;
        const int64_t slot = static_cast<int64_t>(blockIdx.x) + unit;
        float* po = p.part_o + slot * p.rows_pad * D;
        float* pl = p.part_lse + slot * p.rows_pad;
#pragma unroll
        for (int nb = 0; nb < NB_O; ++nb) {
          *reinterpret_cast<float2*>(po + rl0 * D + nb * 8 + 2 * t4) = make_float2(o[nb][0] * inv0, o[nb][1] * inv0);
          *reinterpret_cast<float2*>(po + rl1 * D + nb * 8 + 2 * t4) = make_float2(o[nb][2] * inv1, o[nb][3] * inv1);
        }
        if (t4 == 0) {
          pl[rl0] = L0 > 0.f ? m0 + log2f(L0) : -INFINITY;
          pl[rl1] = L1 > 0.f ? m1 + log2f(L1) : -INFINITY;
        }
      }
      if (last_of_cta) break;
      if (++uir == units_per_req) {
        uir = 0;
        ++b;
        attn_lengths(p, b, P, n, false);
        tiles = attn_tiles(P + n);
      }
      tile = 0;
      seg_first = 0;
      need_setup = true;
    } else {
      ++tile;
    }
  }
}

}  // namespace

size_t attn_mma_smem_bytes(int head_dim, int stages, int num_req, int rows_pad) {
  return mma_layout(head_dim, stages, num_req, rows_pad).total + 1024;  // + alignment slack
}

int attn_mma_threads(int rows_pad) { return kThreadsPerWarp * (1 + rows_pad / 16); }

// The dynamic shared-memory attribute was raised by attn_mma_occupancy, which
// the host plan runs (once per device and shape) before any launch.
cudaError_t launch_attn_mma(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
  const size_t smem = attn_mma_smem_bytes(p.head_dim, p.stages, p.num_req, p.rows_pad);
  const int threads = attn_mma_threads(p.rows_pad);
  const bool bounded = p.wait_ns < kWaitLimitNs;  // a caller-given bound: the bounded-wait variant
  if (p.head_dim == 128)
    return bounded ? launch_pdl(attn_mma_kernel<128, true>, dim3(p.num_ctas), dim3(threads), smem, stream, kmap, vmap, p)
                   : launch_pdl(attn_mma_kernel<128, false>, dim3(p.num_ctas), dim3(threads), smem, stream, kmap, vmap, p);
  return bounded ? launch_pdl(attn_mma_kernel<64, true>, dim3(p.num_ctas), dim3(threads), smem, stream, kmap, vmap, p)
                 : launch_pdl(attn_mma_kernel<64, false>, dim3(p.num_ctas), dim3(threads), smem, stream, kmap, vmap, p);
}

int attn_mma_occupancy(int head_dim, int stages, int num_req, int rows_pad) {
  // raise the kernel's dynamic shared-memory limit to the device maximum once,
  // so every shape's launch fits; occupancy uses this shape's size
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  int nb = 0;
  const size_t smem = attn_mma_smem_bytes(head_dim, stages, num_req, rows_pad);
  if (smem > static_cast<size_t>(optin)) return 0;
  const int threads = attn_mma_threads(rows_pad);
  if (head_dim == 128) {
    if (cudaFuncSetAttribute(attn_mma_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_mma_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
            cudaSuccess)
      return 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, attn_mma_kernel<128, false>, threads, smem);
  } else {
    if (cudaFuncSetAttribute(attn_mma_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_mma_kernel<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
            cudaSuccess)
      return 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, attn_mma_kernel<64, false>, threads, smem);
  }
  return nb;
}

}  // namespace ts
