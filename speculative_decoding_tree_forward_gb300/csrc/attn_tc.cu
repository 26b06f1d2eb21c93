// Tree-masked GQA attention on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory), for KV heads whose packed query rows fill
// one 128-row tile: R = G * n_query = 128, head_dim 128.  This is the NVIDIA
// draft-length article's tile rule (D = 128 / G - 1, G x (1 + D) a multiple
// of 128); the ancestor mask is the SwiftSpec summary's Figure 3 and the key
// split with a combine its §3.3.
//
// One CTA per SM, 192 threads, warp-specialised:
//   warps 0-3  softmax: thread t owns packed row t = TMEM lane t.  Per 64-key
//              tile it loads its row of S = QK^T from TMEM, applies the scale
//              and the ancestor mask, keeps a lazily-updated running max
//              (O is rescaled in TMEM only when the max grows by more than
//              2^8), writes the probabilities as bf16 into a 128-byte-swizzled
//              shared-memory tile (plus the rounding residual on tiles with
//              tree keys), and at the end of a unit reads O from TMEM and
//              writes the bf16 output or an fp32 split-KV partial;
//   warp 4     TMA producer: Q once per unit (3-D box G x n_query rows), K and
//              V tiles into a 4-stage ring;
//   warp 5     MMA issuer (one lane): S_j = Q K_j^T (M 128, N 64, K 128) into
//              one of two TMEM S buffers, issued one tile ahead, then
//              O += P_j V_j (M 128, N 128, K 64, V read MN-major) into TMEM O;
//              completion is signalled with tcgen05.commit on mbarriers.
// TMEM: 256 columns = S0 [0, 64) | S1 [64, 128) | O [128, 256).
// The split-KV schedule and the in-kernel combine of partials are those of
// the warp-MMA kernel (attn_common.cuh).
#include "attn_common.cuh"
#include "tcgen05.cuh"

namespace ts {
namespace {

constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

struct TcLayout {
  uint32_t q, kv, p_hi, p_lo, ctrl, par, cum, total;
  static constexpr uint32_t kQBytes = 128 * 128 * 2;        // two 64-column halves of 128 rows
  static constexpr uint32_t kKvBytes = 64 * 128 * 2;        // one of K or V: two halves of 64 rows
  static constexpr uint32_t kStageBytes = 2 * kKvBytes;
  static constexpr uint32_t kPBytes = 128 * 64 * 2;         // 128 rows x 64 keys
};

// control block (barriers etc.), after the 1024-aligned tiles
struct TcCtrl {
  uint64_t kv_full[kTcStages], kv_empty[kTcStages];
  uint64_t q_full, q_empty, s_full[2], s_free[2], p_full, o_done, o_free, fin;
  uint32_t tmem_base;
  int abort;
  int merge_flag;
};

__host__ __device__ inline TcLayout tc_layout(int num_req) {
  TcLayout L;
  L.q = 0;
  L.kv = L.q + TcLayout::kQBytes;
  L.p_hi = L.kv + kTcStages * TcLayout::kStageBytes;  // two buffers, alternating tiles
  L.p_lo = L.p_hi + 2 * TcLayout::kPBytes;
  L.ctrl = L.p_lo + TcLayout::kPBytes;
  L.par = L.ctrl + ((sizeof(TcCtrl) + 15) & ~size_t(15));
  L.cum = L.par + TS_MAX_TREE * 4;
  L.total = L.cum + 8 * (num_req + 1);
  return L;
}

__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory"); }

// Position of a CTA in its tile sequence: request, unit within the request,
// tile within the unit, and the K/V ring slot.
struct Cursor {
  int b, uir, tile, P, n, tiles, unit;  // unit: CTA-local unit index
  int st;
  uint32_t phase;
  __device__ void start(const AttnParams& p, int b0, int64_t local) {
    b = b0;
    attn_lengths(p, b, P, n, false);
    tiles = attn_tiles(P + n);
    uir = static_cast<int>(local / tiles);
    tile = static_cast<int>(local % tiles);
    unit = 0;
    st = 0;
    phase = 0;
  }
  __device__ void advance(const AttnParams& p, int units_per_req) {
    if (++st == kTcStages) {
      st = 0;
      ++phase;
    }
    if (++tile == tiles) {
      tile = 0;
      ++unit;
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
};

__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                const __grid_constant__ CUtensorMap vmap,
                                                                const __grid_constant__ CUtensorMap qmap,
                                                                const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const TcLayout L = tc_layout(p.num_req);
  TcCtrl* ctl = reinterpret_cast<TcCtrl*>(smem + L.ctrl);
  int* par = reinterpret_cast<int*>(smem + L.par);
  int64_t* cum = reinterpret_cast<int64_t*>(smem + L.cum);
  volatile int* abort_flag = &ctl->abort;

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const int units_per_req = p.hkv;  // one row group: R == 128

  // ---- schedule (identical to the warp-MMA kernel) and barrier set-up
  for (int b = tid; b < p.num_req; b += blockDim.x) {
    int P, n;
    attn_lengths(p, b, P, n, blockIdx.x == 0);
    cum[b + 1] = static_cast<int64_t>(attn_tiles(P + n)) * units_per_req;
  }
  if (tid == 0) {
    cum[0] = 0;
    ctl->abort = 0;
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&ctl->kv_full[s], 1);
      mbar_init(&ctl->kv_empty[s], 1);
    }
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->s_free[i], kSoftmaxThreads / 32);
    }
    mbar_init(&ctl->p_full, kSoftmaxThreads / 32);
    mbar_init(&ctl->o_done, 1);
    mbar_init(&ctl->o_free, kSoftmaxThreads / 32);
    mbar_init(&ctl->fin, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int b = 0; b < p.num_req; ++b) cum[b + 1] += cum[b];
  __syncthreads();
  const int64_t T = cum[p.num_req];
  const int64_t t_begin = sched_begin(blockIdx.x, T, p.num_ctas);
  const int64_t t_end = sched_begin(blockIdx.x + 1, T, p.num_ctas);
  if (t_begin >= t_end) return;
  const int n_tiles = static_cast<int>(t_end - t_begin);
  int b0 = 0;
  {
    int lo = 0, hi = p.num_req - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (cum[mid] <= t_begin) lo = mid; else hi = mid - 1;
    }
    b0 = lo;
  }
  const int64_t local0 = t_begin - cum[b0];

  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;

  if (warp == kProducerWarp) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      prefetch_tmap(&qmap);
      Cursor c;
      c.start(p, b0, local0);
      int issued = 0, q_issued = 0;
      bool ok = true;
      for (int it = 0; it < n_tiles && ok; ++it) {
        if (it == 0 || c.tile == 0) {
          if (c.unit > 0 && !mbar_wait(&ctl->q_empty, (c.unit - 1) & 1)) { ok = false; break; }
          const int kvh = c.uir;
          mbar_arrive_expect_tx(&ctl->q_full, TcLayout::kQBytes);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(smem + L.q + h * (TcLayout::kQBytes / 2), &qmap, h * 64, kvh * p.group, c.b * p.n_query,
                        &ctl->q_full);
          ++q_issued;
        }
        if (it >= kTcStages && !mbar_wait(&ctl->kv_empty[c.st], (c.phase - 1) & 1)) { ok = false; break; }
        uint8_t* ks = smem + L.kv + c.st * TcLayout::kStageBytes;
        uint8_t* vs = ks + TcLayout::kKvBytes;
        const int kvh = c.uir;
        const int key0 = c.tile * kBlockN;
        mbar_arrive_expect_tx(&ctl->kv_full[c.st], TcLayout::kStageBytes);
        if (!p.paged) {
          const int row = c.b * p.max_kv_len + key0;
          for (int h = 0; h < 2; ++h) {
            tma_load_3d(ks + h * (TcLayout::kKvBytes / 2), &kmap, h * 64, kvh, row, &ctl->kv_full[c.st]);
            tma_load_3d(vs + h * (TcLayout::kKvBytes / 2), &vmap, h * 64, kvh, row, &ctl->kv_full[c.st]);
          }
        } else {
          const int pages = kBlockN / p.page_size;
          const int keys = c.P + c.n;
          for (int pg = 0; pg < pages; ++pg) {
            const int lb = key0 / p.page_size + pg;
            int row = p.num_blocks * p.page_size;  // past the pool: TMA fills zeros
            if (lb * p.page_size < keys) {
              const int blk = p.block_table[static_cast<int64_t>(c.b) * p.max_blocks + lb];
              if (blk >= 0 && blk < p.num_blocks) row = blk * p.page_size;
              else report_error(p.err, TS_DEVERR_BAD_BLOCK);
            }
            const uint32_t off = static_cast<uint32_t>(pg * p.page_size) * 128u;
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(ks + h * (TcLayout::kKvBytes / 2) + off, &kmap, h * 64, kvh, row, &ctl->kv_full[c.st]);
              tma_load_3d(vs + h * (TcLayout::kKvBytes / 2) + off, &vmap, h * 64, kvh, row, &ctl->kv_full[c.st]);
            }
          }
        }
        ++issued;
        c.advance(p, units_per_req);
      }
      if (!ok) {
        report_error(p.err, TS_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (*abort_flag) {
        // never leave with copies into this CTA's shared memory in flight
        for (int st = 0; st < kTcStages && st < issued; ++st) {
          const int last = issued - 1 - ((issued - 1 - st) % kTcStages);
          mbar_wait(&ctl->kv_full[st], static_cast<uint32_t>((last / kTcStages) & 1));
        }
        if (q_issued > 0) mbar_wait(&ctl->q_full, static_cast<uint32_t>((q_issued - 1) & 1));
      }
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, true);
      const uint32_t sq = smem_u32(smem + L.q);
      const uint32_t skv = smem_u32(smem + L.kv);
      const uint32_t sph = smem_u32(smem + L.p_hi);
      const uint32_t spl = smem_u32(smem + L.p_lo);
      Cursor cq, cp;  // the QK^T cursor runs one tile ahead of the PV cursor
      cq.start(p, b0, local0);
      cp.start(p, b0, local0);
      bool ok = true;
      auto issue_qk = [&](int j) -> bool {
        if (j == 0 || cq.tile == 0) {
          if (!mbar_wait(&ctl->q_full, cq.unit & 1)) return false;
        }
        if (!mbar_wait(&ctl->kv_full[cq.st], cq.phase & 1)) return false;
        if (j >= 2 && !mbar_wait(&ctl->s_free[j & 1], ((j >> 1) - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t ks = skv + cq.st * TcLayout::kStageBytes;
        const uint32_t d_tmem = tbase + (j & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t half = kk >> 2, off = (kk & 3) * 32;
          tc_mma_bf16(d_tmem, smem_desc_sw128(sq + half * (TcLayout::kQBytes / 2) + off, 16, 1024),
                      smem_desc_sw128(ks + half * (TcLayout::kKvBytes / 2) + off, 16, 1024), kIdescS, kk > 0);
        }
        tc_commit(&ctl->s_full[j & 1]);
        if (cq.tile == cq.tiles - 1 || j == n_tiles - 1) tc_commit(&ctl->q_empty);
        cq.advance(p, units_per_req);
        return true;
      };
      ok = issue_qk(0);
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (j + 1 < n_tiles && !(ok = issue_qk(j + 1))) break;
        if (!mbar_wait(&ctl->p_full, j & 1)) { ok = false; break; }
        tc_fence_after();
        const bool unit_first = (j == 0) || (cp.tile == 0);
        if (unit_first && cp.unit > 0) {
          if (!mbar_wait(&ctl->o_free, (cp.unit - 1) & 1)) { ok = false; break; }
          tc_fence_after();
        }
        const bool tree_tile = cp.tile * kBlockN + kBlockN > cp.P;
        const uint32_t vs = skv + cp.st * TcLayout::kStageBytes + TcLayout::kKvBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(tbase + kColO, smem_desc_sw128(sph + (j & 1) * TcLayout::kPBytes + kk * 32, 16, 1024),
                      smem_desc_sw128(vs + kk * 2048, TcLayout::kKvBytes / 2, 1024), kIdescPV,
                      (unit_first && kk == 0) ? 0u : 1u);
        if (tree_tile) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(tbase + kColO, smem_desc_sw128(spl + kk * 32, 16, 1024),
                        smem_desc_sw128(vs + kk * 2048, TcLayout::kKvBytes / 2, 1024), kIdescPV, 1u);
        }
        tc_commit(&ctl->o_done);
        tc_commit(&ctl->kv_empty[cp.st]);
        cp.advance(p, units_per_req);
      }
      if (!ok) {
        report_error(p.err, TS_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // every MMA this thread issued has completed before TMEM is released
      tc_commit(&ctl->fin);
      mbar_wait(&ctl->fin, 0);
    }
  } else {
    // ======================= softmax / epilogue (rows) =======================
    const int r = tid;  // packed row = TMEM lane
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    uint8_t* sph = smem + L.p_hi;
    uint8_t* spl = smem + L.p_lo;
    Cursor c;
    c.start(p, b0, local0);
    int seg_first = c.tile;
    int anc_req = -1;
    uint32_t anc[4] = {0, 0, 0, 0};
    float m_used = -INFINITY, l = 0.f;
    for (int it = 0; it < n_tiles; ++it) {
      const bool unit_first = (it == 0) || (c.tile == 0);
      if (unit_first) {
        if (anc_req != c.b) {
          softmax_sync();  // every row has finished with the previous parent copy
          for (int i = r; i < c.n; i += kSoftmaxThreads) {
            int q = p.parent[static_cast<int64_t>(c.b) * p.n_tree_max + i];
            if (q < -1 || q >= i) {
              if (blockIdx.x == 0) report_error(p.err, TS_DEVERR_BAD_PARENT);
              q = -1;
            }
            par[i] = q;
          }
          softmax_sync();
          anc_req = c.b;
        }
        ancestor_walk(par, c.n - p.n_query + r / p.group, anc);
        m_used = -INFINITY;
        l = 0.f;
      }
      if (*abort_flag || !mbar_wait(&ctl->s_full[it & 1], (it >> 1) & 1)) {
        report_error(p.err, TS_DEVERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      float x[64];
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(lane_addr + (it & 1) * 64, v0);
        tmem_ld32(lane_addr + (it & 1) * 64 + 32, v1);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          x[e] = __uint_as_float(v0[e]);
          x[32 + e] = __uint_as_float(v1[e]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_free[it & 1]);

      // ---- ancestor mask (tiles holding tree keys only), running max in log2 units
      const int key0 = c.tile * kBlockN;
      const bool tree_tile = key0 + kBlockN > c.P;
      if (tree_tile) {
        const uint64_t vis = tile_visibility(anc, key0 - c.P);
#pragma unroll
        for (int e = 0; e < 64; ++e) x[e] = ((vis >> e) & 1ull) ? x[e] : -INFINITY;
      }
      // eight independent partial maxima keep the dependency chain short
      float pm[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) pm[q] = x[q];
#pragma unroll
      for (int e = 8; e < 64; ++e) pm[e & 7] = fmaxf(pm[e & 7], x[e]);
      const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                             fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      const float mxs = mx * p.scale_log2;  // scale > 0, so the max commutes with it
      float alpha = 1.f;
      bool rescale = false;
      if (m_used == -INFINITY) {
        m_used = mxs;  // O and l hold nothing for this row yet
      } else if (mxs > m_used + kRescaleThreshold) {
        alpha = ex2_approx(m_used - mxs);
        m_used = mxs;
        rescale = !unit_first;
      }
      const float nbase = (m_used == -INFINITY) ? 0.f : -m_used;

      // PV of the previous tile must be complete before O is rescaled or the
      // single residual tile is rewritten.  The bf16 P tile alternates between
      // two buffers: PV of tile it-2 had completed before S of tile it was
      // signalled, so it is written without waiting.  Completion of PV it-1 is
      // confirmed in every iteration before P of tile it is released, so the
      // o_done parity waits never fall two phases behind.
      const bool need_rescale = __any_sync(0xffffffffu, rescale);
      bool pv_prev_done = (it == 0);
      if (!pv_prev_done && (need_rescale || tree_tile)) {
        if (!mbar_wait(&ctl->o_done, (it - 1) & 1)) {
          report_error(p.err, TS_DEVERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        pv_prev_done = true;
      }
      if (need_rescale) {
        const float a = rescale ? alpha : 1.f;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tmem_ld32(lane_addr + kColO + ch * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
          tmem_st32(lane_addr + kColO + ch * 32, v);
        }
        tmem_st_wait();
      }

      // ---- probabilities 2^(s*scale - m) -> bf16 P tile (row r, 128-byte swizzled),
      //      plus the bf16 rounding residual on tiles holding tree keys
      float ps[4] = {0.f, 0.f, 0.f, 0.f};  // partial row sums
      uint8_t* prow = sph + (it & 1) * TcLayout::kPBytes;
#pragma unroll
      for (int ck = 0; ck < 8; ++ck) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float e0 = ex2_approx(fmaf(x[8 * ck + 2 * q], p.scale_log2, nbase));
          const float e1 = ex2_approx(fmaf(x[8 * ck + 2 * q + 1], p.scale_log2, nbase));
          ps[q] += e0 + e1;
          hi[q] = pack_bf16x2(e0, e1);
          if (tree_tile) lo[q] = bf16x2_residual(hi[q], e0, e1);
        }
        const uint32_t off = sw128(r, ck);
        *reinterpret_cast<uint4*>(prow + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (tree_tile) *reinterpret_cast<uint4*>(spl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      // rows past the last key may hold anything; their probability is 0 but
      // 0 * NaN is NaN, so zero them in the V tile before PV reads it
      const int keys = c.P + c.n;
      if (key0 + kBlockN > keys) {
        uint8_t* vs = smem + L.kv + c.st * TcLayout::kStageBytes + TcLayout::kKvBytes;
        const int first = keys - key0;
        const int nvec = (kBlockN - first) * 8;
        for (int h = 0; h < 2; ++h)
          for (int xv = r; xv < nvec; xv += kSoftmaxThreads)
            reinterpret_cast<uint4*>(vs + h * (TcLayout::kKvBytes / 2) + first * 128)[xv] = make_uint4(0, 0, 0, 0);
      }
      if (!pv_prev_done && !mbar_wait(&ctl->o_done, (it - 1) & 1)) {
        report_error(p.err, TS_DEVERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full);

      // ---- end of a unit segment: O from TMEM -> output or partial
      const bool last_of_cta = (it + 1 == n_tiles);
      if (c.tile == c.tiles - 1 || last_of_cta) {
        if (!mbar_wait(&ctl->o_done, it & 1)) {
          report_error(p.err, TS_DEVERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int kvh = c.uir;
        const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
        const bool complete = (seg_first == 0) && (c.tile == c.tiles - 1);
        const int i = r / p.group, h = kvh * p.group + r % p.group;
        const int64_t unit = static_cast<int64_t>(c.b) * units_per_req + c.uir;
        const int64_t slot = static_cast<int64_t>(blockIdx.x) + unit;
        __nv_bfloat16* orow = p.out + ((static_cast<int64_t>(c.b) * p.n_query + i) * p.hq + h) * 128;
        float* prow = p.part_o + (slot * 128 + r) * 128;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tmem_ld32(lane_addr + kColO + ch * 32, v);
          tmem_ld_wait();
          if (complete) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]) * inv, __uint_as_float(v[8 * q + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv);
              reinterpret_cast<uint4*>(orow + ch * 32)[q] = w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<float4*>(prow + ch * 32)[q] =
                  make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                              __uint_as_float(v[4 * q + 2]) * inv, __uint_as_float(v[4 * q + 3]) * inv);
          }
        }
        const float lse2 = l > 0.f ? m_used + log2f(l) : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->o_free);  // O has been read: the next unit's PV may overwrite it
        if (complete) {
          if (p.lse != nullptr)
            p.lse[(static_cast<int64_t>(c.b) * p.hq + h) * p.n_query + i] = lse2 * 0.69314718055994530942f;
        } else {
          p.part_lse[slot * 128 + r] = lse2;
          const int64_t first = cum[c.b] + static_cast<int64_t>(c.uir) * c.tiles;
          if (split_arrive(p, unit, T, first, c.tiles, r, &ctl->merge_flag, softmax_sync))
            // the residual P tile is idle here (PV of this tile is done, the
            // next P is not yet released): it holds the merge weights
            merge_unit_rows(p, unit, c.b, kvh, 0, T, first, c.tiles, r, kSoftmaxThreads,
                            reinterpret_cast<float*>(spl), TcLayout::kPBytes / 4, softmax_sync);
        }
        seg_first = 0;
      }
      c.advance(p, units_per_req);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

bool attn_tc_available() { return true; }

size_t attn_tc_smem_bytes(int /*stages*/, int num_req) { return tc_layout(num_req).total + 1024; }

int attn_tc_threads() { return kTcThreads; }

int attn_tc_occupancy(int stages, int num_req) {
  int nb = 0;
  const size_t smem = attn_tc_smem_bytes(stages, num_req);
  if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, attn_tc_kernel, kTcThreads, smem) != cudaSuccess) return 0;
  return nb;
}

cudaError_t launch_attn_tc(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& qmap, cudaStream_t stream) {
  const size_t smem = attn_tc_smem_bytes(p.stages, p.num_req);
  cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  attn_tc_kernel<<<p.num_ctas, kTcThreads, smem, stream>>>(kmap, vmap, qmap, p);
  return cudaGetLastError();
}

}  // namespace ts
