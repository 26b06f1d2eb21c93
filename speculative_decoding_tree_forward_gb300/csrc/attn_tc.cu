// Tree-masked GQA attention on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory), for KV heads whose packed query rows fit
// one 128-row tile: R = G * n_query <= 128, head_dim 128.  Rows R..127 of the
// tile are padding: an M = 128 instruction costs the same for any R, and the
// kernel is bound by the K/V stream, not by the tensor pipe.  This is the NVIDIA
// draft-length article's tile rule (D = 128 / G - 1, G x (1 + D) a multiple
// of 128); the ancestor mask is the SwiftSpec summary's Figure 3 and the key
// split with a combine its §3.3.
//
// One CTA per SM, 384 threads, warp-specialised:
//   warps 0-3 and 4-7  two softmax warpgroups.  Tile k of the CTA's range
//              belongs to warpgroup k % 2; thread t of a warpgroup owns
//              packed row t (TMEM lane t).  Per 64-key tile it reads its row
//              of S = QK^T from TMEM, applies the scale and the ancestor mask,
//              keeps a lazily-updated running max (its O is rescaled in TMEM
//              only when the max grows by more than 2^8), and writes the
//              probabilities as bf16 pairs over the S they came from (plus
//              the bf16 rounding residual on tiles that hold tree keys).  Each
//              warpgroup keeps its own O, max and sum; at the end of a unit
//              segment the warpgroup that owns its last tile combines both and
//              writes the bf16 output or an fp32 split-KV partial (merged
//              afterwards by the combine kernel, attn_merge.cu).
//   warps 8, 11  TMA producers: warp 8 loads Q once per unit (3-D box
//              G x n_query rows, into one of two Q buffers) and the K tiles
//              into a 4-slot ring (slots 2i and 2i + 1 form one 128-row
//              operand); warp 11 loads the V
//              tiles, tile k into V slot 2 b + w of its S/P buffer (b, w)
//              below.  A K slot is refilled as soon as the S that read it is
//              computed, without queueing behind a V slot.  Tile k uses S/P
//              buffer b = (k / 2) % 2 of warpgroup w = k % 2.
//   warp 9     QK^T issuer (one lane): S = Q K^T (M 128, K 128, both
//              operands in shared memory) for two consecutive tiles of one
//              unit as one N = 128 product, else N = 64 for a single tile.
//              An M = 128 instruction costs about the same at N = 64 as at
//              N = 128, so pairing halves the tensor time of QK^T.
//   warp 10    PV issuer (one lane): O_w += P_k V_k (M 128, N 128, K 64; P
//              from TMEM, V read MN-major from shared memory).
//              The two issuers run on different schedulers, so the waits and
//              commits of one do not leave the tensor pipe idle while the
//              other has work.  Completion is signalled with tcgen05.commit:
//              per S/P buffer one "S ready" and one "PV done" barrier (its P
//              buffer and V slot are then free, O is up to date), and per K
//              slot one "K slot free" barrier.
// TMEM (512 columns): S buffers [0,256), buffer b of warpgroup w at column
// 128 b + 64 w (S as fp32; then, per 32-key chunk j, P as bf16 pairs in
// columns 32 j .. 32 j + 15 and the P residual in 32 j + 16 .. 32 j + 31) |
// O0 [256,384) | O1 [384,512).
// Every mbarrier wait waits for a phase at most one ahead of the last phase
// the same thread confirmed, so the parity waits are never ambiguous.
#include "attn_common.cuh"
#include "tcgen05.cuh"

namespace ts {
namespace {

constexpr int kMaxVSlots = 4;  // V slots (one per S/P buffer)
constexpr int kMaxKSlots = 4;  // K slots
constexpr int kMaxQBufs = 2;   // Q buffers (unit u uses buffer u % kQBufs)
constexpr int kTcThreads = 384;
constexpr int kRowsTc = 128;
constexpr int kProducerWarp = 8;  // Q and K
constexpr int kQkWarp = 9;
constexpr int kPvWarp = 10;
constexpr int kVProducerWarp = 11;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

__host__ __device__ constexpr uint32_t col_o(int w) { return 256u + 128u * w; }

// Shape of the pipeline for HP KV heads per unit.  HP = 1: a tile is 64 keys
// of one head; each warpgroup has two 64-column S/P buffers (tile k of
// warpgroup w = k % 2 uses buffer (k / 2) % 2 and V slot k % 4); K lives in
// four 16 KB slots, two adjacent slots forming the 128-row operand of a tile
// pair; two Q buffers, so the next unit's Q loads while the current unit's
// last tiles are computed.  HP = 2 (packed rows R <= 64, two adjacent KV
// heads share one CTA):
// a tile is 64 keys of both heads, loaded as one TMA box per page-half (keys
// interleaved by head: shared-memory row 2 key + head); each warpgroup has one
// 128-column S/P buffer; K lives in two 32 KB slots and V in three (a V slot
// is then released by its own barrier rather than with its S/P buffer, and
// the extra slot lets V loads run further ahead of the PVs that need them).
template <int HP>
struct TcShape {
  static constexpr int kQBufs = HP == 1 ? 2 : 1;
  static constexpr int kKSlots = HP == 1 ? 4 : 2;
  static constexpr int kVSlots = HP == 1 ? 4 : 3;     // slot of tile k is k % kVSlots
  static constexpr bool kVTied = HP == 1;             // V slot k % 4 = the S/P buffer of tile k
  static constexpr int kSBufs = HP == 1 ? 4 : 2;      // S/P buffers in all: tile k reuses tile k - kSBufs's
  static constexpr uint32_t kKBytes = HP == 1 ? 4u * 16384u : 2u * 32768u;
  static constexpr uint32_t kTileBytes = 64u * 128u * 2u * HP;  // one K or V tile (two 64-column halves)
  static constexpr uint32_t kHalfRows = 64u * HP;    // shared-memory rows of one half of a tile
  __device__ static uint32_t col_s(int w, int b) { return HP == 1 ? 128u * b + 64u * w : 128u * w; }
  __device__ static int buf(int k) { return HP == 1 ? (k >> 1) & 1 : 0; }
  __device__ static int use(int k) { return HP == 1 ? k >> 2 : k >> 1; }  // earlier tiles in the same buffer
  // half h (columns 64 h .. 64 h + 63) of the K tile in slot s; for HP = 1
  // the pair region holds each half as 128 rows, tile 2i in rows 0-63 and
  // tile 2i + 1 in 64-127
  __device__ static uint32_t k_half_off(int s, int h) {
    return HP == 1 ? static_cast<uint32_t>((s >> 1) * 32768 + h * 16384 + (s & 1) * 8192)
                   : static_cast<uint32_t>(s * 32768 + h * 16384);
  }
  __device__ static uint32_t v_half_off(int s, int h) {
    return static_cast<uint32_t>(s * kTileBytes + h * (kTileBytes / 2));
  }
  // packed row r of the tile: head within the unit and row within the head
  __device__ static int head_of(int r) { return HP == 1 ? 0 : r >> 6; }
  __device__ static int local_of(int r) { return HP == 1 ? r : r & 63; }
};

struct TcLayout {
  uint32_t q, k, v, ctrl, par, xch, cum, lenp, lenn, rope, stg, total;
  static constexpr uint32_t kStgWarpBytes = 32 * 128;  // 32 rows x 128 bytes, 128-byte swizzle
  static constexpr uint32_t kQBytes = 128 * 128 * 2;   // two 64-column halves of 128 rows
  static constexpr uint32_t kQKVBytes = 192 * 1024;    // Q buffers + K ring + V ring (split per HP)
};

struct TcCtrl {
  uint64_t k_full[kMaxKSlots], k_empty[kMaxKSlots], v_full[kMaxVSlots], v_empty[kMaxVSlots];
  uint64_t q_full[kMaxQBufs], q_empty[kMaxQBufs];  // Q buffer u % kQBufs holds the CTA's u-th unit
  uint64_t q_rot[kMaxQBufs];  // with RoPE: the buffer's queries have been rotated at their tree positions
  uint64_t s_full[2][2], p_full[2][2], pv_done[2][2];  // per (warpgroup, S/P buffer)
  uint64_t o_free[2], xch_full[2], fin_qk, fin_pv;
  uint64_t stg_free;  // one phase per complete mid-range segment: its finisher's staging tiles are free again
  int64_t t_begin, t_end, local0;  // the CTA's tile range and its offset in request b0
  int b0;
  uint32_t tmem_base;
  int abort;
};

// q_bufs, k_bytes: TcShape<HP>::kQBufs and kKBytes (the V ring takes the
// rest of the Q/K/V region, whose size is the same for every HP)
__host__ __device__ inline TcLayout tc_layout(int num_req, int q_bufs = 2, uint32_t k_bytes = 4u * 16384u) {
  TcLayout L;
  L.q = 0;
  L.k = L.q + q_bufs * TcLayout::kQBytes;
  L.v = L.k + k_bytes;
  L.ctrl = TcLayout::kQKVBytes;
  L.par = L.ctrl + ((sizeof(TcCtrl) + 15) & ~size_t(15));
  L.xch = L.par + 2 * TS_MAX_TREE * 4;
  L.cum = L.xch + 2 * kRowsTc * 8;
  L.lenp = L.cum + 8 * (kMaxRequestsAttn + 1);  // clamped prefix length of every request
  L.lenn = L.lenp + 4 * kMaxRequestsAttn;       // clamped tree size of every request (<= 128)
  L.rope = L.lenn + kMaxRequestsAttn;           // RoPE frequencies as turn fractions (64 x 8 bytes)
  // epilogue staging: 32 rows x 64 bytes of bf16 output per warp of the
  // finishing warpgroup, 128-byte swizzled, 1024-byte aligned
  L.stg = (L.rope + 64 * 8 + 1023) & ~1023u;
  L.total = L.stg + 4 * TcLayout::kStgWarpBytes;  // fixed: launch shape independent of the batch
  (void)num_req;
  return L;
}

// barrier over the 128 threads of one softmax warpgroup (ids 1 and 2)
__device__ __forceinline__ void wg_sync(int w) {
  if (w == 0) asm volatile("bar.sync 1, 128;" ::: "memory");
  else asm volatile("bar.sync 2, 128;" ::: "memory");
}

// Position of a CTA in its tile sequence: request, unit within the request
// and tile within the unit.
struct Cursor {
  int b, uir, tile, P, n, tiles, unit;  // unit: CTA-local unit index
  int tile0;                            // unit tile at which the CTA's range starts
  const int* lp;                        // clamped lengths of every request (shared memory)
  const uint8_t* ln;
  __device__ void start(const int* lp_, const uint8_t* ln_, int b0, int64_t local) {
    lp = lp_;
    ln = ln_;
    b = b0;
    P = lp[b];
    n = ln[b];
    tiles = attn_tiles(P + n);
    uir = static_cast<int>(local / tiles);
    tile = static_cast<int>(local - static_cast<int64_t>(uir) * tiles);
    tile0 = tile;
    unit = 0;
  }
  __device__ void advance(const AttnParams& p, int units_per_req) {
    if (++tile == tiles) {
      tile = 0;
      ++unit;
      if (++uir == units_per_req) {
        uir = 0;
        ++b;
        if (b < p.num_req) {
          P = lp[b];
          n = ln[b];
          tiles = attn_tiles(P + n);
        }
      }
    }
  }
  // CTA-local index of the first / last tile of the segment (the CTA's tiles
  // of one unit) that tile k belongs to, and whether it covers the whole unit
  __device__ int seg_first(int k) const { return k - (tile - (unit == 0 ? tile0 : 0)); }
  __device__ int seg_last(int k, int n_tiles) const { return min(n_tiles - 1, k + tiles - 1 - tile); }
  __device__ bool seg_complete(int k, int n_tiles) const {
    return (unit > 0 || tile0 == 0) && (k + tiles - 1 - tile) <= n_tiles - 1;
  }
};

// Pages per 64-key tile at the smallest supported page size (16 rows).
constexpr int kMaxPagesPerTile = kBlockN / 16;

// Block-table entries of the cursor's tile for paged K/V: the row of each
// page in the pool, or one past the pool (the TMA unit fills zeros there)
// for pages past the request's keys or with an invalid block id.  The loads
// are independent, so they overlap; the producer issues them one tile ahead.
__device__ __forceinline__ void tile_pages(const AttnParams& p, const Cursor& c, int (&row)[kMaxPagesPerTile]) {
  const int pages = kBlockN / p.page_size;
  const int keys = c.P + c.n;
  const int key0 = c.tile * kBlockN;
#pragma unroll
  for (int pg = 0; pg < kMaxPagesPerTile; ++pg) {
    const int lb = key0 / p.page_size + pg;
    row[pg] = -1;
    if (pg < pages && lb * p.page_size < keys) row[pg] = p.block_table[static_cast<int64_t>(c.b) * p.max_blocks + lb];
  }
}

// Loads one 64-key K or V tile (two 64-column halves) of the cursor's tile,
// from the contiguous cache or page by page (block-table entries `blk` from
// tile_pages).  Rows past the pool or the tensor are filled with zeros by
// the TMA unit.
template <int HP>
__device__ __forceinline__ void load_tile(const AttnParams& p, const Cursor& c, const CUtensorMap* map, uint8_t* dst0,
                                          uint8_t* dst1, uint64_t* bar, const int (&blk)[kMaxPagesPerTile],
                                          uint64_t pol) {
  const int kvh = HP * c.uir;  // first KV head of the unit (the box covers HP heads)
  const int key0 = c.tile * kBlockN;
  if (!p.paged) {
    const int row = c.b * p.max_kv_len + key0;
    tma_load_3d_hint(dst0, map, 0, kvh, row, bar, pol);
    tma_load_3d_hint(dst1, map, 64, kvh, row, bar, pol);
    return;
  }
  const int pages = kBlockN / p.page_size;
  const int keys = c.P + c.n;
#pragma unroll
  for (int pg = 0; pg < kMaxPagesPerTile; ++pg) {
    if (pg >= pages) break;
    const int lb = key0 / p.page_size + pg;
    int row = p.num_blocks * p.page_size;  // past the pool: TMA fills zeros
    if (lb * p.page_size < keys) {
      if (blk[pg] >= 0 && blk[pg] < p.num_blocks) row = blk[pg] * p.page_size;
      else report_error(p.err, TS_DEVERR_BAD_BLOCK);
    }
    const uint32_t off = static_cast<uint32_t>(pg * p.page_size) * 128u * HP;
    tma_load_3d_hint(dst0 + off, map, 0, kvh, row, bar, pol);
    tma_load_3d_hint(dst1 + off, map, 64, kvh, row, bar, pol);
  }
}

// Paged K or V tile: lane l < 2 * pages issues the TMA box of page l / 2,
// half l % 2 (16 rows of HP heads: a 2 KB box per half for one head).
template <int HP>
__device__ __forceinline__ void load_tile_paged_lanes(const AttnParams& p, const Cursor& c, const CUtensorMap* map,
                                                      uint8_t* dst0, uint8_t* dst1, uint64_t* bar,
                                                      const int (&blk)[kMaxPagesPerTile], int lane, uint64_t pol) {
  const int pages = kBlockN / p.page_size;
  if (lane >= 2 * pages) return;
  const int pg = lane >> 1, h = lane & 1;
  const int kvh = HP * c.uir;
  const int key0 = c.tile * kBlockN;
  const int keys = c.P + c.n;
  const int lb = key0 / p.page_size + pg;
  const int b = pg == 0 ? blk[0] : pg == 1 ? blk[1] : pg == 2 ? blk[2] : blk[3];
  int row = p.num_blocks * p.page_size;  // past the pool: TMA fills zeros
  if (lb * p.page_size < keys) {
    if (b >= 0 && b < p.num_blocks) row = b * p.page_size;
    else report_error(p.err, TS_DEVERR_BAD_BLOCK);
  }
  const uint32_t off = static_cast<uint32_t>(pg * p.page_size) * 128u * HP;
  tma_load_3d_hint((h == 0 ? dst0 : dst1) + off, map, h * 64, kvh, row, bar, pol);
}

// Pass 2 of the softmax for one row: P = 2^(s * scale_log2 + nbase) (keys
// whose bit in vis is clear count as -inf on tiles holding tree keys),
// written as bf16 pairs over the S chunks they came from (16 pairs per
// 32-column chunk; the chunk's other 16 columns get the bf16 rounding
// residual on tree tiles); the sum of the fp32 probabilities goes to ps.
// HP = 1: the row's 64 scores sv are in registers; a chunk is keys
// 32 ch .. 32 ch + 31, two keys per pair.
template <bool TREE>
__device__ __forceinline__ void write_p1(const float (&sv)[64], uint64_t vis, float scale_log2, float nbase,
                                         uint32_t sbuf, float (&ps)[4]) {
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = 32 * ch + 2 * q;
      const float s0 = (!TREE || ((vis >> e) & 1ull)) ? sv[e] : -INFINITY;
      const float s1 = (!TREE || ((vis >> (e + 1)) & 1ull)) ? sv[e + 1] : -INFINITY;
      const float x0 = ex2_approx(fmaf(s0, scale_log2, nbase));
      const float x1 = ex2_approx(fmaf(s1, scale_log2, nbase));
      ps[q & 3] += x0 + x1;
      hi[q] = pack_bf16x2(x0, x1);
      if constexpr (TREE) lo[q] = bf16x2_residual(hi[q], x0, x1);
    }
    tmem_st16(sbuf + 32 * ch, hi);
    if constexpr (TREE) tmem_st16(sbuf + 32 * ch + 16, lo);
  }
}
// HP = 2: S is re-read chunk by chunk; chunk ch holds keys 16 ch .. 16 ch + 15
// of both heads (column 2 key + head), and pair q of the chunk is key
// 16 ch + q (V rows 2 key, 2 key + 1) with the other head's half zero.
template <bool TREE>
__device__ __forceinline__ void write_p2(uint64_t vis, float scale_log2, float nbase, int hj, uint32_t sbuf,
                                         float (&ps)[4]) {
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t v[32];
    tmem_ld32(sbuf + 32 * ch, v);
    tmem_ld_wait();
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = 16 * ch + q;
      const float s0 = (!TREE || ((vis >> e) & 1ull)) ? __uint_as_float(hj ? v[2 * q + 1] : v[2 * q]) : -INFINITY;
      const float e0 = ex2_approx(fmaf(s0, scale_log2, nbase));
      ps[q & 3] += e0;
      const float x0 = hj ? 0.f : e0, x1 = hj ? e0 : 0.f;
      hi[q] = pack_bf16x2(x0, x1);
      if constexpr (TREE) lo[q] = bf16x2_residual(hi[q], x0, x1);
    }
    tmem_st16(sbuf + 32 * ch, hi);
    if constexpr (TREE) tmem_st16(sbuf + 32 * ch + 16, lo);
  }
}

// First tile of CTA c under the cost-weighted split (common.cuh): cum[b] =
// tiles before request b, every unit of request b has `tiles` = attn_tiles(P +
// n) tiles (lengths from the shared-memory table), E = the weight a unit's
// first tile carries beyond 1.
__device__ __forceinline__ int64_t wsched_begin(int c, const int64_t* cum, const int* lp, const uint8_t* ln,
                                                int num_req, int upr, int E, int64_t T, int NC) {
  const int64_t W = T + static_cast<int64_t>(E) * upr * num_req;
  const int64_t x = wsched_x(c, W, NC);
  if (x >= W) return T;
  int lo = 0, hi = num_req - 1;  // the request whose weighted range holds x
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (cum[mid] + static_cast<int64_t>(E) * upr * mid <= x) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int tiles = attn_tiles(lp[b] + ln[b]);
  const int64_t span = tiles + E;
  if (span <= 0) return cum[b + 1];
  const int64_t off = x - (cum[b] + static_cast<int64_t>(E) * upr * b);
  const int uir = (off < (1ll << 31)) ? static_cast<int>(static_cast<uint32_t>(off) / static_cast<uint32_t>(span))
                                      : static_cast<int>(off / span);
  if (uir >= upr) return cum[b + 1];
  const int j = wsched_tile_in_unit(off - uir * span, E, tiles);
  return cum[b] + static_cast<int64_t>(uir) * tiles + j;
}

// Waits (bounded) for the last copy issued into each slot of a ring.
__device__ __forceinline__ void drain_ring(uint64_t* full, int slots, int issued) {
  for (int st = 0; st < slots && st < issued; ++st) {
    const int last = issued - 1 - ((issued - 1 - st) % slots);
    mbar_wait(&full[st], static_cast<uint32_t>((last / slots) & 1));
  }
}

template <int HP, bool kBounded>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                const __grid_constant__ CUtensorMap vmap,
                                                                const __grid_constant__ CUtensorMap qmap,
                                                                const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const TcLayout L = tc_layout(p.num_req, TcShape<HP>::kQBufs, TcShape<HP>::kKBytes);
  TcCtrl* ctl = reinterpret_cast<TcCtrl*>(smem + L.ctrl);
  int64_t* cum = reinterpret_cast<int64_t*>(smem + L.cum);
  volatile int* abort_flag = &ctl->abort;

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  using Sh = TcShape<HP>;
  const int units_per_req = p.hkv / HP;  // one row group: HP heads x R <= 128 rows

  // ---- set-up that reads no input, done while the previous kernel in the
  //      stream may still be finishing: barriers, TMEM, tensor maps, and the
  //      Q padding rows (fewer than 128 packed rows: the Q loads fill rows
  //      0 .. R-1 of each head's 128 / HP rows only, so the rest of the Q
  //      buffer is zeroed once, before any copy into it)
  if (tid == 0) {
    ctl->abort = 0;
    for (int s = 0; s < Sh::kKSlots; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < Sh::kVSlots; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    for (int i = 0; i < Sh::kQBufs; ++i) {
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 1);
      mbar_init(&ctl->q_rot[i], 8);  // 8 warp arrivals: both warpgroups (first unit) or one, twice
    }
    for (int i = 0; i < 2; ++i) {
      for (int j = 0; j < 2; ++j) {
        mbar_init(&ctl->s_full[i][j], 1);
        mbar_init(&ctl->p_full[i][j], 4);
        mbar_init(&ctl->pv_done[i][j], 1);
      }
      mbar_init(&ctl->o_free[i], 4);
      mbar_init(&ctl->xch_full[i], 4);
    }
    mbar_init(&ctl->stg_free, 4);
    mbar_init(&ctl->fin_qk, 1);
    mbar_init(&ctl->fin_pv, 1);
    fence_mbar_init();
  }
  if (p.rows < kRowsTc / HP) {
    for (int x = tid; x < Sh::kQBufs * static_cast<int>(TcLayout::kQBytes / 16); x += kTcThreads)
      reinterpret_cast<uint4*>(smem + L.q)[x] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == kQkWarp) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (lane == 0 && warp == kProducerWarp) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&qmap);
  }
  if (lane == 0 && warp == kVProducerWarp) prefetch_tmap(&vmap);
  uint64_t* rope_turn = reinterpret_cast<uint64_t*>(smem + L.rope);
  if (p.rope && tid < 64) rope_turn[tid] = p.rope_turn[tid];

  // ---- the inputs: wait for the previous kernel in the stream
  pdl_wait();
  pdl_launch_dependents();
  // ---- schedule (warp 0): every request's lengths, clamped as every kernel
  //      of the call clamps them, into the shared-memory table; the prefix
  //      sums of the tile counts by warp scans; then the CTA's tile range
  //      (lane 0 its start, lane 1 its end) and the request it starts in.
  int* lenp = reinterpret_cast<int*>(smem + L.lenp);
  uint8_t* lenn = smem + L.lenn;
  if (warp == 0) {
    int64_t run = 0;
    for (int base = 0; base < p.num_req; base += 32) {
      const int b = base + lane;
      int64_t t = 0;
      if (b < p.num_req) {
        int P, n;
        attn_lengths(p, b, P, n, blockIdx.x == 0);
        lenp[b] = P;
        lenn[b] = static_cast<uint8_t>(n);
        t = static_cast<int64_t>(attn_tiles(P + n)) * units_per_req;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += v;
      }
      if (b < p.num_req) cum[b + 1] = run + t;
      run += __shfl_sync(0xffffffffu, t, 31);
    }
    if (lane == 0) cum[0] = 0;
    __syncwarp();
    if (lane < 2) {
      const int64_t x = wsched_begin(blockIdx.x + lane, cum, lenp, lenn, p.num_req, units_per_req, p.seg_cost, run,
                                     p.num_ctas);
      if (lane == 0) {
        int lo = 0, hi = p.num_req - 1;  // the request holding the CTA's first tile
        while (lo < hi) {
          const int mid = (lo + hi + 1) / 2;
          if (cum[mid] <= x) lo = mid; else hi = mid - 1;
        }
        ctl->t_begin = x;
        ctl->b0 = lo;
        ctl->local0 = x - cum[lo];
      } else {
        ctl->t_end = x;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;
  const int64_t t_begin = ctl->t_begin, t_end = ctl->t_end;
  if (t_begin >= t_end) {  // no tiles: release TMEM and leave
    if (warp == kQkWarp) tmem_dealloc(tbase, kTmemCols);
    return;
  }
  const int n_tiles = static_cast<int>(t_end - t_begin);
  const int b0 = ctl->b0;
  const int64_t local0 = ctl->local0;

  if (warp == kProducerWarp || warp == kVProducerWarp) {
    // ======================= K / V producers =======================
    // Lane 0 waits for slots and issues the TMA loads; a paged tile's page
    // boxes are issued by several lanes at once.
    const bool kside = warp == kProducerWarp;
    const CUtensorMap* map = kside ? &kmap : &vmap;
    Cursor c;
    c.start(lenp, lenn, b0, local0);
    int issued = 0, q_issued = 0;
    int blk[kMaxPagesPerTile];
    const uint64_t kv_policy = l2_policy_evict_first();  // K/V rows are read once
    if (p.paged) tile_pages(p, c, blk);
    bool ok = true;
    for (int it = 0; it < n_tiles; ++it) {
      if (kside && (it == 0 || c.tile == 0)) {
        // buffer u % Sh::kQBufs is free once the QK^T of unit u - Sh::kQBufs are done
        const int qb = c.unit % Sh::kQBufs;
        if (lane == 0) {
          ok = c.unit < Sh::kQBufs || pipe_wait<kBounded>(&ctl->q_empty[qb], ((c.unit / Sh::kQBufs) - 1) & 1, p.wait_ns);
          if (ok) {
            mbar_arrive_expect_tx(&ctl->q_full[qb], static_cast<uint32_t>(HP * p.rows) * 256u);
            for (int h = 0; h < 2; ++h)
              for (int j = 0; j < HP; ++j)  // head j of the unit at packed row 64 j
                tma_load_3d(smem + L.q + qb * TcLayout::kQBytes + h * (TcLayout::kQBytes / 2) + j * 8192, &qmap,
                            h * 64, (HP * c.uir + j) * p.group, c.b * p.n_query, &ctl->q_full[qb]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++q_issued;
      }
      const int sl = kside ? it % Sh::kKSlots : it % Sh::kVSlots, w = it & 1, bb = Sh::buf(it);
      // a K slot is free once the S that read it is computed, a V slot once
      // the PV that read it is done (HP = 1: the PV of the previous tile in
      // the same S/P buffer)
      if (lane == 0)
        ok = kside ? (it < Sh::kKSlots || pipe_wait<kBounded>(&ctl->k_empty[sl], ((it / Sh::kKSlots) - 1) & 1, p.wait_ns))
                   : (it < Sh::kVSlots || (Sh::kVTied ? pipe_wait<kBounded>(&ctl->pv_done[w][bb], (Sh::use(it) - 1) & 1, p.wait_ns)
                                                      : pipe_wait<kBounded>(&ctl->v_empty[sl], ((it / Sh::kVSlots) - 1) & 1, p.wait_ns)));
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint64_t* full = kside ? &ctl->k_full[sl] : &ctl->v_full[sl];
      uint8_t* dst0 = smem + (kside ? L.k + Sh::k_half_off(sl, 0) : L.v + Sh::v_half_off(sl, 0));
      uint8_t* dst1 = smem + (kside ? L.k + Sh::k_half_off(sl, 1) : L.v + Sh::v_half_off(sl, 1));
      if (lane == 0) mbar_arrive_expect_tx(full, Sh::kTileBytes);
      if (!p.paged) {
        if (lane == 0) load_tile<HP>(p, c, map, dst0, dst1, full, blk, kv_policy);
      } else {
        __syncwarp();  // the transaction count is armed before any box lands
        load_tile_paged_lanes<HP>(p, c, map, dst0, dst1, full, blk, lane, kv_policy);
      }
      ++issued;
      c.advance(p, units_per_req);
      // next tile's block-table entries: in flight while lane 0 waits for the slot
      if (p.paged && it + 1 < n_tiles) tile_pages(p, c, blk);
    }
    if (!ok && lane == 0) {
      report_error(p.err, TS_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
    __syncwarp();
    if (*abort_flag) {
      // never leave with copies into this CTA's shared memory in flight
      if (lane == 0) {
        drain_ring(kside ? ctl->k_full : ctl->v_full, kside ? Sh::kKSlots : Sh::kVSlots, issued);
        for (int u = max(q_issued - Sh::kQBufs, 0); u < q_issued; ++u)
          mbar_wait(&ctl->q_full[u % Sh::kQBufs], static_cast<uint32_t>((u / Sh::kQBufs) & 1));
      }
    }
  } else if (warp == kQkWarp) {
    // ======================= QK^T issuer =======================
    if (lane == 0) {
      constexpr uint32_t kIdescS1 = idesc_bf16_f32(128, 64, false);
      constexpr uint32_t kIdescS2 = idesc_bf16_f32(128, 128, false);
      const uint64_t qdesc0 = smem_desc_sw128(smem_u32(smem + L.q), 16, 1024);
      const uint32_t sk = smem_u32(smem + L.k);
      Cursor cq;
      cq.start(lenp, lenn, b0, local0);
      bool ok = true;
      for (int k = 0; k < n_tiles;) {
        if (*abort_flag) { ok = false; break; }
        // HP = 1: two consecutive tiles of one unit as one N = 128 product
        const bool pair = HP == 1 && (k & 1) == 0 && k + 1 < n_tiles && cq.tile != cq.tiles - 1;
        const int cnt = pair ? 2 : 1;
        const int qb = cq.unit % Sh::kQBufs;
        // the unit's queries: landed (and, with RoPE, rotated by the softmax
        // warpgroup that owns the unit's first tile)
        if ((k == 0 || cq.tile == 0) &&
            !pipe_wait<kBounded>(p.rope ? &ctl->q_rot[qb] : &ctl->q_full[qb], (cq.unit / Sh::kQBufs) & 1, p.wait_ns)) {
          ok = false;
          break;
        }
        for (int t = k; t < k + cnt && ok; ++t)
          ok = pipe_wait<kBounded>(&ctl->k_full[t % Sh::kKSlots], (t / Sh::kKSlots) & 1, p.wait_ns) &&
               (t < Sh::kSBufs || pipe_wait<kBounded>(&ctl->pv_done[t & 1][Sh::buf(t)], (Sh::use(t) - 1) & 1, p.wait_ns));
        if (!ok) break;
        tc_fence_after();
        // the descriptors of the 8 K-slices differ only in the start address
        // field (bits 0-13, shared-memory byte address >> 4)
        const uint64_t kdesc = smem_desc_sw128(sk + Sh::k_half_off(k % Sh::kKSlots, 0), 16, 1024);
        const uint32_t dst = tbase + Sh::col_s(k & 1, Sh::buf(k));
        const uint32_t idesc = (pair || HP == 2) ? kIdescS2 : kIdescS1;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a_off = ((kk >> 2) * (TcLayout::kQBytes / 2) + (kk & 3) * 32) >> 4;
          const uint32_t b_off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;  // 128-row halves, 16 KB apart
          tc_mma_bf16(dst, qdesc0 + qb * (TcLayout::kQBytes >> 4) + a_off, kdesc + b_off, idesc, kk > 0);
        }
        for (int t = k; t < k + cnt; ++t) {
          tc_commit(&ctl->s_full[t & 1][Sh::buf(t)]);
          tc_commit(&ctl->k_empty[t % Sh::kKSlots]);
        }
        if (cq.tile + cnt - 1 == cq.tiles - 1 || k + cnt == n_tiles) tc_commit(&ctl->q_empty[qb]);
        for (int t = 0; t < cnt; ++t) cq.advance(p, units_per_req);
        k += cnt;
      }
      if (!ok) {
        report_error(p.err, TS_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // every MMA this thread issued has completed before TMEM is released
      tc_commit(&ctl->fin_qk);
      mbar_wait(&ctl->fin_qk, 0);
    }
  } else if (warp == kPvWarp) {
    // ======================= PV issuer =======================
    if (lane == 0) {
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, true);
      const uint32_t sv = smem_u32(smem + L.v);
      Cursor cp;
      cp.start(lenp, lenn, b0, local0);
      int part[2] = {0, 0};  // segments each warpgroup has finished taking part in (o_free phases)
      bool ok = true;
      for (int k = 0; k < n_tiles; ++k) {
        if (*abort_flag) { ok = false; break; }
        const int w = k & 1, bb = Sh::buf(k);
        const int sf = cp.seg_first(k), sl = cp.seg_last(k, n_tiles);
        const bool first_owned = (k - sf) < 2;
        if (!pipe_wait<kBounded>(&ctl->p_full[w][bb], Sh::use(k) & 1, p.wait_ns) ||
            (first_owned && part[w] > 0 && !pipe_wait<kBounded>(&ctl->o_free[w], (part[w] - 1) & 1, p.wait_ns)) ||
            !pipe_wait<kBounded>(&ctl->v_full[k % Sh::kVSlots], (k / Sh::kVSlots) & 1, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool tree_tile = cp.tile * kBlockN + kBlockN > cp.P;
        const uint64_t vdesc =
            smem_desc_sw128(sv + Sh::v_half_off(k % Sh::kVSlots, 0), Sh::kTileBytes / 2, 1024);
        const uint32_t pa = tbase + Sh::col_s(w, bb), dst = tbase + col_o(w);
        // K = 16 shared-memory rows per instruction (8 keys of both heads when HP = 2)
#pragma unroll
        for (int kk = 0; kk < 4 * HP; ++kk)
          tc_mma_bf16_ts(dst, pa + 32 * (kk >> 1) + 8 * (kk & 1), vdesc + ((kk * 2048) >> 4), kIdescPV,
                         (first_owned && kk == 0) ? 0u : 1u);
        if (tree_tile) {
#pragma unroll
          for (int kk = 0; kk < 4 * HP; ++kk)
            tc_mma_bf16_ts(dst, pa + 32 * (kk >> 1) + 16 + 8 * (kk & 1), vdesc + ((kk * 2048) >> 4), kIdescPV, 1u);
        }
        tc_commit(&ctl->pv_done[w][bb]);
        if (!Sh::kVTied) tc_commit(&ctl->v_empty[k % Sh::kVSlots]);
        if (k == sl) {  // segment ends: both warpgroups' participation counts
          ++part[sl & 1];
          if (sl > sf) ++part[(sl & 1) ^ 1];
        }
        cp.advance(p, units_per_req);
      }
      if (!ok) {
        report_error(p.err, TS_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      tc_commit(&ctl->fin_pv);
      mbar_wait(&ctl->fin_pv, 0);
    }
  } else {
    // ======================= softmax warpgroups =======================
    const int wg = warp >> 2;            // 0 or 1
    const int r = tid & (kRowsTc - 1);   // packed row = TMEM lane
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    int* par = reinterpret_cast<int*>(smem + L.par) + wg * TS_MAX_TREE;
    float2* xch = reinterpret_cast<float2*>(smem + L.xch);
    Cursor c;
    c.start(lenp, lenn, b0, local0);
    int nonfin[2] = {0, 0};  // segments in which each warpgroup handed its state to the other
    int stg_idx = 0;         // earlier segments whose epilogue used the shared staging tiles
    int anc_req = -1;
    uint32_t anc[4] = {0, 0, 0, 0};
    float m_used = -INFINITY, l = 0.f;
    if (p.rope) {
      // RoPE of the CTA's first unit by both warpgroups (idle until the
      // first S): each rotates half of the pairs of every packed row,
      // thread r row r at position P + depth, once the queries land
      for (int i = r; i < c.n; i += kRowsTc) {
        int q = p.parent[static_cast<int64_t>(c.b) * p.n_tree_max + i];
        if (q < -1 || q >= i) {
          if (blockIdx.x == 0) report_error(p.err, TS_DEVERR_BAD_PARENT);
          q = -1;
        }
        par[i] = q;
      }
      wg_sync(wg);
      anc_req = c.b;
      if (pipe_wait<kBounded>(&ctl->q_full[0], 0, p.wait_ns)) {
        if (Sh::local_of(r) < p.rows) {
          ancestor_walk(par, c.n - p.n_query + Sh::local_of(r) / p.group, anc);
          const int pos = c.P + __popc(anc[0]) + __popc(anc[1]) + __popc(anc[2]) + __popc(anc[3]) - 1;
#pragma unroll 1
          for (int cc = 4 * wg; cc < 4 * wg + 4; ++cc) {
            uint4* pa = reinterpret_cast<uint4*>(smem + L.q + sw128(r, cc));
            uint4* pb = reinterpret_cast<uint4*>(smem + L.q + TcLayout::kQBytes / 2 + sw128(r, cc));
            uint4 va = *pa, vb = *pb;
            rope_rotate8(va, vb, pos, rope_turn, 8 * cc);
            *pa = va;
            *pb = vb;
          }
        }
        fence_proxy_async_smem();  // the tensor cores read the rotated rows
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->q_rot[0]);
      } else {
        report_error(p.err, TS_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
    for (int k = 0; k < n_tiles; ++k) {
      const int sf = c.seg_first(k), sl = c.seg_last(k, n_tiles);
      if ((k & 1) == wg) {
        const bool first_owned = (k - sf) < 2;
        const bool last_owned = k + 2 > sl;
        if (first_owned) {
          if (anc_req != c.b) {
            wg_sync(wg);  // every row has finished with the previous parent copy
            for (int i = r; i < c.n; i += kRowsTc) {
              int q = p.parent[static_cast<int64_t>(c.b) * p.n_tree_max + i];
              if (q < -1 || q >= i) {
                if (blockIdx.x == 0) report_error(p.err, TS_DEVERR_BAD_PARENT);
                q = -1;
              }
              par[i] = q;
            }
            wg_sync(wg);
            anc_req = c.b;
          }
          if (Sh::local_of(r) < p.rows) {
            ancestor_walk(par, c.n - p.n_query + Sh::local_of(r) / p.group, anc);
          } else {  // padding row: sees no tree key, its output is discarded
#pragma unroll
            for (int w = 0; w < 4; ++w) anc[w] = 0u;
          }
          if (p.rope && k == sf && c.unit > 0) {
            // RoPE of a later unit: the owner of the unit's first tile rotates
            // the unit's queries in shared memory once they land, each thread
            // its own packed row at position P + depth (16-byte chunk cc of the
            // two 64-column halves holds pairs 8 cc .. 8 cc + 7); the QK^T
            // issuer waits for q_rot before the unit's first product
            // Rotations run in unit order: first the previous unit's (whose
            // owner may be the other warpgroup).  That keeps each parity wait
            // below within one phase of its barrier even when this warpgroup
            // owns no tile of the previous unit: once unit u - 1 is rotated,
            // its queries have landed, so q_full[qb] has completed every phase
            // before this unit's, and q_rot[qb] cannot run ahead of this
            // warpgroup, which rotates this unit.
            const int qb = c.unit % Sh::kQBufs;
            if (!pipe_wait<kBounded>(&ctl->q_rot[(c.unit - 1) % Sh::kQBufs],
                                         ((c.unit - 1) / Sh::kQBufs) & 1, p.wait_ns)) {
              report_error(p.err, TS_DEVERR_TIMEOUT);
              *abort_flag = 1;
              break;
            }
            if (!pipe_wait<kBounded>(&ctl->q_full[qb], (c.unit / Sh::kQBufs) & 1, p.wait_ns)) {
              report_error(p.err, TS_DEVERR_TIMEOUT);
              *abort_flag = 1;
              break;
            }
            if (Sh::local_of(r) < p.rows) {
              const int pos = c.P + __popc(anc[0]) + __popc(anc[1]) + __popc(anc[2]) + __popc(anc[3]) - 1;
              uint8_t* q0 = smem + L.q + qb * TcLayout::kQBytes;
#pragma unroll 1
              for (int cc = 0; cc < 8; ++cc) {
                uint4* pa = reinterpret_cast<uint4*>(q0 + sw128(r, cc));
                uint4* pb = reinterpret_cast<uint4*>(q0 + TcLayout::kQBytes / 2 + sw128(r, cc));
                uint4 va = *pa, vb = *pb;
                rope_rotate8(va, vb, pos, rope_turn, 8 * cc);
                *pa = va;
                *pb = vb;
              }
            }
            fence_proxy_async_smem();  // the tensor cores read the rotated rows
            __syncwarp();
            if (lane == 0) mbar_arrive_cnt(&ctl->q_rot[qb], 2);  // one warpgroup stands for both
          }
          m_used = -INFINITY;
          l = 0.f;
        }
        const int bb = Sh::buf(k);
        const uint32_t sbuf = lane_addr + Sh::col_s(wg, bb);
        if (*abort_flag || !pipe_wait<kBounded>(&ctl->s_full[wg][bb], Sh::use(k) & 1, p.wait_ns)) {
          report_error(p.err, TS_DEVERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int key0 = c.tile * kBlockN;
        const bool tree_tile = key0 + kBlockN > c.P;
        const uint64_t vis = tree_tile ? tile_visibility(anc, key0 - c.P) : ~0ull;

        // ---- pass 1: row max over the 64 keys (masked on tiles holding tree
        //      keys; every key of a prefix tile is visible).  The row's 64
        //      scores stay in registers for pass 2: HP = 1 reads S columns
        //      0..63; HP = 2 reads column 2 key + head of this row's head.
        //      (HP = 2 re-reads S in pass 2 instead, chunk by chunk.)
        float sv[HP == 1 ? 64 : 1];
        float mx;
        {
          float pm[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) pm[q] = -INFINITY;
          if constexpr (HP == 1) {
            uint32_t v0[32], v1[32];
            tmem_ld32(sbuf, v0);
            tmem_ld32(sbuf + 32, v1);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              sv[e] = __uint_as_float(v0[e]);
              sv[32 + e] = __uint_as_float(v1[e]);
            }
            if (tree_tile) {
#pragma unroll
              for (int e = 0; e < 64; ++e)
                if ((vis >> e) & 1ull) pm[e & 7] = fmaxf(pm[e & 7], sv[e]);
            } else {
#pragma unroll
              for (int e = 0; e < 64; ++e) pm[e & 7] = fmaxf(pm[e & 7], sv[e]);
            }
          } else {
            const int hj = Sh::head_of(r);
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
              uint32_t v[32];
              tmem_ld32(sbuf + 32 * ch, v);
              tmem_ld_wait();
#pragma unroll
              for (int q = 0; q < 16; ++q) {
                const int e = 16 * ch + q;
                if (!tree_tile || ((vis >> e) & 1ull))
                  pm[q & 7] = fmaxf(pm[q & 7], __uint_as_float(hj ? v[2 * q + 1] : v[2 * q]));
              }
            }
          }
          mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
        }
        const float mxs = mx * p.scale_log2;  // scale > 0, so the max commutes with it
        float alpha = 1.f;
        bool rescale = false;
        if (m_used == -INFINITY) {
          m_used = mxs;  // O and l hold nothing for this row yet
        } else if (mxs > m_used + kRescaleThreshold) {
          alpha = ex2_approx(m_used - mxs);
          m_used = mxs;
          rescale = true;
        }
        const float nbase = (m_used == -INFINITY) ? 0.f : -m_used;

        // O may be rescaled only once every earlier PV into it is done: the
        // last one was this warpgroup's previous tile, k - 2 (a rescale
        // implies a previous tile in this segment)
        const bool need_rescale = __any_sync(0xffffffffu, rescale);
        if (need_rescale) {
          if (!pipe_wait<kBounded>(&ctl->pv_done[wg][Sh::buf(k - 2)], Sh::use(k - 2) & 1, p.wait_ns)) {
            report_error(p.err, TS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const float a = rescale ? alpha : 1.f;
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t v[32];
            tmem_ld32(lane_addr + col_o(wg) + ch * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
            tmem_st32(lane_addr + col_o(wg) + ch * 32, v);
          }
        }

        // ---- pass 2: probabilities 2^(s*scale - m) as bf16 pairs, written over
        //      the S chunk they came from: the chunk's first 16 columns hold P,
        //      the other 16 the bf16 rounding residual (tiles holding tree
        //      keys).  HP = 1: a chunk is keys 32 j .. 32 j + 31, two keys per
        //      pair.  HP = 2: a chunk is keys 16 j .. 16 j + 15, one key per
        //      pair (key k's pair is shared-memory rows 2 k, 2 k + 1 of V),
        //      with the other head's half zero.
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (HP == 1) {
          if (tree_tile) write_p1<true>(sv, vis, p.scale_log2, nbase, sbuf, ps);
          else write_p1<false>(sv, vis, p.scale_log2, nbase, sbuf, ps);
        } else {
          if (tree_tile) write_p2<true>(vis, p.scale_log2, nbase, Sh::head_of(r), sbuf, ps);
          else write_p2<false>(vis, p.scale_log2, nbase, Sh::head_of(r), sbuf, ps);
        }
        tmem_st_wait();
        l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
        // rows past the last key may hold anything; their probability is 0 but
        // 0 * NaN is NaN, so zero them in the V tile before PV reads it
        const int keys = c.P + c.n;
        if (key0 + kBlockN > keys) {
          const int vslot = k % Sh::kVSlots;
          if (!pipe_wait<kBounded>(&ctl->v_full[vslot], (k / Sh::kVSlots) & 1, p.wait_ns)) {  // the tile has landed
            report_error(p.err, TS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          // keys first .. 63 are shared-memory rows HP * first .. 64 HP - 1 of each half
          const int first = HP * (keys - key0);
          const int nvec = (static_cast<int>(Sh::kHalfRows) - first) * 8;
          for (int h = 0; h < 2; ++h)
            for (int xv = r; xv < nvec; xv += kRowsTc)
              reinterpret_cast<uint4*>(smem + L.v + Sh::v_half_off(vslot, h) + first * 128)[xv] = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[wg][bb]);

        // ---- this warpgroup's last tile of the segment
        if (last_owned) {
          if (!pipe_wait<kBounded>(&ctl->pv_done[wg][bb], Sh::use(k) & 1, p.wait_ns)) {
            report_error(p.err, TS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const int fin = sl & 1, oth = fin ^ 1;
          const bool other_in = sl > sf;  // then the other warpgroup owns tile sl - 1
          if (wg != fin) {
            // hand (max, sum) to the finishing warpgroup; it reads this O from TMEM
            xch[wg * kRowsTc + r] = make_float2(m_used, l);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->xch_full[wg]);
          } else {
            float mo = -INFINITY, lo_ = 0.f;
            if (other_in) {
              if (!pipe_wait<kBounded>(&ctl->xch_full[oth], nonfin[oth] & 1, p.wait_ns)) {
                report_error(p.err, TS_DEVERR_TIMEOUT);
                *abort_flag = 1;
                break;
              }
              tc_fence_after();
              const float2 x2 = xch[oth * kRowsTc + r];
              mo = x2.x;
              lo_ = x2.y;
            }
            const float M = fmaxf(m_used, mo);
            const float a_own = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - M);
            const float a_oth = (!other_in || mo == -INFINITY) ? 0.f : ex2_approx(mo - M);
            const float Ls = l * a_own + lo_ * a_oth;
            const float inv = Ls > 0.f ? __frcp_rn(Ls) : 0.f;
            const float f_own = a_own * inv, f_oth = a_oth * inv;
            const bool complete = c.seg_complete(k, n_tiles);
            // packed row r: head HP * unit + head_of(r), query local_of(r) / G
            const int loc = Sh::local_of(r);
            const int i = loc / p.group, h = (HP * c.uir + Sh::head_of(r)) * p.group + loc % p.group;
            const int64_t unit = static_cast<int64_t>(c.b) * units_per_req + c.uir;
            const int64_t slot = static_cast<int64_t>(blockIdx.x) + unit;
            const bool last_seg = sl == n_tiles - 1;
            uint32_t v[32], u[32];
            tmem_ld32(lane_addr + col_o(wg), v);
            if (other_in) tmem_ld32(lane_addr + col_o(oth), u);
            tmem_ld_wait();
            if (complete) {
              // bf16 output: each 32-column chunk of this warp's 32 rows goes
              // through shared memory (128-byte rows, 16-byte chunk c of row r
              // at c ^ (r % 8)) and leaves as whole 64-byte row segments.  The
              // CTA's last segment stages in the V ring, idle by now (every
              // tile has been loaded and its PV is done); other segments share
              // one 4 KB tile per warp, taken in turn by the finishers of
              // consecutive complete segments, which may be different
              // warpgroups.
              const uint32_t stg_step = last_seg ? TcLayout::kStgWarpBytes : 0u;  // between chunks
              const uint32_t stg = last_seg ? L.v + (warp & 3) * 4 * TcLayout::kStgWarpBytes
                                            : L.stg + (warp & 3) * TcLayout::kStgWarpBytes;
              const int row0 = (warp & 3) * 32;
              if (!last_seg && stg_idx > 0 && !pipe_wait<kBounded>(&ctl->stg_free, (stg_idx - 1) & 1, p.wait_ns)) {
                report_error(p.err, TS_DEVERR_TIMEOUT);
                *abort_flag = 1;
                break;
              }
              // chunk ch + 1 is read from TMEM while chunk ch is staged and stored
#pragma unroll 1
              for (int ch = 0; ch < 4; ++ch) {
                uint8_t* const cs = smem + stg + ch * stg_step;
                float o[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  o[e] = __uint_as_float(v[e]) * f_own + (other_in ? __uint_as_float(u[e]) * f_oth : 0.f);
                if (ch < 3) {
                  tmem_ld32(lane_addr + col_o(wg) + (ch + 1) * 32, v);
                  if (other_in) tmem_ld32(lane_addr + col_o(oth) + (ch + 1) * 32, u);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  *reinterpret_cast<uint4*>(cs + sw128(lane, q)) =
                      make_uint4(pack_bf16x2(o[8 * q + 0], o[8 * q + 1]), pack_bf16x2(o[8 * q + 2], o[8 * q + 3]),
                                 pack_bf16x2(o[8 * q + 4], o[8 * q + 5]), pack_bf16x2(o[8 * q + 6], o[8 * q + 7]));
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 4; ++it) {  // 8 rows x 64 bytes per instruction
                  const int rr = it * 8 + (lane >> 2), c4 = lane & 3;
                  const int row = row0 + rr, lrow = Sh::local_of(row);
                  if (lrow >= p.rows) continue;
                  const int ii = lrow / p.group, hh = (HP * c.uir + Sh::head_of(row)) * p.group + lrow % p.group;
                  const uint4 val = *reinterpret_cast<const uint4*>(cs + sw128(rr, c4));
                  reinterpret_cast<uint4*>(p.out + ((static_cast<int64_t>(c.b) * p.n_query + ii) * p.hq + hh) * 128 +
                                           ch * 32)[c4] = val;
                }
                __syncwarp();  // the next chunk rewrites the staging rows
                if (ch < 3) tmem_ld_wait();
              }
              if (!last_seg && lane == 0) mbar_arrive(&ctl->stg_free);
            } else {
              // fp32 partial, written straight from registers: float4 j of
              // row r at ((slot * 32 + j) * 128 + r), so a warp's 32 rows
              // store 512 contiguous bytes per instruction.  No staging and
              // no wait for the stores: both O accumulators are free as soon
              // as the last chunk has been read from TMEM.
              float4* prow = reinterpret_cast<float4*>(p.part_o) + slot * (kRowsTc * 32) + r;
              const bool write_row = loc < p.rows;
#pragma unroll 1
              for (int ch = 0; ch < 4; ++ch) {
                float o[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  o[e] = __uint_as_float(v[e]) * f_own + (other_in ? __uint_as_float(u[e]) * f_oth : 0.f);
                if (ch < 3) {
                  tmem_ld32(lane_addr + col_o(wg) + (ch + 1) * 32, v);
                  if (other_in) tmem_ld32(lane_addr + col_o(oth) + (ch + 1) * 32, u);
                }
                if (write_row) {
#pragma unroll
                  for (int q = 0; q < 8; ++q)
                    __stcg(prow + (ch * 8 + q) * kRowsTc, make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]));
                }
                if (ch < 3) tmem_ld_wait();
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&ctl->o_free[wg]);  // both O accumulators have been read
              if (other_in) mbar_arrive(&ctl->o_free[oth]);
            }
            const float lse2 = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
            if (loc < p.rows) {
              if (complete) {
                if (p.lse != nullptr)
                  p.lse[(static_cast<int64_t>(c.b) * p.hq + h) * p.n_query + i] = lse2 * 0.69314718055994530942f;
              } else {
                __stcg(p.part_lse + slot * 128 + r, lse2);
              }
            }
          }
        }
      }
      if (k == sl && sl > sf) ++nonfin[(sl & 1) ^ 1];  // the non-finishing warpgroup handed over
      if (k == sl && sl != n_tiles - 1 && c.seg_complete(k, n_tiles)) ++stg_idx;
      c.advance(p, units_per_req);
    }
  }

  bulk_wait_all();  // bulk copies issued by this thread have completed
  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

bool attn_tc_available() { return true; }

size_t attn_tc_smem_bytes(int /*stages*/, int num_req) { return tc_layout(num_req).total + 1024; }

int attn_tc_threads() { return kTcThreads; }

int attn_tc_occupancy(int stages, int num_req) {
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 0;
  int nb = 0;
  const size_t smem = attn_tc_smem_bytes(stages, num_req);
  if (smem > static_cast<size_t>(optin)) return 0;
  if (cudaFuncSetAttribute(attn_tc_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess ||
      cudaFuncSetAttribute(attn_tc_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess ||
      cudaFuncSetAttribute(attn_tc_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess ||
      cudaFuncSetAttribute(attn_tc_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, attn_tc_kernel<1, false>, kTcThreads, smem) != cudaSuccess)
    return 0;
  return nb;
}

// The dynamic shared-memory attribute was raised by attn_tc_occupancy, which
// the host plan runs (once per device) before any launch.
cudaError_t launch_attn_tc(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                           cudaStream_t stream) {
  const size_t smem = attn_tc_smem_bytes(p.stages, p.num_req);
  const bool bounded = p.wait_ns < kWaitLimitNs;  // a caller-given bound: the bounded-wait variant
  const dim3 grid(p.num_ctas), block(kTcThreads);
  if (p.hp == 2)
    return bounded ? launch_pdl(attn_tc_kernel<2, true>, grid, block, smem, stream, kmap, vmap, qmap, p)
                   : launch_pdl(attn_tc_kernel<2, false>, grid, block, smem, stream, kmap, vmap, qmap, p);
  return bounded ? launch_pdl(attn_tc_kernel<1, true>, grid, block, smem, stream, kmap, vmap, qmap, p)
                 : launch_pdl(attn_tc_kernel<1, false>, grid, block, smem, stream, kmap, vmap, qmap, p);
}

}  // namespace ts
