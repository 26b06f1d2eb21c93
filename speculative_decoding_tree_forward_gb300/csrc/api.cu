// treespec C ABI: argument validation, workspace layout, TMA descriptors and
// kernel launches.  Every entry point returns synchronously with a ts_status
// and launches its kernels asynchronously on the caller's stream.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace ts {

int attn_mma_occupancy(int head_dim, int stages, int num_req, int rows_pad);
int attn_tc_occupancy(int stages, int num_req);
bool attn_tc_available();

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr uint64_t kWaitLimitNsHost = 2000000000ull;  // the kernels' default bound of a wait (2 s)

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn.store(f, std::memory_order_release);
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// Per-device launch facts, computed once per device and kept for the
// process: SM count and the occupancy of each kernel shape (computing the
// occupancy also raises the kernel's dynamic shared-memory limit, which the
// launches rely on).
struct OccEntry {
  int key;  // (tc ? 1 << 20 : 0) | head_dim << 12 | stages << 7 | rows_pad
  int occ;
};
struct DeviceFacts {
  int sms = 0;
  int n = 0;
  OccEntry e[32];
};
constexpr int kMaxDevices = 64;
std::mutex g_facts_mutex;
DeviceFacts g_facts[kMaxDevices];

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lock(g_facts_mutex);
  if (g_facts[dev].sms == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_facts[dev].sms = sms;
  }
  return g_facts[dev].sms;
}

int cached_occupancy(bool tc, int head_dim, int stages, int rows_pad, int num_req) {
  const int dev = current_device();
  if (dev < 0) return 0;
  const int key = (tc ? 1 << 20 : 0) | head_dim << 12 | stages << 7 | rows_pad;
  std::lock_guard<std::mutex> lock(g_facts_mutex);
  DeviceFacts& f = g_facts[dev];
  for (int i = 0; i < f.n; ++i)
    if (f.e[i].key == key) return f.e[i].occ;
  const int occ = tc ? attn_tc_occupancy(stages, num_req) : attn_mma_occupancy(head_dim, stages, num_req, rows_pad);
  if (occ > 0 && f.n < 32) f.e[f.n++] = OccEntry{key, occ};
  return occ;
}

// ------------------------------------------------------------------ attention plan
struct AttnPlan {
  bool use_tc;
  int rows, row_groups, rows_pad, group, stages, num_ctas, hp, merge_half_warp;
  int64_t units, slots;
  size_t ws_bytes, off_o, off_lse;
};

ts_status validate_attn(const ts_attn_args* a) {
  if (a == nullptr) return TS_ERR_INVALID_ARG;
  if (a->num_requests < 1 || a->num_q_heads < 1 || a->num_kv_heads < 1 || a->n_tree_max < 1 || a->n_query < 1 ||
      a->n_query > a->n_tree_max)
    return TS_ERR_INVALID_ARG;
  if (a->num_q_heads % a->num_kv_heads != 0) return TS_ERR_INVALID_ARG;
  if (a->num_requests > kMaxRequestsAttn) return TS_ERR_UNSUPPORTED;
  if (a->head_dim != 64 && a->head_dim != 128) return TS_ERR_UNSUPPORTED;
  if (a->n_tree_max > TS_MAX_TREE) return TS_ERR_UNSUPPORTED;
  if (a->kv_layout == TS_KV_CONTIGUOUS) {
    if (a->max_kv_len < 1) return TS_ERR_INVALID_ARG;
    if (static_cast<int64_t>(a->num_requests) * a->max_kv_len > INT32_MAX - kBlockN) return TS_ERR_UNSUPPORTED;
  } else if (a->kv_layout == TS_KV_PAGED) {
    if (a->page_size != 16 && a->page_size != 32 && a->page_size != 64) return TS_ERR_UNSUPPORTED;
    if (a->max_blocks_per_req < 1 || a->num_blocks < 1 || a->block_table == nullptr) return TS_ERR_INVALID_ARG;
    if (static_cast<int64_t>(a->num_blocks) * a->page_size > INT32_MAX - kBlockN) return TS_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(a->max_blocks_per_req) * a->page_size > INT32_MAX / 2) return TS_ERR_UNSUPPORTED;
  } else {
    return TS_ERR_INVALID_ARG;
  }
  if (!a->prefix_len || !a->n_tree || !a->parent || !a->q || !a->k_cache || !a->v_cache || !a->out)
    return TS_ERR_INVALID_ARG;
  if (!aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->q, 16) || !aligned(a->out, 16) ||
      !aligned(a->lse, 4))
    return TS_ERR_INVALID_ARG;
  if (a->force_path < 0 || a->force_path > 2 || a->num_ctas < 0) return TS_ERR_INVALID_ARG;
  if (!(a->rope_theta >= 0.f) || std::isinf(a->rope_theta) || (a->rope_theta > 0.f && a->rope_theta <= 1.f))
    return TS_ERR_INVALID_ARG;  // NaN, infinite, or a base that does not decay
  return TS_OK;
}

ts_status plan_attn(const ts_attn_args* a, AttnPlan* pl) {
  ts_status st = validate_attn(a);
  if (st != TS_OK) return st;
  const int group = a->num_q_heads / a->num_kv_heads;
  const int rows = group * a->n_query;
  pl->group = group;
  pl->rows = rows;
  pl->row_groups = (rows + kMaxRowsPerUnit - 1) / kMaxRowsPerUnit;
  pl->rows_pad = rows >= kMaxRowsPerUnit ? kMaxRowsPerUnit : ((rows + 15) / 16) * 16;
  // the tcgen05 kernel takes any R <= 128 as one 128-row tile (padded)
  const bool tc_shape = (rows <= kMaxRowsPerUnit) && a->head_dim == 128;
  if (a->force_path == 2) {
    if (!tc_shape) return TS_ERR_UNSUPPORTED;
    if (!attn_tc_available()) return TS_ERR_UNSUPPORTED;
    pl->use_tc = true;
  } else if (a->force_path == 1) {
    pl->use_tc = false;
  } else {
    pl->use_tc = tc_shape && attn_tc_available();
  }
  // the tcgen05 kernel packs two adjacent KV heads into one 128-row tile when
  // their rows fit (R <= 64): one TMA box then carries both heads' keys
  pl->hp = (pl->use_tc && rows <= kMaxRowsPerUnit / 2 && a->num_kv_heads % 2 == 0) ? 2 : 1;
  if (pl->use_tc) pl->rows_pad = kMaxRowsPerUnit;  // partial rows laid out as the 128-row tile
  pl->units = static_cast<int64_t>(a->num_requests) * (a->num_kv_heads / pl->hp) * pl->row_groups;
  const int max_len = a->kv_layout == TS_KV_PAGED ? a->max_blocks_per_req * a->page_size : a->max_kv_len;
  const int64_t t_max = pl->units * ((max_len + a->n_tree_max + kBlockN - 1) / kBlockN);
  int occ = 1;
  if (pl->use_tc) {
    pl->stages = 4;
    occ = cached_occupancy(true, a->head_dim, pl->stages, pl->rows_pad, a->num_requests);
  } else {
    const int rb = pl->rows_pad / 16;
    if (a->head_dim == 128) pl->stages = rb <= 4 ? 3 : 5;
    else pl->stages = rb <= 4 ? 6 : 10;
    occ = cached_occupancy(false, a->head_dim, pl->stages, pl->rows_pad, a->num_requests);
  }
  if (occ < 1) return TS_ERR_UNSUPPORTED;
  if (a->num_ctas > 0) {
    pl->num_ctas = a->num_ctas;
  } else {
    const int sms = device_sm_count();
    if (sms <= 0) return TS_ERR_CUDA;
    int64_t nc = static_cast<int64_t>(sms) * occ;
    if (nc > t_max) nc = t_max;
    // at most one merge round of shares per unit on average: with few units
    // (a draft-side call of one request), more CTAs only split the same
    // tiles into shares the merge reads in a second round (measured on the
    // 8-leaf expansion's calls: 4 units of 34 tiles, 13.6 us per call with
    // 128 CTAs against 14.9 us with one tile per CTA)
    if (pl->use_tc) nc = std::min<int64_t>(nc, static_cast<int64_t>(kMergeSharesPerRound) * pl->units);
    pl->num_ctas = static_cast<int>(nc < 1 ? 1 : nc);
  }
  // The merge runs eight warps per CTA, four CTAs per SM.  One warp per row
  // (eight shares prefetched) while that grid fits one resident wave; past
  // that, one half-warp per row (four prefetched), which keeps twice the rows
  // in flight: a second wave would cost every row of it another round trip.
  pl->merge_half_warp = pl->units * ((pl->rows_pad + 7) / 8) > 4LL * device_sm_count() ? 1 : 0;
  pl->slots = pl->num_ctas + pl->units;
  // [error word][partial O][partial lse]
  pl->off_o = kWsHeader;
  pl->off_lse = pl->off_o + align256(static_cast<size_t>(pl->slots) * pl->rows_pad * a->head_dim * sizeof(float));
  pl->ws_bytes = pl->off_lse + align256(static_cast<size_t>(pl->slots) * pl->rows_pad * sizeof(float));
  return TS_OK;
}

// K or V as a 3-D tensor (head_dim, Hkv, rows); a box is 64 columns of `hp`
// adjacent heads for 64 rows (contiguous) or one page (paged).
bool encode_kv_map(CUtensorMap* map, const void* base, const ts_attn_args* a, int hp) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t rows = a->kv_layout == TS_KV_PAGED
                              ? static_cast<cuuint64_t>(a->num_blocks) * a->page_size
                              : static_cast<cuuint64_t>(a->num_requests) * a->max_kv_len;
  const cuuint32_t box_rows = a->kv_layout == TS_KV_PAGED ? a->page_size : kBlockN;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(a->head_dim), static_cast<cuuint64_t>(a->num_kv_heads), rows};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(a->head_dim) * 2,
                           static_cast<cuuint64_t>(a->head_dim) * 2 * a->num_kv_heads};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(hp), box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Q as a 3-D tensor (head_dim, Hq, num_requests * n_query); one box of
// (64, G, n_query) is the 128 packed rows (node-major, head within the group)
// of one KV head, in two 64-column halves.
bool encode_q_map(CUtensorMap* map, const ts_attn_args* a, const void* q, int group) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(a->head_dim), static_cast<cuuint64_t>(a->num_q_heads),
                        static_cast<cuuint64_t>(a->num_requests) * a->n_query};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(a->head_dim) * 2,
                           static_cast<cuuint64_t>(a->head_dim) * 2 * a->num_q_heads};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(a->n_query)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// Leading workspace bytes that must be zero when a call starts (the error
// word); 0 when the arguments are rejected.
size_t attn_zero_prefix_bytes(const ts_attn_args* a) {
  AttnPlan pl;
  if (plan_attn(a, &pl) != TS_OK) return 0;
  return kWsHeader;
}

}  // namespace ts

using namespace ts;

extern "C" {

int ts_version(void) { return (0 << 16) | 1; }

const char* ts_status_string(ts_status s) {
  switch (s) {
    case TS_OK: return "TS_OK";
    case TS_ERR_INVALID_ARG: return "TS_ERR_INVALID_ARG: invalid argument";
    case TS_ERR_UNSUPPORTED: return "TS_ERR_UNSUPPORTED: shape or option not implemented";
    case TS_ERR_CUDA: return "TS_ERR_CUDA: a CUDA call failed";
    case TS_ERR_WORKSPACE: return "TS_ERR_WORKSPACE: workspace missing, too small or misaligned";
  }
  return "unknown ts_status";
}

ts_status ts_read_device_error(void* workspace, int* code, int clear, void* stream) {
  if (workspace == nullptr || code == nullptr) return TS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return TS_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TS_ERR_CUDA;
  *code = static_cast<int>(v);
  if (clear) {
    if (cudaMemsetAsync(workspace, 0, sizeof(unsigned), st) != cudaSuccess) return TS_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return TS_ERR_CUDA;
  }
  return TS_OK;
}

// ------------------------------------------------------------------ metadata
size_t tree_meta_workspace_size(void) { return kWsHeader; }

ts_status tree_build_mask(const int32_t* parent, const int32_t* n_tree, int num_requests, int n_tree_max,
                          int32_t* depth, uint32_t* anc, void* workspace, size_t workspace_bytes, void* stream) {
  if (!parent || !n_tree || !depth || !anc || num_requests < 1 || n_tree_max < 1) return TS_ERR_INVALID_ARG;
  if (n_tree_max > TS_MAX_TREE) return TS_ERR_UNSUPPORTED;
  if (!aligned(anc, 16)) return TS_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kWsHeader || !aligned(workspace, 256)) return TS_ERR_WORKSPACE;
  cudaError_t e = launch_tree_meta(parent, n_tree, num_requests, n_tree_max, depth, anc,
                                   static_cast<unsigned*>(workspace), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

// ------------------------------------------------------------------ attention
size_t tree_attn_workspace_size(const ts_attn_args* args) {
  AttnPlan pl;
  if (plan_attn(args, &pl) != TS_OK) return 0;
  return pl.ws_bytes;
}

int tree_attn_selected_path(const ts_attn_args* args) {
  AttnPlan pl;
  const ts_status st = plan_attn(args, &pl);
  if (st != TS_OK) return -static_cast<int>(st);
  return pl.use_tc ? 2 : 1;
}

ts_status tree_attn_forward(const ts_attn_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  AttnPlan pl;
  ts_status st = plan_attn(a, &pl);
  if (st != TS_OK) return st;
  if (!workspace || workspace_bytes < pl.ws_bytes || !aligned(workspace, 256)) return TS_ERR_WORKSPACE;
  CUtensorMap kmap, vmap;
  if (!encode_kv_map(&kmap, a->k_cache, a, pl.hp) || !encode_kv_map(&vmap, a->v_cache, a, pl.hp)) return TS_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.num_req = a->num_requests;
  p.hq = a->num_q_heads;
  p.hkv = a->num_kv_heads;
  p.group = pl.group;
  p.head_dim = a->head_dim;
  p.n_query = a->n_query;
  p.n_tree_max = a->n_tree_max;
  p.rows = pl.rows;
  p.hp = pl.hp;
  p.row_groups = pl.row_groups;
  p.rows_pad = pl.rows_pad;
  p.max_kv_len = a->max_kv_len;
  p.paged = a->kv_layout == TS_KV_PAGED;
  p.page_size = p.paged ? a->page_size : 0;
  p.max_blocks = p.paged ? a->max_blocks_per_req : 0;
  p.num_blocks = p.paged ? a->num_blocks : 0;
  p.num_ctas = pl.num_ctas;
  // a segment's epilogue (and the refill after it) costs about 4 tiles of
  // time; a sweep of E = 1..8 on the verify and paged chain workloads
  // measured the best totals at E = 4..6
  p.seg_cost = pl.use_tc ? 4 : 0;
  p.stages = pl.stages;
  p.merge_half_warp = pl.merge_half_warp;
  p.num_units = pl.units;
  p.prefix_len = a->prefix_len;
  p.n_tree = a->n_tree;
  p.parent = a->parent;
  p.q = static_cast<const __nv_bfloat16*>(a->q);
  p.block_table = a->block_table;
  p.out = static_cast<__nv_bfloat16*>(a->out);
  p.lse = a->lse;
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / std::sqrt(static_cast<float>(a->head_dim));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.part_o = reinterpret_cast<float*>(ws + pl.off_o);
  p.part_lse = reinterpret_cast<float*>(ws + pl.off_lse);
  p.wait_ns = a->wait_limit_ns > 0 ? static_cast<uint64_t>(a->wait_limit_ns) : kWaitLimitNsHost;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (a->rope_theta > 0.f) {
    // the kernels rotate the queries at their tree positions as they stage
    // them; each frequency theta^(-2j/d) goes as a 64-bit fraction of a turn
    p.rope = 1;
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    for (int j = 0; j < 64; ++j) {
      const double f = j < a->head_dim / 2 ? std::pow(static_cast<double>(a->rope_theta), -2.0 * j / a->head_dim) : 0.0;
      p.rope_turn[j] = static_cast<uint64_t>(std::ldexp(f / kTwoPi, 64));
    }
  }
  if (pl.use_tc) {
    CUtensorMap qmap;
    if (!encode_q_map(&qmap, a, p.q, pl.group)) return TS_ERR_CUDA;
    e = launch_attn_tc(p, kmap, vmap, qmap, s);
  } else {
    e = launch_attn_mma(p, kmap, vmap, s);
  }
  if (e != cudaSuccess) return TS_ERR_CUDA;
  e = launch_attn_merge(p, pl.use_tc, s);
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

// ------------------------------------------------------------------ acceptance
// Vocab slice per argmax CTA: the scored rows x slices fill one resident wave
// of 256-thread CTAs (eight per SM), each streaming its slice in steps of
// eight 16-byte loads per thread, so the logits stream without a second wave
// of CTA launches.  Slices are multiples of 1024 floats (16-byte aligned).
static int accept_chunk(int vocab, int64_t rows) {
  const int sms = device_sm_count();
  int64_t c = 8192;
  if (sms > 0 && rows > 0) {
    const int64_t slices = std::max<int64_t>(1, static_cast<int64_t>(sms) * 8 / rows);
    c = ((vocab + slices - 1) / slices + 1023) / 1024 * 1024;
  }
  return vocab <= c ? ((vocab + 3) / 4) * 4 : static_cast<int>(c);
}

size_t tree_accept_workspace_size(const ts_accept_args* a) {
  if (a == nullptr || a->num_requests < 1 || a->n_tree_max < 1 || a->vocab < 1) return 0;
  const int64_t rows = static_cast<int64_t>(a->num_requests) * a->n_tree_max;
  const int chunk = accept_chunk(a->vocab, rows);
  const int64_t chunks = (a->vocab + chunk - 1) / chunk;
  return kWsHeader + align256(rows * chunks * sizeof(float)) + align256(rows * chunks * sizeof(int32_t));
}

ts_status tree_accept_greedy(const ts_accept_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  if (a == nullptr || a->num_requests < 1 || a->n_tree_max < 1 || a->vocab < 1) return TS_ERR_INVALID_ARG;
  if (a->n_tree_max > TS_MAX_TREE) return TS_ERR_UNSUPPORTED;
  if (!a->logits || !a->tokens || !a->parent || !a->n_tree || !a->argmax || !a->path || !a->accept_len || !a->bonus)
    return TS_ERR_INVALID_ARG;
  if (!aligned(a->logits, (a->vocab % 4 == 0) ? 16 : 4)) return TS_ERR_INVALID_ARG;
  if (static_cast<int64_t>(a->num_requests) * a->n_tree_max > INT32_MAX) return TS_ERR_UNSUPPORTED;
  const size_t need = tree_accept_workspace_size(a);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return TS_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AcceptParams p;
  p.num_req = a->num_requests;
  p.n_tree_max = a->n_tree_max;
  p.vocab = a->vocab;
  p.chunk = accept_chunk(a->vocab, static_cast<int64_t>(a->num_requests) * a->n_tree_max);
  p.num_chunks = (a->vocab + p.chunk - 1) / p.chunk;
  p.logits = a->logits;
  p.tokens = a->tokens;
  p.parent = a->parent;
  p.n_tree = a->n_tree;
  p.argmax = a->argmax;
  p.path = a->path;
  p.accept_len = a->accept_len;
  p.bonus = a->bonus;
  p.verified = a->verified;
  p.verified_len = a->verified_len;
  p.err = reinterpret_cast<unsigned*>(ws);
  const int64_t rows = static_cast<int64_t>(a->num_requests) * a->n_tree_max;
  p.part_val = reinterpret_cast<float*>(ws + kWsHeader);
  p.part_idx = reinterpret_cast<int32_t*>(ws + kWsHeader + align256(rows * p.num_chunks * sizeof(float)));
  if (p.num_chunks > 65535) return TS_ERR_UNSUPPORTED;
  cudaError_t e = launch_accept(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

// ------------------------------------------------------------------ compaction
size_t tree_compact_workspace_size(const ts_compact_args* a) {
  if (a == nullptr || a->num_requests < 1) return 0;
  return kWsHeader + align256(static_cast<size_t>(a->num_requests) * sizeof(unsigned));
}

}  // extern "C"

// Validates one compaction call and fills its kernel parameters; the CTA
// count per request is sized for `total_requests` requests in the launch.
static ts_status compact_params(const ts_compact_args* a, void* workspace, size_t workspace_bytes, int64_t total_requests,
                                CompactParams& p) {
  if (a == nullptr || a->num_requests < 1 || a->n_tree_max < 1 || a->m_max < 0 || a->num_layers < 1 ||
      a->num_kv_heads < 1 || a->head_dim < 1 || a->elem_bytes < 1)
    return TS_ERR_INVALID_ARG;
  if (a->n_tree_max > TS_MAX_TREE || a->num_requests > 65535) return TS_ERR_UNSUPPORTED;
  const int64_t row_bytes = static_cast<int64_t>(a->num_kv_heads) * a->head_dim * a->elem_bytes;
  if (row_bytes % 16 != 0 || row_bytes > (1 << 20)) return TS_ERR_UNSUPPORTED;
  if (!a->k_layers || !a->v_layers || !a->prefix_len || !a->n_tree || !a->parent || !a->tokens || !a->m ||
      !a->new_prefix_len || !a->new_n_tree || !a->new_parent || !a->new_tokens)
    return TS_ERR_INVALID_ARG;
  if (a->m_max > 0 && a->verified == nullptr) return TS_ERR_INVALID_ARG;
  if (a->kv_layout == TS_KV_CONTIGUOUS) {
    if (a->max_kv_len < 1) return TS_ERR_INVALID_ARG;
  } else if (a->kv_layout == TS_KV_PAGED) {
    if (a->page_size < 1 || a->max_blocks_per_req < 1 || a->num_blocks < 1 || !a->block_table)
      return TS_ERR_INVALID_ARG;
  } else {
    return TS_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(a->num_layers) * a->num_requests > INT32_MAX) return TS_ERR_UNSUPPORTED;
  const size_t need = tree_compact_workspace_size(a);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return TS_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.num_req = a->num_requests;
  p.n_tree_max = a->n_tree_max;
  p.m_max = a->m_max;
  p.num_layers = a->num_layers;
  p.row_bytes = static_cast<int>(row_bytes);
  p.paged = a->kv_layout == TS_KV_PAGED;
  p.max_kv_len = a->max_kv_len;
  p.page_size = a->page_size;
  p.max_blocks = a->max_blocks_per_req;
  p.num_blocks = a->num_blocks;
  // about two CTAs per SM over all requests, each taking a run of
  // (layer, K|V) items; a CTA's vector count stays below 2^31
  const int items = 2 * a->num_layers;
  const int sms = device_sm_count();
  if (sms <= 0) return TS_ERR_CUDA;
  int per_req = static_cast<int>(std::min<int64_t>(items, std::max<int64_t>(1, (2LL * sms + total_requests - 1) /
                                                                                    total_requests)));
  int ipc = (items + per_req - 1) / per_req;
  const int64_t max_item_vecs = static_cast<int64_t>(a->n_tree_max) * (row_bytes / 16);
  ipc = static_cast<int>(std::min<int64_t>(ipc, std::max<int64_t>(1, (INT32_MAX / 2) / max_item_vecs)));
  p.items_per_cta = ipc;
  p.ctas = (items + ipc - 1) / ipc;
  // shared-memory staging: the CTA's largest possible move, at most 96 KB
  const int64_t most = max_item_vecs * ipc;
  p.batch_vecs = static_cast<int>(std::min<int64_t>(most, kCompactBatchBytes / 16));
  p.k_layers = a->k_layers;
  p.v_layers = a->v_layers;
  p.block_table = a->block_table;
  p.prefix_len = a->prefix_len;
  p.n_tree = a->n_tree;
  p.parent = a->parent;
  p.tokens = a->tokens;
  p.verified = a->verified;
  p.m = a->m;
  p.new_prefix_len = a->new_prefix_len;
  p.new_n_tree = a->new_n_tree;
  p.new_parent = a->new_parent;
  p.new_tokens = a->new_tokens;
  p.src_rows = a->src_rows;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.ticket = reinterpret_cast<unsigned*>(ws + kWsHeader);
  return TS_OK;
}

extern "C" {

ts_status tree_cache_compact(const ts_compact_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  if (a == nullptr) return TS_ERR_INVALID_ARG;
  CompactParams p;
  const ts_status st = compact_params(a, workspace, workspace_bytes, a->num_requests, p);
  if (st != TS_OK) return st;
  cudaError_t e = launch_compact(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

ts_status tree_cache_compact_batch(const ts_compact_args* args, int count, void* const* workspaces,
                                   const size_t* workspace_bytes, void* stream) {
  if (args == nullptr || workspaces == nullptr || workspace_bytes == nullptr || count < 1) return TS_ERR_INVALID_ARG;
  if (count > TS_MAX_COMPACT_BATCH) return TS_ERR_UNSUPPORTED;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) {
    if (args[i].num_requests < 1) return TS_ERR_INVALID_ARG;
    total += args[i].num_requests;
  }
  if (total > 65535) return TS_ERR_UNSUPPORTED;
  CompactBatch bt;
  bt.count = count;
  int64_t end = 0;
  for (int i = 0; i < count; ++i) {
    const ts_status st = compact_params(&args[i], workspaces[i], workspace_bytes[i], total, bt.p[i]);
    if (st != TS_OK) return st;
    end += args[i].num_requests;
    bt.req_end[i] = static_cast<int>(end);
  }
  cudaError_t e = launch_compact_batch(bt, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}


// ------------------------------------------------------------------ stochastic acceptance
// Vocab slice per row-statistics CTA (a multiple of 1024 floats): the
// target and draft rows x slices fill about one resident wave, at most 32
// slices per row for the walk's merge.
static int sample_slice(int vocab, int64_t rows) {
  const int sms = device_sm_count();
  int64_t slices = std::min<int64_t>(32, (vocab + 1023) / 1024);
  if (sms > 0 && rows > 0) slices = std::min<int64_t>(slices, std::max<int64_t>(1, static_cast<int64_t>(sms) * 8 / rows));
  slices = std::max<int64_t>(slices, 1);
  return static_cast<int>(((vocab + slices - 1) / slices + 1023) / 1024 * 1024);
}

// CTAs per request in the walk: the SMs shared out among the requests, at
// most kMaxWalkCtas, at least one (the leader alone).
static int sample_walk_ctas(int num_requests) {
  const int sms = device_sm_count();
  if (sms <= 0) return 1;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kMaxWalkCtas, sms / num_requests)));
}

size_t tree_accept_sample_workspace_size(const ts_sample_args* a) {
  if (a == nullptr || a->num_requests < 1 || a->n_tree_max < 1 || a->vocab < 1) return 0;
  const int64_t rows = 2LL * a->num_requests * a->n_tree_max;
  const int slice = sample_slice(a->vocab, rows);
  const int64_t slices = (a->vocab + slice - 1) / slice;
  return kWsHeader + align256(static_cast<size_t>(rows * slices) * sizeof(float2)) +
         align256(static_cast<size_t>(a->num_requests) * sizeof(WalkSync));
}

ts_status tree_accept_sample(const ts_sample_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  if (a == nullptr || a->num_requests < 1 || a->n_tree_max < 1 || a->vocab < 1) return TS_ERR_INVALID_ARG;
  if (!(a->temperature > 0.f) || std::isinf(a->temperature)) return TS_ERR_INVALID_ARG;
  if (a->n_tree_max > TS_MAX_TREE || a->vocab > 262144) return TS_ERR_UNSUPPORTED;
  if (!a->target_logits || !a->draft_logits || !a->tokens || !a->parent || !a->n_tree || !a->u_accept ||
      !a->u_bonus || !a->path || !a->accept_len || !a->bonus)
    return TS_ERR_INVALID_ARG;
  const size_t al = (a->vocab % 4 == 0) ? 16 : 4;
  if (!aligned(a->target_logits, al) || !aligned(a->draft_logits, al)) return TS_ERR_INVALID_ARG;
  const int64_t rows = 2LL * a->num_requests * a->n_tree_max;
  if (rows > INT32_MAX) return TS_ERR_UNSUPPORTED;
  const size_t need = tree_accept_sample_workspace_size(a);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return TS_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SampleParams p;
  p.num_req = a->num_requests;
  p.n_tree_max = a->n_tree_max;
  p.vocab = a->vocab;
  p.slice = sample_slice(a->vocab, rows);
  p.num_slices = (a->vocab + p.slice - 1) / p.slice;
  p.scale2 = static_cast<float>(1.4426950408889634 / static_cast<double>(a->temperature));  // log2(e) / T
  if (!std::isfinite(p.scale2)) return TS_ERR_UNSUPPORTED;
  p.wait_ns = a->wait_limit_ns > 0 ? static_cast<uint64_t>(a->wait_limit_ns) : kWaitLimitNsHost;
  p.tl = a->target_logits;
  p.dl = a->draft_logits;
  p.tokens = a->tokens;
  p.parent = a->parent;
  p.n_tree = a->n_tree;
  p.u_acc = a->u_accept;
  p.u_bonus = a->u_bonus;
  p.path = a->path;
  p.accept_len = a->accept_len;
  p.bonus = a->bonus;
  p.verified = a->verified;
  p.verified_len = a->verified_len;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.part = reinterpret_cast<float2*>(ws + kWsHeader);
  const size_t sync_off = kWsHeader + align256(static_cast<size_t>(rows * p.num_slices) * sizeof(float2));
  p.walk_ctas = sample_walk_ctas(a->num_requests);
  p.sync = reinterpret_cast<WalkSync*>(ws + sync_off);
  cudaError_t e = launch_sample(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

// ------------------------------------------------------------------ draft-side expansion and selection
// Vocab slice per candidate CTA (a multiple of 1024 floats): as many slices
// as keep the SMs busy (about one resident wave of 256-thread CTAs), at most
// 16 per row for the merge.
static int expand_slice(int vocab, int64_t rows) {
  const int sms = device_sm_count();
  int64_t slices = std::min<int64_t>(16, (vocab + 1023) / 1024);
  if (sms > 0 && rows > 0) slices = std::min<int64_t>(slices, std::max<int64_t>(1, static_cast<int64_t>(sms) * 8 / rows));
  slices = std::max<int64_t>(slices, 1);
  return static_cast<int>(((vocab + slices - 1) / slices + 1023) / 1024 * 1024);
}

size_t tree_expand_workspace_size(const ts_expand_args* a) {
  if (a == nullptr || a->num_requests < 1 || a->w < 1 || a->w > TS_MAX_EXPAND || a->vocab < 1) return 0;
  const int64_t rows = static_cast<int64_t>(a->num_requests) * a->w;
  const int slice = expand_slice(a->vocab, rows);
  const int64_t slices = (a->vocab + slice - 1) / slice;
  return kWsHeader + align256(static_cast<size_t>(rows * slices) * sizeof(CandPartial));
}

ts_status tree_expand(const ts_expand_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  if (a == nullptr || a->num_requests < 1 || a->n_tree_max < 1 || a->vocab < 1 || a->w < 1 || a->k < 1)
    return TS_ERR_INVALID_ARG;
  if (a->n_tree_max > TS_MAX_TREE || a->w > TS_MAX_EXPAND || a->k > TS_MAX_EXPAND) return TS_ERR_UNSUPPORTED;
  if (!a->logits || !a->rows || !a->n_tree || !a->parent || !a->tokens || !a->weight || !a->cand_tok ||
      !a->cand_lp || !a->cand_taken || !a->added)
    return TS_ERR_INVALID_ARG;
  if (!aligned(a->logits, (a->vocab % 4 == 0) ? 16 : 4)) return TS_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(a->num_requests) * a->w;
  if (rows > INT32_MAX) return TS_ERR_UNSUPPORTED;
  const size_t need = tree_expand_workspace_size(a);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return TS_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ExpandParams p;
  p.num_req = a->num_requests;
  p.n_tree_max = a->n_tree_max;
  p.vocab = a->vocab;
  p.w = a->w;
  p.k = a->k;
  p.slice = expand_slice(a->vocab, rows);
  p.num_slices = (a->vocab + p.slice - 1) / p.slice;
  p.logits = a->logits;
  p.rows = a->rows;
  p.n_tree = a->n_tree;
  p.parent = a->parent;
  p.tokens = a->tokens;
  p.weight = a->weight;
  p.cand_tok = a->cand_tok;
  p.cand_lp = a->cand_lp;
  p.cand_taken = a->cand_taken;
  p.added = a->added;
  p.err = reinterpret_cast<unsigned*>(ws);
  p.part = reinterpret_cast<CandPartial*>(ws + kWsHeader);
  cudaError_t e = launch_expand(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

size_t tree_select_workspace_size(const ts_select_args* a) { return a == nullptr ? 0 : kWsHeader; }

ts_status tree_select_subtree(const ts_select_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  if (a == nullptr || a->num_requests < 1 || a->n_tree_max < 1 || a->bs < 1) return TS_ERR_INVALID_ARG;
  if (a->n_tree_max > TS_MAX_TREE) return TS_ERR_UNSUPPORTED;
  if (!a->n_tree || !a->parent || !a->tokens || !a->weight || !a->keep || !a->new_parent || !a->new_tokens ||
      !a->new_weight || !a->n_sel)
    return TS_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kWsHeader || !aligned(workspace, 256)) return TS_ERR_WORKSPACE;
  SelectParams p;
  p.num_req = a->num_requests;
  p.n_tree_max = a->n_tree_max;
  p.bs = a->bs;
  p.n_tree = a->n_tree;
  p.parent = a->parent;
  p.tokens = a->tokens;
  p.weight = a->weight;
  p.keep = a->keep;
  p.new_parent = a->new_parent;
  p.new_tokens = a->new_tokens;
  p.new_weight = a->new_weight;
  p.n_sel = a->n_sel;
  p.err = reinterpret_cast<unsigned*>(workspace);
  cudaError_t e = launch_select(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

}  // extern "C"
