// Host/device parameter blocks and launchers shared by the treespec .cu files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "treespec.h"

namespace ts {

// Launches a kernel with programmatic dependent launch allowed: its CTAs may
// be scheduled while the previous kernel in the stream drains.  Every kernel
// of this library begins with pdl_wait() (griddepcontrol.wait), which blocks
// until the previous grid has completed and its writes are visible, so
// stream order is kept; only the launch latency is overlapped.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

constexpr int kBlockN = 64;        // keys per K/V tile
constexpr int kMaxRowsPerUnit = 128;  // packed query rows handled by one CTA
// Shares of one unit the tcgen05 path's merge reads in one round of loads
// (its share groups x shares prefetched per group).
constexpr int kMergeSharesPerRound = 32;
constexpr int kMaxRequestsAttn = 1024;
constexpr size_t kWsHeader = 256;  // error word + padding at the start of every workspace
constexpr int64_t kCompactBatchBytes = 96 * 1024;  // row-move staging per CTA (two CTAs per SM)

// Parameters of one tree_attn_forward call as the kernels see them.
struct AttnParams {
  int num_req, hq, hkv, group, head_dim, n_query, n_tree_max;
  int rows;          // R = G * n_query packed rows per KV head
  int hp;            // KV heads per unit: 2 when the tcgen05 kernel packs two heads (R <= 64), else 1
  int row_groups;    // ceil(R / 128)
  int rows_pad;      // rows per unit rounded up to 16 (<= 128)
  int max_kv_len;
  int paged, page_size, max_blocks, num_blocks;
  int num_ctas;      // NC
  int seg_cost;      // E of the cost-weighted split (tcgen05 path, > 0); 0 = plain split of the tiles
  int stages;
  int merge_half_warp;  // the merge takes one row per half-warp (else one per warp)
  int64_t num_units; // num_req * hkv * row_groups
  const int32_t* prefix_len;
  const int32_t* n_tree;
  const int32_t* parent;
  const __nv_bfloat16* q;
  const int32_t* block_table;
  __nv_bfloat16* out;
  float* lse;
  float scale_log2;  // softmax scale * log2(e)
  unsigned* err;     // workspace error word
  float* part_o;     // warp-MMA path: [slots][rows_pad][head_dim]; tcgen05 path: [slots][32][128] float4
                     // (float4 j of row r at (slot * 32 + j) * 128 + r)
  float* part_lse;   // [slots][rows_pad] (log2 domain)
  uint64_t wait_ns;    // bound of each pipeline wait (the drain waits after an abort keep kWaitLimitNs)
  int rope;            // 1: rotate the queries at their tree positions (rope_turn holds the frequencies)
  uint64_t rope_turn[64];  // theta^(-2j/d) / 2 pi as a 64-bit fraction of a turn, j < d/2
};

// Launchers (one per kernel family); return cudaGetLastError().
cudaError_t launch_attn_mma(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream);
cudaError_t launch_attn_tc(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                           cudaStream_t stream);
size_t attn_zero_prefix_bytes(const ts_attn_args* a);
cudaError_t launch_attn_merge(const AttnParams& p, bool tc_layout, cudaStream_t stream);
size_t attn_mma_smem_bytes(int head_dim, int stages, int num_req, int rows_pad);
size_t attn_tc_smem_bytes(int stages, int num_req);
int attn_mma_threads(int rows_pad);
int attn_tc_threads();

cudaError_t launch_tree_meta(const int32_t* parent, const int32_t* n_tree, int num_req, int n_tree_max,
                             int32_t* depth, uint32_t* anc, unsigned* err, cudaStream_t stream);

struct AcceptParams {
  int num_req, n_tree_max, vocab, chunk, num_chunks;
  const float* logits;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* n_tree;
  int32_t* argmax;
  int32_t* path;
  int32_t* accept_len;
  int32_t* bonus;
  int32_t* verified;
  int32_t* verified_len;
  unsigned* err;
  float* part_val;   // [num_req * n_tree_max][num_chunks]
  int32_t* part_idx; // [num_req * n_tree_max][num_chunks]
};
cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream);

struct CompactParams {
  int num_req, n_tree_max, m_max, num_layers, row_bytes;
  int paged, max_kv_len, page_size, max_blocks, num_blocks;
  int items_per_cta;  // (layer, K|V) items per CTA
  int ctas;           // CTAs per request: ceil(2 * num_layers / items_per_cta)
  int batch_vecs;     // 16-byte vectors staged in shared memory per batch
  void* const* k_layers;
  void* const* v_layers;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* n_tree;
  const int32_t* parent;
  const int32_t* tokens;
  const int32_t* verified;
  const int32_t* m;
  int32_t* new_prefix_len;
  int32_t* new_n_tree;
  int32_t* new_parent;
  int32_t* new_tokens;
  int32_t* src_rows;
  unsigned* err;
  unsigned* ticket;  // [num_req] CTAs of the request that have read its metadata; 0 between calls
};
cudaError_t launch_compact(const CompactParams& p, cudaStream_t stream);
// Up to TS_MAX_COMPACT_BATCH independent compactions in one launch; call i
// owns grid rows req_end[i - 1] .. req_end[i] - 1 (req_end[-1] = 0).
struct CompactBatch {
  CompactParams p[TS_MAX_COMPACT_BATCH];
  int req_end[TS_MAX_COMPACT_BATCH];
  int count;
};
cudaError_t launch_compact_batch(const CompactBatch& bt, cudaStream_t stream);

// One (row, vocab slice) partial of the draft-candidate pass: running max m,
// sum of exp(logit - m), and the slice's TS_MAX_EXPAND largest logits.
struct CandPartial {
  float m, s;
  float val[TS_MAX_EXPAND];
  int idx[TS_MAX_EXPAND];
};

struct ExpandParams {
  int num_req, n_tree_max, vocab, w, k;
  int slice, num_slices;   // vocab floats per candidate CTA (multiple of 1024), slices per row (<= 16)
  const float* logits;
  const int32_t* rows;
  int32_t* n_tree;
  int32_t* parent;
  int32_t* tokens;
  float* weight;
  int32_t* cand_tok;
  float* cand_lp;
  int32_t* cand_taken;
  int32_t* added;
  unsigned* err;
  CandPartial* part;       // [num_req * w][num_slices]
};
cudaError_t launch_expand(const ExpandParams& p, cudaStream_t stream);

struct SelectParams {
  int num_req, n_tree_max, bs;
  const int32_t* n_tree;
  const int32_t* parent;
  const int32_t* tokens;
  const float* weight;
  int32_t* keep;
  int32_t* new_parent;
  int32_t* new_tokens;
  float* new_weight;
  int32_t* n_sel;
  unsigned* err;
};
cudaError_t launch_select(const SelectParams& p, cudaStream_t stream);

// One request's hand-off between the walk's leader CTA and its helpers (in
// the workspace; zero before the first call, left at zero by every call
// that ends without a timeout).  A command is one 64-bit word: its sequence
// number (bits 48..63, from 1), the node (bits 32..47; kWalkStopNode to
// stop) and the pass's threshold a (bits 0..31, fp32); helper k answers in
// slot[k]: the sequence number (bits 32..63) and its slice sum (fp32).
constexpr int kMaxWalkCtas = 16;
struct WalkSync {
  unsigned long long cmd;
  unsigned long long slot[kMaxWalkCtas];  // slot k: helper k's answer (slot 0 unused)
  unsigned long long last;                // the last command number of the previous call
  unsigned long long pad[32 - 2 - kMaxWalkCtas];  // 256 bytes per request
};
constexpr int kWalkStopNode = 0xffff;

struct SampleParams {
  int num_req, n_tree_max, vocab;
  int slice, num_slices;  // vocab floats per statistics CTA (multiple of 1024), slices per row (<= 32)
  float scale2;           // log2(e) / temperature: every exponential is 2^(x scale2 - lse2)
  uint64_t wait_ns;       // bound of each wait in the walk's hand-offs
  const float* tl;
  const float* dl;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* n_tree;
  const float* u_acc;
  const float* u_bonus;
  int32_t* path;
  int32_t* accept_len;
  int32_t* bonus;
  int32_t* verified;
  int32_t* verified_len;
  unsigned* err;
  float2* part;           // [2][num_req * n_tree_max][num_slices]: (max, sum of exp) of logit / T
  int walk_ctas;          // CTAs per request in the walk: one leader and walk_ctas - 1 helpers
  WalkSync* sync;         // [num_req]: the leader's commands and the helpers' slice sums
};
cudaError_t launch_sample(const SampleParams& p, cudaStream_t stream);

}  // namespace ts
