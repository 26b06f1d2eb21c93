/*
 * treespec -- the speculative-decoding verify / expand step on one GB300 GPU.
 *
 * C ABI.  Every pointer named "device" is device memory owned by the caller;
 * the library allocates nothing, keeps no global state besides one cached
 * driver entry point and per-device launch facts (SM count, kernel
 * occupancy; computed on first use, guarded by a mutex), and never
 * synchronises the stream it is given.  Every
 * entry point validates its arguments on the host and returns a ts_status
 * synchronously; kernels are launched asynchronously on `stream` (a
 * cudaStream_t; NULL = the legacy default stream).  Kernel-side faults in the
 * metadata (a parent index out of range, a block-table entry out of range, a
 * bounded wait that expired) never trap: they clamp the offending value and
 * OR a TS_DEVERR_* bit into the error word at the start of the workspace,
 * which ts_read_device_error() reports.
 *
 * Workspace: each call that takes one needs `*_workspace_size()` bytes of
 * device memory, 256-byte aligned.  Its first 4 bytes are the sticky device
 * error word: zero the whole workspace once before its first use
 * (cudaMemset); afterwards the library keeps the rest consistent by itself
 * and only ts_read_device_error(..., clear = 1) resets the word.  Calls that
 * share one workspace must be ordered on one stream.
 *
 * Shapes use the pages' terms: a draft tree of n nodes (n = 1 + D for a
 * verify block, the SwiftSpec summary's bs), the last n_query nodes as
 * queries (w new leaves when expanding), G = num_q_heads / num_kv_heads query
 * heads per KV head (NVIDIA draft-length article), a verified prefix of P
 * tokens, and a parent array.  The KV cache of a request holds its P prefix
 * rows followed by its n tree rows: tree node i is row P + i (SwiftSpec
 * summary, §3.2, the prefix-cache / tree-cache invariant).
 */
#ifndef TREESPEC_H
#define TREESPEC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TS_API __attribute__((visibility("default")))
#else
#define TS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ts_status {
  TS_OK = 0,
  TS_ERR_INVALID_ARG = 1,   /* a null pointer, a negative or inconsistent size */
  TS_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels implement */
  TS_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  TS_ERR_WORKSPACE = 4      /* workspace missing, too small or misaligned */
} ts_status;

typedef enum ts_kv_layout {
  TS_KV_CONTIGUOUS = 0,     /* [num_requests][max_kv_len][num_kv_heads][head_dim] */
  TS_KV_PAGED = 1           /* pool [num_blocks][page_size][num_kv_heads][head_dim] + block table */
} ts_kv_layout;

/* Device error word bits (ts_read_device_error). */
#define TS_DEVERR_BAD_PARENT 0x1u   /* parent[i] outside [-1, i): treated as -1 */
#define TS_DEVERR_BAD_LENGTH 0x2u   /* prefix_len / n_tree / m outside its stated bound: clamped */
#define TS_DEVERR_BAD_BLOCK 0x4u    /* block_table entry outside [0, num_blocks): rows read as zero / not moved */
#define TS_DEVERR_TIMEOUT 0x8u      /* a bounded wait inside a kernel expired; outputs are invalid */
#define TS_DEVERR_BAD_TOKEN 0x10u   /* a draft token outside [0, vocab): never accepted */
#define TS_DEVERR_BAD_WORKSPACE 0x20u /* a workspace word holds what no call wrote (not zeroed before use,
                                       or last used by a call of another shape): ignored, outputs invalid */

/* Largest tree the kernels accept (ancestor sets are 128-bit masks). */
#define TS_MAX_TREE 128

/* ------------------------------------------------------------------------
 * Tree metadata (depth and ancestor-or-self bitmask of every node).
 *
 * SwiftSpec summary, §3.1.3 and Figure 3: a node attends to its ancestors
 * and itself; the mask row of node i is the set anc(i).  Computed for every
 * request by one kernel: depth[b][i] = number of proper ancestors,
 * anc[b][i][w] = bits 32w..32w+31 of the set {j : j is i or an ancestor of i}.
 *
 *   parent  device int32 [num_requests][n_tree_max]; parent[i] in [-1, i)
 *   n_tree  device int32 [num_requests]; n_tree[b] in [0, n_tree_max]
 *   depth   device int32 [num_requests][n_tree_max]   (out; entries >= n_tree[b] set to -1)
 *   anc     device uint32 [num_requests][n_tree_max][4] (out; zero beyond n_tree[b])
 *   workspace  >= tree_meta_workspace_size() bytes (holds the error word)
 * Errors: TS_ERR_UNSUPPORTED if n_tree_max > TS_MAX_TREE.
 * ------------------------------------------------------------------------ */
TS_API size_t tree_meta_workspace_size(void);
TS_API ts_status tree_build_mask(const int32_t* parent, const int32_t* n_tree, int num_requests,
                          int n_tree_max, int32_t* depth, uint32_t* anc, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Tree-masked grouped-query attention (verify and expand).
 *
 * SwiftSpec summary, §3.1.3 / Figure 3 (non-square mask: query rows are the
 * new leaves, key columns are the prefix and the whole tree, each leaf sees
 * the prefix, its ancestors and itself) and §3.3 (one head split across
 * thread blocks, partial results combined).  For request b, query r is tree
 * node u = n_tree[b] - n_query + r; query head h reads KV head h / G; keys are
 * rows [0, prefix_len[b] + n_tree[b]) of the request's cache; key P + j is
 * visible to u iff j is u or an ancestor of u; every prefix key is visible.
 *   out[b][r][h] = sum_j softmax_j(scale * q.k_j) v_j   (bf16, fp32 accumulation)
 *   lse[b][h][r] = log sum_j exp(scale * q.k_j)         (fp32, natural log)
 * The caller has already written the tree's K/V rows at P .. P + n - 1.
 * With rope_theta > 0 the queries are first rotated at their tree positions
 * (SwiftSpec summary §3.3, RoPE inside the verify attention; position of
 * node u = prefix_len[b] + depth(u), the root at depth 0): rotate-half
 * rotary embedding, pair (x_j, x_{j+d/2}) turned by position *
 * rope_theta^(-2j/d) (angles in fp64, rotation in fp32, bf16 result), into
 * workspace scratch; `q` itself is not written.  The K rows are read as
 * stored (rotated by the writer, as in any KV cache).
 * ------------------------------------------------------------------------ */
typedef struct ts_attn_args {
  int num_requests;           /* >= 1 (an empty batch is TS_ERR_INVALID_ARG) */
  int num_q_heads;            /* Hq */
  int num_kv_heads;           /* Hkv; Hq % Hkv == 0, G = Hq / Hkv */
  int head_dim;               /* 64 or 128 */
  int n_tree_max;             /* row stride of `parent`; <= TS_MAX_TREE */
  int n_query;                /* query rows per request, 1 <= n_query <= n_tree[b] */
  int max_kv_len;             /* contiguous: rows allocated per request (>= P + n);
                                 paged: max_blocks_per_req * page_size */
  int kv_layout;              /* ts_kv_layout */
  int page_size;              /* paged only: 16, 32 or 64 rows per block */
  int max_blocks_per_req;     /* paged only: row stride of block_table */
  int num_blocks;             /* paged only: blocks in the pool */
  const int32_t* prefix_len;  /* device [num_requests]: P >= 0 */
  const int32_t* n_tree;      /* device [num_requests]: n in [n_query, n_tree_max] */
  const int32_t* parent;      /* device [num_requests][n_tree_max] */
  const void* q;              /* device bf16 [num_requests][n_query][Hq][head_dim] (16-byte aligned) */
  const void* k_cache;        /* device bf16, layout per kv_layout (16-byte aligned) */
  const void* v_cache;        /* device bf16, same layout as k_cache */
  const int32_t* block_table; /* device [num_requests][max_blocks_per_req] (paged only) */
  void* out;                  /* device bf16 [num_requests][n_query][Hq][head_dim] (out, 16-byte aligned) */
  float* lse;                 /* device fp32 [num_requests][Hq][n_query] (out) or NULL */
  float softmax_scale;        /* <= 0 selects 1 / sqrt(head_dim) */
  int force_path;             /* 0 automatic; 1 warp-mma kernel; 2 tcgen05 kernel (G*n_query <= 128, d 128) */
  int num_ctas;               /* 0 automatic; else the number of split-KV CTAs (testing) */
  float rope_theta;           /* 0: no rotation; > 0: RoPE base of the queries at tree positions */
  unsigned wait_limit_ns;     /* testing: bound of each pipeline wait inside the attention kernels, in ns
                                 (0 = the default, 2 s).  A wait that runs out sets TS_DEVERR_TIMEOUT; the
                                 kernel then waits for its own copies in flight (with the default bound),
                                 frees its tensor memory and returns, and the call's outputs are void. */
} ts_attn_args;

TS_API size_t tree_attn_workspace_size(const ts_attn_args* args);
/* The kernel tree_attn_forward runs for these arguments: 1 = warp-level MMA,
 * 2 = tcgen05/TMEM (R = G * n_query <= 128 and head_dim 128; rows padded to the
 * 128-row tile); -(ts_status) when the arguments are rejected. */
TS_API int tree_attn_selected_path(const ts_attn_args* args);
TS_API ts_status tree_attn_forward(const ts_attn_args* args, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Allocation-free variant of tree_attn_forward (the pages have no
 * counterpart: this is a library convenience).  For callers that cannot
 * allocate device memory -- code inside a host framework that owns all device
 * memory through its own pool, or latency-critical loops where cudaMalloc
 * would synchronize the device -- and so cannot pass a workspace.  The
 * split-KV scratch is a 16 MiB array in device memory that the library
 * reserves on every GPU that loads it, until the process exits.  The first
 * call on each device (with that device current) looks up the array's device
 * address; make that first call before any stream capture.  The address is kept
 * for the life of the process: it does not survive cudaDeviceReset (after a
 * reset the array may sit elsewhere), so do not call this variant after
 * resetting a device.  Same arguments,
 * results and tolerance as tree_attn_forward; when the partials of the
 * requested split would not fit, fewer split-KV CTAs are used; arguments whose
 * partials exceed 16 MiB even unsplit return TS_ERR_UNSUPPORTED.  No
 * cudaMalloc, cudaFree or allocating library call is made.  Every call shares
 * the one array, so calls that overlap on the GPU (other streams, other host
 * threads) race and corrupt each other's results: serialize them.  Device
 * error bits of this variant are cleared at the start of each call and are
 * not reported; use tree_attn_forward with a workspace to read them. */
TS_API ts_status tree_attn_forward_noalloc(const ts_attn_args* args, void* stream);

/* ------------------------------------------------------------------------
 * Greedy tree acceptance.
 *
 * NVIDIA draft-length article ("Speculative Decoding 작동 원리", Acceptance
 * Length): the target accepts draft tokens up to the first mismatch and adds
 * one of its own, so AL is in [1, 1 + D].  SwiftSpec summary Figure 2: the
 * target picks one path of the tree.  For each request b:
 *   argmax[b][i] = argmax_v logits[b][i][v]      (lowest v on ties)
 *   node 0 (the root = last verified token) is accepted; node i >= 1 is
 *   accepted iff parent[i] >= 0 is accepted and tokens[i] == argmax[parent[i]];
 *   path = the longest accepted root path (ties: smallest last index),
 *   accept_len = |path| (AL), bonus = argmax[last node of path],
 *   verified = tokens[path[0..AL-1]] ++ [bonus], verified_len = AL + 1.
 * An empty tree gives accept_len = 0, bonus = -1, verified_len = 0.
 *   logits   device fp32 [num_requests][n_tree_max][vocab] (rows >= n_tree[b] unread)
 *   tokens, parent  device int32 [num_requests][n_tree_max]
 *   n_tree   device int32 [num_requests]
 *   argmax, path    device int32 [num_requests][n_tree_max] (out; unused entries -1)
 *   accept_len, bonus  device int32 [num_requests] (out)
 *   verified device int32 [num_requests][n_tree_max + 1] (out) or NULL
 *   verified_len device int32 [num_requests] (out) or NULL
 * ------------------------------------------------------------------------ */
typedef struct ts_accept_args {
  int num_requests;           /* >= 1 */
  int n_tree_max;             /* <= TS_MAX_TREE */
  int vocab;                  /* >= 1 */
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
} ts_accept_args;

TS_API size_t tree_accept_workspace_size(const ts_accept_args* args);
TS_API ts_status tree_accept_greedy(const ts_accept_args* args, void* workspace, size_t workspace_bytes,
                             void* stream);

/* ------------------------------------------------------------------------
 * Evolving tree cache: re-root and in-place KV compaction.
 *
 * SwiftSpec summary, §3.2 (update procedure, Figure 4) and Figure 2's
 * walkthrough.  For each request b, walk the verified tokens v[0..m) from the
 * prefix tail: at each step take the lowest-index child of the current node
 * (the prefix tail at first: parent == -1) whose token equals v[j]; stop at
 * the first token without such a child.  The matched nodes (`path`) join the
 * prefix.  If all m tokens matched, the proper descendants of the last one
 * (all nodes when m == 0) survive as the new tree, in increasing index
 * order; otherwise nothing survives (a new tree starts from the unmatched
 * token, whose KV does not exist yet).  Then, for every layer and for K and
 * V, new row P + j takes old row P + src[j], src = path ++ survivors, in
 * place; rows below P are not touched; rows at or beyond the new P + n are
 * left with unspecified content.
 *   new_prefix_len = P + |path|, new_n_tree = |survivors|,
 *   new_parent[j] = -1 if the survivor's parent is the last matched node,
 *   else that parent's new index; new_tokens[j] = tokens of survivor j.
 *   new_prefix_len / new_n_tree / new_parent / new_tokens may alias
 *   prefix_len / n_tree / parent / tokens (in-place update);
 *   src_rows (optional) gets src (entries beyond |src| set to -1).
 * One kernel launch: every CTA of a request derives the re-root from the
 * request's tree and moves its share of the (layer, K|V) rows; the new
 * metadata is written by the request's last CTA to have read the old, found
 * with a per-request ticket counter in the workspace (zero before the first
 * call, left at zero by every call).  num_requests <= 65535.
 * Layers: k_layers / v_layers are device arrays of num_layers device
 * pointers, each one layer's cache in the given layout; the paged block
 * table is shared by all layers.  A row is num_kv_heads * head_dim *
 * elem_bytes bytes, a multiple of 16.
 * ------------------------------------------------------------------------ */
typedef struct ts_compact_args {
  int num_requests;           /* >= 1 */
  int n_tree_max;             /* <= TS_MAX_TREE */
  int m_max;                  /* row stride of `verified` */
  int num_layers;
  int num_kv_heads;
  int head_dim;
  int elem_bytes;             /* bytes per cache element (2 for bf16) */
  int kv_layout;              /* ts_kv_layout */
  int max_kv_len;             /* contiguous: rows allocated per request */
  int page_size;              /* paged only */
  int max_blocks_per_req;     /* paged only */
  int num_blocks;             /* paged only */
  void* const* k_layers;      /* device [num_layers] of device pointers */
  void* const* v_layers;      /* device [num_layers] of device pointers */
  const int32_t* block_table; /* device [num_requests][max_blocks_per_req] (paged only) */
  const int32_t* prefix_len;  /* device [num_requests] */
  const int32_t* n_tree;      /* device [num_requests] */
  const int32_t* parent;      /* device [num_requests][n_tree_max] */
  const int32_t* tokens;      /* device [num_requests][n_tree_max] */
  const int32_t* verified;    /* device [num_requests][m_max] */
  const int32_t* m;           /* device [num_requests]: m in [0, m_max] */
  int32_t* new_prefix_len;    /* device [num_requests] (out) */
  int32_t* new_n_tree;        /* device [num_requests] (out) */
  int32_t* new_parent;        /* device [num_requests][n_tree_max] (out, may alias parent) */
  int32_t* new_tokens;        /* device [num_requests][n_tree_max] (out, may alias tokens) */
  int32_t* src_rows;          /* device [num_requests][n_tree_max] (out) or NULL */
} ts_compact_args;

TS_API size_t tree_compact_workspace_size(const ts_compact_args* args);
TS_API ts_status tree_cache_compact(const ts_compact_args* args, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Several independent compactions in one kernel launch, e.g. the target-side
 * and the draft-side cache of one verify step (SwiftSpec summary, §3.2: both
 * the target and the draft keep a prefix cache and a tree cache).  args[i],
 * workspaces[i] and workspace_bytes[i] are exactly what tree_cache_compact
 * would take for call i (each call keeps its own workspace, error word and
 * ticket counters, so the workspaces must be distinct); the calls must not
 * share any written buffer (caches, new metadata), and the result equals
 * `count` tree_cache_compact calls.
 * count in [1, TS_MAX_COMPACT_BATCH]; the requests of all calls together
 * <= 65535.  Every call is validated before anything is launched: the
 * first failing status is returned and nothing runs. */
#define TS_MAX_COMPACT_BATCH 4
TS_API ts_status tree_cache_compact_batch(const ts_compact_args* args, int count, void* const* workspaces,
                                          const size_t* workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Stochastic tree acceptance (speculative sampling at temperature > 0).
 *
 * MineDraft summary (on a rejection one token is resampled from
 * norm(max(0, p - q)); the default temperature is 1.0), generalised to the
 * draft tree of the SwiftSpec summary, Figure 2.  p_u = softmax(
 * target_logits[u] / T) is the target's distribution after node u, q_u =
 * softmax(draft_logits[u] / T) the draft's (u's children were drawn from
 * it).  From the root (node 0, always accepted), at the current node u the
 * children are tried in index order with a running target r = p_u: child c
 * (token t) is accepted iff u_accept[c] < r(t) / q_u(t) (if q_u(t) is 0 in
 * fp32: iff r(t) > 0); on a rejection r becomes norm(max(0, r - q_u)) (kept
 * if that is all zero).  An accepted child becomes the current node.  When
 * every child was rejected, or u has none, the bonus is the smallest token v
 * with r(0) + ... + r(v) > u_bonus[u] * sum(r).  Children drawn
 * independently from q_u make the emitted tokens follow the target's law.
 *   path[b][0..AL) = accepted nodes (root first, -1 after), accept_len[b] =
 *   AL in [1, 1 + depth], bonus[b]; verified[b] = tokens(path) ++ bonus
 *   (-1 after, optional), verified_len[b] = AL + 1 (optional).
 * The uniforms are inputs in [0, 1).  Arithmetic: fp32, each probability
 * 2^(logit * log2(e) / T - the row's base-2 log-sum-exp) by the hardware's
 * approximate 2^x (relative error about 2^-22; below 2^-126 it is 0); a
 * decision within that rounding of its threshold may go either way.  Workspace: tree_accept_sample_workspace_size(),
 * zero-filled before its first use; besides the error word it holds
 * per-request command words whose numbering carries on from one call to the
 * next, so a workspace serves calls of one shape (num_requests, n_tree_max,
 * vocab) on one stream: zero it again before a call of another shape, and
 * after a call that reports TS_DEVERR_TIMEOUT (its outputs are void).
 * Errors: TS_ERR_INVALID_ARG unless temperature > 0 and finite;
 * TS_ERR_UNSUPPORTED if vocab > 262144 or n_tree_max > TS_MAX_TREE, or if
 * log2(e) / temperature overflows fp32 (a temperature below about 4e-39).
 * ------------------------------------------------------------------------ */
typedef struct ts_sample_args {
  int num_requests;           /* >= 1 */
  int n_tree_max;              /* <= TS_MAX_TREE */
  int vocab;                   /* >= 1 */
  float temperature;           /* > 0 */
  const float* target_logits;  /* device [num_requests][n_tree_max][vocab] */
  const float* draft_logits;   /* device [num_requests][n_tree_max][vocab] */
  const int32_t* tokens;       /* device [num_requests][n_tree_max] */
  const int32_t* parent;       /* device [num_requests][n_tree_max] */
  const int32_t* n_tree;       /* device [num_requests] */
  const float* u_accept;       /* device [num_requests][n_tree_max] */
  const float* u_bonus;        /* device [num_requests][n_tree_max] */
  int32_t* path;               /* device [num_requests][n_tree_max] (out) */
  int32_t* accept_len;         /* device [num_requests] (out) */
  int32_t* bonus;              /* device [num_requests] (out) */
  int32_t* verified;           /* device [num_requests][n_tree_max + 1] (out) or NULL */
  int32_t* verified_len;       /* device [num_requests] (out) or NULL */
  unsigned wait_limit_ns;      /* testing: bound of each wait in the walk's hand-offs between CTAs, in ns
                                  (0 = the default, 2 s).  A wait that runs out sets TS_DEVERR_TIMEOUT and
                                  its CTA returns; the call's outputs are void and the workspace must be
                                  zeroed before its next use. */
} ts_sample_args;

TS_API size_t tree_accept_sample_workspace_size(const ts_sample_args* args);
TS_API ts_status tree_accept_sample(const ts_sample_args* args, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* ------------------------------------------------------------------------
 * Draft-side tree growth: maximum-likelihood expansion (one step) and the
 * selection of the most promising subtree.
 *
 * SwiftSpec summary, §3.1.1 (the draft worker's iteration: Expand the w most
 * probable leaves d times while the target verifies, then Select a subtree
 * of size bs) and §3.1.3 (a node's value is the log-softmax probability of
 * its token under the draft model, its weight the sum of the values from
 * the root; the leaves to expand come from a priority queue); Figure 2
 * (w = 2 nodes per expansion, six in d = 3 steps).
 *
 * Per request b and node i < n_tree[b] (row stride n_tree_max): parent,
 * token, weight (fp32), and the node's candidate children
 * cand_tok[b][i][0..k), cand_lp[b][i][0..k) (token ids and log-softmax
 * values in decreasing order, ties to the lower token id; token -1 with
 * -inf past the vocabulary), of which the first cand_taken[b][i] have become
 * children (k: none known).
 *
 * tree_expand, one step, per request:
 *  1. each row r of `logits` with rows[b][r] in [0, n) gives that node its k
 *     candidates (the row's k largest logits, value = logit - log-sum-exp of
 *     the row) and cand_taken = 0;
 *  2. w times: among the nodes with a candidate left, the one whose next
 *     candidate has the largest weight[node] + cand_lp (ties: the lower node
 *     index) gives it up: node n is appended with that parent, token and
 *     weight, cand_taken = k, and the parent's cand_taken grows by one.
 *     Growth stops at n_tree_max or when no candidate is left;
 *  3. added[b][0..w) gets the new nodes in order (-1 past the last): the
 *     next draft queries.  n_tree grows accordingly.
 *  `added` may alias `rows`.  Workspace: tree_expand_workspace_size().
 *  Errors: TS_ERR_UNSUPPORTED if n_tree_max > TS_MAX_TREE, w or k > 16.
 *  Device: a row node outside [0, n) is ignored (TS_DEVERR_BAD_LENGTH).
 *
 * tree_select_subtree, per request: the min(bs, n) nodes of largest weight
 *  (ties: lower index), in index order: keep[b][j] = old index,
 *  new_parent[b][j] (remapped; -1 where the old parent is -1), new_tokens,
 *  new_weight, n_sel[b]; entries past n_sel are -1 / 0 / -inf.  Weights built
 *  by tree_expand never increase from a parent to a child, so the set holds
 *  every selected node's parent; a selected node whose parent is not
 *  selected (weights from elsewhere) gets new parent -1 and
 *  TS_DEVERR_BAD_PARENT.  Workspace: tree_select_workspace_size().
 * ------------------------------------------------------------------------ */
#define TS_MAX_EXPAND 16

typedef struct ts_expand_args {
  int num_requests;           /* >= 1 */
  int n_tree_max;          /* capacity and row stride, <= TS_MAX_TREE */
  int vocab;               /* >= 1 */
  int w;                   /* rows of logits and nodes added per step, 1..TS_MAX_EXPAND */
  int k;                   /* candidates per node, 1..TS_MAX_EXPAND */
  const float* logits;     /* device [num_requests][w][vocab] */
  const int32_t* rows;     /* device [num_requests][w]: node of each logits row, -1 = none */
  int32_t* n_tree;         /* device [num_requests] (in/out) */
  int32_t* parent;         /* device [num_requests][n_tree_max] (in/out) */
  int32_t* tokens;         /* device [num_requests][n_tree_max] (in/out) */
  float* weight;           /* device [num_requests][n_tree_max] (in/out) */
  int32_t* cand_tok;       /* device [num_requests][n_tree_max][k] (in/out) */
  float* cand_lp;          /* device [num_requests][n_tree_max][k] (in/out) */
  int32_t* cand_taken;     /* device [num_requests][n_tree_max] (in/out) */
  int32_t* added;          /* device [num_requests][w] (out; may alias rows) */
} ts_expand_args;

TS_API size_t tree_expand_workspace_size(const ts_expand_args* args);
TS_API ts_status tree_expand(const ts_expand_args* args, void* workspace, size_t workspace_bytes, void* stream);

typedef struct ts_select_args {
  int num_requests;           /* >= 1 */
  int n_tree_max;          /* row stride of the inputs, <= TS_MAX_TREE */
  int bs;                  /* nodes to keep, >= 1; row stride of the outputs */
  const int32_t* n_tree;   /* device [num_requests] */
  const int32_t* parent;   /* device [num_requests][n_tree_max] */
  const int32_t* tokens;   /* device [num_requests][n_tree_max] */
  const float* weight;     /* device [num_requests][n_tree_max] */
  int32_t* keep;           /* device [num_requests][bs] (out) */
  int32_t* new_parent;     /* device [num_requests][bs] (out) */
  int32_t* new_tokens;     /* device [num_requests][bs] (out) */
  float* new_weight;       /* device [num_requests][bs] (out) */
  int32_t* n_sel;          /* device [num_requests] (out) */
} ts_select_args;

TS_API size_t tree_select_workspace_size(const ts_select_args* args);
TS_API ts_status tree_select_subtree(const ts_select_args* args, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* ------------------------------------------------------------------------
 * Status and error reporting.
 * ------------------------------------------------------------------------ */
TS_API const char* ts_status_string(ts_status status);

/* Copies the device error word of `workspace` into *code (TS_DEVERR_* bits)
 * and, if `clear` is non-zero, resets it.  Synchronises `stream`. */
TS_API ts_status ts_read_device_error(void* workspace, int* code, int clear, void* stream);

/* Library version, (major << 16) | minor. */
TS_API int ts_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TREESPEC_H */
