// Evolving tree cache: re-root walk and in-place KV-row compaction, one kernel.
//
// SwiftSpec summary, §3.2 (the prefix-cache / tree-cache invariant and its
// update procedure), Figure 4 (t12, t15 promoted, t17, t18 moved to the front
// of the tree cache, the rest dropped) and Figure 2 with its walkthrough
// (re-rooting at t6 reuses its subtree; an out-of-tree token reuses nothing).
//
// Grid (G, num_requests): the G CTAs of request b share its (layer, K|V)
// row moves.  A batch of independent calls (e.g. the target-side and the
// draft-side cache of one verify step) runs as one launch whose grid rows
// are the requests of all calls.  Every CTA derives the re-root itself from the request's tree,
// held in shared memory (at most TS_MAX_TREE nodes):
//   1. one warp walks the verified tokens down the tree, taking at each step
//      the lowest-index child of the current node that carries the token
//      (each lane holds four nodes in registers; a warp min-reduction per
//      step, no block barriers);
//   2. survivors = proper descendants of the last matched node (every node
//      when no token was verified), found by walking each node's parent
//      chain up to that node's index, ranked in index order;
//   3. src = path ++ survivors; row j of the new tree cache takes old row
//      src[j].  Only rows with src[j] != j move.
// The new metadata (prefix length, tree size, parents, tokens, src) may
// overwrite the old in place, so it is written by exactly one CTA per
// request, the one that takes the last of the request's G tickets: every
// CTA takes its ticket only after it has read the old metadata.  That CTA
// resets the ticket for the next call.  No CTA waits for another.
//
// Row moves: the CTA's items are (layer, K|V) pairs; their moved rows form a
// sequence of 16-byte vectors (item, moved row in increasing destination
// order, vector).  The sequence goes through shared memory in batches: load
// the whole batch, then store it.  A source row is never below its
// destination (src is strictly increasing and src[j] >= j), so within an
// item a row is read, at the latest, in the batch that overwrites it, and
// every read of a batch precedes its stores: no row is overwritten before it
// is read.  Items of different CTAs are disjoint.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kCompactThreads = 256;
constexpr int kLoadsInFlight = 8;  // 16-byte loads per thread before the first store to shared memory
constexpr int kItemPtrs = 32;      // item base pointers a CTA keeps in shared memory

// One CTA's share of one request's compaction: request b of the call whose
// parameters are p, CTA `cta` of its p.ctas.
__device__ __forceinline__ void compact_body(const CompactParams& p, const int b, const int cta) {
  extern __shared__ uint4 buf[];  // [batch_vecs]
  __shared__ int par_s[TS_MAX_TREE];
  __shared__ int tok_s[TS_MAX_TREE];
  __shared__ int ver_s[TS_MAX_TREE + 1];
  __shared__ int path_s[TS_MAX_TREE + 1];
  __shared__ int surv_s[TS_MAX_TREE];     // survivors' old indices, by rank
  __shared__ int newidx[TS_MAX_TREE];     // old index -> survivor rank, or -1
  __shared__ int64_t mv_src[TS_MAX_TREE]; // moved row k: source / destination row within a layer's cache
  __shared__ int64_t mv_dst[TS_MAX_TREE];
  __shared__ int cnt[kCompactThreads / 32];
  __shared__ int blk_s[TS_MAX_TREE + 2];  // paged: block-table entries of the pages holding rows P .. P + n - 1
  __shared__ int walk_cur, walk_plen, walk_all, last_ticket;
  __shared__ void* item_ptr[kItemPtrs];   // base pointers of the CTA's first (layer, K|V) items

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t rowbase = static_cast<int64_t>(b) * p.n_tree_max;

  // ---- the request's lengths, tree and verified tokens, requested together
  //      (bounded by the arrays' sizes; the lengths then clamp what is used),
  //      and the base pointers of the CTA's first (layer, K|V) items, which
  //      only the row moves need
  const int items = 2 * p.num_layers;
  const int it0 = cta * p.items_per_cta;
  const int it1 = min(items, it0 + p.items_per_cta);
  int n = p.n_tree[b];
  int m = p.m[b];
  int P = p.prefix_len[b];
  const int ver = tid < min(p.m_max, TS_MAX_TREE + 1) ? p.verified[static_cast<int64_t>(b) * p.m_max + tid] : 0;
  const int raw_par = tid < p.n_tree_max ? p.parent[rowbase + tid] : -1;
  const int raw_tok = tid < p.n_tree_max ? p.tokens[rowbase + tid] : 0;
  if (tid < min(it1 - it0, kItemPtrs)) {
    const int it = it0 + tid;
    item_ptr[tid] = (it & 1) ? p.v_layers[it >> 1] : p.k_layers[it >> 1];
  }
  bool bad = false;
  if (n < 0 || n > p.n_tree_max) { n = min(max(n, 0), p.n_tree_max); bad = true; }
  if (m < 0 || m > p.m_max) { m = min(max(m, 0), p.m_max); bad = true; }
  const int cap = p.paged ? p.max_blocks * p.page_size : p.max_kv_len;
  if (P < 0 || P + n > cap) { P = min(max(P, 0), max(cap - n, 0)); bad = true; }
  if (bad && tid == 0 && cta == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);
  // A walk step matches at most one node, so with n <= TS_MAX_TREE nodes the
  // walk has always ended by step TS_MAX_TREE + 1: later tokens are never read.
  const int mw = min(m, TS_MAX_TREE + 1);
  if (tid < mw) ver_s[tid] = ver;  // mw <= TS_MAX_TREE + 1 < kCompactThreads
  int my_par = -1, my_tok = 0;
  if (tid < n) {
    my_par = raw_par;
    if (my_par < -1 || my_par >= tid) {
      if (cta == 0) report_error(p.err, TS_DEVERR_BAD_PARENT);
      my_par = -1;
    }
    my_tok = raw_tok;
    par_s[tid] = my_par;
    tok_s[tid] = my_tok;
  }
  __syncthreads();  // every read of the old metadata is done

  // ---- ticket: the request's last CTA writes the new metadata (requested
  //      by warp 1 while warp 0 walks); paged: the tree rows' block-table
  //      entries, read by warps 2.. while warp 0 walks
  const int pg0 = p.paged ? P / p.page_size : 0;
  if (p.paged && tid >= 64) {
    const int npg = n > 0 ? (P + n - 1) / p.page_size - pg0 + 1 : 0;
    for (int j = tid - 64; j < npg; j += kCompactThreads - 64)
      blk_s[j] = p.block_table[static_cast<int64_t>(b) * p.max_blocks + pg0 + j];
  }
  // the ticket is taken here and its value used just before the barrier that
  // precedes the metadata write, so the atomic's round trip overlaps the walk
  unsigned ticket_before = 0;
  if (tid == 32) {
    __threadfence();
    ticket_before = atomicAdd(p.ticket + b, 1u);
  }

  // ---- 1. walk (warp 0): lane l holds nodes l, l + 32, l + 64, l + 96
  if (warp == 0) {
    int wp[TS_MAX_TREE / 32], wt[TS_MAX_TREE / 32];
#pragma unroll
    for (int q = 0; q < TS_MAX_TREE / 32; ++q) {
      const int i = lane + 32 * q;
      wp[q] = i < n ? par_s[i] : -2;  // -2: never a child of anything
      wt[q] = i < n ? tok_s[i] : 0;
    }
    int cur = -1, plen = 0, all = 1;
    for (int j = 0; j < mw; ++j) {
      const int v = ver_s[j];
      int cand = INT32_MAX;
#pragma unroll
      for (int q = TS_MAX_TREE / 32 - 1; q >= 0; --q)  // the lane's lowest matching index wins
        if (wp[q] == cur && wt[q] == v) cand = lane + 32 * q;
      cand = __reduce_min_sync(0xffffffffu, cand);
      if (cand == INT32_MAX) {
        all = 0;
        break;
      }
      if (lane == 0) path_s[plen] = cand;
      ++plen;
      cur = cand;
    }
    if (lane == 0) {
      walk_cur = cur;
      walk_plen = plen;
      walk_all = all;
    }
  }
  __syncthreads();
  const int cur = walk_cur, plen = walk_plen;
  const bool all = walk_all != 0;

  // ---- 2. survivors: proper descendants of cur (every node when cur = -1)
  bool surv = false;
  if (all && tid < n && tid != cur) {
    if (cur < 0) {
      surv = true;
    } else if (tid > cur) {
      int u = my_par;  // parent indices strictly decrease: at most n steps
      while (u > cur) u = par_s[u];
      surv = u == cur;
    }
  }
  const unsigned bal = __ballot_sync(0xffffffffu, surv);
  if (lane == 0) cnt[warp] = __popc(bal);
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kCompactThreads / 32; ++w) {
    if (w < warp) before += cnt[w];
    total += cnt[w];
  }
  const int rank = before + __popc(bal & ((1u << lane) - 1u));
  if (tid < n) newidx[tid] = surv ? rank : -1;
  if (surv) surv_s[rank] = tid;
  __syncthreads();  // cnt is reused below; surv_s / newidx complete

  // ---- 3. moved rows: destination j < plen + total whose source differs
  const int L = plen + total;
  const int srcj = tid < L ? (tid < plen ? path_s[tid] : surv_s[tid - plen]) : tid;
  const bool moves = tid < L && srcj != tid;
  const unsigned mbal = __ballot_sync(0xffffffffu, moves);
  if (lane == 0) cnt[warp] = __popc(mbal);
  if (tid == 32) {
    const int last = ticket_before + 1u == static_cast<unsigned>(p.ctas);
    if (last) p.ticket[b] = 0u;
    __threadfence();
    last_ticket = last;
  }
  __syncthreads();  // cnt, last_ticket
  int mbefore = 0, nmv = 0;
#pragma unroll
  for (int w = 0; w < kCompactThreads / 32; ++w) {
    if (w < warp) mbefore += cnt[w];
    nmv += cnt[w];
  }
  if (moves) {
    const int k = mbefore + __popc(mbal & ((1u << lane) - 1u));
    const int rs = P + srcj, rd = P + tid;
    int64_t s = -1, d = -1;
    if (!p.paged) {
      s = static_cast<int64_t>(b) * p.max_kv_len + rs;
      d = static_cast<int64_t>(b) * p.max_kv_len + rd;
    } else {
      const int bs = blk_s[rs / p.page_size - pg0];
      const int bd = blk_s[rd / p.page_size - pg0];
      if (bs < 0 || bs >= p.num_blocks || bd < 0 || bd >= p.num_blocks) {
        report_error(p.err, TS_DEVERR_BAD_BLOCK);  // the row is not moved
      } else {
        s = static_cast<int64_t>(bs) * p.page_size + rs % p.page_size;
        d = static_cast<int64_t>(bd) * p.page_size + rd % p.page_size;
      }
    }
    mv_src[k] = s;
    mv_dst[k] = d;
  }

  // ---- new metadata (one CTA per request)
  if (last_ticket) {
    if (tid == 0) {
      p.new_prefix_len[b] = P + plen;
      p.new_n_tree[b] = total;
    }
    if (tid < p.n_tree_max) {
      int np = -1, nt = 0;
      if (tid < total) {
        const int i = surv_s[tid];
        const int q = par_s[i];
        np = q == cur ? -1 : newidx[q];
        nt = tok_s[i];
      }
      p.new_parent[rowbase + tid] = np;
      p.new_tokens[rowbase + tid] = nt;
      if (p.src_rows != nullptr) p.src_rows[rowbase + tid] = tid < L ? srcj : -1;
    }
  }
  __syncthreads();  // mv_src / mv_dst complete

  // ---- row moves: items it0 .. it1 - 1 of this CTA, as 16-byte vectors
  if (nmv == 0 || it0 >= it1) return;
  const int vr = p.row_bytes / 16;
  const int64_t per_item = static_cast<int64_t>(nmv) * vr;
  const int64_t nvec = per_item * (it1 - it0);
  // nvec < 2^31 (the host bounds items_per_cta), so 32-bit arithmetic
  // suffices.  x / per_item is a multiply-high by a constant fixed for the CTA
  // (division by an invariant integer, Granlund and Montgomery 1994: with
  // l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, t = mulhi(m, x),
  // x / d = (t + ((x - t) >> min(l, 1))) >> max(l - 1, 0), exact for every
  // 32-bit x); a row's vector count is a power of two for the usual shapes,
  // and then its quotient and remainder are a shift and a mask.
  const uint32_t per_item32 = static_cast<uint32_t>(per_item), vr32 = static_cast<uint32_t>(vr);
  const uint32_t pi_l = per_item32 <= 1 ? 0u : 32u - static_cast<uint32_t>(__clz(per_item32 - 1));
  const uint32_t pi_m =
      static_cast<uint32_t>((4294967296ull * ((1ull << pi_l) - per_item32)) / per_item32 + 1ull);
  const uint32_t pi_s1 = pi_l > 0 ? 1u : 0u, pi_s2 = pi_l > 0 ? pi_l - 1u : 0u;
  const bool vr_pow2 = (vr32 & (vr32 - 1u)) == 0u;
  const uint32_t vr_sh = static_cast<uint32_t>(__ffs(static_cast<int>(vr32)) - 1);
  auto address = [&](int64_t x, bool dst) -> uint4* {
    const uint32_t x32 = static_cast<uint32_t>(x);
    const uint32_t t = __umulhi(pi_m, x32);
    const uint32_t itn = (t + ((x32 - t) >> pi_s1)) >> pi_s2;  // x32 / per_item32
    const int it = it0 + static_cast<int>(itn);
    const uint32_t rem = x32 - itn * per_item32;
    int k, e;
    if (vr_pow2) {
      k = static_cast<int>(rem >> vr_sh);
      e = static_cast<int>(rem & (vr32 - 1u));
    } else {
      k = static_cast<int>(rem / vr32);
      e = static_cast<int>(rem % vr32);
    }
    const int64_t row = dst ? mv_dst[k] : mv_src[k];  // both -1 when the row does not move
    if (row < 0) return nullptr;
    void* base = it - it0 < kItemPtrs ? item_ptr[it - it0] : ((it & 1) ? p.v_layers[it >> 1] : p.k_layers[it >> 1]);
    return reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + row * p.row_bytes) + e;
  };
  for (int64_t x0 = 0; x0 < nvec; x0 += p.batch_vecs) {
    const int nb = static_cast<int>(min(static_cast<int64_t>(p.batch_vecs), nvec - x0));
    for (int y0 = tid; y0 < nb; y0 += kLoadsInFlight * kCompactThreads) {
      uint4 v[kLoadsInFlight];
#pragma unroll
      for (int q = 0; q < kLoadsInFlight; ++q) {
        const int y = y0 + q * kCompactThreads;
        v[q] = make_uint4(0, 0, 0, 0);
        if (y < nb) {
          const uint4* s = address(x0 + y, false);
          if (s != nullptr) v[q] = *s;
        }
      }
#pragma unroll
      for (int q = 0; q < kLoadsInFlight; ++q) {
        const int y = y0 + q * kCompactThreads;
        if (y < nb) buf[y] = v[q];
      }
    }
    __syncthreads();
    for (int y = tid; y < nb; y += kCompactThreads) {
      uint4* d = address(x0 + y, true);
      if (d != nullptr) *d = buf[y];
    }
    __syncthreads();  // the next batch rewrites buf
  }
}

__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const CompactParams p) {
  pdl_wait();
  pdl_launch_dependents();
  compact_body(p, blockIdx.y, blockIdx.x);
}

// Several independent compactions in one launch: row y of the grid is
// request y - req_end[i - 1] of call i; call i uses the first p[i].ctas CTAs
// of the row.  Each branch passes a fixed element, so the parameters are
// read from the constant bank as in the single kernel.
__global__ void __launch_bounds__(kCompactThreads) compact_batch_kernel(const CompactBatch bt) {
  pdl_wait();
  pdl_launch_dependents();
  const int y = blockIdx.y, x = blockIdx.x;
  if (y < bt.req_end[0]) {
    if (x < bt.p[0].ctas) compact_body(bt.p[0], y, x);
  } else if (bt.count > 1 && y < bt.req_end[1]) {
    if (x < bt.p[1].ctas) compact_body(bt.p[1], y - bt.req_end[0], x);
  } else if (bt.count > 2 && y < bt.req_end[2]) {
    if (x < bt.p[2].ctas) compact_body(bt.p[2], y - bt.req_end[1], x);
  } else if (bt.count > 3 && y < bt.req_end[3]) {
    if (x < bt.p[3].ctas) compact_body(bt.p[3], y - bt.req_end[2], x);
  }
}

}  // namespace

// The dynamic shared-memory limit is raised once per device (to the largest
// staging batch), so a launch is a plain stream operation (graph capture).
static bool compact_smem_ready() {
  static std::mutex m;
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(m);
  if (!done[dev]) {
    if (cudaFuncSetAttribute(compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kCompactBatchBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(compact_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kCompactBatchBytes)) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

cudaError_t launch_compact(const CompactParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(p.batch_vecs) * 16;
  if (smem > 48 * 1024 && !compact_smem_ready()) return cudaErrorInvalidValue;
  return launch_pdl(compact_kernel, dim3(p.ctas, p.num_req), dim3(kCompactThreads), smem, stream, p);
}

cudaError_t launch_compact_batch(const CompactBatch& bt, cudaStream_t stream) {
  int vecs = 0, ctas = 0;
  for (int i = 0; i < bt.count; ++i) {
    vecs = std::max(vecs, bt.p[i].batch_vecs);
    ctas = std::max(ctas, bt.p[i].ctas);
  }
  const size_t smem = static_cast<size_t>(vecs) * 16;
  if (smem > 48 * 1024 && !compact_smem_ready()) return cudaErrorInvalidValue;
  return launch_pdl(compact_batch_kernel, dim3(ctas, bt.req_end[bt.count - 1]), dim3(kCompactThreads), smem, stream,
                    bt);
}

}  // namespace ts
