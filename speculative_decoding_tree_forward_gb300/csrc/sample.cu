// Stochastic tree acceptance: speculative sampling at temperature T > 0 on a
// draft tree.
//
// MineDraft summary (a rejection resamples from norm(max(0, p - q)); default
// temperature 1.0), generalised to the tree of the SwiftSpec summary, Figure
// 2: at the current node the children are tried in index order, each
// accepted with probability min(1, r(t) / q(t)), r turning into
// norm(max(0, r - q)) after each rejection; an accepted child becomes the
// current node; when all are rejected the bonus is drawn from r.
//
// Kernel 1 (row statistics) streams every target and draft row of the tree
// once in vocab slices and keeps (max, sum of 2^(z - max)) of z = logit log2(e) / T.
// Kernel 2 (walk) runs a leader CTA and up to 15 helper CTAs per request
// (512 threads each): every CTA folds all nodes' slice statistics into their
// log-sum-exps, and warp 0 of the leader lists a node's children with
// ballots and tests each child from p and q at its token.  The running target
// after j rejections has the closed form max(0, p - a_j q) / S(a_j) (derived
// at the walk's passes below), so a rejection is one sum over the vocab and no
// residual row is written; the request's CTAs split that sum by vocab slices,
// each keeping its slice's 128-token block sums, and hand commands and slice
// sums over through the workspace with bounded waits.  The bonus is drawn by
// inverse transform: the slice that holds the target from the slice sums of
// the last pass, then, in the CTA that owns that slice, a block scan of its
// block sums and one warp's scan inside the block that holds the target.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kLseThreads = 256;
constexpr int kWalkThreads = 512;
constexpr int kWalkWarps = kWalkThreads / 32;

// Logits enter every exponential as x * scale2 with scale2 = log2(e) / T, so
// a row's statistics are (m, s) with m = max_v x_v scale2 and
// s = sum_v 2^(x_v scale2 - m), its log-sum-exp in base 2 is m + log2(s), and
// p(v) = 2^(x_v scale2 - lse2): the same softmax at temperature T, each
// exponential one ex2 instruction.
__device__ __forceinline__ void lse_pair(float& m, float& s, float om, float os) {
  if (om > m) {
    s = s * ex2_approx(m - om) + os;
    m = om;
  } else if (om != -INFINITY) {
    s += os * ex2_approx(om - m);
  }
}

__device__ __forceinline__ int tree_size(const SampleParams& p, int b) {
  return min(max(p.n_tree[b], 0), p.n_tree_max);
}

// At most 32 registers: eight CTAs per SM, the residency the host's slice
// sizing assumes (target and draft rows x slices = about one wave).
__global__ void __launch_bounds__(kLseThreads, 8) sample_lse_kernel(const SampleParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int rows = p.num_req * p.n_tree_max;
  const int which = blockIdx.x / rows;  // 0: target, 1: draft
  const int row = blockIdx.x % rows;
  if (row % p.n_tree_max >= tree_size(p, row / p.n_tree_max)) return;
  const float* lg = (which == 0 ? p.tl : p.dl) + static_cast<int64_t>(row) * p.vocab;
  const int64_t v0 = static_cast<int64_t>(blockIdx.y) * p.slice;
  const int64_t v1 = min(static_cast<int64_t>(p.vocab), v0 + p.slice);
  float m = -INFINITY, s = 0.f;
  if ((p.vocab & 3) == 0) {
    constexpr int kLoads = 4;  // 16-byte loads in flight per thread (eight CTAs per SM)
    const float4* lg4 = reinterpret_cast<const float4*>(lg);
    const int e4 = static_cast<int>(v1 / 4);  // vocab < 2^31
    for (int x0 = static_cast<int>(v0 / 4) + static_cast<int>(threadIdx.x); x0 < e4; x0 += kLoads * kLseThreads) {
      float4 f[kLoads];
#pragma unroll
      for (int q = 0; q < kLoads; ++q)
        f[q] = x0 + q * kLseThreads < e4 ? __ldcs(lg4 + x0 + q * kLseThreads)
                                         : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      float bm = m;
#pragma unroll
      for (int q = 0; q < kLoads; ++q)
        bm = fmaxf(bm, fmaxf(fmaxf(f[q].x, f[q].y), fmaxf(f[q].z, f[q].w)) * p.scale2);
      if (bm > m) {
        s *= ex2_approx(m - bm);
        m = bm;
      }
#pragma unroll
      for (int q = 0; q < kLoads; ++q)
        s += (ex2_approx(fmaf(f[q].x, p.scale2, -m)) + ex2_approx(fmaf(f[q].y, p.scale2, -m))) +
             (ex2_approx(fmaf(f[q].z, p.scale2, -m)) + ex2_approx(fmaf(f[q].w, p.scale2, -m)));
    }
  } else {
    for (int64_t x = v0 + threadIdx.x; x < v1; x += kLseThreads) lse_pair(m, s, __ldcs(lg + x) * p.scale2, 1.f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lse_pair(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
  __shared__ float wm[kLseThreads / 32], ws[kLseThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    wm[warp] = m;
    ws[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kLseThreads / 32; ++w) lse_pair(m, s, wm[w], ws[w]);
    p.part[(static_cast<int64_t>(which) * rows + row) * p.num_slices + blockIdx.y] = make_float2(m, s);
  }
}

// block-wide sum of one float per thread (all threads get the total)
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();  // red may still be read from the previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < kWalkWarps ? red[lane] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

// ---- the walk's passes --------------------------------------------------------
// After j rejections at node u the running target has a closed form.  With
// p = p_u and q = q_u, r_0 = p and r_{j+1} = norm(max(0, r_j - q)) give
//   r_j = max(0, p - a_j q) / S(a_j),  S(a) = sum_v max(0, p(v) - a q(v)),
//   a_0 = 0 (S(0) = 1),  a_{j+1} = a_j + S(a_j),
// since max(0, max(0, p - a q) / S - q) = max(0, p - (a + S) q) / S; when
// S(a_{j+1}) is 0 the residual is all zero and r_j is kept.  A rejection is
// therefore one sum of max(0, p - a q) over the vocab, with no residual row
// written, and the sum splits into slices: CTA k of a request's walk_ctas sums
// slice k.  The bonus is drawn from the unnormalised max(0, p - a q).
constexpr int kBonusBlock = 128;  // tokens per first-level block of the inverse transform
constexpr int kBlocksPerThread = 4;
constexpr int kMaxBonusBlocks = kBlocksPerThread * kWalkThreads;  // slice <= 262144 tokens
constexpr int kBlocksInFlight = 8;                                // a warp's block sums in flight

__device__ __forceinline__ float r_of(float xt, float xd, float scale2, float lt, float ld, float a) {
  return fmaxf(0.f, ex2_approx(fmaf(xt, scale2, -lt)) - a * ex2_approx(fmaf(xd, scale2, -ld)));
}

// Slice k of K of a row of V tokens: [v0, v1), v0 a multiple of 4.
__device__ __forceinline__ void walk_slice(int V, int K, int k, int& v0, int& v1) {
  const int len = ((V + K - 1) / K + 3) & ~3;
  v0 = min(V, k * len);
  v1 = min(V, v0 + len);
}

// Sums of r over the slice's blocks of kBonusBlock tokens (block i is
// [v0 + 128 i, ...)), warp per block with kBlocksInFlight blocks of a warp
// requested before any is summed, into bsum[0 .. ceil((v1 - v0) / 128)).
__device__ __forceinline__ void slice_block_sums(const float* __restrict__ tl, const float* __restrict__ dl, int V,
                                                 int v0, int v1, float scale2, float lt, float ld, float a, float* bsum) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = (v1 - v0 + kBonusBlock - 1) / kBonusBlock;
  for (int b0 = warp; b0 < nb; b0 += kBlocksInFlight * kWalkWarps) {
    float t[kBlocksInFlight];
    if ((V & 3) == 0) {  // lane l: tokens 4l .. 4l + 3 of the block, whole 16-byte groups (v1 - v0 % 4 == 0)
      float4 ft[kBlocksInFlight], fd[kBlocksInFlight];
      unsigned in = 0u;
#pragma unroll
      for (int j = 0; j < kBlocksInFlight; ++j) {
        const int v = v0 + (b0 + j * kWalkWarps) * kBonusBlock + 4 * lane;
        if (b0 + j * kWalkWarps < nb && v < v1) {
          ft[j] = __ldcg(reinterpret_cast<const float4*>(tl + v));
          fd[j] = __ldcg(reinterpret_cast<const float4*>(dl + v));
          in |= 1u << j;
        }
      }
#pragma unroll
      for (int j = 0; j < kBlocksInFlight; ++j)
        t[j] = ((in >> j) & 1u) ? (r_of(ft[j].x, fd[j].x, scale2, lt, ld, a) + r_of(ft[j].y, fd[j].y, scale2, lt, ld, a)) +
                                      (r_of(ft[j].z, fd[j].z, scale2, lt, ld, a) + r_of(ft[j].w, fd[j].w, scale2, lt, ld, a))
                                : 0.f;
    } else {
#pragma unroll
      for (int j = 0; j < kBlocksInFlight; ++j) {
        t[j] = 0.f;
#pragma unroll
        for (int e = 0; e < kBonusBlock / 32; ++e) {
          const int v = v0 + (b0 + j * kWalkWarps) * kBonusBlock + e * 32 + lane;
          if (b0 + j * kWalkWarps < nb && v < v1) t[j] += r_of(__ldcg(tl + v), __ldcg(dl + v), scale2, lt, ld, a);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kBlocksInFlight; ++j) {
      float x = t[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == 0 && b0 + j * kWalkWarps < nb) bsum[b0 + j * kWalkWarps] = x;
    }
  }
}

// Inside block blk of the slice: the smallest token with excl + r(block start
// .. v) > target (warp-wide: lane l holds tokens 4l .. 4l + 3 of the block), or -1.
__device__ __forceinline__ int scan_block(const float* __restrict__ tl, const float* __restrict__ dl, int v0, int v1,
                                          float scale2, float lt, float ld, float a, int blk, float excl, float target) {
  const int lane = threadIdx.x & 31;
  float r4[4];
  float mine = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int v = v0 + blk * kBonusBlock + lane * 4 + e;
    r4[e] = v < v1 ? r_of(__ldcg(tl + v), __ldcg(dl + v), scale2, lt, ld, a) : 0.f;
    mine += r4[e];
  }
  float inc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  float acc = excl + inc - mine;
  int pick = -1;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    acc += r4[e];
    if (pick < 0 && acc > target) pick = v0 + blk * kBonusBlock + lane * 4 + e;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, pick >= 0);
  return hit ? __shfl_sync(0xffffffffu, pick, __ffs(hit) - 1) : -1;
}

// Shared scratch of a bonus draw inside one slice.
struct DrawScratch {
  float scan[kWalkWarps];
  int cnt[kWalkWarps];
  int blk, bonus;
  float blk_excl;
};

// This CTA's part of a pass over node rows tl, dl: r's 128-token block sums
// over its slice [v0, v1) into bsum (kept for a bonus draw in the slice) and
// their total, which every thread returns.
__device__ __forceinline__ float slice_pass(const float* __restrict__ tl, const float* __restrict__ dl, int V, int v0,
                                            int v1, float scale2, float lt, float ld, float a, float* bsum, float* red) {
  __syncthreads();  // bsum may still be read from the previous pass
  slice_block_sums(tl, dl, V, v0, v1, scale2, lt, ld, a, bsum);
  __syncthreads();
  const int nbk = (v1 - v0 + kBonusBlock - 1) / kBonusBlock;
  float t = 0.f;
  for (int i = static_cast<int>(threadIdx.x); i < nbk; i += kWalkThreads) t += bsum[i];
  return block_sum(t, red);
}

// The bonus inside slice [v0, v1) of node rows tl, dl, from the block sums
// in bsum (those of a pass at the same a): the smallest v whose sum of r over
// [v0, v] exceeds ltarget; with take_last, or when rounding leaves no such v,
// the slice's last token with r > 0 (-1 if there is none).  Every thread
// returns it.
__device__ int draw_in_slice(const float* __restrict__ tl, const float* __restrict__ dl, int v0, int v1, float scale2,
                             float lt, float ld, float a, const float* bsum, float ltarget, bool take_last,
                             DrawScratch& ds) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nbk = (v1 - v0 + kBonusBlock - 1) / kBonusBlock;
  if (tid == 0) {
    ds.bonus = -1;
    ds.blk = -1;
  }
  __syncthreads();
  if (!take_last) {
    // consecutive block sums per thread (nbk <= kMaxBonusBlocks), block exclusive scan
    const int per = (nbk + kWalkThreads - 1) / kWalkThreads;
    float bs[kBlocksPerThread];
    float mine = 0.f;
#pragma unroll
    for (int e = 0; e < kBlocksPerThread; ++e) {
      bs[e] = (e < per && tid * per + e < nbk) ? bsum[tid * per + e] : 0.f;
      mine += bs[e];
    }
    float inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) ds.scan[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      float w = lane < kWalkWarps ? ds.scan[lane] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < kWalkWarps) ds.scan[lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    float excl = (warp > 0 ? ds.scan[warp - 1] : 0.f) + inc - mine;
#pragma unroll
    for (int e = 0; e < kBlocksPerThread; ++e) {
      if (bs[e] > 0.f && excl <= ltarget && ltarget < excl + bs[e]) {
        ds.blk = tid * per + e;
        ds.blk_excl = excl;
      }
      excl += bs[e];
    }
    __syncthreads();
    if (warp == 0 && ds.blk >= 0) {
      const int v = scan_block(tl, dl, v0, v1, scale2, lt, ld, a, ds.blk, ds.blk_excl, ltarget);
      if (lane == 0) ds.bonus = v;
    }
    __syncthreads();
  }
  if (ds.bonus < 0) {  // the last token of the slice with r > 0
    int lastb = -1;
    for (int blk = nbk - 1 - tid; blk >= 0; blk -= kWalkThreads)
      if (bsum[blk] > 0.f) {
        lastb = blk;
        break;
      }
    lastb = __reduce_max_sync(0xffffffffu, lastb);
    if (lane == 0) ds.cnt[warp] = lastb;
    __syncthreads();
    if (warp == 0) {
      int blk = lane < kWalkWarps ? ds.cnt[lane] : -1;
      blk = __reduce_max_sync(0xffffffffu, blk);
      int v = -1;
      if (blk >= 0) {
        for (int e = lane; e < kBonusBlock; e += 32) {
          const int t = v0 + blk * kBonusBlock + e;
          if (t < v1 && r_of(__ldcg(tl + t), __ldcg(dl + t), scale2, lt, ld, a) > 0.f) v = t;
        }
      }
      v = __reduce_max_sync(0xffffffffu, v);
      if (lane == 0) ds.bonus = v;
    }
    __syncthreads();
  }
  const int v = ds.bonus;
  __syncthreads();  // ds is rewritten by the next draw
  return v;
}

// Global-memory hand-off between a request's leader and helper CTAs: one
// 64-bit word each way.  A word carries its whole message (the command
// number with the node and a, or with the slice sum) and neither side reads
// any other memory the other writes, so the words need no ordering against
// other accesses: relaxed loads and stores at GPU scope (single-copy atomic
// for an aligned 64-bit word), with no fence and no L1 invalidation per poll.
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* ptr) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed64(unsigned long long* ptr, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(ptr), "l"(v) : "memory");
}
// Waits until the word's bits from `shift` up equal `want`, for at most
// limit_ns of %globaltimer (read after the first poll, then every 32); the
// word read last goes to *got.
__device__ __forceinline__ bool poll_tag(const unsigned long long* ptr, int shift, unsigned long long want,
                                         unsigned long long* got, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (unsigned i = 1;; ++i) {
    const unsigned long long v = ld_relaxed64(ptr);
    if ((v >> shift) == want) {
      *got = v;
      return true;
    }
    if ((i & 31u) == 1u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ unsigned long long walk_cmd(unsigned seq, int u, float a) {
  return (static_cast<unsigned long long>(seq & 0xffffu) << 48) | (static_cast<unsigned long long>(u & 0xffff) << 32) |
         __float_as_uint(a);
}
// A bonus command in the node field: the flag, the slice whose owner draws
// (bits 10..14) and the path length (bits 0..9, at most TS_MAX_TREE, so never
// the stop word's 1023); the float is the target within that slice, or -1 for
// the slice's last token with r > 0.
constexpr int kWalkBonusFlag = 0x8000;
__device__ __forceinline__ unsigned long long walk_bonus_cmd(unsigned seq, int slice, int len, float ltarget) {
  return walk_cmd(seq, kWalkBonusFlag | (slice << 10) | len, ltarget);
}

// Node u's next child after node `after` (children in index order; parent[j]
// < j, so they all follow u), or -1: warp-wide, one ballot per 32 nodes.
__device__ __forceinline__ int next_child(const int* par_s, int n, int u, int after, int lane) {
  for (int w0 = (after + 1) & ~31; w0 < n; w0 += 32) {
    const int j = w0 + lane;
    const unsigned bal = __ballot_sync(0xffffffffu, j > after && j < n && par_s[j] == u);
    if (bal) return w0 + __ffs(bal) - 1;
  }
  return -1;
}

// The walk: walk_ctas CTAs per request.  CTA 0 (the leader) walks the tree;
// every pass (a rejection, or the bonus draw's slice totals) is a sum of
// max(0, p - a q) over the vocab that the leader and its helpers compute
// over their slices: the leader posts (command number, node, a) in the
// request's command word, helper k answers (command number, slice sum) in
// its slot, and the leader adds the slice sums in slice order.  A helper
// handles every command in order (the leader posts the next only after every
// helper has answered this one) until the last one, which it does not
// answer: the stop, or the bonus command, on which the helper that owns the
// bonus's slice draws it from its block sums and writes it while the others
// stop (when the leader owns that slice it draws the bonus itself and posts
// the stop).  Command numbers continue from one call to the next (the leader
// leaves the last one in the request's words), so no word is reset and a
// stale word never carries the number a CTA waits for.  The tree, the
// uniforms and the logits at the draft tokens are inputs of the call, final
// before the statistics kernel passed its own wait, which precedes this
// grid's launch: the leader reads them before waiting.  After the wait every
// CTA forms the log-sum-exps of all the request's nodes, and the leader p and
// q of every node's own token under its parent, so testing a child costs no
// memory round trip.  Warp 0 of the leader walks alone (a ballot lists a
// node's children) and the whole CTA joins it for each pass.  Every wait is
// bounded; one that runs out reports TS_DEVERR_TIMEOUT and ends the walk
// (the call's outputs are void and the workspace must be zeroed before its
// next use).  No CTA reads another's shared memory.
__global__ void __launch_bounds__(kWalkThreads) sample_walk_kernel(const SampleParams p) {
  const int K = p.walk_ctas;
  const int b = blockIdx.x / K, part = blockIdx.x % K;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nb = static_cast<int64_t>(b) * p.n_tree_max;
  const int rows = p.num_req * p.n_tree_max;
  const int V = p.vocab;
  WalkSync* const sync = p.sync + b;
  __shared__ float red[kWalkWarps];
  __shared__ float lt_s[TS_MAX_TREE], ld_s[TS_MAX_TREE];  // base-2 log-sum-exps of every node's rows
  __shared__ int par_s[TS_MAX_TREE], tok_s[TS_MAX_TREE];
  __shared__ float pc_s[TS_MAX_TREE], qc_s[TS_MAX_TREE];  // logits of node c's token under its parent, then p and q
  __shared__ int s_ok;
  __shared__ float bsum[kMaxBonusBlocks];  // this CTA's block sums of the last pass
  __shared__ DrawScratch ds;
  const int n = tree_size(p, b);  // the same for every CTA of the request
  float ua = 0.f, ub = 0.f;
  if (part == 0) {
    if (n != p.n_tree[b] && tid == 0) report_error(p.err, TS_DEVERR_BAD_LENGTH);
    if (tid < n) {
      int q = p.parent[nb + tid];
      if (q < -1 || q >= tid) {
        report_error(p.err, TS_DEVERR_BAD_PARENT);
        q = -1;
      }
      par_s[tid] = q;
      int t = p.tokens[nb + tid];
      if (t < 0 || t >= V) {
        if (tid > 0) report_error(p.err, TS_DEVERR_BAD_TOKEN);  // the root's own token is not tested
        t = -1;
      }
      tok_s[tid] = t;
      float xt = 0.f, xd = 0.f;
      if (q >= 0 && t >= 0) {
        const int64_t row = (nb + q) * V;
        xt = p.tl[row + t];
        xd = p.dl[row + t];
      }
      pc_s[tid] = xt;
      qc_s[tid] = xd;
      ua = p.u_acc[nb + tid];
      ub = p.u_bonus[nb + tid];
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  const unsigned base = static_cast<unsigned>(sync->last);  // the previous call's last command number
  if (tid < n) {  // node tid's two log-sum-exps from the statistics partials
    float m[2] = {-INFINITY, -INFINITY}, sm[2] = {0.f, 0.f};
    for (int j0 = 0; j0 < p.num_slices; j0 += 8) {  // eight slices of both rows requested together
      float2 x[2][8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
#pragma unroll
        for (int which = 0; which < 2; ++which)
          x[which][jj] = j0 + jj < p.num_slices
                             ? p.part[(static_cast<int64_t>(which) * rows + nb + tid) * p.num_slices + j0 + jj]
                             : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
#pragma unroll
        for (int which = 0; which < 2; ++which) lse_pair(m[which], sm[which], x[which][jj].x, x[which][jj].y);
    }
    lt_s[tid] = m[0] + log2f(sm[0]);
    ld_s[tid] = m[1] + log2f(sm[1]);
  }
  __syncthreads();
  // ======================= helpers =======================
  if (part > 0) {
    if (n == 0) return;  // the leader posts nothing
    __shared__ int s_u;
    __shared__ float s_a;
    int v0, v1;
    walk_slice(V, K, part, v0, v1);
    int last_u = 0;      // the node and a of the last pass
    float last_a = 0.f;
    for (unsigned seq = base + 1;; ++seq) {
      if (tid == 0) {
        unsigned long long c = 0;
        s_ok = poll_tag(&sync->cmd, 48, static_cast<unsigned long long>(seq & 0xffffu), &c, p.wait_ns);
        s_u = static_cast<int>((c >> 32) & 0xffff);
        s_a = __uint_as_float(static_cast<unsigned>(c));
        if (!s_ok) report_error(p.err, TS_DEVERR_TIMEOUT);
      }
      __syncthreads();
      if (!s_ok) return;
      const int u = s_u;
      if (u == kWalkStopNode) return;
      if (u & kWalkBonusFlag) {  // the bonus: drawn by the slice's owner from its last pass; the others stop
        if (((u >> 10) & 31) != part) return;
        const float ltarget = s_a;
        const int len = u & 1023;
        if (len < 1 || len > n || seq == base + 1) {  // no call posts this: a word the workspace held before
          if (tid == 0) report_error(p.err, TS_DEVERR_BAD_WORKSPACE);
          return;
        }
        const int64_t row = (nb + last_u) * V;
        const int v = draw_in_slice(p.tl + row, p.dl + row, v0, v1, p.scale2, lt_s[last_u], ld_s[last_u], last_a, bsum,
                                    ltarget, ltarget < 0.f, ds);
        if (tid == 0) {
          p.bonus[b] = v;
          if (p.verified != nullptr) p.verified[static_cast<int64_t>(b) * (p.n_tree_max + 1) + len] = v;
          if (p.verified_len != nullptr) p.verified_len[b] = len + 1;
        }
        return;
      }
      if (u >= n) {  // no call posts this: a word the workspace held before
        if (tid == 0) report_error(p.err, TS_DEVERR_BAD_WORKSPACE);
        return;
      }
      const int64_t row = (nb + u) * V;
      last_u = u;
      last_a = s_a;
      const float t = slice_pass(p.tl + row, p.dl + row, V, v0, v1, p.scale2, lt_s[u], ld_s[u], last_a, bsum, red);
      if (tid == 0)
        st_relaxed64(&sync->slot[part], (static_cast<unsigned long long>(seq) << 32) | __float_as_uint(t));
      __syncthreads();  // s_u, s_a are rewritten by the next command
    }
  }
  // ======================= leader =======================
  __shared__ int path_s[TS_MAX_TREE];
  __shared__ float ua_s[TS_MAX_TREE], ub_s[TS_MAX_TREE];  // the uniforms of every node
  __shared__ int s_op, s_u, s_len;
  __shared__ float s_a;
  __shared__ int s_slice;
  __shared__ float s_slice_excl;
  __shared__ float s_tot[kMaxWalkCtas];  // slice sums of the last pass
  if (tid < n) {
    const int q = par_s[tid], t = tok_s[tid];
    const bool real = q >= 0 && t >= 0;
    pc_s[tid] = real ? ex2_approx(fmaf(pc_s[tid], p.scale2, -lt_s[q])) : 0.f;
    qc_s[tid] = real ? ex2_approx(fmaf(qc_s[tid], p.scale2, -ld_s[q])) : 0.f;
    ua_s[tid] = ua;
    ub_s[tid] = ub;
  }
  if (tid == 0) {
    s_ok = 1;
    path_s[0] = 0;
  }
  __syncthreads();
  unsigned seq = base;  // commands posted
  // One pass: the slice sums of max(0, p - a q) over node u's rows into
  // s_tot[0 .. K), the leader's own slice first.  Returns their sum (slice order).
  auto pass = [&](int u, float a) -> float {
    ++seq;
    if (K > 1 && tid == 0) st_relaxed64(&sync->cmd, walk_cmd(seq, u, a));
    const int64_t row = (nb + u) * V;
    int v0, v1;
    walk_slice(V, K, 0, v0, v1);
    const float mine = slice_pass(p.tl + row, p.dl + row, V, v0, v1, p.scale2, lt_s[u], ld_s[u], a, bsum, red);
    if (tid == 0) s_tot[0] = mine;
    if (warp == 0 && lane + 1 < K) {  // lane k - 1 collects helper k's answer
      unsigned long long v = 0;
      if (poll_tag(&sync->slot[lane + 1], 32, static_cast<unsigned long long>(seq), &v, p.wait_ns)) {
        s_tot[lane + 1] = __uint_as_float(static_cast<unsigned>(v));
      } else {
        report_error(p.err, TS_DEVERR_TIMEOUT);
        s_ok = 0;
      }
    }
    __syncthreads();
    float total = 0.f;
    for (int k = 0; k < K; ++k) total += s_tot[k];
    return total;
  };
  int len = 0, bonus = -1;
  bool drawn_by_helper = false;
  if (n > 0) {
    // Warp 0's walk state (the same in every lane): node wu, the last child
    // tried at wu, and r = max(0, p - wa q) / sa at wu; tot_a is the a that
    // s_tot holds slice sums for (-1: none).
    int wu = 0, after = 0, wlen = 1;
    float wa = 0.f, sa = 1.f, tot_a = -1.f;
    constexpr int kOpReject = 1, kOpBonusSums = 2, kOpBonus = 3;
    for (;;) {
      if (warp == 0) {
        int op = kOpBonus;
        float pa = 0.f;  // the pass's a
        for (;;) {  // children of wu in index order, until a rejection or none is left
          const int c = next_child(par_s, n, wu, after, lane);
          if (c < 0) break;
          // U < r(t) / q(t) with r = max(0, p - wa q) / sa, as U q(t) sa <
          // max(0, p(t) - wa q(t)) (sa > 0): no division, and with q(t) = 0 it
          // reads r(t) > 0
          const float qt = qc_s[c];
          const bool acc = tok_s[c] >= 0 && ua_s[c] * qt * sa < fmaxf(0.f, pc_s[c] - wa * qt);
          after = c;
          if (acc) {  // c becomes the current node, with r = p at c
            if (lane == 0) path_s[wlen] = c;
            ++wlen;
            wu = c;
            wa = 0.f;
            sa = 1.f;
            tot_a = -1.f;
            continue;
          }
          op = kOpReject;  // r becomes max(0, p - (wa + sa) q) / S(wa + sa), kept if S is 0
          pa = wa + sa;
          break;
        }
        if (op == kOpBonus) {
          pa = wa;  // the bonus draws from r at the node where the walk ended
          if (tot_a != wa) op = kOpBonusSums;  // and needs its slice sums
        }
        if (lane == 0) {
          s_op = op;
          s_u = wu;
          s_a = pa;
          s_len = wlen;
        }
      }
      __syncthreads();
      const int op = s_op;
      if (op == kOpBonus) break;
      const float z = pass(s_u, s_a);
      if (!s_ok || op == kOpBonusSums) break;
      if (warp == 0) {
        if (z > 0.f) {
          wa += sa;  // the pass's a
          sa = z;
          tot_a = wa;
        } else {
          tot_a = -1.f;  // s_tot holds the sums for wa + sa, not for the wa that is kept
        }
      }
    }
    len = s_len;
    if (s_ok) {
      // ---- the bonus: the smallest v with r(0) + ... + r(v) > U * sum(r),
      //      r = max(0, p - a q) unnormalised: the slice that holds the
      //      target from the last pass's slice sums (a pass at this a), then,
      //      in the CTA that owns that slice, a scan of its block sums from
      //      that pass and a scan inside the block
      const int u = s_u;
      const float a = s_a;
      float total = 0.f;
      for (int k = 0; k < K; ++k) total += s_tot[k];
      const float target = ub_s[u] * total;
      if (tid == 0) {
        float excl = 0.f;
        int sl = -1, last_pos = -1;
        for (int k = 0; k < K; ++k) {
          if (s_tot[k] > 0.f) {
            last_pos = k;
            if (sl < 0 && excl <= target && target < excl + s_tot[k]) {
              sl = k;
              s_slice_excl = excl;
            }
          }
          excl += s_tot[k];
        }
        if (sl < 0) {  // rounding put the target at or past the total: the last slice with r > 0
          sl = last_pos;
          s_slice_excl = -1.f;  // take its last token with r > 0
        }
        s_slice = sl;
      }
      __syncthreads();
      const int sl = s_slice;
      const bool take_last = s_slice_excl < 0.f;
      const float ltarget = take_last ? -1.f : fmaxf(0.f, target - s_slice_excl);
      if (sl == 0) {  // the leader's own slice
        int v0, v1;
        walk_slice(V, K, 0, v0, v1);
        const int64_t row = (nb + u) * V;
        bonus = draw_in_slice(p.tl + row, p.dl + row, v0, v1, p.scale2, lt_s[u], ld_s[u], a, bsum, ltarget, take_last,
                              ds);
      } else if (sl > 0) {  // helper sl draws and writes the bonus; the command stops the other helpers
        drawn_by_helper = true;
        if (tid == 0) {
          st_relaxed64(&sync->cmd, walk_bonus_cmd(seq + 1, sl, len, ltarget));
          sync->last = seq + 1;
        }
      }
    }
    // the helpers stop (without answering); the next call's commands continue from here
    if (K > 1 && s_ok && !drawn_by_helper && tid == 0) {
      st_relaxed64(&sync->cmd, walk_cmd(seq + 1, kWalkStopNode, 0.f));
      sync->last = seq + 1;
    }
  }
  __syncthreads();
  // ---- outputs (the path written from shared memory; the bonus, its place
  //      in `verified` and verified_len by the helper that drew it, if one did)
  for (int j = tid; j < p.n_tree_max; j += kWalkThreads) p.path[nb + j] = j < len ? path_s[j] : -1;
  if (p.verified != nullptr) {
    int32_t* vrow = p.verified + static_cast<int64_t>(b) * (p.n_tree_max + 1);
    for (int j = tid; j <= p.n_tree_max; j += kWalkThreads) {
      if (j < len) vrow[j] = p.tokens[nb + path_s[j]];
      else if (j > len || n == 0) vrow[j] = -1;
      else if (!drawn_by_helper) vrow[j] = bonus;
    }
  }
  if (tid == 0) {
    p.accept_len[b] = len;
    if (!drawn_by_helper) {
      p.bonus[b] = bonus;
      if (p.verified_len != nullptr) p.verified_len[b] = n > 0 ? len + 1 : 0;
    }
  }
}

}  // namespace

cudaError_t launch_sample(const SampleParams& p, cudaStream_t stream) {
  const dim3 grid(2 * p.num_req * p.n_tree_max, p.num_slices);
  cudaError_t e = launch_pdl(sample_lse_kernel, grid, dim3(kLseThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(sample_walk_kernel, dim3(p.num_req * p.walk_ctas), dim3(kWalkThreads), 0, stream, p);
}

}  // namespace ts
