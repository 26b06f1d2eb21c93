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
// once in vocab slices and keeps (max, sum of exp(z - max)) of z = logit / T.
// Kernel 2 (walk) runs one 1024-thread CTA per request: it merges a visited
// node's slices into the two log-sum-exps, lists its children with a ballot,
// tests the first child from two logits, and on each rejection makes one
// coalesced pass over the vocab that writes max(0, r - q) into a workspace
// row (two rows per request, swapped when the new residual is not all zero)
// and sums it (four 16-byte loads per row in flight per thread).  The bonus
// is drawn by inverse transform in three levels: coalesced sums of
// 128-token blocks, a block scan of those sums for the block that holds the
// target, and one warp's scan inside that block.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

constexpr int kLseThreads = 256;
constexpr int kWalkThreads = 512;
constexpr int kWalkWarps = kWalkThreads / 32;

__device__ __forceinline__ void lse_pair(float& m, float& s, float om, float os) {
  if (om > m) {
    s = s * expf(m - om) + os;
    m = om;
  } else if (om != -INFINITY) {
    s += os * expf(om - m);
  }
}

__device__ __forceinline__ int64_t nb_row(const SampleParams& p, int b) { return static_cast<int64_t>(b) * p.n_tree_max; }

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
        bm = fmaxf(bm, fmaxf(fmaxf(f[q].x, f[q].y), fmaxf(f[q].z, f[q].w)) * p.inv_t);
      if (bm > m) {
        s *= expf(m - bm);
        m = bm;
      }
#pragma unroll
      for (int q = 0; q < kLoads; ++q)
        s += (expf(f[q].x * p.inv_t - m) + expf(f[q].y * p.inv_t - m)) +
             (expf(f[q].z * p.inv_t - m) + expf(f[q].w * p.inv_t - m));
    }
  } else {
    for (int64_t x = v0 + threadIdx.x; x < v1; x += kLseThreads) lse_pair(m, s, __ldcs(lg + x) * p.inv_t, 1.f);
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

constexpr int kBonusBlock = 128;  // tokens per first-level block of the inverse transform
constexpr int kBlocksPerThread = 4;
constexpr int kMaxBonusBlocks = kBlocksPerThread * kWalkThreads;  // vocab <= 262144

// r(v) for the current node: from the target logits (no rejection yet) or
// from the residual row (unnormalised)
template <bool FROM_LOGITS>
__device__ __forceinline__ float r_of(float x, float inv_t, float lt) {
  return FROM_LOGITS ? expf(x * inv_t - lt) : x;
}

// One rejection: out = max(0, r - q) over the vocab (r = src scaled by
// r_scale), returns this thread's share of its sum.  Four 16-byte loads of
// each row in flight per thread.
template <bool FROM_LOGITS>
__device__ __forceinline__ float residual_pass(const float* __restrict__ src, const float* __restrict__ dl,
                                               float* __restrict__ out, int V, float inv_t, float lt, float ld,
                                               float r_scale) {
  float part = 0.f;
  if ((V & 3) == 0) {
    constexpr int kLoads = 4;
    const int V4 = V / 4;
    const float4* s4 = reinterpret_cast<const float4*>(src);
    const float4* d4 = reinterpret_cast<const float4*>(dl);
    float4* o4 = reinterpret_cast<float4*>(out);
    for (int x0 = threadIdx.x; x0 < V4; x0 += kLoads * kWalkThreads) {
      float4 a[kLoads], d[kLoads];
#pragma unroll
      for (int q = 0; q < kLoads; ++q) {
        const int x = x0 + q * kWalkThreads;
        if (x < V4) {
          a[q] = __ldcg(s4 + x);
          d[q] = __ldcg(d4 + x);
        }
      }
#pragma unroll
      for (int q = 0; q < kLoads; ++q) {
        const int x = x0 + q * kWalkThreads;
        if (x < V4) {
          float4 o;
          o.x = fmaxf(0.f, r_of<FROM_LOGITS>(a[q].x, inv_t, lt) * r_scale - expf(d[q].x * inv_t - ld));
          o.y = fmaxf(0.f, r_of<FROM_LOGITS>(a[q].y, inv_t, lt) * r_scale - expf(d[q].y * inv_t - ld));
          o.z = fmaxf(0.f, r_of<FROM_LOGITS>(a[q].z, inv_t, lt) * r_scale - expf(d[q].z * inv_t - ld));
          o.w = fmaxf(0.f, r_of<FROM_LOGITS>(a[q].w, inv_t, lt) * r_scale - expf(d[q].w * inv_t - ld));
          o4[x] = o;
          part += (o.x + o.y) + (o.z + o.w);
        }
      }
    }
  } else {
#pragma unroll 4
    for (int v = threadIdx.x; v < V; v += kWalkThreads) {
      const float res = fmaxf(0.f, r_of<FROM_LOGITS>(__ldcg(src + v), inv_t, lt) * r_scale -
                                       expf(__ldcg(dl + v) * inv_t - ld));
      out[v] = res;
      part += res;
    }
  }
  return part;
}

// Sums of r over blocks of kBonusBlock tokens (warp per block, coalesced),
// into bsum[0 .. ceil(V / kBonusBlock)).  16-byte rows: lane l takes tokens
// 4l .. 4l + 3 of a block, and a warp requests kBlocksInFlight blocks before
// it sums any, so a row of ~10^5 tokens is a few dozen dependent round trips
// per warp rather than one per block.
constexpr int kBlocksInFlight = 8;
template <bool FROM_LOGITS>
__device__ __forceinline__ void block_sums(const float* __restrict__ src, int V, float inv_t, float lt, float* bsum) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = (V + kBonusBlock - 1) / kBonusBlock;
  if ((V & 3) == 0) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
    for (int b0 = warp; b0 < nb; b0 += kBlocksInFlight * kWalkWarps) {
      float4 f[kBlocksInFlight];
      unsigned in = 0u;  // bit j: this lane's group of block j lies in the row
#pragma unroll
      for (int j = 0; j < kBlocksInFlight; ++j) {
        const int v = (b0 + j * kWalkWarps) * kBonusBlock + 4 * lane;  // a whole 16-byte group or none: V % 4 == 0
        f[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b0 + j * kWalkWarps < nb && v < V) {
          f[j] = __ldcg(s4 + v / 4);
          in |= 1u << j;
        }
      }
#pragma unroll
      for (int j = 0; j < kBlocksInFlight; ++j) {
        float t = 0.f;
        if ((in >> j) & 1u)
          t = (r_of<FROM_LOGITS>(f[j].x, inv_t, lt) + r_of<FROM_LOGITS>(f[j].y, inv_t, lt)) +
              (r_of<FROM_LOGITS>(f[j].z, inv_t, lt) + r_of<FROM_LOGITS>(f[j].w, inv_t, lt));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0 && b0 + j * kWalkWarps < nb) bsum[b0 + j * kWalkWarps] = t;
      }
    }
    return;
  }
  for (int blk = warp; blk < nb; blk += kWalkWarps) {
    float t = 0.f;
#pragma unroll
    for (int e = 0; e < kBonusBlock / 32; ++e) {
      const int v = blk * kBonusBlock + e * 32 + lane;
      if (v < V) t += r_of<FROM_LOGITS>(__ldcg(src + v), inv_t, lt);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) bsum[blk] = t;
  }
}

// Inside one block: the smallest token with excl + r(blk start .. v) > target
// (warp-wide: lane l holds tokens 4l .. 4l + 3 of the block), or -1.
template <bool FROM_LOGITS>
__device__ __forceinline__ int scan_block(const float* __restrict__ src, int V, float inv_t, float lt, int blk,
                                          float excl, float target) {
  const int lane = threadIdx.x & 31;
  float r4[4];
  float mine = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int v = blk * kBonusBlock + lane * 4 + e;
    r4[e] = v < V ? r_of<FROM_LOGITS>(__ldcg(src + v), inv_t, lt) : 0.f;
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
    if (pick < 0 && acc > target) pick = blk * kBonusBlock + lane * 4 + e;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, pick >= 0);
  return hit ? __shfl_sync(0xffffffffu, pick, __ffs(hit) - 1) : -1;
}

__global__ void __launch_bounds__(kWalkThreads) sample_walk_kernel(const SampleParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nb = static_cast<int64_t>(b) * p.n_tree_max;
  const int rows = p.num_req * p.n_tree_max;
  const int V = p.vocab;
  __shared__ int par_s[TS_MAX_TREE], tok_s[TS_MAX_TREE], kids[TS_MAX_TREE], path_s[TS_MAX_TREE];
  __shared__ int cnt[kWalkWarps];
  __shared__ float red[kWalkWarps];
  __shared__ float lse_t, lse_d;
  __shared__ int s_accept;
  __shared__ int s_bonus, s_blk;
  __shared__ float s_blk_excl;
  __shared__ float s_scan[kWalkWarps];
  __shared__ float bsum[kMaxBonusBlocks];
  const int n = tree_size(p, b);
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
  }
  __syncthreads();
  float* const row0 = p.resid + static_cast<int64_t>(b) * 2 * V;
  float* const row1 = row0 + V;
  int len = 0, bonus = -1;
  if (n > 0) {
    int u = 0;
    len = 1;
    if (tid == 0) path_s[0] = 0;
    for (int guard = 0; guard < n; ++guard) {
      // ---- the two log-sum-exps of node u (scaled logits)
      if (warp == 0) {
        for (int which = 0; which < 2; ++which) {
          float m = -INFINITY, s = 0.f;
          if (lane < p.num_slices) {  // num_slices <= 32
            const float2 ms = p.part[(static_cast<int64_t>(which) * rows + nb + u) * p.num_slices + lane];
            m = ms.x;
            s = ms.y;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
            lse_pair(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
          if (lane == 0) {
            if (which == 0) lse_t = m + logf(s);
            else lse_d = m + logf(s);
          }
        }
      }
      // ---- children of u in index order
      const bool kid = tid < n && par_s[tid] == u;
      const unsigned bal = __ballot_sync(0xffffffffu, kid);
      if (lane == 0 && warp < TS_MAX_TREE / 32) cnt[warp] = __popc(bal);
      __syncthreads();
      int before = 0, nk = 0;
      for (int w = 0; w < TS_MAX_TREE / 32; ++w) {
        if (w < warp) before += cnt[w];
        nk += cnt[w];
      }
      if (kid) kids[before + __popc(bal & ((1u << lane) - 1u))] = tid;
      __syncthreads();
      const float* tl = p.tl + (nb + u) * V;
      const float* dl = p.dl + (nb + u) * V;
      const float lt = lse_t, ld = lse_d;
      int mode = 0, cur = 0;  // mode 0: r = p_u (from the logits); 1: r = (residual row cur) / rsum
      float rsum = 1.f;
      int next = -1;
      for (int k = 0; k < nk; ++k) {
        const int c = kids[k];
        if (tid == 0) {
          const int t = tok_s[c];
          bool acc = false;
          if (t >= 0) {
            const float rt = mode == 0 ? expf(tl[t] * p.inv_t - lt) : (cur ? row1 : row0)[t] / rsum;
            const float qt = expf(dl[t] * p.inv_t - ld);
            acc = qt > 0.f ? (p.u_acc[nb + c] < rt / qt) : rt > 0.f;
          }
          s_accept = acc;
        }
        __syncthreads();
        if (s_accept) {
          next = c;
          break;
        }
        // rejected: the next r is norm(max(0, r - q)), written to the other row
        float* const dst = cur ? row0 : row1;
        const float part = mode == 0 ? residual_pass<true>(tl, dl, dst, V, p.inv_t, lt, ld, 1.f)
                                     : residual_pass<false>(cur ? row1 : row0, dl, dst, V, p.inv_t, lt, ld, 1.f / rsum);
        const float z = block_sum(part, red);  // also orders the writes before later reads
        if (z > 0.f) {
          mode = 1;
          cur ^= 1;
          rsum = z;
        }
      }
      if (next >= 0) {
        u = next;
        if (tid == 0) path_s[len] = u;
        ++len;
        __syncthreads();
        continue;
      }
      // ---- the bonus: smallest v with r(0) + ... + r(v) > U * sum(r):
      //      block sums, a scan of them for the block, a scan inside it
      const float* src = mode == 0 ? tl : (cur ? row1 : row0);
      if (mode == 0) block_sums<true>(src, V, p.inv_t, lt, bsum);
      else block_sums<false>(src, V, p.inv_t, lt, bsum);
      __syncthreads();
      const int nb = (V + kBonusBlock - 1) / kBonusBlock;
      // consecutive block sums per thread (nb <= kMaxBonusBlocks), block exclusive scan
      const int per = (nb + kWalkThreads - 1) / kWalkThreads;
      float bs[kBlocksPerThread];
      float mine = 0.f;
#pragma unroll
      for (int e = 0; e < kBlocksPerThread; ++e) {
        bs[e] = (e < per && tid * per + e < nb) ? bsum[tid * per + e] : 0.f;
        mine += bs[e];
      }
      float inc = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) s_scan[warp] = inc;
      if (tid == 0) {
        s_bonus = -1;
        s_blk = -1;
      }
      __syncthreads();
      if (warp == 0) {
        float w = lane < kWalkWarps ? s_scan[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += y;
        }
        if (lane < kWalkWarps) s_scan[lane] = w;  // inclusive warp totals
      }
      __syncthreads();
      const float total = s_scan[kWalkWarps - 1];
      const float target = p.u_bonus[nb_row(p, b) + u] * total;
      float excl = (warp > 0 ? s_scan[warp - 1] : 0.f) + inc - mine;
#pragma unroll
      for (int e = 0; e < kBlocksPerThread; ++e) {
        if (bs[e] > 0.f && excl <= target && target < excl + bs[e]) {
          s_blk = tid * per + e;
          s_blk_excl = excl;
        }
        excl += bs[e];
      }
      __syncthreads();
      if (warp == 0 && s_blk >= 0) {
        const int v = mode == 0 ? scan_block<true>(src, V, p.inv_t, lt, s_blk, s_blk_excl, target)
                                : scan_block<false>(src, V, p.inv_t, lt, s_blk, s_blk_excl, target);
        if (lane == 0) s_bonus = v;
      }
      __syncthreads();
      if (s_bonus < 0) {  // rounding put the target at or past the total: the last token with r > 0
        int last = -1;
        for (int blk = nb - 1 - tid; blk >= 0; blk -= kWalkThreads)
          if (bsum[blk] > 0.f) {
            last = blk;
            break;
          }
        last = __reduce_max_sync(0xffffffffu, last);
        if (lane == 0) cnt[warp] = last;
        __syncthreads();
        if (warp == 0) {
          int blk = lane < kWalkWarps ? cnt[lane] : -1;
          blk = __reduce_max_sync(0xffffffffu, blk);
          int v = -1;
          if (blk >= 0) {
            for (int e = lane; e < kBonusBlock; e += 32) {
              const int t = blk * kBonusBlock + e;
              if (t < V && (mode == 0 ? expf(__ldcg(src + t) * p.inv_t - lt) : __ldcg(src + t)) > 0.f) v = t;
            }
          }
          v = __reduce_max_sync(0xffffffffu, v);
          if (lane == 0) s_bonus = v;
        }
        __syncthreads();
      }
      bonus = s_bonus;
      break;
    }
  }
  __syncthreads();
  // ---- outputs (the path written from shared memory)
  for (int j = tid; j < p.n_tree_max; j += kWalkThreads) p.path[nb + j] = j < len ? path_s[j] : -1;
  if (p.verified != nullptr) {
    int32_t* vrow = p.verified + static_cast<int64_t>(b) * (p.n_tree_max + 1);
    for (int j = tid; j <= p.n_tree_max; j += kWalkThreads)
      vrow[j] = j < len ? p.tokens[nb + path_s[j]] : (j == len && n > 0 ? bonus : -1);
  }
  if (tid == 0) {
    p.accept_len[b] = len;
    p.bonus[b] = bonus;
    if (p.verified_len != nullptr) p.verified_len[b] = n > 0 ? len + 1 : 0;
  }
}

}  // namespace

cudaError_t launch_sample(const SampleParams& p, cudaStream_t stream) {
  const dim3 grid(2 * p.num_req * p.n_tree_max, p.num_slices);
  cudaError_t e = launch_pdl(sample_lse_kernel, grid, dim3(kLseThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(sample_walk_kernel, dim3(p.num_req), dim3(kWalkThreads), 0, stream, p);
}

}  // namespace ts
