// Device helpers shared by the treespec kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA tensor loads, ldmatrix and the
// warp-level bf16 MMA; bounded waits that never hang; the tree-metadata
// builder (ancestor-or-self bitmasks); and the split-KV schedule used by the
// attention kernels and their merge.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "treespec.h"

namespace ts {

// A bounded wait gives up after this long (ns of %globaltimer) and reports
// TS_DEVERR_TIMEOUT instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch: wait for the previous grid in the stream
// (no-op when the kernel was not launched as a dependent), and allow the
// next grid to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report_error(unsigned* err_word, unsigned bits) {
  if (err_word) atomicOr(err_word, bits);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of whether the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most
// kWaitLimitNs of %globaltimer; returns false when the limit expires.  The
// loop spins on try_wait, which may suspend the thread in hardware until the
// phase completes.  One PTX block, so the wait adds no register pressure to
// the loop around it.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t.reg .u64 t0, t1;\n\t"
      "mov.u64 t0, %%globaltimer;\n"
      "LAB_WAIT:\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "@P1 bra.uni DONE;\n\t"
      "mov.u64 t1, %%globaltimer;\n\t"
      "sub.u64 t1, t1, t0;\n\t"
      "setp.lt.u64 P1, t1, %3;\n\t"
      "@P1 bra.uni LAB_WAIT;\n"
      "DONE:\n\t"
      "selp.u32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "l"(kWaitLimitNs)
      : "memory");
  return ok != 0;
}

// The same wait with a caller-given bound, for the kernels' bounded-wait
// variant (a test that makes a wait run out): it spins on the non-blocking
// test_wait, so the bound holds to the nanosecond.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t.reg .u64 t0, t1;\n\t"
      "mov.u64 t0, %%globaltimer;\n"
      "LAB_TEST:\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "@P1 bra.uni DONE_TEST;\n\t"
      "mov.u64 t1, %%globaltimer;\n\t"
      "sub.u64 t1, t1, t0;\n\t"
      "setp.lt.u64 P1, t1, %3;\n\t"
      "@P1 bra.uni LAB_TEST;\n"
      "DONE_TEST:\n\t"
      "selp.u32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "l"(limit_ns)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled TMA store from shared memory (bulk-group completion), the
// commit of the issued stores, and the waits: `.read` returns once the
// shared-memory source may be rewritten, the plain form once the writes are done.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// L2 policy for data read exactly once (streamed K/V): evicted first, so it
// does not push out data that is read again soon (the split partials).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- warp MMA
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x by the hardware approximation (ex2.approx, flush-to-zero): exact 0
// for x = -inf, relative error of a few ulp, far below the bf16 rounding the
// probabilities go through.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair holding (lo - bf16(lo), hi - bf16(hi)) given `rounded` = the
// bf16 pair of (lo, hi): the part of two fp32 values that one bf16 rounding drops.
__device__ __forceinline__ uint32_t bf16x2_residual(uint32_t rounded, float lo, float hi) {
  const __nv_bfloat162 r = *reinterpret_cast<const __nv_bfloat162*>(&rounded);
  return pack_bf16x2(lo - __low2float(r), hi - __high2float(r));
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a tile whose
// rows are 128 bytes and which TMA wrote with 128-byte swizzling from a
// 1024-byte-aligned base: chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return row * 128u + (((chunk ^ row) & 7u) << 4);
}

// ---------------------------------------------------------------- tree metadata
// Ancestor-or-self sets of the first n nodes of one tree, as 128-bit masks in
// shared memory, by pointer jumping: after round k every node has OR-ed in
// the sets of all ancestors less than 2^k hops away, so ceil(log2 n) rounds
// cover any depth below n.  A parent outside [-1, i) is reported and treated
// as -1.  `nthr` threads with ids `tid` in [0, nthr) take part (nthr >= 32);
// `sync()` must be a barrier over exactly those threads.
template <class Sync>
__device__ __forceinline__ void build_ancestor_masks(const int32_t* parent, int n, uint32_t (*anc)[4],
                                                     int* jmp, int tid, int nthr, unsigned* err_word,
                                                     Sync sync) {
  for (int i = tid; i < n; i += nthr) {
    int p = parent[i];
    if (p < -1 || p >= i) {
      report_error(err_word, TS_DEVERR_BAD_PARENT);
      p = -1;
    }
    jmp[i] = p;
#pragma unroll
    for (int w = 0; w < 4; ++w) anc[i][w] = (w == (i >> 5)) ? (1u << (i & 31)) : 0u;
  }
  sync();
  int rounds = 0;
  while ((1 << rounds) < n) ++rounds;
  for (int r = 0; r < rounds; ++r) {
    uint32_t a[4][4];
    int jn[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = tid + k * nthr;
      if (i < n) {
        const int q = jmp[i];
#pragma unroll
        for (int w = 0; w < 4; ++w) a[k][w] = anc[i][w] | (q >= 0 ? anc[q][w] : 0u);
        jn[k] = q >= 0 ? jmp[q] : -1;
      }
    }
    sync();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = tid + k * nthr;
      if (i < n) {
#pragma unroll
        for (int w = 0; w < 4; ++w) anc[i][w] = a[k][w];
        jmp[i] = jn[k];
      }
    }
    sync();
  }
}

// ---------------------------------------------------------------- split-KV schedule
// Work is cut into "units" (request b, KV head, row group) and each unit's
// keys into tiles of kBlockN.  Units are ordered request-major; the tiles of
// all units form one sequence of T tiles that CTA c takes the contiguous
// range [c*T/NC, (c+1)*T/NC) of.  A CTA that finishes a unit it did not
// start (or starts one it does not finish) writes a partial result into slot
// c + u, which is unique because ranges are monotone in c (if c covers unit u
// and c' > c covers u' then u' >= u).
__host__ __device__ __forceinline__ int64_t sched_begin(int c, int64_t T, int NC) {
  return (static_cast<int64_t>(c) * T) / NC;
}
// The CTA whose range holds tile t: the largest c with sched_begin(c) <= t.
__host__ __device__ __forceinline__ int sched_cta_of(int64_t t, int64_t T, int NC) {
  return static_cast<int>(((t + 1) * NC + T - 1) / T - 1);
}

// Cost-weighted split (the tcgen05 path).  The tile sequence is laid on a
// weighted line: the first tile of every unit weighs 1 + E, the others 1 (a
// unit segment ends in an epilogue that costs about E tiles of time, so a CTA
// whose range crosses unit boundaries should take fewer tiles).  With
// pos(t) = the weight before tile t and W = T + E * units, CTA c takes the
// tiles whose pos lies in [ceil(c W / NC), ceil((c + 1) W / NC)), i.e. the
// CTA of tile t is floor(pos(t) NC / W).  A unit of `tiles` tiles starting at
// weighted position pf: tile 0 at pf, tile j >= 1 at pf + E + j.
// (32-bit division when the operands fit: 64-bit division is a long
// software sequence on the GPU; the results are identical.)
__host__ __device__ __forceinline__ int64_t wsched_x(int c, int64_t W, int NC) {
  const int64_t num = static_cast<int64_t>(c) * W + NC - 1;
  if (num < (1ll << 31)) return static_cast<int64_t>(static_cast<uint32_t>(num) / static_cast<uint32_t>(NC));
  return num / NC;
}
// first tile (0 .. tiles, tiles meaning "past the unit") with pos >= pf + r
__host__ __device__ __forceinline__ int wsched_tile_in_unit(int64_t r, int E, int tiles) {
  const int j = r <= 0 ? 0 : (r <= E + 1 ? 1 : static_cast<int>(r - E));
  return j < tiles ? j : tiles;
}
__host__ __device__ __forceinline__ int wsched_cta_of_pos(int64_t pos, int64_t W, int NC) {
  const int64_t num = pos * NC;
  if (num < (1ll << 31) && W < (1ll << 31))
    return static_cast<int>(static_cast<uint32_t>(num) / static_cast<uint32_t>(W));
  return static_cast<int>(num / W);
}

}  // namespace ts
