// csa2_device.cuh -- device-side building blocks shared by the CSA2 kernels:
// error word, bounded mbarrier waits, TMA, tcgen05 (UMMA) descriptors and
// instructions, and the FP4 / FP8 numerics of the cache format.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "csa2_kernels.h"

namespace csa2 {

// ---------------------------------------------------------------- errors
// Sticky device error word: bit 0 = a bounded wait ran out, bit 1 = a bad
// index was seen (and skipped).
constexpr uint32_t kErrTimeout = kErrTimeoutBit;
constexpr uint32_t kErrIndex = kErrIndexBit;

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// Bounds checks of the CSA2_DEBUG build (libcsa2_debug.so): a computed index
// that falls outside its buffer records kErrIndex in the device error word
// and the access is skipped.  In the normal build the check is `true` and
// compiles away.
#ifdef CSA2_DEBUG
#define CSA2_IN_BOUNDS(cond, err) \
  ((cond) ? true : (::csa2::set_error((err), ::csa2::kErrIndex), false))
#else
#define CSA2_IN_BOUNDS(cond, err) true
#endif

// ~2^31 cycles (about one second at GB300 clocks) before a wait gives up,
// unless the launch sets a limit of its own (csa2_cache_set_wait_limit).
constexpr long long kWaitCycles = 1ll << 31;
__device__ __forceinline__ long long wait_limit(long long cycles) {
  return cycles > 0 ? cycles : kWaitCycles;
}

// ---------------------------------------------------------------- smem / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread up to `ns` nanoseconds (it resumes
// when the phase completes), so waiting warps leave the issue slots to
// working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// mbar_wait for consumers that usually wait long: suspending try_wait.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t* err,
                                                long long limit = kWaitCycles) {
  if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
    if (clock64() - t0 > limit) {
      set_error(err, kErrTimeout);
      return false;
    }
  }
}

// Waits for the phase with the given parity; gives up after `limit` cycles,
// records kErrTimeout and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          long long limit = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) {
      set_error(err, kErrTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------- launch order
// A kernel launched with programmatic stream serialisation may be scheduled
// while the kernel before it in the stream is still finishing; this waits
// until that kernel has completed and its memory operations are visible (at
// once when there is no such predecessor).  Every kernel of this library
// launched that way calls it before touching global memory.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled bulk tensor load into shared memory, completion on `bar`.
// x is the innermost (column) coordinate in elements, y the row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 3-D tiled bulk tensor load (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, int32_t x,
                                            int32_t y, int32_t z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// L2 policy for data read exactly once in a stream much larger than L2
// (the indexer keys): its lines are the first to go, so that what other
// kernels keep in L2 (scores on their way to the top-k, prefetched gathers)
// is not pushed out by the stream.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// The loads above, with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int32_t x,
                                            int32_t y, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, int32_t x,
                                            int32_t y, int32_t z, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, int32_t c0, int32_t c1,
                                            int32_t c2, int32_t c3, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "l"(pol)
      : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of
// 16), completion on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
      "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
      "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Generic-proxy shared-memory writes become visible to the async proxy
// (tensor core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle.  K-major operands:
// rows of 128 B (64 bf16 along K), 8-row groups `sbo` bytes apart.  MN-major
// operands: 8 K-rows of 128 B (64 elements along MN) per atom, atoms along
// MN `lbo` bytes apart, 8-row groups along K `sbo` bytes apart.  Buffers are
// 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;           // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;           // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4)                         // D = f32
         | (1u << 7)                       // A = bf16
         | (1u << 10)                      // B = bf16
         | ((a_mn_major ? 1u : 0u) << 15)  // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)  // B major-ness
         | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once all prior tcgen05.mma of this thread have completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Warp-collective TMEM loads: thread i of the warp reads lane (base lane + i)
// and N consecutive 32-bit columns.  The wait is inside the same asm
// statement so that no use of the destination registers can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
      "14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// Two 16-column loads (addresses ta, tb), one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16],
                                            uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
      "14,%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%"
      "27,%28,%29,%30,%31}, [%33];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
        "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]),
        "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]),
        "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]),
        "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
      : "r"(ta), "r"(tb)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
      "14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Two x32 loads (columns at ta and at tb) under one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t (&a)[32],
                                            uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(ta), "r"(tb)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%"
      "13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- pinned loads
// Read-only global loads issued exactly where they are written (volatile
// asm: the compiler neither sinks them towards their use nor merges them),
// for prefetches whose results are consumed much later.
// 32 bytes (32-byte aligned) in one 256-bit load.
__device__ __forceinline__ void ldg_now_v8(const void* a, uint4& lo, uint4& hi) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y),
                 "=r"(hi.z), "=r"(hi.w)
               : "l"(a));
}

__device__ __forceinline__ uint4 ldg_now_v4(const void* a) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(a));
  return v;
}
__device__ __forceinline__ uint32_t ldg_now_u32(const void* a) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(a));
  return v;
}
__device__ __forceinline__ uint32_t ldg_now_u16(const void* a) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(a));
  return v;
}
__device__ __forceinline__ uint32_t ldg_now_u8(const void* a) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(a));
  return v;
}

// ---------------------------------------------------------------- clusters
// Rank of this CTA in its cluster (0 outside a cluster launch).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address in the shared window of cluster CTA `rank` of the variable that
// sits at `saddr` in this CTA's shared memory.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Cluster-wide barrier in two halves: every thread of every CTA of the
// cluster arrives (release: its shared-memory writes become visible to the
// cluster) and later waits (acquire).  The hardware guarantees that the
// CTAs of a cluster are resident together; all threads must take both.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive (release, cluster scope) on an mbarrier of another CTA of the
// cluster; `addr` comes from dsmem_addr.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
               : "memory");
}
// Bounded wait (acquire, cluster scope) for a phase that another CTA of the
// cluster completes.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      set_error(err, kErrTimeout);
      return false;
    }
  }
  return true;
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this CTA's shared memory into another CTA's, completing as
// transaction bytes on that CTA's mbarrier (`dst` and `bar` from dsmem_addr).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, const void* src, uint32_t bytes,
                                                  uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "r"(smem_u32(src)), "r"(bytes), "r"(bar)
      : "memory");
}
// Waits until the bulk copies issued by this thread have read their sources.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\ncp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ---------------------------------------------------------------- score keys
// Order-preserving 32-bit key of an fp32 score (-0 folded to +0): the
// sign bit is set for non-negative values, all bits are inverted for
// negative ones, so unsigned key order is score order.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
constexpr int kKeyHistBins = kKeyHistBinsHost;   // top 11 bits of the key

// ---------------------------------------------------------------- numerics
// E2M1 code of v (round to nearest, ties to the even code, saturating at 6);
// the sign bit of v becomes bit 3.  Decision boundaries are the midpoints of
// the grid {0, .5, 1, 1.5, 2, 3, 4, 6}; a midpoint goes to the code whose
// mantissa bit is 0.
__device__ __forceinline__ uint32_t e2m1_encode(float v) {
  const float a = fabsf(v);
  uint32_t c;
  if (a <= 0.25f) c = 0;
  else if (a < 0.75f) c = 1;
  else if (a <= 1.25f) c = 2;
  else if (a < 1.75f) c = 3;
  else if (a <= 2.5f) c = 4;
  else if (a < 3.5f) c = 5;
  else if (a <= 5.0f) c = 6;
  else c = 7;
  return c | ((__float_as_uint(v) >> 28) & 8u);
}

// UE8M0 scale byte for a block maximum (OCP MX: floor(log2 amax) - 2,
// biased by 127, clamped at 0; zero and subnormal maxima give byte 0).
__device__ __forceinline__ uint32_t ue8m0_for_amax(float amax) {
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  return (uint32_t)(e >= 2 ? e - 2 : 0);
}
__device__ __forceinline__ float ue8m0_value(uint32_t b) {
  return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// E4M3 (OCP FP8) byte of a non-negative value, round to nearest even with
// saturation at 448, via the hardware conversion.
__device__ __forceinline__ uint32_t e4m3_encode_rn_sat(float v) {
  return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  const float mag = e ? ldexpf((float)(8u + m), (int)e - 10) : ldexpf((float)m, -9);
  return (b & 0x80u) ? -mag : mag;
}

// Eight E2M1 codes (nibbles of `codes`, code i at bits 4i..4i+3) to eight
// bf16 values, packed two per word (code 2k in the low half of out[k]).
// The magnitude bytes come from two 8-entry byte tables via PRMT; the sign
// bit is moved into bit 15 of each half.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ void e2m1x8_to_bf16x8(uint32_t codes, uint32_t (&out)[4]) {
  // bf16 of 0, .5, 1, 1.5, 2, 3, 4, 6 = 0000 3F00 3F80 3FC0 4000 4040 4080 40C0
  constexpr uint32_t kLoA = 0xC0800000u, kLoB = 0xC0804000u;
  constexpr uint32_t kHiA = 0x3F3F3F00u, kHiB = 0x40404040u;
  const uint32_t s0 = codes & 0x7777u, s1 = (codes >> 16) & 0x7777u;
  // sign bytes: PRMT's sign-replicate mode copies bit 7 of the selected byte;
  // bit 7 of byte i holds the sign of code 2i+1, and after a shift by 4 the
  // sign of code 2i.
  const uint32_t ev = codes << 4;
  const uint32_t sg0 = prmt(ev, codes, 0xD9C8u) & 0x80808080u;  // codes 0..3
  const uint32_t sg1 = prmt(ev, codes, 0xFBEAu) & 0x80808080u;  // codes 4..7
  const uint32_t l0 = prmt(kLoA, kLoB, s0), h0 = prmt(kHiA, kHiB, s0) | sg0;
  const uint32_t l1 = prmt(kLoA, kLoB, s1), h1 = prmt(kHiA, kHiB, s1) | sg1;
  out[0] = prmt(l0, h0, 0x5140u);
  out[1] = prmt(l0, h0, 0x7362u);
  out[2] = prmt(l1, h1, 0x5140u);
  out[3] = prmt(l1, h1, 0x7362u);
}

// Value of an E2M1 code (sign bit 3): 0, 0.5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t m = code & 7u;
  const float mag = (m < 2u) ? 0.5f * (float)m : __uint_as_float((126u + (m >> 1)) << 23) *
                                                  (1.0f + 0.5f * (float)(m & 1u));
  return (code & 8u) ? -mag : mag;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

__device__ __forceinline__ uint32_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return (uint32_t)(*reinterpret_cast<uint16_t*>(&h));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Indexer score of one entry from its 32 head logits r (fp32 bits) and the
// query's head weights w (shared memory, 16-byte aligned):
//     sum_h w[h] * max(r[h], 0)
// summed in four fp32 chains (chain c takes heads h = c mod 4, in order),
// then (c0 + c1) + (c2 + c3).  Chains (0, 1) and (2, 3) run as the two lanes
// of packed f32x2 FMAs (each lane an fp32 fma, round to nearest), which
// halves the FMA issues; the ReLU stays one fmax per head.
__device__ __forceinline__ float relu_dot32(const float* w, const uint32_t (&r)[32]) {
  uint64_t a = 0, b = 0;   // (c0, c1), (c2, c3); +0.0f bits
#pragma unroll
  for (int h = 0; h < 32; h += 4) {
    const float4 wv = *reinterpret_cast<const float4*>(w + h);
    uint64_t w01, w23, x01, x23;
    asm("mov.b64 %0, {%1, %2};" : "=l"(w01) : "f"(wv.x), "f"(wv.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(w23) : "f"(wv.z), "f"(wv.w));
    asm("mov.b64 %0, {%1, %2};" : "=l"(x01)
        : "f"(fmaxf(__uint_as_float(r[h]), 0.0f)), "f"(fmaxf(__uint_as_float(r[h + 1]), 0.0f)));
    asm("mov.b64 %0, {%1, %2};" : "=l"(x23)
        : "f"(fmaxf(__uint_as_float(r[h + 2]), 0.0f)), "f"(fmaxf(__uint_as_float(r[h + 3]), 0.0f)));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(w01), "l"(x01));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(b) : "l"(w23), "l"(x23));
  }
  float c0, c1, c2, c3;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(c0), "=f"(c1) : "l"(a));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(c2), "=f"(c3) : "l"(b));
  return (c0 + c1) + (c2 + c3);
}

}  // namespace csa2
