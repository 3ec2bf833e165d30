// Device helpers shared by the kernels: PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor),
// and the 5th-generation tensor core (tcgen05: TMEM allocation, MMA, commit, TMEM loads),
// plus bounded waits that report a timeout instead of hanging.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Bits of the workspace error word.
enum : int {
  DEVERR_TOKEN_ID = 1,     // token id outside [0, vocab) (clamped)
  DEVERR_TID2EID = 2,      // tid2eid entry outside [0, E) (clamped)
  DEVERR_TOPK_ID = 4,      // topk id outside [0, E) (clamped)
  DEVERR_TIMEOUT = 8,      // a pipeline wait exceeded its limit; the kernel stopped early
  DEVERR_BOUNDS = 16,      // (MOE_DEBUG_BOUNDS builds) an internal row index out of range; skipped
};

// MOE_DEBUG_BOUNDS=1 builds check internal row indices before they are used to address memory
// (dispatch rows, grouped-GEMM output rows, combine rows).  A failed check records DEVERR_BOUNDS
// in the error word and the access is skipped.  Default builds compile the checks away.
#ifndef MOE_DEBUG_BOUNDS
#define MOE_DEBUG_BOUNDS 0
#endif
__device__ __forceinline__ bool bad_index(long long i, long long n, int* err) {
#if MOE_DEBUG_BOUNDS
  if (i < 0 || i >= n) {
    if (err != nullptr) atomicOr(err, DEVERR_BOUNDS);
    return true;
  }
#endif
  return false;
}

// Longest a pipeline wait may last before the kernel gives up (2 s; a build may set it lower).
#ifndef MOE_WAIT_LIMIT_NS
#define MOE_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr unsigned long long WAIT_LIMIT_NS = MOE_WAIT_LIMIT_NS;

// Quiet period before a CTA that gave up a wait releases its shared memory and Tensor Memory.
// When a role stops early, asynchronous operations issued before (TMA loads into this CTA's
// shared memory, by this CTA or its pair peer; tensor-core MMAs reading it and writing Tensor
// Memory; the mbarrier arrivals of their commits) may still be completing.  None of them waits
// on anything once issued, and each completes within microseconds; 1 ms lets them all land.
constexpr unsigned long long QUIET_NS = 1000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// MOE_WAIT_HINT_NS > 0: ask the hardware to suspend a waiting thread up to that many ns (it
// resumes when the phase completes) instead of returning at once, so idle roles poll less
// (V4-Flash T=8192 layer: 3.17 -> 3.12 ms; 0.2 to 20 us measured alike).
#ifndef MOE_WAIT_HINT_NS
#define MOE_WAIT_HINT_NS 2000
#endif
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
#if MOE_WAIT_HINT_NS > 0
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(MOE_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after WAIT_LIMIT_NS, or as
// soon as another role of the CTA raised `abort_flag`; on a timeout it raises the flag and
// records DEVERR_TIMEOUT in the global error word.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort_flag = 1;
        atomicOr(err, DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// End of a warp-specialised kernel, called by every thread after its role's loop: a CTA barrier,
// then, if any role of this CTA gave up a wait, the quiet period (one thread sleeps, the others
// wait at a second barrier).  After the first barrier no role writes the flag any more, so every
// thread takes the same branch.
__device__ __forceinline__ void sync_and_quiesce(volatile int* abort_flag) {
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      const unsigned long long t0 = global_timer_ns();
      while (global_timer_ns() - t0 < QUIET_NS) __nanosleep(1000);
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------------------------- TMA

// 2-D tiled bulk tensor load global -> shared, completion counted on `bar` in bytes.
// Coordinates are (inner, outer) in elements; the inner one times the element size must be a
// multiple of 16 bytes (all callers pass multiples of 64 bf16 elements).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* tmap, uint32_t bar,
                                                 int32_t c0, int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// 3-D tiled load (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0, int32_t c1,
                                            int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// L2 eviction-priority policies for the cache-hint form.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------------------------------- tcgen05

// Allocate `ncols` TMEM columns (power of two >= 32); the base address is written to smem.
// Executed by one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// 16-byte shared-memory load.
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
// 16-byte shared-memory store.
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 16-byte global -> shared copy that bypasses L1 (cp.async.cg), completed through the per-thread
// commit / wait groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrive on a local mbarrier once all of this thread's earlier cp.async copies have landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Order this thread's completed generic-proxy writes to shared memory before later async-proxy
// reads of it (tensor-core operand loads), once a barrier has passed the ordering on.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of `row_bytes`
// (128 or 64 bytes: 64 or 32 bf16) with the matching swizzle that TMA's SWIZZLE_128B /
// SWIZZLE_64B writes: 8-row core-matrix groups 8*row_bytes apart (stride byte offset),
// descriptor version 1, layout type 2 (128B swizzle) or 4 (64B swizzle).  The tile base must
// be aligned to 8*row_bytes.
__device__ __forceinline__ uint64_t smem_desc_sw(uint32_t saddr, uint32_t row_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);            // start address >> 4, bits [0,14)
  d |= (uint64_t)(16u >> 4) << 16;                     // leading byte offset (unused here)
  d |= (uint64_t)((8u * row_bytes) >> 4) << 32;        // stride byte offset, bits [32,46)
  d |= (uint64_t)1 << 46;                              // descriptor version, bits [46,48)
  d |= (uint64_t)(row_bytes == 128 ? 2 : 4) << 61;     // swizzle mode, bits [61,64)
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 accumulator, both
// operands K-major, M = 128, N = n (multiple of 16, 16..256).
__device__ __forceinline__ uint32_t idesc_bf16_f32(uint32_t n) {
  return (1u << 4)            // accumulator format f32, bits [4,6)
         | (1u << 7)          // A format bf16, bits [7,10)
         | (1u << 10)         // B format bf16, bits [10,13)
         | ((n >> 3) << 17)   // N >> 3, bits [17,23)
         | ((128u >> 4) << 24);  // M >> 4, bits [24,29)
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with E4M3 A and B (format code 0 in both
// operand fields), fp32 accumulator, both operands K-major, M = 128, N = n (multiple of 16).
__device__ __forceinline__ uint32_t idesc_e4m3_f32(uint32_t n) {
  return (1u << 4)               // accumulator format f32, bits [4,6)
         | ((n >> 3) << 17)      // N >> 3, bits [17,23)
         | ((128u >> 4) << 24);  // M >> 4, bits [24,29)
}

// D[tmem] (+)= A[smem] * B[smem]^T on 8-bit operands (K = 32 per instruction), one thread.
__device__ __forceinline__ void tc_mma_f8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.  The
// registers are valid only after tmem_ld_wait(); pass them through reg_fence16() after the
// wait so that the compiler cannot move their first use above it.
// D (+)= A * B^T with A read from Tensor Memory at tmem_a (M = 128 rows in the 128 lanes, K = 16
// bf16 values packed two per 32-bit column, 8 columns) and B from shared memory.
__device__ __forceinline__ void tc_mma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Store 16 consecutive 32-bit columns of this warp's 32 TMEM lanes (lane quadrant warp % 4).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// Wait until this thread's tcgen05.st stores have completed.
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// ----------------------------------------------------------------------------- CTA pairs
// Helpers for kernels launched as clusters of two CTAs that share one 2-SM MMA
// (tcgen05 .cta_group::2): each CTA holds half of A (M/2 rows) and half of B (N/2 rows) in its
// own shared memory, and the even CTA of the pair issues the MMA for both.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the cluster shared-memory window, of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Arrive on an mbarrier of any CTA of the cluster, releasing this thread's prior writes
// (and, after tcgen05.fence::before_thread_sync, its completed TMEM reads) at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
#if MOE_WAIT_HINT_NS > 0
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(MOE_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}

// mbar_wait with cluster-scope acquire (for phases completed by arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  int* err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort_flag = 1;
        atomicOr(err, DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// 2-D tiled TMA load into this CTA's shared memory whose completion is counted on an mbarrier
// of either CTA of the pair (`bar_cluster` is a cluster-window address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// TMEM allocation shared by the CTA pair: one warp of EACH CTA executes these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Instruction descriptor for a 2-SM MMA: bf16 A/B, fp32 accumulator, K-major, M = 256.
__device__ __forceinline__ uint32_t idesc_bf16_f32_m256(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((256u >> 4) << 24);
}

// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]^T; issued by one thread of the
// even CTA.
__device__ __forceinline__ void tc_mma_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (+)= (A[smem] . 2^SFA) * (B[smem] . 2^SFB)^T: E2M1 A in the 16-byte-chunk form, E4M3 B, K = 32
// per instruction, UE8M0 scales read from Tensor Memory at sfa / sfb; issued by one thread.
__device__ __forceinline__ void tc_mma_mx(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with E2M1 A (format 5) and E4M3 B (format 0), fp32
// accumulator, both K-major, UE8M0 scales (bit 23), M = 128, N = n, B scale byte 0 (bits [4,6)),
// A scale byte `ida` (bits [29,31)).
__device__ __forceinline__ uint32_t idesc_mx_e2m1_e4m3(uint32_t n, uint32_t ida) {
  return (5u << 7)                // A format E2M1, bits [7,10)
         | ((n >> 3) << 17)       // N >> 3, bits [17,23)
         | (1u << 23)             // scale format UE8M0
         | ((128u >> 4) << 24)    // M >> 4, bits [24,29)
         | (ida << 29);           // A scale byte, bits [29,31)
}

// Store one 32-bit column of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// Arrive once on the mbarrier at offset `bar` in every CTA of `cta_mask` when all tcgen05
// operations issued so far by this thread complete.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// Named barrier for `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace moe
