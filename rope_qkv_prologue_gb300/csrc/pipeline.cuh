// Shared-memory staging pipeline for the streaming kernels (sm_103a):
// one producer warp moves whole token rows from HBM into a ring of shared-
// memory stages with bulk asynchronous copies (cp.async.bulk, completion
// counted in bytes on an mbarrier), and the consumer warps release a stage
// with an arrive on its "empty" mbarrier once they have read it.
//
// Every wait is bounded: after kWaitLimitNs of %globaltimer time without the
// phase completing, the waiting thread records kErrWaitTimeout in the
// library's device error word (a __device__ int whose address the host passes
// in the kernel arguments) and gives up; the kernel then drains the copies it
// issued (again bounded) and returns, so a broken pipeline never spins
// forever.
#pragma once

#include <stdint.h>

namespace qkvp {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kErrWaitTimeout = 1;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the other threads and to the bulk
// copy engine before first use (followed by __syncthreads by the caller).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete, for at most
// kWaitLimitNs. Returns false if it never did, after OR-ing kErrWaitTimeout
// into the library's device error word *err.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

// Grid-wide "who finished last" without a counter that would need clearing:
// CTA b publishes the call's generation in its own word flags[b]
// (release: everything it wrote before is visible to a reader that sees the
// flag), then an SC fence, then reads every CTA's word. The CTA whose fence
// comes last in the fences' total order sees every flag, so at least one CTA
// sees all of them; the first of those to swap the call's generation into
// the election word wins. Words left by earlier calls (other generations) or
// any initial contents count as "not arrived".
__device__ __forceinline__ void fence_sc_gpu() { asm volatile("fence.sc.gpu;" ::: "memory"); }
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One warp (all 32 lanes) of CTA `me` of `n`: publish, look, elect. Returns
// true (in every lane) for exactly one CTA of the call. The caller orders
// the data it publishes before this (a fence by every writer, then a barrier).
__device__ __forceinline__ bool warp_publish_and_elect(uint32_t* flags, uint32_t* elect, uint32_t me, uint32_t n,
                                                       uint32_t gen) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) st_relaxed_gpu(flags + me, gen);
  __syncwarp();
  fence_sc_gpu();
  bool all = true;
  for (uint32_t i = lane; i < n; i += 32) all &= ld_relaxed_gpu(flags + i) == gen;
  all = __all_sync(0xffffffffu, all);
  uint32_t won = 0;
  if (all && lane == 0) won = atomicExch(elect, gen) != gen ? 1u : 0u;
  return __shfl_sync(0xffffffffu, won, 0) != 0;
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The default L2 policy (lines age like any other).
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bulk copy global -> this CTA's shared memory; `bytes` and both addresses
// must be multiples of 16. Completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

}  // namespace qkvp
