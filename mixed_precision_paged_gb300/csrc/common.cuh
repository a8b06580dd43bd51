// common.cuh -- shared device helpers of the ekv kernels (sm_103a).
//
// mbarrier + TMA (cp.async.bulk.tensor) wrappers written as inline PTX, the shared
// memory swizzle that TMA applies, bounded waits and the sticky error word.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/ekv.h"

namespace ekv {

constexpr int kPage = 16;                 // tokens per page (page size 16)
constexpr int kMaxKvHeads = 8;
constexpr int kMaxBatch = 4096;
#ifdef EKV_TEST_WAIT_TIMEOUT
// Test build only (libekv_waittest.so): a short bound, so a test can run a wait out
constexpr uint64_t kWaitTimeoutNs = 5000000ull;      // 5 ms
#else
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;   // 1 s bound on every pipeline wait
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- sticky error word
// err[0] = ekv_status, err[1] = ekv_detail, err[2] = first offending index.
__device__ __forceinline__ void report_error(int* err, int code, int detail, int index) {
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = detail;
    err[2] = index;
  }
}

// ----------------------------------------------------------------------- mbarriers
// Release/acquire fence at GPU scope: lighter than __threadfence (a sequentially
// consistent fence); with a relaxed atomic after it (release) or before it (acquire) it
// forms the message-passing pattern of the PTX memory model.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Programmatic dependent launch (sm_90+). launch_dependents lets the next kernel of the
// stream, when it was launched with programmatic serialization, be scheduled once every
// CTA of this grid has executed it; wait blocks until the preceding grid has completed
// and its memory operations are visible (it returns at once when there is none).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

#ifdef EKV_TEST_WAIT_TIMEOUT
// Test build only: raise the byte count the barrier's current phase waits for, without
// arriving. Bytes that no copy delivers keep the phase open, so the wait on it runs out
// while no copy is left in flight.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
#endif

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Wait for the phase of `parity` to complete; gives up after kWaitTimeoutNs and
// returns false (the caller then reports EKV_DETAIL_TIMEOUT and winds down).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// --------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 4-D tiled bulk tensor load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

// 5-D tiled bulk tensor load global -> shared (see tma_load_4d).
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, int c3, int c4, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy global -> shared of `bytes` (multiple of 16; both addresses 16-byte
// aligned), completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 (cp.async, LSU path), and the
// wait for all of this thread's such copies.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Order this thread's generic-proxy reads of shared memory before the TMA (async-proxy)
// writes that refill it.
__device__ __forceinline__ void fence_reads_before_refill() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset inside a 1024-byte-aligned TMA box after the hardware swizzle:
// 128B mode XORs the 16-byte chunk index (bits 4..6) with bits 7..9, 64B mode XORs
// bits 4..5 with bits 7..8.
__device__ __forceinline__ uint32_t swz128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }
__device__ __forceinline__ uint32_t swz64(uint32_t off) { return off ^ (((off >> 7) & 3u) << 4); }

// ----------------------------------------------------------------- conversions
// Two E4M3 codes (low byte = first element) -> two fp16 values, exact.
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint16_t two_codes) {
  __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes), __NV_E4M3);
  return *reinterpret_cast<__half2*>(&r);
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two_codes) {
  return __half22float2(e4m3x2_to_half2(two_codes));
}

// Round two fp32 values to E4M3 (RN, saturating to +-448); low byte = x.
__device__ __forceinline__ uint16_t float2_to_e4m3x2(float x, float y) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(x, y), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ bool scale_ok(float s) { return s > 0.f && s <= 3.0e38f; }

// x / s rounded to nearest-even in fp32, from r = the correctly rounded reciprocal of s:
// q0 = RN(x * r) is within one ulp of x / s, the remainder x - q0 * s is exact in one
// FMA, and RN(q0 + rem * r) is the correctly rounded quotient (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J.
// Res. Dev. 34(1), 1990; Muller et al., Handbook of Floating-Point Arithmetic, Sec. 4.7).
// The sign of a zero quotient is restored from x (s > 0). Valid while nothing
// overflows or underflows: s a positive normal float, |x / s| far from the fp32 limits,
// which holds for fp16 x and s = absmax / 448 of fp16 values. The unit test checks it
// bit for bit against __fdiv_rn over that whole domain.
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float rem = __fmaf_rn(-q0, s, x);
  return copysignf(__fmaf_rn(rem, r, q0), x);
}

}  // namespace ekv
