// Device helpers: mbarriers with bounded waits, TMA tile loads, numeric unpacking.
// Hand-written PTX for sm_103a; every wait gives up after a fixed time and flags
// PSD_FAULT_WAIT_TIMEOUT instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/psd.h"
#include "kernels.h"

namespace psd {

// ~2 s at 2 GHz; no correct launch waits anywhere near this long.
constexpr long long kWaitLimitCycles = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Flags `bits` in a call's fault word (FaultRef): OR into the word when it carries
// the call's epoch, replace it otherwise.
__device__ __forceinline__ void raise_fault(const FaultRef &f, uint32_t bits) {
  unsigned long long seen = *reinterpret_cast<volatile unsigned long long *>(f.word);
  for (int tries = 0; tries < 64; ++tries) {
    const uint32_t mine = uint32_t(seen >> 32) == f.epoch ? uint32_t(seen) : 0u;
    const unsigned long long want = (static_cast<unsigned long long>(f.epoch) << 32) | (mine | bits);
    if (want == seen) return;
    const unsigned long long prev = atomicCAS(f.word, seen, want);
    if (prev == seen) return;
    seen = prev;
  }
}

// Waits for phase `parity` of the barrier; returns false (and flags the fault
// word) if it has not completed within `limit` cycles (kWaitLimitCycles unless a
// launch was given a shorter limit for testing).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const FaultRef &fault,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      raise_fault(fault, PSD_FAULT_WAIT_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t *fault) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) {
      atomicOr(fault, PSD_FAULT_WAIT_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start once every block of the kernel before it on the stream
// has called dependents_may_launch(); it must call wait_for_prior_grid() before it
// touches anything that kernel writes (the wait returns at once when there is no
// such kernel).
__device__ __forceinline__ void dependents_may_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void wait_for_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 4-D tiled TMA load into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two bf16 packed in a 32-bit word -> two floats (exact: a bf16 is the top half
// of an f32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two e4m3 codes (low 16 bits of w) -> two floats, exact, via the hardware
// e4m3x2 -> f16x2 conversion.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t w) {
  uint32_t h2;
  asm("{\n\t.reg .b16 lo;\n\tmov.b32 {lo, _}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(h2)
      : "r"(w));
  __half2 h = *reinterpret_cast<__half2 *>(&h2);
  return __half22float2(h);
}

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

}  // namespace psd
