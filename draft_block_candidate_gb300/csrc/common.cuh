// Shared device helpers of the LiLiCorr sm_103a kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lilicorr.h"

namespace lilicorr {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Each translation unit with bounded waits keeps its own device-side error word; a
// kernel whose wait gives up ORs a site bit into it and returns.  The host reads and
// clears the words through lilicorr_device_error().
enum ErrSite : uint32_t {
  ERR_K1_FULL_WAIT = 1u << 0,
  ERR_K1_DRAIN = 1u << 1,
  ERR_K1_EMPTY_WAIT = 1u << 2,
};

// About one second at GB300 clocks: any wait longer than this is treated as a failure.
constexpr long long WAIT_LIMIT_CYCLES = 2000000000ll;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

// Non-blocking probe: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, at most `limit` SM cycles (default
// WAIT_LIMIT_CYCLES).  Returns false (and records `site`) if the limit was hit.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t* err_word, uint32_t site,
                                                  long long limit = WAIT_LIMIT_CYCLES) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0 && clock64() - t0 > limit) {
      atomicOr(err_word, site);
      return false;
    }
  }
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Barrier among the first nthreads (a multiple of 32) threads that use barrier id.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Ordered key of a float: signed-int comparison of keys matches float comparison
// (with -0.0 ordered just below +0.0, which only ever loosens a lower bound).
__device__ __forceinline__ int float_key(float f) {
  int b = __float_as_int(f);
  return b >= 0 ? b : (b ^ 0x7fffffff);
}
__device__ __forceinline__ float key_float(int k) {
  return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff));
}

// Split an f32 value into bf16 hi + bf16 lo with hi + lo == v to ~16 significant bits.
__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}
// The same for a pair, as packed words (a in the low half): one paired conversion per
// word instead of two single ones (the conversions, not the arithmetic, set the pace of the
// split epilogues).  Bit-identical to split_bf16 on each element.
__device__ __forceinline__ void split2_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const uint32_t hw = *reinterpret_cast<const uint32_t*>(&h);
  const __nv_bfloat162 l2 = __floats2bfloat162_rn(a - __uint_as_float(hw << 16),
                                                  b - __uint_as_float(hw & 0xffff0000u));
  hi = hw;
  lo = *reinterpret_cast<const uint32_t*>(&l2);
}

// Programmatic dependent launch.  pdl_wait: every memory access of the kernel comes after
// it; it returns once the kernel before this one on the stream has completed and its
// writes are visible (at once when this launch was not programmatic).  pdl_trigger: the
// next kernel on the stream may start launching (its CTAs then wait in their own
// pdl_wait); issued right after the wait, so that the next kernel's launch and set-up
// overlap this one.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// x * sigmoid(x); fast exponential and division (relative error ~1e-6, below the
// ~16-bit precision the split operands carry).
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

}  // namespace lilicorr

// Host-side launch bookkeeping (defined in lilicorr_api.cu).
namespace lilicorr {
void note_launch(int n = 1);
}
