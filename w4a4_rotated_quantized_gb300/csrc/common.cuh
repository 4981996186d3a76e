// Shared helpers of the sm_103a kernels: the device error word, bounded
// waits on mbarriers, and small PTX wrappers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/quarot.h"

namespace quarot {

// Device error word: one bit per status code, bit (1 << code).  A kernel
// sets the bit of QUAROT_ERR_TIMEOUT when a bounded wait expires;
// quarot_check_error() reads the word, clears it and maps the bits back.
extern __device__ unsigned int g_error_word;  // defined in abi.cu (relocatable device code)

// ~1 s: far above any legitimate wait, short enough to keep a shared GPU
// usable if a barrier is never satisfied.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Sizes the decode attention supports (quarot_decode_attn and its variants):
// head_dim 128 and up to 8 query heads per KV head.
constexpr int kDecodeHeadDim = 128;
constexpr int kDecodeMaxGroup = 8;

// Unique id (cuCtxGetId) of the calling thread's current CUDA context, or 0
// when no context is current or the driver cannot say.  Defined in abi.cu.
unsigned long long current_context_id();

// Dynamic shared memory above 48 KB is an attribute of a kernel in one CUDA
// context: set it the first time the kernel is launched in each context.
// ctx[d] remembers the context of device d (0..63) in which it was set; after
// a cudaDeviceReset (a new context, a new id) it is set again.  A device
// beyond 64 sets it every time.
struct AttrCache {
  std::atomic<unsigned long long> ctx[64];
};
template <typename Kernel>
inline bool smem_attr_once(Kernel* kern, int bytes, AttrCache& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const bool cached = dev >= 0 && dev < 64;
  if (cached) {
    const unsigned long long id = current_context_id();
    if (id != 0 && done.ctx[dev].load(std::memory_order_acquire) == id) return true;
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  if (cached) done.ctx[dev].store(current_context_id(), std::memory_order_release);
  return true;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_error(unsigned int code) { atomicOr(&g_error_word, 1u << (code & 31u)); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
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

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or `ns` elapse, instead of returning at once and spinning
// (a spinning waiter takes issue slots from the warps that share its
// scheduler, which are usually the ones it is waiting for).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// records QUAROT_ERR_TIMEOUT) if it does not within kWaitLimitNs, or if
// *abort is set by another thread of the CTA.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      record_error(QUAROT_ERR_TIMEOUT);
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- fp helpers
__device__ __forceinline__ float2 h2_to_f2(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}

// Round-half-even of y (|y| < 2^22) into a two's complement nibble: adding
// 1.5 * 2^23 in round-to-nearest-even fp32 leaves the integer in the low
// mantissa bits.
__device__ __forceinline__ uint32_t nibble_rne(float y) {
  return static_cast<uint32_t>(__float_as_int(__fadd_rn(y, 12582912.0f))) & 0xFu;
}

// The per-row scale of the symmetric INT4 quantizer, rounded to fp16.
__device__ __forceinline__ __half quant_scale_fp16(float absmax, float clip_ratio) {
  float s = fmaxf(clip_ratio * absmax, 1e-5f) / 7.0f;
  s = fminf(s, 65504.0f);
  return __float2half_rn(s);
}

}  // namespace quarot
