// quarot_legacy_imma_probe: the issue rate of the legacy warp-level
// tensor-core instructions (mma.sync, s8 m16n8k32, s4 m16n8k64, and the fp16
// m16n8k16 with fp32 accumulators) on this GPU, measured by a launch that does
// nothing else.
//
// Why it exists: "QuaRot: Outlier-Free 4-Bit Inference in Rotated LLMs"
// (paper summary), "Kernel Implementation and Hardware Efficiency", runs its
// 4-bit GEMM as CUTLASS INT4 warp-level MMAs on Ampere.  sm_103a keeps those
// instructions for compatibility only; its W4A4 GEMM here runs on tcgen05
// (kind::f8f6f4).  The probe gives the integer rate the pages' kernel class
// would reach on this chip, the context for reporting the tcgen05 GEMM's
// throughput as a fraction of an "INT8 tensor core" peak.  The fp16 form is
// the instruction of this library's decode and prefill attention kernels, so
// its rate bounds their tensor-core share.
//
// Every warp keeps eight independent accumulator chains in registers, so the
// rate is limited by the tensor pipe, not by the dependency latency; operands
// come from registers and nothing touches memory but one guarded store.
#include "common.cuh"

namespace quarot {
namespace imma {

constexpr int kThreads = 256;
constexpr int kChains = 8;
constexpr int kBlocksPerSm = 4;

__device__ __forceinline__ void mma_s8(int32_t* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_f16(float* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_s4(int32_t* c, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k64.row.col.s32.s4.s4.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) imma_probe_kernel(int iters, int32_t* sink) {
  const uint32_t t = threadIdx.x + 1u;
  const uint32_t a[4] = {t * 0x01030507u, t * 0x0b0d1113u, t * 0x17191d1fu, t * 0x25292b2fu};
  const uint32_t b[2] = {t * 0x35373b3du, t * 0x43474953u};
  int32_t c[kChains][4];
#pragma unroll
  for (int j = 0; j < kChains; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0;
#pragma unroll 1
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) {
      if constexpr (BITS == 8) mma_s8(c[j], a, b);
      else mma_s4(c[j], a, b);
    }
  }
  int32_t s = 0;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s ^= c[j][0] ^ c[j][1] ^ c[j][2] ^ c[j][3];
  if (s == 0x13572468) sink[0] = s;  // keeps the chains live; practically never taken
}

__global__ void __launch_bounds__(kThreads) hmma_probe_kernel(int iters, int32_t* sink) {
  const uint32_t t = threadIdx.x + 1u;
  // small fp16 operands (exponent fields 12..13, about 2^-3): the
  // accumulators stay finite over any trip count the caller can pass
  const uint32_t a[4] = {0x30003000u | (t & 0x03FF03FFu), 0x31003100u | (t & 0x00FF00FFu),
                         0x32003200u | (t & 0x007F007Fu), 0x33003300u | (t & 0x003F003Fu)};
  const uint32_t b[2] = {0x34003400u | (t & 0x001F001Fu), 0x35003500u | (t & 0x000F000Fu)};
  float c[kChains][4];
#pragma unroll
  for (int j = 0; j < kChains; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
#pragma unroll 1
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kChains; ++j) mma_f16(c[j], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kChains; ++j) s += (c[j][0] + c[j][1]) + (c[j][2] + c[j][3]);
  if (s == 1.2345678f) sink[0] = 1;  // keeps the chains live; practically never taken
}

}  // namespace imma
}  // namespace quarot

extern "C" int quarot_legacy_imma_probe(int bits, int iters, int32_t* sink, int64_t* ops, void* stream) {
  using namespace quarot::imma;
  if ((bits != 8 && bits != 4 && bits != 16) || iters <= 0 || sink == nullptr || ops == nullptr)
    return QUAROT_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(sink) & 3) return QUAROT_ERR_ALIGNMENT;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return QUAROT_ERR_CUDA;
  const int blocks = sms * kBlocksPerSm;
  const int64_t k = bits == 8 ? 32 : bits == 4 ? 64 : 16;
  // 2 ops (multiply, add) per MAC of each 16 x 8 x k instruction
  *ops = int64_t(blocks) * (kThreads / 32) * int64_t(iters) * kChains * (2 * 16 * 8 * k);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (bits == 8)
    imma_probe_kernel<8><<<blocks, kThreads, 0, st>>>(iters, sink);
  else if (bits == 4)
    imma_probe_kernel<4><<<blocks, kThreads, 0, st>>>(iters, sink);
  else
    hmma_probe_kernel<<<blocks, kThreads, 0, st>>>(iters, sink);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}
