// quarot_crosshead_rotate_quant: the online cross-head Hadamard of the
// attention output, fused with per-token INT4 quantization and packing.
//
// What it computes -- "QuaRot: Outlier-Free 4-Bit Inference in Rotated LLMs"
// (paper summary), Stage 1c, "The online Hadamard heads transform": a full
// Hadamard over the nh * dh concatenated head dimensions factors as
// (I_nh (x) H_dh)(H_nh (x) I_dh).  The head-wise factor is carried by the
// rotated values (the decode output stays in that basis), so the output
// projection's input only needs Z <- Z (H_nh (x) I_dh) online: a size-nh
// Walsh-Hadamard across heads at every in-head position.  Stage 2b quantizes
// the result per token (S = max|x~| / 7, clipping ratio) for the W4A4 output
// projection.
//
// Design: one CTA of dh threads per row.  Thread j loads element j of every
// head (fp16, coalesced across threads for each head), runs the nh-point FWHT
// in registers, scales by 1/sqrt(nh), and the row abs-max is reduced over the
// CTA; codes go to shared memory and leave as packed 32-bit words.
#include <math.h>

#include "common.cuh"

namespace quarot {
namespace crosshead {

template <int N>
__device__ __forceinline__ void fwht_n(float* v) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1)
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
}

template <int NH, int DH>
__global__ void __launch_bounds__(DH)
crosshead_quant_kernel(const __half* __restrict__ z, int64_t ld_z, float clip_ratio, uint8_t* __restrict__ q_out,
                       __half* __restrict__ scale_out, float* __restrict__ rot_out) {
  constexpr int D = NH * DH;
  constexpr int NW = DH / 32;
  __shared__ float red[NW];
  __shared__ __align__(16) uint8_t codes[D];
  const int j = threadIdx.x, lane = j & 31, w = j >> 5;
  const int64_t row = blockIdx.x;
  const __half* zr = z + row * ld_z;

  float v[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) v[h] = __half2float(zr[h * DH + j]);
  fwht_n<NH>(v);
  // 1/sqrt(nh): exact for even powers of two, else the correctly rounded quotient
  float s_norm;
  if constexpr (NH == 1) s_norm = 1.0f;
  else if constexpr (NH == 4) s_norm = 0.5f;
  else if constexpr (NH == 16) s_norm = 0.25f;
  else if constexpr (NH == 64) s_norm = 0.125f;
  else s_norm = 1.0f / sqrtf(float(NH));
  float amax = 0.f;
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    v[h] *= s_norm;
    amax = fmaxf(amax, fabsf(v[h]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[w] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < NW; ++i) amax = fmaxf(amax, red[i]);
  const __half S = quant_scale_fp16(amax, clip_ratio);
  const float inv = 1.0f / __half2float(S);
  if (j == 0) scale_out[row] = S;
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const float y = fminf(fmaxf(v[h] * inv, -8.0f), 7.0f);
    codes[h * DH + j] = static_cast<uint8_t>(nibble_rne(y));
    if (rot_out != nullptr) rot_out[row * D + h * DH + j] = v[h];
  }
  __syncthreads();
  // 8 codes (one 32-bit word) per step, coalesced
  uint32_t* qrow = reinterpret_cast<uint32_t*>(q_out + row * (D / 2));
  for (int wi = j; wi < D / 8; wi += DH) {
    const uint2 cb = *reinterpret_cast<const uint2*>(codes + 8 * wi);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      packed |= ((cb.x >> (8 * i)) & 0xFu) << (4 * i);
      packed |= ((cb.y >> (8 * i)) & 0xFu) << (4 * (i + 4));
    }
    qrow[wi] = packed;
  }
}

template <int NH, int DH>
static int launch(const void* z, int64_t M, int64_t ld_z, float clip, uint8_t* q, void* s, float* rot,
                  cudaStream_t st) {
  crosshead_quant_kernel<NH, DH><<<dim3(unsigned(M)), dim3(DH), 0, st>>>(static_cast<const __half*>(z), ld_z, clip, q,
                                                                         static_cast<__half*>(s), rot);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

template <int DH>
static int dispatch_nh(int64_t nh, const void* z, int64_t M, int64_t ld_z, float clip, uint8_t* q, void* s,
                       float* rot, cudaStream_t st) {
  switch (nh) {
    case 1: return launch<1, DH>(z, M, ld_z, clip, q, s, rot, st);
    case 2: return launch<2, DH>(z, M, ld_z, clip, q, s, rot, st);
    case 4: return launch<4, DH>(z, M, ld_z, clip, q, s, rot, st);
    case 8: return launch<8, DH>(z, M, ld_z, clip, q, s, rot, st);
    case 16: return launch<16, DH>(z, M, ld_z, clip, q, s, rot, st);
    case 32: return launch<32, DH>(z, M, ld_z, clip, q, s, rot, st);
    case 64: return launch<64, DH>(z, M, ld_z, clip, q, s, rot, st);
    default: return QUAROT_ERR_UNSUPPORTED;
  }
}

}  // namespace crosshead
}  // namespace quarot

extern "C" int quarot_crosshead_rotate_quant(const void* z, int64_t M, int64_t nh, int64_t dh, int64_t ld_z,
                                             float clip_ratio, uint8_t* q_out, void* scale_out, float* rot_out,
                                             void* stream) {
  using namespace quarot::crosshead;
  if (M < 0 || nh <= 0 || dh <= 0 || ld_z < nh * dh) return QUAROT_ERR_INVALID_ARG;
  if (!(clip_ratio > 0.f && clip_ratio <= 1.f)) return QUAROT_ERR_INVALID_ARG;
  if ((nh & (nh - 1)) != 0 || nh > 64 || (dh != 64 && dh != 128)) return QUAROT_ERR_UNSUPPORTED;
  if (M == 0) return QUAROT_OK;
  if (M > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  if (z == nullptr || q_out == nullptr || scale_out == nullptr) return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(z) & 1) || (reinterpret_cast<uintptr_t>(q_out) & 3) ||
      (reinterpret_cast<uintptr_t>(scale_out) & 1) || (rot_out && (reinterpret_cast<uintptr_t>(rot_out) & 3)))
    return QUAROT_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return dh == 64 ? dispatch_nh<64>(nh, z, M, ld_z, clip_ratio, q_out, scale_out, rot_out, st)
                  : dispatch_nh<128>(nh, z, M, ld_z, clip_ratio, q_out, scale_out, rot_out, st);
}
