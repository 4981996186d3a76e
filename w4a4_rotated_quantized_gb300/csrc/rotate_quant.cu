// quarot_rotate_quant: randomized Hadamard rotation of each row fused with
// per-token symmetric INT4 quantization and nibble packing.
//
// What it computes -- "QuaRot: Outlier-Free 4-Bit Inference in Rotated LLMs"
// (paper summary), section 3: Stage 1a (Q = H diag(s); d = 2^n m handled as a
// Kronecker product H_{2^n} (x) H_m), Stage 1b (online FWHT in FP32 before
// the quantized down-projection), Stage 2b (per-token scale max|x| / 7 with
// a clipping ratio) and "Kernel Implementation" (quantize, pack two INT4 per
// byte).  "QuaRot Guide: Outlier-Free 4-Bit W4A4 LLM Quantization": Sylvester
// doubling and the FWHT butterfly, round and clip to [-8, 7].  The 12288 case
// uses a Paley-12 block as in the QuaRot paper-viz explainer.
//
// Design (HBM-bound kernel): a group of TPR threads owns one row.
//   1. load pass   -- 16-byte vector loads of 8 fp16, sign flip, the three
//                     butterfly stages of index bits 0..2 in registers,
//                     store fp32 to a padded shared-memory row;
//   2. middle pass -- (rows with >= 256 power-of-two width) bits 3..7 as a
//                     radix-32 FWHT in registers, back to shared memory;
//   3. final pass  -- the remaining power-of-two bits and, for 12 * 2^n, the
//                     dense 12-point Paley transform, all values kept in
//                     registers; row abs-max, fp16 scale, round half-even,
//                     clamp, code bytes to shared memory;
//   4. pack        -- 8 codes -> one 32-bit coalesced store.
// Padding: element i lives at i + 4 * (i >> 7) so that the strided passes
// are free of shared-memory bank conflicts while 8-element chunks stay
// 16-byte aligned.
#include "common.cuh"

namespace quarot {

// ----------------------------------------------------------- Paley-12 table
// H12 = I + S, S = [[0, 1^T], [-1, Q]], Q_ij = chi(j - i) with chi the
// Legendre symbol mod 11 (nonzero squares mod 11: 1, 3, 4, 5, 9).
__host__ __device__ constexpr int legendre11(int a) {
  a = ((a % 11) + 11) % 11;
  return a == 0 ? 0 : ((a == 1 || a == 3 || a == 4 || a == 5 || a == 9) ? 1 : -1);
}
__host__ __device__ constexpr int paley12_entry(int i, int j) {
  return i == j ? 1 : (i == 0 ? 1 : (j == 0 ? -1 : legendre11((j - 1) - (i - 1))));
}

__device__ __forceinline__ int pad_idx(int i) { return i + 4 * (i >> 7); }

// In-register FWHT of N values (natural order, unnormalized).
template <int N>
__device__ __forceinline__ void fwht_regs(float* v) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
}

template <int LOGP, bool M12>
struct RQPlan {
  static constexpr int P = 1 << LOGP;
  static constexpr int NA = M12 ? 12 : 1;
  static constexpr int D = NA * P;
  static constexpr bool HAS_MID = LOGP >= 8;
  static constexpr int FINAL_LO = HAS_MID ? 8 : 3;
  static constexpr int FINAL_BITS = LOGP - FINAL_LO;
  static constexpr int FJ = 1 << FINAL_BITS;     // power-of-two values per final group
  static constexpr int GROUP = FJ * NA;          // values per final group
  static constexpr int NGROUPS = D / GROUP;      // = 2^FINAL_LO
  static constexpr int TPR = (LOGP < 8) ? 8 : ((M12 || LOGP >= 13) ? 256 : 128);
  static constexpr int GPT = NGROUPS / TPR;      // final groups per thread
  static constexpr int RPC = (TPR >= 256) ? 1 : 256 / TPR;  // rows per CTA
  static constexpr int NT = TPR * RPC;
  static constexpr int ROW_STRIDE = D + 4 * (D / 128) + 4;  // floats
  static constexpr size_t SMEM = size_t(RPC) * (ROW_STRIDE * 4 + D) + 64 * 4;
  static_assert(GPT >= 1 && GPT * TPR == NGROUPS, "final pass must cover the groups exactly");
  static_assert(GPT * GROUP <= 64, "final pass register budget");
};

template <int LOGP, bool M12>
__global__ void __launch_bounds__(RQPlan<LOGP, M12>::NT)
rotate_quant_kernel(const __half* __restrict__ x, int64_t M, int64_t ld_x,
                    const int8_t* __restrict__ signs, float clip_ratio, uint8_t* __restrict__ q_out,
                    __half* __restrict__ scale_out, float* __restrict__ rot_out) {
  using PL = RQPlan<LOGP, M12>;
  constexpr int D = PL::D, P = PL::P, TPR = PL::TPR;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* red = reinterpret_cast<float*>(smem_raw);  // [64] cross-warp max
  float* rows = reinterpret_cast<float*>(smem_raw + 64 * 4);

  const int tid = threadIdx.x;
  const int r_local = tid / TPR;
  const int t = tid % TPR;
  const int64_t row = int64_t(blockIdx.x) * PL::RPC + r_local;
  const bool valid = row < M;
  float* buf = rows + r_local * PL::ROW_STRIDE;
  uint8_t* codes = reinterpret_cast<uint8_t*>(rows + PL::RPC * PL::ROW_STRIDE) + r_local * D;

  // ---- 1. load pass: bits 0..2
  const __half* xr = x + (valid ? row : 0) * ld_x;
  for (int c = t; c < D / 8; c += TPR) {
    float v[8];
    if (valid) {
      const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(xr + 8 * c));
      const float2 f0 = h2_to_f2(raw.x), f1 = h2_to_f2(raw.y), f2 = h2_to_f2(raw.z),
                   f3 = h2_to_f2(raw.w);
      v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
      v[4] = f2.x; v[5] = f2.y; v[6] = f3.x; v[7] = f3.y;
      if (signs != nullptr) {
        const uint2 sraw = __ldg(reinterpret_cast<const uint2*>(signs + 8 * c));
        const uint32_t sw[2] = {sraw.x, sraw.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int8_t s = static_cast<int8_t>((sw[i >> 2] >> (8 * (i & 3))) & 0xFF);
          v[i] = s < 0 ? -v[i] : v[i];
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    fwht_regs<8>(v);
    float4* dst = reinterpret_cast<float4*>(buf + pad_idx(8 * c));
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  __syncthreads();

  // ---- 2. middle pass: bits 3..7 (radix 32)
  if constexpr (PL::HAS_MID) {
    for (int q = t; q < D / 32; q += TPR) {
      const int base = (q & 7) + ((q >> 3) << 8);
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = buf[pad_idx(base + 8 * j)];
      fwht_regs<32>(v);
#pragma unroll
      for (int j = 0; j < 32; ++j) buf[pad_idx(base + 8 * j)] = v[j];
    }
    __syncthreads();
  }

  // ---- 3. final pass: remaining bits (+ Paley-12), values stay in registers
  constexpr int GPT = PL::GPT, FJ = PL::FJ, NA = PL::NA, FLO = PL::FINAL_LO;
  float v[GPT][NA][FJ];
  float amax = 0.f;
#pragma unroll
  for (int g = 0; g < GPT; ++g) {
    const int base = t + g * TPR;
#pragma unroll
    for (int a = 0; a < NA; ++a) {
#pragma unroll
      for (int j = 0; j < FJ; ++j) v[g][a][j] = buf[pad_idx(base + (j << FLO) + a * P)];
      if constexpr (FJ > 1) fwht_regs<FJ>(v[g][a]);
    }
    if constexpr (M12) {
#pragma unroll
      for (int j = 0; j < FJ; ++j) {
        float in[12], out[12];
#pragma unroll
        for (int a = 0; a < 12; ++a) in[a] = v[g][a][j];
#pragma unroll
        for (int c = 0; c < 12; ++c) {
          float acc = 0.f;
#pragma unroll
          for (int a = 0; a < 12; ++a) acc = paley12_entry(a, c) > 0 ? acc + in[a] : acc - in[a];
          out[c] = acc;
        }
#pragma unroll
        for (int c = 0; c < 12; ++c) v[g][c][j] = out[c];
      }
    }
  }
  // 1/sqrt(d): an exact power of two for even powers of two, otherwise the
  // correctly rounded fp32 quotient.
  float inv_sqrt_d;
  if constexpr (!M12 && (LOGP % 2 == 0)) inv_sqrt_d = 1.0f / float(1 << (LOGP / 2));
  else inv_sqrt_d = 1.0f / sqrtf(float(D));
#pragma unroll
  for (int g = 0; g < GPT; ++g)
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
      for (int j = 0; j < FJ; ++j) {
        v[g][a][j] *= inv_sqrt_d;
        amax = fmaxf(amax, fabsf(v[g][a][j]));
      }

  // row abs-max: lanes of the row, then warps of the row
  constexpr int LANES = TPR < 32 ? TPR : 32;
#pragma unroll
  for (int o = LANES / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if constexpr (TPR > 32) {
    constexpr int WPR = TPR / 32;
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = red[(r_local * WPR)];
#pragma unroll
    for (int w = 1; w < WPR; ++w) amax = fmaxf(amax, red[r_local * WPR + w]);
  }
  const __half S = quant_scale_fp16(amax, clip_ratio);
  const float inv = 1.0f / __half2float(S);
  if (valid && t == 0) scale_out[row] = S;

#pragma unroll
  for (int g = 0; g < GPT; ++g) {
    const int base = t + g * TPR;
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
      for (int j = 0; j < FJ; ++j) {
        const int idx = base + (j << FLO) + a * P;
        const float y = fminf(fmaxf(v[g][a][j] * inv, -8.0f), 7.0f);
        codes[idx] = static_cast<uint8_t>(nibble_rne(y));
        if (rot_out != nullptr && valid) rot_out[row * D + idx] = v[g][a][j];
      }
  }
  __syncthreads();

  // ---- 4. pack 8 codes per 32-bit store
  if (valid) {
    uint32_t* qrow = reinterpret_cast<uint32_t*>(q_out + row * (D / 2));
    for (int w = t; w < D / 8; w += TPR) {
      const uint2 cb = *reinterpret_cast<const uint2*>(codes + 8 * w);
      uint32_t packed = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        packed |= ((cb.x >> (8 * i)) & 0xFu) << (4 * i);
        packed |= ((cb.y >> (8 * i)) & 0xFu) << (4 * (i + 4));
      }
      __stcs(qrow + w, packed);
    }
  }
}

template <int LOGP, bool M12>
static int launch_rq(const void* x, int64_t M, int64_t ld_x, const int8_t* signs, float clip,
                     uint8_t* q, void* s, float* rot, cudaStream_t st) {
  using PL = RQPlan<LOGP, M12>;
  auto kern = rotate_quant_kernel<LOGP, M12>;
  static bool attr_set = false;  // per-process; sizes are below the opt-in limit
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(PL::SMEM)) !=
        cudaSuccess)
      return QUAROT_ERR_LAUNCH;
    attr_set = true;
  }
  const int64_t blocks = (M + PL::RPC - 1) / PL::RPC;
  if (blocks > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  kern<<<dim3(unsigned(blocks)), dim3(PL::NT), PL::SMEM, st>>>(
      static_cast<const __half*>(x), M, ld_x, signs, clip, q, static_cast<__half*>(s), rot);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

}  // namespace quarot

using namespace quarot;

extern "C" int quarot_rotate_quant(const void* x, int64_t M, int64_t d, int64_t ld_x,
                                   const int8_t* signs, float clip_ratio, uint8_t* q_out,
                                   void* scale_out, float* rot_out, void* stream) {
  if (M < 0 || d <= 0 || ld_x < d) return QUAROT_ERR_INVALID_ARG;
  if (!(clip_ratio > 0.f && clip_ratio <= 1.f)) return QUAROT_ERR_INVALID_ARG;
  if (M == 0) return QUAROT_OK;
  if (x == nullptr || q_out == nullptr || scale_out == nullptr) return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (ld_x % 8) || (reinterpret_cast<uintptr_t>(q_out) & 15) ||
      (reinterpret_cast<uintptr_t>(scale_out) & 1) || (signs && (reinterpret_cast<uintptr_t>(signs) & 7)) ||
      (rot_out && (reinterpret_cast<uintptr_t>(rot_out) & 15)))
    return QUAROT_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (d) {
    case 16: return launch_rq<4, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 32: return launch_rq<5, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 64: return launch_rq<6, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 128: return launch_rq<7, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 256: return launch_rq<8, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 512: return launch_rq<9, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 1024: return launch_rq<10, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 2048: return launch_rq<11, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 4096: return launch_rq<12, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 8192: return launch_rq<13, false>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 3072: return launch_rq<8, true>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 6144: return launch_rq<9, true>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    case 12288: return launch_rq<10, true>(x, M, ld_x, signs, clip_ratio, q_out, scale_out, rot_out, st);
    default: return QUAROT_ERR_UNSUPPORTED;
  }
}
