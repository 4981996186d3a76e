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

// Nearest fp16 value (ties to even), kept in fp32.  For two fp16 operands
// the fp32 sum or product rounded this way equals the fp16 operation
// (fp32 carries more than 2 * 11 + 2 significand bits, so the double rounding
// is harmless).
__device__ __forceinline__ float r16(float x) { return __half2float(__float2half_rn(x)); }

// In-register FWHT of N values (natural order, unnormalized).  H16: the FP16
// arithmetic variant, every butterfly output rounded to fp16.
template <int N, bool H16 = false>
__device__ __forceinline__ void fwht_regs(float* v) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        if constexpr (H16) {
          v[i] = r16(a + b);
          v[i + h] = r16(a - b);
        } else {
          v[i] = a + b;
          v[i + h] = a - b;
        }
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

// H16: the FP16-arithmetic rotation ([S] "Kernel Implementation and Hardware
// Efficiency": FP32 online Hadamard by default, FP16 as the alternative):
// y = fp16(s x h16_c) with h16_c = fp16(1/sqrt(d)), then every butterfly and
// every Paley-12 partial sum (in index order) rounded to fp16.
template <int LOGP, bool M12, bool RMS, bool H16 = false>
__global__ void __launch_bounds__(RQPlan<LOGP, M12>::NT)
rotate_quant_kernel(const __half* __restrict__ x, int64_t M, int64_t ld_x,
                    const int8_t* __restrict__ signs, float clip_ratio, float rms_eps, uint8_t* __restrict__ q_out,
                    __half* __restrict__ scale_out, float* __restrict__ rot_out, float h16_c) {
  static_assert(!(RMS && H16), "the FP16 variant has no fused RMSNorm");
  using PL = RQPlan<LOGP, M12>;
  constexpr int D = PL::D, P = PL::P, TPR = PL::TPR;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* red = reinterpret_cast<float*>(smem_raw);  // [64]: cross-warp max [0, 32), sum of squares [32, 64)
  float* rows = reinterpret_cast<float*>(smem_raw + 64 * 4);

  const int tid = threadIdx.x;
  const int r_local = tid / TPR;
  const int t = tid % TPR;
  const int64_t row = int64_t(blockIdx.x) * PL::RPC + r_local;
  const bool valid = row < M;
  float* buf = rows + r_local * PL::ROW_STRIDE;
  uint8_t* codes = reinterpret_cast<uint8_t*>(rows + PL::RPC * PL::ROW_STRIDE) + r_local * D;

  // ---- 1. load pass: bits 0..2 (and the row's sum of squares for RMSNorm)
  const __half* xr = x + (valid ? row : 0) * ld_x;
  float sq = 0.f;
  for (int c = t; c < D / 8; c += TPR) {
    float v[8];
    if (valid) {
      const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(xr + 8 * c));
      const float2 f0 = h2_to_f2(raw.x), f1 = h2_to_f2(raw.y), f2 = h2_to_f2(raw.z),
                   f3 = h2_to_f2(raw.w);
      v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
      v[4] = f2.x; v[5] = f2.y; v[6] = f3.x; v[7] = f3.y;
      if constexpr (RMS) {
#pragma unroll
        for (int i = 0; i < 8; ++i) sq = fmaf(v[i], v[i], sq);
      }
      if (signs != nullptr) {
        const uint2 sraw = __ldg(reinterpret_cast<const uint2*>(signs + 8 * c));
        const uint32_t sw[2] = {sraw.x, sraw.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int8_t s = static_cast<int8_t>((sw[i >> 2] >> (8 * (i & 3))) & 0xFF);
          v[i] = s < 0 ? -v[i] : v[i];
        }
      }
      if constexpr (H16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = r16(v[i] * h16_c);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    fwht_regs<8, H16>(v);
    float4* dst = reinterpret_cast<float4*>(buf + pad_idx(8 * c));
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  constexpr int LANES = TPR < 32 ? TPR : 32;  // lanes of one row within a warp
  if constexpr (RMS) {
#pragma unroll
    for (int o = LANES / 2; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if constexpr (TPR > 32) {
      if ((tid & 31) == 0) red[32 + (tid >> 5)] = sq;
    }
  }
  __syncthreads();

  // ---- 2. middle pass: bits 3..7 (radix 32)
  if constexpr (PL::HAS_MID) {
    for (int q = t; q < D / 32; q += TPR) {
      const int base = (q & 7) + ((q >> 3) << 8);
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = buf[pad_idx(base + 8 * j)];
      fwht_regs<32, H16>(v);
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
      if constexpr (FJ > 1) fwht_regs<FJ, H16>(v[g][a]);
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
          for (int a = 0; a < 12; ++a) {
            acc = paley12_entry(a, c) > 0 ? acc + in[a] : acc - in[a];
            if constexpr (H16) acc = r16(acc);
          }
          out[c] = acc;
        }
#pragma unroll
        for (int c = 0; c < 12; ++c) v[g][c][j] = out[c];
      }
    }
  }
  // 1/sqrt(d): an exact power of two for even powers of two, otherwise the
  // correctly rounded fp32 quotient.  With RMSNorm the row is also divided by
  // sqrt(mean(x^2) + eps) (the rotation preserves the row norm, so the sum of
  // squares of the input row serves).
  float inv_sqrt_d;
  if constexpr (!M12 && (LOGP % 2 == 0)) inv_sqrt_d = 1.0f / float(1 << (LOGP / 2));
  else inv_sqrt_d = 1.0f / sqrtf(float(D));
  float post = H16 ? 1.0f : inv_sqrt_d;  // the FP16 variant scaled on load
  if constexpr (RMS) {
    float tot = sq;
    if constexpr (TPR > 32) {
      constexpr int WPR = TPR / 32;
      tot = 0.f;
#pragma unroll
      for (int w = 0; w < WPR; ++w) tot += red[32 + r_local * WPR + w];
    }
    post = inv_sqrt_d * (1.0f / sqrtf(tot / float(D) + rms_eps));
  }
#pragma unroll
  for (int g = 0; g < GPT; ++g)
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
      for (int j = 0; j < FJ; ++j) {
        v[g][a][j] *= post;
        amax = fmaxf(amax, fabsf(v[g][a][j]));
      }

  // row abs-max: lanes of the row, then warps of the row
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

// ===================================================================== d = m x 1024
// Segment kernel for the hot widths d = 4096 (m = 4, Sylvester: H4 (x) H1024)
// and d = 12288 (m = 12, H12 (x) H1024).  Four warps own a row; warp w owns
// segments a = w * m/4 .. of 1024 elements.
//   pass 1  lane l loads 16-byte chunks l + 32 i (i = 0..3) of its segment:
//            element bits {0,1,2} (within the chunk) and {8,9} (i) are local;
//            sign flip on the fp16 bits, 32-point FWHT in registers, store to
//            the fp32 segment in shared memory transposed (one scalar store
//            per element, the warp's 32 lanes filling 32 consecutive words);
//   pass 2  lane l re-reads the 32 elements whose bits {0,1,2,8,9} equal l as
//            eight 16-byte loads, runs the 32-point FWHT over bits 3..7 and
//            stores them back in natural order;
//   pass 3  thread t takes elements 8t .. 8t+7 of every segment, applies the
//            m-point transform across segments (H4, or Paley-12 in the form
//            y_0 = x_0 - T, y_{j+1} = 2 (z_j + A_j) + y_0 with z = x_1..x_11,
//            T = sum z and A_j = sum of z_{j-r} over the quadratic residues r
//            of 11), then abs-max, fp16 scale, round, clamp and pack: one
//            32-bit store per segment.
// Packed fp32x2 arithmetic (__fadd2_rn / __ffma2_rn) carries the butterflies.
// Shared-memory layout between passes 2 and 3 (natural order): float4 slot V
// of a segment lives at V ^ (((V >> 6) & 3) << 1) ^ ((V >> 3) & 1), which
// keeps the strided scalar stores of pass 2 and the 16-byte loads of pass 3
// free of bank conflicts.  Between passes 1 and 2 (transposed) element bits
// g = {0,1,2,8,9} and k = 3..7 sit at word g * 32 + ((k >> 2) ^ (g & 7)) * 4 +
// (k & 3): pass 1's stores and pass 2's 16-byte loads are conflict-free, and
// pass 2's loads, which feed its butterflies, are 8 per lane instead of 32
// (27.7 -> 27.3 us at 2048 x 12288, bit-identical).
__device__ __forceinline__ int seg_swz(int V) { return V ^ (((V >> 6) & 3) << 1) ^ ((V >> 3) & 1); }

__device__ __forceinline__ void bfly2(float2& a, float2& b) {
  const float2 s = __fadd2_rn(a, b);
  b = __ffma2_rn(b, make_float2(-1.f, -1.f), a);
  a = s;
}
__device__ __forceinline__ void bfly_in(float2& a) {  // (x, y) -> (x + y, x - y)
  const float x = a.x, y = a.y;
  a = make_float2(x + y, x - y);
}

// 32-point FWHT of p[16] holding elements (2n, 2n+1) in p[n]: bit 0 inside
// each pair, bits 1..4 across pairs.
__device__ __forceinline__ void fwht32_pairs(float2* p) {
#pragma unroll
  for (int n = 0; n < 16; ++n) bfly_in(p[n]);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int n = 0; n < 16; ++n)
      if ((n & h) == 0) bfly2(p[n], p[n + h]);
}

template <int MSEG, bool STAGED>
struct SegPlan {
  static constexpr int D = MSEG * 1024;
  static constexpr int TPR = 128;
  static constexpr int SPW = MSEG / 4;  // segments per warp
  static constexpr int RPC = STAGED ? 1 : 2;
  static constexpr int NT = TPR * RPC;
  // [red 256 B][fp32 rows][fp16 staging row (STAGED)][mbarrier (STAGED)]
  static constexpr size_t OFF_BUF = 64 * 4;
  static constexpr size_t OFF_STAGE = OFF_BUF + size_t(RPC) * D * 4;
  static constexpr size_t OFF_MBAR = OFF_STAGE + (STAGED ? size_t(D) * 2 : 0);
  static constexpr size_t SMEM = OFF_MBAR + 16;
};

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// STAGED = true: persistent CTAs, one row at a time; while a row runs passes 2
// and 3, the next row's fp16 data arrives in a staging buffer by a bulk
// asynchronous copy, so the load latency of one row hides behind the
// arithmetic of the previous one.
//
// A8 = true writes the tensor-core operand form of the codes instead of
// packed nibbles: one byte per code holding u = v + 8 (the e4m3 byte whose
// value is u * 2^-9), in the order (0, 2, 4, 6, 1, 3, 5, 7) within each group
// of 8 codes, and the row's code sum sum_k v_k into rowsum_out[row].
template <int MSEG, bool STAGED, bool RMS, bool A8 = false, bool RS = false>
__global__ void __launch_bounds__(SegPlan<MSEG, STAGED>::NT, STAGED ? 3 : (RS ? 4 : 1))
rotate_quant_seg_kernel(const __half* __restrict__ x, int64_t M, int64_t ld_x, const int8_t* __restrict__ signs,
                        float clip_ratio, float rms_eps, uint8_t* __restrict__ q_out, __half* __restrict__ scale_out,
                        float* __restrict__ rot_out, int32_t* __restrict__ rowsum_out = nullptr) {
  using PL = SegPlan<MSEG, STAGED>;
  constexpr int D = PL::D;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* red = reinterpret_cast<float*>(smem_raw);
  const int tid = threadIdx.x;
  const int r_local = tid / PL::TPR;
  const int t = tid % PL::TPR;
  const int lane = t & 31, w = t >> 5;
  float4* buf = reinterpret_cast<float4*>(smem_raw + PL::OFF_BUF) + size_t(r_local) * (D / 4);
  const __half* stage = reinterpret_cast<const __half*>(smem_raw + PL::OFF_STAGE);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem_raw + PL::OFF_MBAR);
  const int64_t row_stride = STAGED ? int64_t(gridDim.x) : int64_t(0);
  int64_t row = STAGED ? int64_t(blockIdx.x) : int64_t(blockIdx.x) * PL::RPC + r_local;
  if constexpr (STAGED) {
    if (tid == 0) {
      mbar_init(mbar, 1);
      fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0 && row < M) {
      mbar_arrive_expect_tx(mbar, uint32_t(D) * 2u);
      bulk_copy_g2s(smem_u32(stage), x + row * ld_x, uint32_t(D) * 2u, mbar);
    }
  }
  for (int it = 0;; ++it, row += row_stride) {
  if constexpr (STAGED) {
    if (row >= M) break;
    if (!mbar_wait_bounded(mbar, uint32_t(it & 1), nullptr)) break;
  } else {
    if (it > 0) break;
  }
  const bool valid = row < M;
  const __half* xr = x + (valid ? row : 0) * ld_x;

  // ---- pass 1 (and the row's sum of squares for RMSNorm)
  float sq = 0.f;
  // the warp's segments unrolled: their load / butterfly / store chains are
  // independent and overlap (launch bounds hold the persistent 12288 kernel
  // at 3 CTAs per SM, and the two-row 4096 kernel with row sums at 4, i.e. 64
  // registers: without them it took 72 and ran 3 CTAs per SM)
#pragma unroll
  for (int sgi = 0; sgi < PL::SPW; ++sgi) {
    const int a = w * PL::SPW + sgi;
    float2 p[16];  // p[4 i + jj] = elements (2 jj, 2 jj + 1) of chunk lane + 32 i
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int chunk = lane + 32 * i;
      uint4 raw = make_uint4(0, 0, 0, 0);
      if constexpr (STAGED) raw = *reinterpret_cast<const uint4*>(stage + a * 1024 + 8 * chunk);
      else if (valid) raw = __ldcs(reinterpret_cast<const uint4*>(xr + a * 1024 + 8 * chunk));
      if (signs != nullptr) {
        const uint2 sg = __ldg(reinterpret_cast<const uint2*>(signs + a * 1024 + 8 * chunk));
        // sign bit of byte k of the sign word -> bit 15 / 31 of the fp16 pair
        raw.x ^= __byte_perm(sg.x, 0u, 0x1404) & 0x80008000u;
        raw.y ^= __byte_perm(sg.x, 0u, 0x3424) & 0x80008000u;
        raw.z ^= __byte_perm(sg.y, 0u, 0x1404) & 0x80008000u;
        raw.w ^= __byte_perm(sg.y, 0u, 0x3424) & 0x80008000u;
      }
      p[4 * i + 0] = h2_to_f2(raw.x);
      p[4 * i + 1] = h2_to_f2(raw.y);
      p[4 * i + 2] = h2_to_f2(raw.z);
      p[4 * i + 3] = h2_to_f2(raw.w);
      if constexpr (RMS) {
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2)
          sq = fmaf(p[4 * i + k2].x, p[4 * i + k2].x, fmaf(p[4 * i + k2].y, p[4 * i + k2].y, sq));
      }
    }
    fwht32_pairs(p);  // pair index n = 4 i + jj: bits 1,2 = jj, bits 3,4 = i
    // transposed for pass 2: element e with g = bits {0, 1, 2, 8, 9} and
    // k = bits 3..7 (here k = lane) at float g * 32 + ((k >> 2) ^ (g & 7)) * 4 + (k & 3)
    float* segf = reinterpret_cast<float*>(buf + a * 256);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int g0 = 2 * jj + 8 * i;
        segf[g0 * 32 + ((((lane >> 2) ^ (2 * jj)) << 2) | (lane & 3))] = p[4 * i + jj].x;
        segf[(g0 + 1) * 32 + ((((lane >> 2) ^ (2 * jj + 1)) << 2) | (lane & 3))] = p[4 * i + jj].y;
      }
  }
  __syncwarp();
  // per-warp partial sums of squares, double-buffered by row parity (a warp
  // can start the next row's pass 1 while another still reads this row's)
  if constexpr (RMS) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) red[16 + (it & 1) * 8 + r_local * 4 + w] = sq;
  }

  // ---- pass 2: bits 3..7; element e = (lane & 7) + 8 k + 256 (lane >> 3)
  {
    const int lh = lane >> 3;
    const int base0 = ((lane & 7) >> 2) | (lh << 6);  // float4 slot bits 0 and 6,7
    int addr[2][4];
#pragma unroll
    for (int par = 0; par < 2; ++par)
#pragma unroll
      for (int kl = 0; kl < 4; ++kl) addr[par][kl] = ((base0 ^ par) + 2 * (kl ^ lh)) * 4 + (lane & 3);
#pragma unroll
    for (int sgi = 0; sgi < PL::SPW; ++sgi) {
      const int a = w * PL::SPW + sgi;
      float* seg = reinterpret_cast<float*>(buf + a * 256);
      float2 p[16];
      // the lane's 32 values (g = lane, k = 0 .. 31) as 8 conflict-free 16-byte loads
      const float4* src = reinterpret_cast<const float4*>(seg) + lane * 8;
#pragma unroll
      for (int qd = 0; qd < 8; ++qd) {
        const float4 v4 = src[qd ^ (lane & 7)];
        p[2 * qd] = make_float2(v4.x, v4.y);
        p[2 * qd + 1] = make_float2(v4.z, v4.w);
      }
      __syncwarp();  // every lane has read the segment before it is rewritten in natural order
      fwht32_pairs(p);
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        seg[addr[(k >> 2) & 1][k & 3] + 32 * (k >> 2)] = p[k >> 1].x;
        seg[addr[(k >> 2) & 1][(k + 1) & 3] + 32 * (k >> 2)] = p[k >> 1].y;
      }
    }
  }
  __syncthreads();
  if constexpr (STAGED) {
    // every warp is past pass 1: the staging buffer may take the next row
    const int64_t next = row + row_stride;
    if (tid == 0 && next < M) {
      mbar_arrive_expect_tx(mbar, uint32_t(D) * 2u);
      bulk_copy_g2s(smem_u32(stage), x + next * ld_x, uint32_t(D) * 2u, mbar);
    }
  }

  // ---- pass 3: cross-segment transform on elements 8t .. 8t+7
  float2 v[MSEG][4];
#pragma unroll
  for (int a = 0; a < MSEG; ++a) {
    const float4 lo = buf[a * 256 + seg_swz(2 * t)];
    const float4 hi = buf[a * 256 + seg_swz(2 * t + 1)];
    v[a][0] = make_float2(lo.x, lo.y);
    v[a][1] = make_float2(lo.z, lo.w);
    v[a][2] = make_float2(hi.x, hi.y);
    v[a][3] = make_float2(hi.z, hi.w);
  }
  if constexpr (MSEG == 4) {
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      bfly2(v[0][jj], v[1][jj]);
      bfly2(v[2][jj], v[3][jj]);
      bfly2(v[0][jj], v[2][jj]);
      bfly2(v[1][jj], v[3][jj]);
    }
  } else {
    // Paley-12: z_j = v[1 + j], T = sum z, A_j = z_{j-1} + z_{j-3} + z_{j-4} + z_{j-5} + z_{j-9}
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      float2 z[11];
#pragma unroll
      for (int j = 0; j < 11; ++j) z[j] = v[1 + j][jj];
      const float2 t01 = __fadd2_rn(z[0], z[1]), t23 = __fadd2_rn(z[2], z[3]), t45 = __fadd2_rn(z[4], z[5]);
      const float2 t67 = __fadd2_rn(z[6], z[7]), t89 = __fadd2_rn(z[8], z[9]);
      const float2 T = __fadd2_rn(__fadd2_rn(__fadd2_rn(t01, t23), __fadd2_rn(t45, t67)), __fadd2_rn(t89, z[10]));
      const float2 y0 = __ffma2_rn(T, make_float2(-1.f, -1.f), v[0][jj]);
      v[0][jj] = y0;
#pragma unroll
      for (int j = 0; j < 11; ++j) {
        const float2 A = __fadd2_rn(__fadd2_rn(__fadd2_rn(z[(j + 10) % 11], z[(j + 8) % 11]),
                                               __fadd2_rn(z[(j + 7) % 11], z[(j + 6) % 11])),
                                    __fadd2_rn(z[(j + 2) % 11], z[j]));
        v[1 + j][jj] = __ffma2_rn(A, make_float2(2.f, 2.f), y0);
      }
    }
  }
  float am[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // independent partial maxima
#pragma unroll
  for (int a = 0; a < MSEG; ++a)
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      am[2 * jj] = fmaxf(am[2 * jj], fabsf(v[a][jj].x));
      am[2 * jj + 1] = fmaxf(am[2 * jj + 1], fabsf(v[a][jj].y));
    }
  float amax = fmaxf(fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3])), fmaxf(fmaxf(am[4], am[5]), fmaxf(am[6], am[7])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[r_local * 4 + w] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[r_local * 4], red[r_local * 4 + 1]), fmaxf(red[r_local * 4 + 2], red[r_local * 4 + 3]));
  // 1/sqrt(d): 1/64 for 4096; the correctly rounded quotient for 12288.  With
  // RMSNorm the row is also divided by sqrt(mean(x^2) + eps) (the rotation
  // preserves the row norm, so the input row's sum of squares serves).
  const float inv_sqrt_d = MSEG == 4 ? (1.0f / 64.0f) : 1.0f / sqrtf(float(D));
  float post = inv_sqrt_d;
  if constexpr (RMS) {
    const float* rs = red + 16 + (it & 1) * 8 + r_local * 4;
    const float tot = (rs[0] + rs[1]) + (rs[2] + rs[3]);
    post = inv_sqrt_d * (1.0f / sqrtf(tot / float(D) + rms_eps));
  }
  const __half S = quant_scale_fp16(amax * post, clip_ratio);
  const float f = post * (1.0f / __half2float(S));
  if (valid && t == 0) scale_out[row] = S;
  if constexpr (A8) {
    const float2 fv = make_float2(f, f);
    const float2 magic = make_float2(12582912.0f, 12582912.0f);
    const bool need_clamp = clip_ratio < 1.0f || __half2float(S) >= 65504.0f;
    int vsum = 0;
#pragma unroll
    for (int a = 0; a < MSEG; ++a) {
      uint32_t ev = 0, od = 0;  // bytes of codes 0, 2, 4, 6 and 1, 3, 5, 7
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        float2 yv = __fmul2_rn(v[a][jj], fv);
        if (need_clamp) {
          yv.x = fminf(fmaxf(yv.x, -8.0f), 7.0f);
          yv.y = fminf(fmaxf(yv.y, -8.0f), 7.0f);
        }
        const float2 rr = __fadd2_rn(yv, magic);
        // the integer sits in the low mantissa bits of 1.5 * 2^23 + v
        const int vx = __float_as_int(rr.x) - 0x4B400000, vy = __float_as_int(rr.y) - 0x4B400000;
        vsum += vx + vy;
        ev |= uint32_t(vx + 8) << (8 * jj);
        od |= uint32_t(vy + 8) << (8 * jj);
      }
      if (valid) __stcs(reinterpret_cast<uint2*>(q_out + row * D + a * 1024 + 8 * t), make_uint2(ev, od));
    }
    vsum = __reduce_add_sync(0xffffffffu, vsum);
    int* isum = reinterpret_cast<int*>(red) + 40;  // [RPC][4]
    if (lane == 0) isum[r_local * 4 + w] = vsum;
    __syncthreads();
    if (valid && t == 0)
      rowsum_out[row] = (isum[r_local * 4] + isum[r_local * 4 + 1]) + (isum[r_local * 4 + 2] + isum[r_local * 4 + 3]);
  } else {
    // RS: also the row's code sum sum_k v_k into rowsum_out[row].  The
    // rounded values' bit patterns are 0x4B400000 + v; their sum is kept
    // modulo 2^32 and the offsets come off once per thread.
    uint32_t vsum_u = 0;
    if (valid) {
    uint32_t* qrow = reinterpret_cast<uint32_t*>(q_out + row * (D / 2));
    const float2 fv = make_float2(f, f);
    const float2 magic = make_float2(12582912.0f, 12582912.0f);
    // With clip ratio 1 the scale is max|x~| / 7 rounded to fp16, so
    // |x~ / S| <= 7 (1 + 2^-11) + rounding < 7.5 and the clamp cannot bind --
    // unless the scale saturated at the fp16 maximum.
    const bool need_clamp = clip_ratio < 1.0f || __half2float(S) >= 65504.0f;
#pragma unroll
    for (int a = 0; a < MSEG; ++a) {
      uint32_t byte[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        float2 yv = __fmul2_rn(v[a][jj], fv);
        if (need_clamp) {
          yv.x = fminf(fmaxf(yv.x, -8.0f), 7.0f);
          yv.y = fminf(fmaxf(yv.y, -8.0f), 7.0f);
        }
        const float2 rr = __fadd2_rn(yv, magic);
        // low nibble of each: the round-half-even integer in two's complement
        byte[jj] = (uint32_t(__float_as_int(rr.x)) & 0x0Fu) | ((uint32_t(__float_as_int(rr.y)) << 4) & 0xF0u);
        if constexpr (RS) vsum_u += uint32_t(__float_as_int(rr.x)) + uint32_t(__float_as_int(rr.y));
      }
      const uint32_t word = __byte_perm(__byte_perm(byte[0], byte[1], 0x0040), __byte_perm(byte[2], byte[3], 0x0040),
                                        0x5410);
      __stcs(qrow + a * 128 + t, word);
      if (rot_out != nullptr) {
        float4* ro = reinterpret_cast<float4*>(rot_out + row * D + a * 1024 + 8 * t);
        ro[0] = make_float4(v[a][0].x * post, v[a][0].y * post, v[a][1].x * post, v[a][1].y * post);
        ro[1] = make_float4(v[a][2].x * post, v[a][2].y * post, v[a][3].x * post, v[a][3].y * post);
      }
    }
    }  // valid
    if constexpr (RS) {
      // valid rows: 8 MSEG values per thread
      const int vsum = __reduce_add_sync(0xffffffffu, valid ? int(vsum_u - uint32_t(8 * MSEG) * 0x4B400000u) : 0);
      int* isum = reinterpret_cast<int*>(red) + 40;  // [RPC][4]
      if (lane == 0) isum[r_local * 4 + w] = vsum;
      __syncthreads();
      if (valid && t == 0)
        rowsum_out[row] = (isum[r_local * 4] + isum[r_local * 4 + 1]) + (isum[r_local * 4 + 2] + isum[r_local * 4 + 3]);
    }
  }
  }  // row loop
}

// ===================================================================== FP16 arithmetic, d = m x 1024
// The FP16-arithmetic rotation for d = 4096 (Sylvester, bits 10 and 11 across
// segments) and 12288 (Paley-12 across segments) on persistent CTAs that
// stage the next row while the current one is transformed.  Values stay
// fp16 throughout: every butterfly is one fp16x2 add or subtract, i.e. the
// correctly rounded fp16(a + b) and fp16(a - b), so the passes follow the
// Sylvester order h = 1, 2, ..., 512 exactly:
//   pass 1  lane l of warp w takes elements 32 l .. 32 l + 31 of each of the
//           warp's segments: sign flip, y = fp16(x c) with c = fp16(1/sqrt d),
//           bits 0..4 in registers;
//   pass 2  lane l takes the element pairs with bits 1..4 = l & 15 and
//           bit 9 = l >> 4: bits 5..8;
//   pass 3  thread t takes elements 4t .. 4t + 3 and 512 + 4t .. 515 + 4t of
//           every segment: bit 9, then bits 10 and 11 (4096) or the Paley-12
//           partial sums acc = fp16(acc +- y_a), a = 0 .. 11 (12288); then the
//           row abs-max, fp16 scale, round, clamp and pack.
// The fp16 work row holds 32 rows of 16 words (half2) per segment.  Logical
// row r (the pass-1 lane) lives at r ^ (r >> 4), its 16-byte slot m at
// m ^ ((r >> 1) & 3): the 16-byte stores of pass 1, the 32-bit accesses of
// pass 2 and the 8-byte loads of pass 3 are all free of bank conflicts.
__device__ __forceinline__ void hbfly(__half2& a, __half2& b) {
  const __half2 s = __hadd2(a, b);
  b = __hsub2(a, b);
  a = s;
}
__device__ __forceinline__ __half2 hbfly_in(__half2 p) {  // (a, b) -> (a + b, a - b)
  return __hfma2(__high2half2(p), __floats2half2_rn(1.f, -1.f), __low2half2(p));
}
__device__ __forceinline__ int seg16_word(int r, int w) {
  return 16 * (r ^ ((r >> 4) & 1)) + 4 * ((w >> 2) ^ ((r >> 1) & 3)) + (w & 3);
}

template <int MSEG>
struct Seg16Plan {
  static constexpr int D = MSEG * 1024;
  static constexpr int NT = 128;
  static constexpr int SPW = MSEG / 4;
  // [red 256 B][fp16 work row][fp16 staging row][mbarrier]
  static constexpr size_t OFF_BUF = 64 * 4;
  static constexpr size_t OFF_STAGE = OFF_BUF + size_t(D) * 2;
  static constexpr size_t OFF_MBAR = OFF_STAGE + size_t(D) * 2;
  static constexpr size_t SMEM = OFF_MBAR + 16;
  static constexpr int MIN_CTAS = MSEG == 4 ? 8 : 4;
};

template <int MSEG>
__global__ void __launch_bounds__(128, Seg16Plan<MSEG>::MIN_CTAS)
rotate_quant_seg16_kernel(const __half* __restrict__ x, int64_t M, int64_t ld_x, const int8_t* __restrict__ signs,
                          float clip_ratio, __half h16_c, uint8_t* __restrict__ q_out, __half* __restrict__ scale_out,
                          float* __restrict__ rot_out) {
  using PL = Seg16Plan<MSEG>;
  constexpr int D = PL::D;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* red = reinterpret_cast<float*>(smem_raw);
  const int t = threadIdx.x;
  const int lane = t & 31, w = t >> 5;
  uint32_t* buf = reinterpret_cast<uint32_t*>(smem_raw + PL::OFF_BUF);  // half2 words, 512 per segment
  const __half* stage = reinterpret_cast<const __half*>(smem_raw + PL::OFF_STAGE);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem_raw + PL::OFF_MBAR);
  const __half2 c2 = __half2half2(h16_c);
  int64_t row = blockIdx.x;
  if (t == 0) {
    mbar_init(mbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (t == 0 && row < M) {
    mbar_arrive_expect_tx(mbar, uint32_t(D) * 2u);
    bulk_copy_g2s(smem_u32(stage), x + row * ld_x, uint32_t(D) * 2u, mbar);
  }
  for (int it = 0; row < M; ++it, row += gridDim.x) {
    if (!mbar_wait_bounded(mbar, uint32_t(it & 1), nullptr)) break;

    // ---- pass 1: bits 0..4
#pragma unroll
    for (int sgi = 0; sgi < PL::SPW; ++sgi) {
      const int a = w * PL::SPW + sgi;
      __half2 p[16];  // p[n] = elements (2n, 2n + 1) of the lane's 32
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 raw = *reinterpret_cast<const uint4*>(stage + a * 1024 + 32 * lane + 8 * i);
        if (signs != nullptr) {
          const uint2 sg = __ldg(reinterpret_cast<const uint2*>(signs + a * 1024 + 32 * lane + 8 * i));
          raw.x ^= __byte_perm(sg.x, 0u, 0x1404) & 0x80008000u;
          raw.y ^= __byte_perm(sg.x, 0u, 0x3424) & 0x80008000u;
          raw.z ^= __byte_perm(sg.y, 0u, 0x1404) & 0x80008000u;
          raw.w ^= __byte_perm(sg.y, 0u, 0x3424) & 0x80008000u;
        }
        const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) p[4 * i + k] = __hmul2(*reinterpret_cast<const __half2*>(&rw[k]), c2);
      }
#pragma unroll
      for (int n = 0; n < 16; ++n) p[n] = hbfly_in(p[n]);
#pragma unroll
      for (int h = 1; h < 16; h <<= 1)
#pragma unroll
        for (int n = 0; n < 16; ++n)
          if ((n & h) == 0) hbfly(p[n], p[n + h]);
      uint4* seg = reinterpret_cast<uint4*>(buf + a * 512);
      const int prow = lane ^ ((lane >> 4) & 1), sx = (lane >> 1) & 3;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint4 o;
        o.x = *reinterpret_cast<const uint32_t*>(&p[4 * m]);
        o.y = *reinterpret_cast<const uint32_t*>(&p[4 * m + 1]);
        o.z = *reinterpret_cast<const uint32_t*>(&p[4 * m + 2]);
        o.w = *reinterpret_cast<const uint32_t*>(&p[4 * m + 3]);
        seg[4 * prow + (m ^ sx)] = o;
      }
    }
    __syncwarp();

    // ---- pass 2: bits 5..8 of the warp's own segments
    {
      const int b = lane & 15, hb = lane >> 4;
      // word of (row k + 16 hb, column b): 16 k + addr[k & 1][(k >> 1) & 3]
      int addr[2][4];
#pragma unroll
      for (int par = 0; par < 2; ++par)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          addr[par][kk] = 256 * hb + (par ? -16 * hb : 16 * hb) + 4 * ((b >> 2) ^ kk) + (b & 3);
#pragma unroll
      for (int sgi = 0; sgi < PL::SPW; ++sgi) {
        uint32_t* seg = buf + (w * PL::SPW + sgi) * 512;
        __half2 p[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint32_t u = seg[16 * k + addr[k & 1][(k >> 1) & 3]];
          p[k] = *reinterpret_cast<const __half2*>(&u);
        }
#pragma unroll
        for (int h = 1; h < 16; h <<= 1)
#pragma unroll
          for (int k = 0; k < 16; ++k)
            if ((k & h) == 0) hbfly(p[k], p[k + h]);
#pragma unroll
        for (int k = 0; k < 16; ++k) seg[16 * k + addr[k & 1][(k >> 1) & 3]] = *reinterpret_cast<const uint32_t*>(&p[k]);
      }
    }
    __syncthreads();
    {
      // every warp is past pass 1: the staging buffer may take the next row
      const int64_t next = row + gridDim.x;
      if (t == 0 && next < M) {
        mbar_arrive_expect_tx(mbar, uint32_t(D) * 2u);
        bulk_copy_g2s(smem_u32(stage), x + next * ld_x, uint32_t(D) * 2u, mbar);
      }
    }

    // ---- pass 3: bit 9, then across segments
    __half2 v[MSEG][4];  // [a][0..1]: elements 4t .. 4t+3, [a][2..3]: the same + 512
    {
      const int off = 4 * (((t & 7) >> 1) ^ ((t >> 4) & 3)) + 2 * (t & 1);
      const int w0 = 16 * (t >> 3) + off, w1 = 16 * (((t >> 3) + 16) ^ 1) + off;
#pragma unroll
      for (int a = 0; a < MSEG; ++a) {
        const uint2 lo = *reinterpret_cast<const uint2*>(buf + a * 512 + w0);
        const uint2 hi = *reinterpret_cast<const uint2*>(buf + a * 512 + w1);
        v[a][0] = *reinterpret_cast<const __half2*>(&lo.x);
        v[a][1] = *reinterpret_cast<const __half2*>(&lo.y);
        v[a][2] = *reinterpret_cast<const __half2*>(&hi.x);
        v[a][3] = *reinterpret_cast<const __half2*>(&hi.y);
        hbfly(v[a][0], v[a][2]);
        hbfly(v[a][1], v[a][3]);
      }
    }
    if constexpr (MSEG == 4) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        hbfly(v[0][j], v[1][j]);
        hbfly(v[2][j], v[3][j]);
        hbfly(v[0][j], v[2][j]);
        hbfly(v[1][j], v[3][j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __half2 in[12];
#pragma unroll
        for (int a = 0; a < 12; ++a) in[a] = v[a][j];
#pragma unroll
        for (int c = 0; c < 12; ++c) {
          __half2 acc = in[0];  // row 0 of the Paley matrix is all +1
#pragma unroll
          for (int a = 1; a < 12; ++a) acc = paley12_entry(a, c) > 0 ? __hadd2(acc, in[a]) : __hsub2(acc, in[a]);
          v[c][j] = acc;
        }
      }
    }
    __half2 am2 = __float2half2_rn(0.f);
#pragma unroll
    for (int a = 0; a < MSEG; ++a)
#pragma unroll
      for (int j = 0; j < 4; ++j) am2 = __hmax2(am2, __habs2(v[a][j]));
    float amax = fmaxf(__low2float(am2), __high2float(am2));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[w] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const __half S = quant_scale_fp16(amax, clip_ratio);
    const float f = 1.0f / __half2float(S);
    if (t == 0) scale_out[row] = S;
    const float2 fv = make_float2(f, f);
    const float2 magic = make_float2(12582912.0f, 12582912.0f);
    // as in the fp32 kernels: with clip ratio 1 the clamp binds only when the
    // scale saturated at the fp16 maximum
    const bool need_clamp = clip_ratio < 1.0f || __half2float(S) >= 65504.0f;
    uint16_t* qrow = reinterpret_cast<uint16_t*>(q_out + row * (D / 2));
#pragma unroll
    for (int a = 0; a < MSEG; ++a) {
      uint32_t byte[4];
      float2 fl[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        fl[j] = __half22float2(v[a][j]);
        float2 yv = __fmul2_rn(fl[j], fv);
        if (need_clamp) {
          yv.x = fminf(fmaxf(yv.x, -8.0f), 7.0f);
          yv.y = fminf(fmaxf(yv.y, -8.0f), 7.0f);
        }
        const float2 rr = __fadd2_rn(yv, magic);
        byte[j] = (uint32_t(__float_as_int(rr.x)) & 0x0Fu) | ((uint32_t(__float_as_int(rr.y)) << 4) & 0xF0u);
      }
      // codes 4t .. 4t + 3 of segment a are packed bytes 512 a + 2t, 2t + 1
      __stcs(qrow + a * 256 + t, uint16_t(byte[0] | (byte[1] << 8)));
      __stcs(qrow + a * 256 + 128 + t, uint16_t(byte[2] | (byte[3] << 8)));
      if (rot_out != nullptr) {
        float* ro = rot_out + row * D + a * 1024 + 4 * t;
        *reinterpret_cast<float4*>(ro) = make_float4(fl[0].x, fl[0].y, fl[1].x, fl[1].y);
        *reinterpret_cast<float4*>(ro + 512) = make_float4(fl[2].x, fl[2].y, fl[3].x, fl[3].y);
      }
    }
  }
}

template <int MSEG>
static int launch_seg16(const void* x, int64_t M, int64_t ld_x, const int8_t* signs, float clip, uint8_t* q, void* s,
                        float* rot, cudaStream_t st) {
  using PL = Seg16Plan<MSEG>;
  auto kern = rotate_quant_seg16_kernel<MSEG>;
  static quarot::AttrCache attr_done;
  static std::atomic<int> per_sm_dev[64];
  if (!smem_attr_once(kern, int(PL::SMEM), attr_done)) return QUAROT_ERR_LAUNCH;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || ((ld_x * 2) & 15)) return QUAROT_ERR_ALIGNMENT;
  int dev = 0, sms = 1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return QUAROT_ERR_CUDA;
  const bool known = dev >= 0 && dev < 64;
  int per_sm = known ? per_sm_dev[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm < 1) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, PL::NT, PL::SMEM) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    if (known) per_sm_dev[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t cap = int64_t(sms) * per_sm;
  const int64_t blocks = M < cap ? M : cap;
  const __half c = __double2half(1.0 / sqrt(double(PL::D)));
  kern<<<dim3(unsigned(blocks)), dim3(PL::NT), PL::SMEM, st>>>(static_cast<const __half*>(x), M, ld_x, signs, clip, c,
                                                                q, static_cast<__half*>(s), rot);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

template <int MSEG, bool STAGED, bool RMS, bool A8 = false, bool RS = false>
static int launch_seg_t(const void* x, int64_t M, int64_t ld_x, const int8_t* signs, float clip, float eps, uint8_t* q,
                      void* s, float* rot, cudaStream_t st, int32_t* rowsum = nullptr) {
  using PL = SegPlan<MSEG, STAGED>;
  auto kern = rotate_quant_seg_kernel<MSEG, STAGED, RMS, A8, RS>;
  static quarot::AttrCache attr_done;
  static std::atomic<int> per_sm_dev[64];  // resident CTAs per SM on devices 0..63; 0 until measured
  if (!smem_attr_once(kern, int(PL::SMEM), attr_done)) return QUAROT_ERR_LAUNCH;
  int64_t blocks = (M + PL::RPC - 1) / PL::RPC;
  if constexpr (STAGED) {
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return QUAROT_ERR_CUDA;
    const bool known = dev >= 0 && dev < 64;
    int per_sm = known ? per_sm_dev[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm < 1) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, PL::NT, PL::SMEM) != cudaSuccess || per_sm < 1)
        per_sm = 1;
      if (known) per_sm_dev[dev].store(per_sm, std::memory_order_relaxed);
    }
    const int64_t cap = int64_t(sms) * per_sm;
    blocks = blocks < cap ? blocks : cap;
    if ((reinterpret_cast<uintptr_t>(x) & 15) || ((ld_x * 2) & 15)) return QUAROT_ERR_ALIGNMENT;
  }
  if (blocks > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  kern<<<dim3(unsigned(blocks)), dim3(PL::NT), PL::SMEM, st>>>(static_cast<const __half*>(x), M, ld_x, signs, clip,
                                                                eps, q, static_cast<__half*>(s), rot, rowsum);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

template <int LOGP, bool M12, bool RMS, bool H16 = false>
static int launch_rq_t(const void* x, int64_t M, int64_t ld_x, const int8_t* signs, float clip, float eps,
                     uint8_t* q, void* s, float* rot, cudaStream_t st) {
  using PL = RQPlan<LOGP, M12>;
  auto kern = rotate_quant_kernel<LOGP, M12, RMS, H16>;
  // fp16(1/sqrt(d)), rounded once from double (used by the FP16 variant)
  const float h16_c = __half2float(__double2half(1.0 / sqrt(double(PL::D))));
  static quarot::AttrCache attr_done;
  if (!smem_attr_once(kern, int(PL::SMEM), attr_done)) return QUAROT_ERR_LAUNCH;
  const int64_t blocks = (M + PL::RPC - 1) / PL::RPC;
  if (blocks > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  kern<<<dim3(unsigned(blocks)), dim3(PL::NT), PL::SMEM, st>>>(
      static_cast<const __half*>(x), M, ld_x, signs, clip, eps, q, static_cast<__half*>(s), rot, h16_c);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

// RMSNorm on (rms_eps >= 0) or off: separate instantiations, so the plain
// rotation carries no sum-of-squares work.
template <int MSEG, bool STAGED>
static int launch_seg(const void* x, int64_t M, int64_t ld_x, const int8_t* signs, float clip, float eps,
                      uint8_t* q, void* s, float* rot, cudaStream_t st) {
  return eps >= 0.f ? launch_seg_t<MSEG, STAGED, true>(x, M, ld_x, signs, clip, eps, q, s, rot, st)
                    : launch_seg_t<MSEG, STAGED, false>(x, M, ld_x, signs, clip, eps, q, s, rot, st);
}
template <int LOGP, bool M12>
static int launch_rq(const void* x, int64_t M, int64_t ld_x, const int8_t* signs, float clip, float eps,
                     uint8_t* q, void* s, float* rot, cudaStream_t st) {
  return eps >= 0.f ? launch_rq_t<LOGP, M12, true>(x, M, ld_x, signs, clip, eps, q, s, rot, st)
                    : launch_rq_t<LOGP, M12, false>(x, M, ld_x, signs, clip, eps, q, s, rot, st);
}

}  // namespace quarot

using namespace quarot;

// Shared by both entry points: rms_eps < 0 disables the RMSNorm.
static int rotate_quant_dispatch(const void* x, int64_t M, int64_t d, int64_t ld_x, const int8_t* signs,
                                 float clip_ratio, float rms_eps, uint8_t* q_out, void* scale_out, float* rot_out,
                                 void* stream) {
  if (M < 0 || d <= 0 || ld_x < d) return QUAROT_ERR_INVALID_ARG;
  if (!(clip_ratio > 0.f && clip_ratio <= 1.f)) return QUAROT_ERR_INVALID_ARG;
  if (M == 0) return QUAROT_OK;
  if (x == nullptr || q_out == nullptr || scale_out == nullptr) return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (ld_x % 8) || (reinterpret_cast<uintptr_t>(q_out) & 15) ||
      (reinterpret_cast<uintptr_t>(scale_out) & 1) || (signs && (reinterpret_cast<uintptr_t>(signs) & 7)) ||
      (rot_out && (reinterpret_cast<uintptr_t>(rot_out) & 15)))
    return QUAROT_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float e = rms_eps;
  switch (d) {
    case 16: return launch_rq<4, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 32: return launch_rq<5, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 64: return launch_rq<6, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 128: return launch_rq<7, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 256: return launch_rq<8, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 512: return launch_rq<9, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 1024: return launch_rq<10, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 2048: return launch_rq<11, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 4096: return launch_seg<4, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 8192: return launch_rq<13, false>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 3072: return launch_rq<8, true>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 6144: return launch_rq<9, true>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    case 12288: return launch_seg<12, true>(x, M, ld_x, signs, clip_ratio, e, q_out, scale_out, rot_out, st);
    default: return QUAROT_ERR_UNSUPPORTED;
  }
}

extern "C" int quarot_rotate_quant(const void* x, int64_t M, int64_t d, int64_t ld_x,
                                   const int8_t* signs, float clip_ratio, uint8_t* q_out,
                                   void* scale_out, float* rot_out, void* stream) {
  return rotate_quant_dispatch(x, M, d, ld_x, signs, clip_ratio, -1.0f, q_out, scale_out, rot_out, stream);
}

extern "C" int quarot_rotate_quant_fp16(const void* x, int64_t M, int64_t d, int64_t ld_x, const int8_t* signs,
                                        float clip_ratio, uint8_t* q_out, void* scale_out, float* rot_out,
                                        void* stream) {
  if (M < 0 || d <= 0 || ld_x < d) return QUAROT_ERR_INVALID_ARG;
  if (!(clip_ratio > 0.f && clip_ratio <= 1.f)) return QUAROT_ERR_INVALID_ARG;
  if (M == 0) return QUAROT_OK;
  if (x == nullptr || q_out == nullptr || scale_out == nullptr) return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (ld_x % 8) || (reinterpret_cast<uintptr_t>(q_out) & 15) ||
      (reinterpret_cast<uintptr_t>(scale_out) & 1) || (signs && (reinterpret_cast<uintptr_t>(signs) & 7)) ||
      (rot_out && (reinterpret_cast<uintptr_t>(rot_out) & 15)))
    return QUAROT_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float c = clip_ratio;
  switch (d) {
    case 16: return launch_rq_t<4, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 32: return launch_rq_t<5, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 64: return launch_rq_t<6, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 128: return launch_rq_t<7, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 256: return launch_rq_t<8, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 512: return launch_rq_t<9, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 1024: return launch_rq_t<10, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 2048: return launch_rq_t<11, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 4096: return launch_seg16<4>(x, M, ld_x, signs, c, q_out, scale_out, rot_out, st);
    case 8192: return launch_rq_t<13, false, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 3072: return launch_rq_t<8, true, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 6144: return launch_rq_t<9, true, false, true>(x, M, ld_x, signs, c, -1.f, q_out, scale_out, rot_out, st);
    case 12288: return launch_seg16<12>(x, M, ld_x, signs, c, q_out, scale_out, rot_out, st);
    default: return QUAROT_ERR_UNSUPPORTED;
  }
}

extern "C" int quarot_rotate_quant_a8(const void* x, int64_t M, int64_t d, int64_t ld_x, const int8_t* signs,
                                      float clip_ratio, uint8_t* a8_out, void* scale_out, int32_t* rowsum_out,
                                      void* stream) {
  if (M < 0 || d <= 0 || ld_x < d) return QUAROT_ERR_INVALID_ARG;
  if (!(clip_ratio > 0.f && clip_ratio <= 1.f)) return QUAROT_ERR_INVALID_ARG;
  if (d != 4096 && d != 12288) return QUAROT_ERR_UNSUPPORTED;
  if (M == 0) return QUAROT_OK;
  if (x == nullptr || a8_out == nullptr || scale_out == nullptr || rowsum_out == nullptr) return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (ld_x % 8) || (reinterpret_cast<uintptr_t>(a8_out) & 15) ||
      (reinterpret_cast<uintptr_t>(scale_out) & 1) || (reinterpret_cast<uintptr_t>(rowsum_out) & 3) ||
      (signs && (reinterpret_cast<uintptr_t>(signs) & 7)))
    return QUAROT_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 4096)
    return launch_seg_t<4, false, false, true>(x, M, ld_x, signs, clip_ratio, -1.f, a8_out, scale_out, nullptr, st,
                                               rowsum_out);
  return launch_seg_t<12, true, false, true>(x, M, ld_x, signs, clip_ratio, -1.f, a8_out, scale_out, nullptr, st,
                                             rowsum_out);
}

extern "C" int quarot_rotate_quant_rowsum(const void* x, int64_t M, int64_t d, int64_t ld_x, const int8_t* signs,
                                          float clip_ratio, uint8_t* q_out, void* scale_out, int32_t* rowsum_out,
                                          void* stream) {
  if (M < 0 || d <= 0 || ld_x < d) return QUAROT_ERR_INVALID_ARG;
  if (!(clip_ratio > 0.f && clip_ratio <= 1.f)) return QUAROT_ERR_INVALID_ARG;
  if (d != 4096 && d != 12288) return QUAROT_ERR_UNSUPPORTED;
  if (M == 0) return QUAROT_OK;
  if (x == nullptr || q_out == nullptr || scale_out == nullptr || rowsum_out == nullptr) return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (ld_x % 8) || (reinterpret_cast<uintptr_t>(q_out) & 15) ||
      (reinterpret_cast<uintptr_t>(scale_out) & 1) || (reinterpret_cast<uintptr_t>(rowsum_out) & 3) ||
      (signs && (reinterpret_cast<uintptr_t>(signs) & 7)))
    return QUAROT_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 4096)
    return launch_seg_t<4, false, false, false, true>(x, M, ld_x, signs, clip_ratio, -1.f, q_out, scale_out, nullptr,
                                                      st, rowsum_out);
  return launch_seg_t<12, true, false, false, true>(x, M, ld_x, signs, clip_ratio, -1.f, q_out, scale_out, nullptr, st,
                                                    rowsum_out);
}

extern "C" int quarot_rmsnorm_rotate_quant(const void* x, int64_t M, int64_t d, int64_t ld_x, float eps,
                                           const int8_t* signs, float clip_ratio, uint8_t* q_out, void* scale_out,
                                           float* rot_out, void* stream) {
  if (!(eps > 0.f && eps < 1e30f)) return QUAROT_ERR_INVALID_ARG;
  return rotate_quant_dispatch(x, M, d, ld_x, signs, clip_ratio, eps, q_out, scale_out, rot_out, stream);
}
