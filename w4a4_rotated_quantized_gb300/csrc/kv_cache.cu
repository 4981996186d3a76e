// Rotated INT4 KV cache: quarot_kv_write ("Append") and quarot_decode_attn
// ("Decode").
//
// What it computes -- "QuaRot: Outlier-Free 4-Bit Inference in Rotated LLMs"
// (paper summary), section 3: Stage 1c (head-wise Hadamard on the values),
// Stage 1d (head-wise Hadamard on keys and queries after RoPE, so the scores
// are unchanged), Stage 2c (the KV cache procedure during decoding: rotate the
// query, load the quantized cache, dequantize on the fly, dot products,
// append), and the "Append"/"Decode" routines of "Kernel Implementation and
// Hardware Efficiency".  "QuaRot Guide: Outlier-Free 4-Bit W4A4 LLM
// Quantization", "4-Bit Rotated Key-Value (KV) Cache Compression".
//
// Cache layout (chosen here; the pages fix none): codes [B, Hkv, T_max, d/2]
// (two per byte, even dim in the low nibble), fp16 scales [B, Hkv, T_max].
#include <math.h>

#include "common.cuh"

namespace quarot {
namespace kv {

// ------------------------------------------------------------------ append
// D/32 threads own one (token, head) vector, 32 consecutive elements each:
// a 32-point FWHT in registers, then the cross-thread butterflies with warp
// shuffles, row abs-max, fp16 scale, round half-even, pack 32 codes into one
// 16-byte store.  Vectors are enumerated (b, h, t) with t fastest so that the
// code and scale stores of neighbouring vectors are contiguous.
template <int N>
__device__ __forceinline__ void fwht32(float* v) {
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

// ASYM selects the asymmetric quantizer ([S] Stage 2c, per-group asymmetric
// with group = the head vector): a = clip * (min, max), s = fp16(range / 15),
// integer zero point z = rne(a_min / s) (int16), codes q = clamp(rne(x / s) - z,
// 0, 15) stored as unsigned nibbles; x^ = s (q + z).
template <int D, bool ASYM, bool STRIDED>
__global__ void __launch_bounds__(256)
kv_write_kernel(const __half* __restrict__ k_src, const __half* __restrict__ v_src, int64_t B, int64_t T_new,
                int64_t Hkv, int64_t t_start, int64_t T_max, uint8_t* __restrict__ k_q, __half* __restrict__ k_s,
                uint8_t* __restrict__ v_q, __half* __restrict__ v_s, int16_t* __restrict__ k_z,
                int16_t* __restrict__ v_z, float clip_ratio) {
  constexpr int TPV = D / 32;
  // blockIdx.y selects the tensor: 0 = keys, 1 = values
  const __half* __restrict__ src = blockIdx.y == 0 ? k_src : v_src;
  uint8_t* __restrict__ cq = blockIdx.y == 0 ? k_q : v_q;
  __half* __restrict__ cs = blockIdx.y == 0 ? k_s : v_s;
  int16_t* __restrict__ cz = blockIdx.y == 0 ? k_z : v_z;
  // STRIDED: resident CTAs walk the (vector, part) items with a grid stride,
  // and every thread loads its next item's 64 bytes before it transforms the
  // current one, so the loads stay in flight across the whole launch.  The
  // stride is block-uniform and a multiple of the warp size, so the threads
  // of one vector share every iteration (and the warp its shuffles).  Without
  // it (launches of at most one wave, such as a one-token append) each thread
  // takes one item and carries no prefetch state.
  const int64_t nvec = B * Hkv * T_new;
  const int64_t total = nvec * TPV;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int64_t gt = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  auto src_of = [&](int64_t g) {
    const int64_t vv = g / TPV, tt = vv % T_new, bb = vv / T_new;
    return reinterpret_cast<const uint4*>(src + ((bb / Hkv * T_new + tt) * Hkv + bb % Hkv) * D + (g % TPV) * 32);
  };
  uint4 nx[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
  if (gt < total) {
    const uint4* p0 = src_of(gt);
#pragma unroll
    for (int i = 0; i < 4; ++i) nx[i] = __ldcs(p0 + i);
  }
  for (int64_t base = int64_t(blockIdx.x) * blockDim.x; base < total; base += stride, gt += stride) {
  const int64_t vi = gt / TPV;
  const int part = int(gt % TPV);
  const bool valid = gt < total;
  const int64_t t = valid ? vi % T_new : 0;
  const int64_t bh = valid ? vi / T_new : 0;
  const int64_t h = bh % Hkv, b = bh / Hkv;
  const uint4 cur[4] = {nx[0], nx[1], nx[2], nx[3]};
  if constexpr (STRIDED) {
    if (gt + stride < total) {
      const uint4* pn = src_of(gt + stride);
#pragma unroll
      for (int i = 0; i < 4; ++i) nx[i] = __ldcs(pn + i);
    }
  }

  float v[32];
  if (valid) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 r = cur[i];
      const float2 f0 = h2_to_f2(r.x), f1 = h2_to_f2(r.y), f2 = h2_to_f2(r.z), f3 = h2_to_f2(r.w);
      v[8 * i + 0] = f0.x; v[8 * i + 1] = f0.y; v[8 * i + 2] = f1.x; v[8 * i + 3] = f1.y;
      v[8 * i + 4] = f2.x; v[8 * i + 5] = f2.y; v[8 * i + 6] = f3.x; v[8 * i + 7] = f3.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
  }
  fwht32<32>(v);
#pragma unroll
  for (int o = 1; o < TPV; o <<= 1) {
    const bool upper = (part & o) != 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, v[i], o);
      v[i] = upper ? other - v[i] : v[i] + other;
    }
  }
  const float inv_sqrt_d = 1.0f / sqrtf(float(D));
  __half S;
  int zp = 0;
  uint32_t w[4] = {0, 0, 0, 0};
  if constexpr (!ASYM) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] *= inv_sqrt_d;
      amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 1; o < TPV; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    S = quant_scale_fp16(amax, 1.0f);
    const float inv = 1.0f / __half2float(S);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float y = fminf(fmaxf(v[i] * inv, -8.0f), 7.0f);
      w[i >> 3] |= nibble_rne(y) << (4 * (i & 7));
    }
  } else {
    float vmin = INFINITY, vmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] *= inv_sqrt_d;
      vmin = fminf(vmin, v[i]);
      vmax = fmaxf(vmax, v[i]);
    }
#pragma unroll
    for (int o = 1; o < TPV; o <<= 1) {
      vmin = fminf(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
      vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    }
    const float a_min = clip_ratio * vmin, a_max = clip_ratio * vmax;
    S = __float2half_rn(fminf(fmaxf(a_max - a_min, 1e-5f) / 15.0f, 65504.0f));
    const float sf = __half2float(S);
    zp = __float2int_rn(fminf(fmaxf(__fdiv_rn(a_min, sf), -32768.0f), 32767.0f));
    const float inv = 1.0f / sf;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      // |x / s| is below 2^24 (fp16 inputs, s >= fp16(1e-5 / 15)), so the
      // fp32 product and the int conversion are exact enough to round
      const int qi = min(max(__float2int_rn(fminf(fmaxf(v[i] * inv, -1.6e7f), 1.6e7f)) - zp, 0), 15);
      w[i >> 3] |= uint32_t(qi) << (4 * (i & 7));
    }
  }
  if (valid) {
    const int64_t pos = (b * Hkv + h) * T_max + t_start + t;
    __stcs(reinterpret_cast<uint4*>(cq + pos * (D / 2) + part * 16), make_uint4(w[0], w[1], w[2], w[3]));
    if (part == 0) {
      cs[pos] = S;
      if constexpr (ASYM) cz[pos] = int16_t(zp);
    }
  }
  if constexpr (!STRIDED) break;
  }  // item loop
}

// ------------------------------------------------------------------ decode
constexpr int HD = kDecodeHeadDim;     // head_dim of the decode kernel
constexpr int MAXG = kDecodeMaxGroup;  // query heads per KV head
constexpr int CHUNK = 256;    // smallest split; the workspace is sized for T / CHUNK splits
constexpr int DT = 128;       // threads per CTA

__host__ __device__ inline int64_t num_splits(int64_t T) {
  const int64_t s = (T + CHUNK - 1) / CHUNK;
  return s < 1 ? 1 : s;
}

// ------------------------------------------------------------------ tensor-core helpers
// The INT4 codes are exact in fp16.  A byte holding codes (lo, hi) becomes an
// fp16x2 pair with the magic-number trick: 0x6400 | (n ^ 8) is 1024 + (v + 8)
// for the low nibble, 0x6400 | ((n ^ 8) << 4) is 1024 + 16 (v + 8) for the
// high nibble; one fused multiply-add per pair recovers v exactly.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t x, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(x), "r"(m), "r"(c));
  return d;
}
constexpr uint32_t H2_ONE = 0x3C003C00u;       // (1, 1)
constexpr uint32_t H2_M1032 = 0xE408E408u;     // (-1032, -1032)
constexpr uint32_t H2_SIXTEENTH = 0x2C002C00u; // (1/16, 1/16)
constexpr uint32_t H2_M72 = 0xD480D480u;       // (-72, -72)
constexpr uint32_t H2_ONE_SIXTEENTH = 0x2C003C00u;  // (lo 1, hi 1/16)
constexpr uint32_t H2_M1032_M72 = 0xD480E408u;      // (lo -1032, hi -72)

// Byte `p` of `w` -> (code_lo, code_hi) as fp16x2.
__device__ __forceinline__ uint32_t byte_pair(uint32_t w, int p) {
  const uint32_t x = prmt(w, 0u, uint32_t(p) | (4u << 4) | (uint32_t(p) << 8) | (4u << 12));
  const uint32_t h = (x & 0x00F0000Fu) ^ 0x64806408u;
  return hfma2_u32(h, H2_ONE_SIXTEENTH, H2_M1032_M72);
}
// Byte `p` of `wa` and byte `p` of `wb` -> low nibbles (lo_a, lo_b) and high
// nibbles (hi_a, hi_b) as fp16x2.
// ASYM: unsigned codes q (no offset): 1024 + q and 1024 + 16 q, minus 1024 / 64.
template <bool ASYM = false>
__device__ __forceinline__ void byte_cross(uint32_t wa, uint32_t wb, int p, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = prmt(wa, wb, uint32_t(p) | (uint32_t(p + 4) << 8));
  if constexpr (ASYM) {
    lo = hfma2_u32((x & 0x000F000Fu) | 0x64006400u, H2_ONE, 0xE400E400u);        // - 1024
    hi = hfma2_u32((x & 0x00F000F0u) | 0x64006400u, H2_SIXTEENTH, 0xD400D400u);  // /16 - 64
  } else {
    lo = hfma2_u32((x & 0x000F000Fu) ^ 0x64086408u, H2_ONE, H2_M1032);
    hi = hfma2_u32((x & 0x00F000F0u) ^ 0x64806480u, H2_SIXTEENTH, H2_M72);
  }
}

// 2^x by the hardware approximation (relative error ~2^-22; -inf -> +0).
// Arguments are scores minus the running max, so results below 2^-126, which
// it flushes to zero, weigh nothing in the softmax.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  return uint32_t(__half_as_ushort(lo)) | (uint32_t(__half_as_ushort(hi)) << 16);
}

// One CTA per (split, b, g): the partial softmax state of the group's G query
// heads over `chunk` tokens (a multiple of 16), on tensor cores.  Four warps
// take 16-token tiles in turn.  Each warp keeps a ring of NS tiles in shared
// memory, filled by bulk asynchronous copies (keys 1 KB, values 1 KB, their
// scales 32 B each) issued NS tiles ahead.  Per tile:
//   scores  S^T[16 tok x 2G] = Kcodes[16 x 128] . Q~^T, m16n8k16 with the
//           query split into fp16 hi and lo halves (the 2G columns), so the
//           product keeps fp32-level precision; the key scale multiplies the
//           fp32 result.  Head dims are permuted identically on both operands
//           so that fragment pairs come from one masked word.
//   softmax online per head, exp2 (log2 e folded into q~); the running max is
//           raised (and the accumulators rescaled) only when a tile exceeds it
//           by more than 8, so p stays below 2^8.
//   output  O^T[128 x 2G] += Vcodes^T[128 x 16 tok] . P'^T, with P' = p * v_scale
//           in fp16 (even columns; odd columns zero); output dims are permuted
//           so each thread's value bytes are one 8-byte load per token.
constexpr int NS = 3;                 // tiles in flight per warp
constexpr int TILE_BYTES = 2 * 16 * (HD / 2) + 2 * 32;  // K, V codes + scales = 2112
constexpr int TILE_STRIDE = 2176;     // rounded to 128 bytes
constexpr int QS = HD + 16;           // padded q~ row: dim d at d + 4 (d >> 5)
constexpr int WO = HD + 4;            // padded merge row

template <int G>
constexpr size_t decode_smem_bytes() {
  static_assert(2 * G * HD * 2 + 2 * G * 4 <= G * QS * 4, "query halves and per-head constants fit the q region");
  return size_t(G) * QS * 4 + size_t(DT / 32) * NS * TILE_STRIDE + size_t(DT / 32) * NS * 8 + 64;
}

// ASYM: the asymmetric cache (unsigned codes q, fp16 scale s, int16 zero point
// z per token; k^ = s (q + z)).  The keys' magic form is 1024 + q (1024 + 16 q
// for odd dims), so the per-head offset is 1024 * sum(weights); the zero point
// adds z_t * sum_d q~_d to each score; the values' zero points add
// sum_t p'_t z_t to every output dim of the head.  Tiles also carry the 16 K
// and 16 V zero points (bytes 2112 .. 2175).
template <int G, bool ASYM>
__global__ void __launch_bounds__(DT, 4)
decode_mma_kernel(const __half* __restrict__ q, const uint8_t* __restrict__ kq, const __half* __restrict__ ks,
                  const uint8_t* __restrict__ vq, const __half* __restrict__ vs, int Hq, int Hkv, int T,
                  int T_max, float qscale, float* __restrict__ ws_o, float* __restrict__ ws_ml, int splits,
                  int chunk, int bulk_ok, const int16_t* __restrict__ kz, const int16_t* __restrict__ vz) {
  constexpr int NT = (2 * G + 7) / 8;  // n8 tiles of (head, hi/lo) columns
  constexpr int NW = DT / 32;
  extern __shared__ __align__(128) unsigned char dsm[];
  unsigned char* ring = dsm;                                        // [NW][NS][TILE_STRIDE]
  float* qs = reinterpret_cast<float*>(dsm + NW * NS * TILE_STRIDE);  // [G][QS]
  uint64_t* tbar = reinterpret_cast<uint64_t*>(dsm + NW * NS * TILE_STRIDE + G * QS * 4);  // [NW][NS]
  __shared__ float wm[NW][G], wl[NW][G], wz[NW][G];
  float* wo = reinterpret_cast<float*>(ring);  // merge rows, reuse the ring after the last tile

  const int split = blockIdx.x;
  const int bg = blockIdx.y;
  const int b = bg / Hkv, g = bg % Hkv;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int r = lane >> 2, c = lane & 3;
  const int t0 = split * chunk;
  const int tn = min(chunk, T - t0);
  const int64_t cache_row = (int64_t(b) * Hkv + g) * T_max + t0;
  const uint8_t* kbase = kq + cache_row * (HD / 2);
  const uint8_t* vbase = vq + cache_row * (HD / 2);
  const __half* ksb = ks + cache_row;
  const __half* vsb = vs + cache_row;
  const int16_t* kzb = ASYM ? kz + cache_row : nullptr;
  const int16_t* vzb = ASYM ? vz + cache_row : nullptr;
  unsigned char* wring = ring + wid * NS * TILE_STRIDE;
  uint64_t* wbar = tbar + wid * NS;

  if (lane == 0) {
    for (int st = 0; st < NS; ++st) mbar_init(&wbar[st], 1);
    fence_barrier_init();
  }
  __syncwarp();
  // tile i of this warp starts at token wid * 16 + i * NW * 16
  auto issue = [&](int i) {
    const int tt = wid * 16 + i * NW * 16;
    if (tt >= tn) return;
    unsigned char* dst = wring + (i % NS) * TILE_STRIDE;
    if (bulk_ok && tt + 16 <= tn) {
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&wbar[i % NS], TILE_BYTES + (ASYM ? 64 : 0));
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 1024, [%2];" ::"r"(
                         smem_u32(dst)), "l"(kbase + int64_t(tt) * (HD / 2)), "r"(smem_u32(&wbar[i % NS])) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 1024, [%2];" ::"r"(
                         smem_u32(dst + 1024)), "l"(vbase + int64_t(tt) * (HD / 2)), "r"(smem_u32(&wbar[i % NS])) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 32, [%2];" ::"r"(
                         smem_u32(dst + 2048)), "l"(ksb + tt), "r"(smem_u32(&wbar[i % NS])) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 32, [%2];" ::"r"(
                         smem_u32(dst + 2080)), "l"(vsb + tt), "r"(smem_u32(&wbar[i % NS])) : "memory");
        if constexpr (ASYM) {
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 32, [%2];" ::"r"(
                           smem_u32(dst + 2112)), "l"(kzb + tt), "r"(smem_u32(&wbar[i % NS])) : "memory");
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 32, [%2];" ::"r"(
                           smem_u32(dst + 2144)), "l"(vzb + tt), "r"(smem_u32(&wbar[i % NS])) : "memory");
        }
      }
    } else {
      // ragged last tile (or unaligned cache): plain loads, zero beyond tn
      for (int k = lane; k < 128; k += 32) {  // 64 x 16 B of codes
        const int tok = (k & 63) >> 2, part = k & 3;
        const uint8_t* srcb = (k < 64 ? kbase : vbase) + int64_t(tt + tok) * (HD / 2);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (tt + tok < tn) val = __ldcs(reinterpret_cast<const uint4*>(srcb) + part);
        *reinterpret_cast<uint4*>(dst + (k < 64 ? 0 : 1024) + tok * 64 + part * 16) = val;
      }
      if (lane < 16) {
        const bool in = tt + lane < tn;
        reinterpret_cast<__half*>(dst + 2048)[lane] = in ? ksb[tt + lane] : __float2half(0.f);
        reinterpret_cast<__half*>(dst + 2080)[lane] = in ? vsb[tt + lane] : __float2half(0.f);
        if constexpr (ASYM) {
          reinterpret_cast<int16_t*>(dst + 2112)[lane] = in ? kzb[tt + lane] : int16_t(0);
          reinterpret_cast<int16_t*>(dst + 2144)[lane] = in ? vzb[tt + lane] : int16_t(0);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&wbar[i % NS]);
    }
  };
#pragma unroll 1
  for (int i = 0; i < NS; ++i) issue(i);

  // This CTA's inputs are read only after the loop; the combine kernel may be
  // scheduled now (it waits in griddepcontrol.wait for this grid to finish).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- q~ = q H / sqrt(d): one warp per query head; lane l holds dims
  // 4l .. 4l+3.  Butterflies of spans 1 and 2 run in registers, spans 4 .. 64
  // across lanes, in the stage order of a natural-order FWHT (lower index
  // a + b, upper a - b).  Each scaled value x (odd dims divided by 16) splits
  // into fp16 hi + lo halves; the head's score offset
  // sum_d (hi + lo)(d) * (1032 for even d, 1152 for odd d) is a warp sum (a
  // per-head constant, so its rounding does not change the softmax).
  __half* qh = reinterpret_cast<__half*>(qs);                   // [G][2][HD]: hi row, lo row
  float* qoff_s = reinterpret_cast<float*>(qh + 2 * G * HD);    // [G]
  float* qsum_s = qoff_s + G;                                   // [G] (ASYM): sum_d q~_d qscale
  for (int hh = wid; hh < G; hh += NW) {
    const uint2 raw = *reinterpret_cast<const uint2*>(q + (int64_t(b) * Hq + g * G + hh) * HD + 4 * lane);
    const float2 x01 = h2_to_f2(raw.x), x23 = h2_to_f2(raw.y);
    float x[4] = {x01.x, x01.y, x23.x, x23.y};
    float u0 = x[0], u1 = x[1];
    x[0] = u0 + u1;
    x[1] = u0 - u1;
    u0 = x[2];
    u1 = x[3];
    x[2] = u0 + u1;
    x[3] = u0 - u1;
    u0 = x[0];
    u1 = x[2];
    x[0] = u0 + u1;
    x[2] = u0 - u1;
    u0 = x[1];
    u1 = x[3];
    x[1] = u0 + u1;
    x[3] = u0 - u1;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const bool upper = (lane & s) != 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float other = __shfl_xor_sync(0xffffffffu, x[k], s);
        x[k] = upper ? other - x[k] : x[k] + other;
      }
    }
    float part = 0.f, qsum = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int dd = 4 * lane + k;
      const float xs = x[k] * qscale * ((dd & 1) ? 0.0625f : 1.0f);
      const __half hi = __float2half_rn(xs);
      const __half lo = __float2half_rn(xs - __half2float(hi));
      const float wsum = __half2float(hi) + __half2float(lo);
      part += wsum * (ASYM ? 1024.0f : ((dd & 1) ? 1152.0f : 1032.0f));
      qsum += wsum * ((dd & 1) ? 16.0f : 1.0f);
      qh[(2 * hh) * HD + dd] = hi;
      qh[(2 * hh + 1) * HD + dd] = lo;
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      part += __shfl_xor_sync(0xffffffffu, part, o2);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, o2);
    }
    if (lane == 0) {
      qoff_s[hh] = part;
      qsum_s[hh] = qsum;
    }
  }
  __syncthreads();

  // ---- B fragments of Q~^T.  Column n = lane/4 of n-tile nt is head
  // 4 nt + n/2 (hi half for even n, lo half for odd n).  Step j pairs head dims
  // d0 = 32c + 8 (j >> 1) + 2 (j & 1): b0 = (d0, d0 + 4), b1 = (d0 + 1, d0 + 5),
  // matching the key fragments built by masking one word of packed codes.
  // The key fragments keep the fp16 magic offsets: a low-nibble code u + 8
  // arrives as 1024 + (v + 8) and a high-nibble code as 1024 + 16 (v + 8), so
  // the query weights of high-nibble dims (odd d) are divided by 16 and every
  // score carries the per-head constant sum_even 1032 q~ + sum_odd 72 q~,
  // subtracted after the product.
  uint32_t qb[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 4 + (r >> 1);
    const int part = r & 1;  // 0: hi, 1: lo
#pragma unroll
    for (int m4 = 0; m4 < 4; ++m4) {
      __half hv[8];
#pragma unroll
      for (int e2 = 0; e2 < 8; ++e2)
        hv[e2] = hh < G ? qh[(2 * hh + part) * HD + 32 * c + 8 * m4 + e2] : __float2half(0.f);
      qb[nt][2 * m4][0] = pack_h2(hv[0], hv[4]);
      qb[nt][2 * m4][1] = pack_h2(hv[1], hv[5]);
      qb[nt][2 * m4 + 1][0] = pack_h2(hv[2], hv[6]);
      qb[nt][2 * m4 + 1][1] = pack_h2(hv[3], hv[7]);
    }
  }
  // per-head offset constant of the scores (the head whose scores this
  // thread holds)
  float qoff[NT], qsum[NT], zacc[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 4 + c;
    qoff[nt] = hh < G ? qoff_s[hh] : 0.f;
    qsum[nt] = hh < G ? qsum_s[hh] : 0.f;
    zacc[nt] = 0.f;  // ASYM: sum_t p'_t z_t of the head over this thread's tokens
  }

  float o[NT][8][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][i][e] = 0.f;
  float m_run[NT], l_run[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.f;
  }

  int i = 0;
  for (int tt = wid * 16; tt < tn; tt += NW * 16, ++i) {
    const unsigned char* src = wring + (i % NS) * TILE_STRIDE;
    if (!mbar_wait_bounded(&wbar[i % NS], uint32_t((i / NS) & 1), nullptr)) break;
    // ---- fragments: keys of tokens r, r+8 (bytes 16c..16c+15), values of
    // tokens 2c, 2c+1, 2c+8, 2c+9 (bytes 8r..8r+7), scales
    const uint4 k0 = *reinterpret_cast<const uint4*>(src + r * 64 + 16 * c);
    const uint4 k1 = *reinterpret_cast<const uint4*>(src + (r + 8) * 64 + 16 * c);
    uint2 vw[4];
    float vsc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tok = 2 * c + (u & 1) + 8 * (u >> 1);
      vw[u] = *reinterpret_cast<const uint2*>(src + 1024 + tok * 64 + 8 * r);
      vsc[u] = __half2float(reinterpret_cast<const __half*>(src + 2080)[tok]);
    }
    const float ks0 = __half2float(reinterpret_cast<const __half*>(src + 2048)[r]);
    const float ks1 = __half2float(reinterpret_cast<const __half*>(src + 2048)[r + 8]);
    // ASYM: zero points of this thread's score tokens r, r + 8 (keys and values)
    float kz0 = 0.f, kz1 = 0.f, vzp0 = 0.f, vzp1 = 0.f;
    if constexpr (ASYM) {
      kz0 = float(reinterpret_cast<const int16_t*>(src + 2112)[r]);
      kz1 = float(reinterpret_cast<const int16_t*>(src + 2112)[r + 8]);
      vzp0 = float(reinterpret_cast<const int16_t*>(src + 2144)[r]) *
             __half2float(reinterpret_cast<const __half*>(src + 2080)[r]);
      vzp1 = float(reinterpret_cast<const int16_t*>(src + 2144)[r + 8]) *
             __half2float(reinterpret_cast<const __half*>(src + 2080)[r + 8]);
    }
    __syncwarp();
    issue(i + NS);  // refill this stage NS tiles ahead

    const int tr0 = tt + r, tr1 = tt + r + 8;
    // ---- scores
    const uint32_t kw0[4] = {k0.x, k0.y, k0.z, k0.w};
    const uint32_t kw1[4] = {k1.x, k1.y, k1.z, k1.w};
    float sacc[NT][2][4];  // two accumulation chains (even / odd steps)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][0][e] = sacc[nt][1][e] = 0.f;
#pragma unroll
    for (int m4 = 0; m4 < 4; ++m4) {
      const uint32_t w0 = kw0[m4], w1 = kw1[m4], w0s = w0 >> 8, w1s = w1 >> 8;
      // magic fp16: 0x6400 | nibble bits (XOR 8 on the nibble for signed codes)
      constexpr uint32_t ML = ASYM ? 0x64006400u : 0x64086408u, MH = ASYM ? 0x64006400u : 0x64806480u;
      const uint32_t p0a = (w0 & 0x000F000Fu) ^ ML, p1a = (w0 & 0x00F000F0u) ^ MH;
      const uint32_t p2a = (w0s & 0x000F000Fu) ^ ML, p3a = (w0s & 0x00F000F0u) ^ MH;
      const uint32_t p0b = (w1 & 0x000F000Fu) ^ ML, p1b = (w1 & 0x00F000F0u) ^ MH;
      const uint32_t p2b = (w1s & 0x000F000Fu) ^ ML, p3b = (w1s & 0x00F000F0u) ^ MH;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma16816(sacc[nt][0], p0a, p0b, p1a, p1b, qb[nt][2 * m4][0], qb[nt][2 * m4][1]);
        mma16816(sacc[nt][1], p2a, p2b, p3a, p3b, qb[nt][2 * m4 + 1][0], qb[nt][2 * m4 + 1][1]);
      }
    }

#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // thread holds head 4 nt + c for tokens tr0 (sacc 0 + 1) and tr1 (sacc 2 + 3)
      float i0 = ((sacc[nt][0][0] + sacc[nt][1][0]) + (sacc[nt][0][1] + sacc[nt][1][1])) - qoff[nt];
      float i1 = ((sacc[nt][0][2] + sacc[nt][1][2]) + (sacc[nt][0][3] + sacc[nt][1][3])) - qoff[nt];
      if constexpr (ASYM) {
        i0 += kz0 * qsum[nt];
        i1 += kz1 * qsum[nt];
      }
      const float s0 = tr0 < tn ? i0 * ks0 : -INFINITY;
      const float s1 = tr1 < tn ? i1 * ks1 : -INFINITY;
      // raise the running max only when it grows by more than 8 (p <= 2^8).
      // The head's tile max exceeds m_run + 8 exactly when one of its lanes'
      // own maxima does, so the lanes test their two scores first and the
      // head-wide max (over the lanes of column c) is formed only in the
      // rare rescale branch, off the common dependency chain.
      float mt = fmaxf(s0, s1);
      if (__any_sync(0xffffffffu, mt > m_run[nt] + 8.0f)) {
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        const float m_new = mt > m_run[nt] + 8.0f ? mt : m_run[nt];
        const float alpha = exp2f(m_run[nt] - m_new);  // 0 when the old max is -inf
        m_run[nt] = m_new;
        l_run[nt] *= alpha;
        zacc[nt] *= alpha;
#pragma unroll
        for (int ii = 0; ii < 8; ++ii)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nt][ii][e] *= alpha;
      }
      // m_run is finite here: a warp's first tile holds at least one valid
      // token (tt < tn), whose finite score raised it from -inf just above
      const float P0 = ex2_approx(s0 - m_run[nt]), P1 = ex2_approx(s1 - m_run[nt]);
      if constexpr (ASYM) zacc[nt] = fmaf(P0, vzp0, fmaf(P1, vzp1, zacc[nt]));
      l_run[nt] += P0 + P1;

      // B fragment of P'^T: column n = r is head 4 nt + r/2 (hi for even r, lo
      // for odd r); rows are tokens 2c, 2c+1 (b0) and 2c+8, 2c+9 (b1).
      const int src0 = 8 * c + (r >> 1), src1 = 8 * c + 4 + (r >> 1);
      const float pv[4] = {__shfl_sync(0xffffffffu, P0, src0) * vsc[0], __shfl_sync(0xffffffffu, P0, src1) * vsc[1],
                           __shfl_sync(0xffffffffu, P1, src0) * vsc[2], __shfl_sync(0xffffffffu, P1, src1) * vsc[3]};
      // fp16 p' (relative rounding 2^-11, uncorrelated across tokens); the odd
      // columns stay zero
      const uint32_t pb0 = (r & 1) ? 0u : pack_h2(__float2half_rn(pv[0]), __float2half_rn(pv[1]));
      const uint32_t pb1 = (r & 1) ? 0u : pack_h2(__float2half_rn(pv[2]), __float2half_rn(pv[3]));
      // ---- O^T += V^T P'^T over 8 m-tiles of 16 dims: m-tile ii, row r is dim
      // 16r + 2ii, row r + 8 is dim 16r + 2ii + 1 (byte ii of the 8-byte chunk)
      const uint32_t va[2] = {vw[0].x, vw[0].y}, vb[2] = {vw[1].x, vw[1].y};
      const uint32_t vc[2] = {vw[2].x, vw[2].y}, vd[2] = {vw[3].x, vw[3].y};
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        uint32_t a0, a1, a2, a3;
        byte_cross<ASYM>(va[ii >> 2], vb[ii >> 2], ii & 3, a0, a1);
        byte_cross<ASYM>(vc[ii >> 2], vd[ii >> 2], ii & 3, a2, a3);
        mma16816(o[nt][ii], a0, a1, a2, a3, pb0, pb1);
      }
    }
  }

  // ---- merge the warps of the CTA (the ring is free: reuse it), then write
  // the split's partial state
  __syncthreads();
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 4 + c;
    float l = l_run[nt], zs = zacc[nt];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    zs += __shfl_xor_sync(0xffffffffu, zs, 4);
    zs += __shfl_xor_sync(0xffffffffu, zs, 8);
    zs += __shfl_xor_sync(0xffffffffu, zs, 16);
    if (hh < G) {
      if (r == 0) {
        wm[wid][hh] = m_run[nt];
        wz[wid][hh] = zs;  // ASYM: the values' zero-point term, common to all dims
        wl[wid][hh] = l;
      }
      float* wrow = wo + (wid * G + hh) * WO + 16 * r;
#pragma unroll
      for (int ii = 0; ii < 8; ++ii)
        *reinterpret_cast<float2*>(wrow + 2 * ii) = make_float2(o[nt][ii][0] + o[nt][ii][1], o[nt][ii][2] + o[nt][ii][3]);
    }
  }
  __syncthreads();
  const int e = tid;  // output dim
  const int64_t base = (int64_t(b) * Hq + g * G) * splits + split;
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) m = fmaxf(m, wm[w][hh]);
    const float m_use = m == -INFINITY ? 0.f : m;
    float l = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = exp2f(wm[w][hh] - m_use);
      l += f * wl[w][hh];
      acc += f * (wo[(w * G + hh) * WO + e] + wz[w][hh]);
    }
    const int64_t slot = base + int64_t(hh) * splits;
    ws_o[slot * HD + e] = acc;
    if (tid == 0) {
      ws_ml[slot * 2 + 0] = m;
      ws_ml[slot * 2 + 1] = l;
    }
  }
}

// Merge the splits of one (b, h): o = sum_s 2^(m_s - m) o_s / sum_s 2^(m_s - m) l_s,
// then optionally rotate back by H / sqrt(d); fp16 out.
__global__ void __launch_bounds__(HD)
decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml, int splits,
                      int unrotate, __half* __restrict__ out) {
  // launched as a programmatic dependent of the decode kernel: wait for it to
  // complete (and its writes to be visible) before reading the workspace
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float ov[HD];
  const int bh = blockIdx.x, e = threadIdx.x;
  const int64_t base = int64_t(bh) * splits;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s) m = fmaxf(m, ws_ml[(base + s) * 2]);
  float l = 0.f, acc = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ms = ws_ml[(base + s) * 2];
    const float f = ms == -INFINITY ? 0.f : exp2f(ms - m);
    l += f * ws_ml[(base + s) * 2 + 1];
    acc += f * ws_o[(base + s) * HD + e];
  }
  float r = acc / l;
  if (unrotate) {
    ov[e] = r;
    __syncthreads();
    for (int hspan = 1; hspan < HD; hspan <<= 1) {
      const int partner = e ^ hspan;
      const float mine = ov[e], other = ov[partner];
      __syncthreads();
      ov[e] = (e & hspan) ? other - mine : mine + other;
      __syncthreads();
    }
    r = ov[e] * (1.0f / sqrtf(float(HD)));
  }
  out[int64_t(bh) * HD + e] = __float2half_rn(r);
}

// Resident CTAs per SM of the decode kernel for group size G (queried once).
template <bool ASYM>
int decode_ctas_per_sm(int G) {
  static int cache[4] = {0, 0, 0, 0};
  const int slot = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  if (cache[slot] == 0) {
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (G) {
      case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<1, ASYM>, DT, decode_smem_bytes<1>()); break;
      case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<2, ASYM>, DT, decode_smem_bytes<2>()); break;
      case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<4, ASYM>, DT, decode_smem_bytes<4>()); break;
      default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<8, ASYM>, DT, decode_smem_bytes<8>()); break;
    }
    cache[slot] = (e == cudaSuccess && n > 0) ? n : 1;
  }
  return cache[slot];
}

// Resident CTAs per SM of the strided KV-write instantiation (256 threads),
// measured once.
template <int D, bool ASYM>
int kv_write_ctas_per_sm() {
  static std::atomic<int> cache{0};
  int n = cache.load(std::memory_order_relaxed);
  if (n < 1) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kv_write_kernel<D, ASYM, true>, 256, 0) != cudaSuccess || n < 1)
      n = 1;
    cache.store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace kv
}  // namespace quarot

using namespace quarot;

static int kv_write_impl(bool asym, const void* k, const void* v, int64_t B, int64_t T_new, int64_t Hkv, int64_t d,
                         int64_t t_start, int64_t T_max, float clip_ratio, uint8_t* k_q, void* k_s, int16_t* k_z,
                         uint8_t* v_q, void* v_s, int16_t* v_z, void* stream) {
  if (B < 0 || T_new < 0 || Hkv <= 0 || t_start < 0 || T_max <= 0) return QUAROT_ERR_INVALID_ARG;
  if (t_start + T_new > T_max) return QUAROT_ERR_INVALID_ARG;
  if (asym && !(clip_ratio > 0.f && clip_ratio <= 1.f)) return QUAROT_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return QUAROT_ERR_UNSUPPORTED;
  if (B == 0 || T_new == 0) return QUAROT_OK;
  if (!k || !v || !k_q || !k_s || !v_q || !v_s || (asym && (!k_z || !v_z))) return QUAROT_ERR_INVALID_ARG;
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(k, 16) || mis(v, 16) || mis(k_q, 16) || mis(v_q, 16) || mis(k_s, 2) || mis(v_s, 2) ||
      (asym && (mis(k_z, 2) || mis(v_z, 2))))
    return QUAROT_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t threads = B * Hkv * T_new * (d / 32);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return QUAROT_ERR_CUDA;
  const int64_t need = (threads + 255) / 256;
  auto go = [&](auto kern_one, auto kern_strided, int per_sm) {
    // more items than one wave of resident CTAs (keys and values share it):
    // that wave walks them with the grid stride; else one item per thread
    int64_t cap = int64_t(sms) * per_sm / 2;
    if (cap < 1) cap = 1;
    const bool strided = need > cap;
    const int64_t blocks = strided ? cap : need;
    auto kern = strided ? kern_strided : kern_one;
    kern<<<dim3(unsigned(blocks), 2), 256, 0, st>>>(static_cast<const __half*>(k), static_cast<const __half*>(v),
                                                    B, T_new, Hkv, t_start, T_max, k_q, static_cast<__half*>(k_s),
                                                    v_q, static_cast<__half*>(v_s), k_z, v_z, clip_ratio);
  };
  if (asym) {
    if (d == 64) go(kv::kv_write_kernel<64, true, false>, kv::kv_write_kernel<64, true, true>, kv::kv_write_ctas_per_sm<64, true>());
    else if (d == 128) go(kv::kv_write_kernel<128, true, false>, kv::kv_write_kernel<128, true, true>, kv::kv_write_ctas_per_sm<128, true>());
    else go(kv::kv_write_kernel<256, true, false>, kv::kv_write_kernel<256, true, true>, kv::kv_write_ctas_per_sm<256, true>());
  } else {
    if (d == 64) go(kv::kv_write_kernel<64, false, false>, kv::kv_write_kernel<64, false, true>, kv::kv_write_ctas_per_sm<64, false>());
    else if (d == 128) go(kv::kv_write_kernel<128, false, false>, kv::kv_write_kernel<128, false, true>, kv::kv_write_ctas_per_sm<128, false>());
    else go(kv::kv_write_kernel<256, false, false>, kv::kv_write_kernel<256, false, true>, kv::kv_write_ctas_per_sm<256, false>());
  }
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

extern "C" int quarot_kv_write(const void* k, const void* v, int64_t B, int64_t T_new, int64_t Hkv,
                               int64_t d, int64_t t_start, int64_t T_max, uint8_t* k_q, void* k_s,
                               uint8_t* v_q, void* v_s, void* stream) {
  return kv_write_impl(false, k, v, B, T_new, Hkv, d, t_start, T_max, 1.0f, k_q, k_s, nullptr, v_q, v_s, nullptr,
                       stream);
}

extern "C" int quarot_kv_write_asym(const void* k, const void* v, int64_t B, int64_t T_new, int64_t Hkv, int64_t d,
                                    int64_t t_start, int64_t T_max, float clip_ratio, uint8_t* k_q, void* k_s,
                                    int16_t* k_z, uint8_t* v_q, void* v_s, int16_t* v_z, void* stream) {
  return kv_write_impl(true, k, v, B, T_new, Hkv, d, t_start, T_max, clip_ratio, k_q, k_s, k_z, v_q, v_s, v_z,
                       stream);
}

extern "C" size_t quarot_decode_workspace_bytes(int64_t B, int64_t Hq, int64_t d, int64_t T) {
  if (B <= 0 || Hq <= 0 || d != kv::HD || T < 0) return 0;
  const int64_t s = kv::num_splits(T);
  const size_t bytes = size_t(B * Hq * s) * (kv::HD + 2) * sizeof(float);
  return (bytes + 255) & ~size_t(255);
}

template <bool ASYM>
static int decode_impl(const void* q, const uint8_t* k_q, const void* k_s, const int16_t* k_z, const uint8_t* v_q,
                       const void* v_s, const int16_t* v_z, int64_t B, int64_t Hq, int64_t Hkv, int64_t d, int64_t T,
                       int64_t T_max, float sm_scale, int unrotate_out, void* out, void* workspace, size_t ws_bytes,
                       void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || T < 0 || T_max < 0 || T > T_max) return QUAROT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return QUAROT_ERR_INVALID_ARG;
  if (d != kv::HD || Hq / Hkv > kv::MAXG) return QUAROT_ERR_UNSUPPORTED;
  if (B == 0) return QUAROT_OK;
  if (!q || !out) return QUAROT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    return cudaMemsetAsync(out, 0, size_t(B * Hq * d) * 2, st) == cudaSuccess ? QUAROT_OK : QUAROT_ERR_CUDA;
  }
  if (!k_q || !k_s || !v_q || !v_s || !workspace || (ASYM && (!k_z || !v_z))) return QUAROT_ERR_INVALID_ARG;
  if (ws_bytes < quarot_decode_workspace_bytes(B, Hq, d, T)) return QUAROT_ERR_INVALID_ARG;
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k_q, 16) || mis(v_q, 16) || mis(k_s, 2) || mis(v_s, 2) || mis(out, 16) ||
      mis(workspace, 256) || (ASYM && (mis(k_z, 2) || mis(v_z, 2))))
    return QUAROT_ERR_ALIGNMENT;
  if (B * Hkv > 65535 || T > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  // Splits: as many as fit one wave of resident CTAs (no tail wave), at least
  // one, never more than the workspace bound of one split per kv::CHUNK
  // tokens; chunks are multiples of 16 tokens.
  const int G = int(Hq / Hkv);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_sm = kv::decode_ctas_per_sm<ASYM>(G);
  const int64_t max_splits = kv::num_splits(T);
  int64_t want = (int64_t(per_sm) * sms) / (B * Hkv);
  want = want < 1 ? 1 : (want > max_splits ? max_splits : want);
  int64_t chunk = (T + want - 1) / want;
  chunk = (chunk + 15) / 16 * 16;
  const int splits = int((T + chunk - 1) / chunk);
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(float(d));
  const float qscale = scale * 1.4426950408889634f / sqrtf(float(d));  // 1/sqrt(d) of H, log2(e)
  float* ws_o = static_cast<float*>(workspace);
  float* ws_ml = ws_o + size_t(B * Hq * splits) * kv::HD;
  dim3 grid(unsigned(splits), unsigned(B * Hkv));
  // bulk copies need 16-byte aligned sources: every (b, g) row of the scale
  // arrays starts at a multiple of 8 tokens
  const int bulk_ok = (T_max % 8) == 0 && !mis(k_s, 16) && !mis(v_s, 16) &&
                      (!ASYM || (!mis(k_z, 16) && !mis(v_z, 16)));
  int lrc = QUAROT_OK;
  auto args = [&](auto kern, size_t smem) {
    static quarot::AttrCache attr[4];  // per group size: the kernels differ
    const int slot = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
    if (!smem_attr_once(kern, int(smem), attr[slot])) {
      lrc = QUAROT_ERR_LAUNCH;
      return;
    }
    kern<<<grid, kv::DT, smem, st>>>(static_cast<const __half*>(q), k_q, static_cast<const __half*>(k_s), v_q,
                                     static_cast<const __half*>(v_s), int(Hq), int(Hkv), int(T), int(T_max),
                                     qscale, ws_o, ws_ml, splits, int(chunk), bulk_ok, k_z, v_z);
  };
  switch (G) {
    case 1: args(kv::decode_mma_kernel<1, ASYM>, kv::decode_smem_bytes<1>()); break;
    case 2: args(kv::decode_mma_kernel<2, ASYM>, kv::decode_smem_bytes<2>()); break;
    case 4: args(kv::decode_mma_kernel<4, ASYM>, kv::decode_smem_bytes<4>()); break;
    case 8: args(kv::decode_mma_kernel<8, ASYM>, kv::decode_smem_bytes<8>()); break;
    default: return QUAROT_ERR_UNSUPPORTED;
  }
  if (lrc != QUAROT_OK) return lrc;
  // the combine kernel is a programmatic dependent launch: it is scheduled
  // while the decode kernel runs and waits for it in griddepcontrol.wait, so
  // its launch latency overlaps the decode
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(B * Hq));
  cfg.blockDim = dim3(kv::HD);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kv::decode_combine_kernel, static_cast<const float*>(ws_o),
                         static_cast<const float*>(ws_ml), splits, unrotate_out, static_cast<__half*>(out)) !=
      cudaSuccess)
    return QUAROT_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

extern "C" int quarot_decode_attn(const void* q, const uint8_t* k_q, const void* k_s, const uint8_t* v_q,
                                  const void* v_s, int64_t B, int64_t Hq, int64_t Hkv, int64_t d, int64_t T,
                                  int64_t T_max, float sm_scale, int unrotate_out, void* out,
                                  void* workspace, size_t ws_bytes, void* stream) {
  return decode_impl<false>(q, k_q, k_s, nullptr, v_q, v_s, nullptr, B, Hq, Hkv, d, T, T_max, sm_scale, unrotate_out,
                            out, workspace, ws_bytes, stream);
}

extern "C" int quarot_decode_attn_asym(const void* q, const uint8_t* k_q, const void* k_s, const int16_t* k_z,
                                       const uint8_t* v_q, const void* v_s, const int16_t* v_z, int64_t B,
                                       int64_t Hq, int64_t Hkv, int64_t d, int64_t T, int64_t T_max, float sm_scale,
                                       int unrotate_out, void* out, void* workspace, size_t ws_bytes, void* stream) {
  return decode_impl<true>(q, k_q, k_s, k_z, v_q, v_s, v_z, B, Hq, Hkv, d, T, T_max, sm_scale, unrotate_out, out,
                           workspace, ws_bytes, stream);
}
