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

template <int D>
__global__ void __launch_bounds__(256)
kv_write_kernel(const __half* __restrict__ k_src, const __half* __restrict__ v_src, int64_t B, int64_t T_new,
                int64_t Hkv, int64_t t_start, int64_t T_max, uint8_t* __restrict__ k_q, __half* __restrict__ k_s,
                uint8_t* __restrict__ v_q, __half* __restrict__ v_s) {
  constexpr int TPV = D / 32;
  // blockIdx.y selects the tensor: 0 = keys, 1 = values
  const __half* __restrict__ src = blockIdx.y == 0 ? k_src : v_src;
  uint8_t* __restrict__ cq = blockIdx.y == 0 ? k_q : v_q;
  __half* __restrict__ cs = blockIdx.y == 0 ? k_s : v_s;
  const int64_t gt = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nvec = B * Hkv * T_new;
  const int64_t vi = gt / TPV;
  const int part = int(gt % TPV);
  const bool valid = vi < nvec;
  const int64_t t = valid ? vi % T_new : 0;
  const int64_t bh = valid ? vi / T_new : 0;
  const int64_t h = bh % Hkv, b = bh / Hkv;

  float v[32];
  if (valid) {
    const uint4* p = reinterpret_cast<const uint4*>(src + ((b * T_new + t) * Hkv + h) * D + part * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 r = __ldcs(p + i);
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
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] *= inv_sqrt_d;
    amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 1; o < TPV; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const __half S = quant_scale_fp16(amax, 1.0f);
  const float inv = 1.0f / __half2float(S);
  uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float y = fminf(fmaxf(v[i] * inv, -8.0f), 7.0f);
    w[i >> 3] |= nibble_rne(y) << (4 * (i & 7));
  }
  if (valid) {
    const int64_t pos = (b * Hkv + h) * T_max + t_start + t;
    __stcs(reinterpret_cast<uint4*>(cq + pos * (D / 2) + part * 16), make_uint4(w[0], w[1], w[2], w[3]));
    if (part == 0) cs[pos] = S;
  }
}

// ------------------------------------------------------------------ decode
constexpr int HD = 128;       // head_dim of the decode kernel
constexpr int MAXG = 8;       // query heads per KV head
constexpr int CHUNK = 256;    // tokens per split
constexpr int DT = 128;       // threads per CTA

__host__ __device__ inline int64_t num_splits(int64_t T) {
  const int64_t s = (T + CHUNK - 1) / CHUNK;
  return s < 1 ? 1 : s;
}

// Nibble n (0..15) of a two's complement code -> float value, exactly:
// 2^23 + (n ^ 8) as fp32 bits, minus 2^23 + 8.
__device__ __forceinline__ float code_f(uint32_t n) {
  return __int_as_float(0x4B000000 | ((n ^ 8u) & 0xFu)) - 8388616.0f;
}

// One CTA per (split, b, g): partial softmax state of the GQA group's heads
// over one chunk of tokens.  Scores use exp2 with log2(e) folded into q~.
template <int G>
__global__ void __launch_bounds__(DT)
decode_partial_kernel(const __half* __restrict__ q, const uint8_t* __restrict__ kq,
                      const __half* __restrict__ ks, const uint8_t* __restrict__ vq,
                      const __half* __restrict__ vs, int Hq, int Hkv, int T, int T_max,
                      float qscale, float* __restrict__ ws_o, float* __restrict__ ws_ml, int splits) {
  __shared__ float qs[G][HD];
  __shared__ float sc[CHUNK][G];          // scores, then p * v_scale
  __shared__ __align__(16) uint8_t vcode[CHUNK][HD / 2];
  __shared__ float red[DT / 32][G];
  __shared__ float mrow[G], lrow[G];

  const int split = blockIdx.x;
  const int bg = blockIdx.y;
  const int b = bg / Hkv, g = bg % Hkv;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int t0 = split * CHUNK;
  const int tn = min(CHUNK, T - t0);      // tokens in this chunk (may be <= 0)
  const int64_t cache_row = (int64_t(b) * Hkv + g) * T_max;

  // q~ = q H / sqrt(d) * qscale, head-wise FWHT in shared memory
  for (int i = tid; i < G * HD; i += DT) {
    const int hh = i / HD, e = i % HD;
    qs[hh][e] = __half2float(q[(int64_t(b) * Hq + g * G + hh) * HD + e]);
  }
  __syncthreads();
  for (int hspan = 1; hspan < HD; hspan <<= 1) {
    for (int i = tid; i < G * HD / 2; i += DT) {
      const int hh = i / (HD / 2), pr = i % (HD / 2);
      const int lo = (pr / hspan) * 2 * hspan + (pr % hspan);
      const float a = qs[hh][lo], c = qs[hh][lo + hspan];
      qs[hh][lo] = a + c;
      qs[hh][lo + hspan] = a - c;
    }
    __syncthreads();
  }
  for (int i = tid; i < G * HD; i += DT) (&qs[0][0])[i] *= qscale;
  // stage the chunk's value codes
  for (int i = tid; i < CHUNK * (HD / 2) / 16; i += DT) {
    const int tok = i / (HD / 32), part = i % (HD / 32);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (tok < tn) val = __ldcs(reinterpret_cast<const uint4*>(vq + (cache_row + t0 + tok) * (HD / 2)) + part);
    *reinterpret_cast<uint4*>(&vcode[tok][part * 16]) = val;
  }
  __syncthreads();

  // scores: one thread per token
  float lmax[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) lmax[hh] = -INFINITY;
  for (int tok = tid; tok < tn; tok += DT) {
    const uint4* kp = reinterpret_cast<const uint4*>(kq + (cache_row + t0 + tok) * (HD / 2));
    float acc[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) acc[hh] = 0.f;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      const uint4 r = __ldcs(kp + c);
      const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int wi = 0; wi < 4; ++wi)
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const float kv = code_f(wv[wi] >> (4 * n));
          const int e = c * 32 + wi * 8 + n;
#pragma unroll
          for (int hh = 0; hh < G; ++hh) acc[hh] = fmaf(qs[hh][e], kv, acc[hh]);
        }
    }
    const float ksc = __half2float(ks[cache_row + t0 + tok]);
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float s = acc[hh] * ksc;
      sc[tok][hh] = s;
      lmax[hh] = fmaxf(lmax[hh], s);
    }
  }
  // chunk max per head
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    float m = lmax[hh];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[wid][hh] = m;
  }
  __syncthreads();
  if (tid < G) {
    float m = red[0][tid];
#pragma unroll
    for (int w = 1; w < DT / 32; ++w) m = fmaxf(m, red[w][tid]);
    mrow[tid] = m;
  }
  __syncthreads();
  // p = exp2(s - m); keep p * v_scale for the PV sweep, sum p for l
  float lsum[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) lsum[hh] = 0.f;
  for (int tok = tid; tok < tn; tok += DT) {
    const float vsc = __half2float(vs[cache_row + t0 + tok]);
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float p = exp2f(sc[tok][hh] - mrow[hh]);
      lsum[hh] += p;
      sc[tok][hh] = p * vsc;
    }
  }
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    float l = lsum[hh];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) red[wid][hh] = l;
  }
  __syncthreads();
  if (tid < G) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < DT / 32; ++w) l += red[w][tid];
    lrow[tid] = l;
  }
  // PV: thread = output dim
  float o[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) o[hh] = 0.f;
  const int e = tid;
  for (int tok = 0; tok < tn; ++tok) {
    const float vv = code_f(uint32_t(vcode[tok][e >> 1]) >> (4 * (e & 1)));
#pragma unroll
    for (int hh = 0; hh < G; ++hh) o[hh] = fmaf(sc[tok][hh], vv, o[hh]);
  }
  __syncthreads();
  const int64_t base = (int64_t(b) * Hq + g * G) * splits + split;
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const int64_t slot = base + int64_t(hh) * splits;
    ws_o[slot * HD + e] = o[hh];
    if (tid == 0) {
      ws_ml[slot * 2 + 0] = mrow[hh];
      ws_ml[slot * 2 + 1] = lrow[hh];
    }
  }
}

// Merge the splits of one (b, h): o = sum_s 2^(m_s - m) o_s / sum_s 2^(m_s - m) l_s,
// then optionally rotate back by H / sqrt(d); fp16 out.
__global__ void __launch_bounds__(HD)
decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml, int splits,
                      int unrotate, __half* __restrict__ out) {
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

}  // namespace kv
}  // namespace quarot

using namespace quarot;

extern "C" int quarot_kv_write(const void* k, const void* v, int64_t B, int64_t T_new, int64_t Hkv,
                               int64_t d, int64_t t_start, int64_t T_max, uint8_t* k_q, void* k_s,
                               uint8_t* v_q, void* v_s, void* stream) {
  if (B < 0 || T_new < 0 || Hkv <= 0 || t_start < 0 || T_max <= 0) return QUAROT_ERR_INVALID_ARG;
  if (t_start + T_new > T_max) return QUAROT_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return QUAROT_ERR_UNSUPPORTED;
  if (B == 0 || T_new == 0) return QUAROT_OK;
  if (!k || !v || !k_q || !k_s || !v_q || !v_s) return QUAROT_ERR_INVALID_ARG;
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(k, 16) || mis(v, 16) || mis(k_q, 16) || mis(v_q, 16) || mis(k_s, 2) || mis(v_s, 2))
    return QUAROT_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t threads = B * Hkv * T_new * (d / 32);
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  auto go = [&](auto kern) {
    kern<<<dim3(unsigned(blocks), 2), 256, 0, st>>>(static_cast<const __half*>(k), static_cast<const __half*>(v),
                                                    B, T_new, Hkv, t_start, T_max, k_q, static_cast<__half*>(k_s),
                                                    v_q, static_cast<__half*>(v_s));
  };
  if (d == 64) go(kv::kv_write_kernel<64>);
  else if (d == 128) go(kv::kv_write_kernel<128>);
  else go(kv::kv_write_kernel<256>);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

extern "C" size_t quarot_decode_workspace_bytes(int64_t B, int64_t Hq, int64_t d, int64_t T) {
  if (B <= 0 || Hq <= 0 || d != kv::HD || T < 0) return 0;
  const int64_t s = kv::num_splits(T);
  const size_t bytes = size_t(B * Hq * s) * (kv::HD + 2) * sizeof(float);
  return (bytes + 255) & ~size_t(255);
}

extern "C" int quarot_decode_attn(const void* q, const uint8_t* k_q, const void* k_s, const uint8_t* v_q,
                                  const void* v_s, int64_t B, int64_t Hq, int64_t Hkv, int64_t d, int64_t T,
                                  int64_t T_max, float sm_scale, int unrotate_out, void* out,
                                  void* workspace, size_t ws_bytes, void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || T < 0 || T_max < 0 || T > T_max) return QUAROT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return QUAROT_ERR_INVALID_ARG;
  if (d != kv::HD || Hq / Hkv > kv::MAXG) return QUAROT_ERR_UNSUPPORTED;
  if (B == 0) return QUAROT_OK;
  if (!q || !out) return QUAROT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    return cudaMemsetAsync(out, 0, size_t(B * Hq * d) * 2, st) == cudaSuccess ? QUAROT_OK : QUAROT_ERR_CUDA;
  }
  if (!k_q || !k_s || !v_q || !v_s || !workspace) return QUAROT_ERR_INVALID_ARG;
  if (ws_bytes < quarot_decode_workspace_bytes(B, Hq, d, T)) return QUAROT_ERR_INVALID_ARG;
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k_q, 16) || mis(v_q, 16) || mis(k_s, 2) || mis(v_s, 2) || mis(out, 16) ||
      mis(workspace, 256))
    return QUAROT_ERR_ALIGNMENT;
  if (B * Hkv > 65535 || T > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  const int splits = int(kv::num_splits(T));
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(float(d));
  const float qscale = scale * 1.4426950408889634f / sqrtf(float(d));  // 1/sqrt(d) of H, log2(e)
  float* ws_o = static_cast<float*>(workspace);
  float* ws_ml = ws_o + size_t(B * Hq * splits) * kv::HD;
  dim3 grid(unsigned(splits), unsigned(B * Hkv));
  const int G = int(Hq / Hkv);
  auto args = [&](auto kern) {
    kern<<<grid, kv::DT, 0, st>>>(static_cast<const __half*>(q), k_q, static_cast<const __half*>(k_s), v_q,
                                  static_cast<const __half*>(v_s), int(Hq), int(Hkv), int(T), int(T_max),
                                  qscale, ws_o, ws_ml, splits);
  };
  switch (G) {
    case 1: args(kv::decode_partial_kernel<1>); break;
    case 2: args(kv::decode_partial_kernel<2>); break;
    case 4: args(kv::decode_partial_kernel<4>); break;
    case 8: args(kv::decode_partial_kernel<8>); break;
    default: return QUAROT_ERR_UNSUPPORTED;
  }
  kv::decode_combine_kernel<<<unsigned(B * Hq), kv::HD, 0, st>>>(ws_o, ws_ml, splits, unrotate_out,
                                                                 static_cast<__half*>(out));
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}
