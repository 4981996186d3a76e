// quarot_w4a4_gemm: packed INT4 x packed INT4 GEMM on the sm_103a tensor
// cores (tcgen05, TMEM accumulator, TMA loads) with the per-token x
// per-output-channel dequantization epilogue.
//
// What it computes -- "QuaRot: Outlier-Free 4-Bit Inference in Rotated LLMs"
// (paper summary), Stage 2b "dequantization step" and "Kernel Implementation
// and Hardware Efficiency": an INT4 GEMM with an INT32 accumulator whose
// result is scaled by scale_x[i] * scale_w[j]; "QuaRot Guide: Outlier-Free
// 4-Bit W4A4 LLM Quantization", "Pure INT4 Tensor Core GEMM Execution".
//
// How, on sm_103a: tcgen05 has no INT4 kind and no INT8 kind on this target,
// so the contraction runs on kind::f8f6f4 (e4m3 x e4m3 -> fp32 in TMEM) with
// an exact encoding:
//   * a code v in [-8, 7] is offset to u = v + 8 in [0, 15] (one XOR of the
//     nibble with 8);
//   * the e4m3 byte with value u (0x00..0x0F) is exactly u * 2^-9: bytes
//     0x01..0x07 are the subnormals u * 2^-9 and 0x08..0x0F the first binade
//     (8 + m) * 2^-9, so the nibble itself is the fp8 operand;
//   * every product is a multiple of 2^-18 and every partial sum is a
//     non-negative integer multiple of 2^-18 below 225 * K * 2^-18 <= 2^24 *
//     2^-18 for K <= 65536, so fp32 accumulation is exact;
//   * sum_k a_k w_k = sum_k u_k u'_k - 8 sum_k u_k - 8 sum_k u'_k + 64 K,
//     with the row sums of the offset codes gathered while unpacking.
// Within each group of 8 codes the unpacked byte order is (0,2,4,6,1,3,5,7);
// the same permutation of K on both operands leaves the product unchanged.
//
// Persistent kernel, one CTA per SM, 576 threads in five roles:
//   warp 0        TMA producer: packed A/W k-blocks into a 4-stage ring (64B swizzle)
//   warp 1        TMEM allocator and single-thread MMA issuer
//   warps 2-5     A converters: packed nibbles -> e4m3 bytes written straight
//                 into tensor memory (tcgen05.st), the MMA's A operand, 2 stages
//   warps 6-13    W converters: packed nibbles -> e4m3 bytes in a 2-stage
//                 shared-memory ring laid out for the 128B-swizzled K-major
//                 UMMA descriptor; both converter groups also sum the offset
//                 codes of their rows
//   warps 14-17   epilogue: TMEM -> registers -> integer correction -> fp16
// Tiles are 128 x BN (BN in {128..224} chosen per shape so the tiles split
// evenly over the SMs).  Tensor memory holds the accumulator (columns
// [0, BN)) and four A stages (columns 256 + 32 s).  Four unpacked stages give
// the MMA issue chain (MMA done -> commit -> converter -> barrier -> next MMA)
// three k-blocks of tensor work to hide behind; with two stages the tensor
// pipe idled between k-blocks.  Every wait is bounded; an expired wait
// records QUAROT_ERR_TIMEOUT and the CTA drains its copies and MMAs, frees
// TMEM and returns.
//
// The file holds three kernels: the one-SM kernel above (M <= 128 or an odd
// k-block count), the CTA-pair kernel (namespace pair) and the CTA-pair kernel
// for activations already widened to operand bytes by quarot_rotate_quant_a8
// (namespace pair::a8, entry point quarot_w4a4_gemm_a8).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace quarot {
namespace gemm {

constexpr int BM = 128, BN_MAX = 224, BK = 128;  // tile in codes
constexpr int BKB = BK / 2;                      // packed bytes per row per k-block
constexpr int SP = 4;                            // packed ring stages
constexpr int SU = 4;                            // unpacked ring stages (A in TMEM, W in smem)
constexpr int NCONV = 384;                       // converter threads (12 warps)
constexpr int NEPI = 128;                        // epilogue threads (4 warps)
constexpr int EPI_WARP0 = 2 + NCONV / 32;        // 14
constexpr int NTHREADS = 64 + NCONV + NEPI;      // 576
constexpr int A_PK = BM * BKB, B_PK = BN_MAX * BKB;  // 8 KB, 14 KB
constexpr int B_UN = BN_MAX * BK;                    // 28 KB
constexpr int OFF_BU = 0;
constexpr int OFF_AP = OFF_BU + SU * B_UN;
constexpr int OFF_BP = OFF_AP + SP * A_PK;
constexpr int OFF_BAR = OFF_BP + SP * B_PK;
constexpr int NBAR = 2 * SP + 2 * SU + 8 + 1;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int OFF_RSA = OFF_MISC + 16;             // int [2][BM]
constexpr int OFF_RSB = OFF_RSA + 2 * BM * 4;      // float [2][BN_MAX]: -8 x the W row sums (exact)
constexpr int SMEM_USED = OFF_RSB + 2 * BN_MAX * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
constexpr uint32_t TMEM_COLS = 512;           // accumulator (up to 224 columns) + A stages
constexpr uint32_t TMEM_A_COL = 256;          // A stage s at column 256 + 32 s (128 bytes per row)
constexpr int NCONV_WARPS = NCONV / 32;       // arrivals per converter barrier phase
constexpr int NEPI_WARPS = NEPI / 32;
constexpr int MAX_K = 65536;

// Instruction descriptor, kind::f8f6f4: D fp32, A/B e4m3, both K-major,
// M = 128; N (bits 17-22, N >> 3) is filled in at run time.
constexpr uint32_t IDESC_BASE = (1u << 4) | (0u << 7) | (0u << 10) | (uint32_t(BM >> 4) << 24);

// Shared-memory matrix descriptor for a K-major operand in the 128B swizzle
// layout: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFF) >> 4);
  d |= uint64_t(1) << 16;             // leading byte offset (unused for this layout)
  d |= uint64_t(1024 >> 4) << 32;     // stride byte offset
  d |= uint64_t(1) << 46;             // descriptor version
  d |= uint64_t(2) << 61;             // SWIZZLE_128B
  return d;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_f8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_f8_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define QUAROT_TMEM_LD32(taddr, r)                                                                 \
  asm volatile(                                                                                    \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"               \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),       \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),   \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),             \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),             \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])              \
      : "r"(taddr))

#define QUAROT_TMEM_ST32(taddr, r)                                                                 \
  asm volatile(                                                                                    \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),       \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),     \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), \
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),          \
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),          \
      "r"(r[30]), "r"(r[31])                                                                       \
      : "memory")

// 8 packed codes (one 32-bit word) -> 8 offset codes as bytes, order
// (0,2,4,6 | 1,3,5,7); also returns their byte-wise sum word.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = (w ^ 0x88888888u) & 0x0F0F0F0Fu;
  hi = ((w >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;
}

// One packed 64-byte row chunk set (4 x 16 B, 64B-swizzled source) -> 128
// e4m3 bytes (128B-swizzled destination); returns the byte sum of the offset
// codes.
__device__ __forceinline__ uint32_t convert_row(const unsigned char* src_row, int r, unsigned char* dst_row) {
  uint4 w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint4*>(src_row + ((c ^ ((r >> 1) & 3)) << 4));
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
    unpack_word(w[c].x, l0, h0);
    unpack_word(w[c].y, l1, h1);
    unpack_word(w[c].z, l2, h2);
    unpack_word(w[c].w, l3, h3);
    acc = __dp4a((l0 + h0) + (l1 + h1) + (l2 + h2) + (l3 + h3), 0x01010101u, acc);
    *reinterpret_cast<uint4*>(dst_row + (((2 * c) ^ (r & 7)) << 4)) = make_uint4(l0, h0, l1, h1);
    *reinterpret_cast<uint4*>(dst_row + (((2 * c + 1) ^ (r & 7)) << 4)) = make_uint4(l2, h2, l3, h3);
  }
  return acc;
}

static_assert(OFF_AP % 1024 == 0 && OFF_BP % 1024 == 0 && OFF_BAR % 8 == 0, "stage alignment");

// The A-side variant: the 128 converted bytes of the row go to 32 registers
// (K order identical to convert_row) for one tcgen05.st.
__device__ __forceinline__ uint32_t convert_row_regs(const unsigned char* src_row, int r, uint32_t* o) {
  uint4 w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = *reinterpret_cast<const uint4*>(src_row + ((c ^ ((r >> 1) & 3)) << 4));
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    unpack_word(w[c].x, o[8 * c + 0], o[8 * c + 1]);
    unpack_word(w[c].y, o[8 * c + 2], o[8 * c + 3]);
    unpack_word(w[c].z, o[8 * c + 4], o[8 * c + 5]);
    unpack_word(w[c].w, o[8 * c + 6], o[8 * c + 7]);
    acc = __dp4a((o[8 * c] + o[8 * c + 1]) + (o[8 * c + 2] + o[8 * c + 3]) + (o[8 * c + 4] + o[8 * c + 5]) +
                     (o[8 * c + 6] + o[8 * c + 7]),
                 0x01010101u, acc);
  }
  return acc;
}

__global__ void __launch_bounds__(NTHREADS, 1)
w4a4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __half* __restrict__ sx, const __half* __restrict__ sw, int M, int N, int K, int BN,
                 __half* __restrict__ y, int32_t* __restrict__ acc_out) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* pk_full = bars;
  uint64_t* pk_empty = bars + SP;
  uint64_t* un_full = bars + 2 * SP;
  uint64_t* un_empty = bars + 2 * SP + SU;
  uint64_t* acc_full = bars + 2 * SP + 2 * SU;   // [2]
  uint64_t* acc_empty = acc_full + 2;            // [2]
  uint64_t* rs_full = acc_full + 4;              // [2]
  uint64_t* rs_empty = acc_full + 6;             // [2]
  uint64_t* drain = acc_full + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 4);
  int* rsA = reinterpret_cast<int*>(sm + OFF_RSA);
  float* rsB = reinterpret_cast<float*>(sm + OFF_RSB);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = K / BK;
  const int n_tiles_n = (N + BN - 1) / BN;
  const int n_tiles = ((M + BM - 1) / BM) * n_tiles_n;
  const uint32_t idesc = IDESC_BASE | (uint32_t(BN >> 3) << 17);
  const int b_bytes = BN * BKB;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < SP; ++s) {
      mbar_init(&pk_full[s], 1);
      mbar_init(&pk_empty[s], NCONV_WARPS);
    }
    for (int s = 0; s < SU; ++s) {
      mbar_init(&un_full[s], NCONV_WARPS);
      mbar_init(&un_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], NEPI_WARPS);
      mbar_init(&rs_full[s], NCONV_WARPS);
      mbar_init(&rs_empty[s], NEPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(const_cast<uint32_t*>(tmem_slot))),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      long issued = 0;
      long it = 0;
      for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
        const int m0 = (tile / n_tiles_n) * BM, n0 = (tile % n_tiles_n) * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = int(it % SP);
          if (!mbar_wait_bounded(&pk_empty[s], uint32_t((it / SP) & 1) ^ 1u, abort_flag)) break;
          mbar_arrive_expect_tx(&pk_full[s], A_PK + b_bytes);
          tma_load_2d(smem_u32(sm + OFF_AP + s * A_PK), &tmA, kb * BKB, m0, &pk_full[s]);
          tma_load_2d(smem_u32(sm + OFF_BP + s * B_PK), &tmB, kb * BKB, n0, &pk_full[s]);
          issued = it + 1;
        }
      }
      if (*abort_flag) {
        // drain: every issued copy must land before the CTA exits
        for (long j = (issued > SP ? issued - SP : 0); j < issued; ++j)
          mbar_wait_bounded(&pk_full[j % SP], uint32_t((j / SP) & 1), nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      long it = 0;
      int ti = 0;
      for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x, ++ti) {
        const int a = 0;  // one accumulator: the epilogue must drain it first
        if (!mbar_wait_bounded(&acc_empty[0], uint32_t(ti & 1) ^ 1u, abort_flag)) break;
        fence_after_sync();
        const uint32_t tmem_d = tmem_base;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = int(it % SU);
          if (!mbar_wait_bounded(&un_full[s], uint32_t((it / SU) & 1), abort_flag)) {
            ok = false;
            break;
          }
          fence_after_sync();
          const uint32_t ta = tmem_base + TMEM_A_COL + uint32_t(32 * s);
          const uint64_t bd = sw128_desc(smem_u32(sm + OFF_BU + s * B_UN));
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            mma_f8_ts(tmem_d, ta + uint32_t(8 * kk), bd + uint64_t(2 * kk), idesc, (kb | kk) != 0);
          mma_commit(&un_empty[s]);
        }
        if (!ok) break;
        mma_commit(&acc_full[a]);  // a == 0
      }
      // every issued MMA must finish before TMEM is freed
      mma_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ converters
    // warps 2-5: A rows 32 * (warp % 4) + lane (the TMEM lane quadrant the warp
    // may access); warps 6-13: W rows 0..255
    const bool is_a = warp < 6;
    const int r = is_a ? 32 * (warp & 3) + lane : int(threadIdx.x) - 64 - BM;
    const uint32_t tmem_a_row = tmem_base + TMEM_A_COL + (uint32_t(32 * (warp & 3)) << 16);
    long it = 0;
    int ti = 0;
    for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x, ++ti) {
      uint32_t sum = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int sp = int(it % SP), su = int(it % SU);
        if (!mbar_wait_bounded(&pk_full[sp], uint32_t((it / SP) & 1), abort_flag) ||
            !mbar_wait_bounded(&un_empty[su], uint32_t((it / SU) & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (is_a) {
          uint32_t o[32];
          sum += convert_row_regs(sm + OFF_AP + sp * A_PK + r * 64, r, o);
          QUAROT_TMEM_ST32(tmem_a_row + uint32_t(32 * su), o);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          fence_before_sync();
        } else {
          if (r < BN) sum += convert_row(sm + OFF_BP + sp * B_PK + r * 64, r, sm + OFF_BU + su * B_UN + r * 128);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&un_full[su]);
          mbar_arrive(&pk_empty[sp]);
        }
      }
      if (!ok) break;
      const int a = ti & 1;
      if (!mbar_wait_bounded(&rs_empty[a], uint32_t((ti >> 1) & 1) ^ 1u, abort_flag)) break;
      if (is_a) rsA[a * BM + r] = int(sum);
      else if (r < BN_MAX) rsB[a * BN_MAX + r] = -8.0f * float(int(sum));  // exact: |8 sum| < 2^24
      __syncwarp();
      if (lane == 0) mbar_arrive(&rs_full[a]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int r = 32 * q + lane;
    const bool vec_ok = (N % 8) == 0;
    int ti = 0;
    for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x, ++ti) {
      const int a = ti & 1;  // row-sum buffer (double-buffered); the accumulator is single
      const uint32_t par = uint32_t((ti >> 1) & 1);
      if (!mbar_wait_bounded(&acc_full[0], uint32_t(ti & 1), abort_flag) ||
          !mbar_wait_bounded(&rs_full[a], par, abort_flag))
        break;
      fence_after_sync();
      const int m0 = (tile / n_tiles_n) * BM, n0 = (tile % n_tiles_n) * BN;
      const int gm = m0 + r;
      const float sxr = gm < M ? __half2float(sx[gm]) : 0.f;
      const float bias_r = 64.0f * float(K) - 8.0f * float(rsA[a * BM + r]);
      const float* rsb = rsB + a * BN_MAX;
      const uint32_t tmem_row = tmem_base + (uint32_t(32 * q) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        __syncwarp();
        QUAROT_TMEM_LD32(tmem_row + uint32_t(c0), v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int gn = n0 + c0;
        if (gm < M && gn < N) {
          float acc[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            acc[j] = __fadd_rn(__fmaf_rn(__uint_as_float(v[j]), 262144.0f, rsb[c0 + j]), bias_r);
          __half* yrow = y + size_t(gm) * N + gn;
          if (vec_ok && gn + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              const uint4 s8 = __ldg(reinterpret_cast<const uint4*>(sw + gn + j));
              const uint32_t sws[4] = {s8.x, s8.y, s8.z, s8.w};
              uint32_t o[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 wsc = h2_to_f2(sws[e]);
                const __half2 hv = __floats2half2_rn(__fmul_rn(__fmul_rn(acc[j + 2 * e], sxr), wsc.x),
                                                     __fmul_rn(__fmul_rn(acc[j + 2 * e + 1], sxr), wsc.y));
                o[e] = *reinterpret_cast<const uint32_t*>(&hv);
              }
              *reinterpret_cast<uint4*>(yrow + j) = make_uint4(o[0], o[1], o[2], o[3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gn + j < N) yrow[j] = __float2half_rn(__fmul_rn(__fmul_rn(acc[j], sxr), __half2float(sw[gn + j])));
          }
          if (acc_out != nullptr) {
            int32_t* arow = acc_out + size_t(gm) * N + gn;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gn + j < N) arow[j] = __float2int_rn(acc[j]);
          }
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&acc_empty[0]);
        mbar_arrive(&rs_empty[a]);
      }
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ===================================================================== 2-SM kernel
// The same contraction on CTA pairs (thread-block clusters of 2) with the
// 2-SM MMA, tcgen05.mma.cta_group::2: a pair computes a 256 x BN tile; each
// CTA holds its 128 rows of A (converted into its own tensor memory) and one
// half of the BN weight rows (converted into its own shared memory), so each
// SM converts 128 + BN/2 rows per k-block instead of 128 + BN.  The leader
// CTA (rank 0) issues the MMAs; completion is committed to both CTAs'
// barriers (multicast); the peer's converters and epilogue signal the
// leader's barriers remotely.  Per CTA, tensor memory holds two accumulators
// (columns [0, BN) and [BN, 2 BN)) and two A stages (columns 448, 480).
namespace pair {

// 2-SM variant for M > 128: clusters of two CTAs on one TPC share a 256 x BN
// tile through tcgen05.mma.cta_group::2 (M = 256).  Each CTA converts its own
// 128 activation rows (into its tensor memory, as the A operand) and HALF of
// the BN weight rows (into its shared memory); the pair's tensor cores read
// both halves of W, so per SM a k-block needs 128 + BN/2 converted rows
// instead of 128 + BN.  Only the leader CTA (rank 0) issues MMAs and its
// commits are multicast back to both CTAs.  Warps signal only barriers of
// their own CTA (cta-scope release, no cluster-wide fence on the converters'
// critical path); in the other CTA one relay thread (warp 1, idle there)
// forwards each completed stage to the leader with a single remote arrival.
//
// Converted operands go through one ring of S = 8 stages: stage s holds the A
// k-block in tensor memory (columns 256 + 32 s) and this CTA's W half in shared
// memory, behind one full and one empty barrier.  Tensor memory also holds one
// accumulator in columns [0, BN).  Eight stages let the converters run ahead
// of the MMA by 8 k-blocks, which hides the cross-SM round trip (converters
// done -> relay -> leader MMA -> multicast commit -> stage free, about 2 us)
// and the epilogue of the previous tile (the MMA of the next tile waits for
// the epilogue to drain the accumulator, the converters do not).  Row sums of the converted W rows are
// written into both CTAs' shared memory so that each epilogue reads its
// correction terms locally.
//
// The MMA issuer and the relay take the converted stages in pairs (one wait
// per pair, eight MMAs back to back): a tcgen05.mma issue blocks about as
// long as the MMA runs, so any per-stage wait between two k-blocks idled the
// tensor pipe (85.0 -> 79.2 us at 2048 x 4096 x 12288; groups of four were
// slower, 81.7 us).
//
//   warp 0         TMA producer (this CTA's 128 A rows and BN/2 W rows)
//   warp 1         TMEM allocator; MMA issuer in the leader, relay in the peer
//   warps 2-9      A converters (packed -> e4m3 bytes -> TMEM), two warps per
//                  TMEM lane quadrant, each converting half of every row
//   warps 10-17    W converters (packed -> e4m3 bytes -> shared memory), 16
//                  rows per warp, lanes l and l + 16 converting the two halves
//                  of one row
//   warps 18-21    epilogue, one warp per TMEM lane quadrant
// Converting half rows gives each thread a short dependency chain per k-block
// and four converter warps per scheduler to hide it.
constexpr int BM = 128;          // rows per CTA (256 per pair)
constexpr int BNH_MAX = 112;     // weight rows per CTA (BN <= 224)
// Packed ring: SP k-block stages, loaded as SP / 2 double stages.  One TMA box
// of 128-byte rows (128B swizzle) covers k-blocks kb and kb + 1 of a row, so
// stage pair (s, s + 1) is one box per operand behind the barriers of stage s
// (the barriers of odd stages are unused).  Half as many TMA row requests as
// 64-byte boxes: 86.1 -> 85.0 us at 2048 x 4096 x 12288.
constexpr int SP = 6;
constexpr int S = 8;             // converted stages (A in tensor memory, W in shared memory)
constexpr int NAW = 8, NBW = 8;  // A / W converter warps
constexpr int NCW = NAW + NBW;
constexpr int NEW = 4;           // epilogue warps
constexpr int EPI_WARP0 = 2 + NCW;
constexpr int NTHREADS = 32 * (2 + NCW + NEW);  // 704
constexpr int A_PK = BM * BKB, B_PK = BNH_MAX * BKB;  // 8 KB, 7 KB
constexpr int B_UN = BNH_MAX * BK;                     // 14 KB
constexpr int OFF_BU = 0;
constexpr int OFF_AP = OFF_BU + S * B_UN;
constexpr int OFF_BP = OFF_AP + SP * A_PK;
constexpr int OFF_BAR = ((OFF_BP + SP * B_PK) + 1023) / 1024 * 1024;
// barriers: pk_full[SP] pk_empty[SP] full[S] empty[S] acc_full acc_empty
//           rs_full[2] rs_empty[2] drain
constexpr int NBAR = 2 * SP + 2 * S + 2 + 4 + 1;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int OFF_RSA = (OFF_MISC + 16 + 127) / 128 * 128;  // int [2][2][BM]: per half row
constexpr int OFF_RSB = OFF_RSA + 4 * BM * 4;      // float [2][BN_MAX]: -8 x the tile's W row sums (exact)
constexpr int OFF_SW = OFF_RSB + 2 * BN_MAX * 4;   // float [NEW][BN_MAX]: each epilogue warp's weight scales
constexpr int SMEM_USED = OFF_SW + NEW * BN_MAX * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_A_COL = 256;
constexpr uint32_t IDESC_BASE = (1u << 4) | (0u << 7) | (0u << 10) | (uint32_t(256 >> 4) << 24);
static_assert(OFF_AP % 1024 == 0 && OFF_BP % 1024 == 0, "stage alignment");
static_assert(B_PK % 1024 == 0 && B_UN % 1024 == 0 && A_PK % 1024 == 0, "stage alignment");
static_assert(TMEM_A_COL + 32 * S <= TMEM_COLS && BN_MAX <= int(TMEM_A_COL), "tensor memory plan");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
static_assert(SP % 2 == 0 && S % 2 == 0, "converters take stages in pairs");
static_assert(OFF_RSB % 16 == 0 && OFF_SW % 16 == 0 && (BN_MAX * 4) % 16 == 0, "16-byte shared loads of row sums and scales");

// The three forms of the pair kernel.  V = 0: eight converted stages, A
// stages at tensor-memory columns [256, 512), one accumulator at [0, BN) with
// BN up to 224.  V = 1 and 2, for pairs that run many tiles (each tile's
// accumulator drain would otherwise idle the tensor pipe): two accumulators
// -- the epilogue drains tile i's while the MMAs of tile i + 1 fill the
// other -- at [0, 160) and [160, 320) with six converted stages at
// [320, 512) and BN up to 160 (V = 1), or at [0, 192) and [192, 384) with
// four converted stages at [384, 512) and BN up to 192 (V = 2).
template <int V>
struct Layout {
  static constexpr bool DBL = V != 0;
  static constexpr int S = V == 0 ? pair::S : (V == 1 ? 6 : 4);
  static constexpr int NACC = DBL ? 2 : 1;
  static constexpr uint32_t ACC_COLS = V == 0 ? 0u : (V == 1 ? 160u : 192u);
  static constexpr uint32_t A_COL = V == 0 ? TMEM_A_COL : (V == 1 ? 320u : 384u);
  static constexpr int BN_LIMIT = V == 0 ? BN_MAX : int(ACC_COLS);
  static constexpr int OFF_BU = 0;
  static constexpr int OFF_AP = OFF_BU + S * B_UN;
  static constexpr int OFF_BP = OFF_AP + SP * A_PK;
  static constexpr int OFF_BAR = ((OFF_BP + SP * B_PK) + 1023) / 1024 * 1024;
  // barriers: pk_full[SP] pk_empty[SP] full[S] empty[S] acc_full[NACC]
  //           acc_empty[NACC] rs_full[2] rs_empty[2] drain
  static constexpr int NBAR = 2 * SP + 2 * S + 2 * NACC + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_RSA = (OFF_MISC + 16 + 127) / 128 * 128;
  static constexpr int OFF_RSB = OFF_RSA + 4 * BM * 4;
  static constexpr int OFF_SW = OFF_RSB + 2 * BN_MAX * 4;
  // each epilogue warp's column corrections of the tile when the weight row
  // sums are given (float [NEW][BN_MAX])
  static constexpr int OFF_RW = OFF_SW + NEW * BN_MAX * 4;
  static constexpr int SMEM_BYTES = OFF_RW + NEW * BN_MAX * 4 + 1024;
  static_assert(OFF_AP % 1024 == 0 && OFF_BP % 1024 == 0, "stage alignment");
  static_assert(A_COL + 32 * S <= TMEM_COLS, "A stages in tensor memory");
  static_assert(uint32_t(NACC - 1) * ACC_COLS + uint32_t(BN_LIMIT) <= A_COL, "accumulators below the A stages");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(S % 2 == 0, "converters take stages in pairs");
  static_assert(OFF_RSB % 16 == 0 && OFF_SW % 16 == 0, "16-byte shared loads of row sums and scales");
};
static_assert(Layout<0>::OFF_BAR == OFF_BAR && Layout<0>::OFF_SW == OFF_SW, "single form keeps its layout");

#define QUAROT_TMEM_ST16(taddr, r)                                                                 \
  asm volatile(                                                                                    \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
      "%15,%16};" ::"r"(taddr),                                                                    \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),     \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) \
      : "memory")

// Half `part` of a packed row (its 16-byte chunks 2 part and 2 part + 1,
// 64B-swizzled source) -> 16 words of e4m3 bytes, the row's TMEM columns
// [16 part, 16 part + 16) in the K order of convert_row_regs; returns the byte
// sum of the offset codes.
__device__ __forceinline__ uint32_t convert_half_regs(const unsigned char* src_row, int r, int part, uint32_t* o) {
  uint4 w[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) w[c] = *reinterpret_cast<const uint4*>(src_row + (((2 * part + c) ^ ((r >> 1) & 3)) << 4));
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    unpack_word(w[c].x, o[8 * c + 0], o[8 * c + 1]);
    unpack_word(w[c].y, o[8 * c + 2], o[8 * c + 3]);
    unpack_word(w[c].z, o[8 * c + 4], o[8 * c + 5]);
    unpack_word(w[c].w, o[8 * c + 6], o[8 * c + 7]);
    acc = __dp4a((o[8 * c] + o[8 * c + 1]) + (o[8 * c + 2] + o[8 * c + 3]) + (o[8 * c + 4] + o[8 * c + 5]) +
                     (o[8 * c + 6] + o[8 * c + 7]),
                 0x01010101u, acc);
  }
  return acc;
}
// Half `part` of a packed row -> its 64 e4m3 bytes in the 128B-swizzled
// K-major destination row (the same layout as convert_row).
__device__ __forceinline__ uint32_t convert_half(const unsigned char* src_row, int r, int part, unsigned char* dst_row) {
  uint4 w[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) w[c] = *reinterpret_cast<const uint4*>(src_row + (((2 * part + c) ^ ((r >> 1) & 3)) << 4));
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int cc = 2 * part + c;
    uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
    unpack_word(w[c].x, l0, h0);
    unpack_word(w[c].y, l1, h1);
    unpack_word(w[c].z, l2, h2);
    unpack_word(w[c].w, l3, h3);
    acc = __dp4a((l0 + h0) + (l1 + h1) + (l2 + h2) + (l3 + h3), 0x01010101u, acc);
    *reinterpret_cast<uint4*>(dst_row + (((2 * cc) ^ (r & 7)) << 4)) = make_uint4(l0, h0, l1, h1);
    *reinterpret_cast<uint4*>(dst_row + (((2 * cc + 1) ^ (r & 7)) << 4)) = make_uint4(l2, h2, l3, h3);
  }
  return acc;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrival on a barrier of CTA `rank` that publishes generic-proxy shared-memory
// data written for that CTA (release at cluster scope: costs a cluster-wide
// fence of ~0.5 us on the issuing thread, so used once per tile only).
__device__ __forceinline__ void arrive_at(uint64_t* bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mapa(smem_u32(bar), rank))
               : "memory");
}
// Stage hand-off to the leader (release at CTA scope, no cluster-wide fence).
// What the leader's MMA reads was published before this arrival by the
// writers themselves: shared-memory operands by fence.proxy.async (visible to
// the tensor cores), tensor-memory operands by tcgen05.wait::st, and drained
// accumulator reads by tcgen05.wait::ld.
__device__ __forceinline__ void handoff_at(uint64_t* bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(mapa(smem_u32(bar), rank)) : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (QUAROT_ERR_TIMEOUT after
// kWaitLimitNs), for barriers that publish generic-proxy data written by the
// other CTA.  The acquire costs ~0.4 us per call, so it is used once per tile;
// the per-k-block stage barriers use CTA-scope waits.
__device__ __forceinline__ bool wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (try_wait_cluster(bar, parity, 20000u)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      record_error(QUAROT_ERR_TIMEOUT);
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}
// Warp-uniform forms for the single-issuer roles: the whole warp waits and
// loops (lane 0 issues), so no lane of these warps sits at the final CTA
// barrier while lane 0 is still working.  (With lane 0 alone in the loop, the
// converter warps sharing its scheduler woke ~1.3 us late from every barrier
// phase.)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort));
}
__device__ __forceinline__ bool warp_flag(volatile int* flag) {
  return __shfl_sync(0xffffffffu, *flag, 0) != 0;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 256-bit global store (one full 32-byte sector per thread; p 32-byte aligned)
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* o) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(o[0]), "r"(o[1]), "r"(o[2]),
               "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
               : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void commit2(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(uint16_t(3))
      : "memory");
}

// PRE: the code sums of the activation rows (sum_k a) and of the weight rows
// (sum_k w) are given, so the converters only unpack and the epilogue forms
// the offset corrections from them: -8 sum_k a for the row and
// -8 (sum_k w + 8 K) for the column (both exact in fp32), the same values the
// converters' sums give.
template <int V, bool PRE>
__global__ void __launch_bounds__(NTHREADS, 1)
w4a4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __half* __restrict__ sx, const __half* __restrict__ sw, int M, int N, int K, int BN,
                      __half* __restrict__ y, int32_t* __restrict__ acc_out, const int32_t* __restrict__ a_rowsum,
                      const int32_t* __restrict__ w_rowsum) {
  using L = Layout<V>;
  constexpr bool DBL = L::DBL;
  constexpr bool EARLY_PK = V != 2;
  // Converters wait for a free converted stage pair after loading and
  // unpacking the packed one, not before, where that was measured to pay:
  // with the row sums given (2048 x 4096 x 12288 70.5 -> 68.2 us,
  // 8192 x 4096 x 12288 306 -> 285 us) and in the four-stage layout (the
  // latter shape without row sums 347 -> 330 us); without the row sums the
  // one-accumulator and 160-wide forms ran ~5 % slower with it.
  constexpr bool LATE_EMPTY = PRE || V == 2;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  uint64_t* pk_full = bars;
  uint64_t* pk_empty = pk_full + SP;
  uint64_t* full = pk_empty + SP;
  uint64_t* empty = full + L::S;
  uint64_t* acc_full = empty + L::S;
  uint64_t* acc_empty = acc_full + L::NACC;
  uint64_t* rs_full = acc_empty + L::NACC;
  uint64_t* rs_empty = rs_full + 2;
  uint64_t* drain = rs_empty + 2;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::OFF_MISC + 4);
  int* rsA = reinterpret_cast<int*>(sm + L::OFF_RSA);
  float* rsB = reinterpret_cast<float*>(sm + L::OFF_RSB);
  float* swS = reinterpret_cast<float*>(sm + L::OFF_SW);
  float* rwS = reinterpret_cast<float*>(sm + L::OFF_RW);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair_id = int(blockIdx.x) >> 1, n_pairs = int(gridDim.x) >> 1;
  const int BNH = BN / 2;
  const int nkb = K / BK;
  const int n_tiles_n = (N + BN - 1) / BN;
  const int n_tiles = ((M + 2 * BM - 1) / (2 * BM)) * n_tiles_n;
  const uint32_t idesc = IDESC_BASE | (uint32_t(BN >> 3) << 17);

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < SP; ++s) {
      mbar_init(&pk_full[s], 1);
      mbar_init(&pk_empty[s], NCW);
    }
    // the leader's full barriers count its own converter warps plus the relay
    for (int s = 0; s < L::S; ++s) {
      mbar_init(&full[s], leader ? NCW + 1 : NCW);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < L::NACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], leader ? NEW + 1 : NEW);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&rs_full[s], 2 * NCW);   // every converter warp of the pair
      mbar_init(&rs_empty[s], 2 * NEW);  // every epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(const_cast<uint32_t*>(tmem_slot))),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival
  fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    long issued = 0, it = 0;
    const int b_bytes = BNH * BKB;
    for (int tile = pair_id; tile < n_tiles && !warp_flag(abort_flag); tile += n_pairs) {
      const int m0 = (tile / n_tiles_n) * 2 * BM + int(rank) * BM;
      const int n0 = (tile % n_tiles_n) * BN + int(rank) * BNH;
      // k-blocks in pairs: the converters release packed stages in pairs (the
      // second stage's phase completes after the first's), so one wait per
      // pair and both k-blocks' loads issued back to back
      for (int kb = 0; kb < nkb; kb += 2, it += 2) {
        const int s = int(it % SP);
        if (!warp_wait(&pk_empty[s], uint32_t((it / SP) & 1) ^ 1u, abort_flag)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&pk_full[s], 2 * (A_PK + b_bytes));
          tma_load_2d(smem_u32(sm + L::OFF_AP + s * A_PK), &tmA, kb * BKB, m0, &pk_full[s]);
          tma_load_2d(smem_u32(sm + L::OFF_BP + s * B_PK), &tmB, kb * BKB, n0, &pk_full[s]);
        }
        __syncwarp();
        issued = it + 2;
      }
    }
    if (warp_flag(abort_flag) && lane == 0) {
      for (long j = (issued > SP ? issued - SP : 0); j < issued; j += 2)
        mbar_wait_bounded(&pk_full[j % SP], uint32_t((j / SP) & 1), nullptr);
    }
  } else if (warp == 1) {
    if (leader) {
      // ---------------------------------------------------------- MMA issuer
      long it = 0;
      int ti = 0;
      for (int tile = pair_id; tile < n_tiles && !warp_flag(abort_flag); tile += n_pairs, ++ti) {
        // accumulator slot of this tile and how often the slot was used before
        const int sa = DBL ? (ti & 1) : 0;
        const uint32_t use = DBL ? uint32_t(ti >> 1) : uint32_t(ti);
        if (!warp_wait(&acc_empty[sa], (use & 1u) ^ 1u, abort_flag)) break;
        const uint32_t tmem_d = tmem_base + uint32_t(sa) * L::ACC_COLS;
        fence_after_sync();
        bool ok = true;
        // stages in pairs, as the converters complete them: each converter
        // warp and the relay arrive once per pair, on its second stage, after
        // their writes of both stages, so one wait covers both, and the eight
        // MMAs of the pair issue back to back
        for (int kb = 0; kb < nkb; kb += 2, it += 2) {
          const int s = int(it % L::S);
          if (!warp_wait(&full[s + 1], uint32_t((it / L::S) & 1), abort_flag)) {
            ok = false;
            break;
          }
          fence_after_sync();
          if (lane == 0) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t ta = tmem_base + L::A_COL + uint32_t(32 * (s + u));
              const uint64_t bd = sw128_desc(smem_u32(sm + L::OFF_BU + (s + u) * B_UN));
#pragma unroll
              for (int kk = 0; kk < BK / 32; ++kk)
                mma2_ts(tmem_d, ta + uint32_t(8 * kk), bd + uint64_t(2 * kk), idesc, ((kb + u) | kk) != 0);
            }
            // one commit frees the pair: it tracks every earlier MMA of this
            // thread, those of stage s included
            commit2(&empty[s + 1]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) commit2(&acc_full[sa]);
        __syncwarp();
      }
      if (lane == 0) {
        commit2(drain);
        mbar_wait_bounded(drain, 0, nullptr);
      }
    } else {
      // ---------------------------------------------------------- relay
      // forward this CTA's completed stages to the leader, in the order the
      // MMA issuer consumes them
      long it = 0;
      int ti = 0;
      bool ok = true;
      for (int tile = pair_id; ok && tile < n_tiles && !warp_flag(abort_flag); tile += n_pairs, ++ti) {
        for (int kb = 0; kb < nkb; kb += 2, it += 2) {
          const int s = int(it % L::S);
          if (!warp_wait(&full[s + 1], uint32_t((it / L::S) & 1), abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            handoff_at(&full[s + 1], 0);  // the issuer waits on the pair's second stage only
          }
          __syncwarp();
        }
        if (!ok) break;
        // forward this CTA's drain of a tile's accumulator to the leader.  With
        // two accumulators the drain of tile ti - 1 is forwarded after tile
        // ti's stages, so the relay never holds back the stages of the tile
        // that overlaps the drain; the leader needs it only before tile ti + 1.
        if (!DBL || ti >= 1) {
          const int pt = DBL ? ti - 1 : ti;
          const int pa = DBL ? (pt & 1) : 0;
          const uint32_t pu = DBL ? uint32_t(pt >> 1) : uint32_t(pt);
          if (!warp_wait(&acc_empty[pa], pu & 1u, abort_flag)) break;
          if (lane == 0) handoff_at(&acc_empty[pa], 0);
        }
        __syncwarp();
      }
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ converters
    // A: row 32 * (warp % 4) + lane (the warp's TMEM lane quadrant), half
    // (warp - 2) / 4; W: row 16 * (warp - 10) + lane % 16 of this CTA's half of
    // the weight rows, half lane / 16
    const bool is_a = warp < 2 + NAW;
    const int r = is_a ? 32 * (warp & 3) + lane : 16 * (warp - 2 - NAW) + (lane & 15);
    const uint32_t part = is_a ? uint32_t(warp - 2) >> 2 : uint32_t(lane) >> 4;
    const bool active = is_a || r < BNH;
    const uint32_t tmem_a_row = tmem_base + L::A_COL + (uint32_t(32 * (warp & 3)) << 16) + 16u * part;
    // 32-bit shared addresses, swizzled chunk offsets hoisted out of the loop:
    // the packed half row is 16-byte chunks 2 part and 2 part + 1 (64B swizzle),
    // the unpacked half row chunks 4 part .. 4 part + 3 (128B swizzle)
    const uint32_t swz_dst = uint32_t(r) & 7u;
    const uint32_t src_row = smem_u32(sm + (is_a ? L::OFF_AP : L::OFF_BP)) + uint32_t(r) * 128u;
    const uint32_t src0 = src_row + (((2u * part) ^ swz_dst) << 4), src1 = src_row + (((2u * part + 1u) ^ swz_dst) << 4);
    const uint32_t src2 = src_row + (((2u * part + 4u) ^ swz_dst) << 4), src3 = src_row + (((2u * part + 5u) ^ swz_dst) << 4);
    const uint32_t pk_stride = is_a ? uint32_t(A_PK) : uint32_t(B_PK);
    const uint32_t dst_row = smem_u32(sm + L::OFF_BU) + uint32_t(r) * 128u;
    const uint32_t d0 = ((4u * part) ^ swz_dst) << 4, d1 = ((4u * part + 1u) ^ swz_dst) << 4;
    const uint32_t d2 = ((4u * part + 2u) ^ swz_dst) << 4, d3 = ((4u * part + 3u) ^ swz_dst) << 4;
    // Each iteration converts two consecutive k-blocks (stages sp, sp + 1 and
    // ss, ss + 1: both rings have even sizes and the k-block count is even, so
    // a pair never straddles a wrap): twice the independent work per thread
    // and one set of waits, fences and arrivals per two k-blocks.
    uint32_t sp = 0, pk_par = 0, ss = 0, s_par = 0;  // ring positions and phase parities
    int ti = 0;
    for (int tile = pair_id; tile < n_tiles && !*abort_flag; tile += n_pairs, ++ti) {
      uint32_t sum = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; kb += 2) {
        if (!mbar_wait_bounded(&pk_full[sp], pk_par, abort_flag) ||
            (!LATE_EMPTY && !mbar_wait_bounded(&empty[ss + 1], s_par ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        uint32_t o[32];
        if (active) {
          const uint32_t pk = sp * pk_stride;
          const uint4 w0 = lds128(src0 + pk), w1 = lds128(src1 + pk);
          const uint4 w2 = lds128(src2 + pk), w3 = lds128(src3 + pk);
          unpack_word(w0.x, o[0], o[1]);
          unpack_word(w0.y, o[2], o[3]);
          unpack_word(w0.z, o[4], o[5]);
          unpack_word(w0.w, o[6], o[7]);
          unpack_word(w1.x, o[8], o[9]);
          unpack_word(w1.y, o[10], o[11]);
          unpack_word(w1.z, o[12], o[13]);
          unpack_word(w1.w, o[14], o[15]);
          unpack_word(w2.x, o[16], o[17]);
          unpack_word(w2.y, o[18], o[19]);
          unpack_word(w2.z, o[20], o[21]);
          unpack_word(w2.w, o[22], o[23]);
          unpack_word(w3.x, o[24], o[25]);
          unpack_word(w3.y, o[26], o[27]);
          unpack_word(w3.z, o[28], o[29]);
          unpack_word(w3.w, o[30], o[31]);
          // byte lanes of each 16-word sum stay below 16 * 15 = 240
          if constexpr (!PRE) {
            sum = __dp4a((((o[0] + o[1]) + (o[2] + o[3])) + ((o[4] + o[5]) + (o[6] + o[7]))) +
                             (((o[8] + o[9]) + (o[10] + o[11])) + ((o[12] + o[13]) + (o[14] + o[15]))),
                         0x01010101u, sum);
            sum = __dp4a((((o[16] + o[17]) + (o[18] + o[19])) + ((o[20] + o[21]) + (o[22] + o[23]))) +
                             (((o[24] + o[25]) + (o[26] + o[27])) + ((o[28] + o[29]) + (o[30] + o[31]))),
                         0x01010101u, sum);
          }
        }
        // the packed stage pair is in registers: hand it back to the producer
        // before the stores (not in the four-stage layout, whose converters
        // already run at most two pairs ahead; measured there 316.3 -> 318.8 us
        // at 8192 x 4096 x 12288, elsewhere 0.2-1.0 us faster)
        if constexpr (EARLY_PK) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&pk_empty[sp]);
        }
        // the converted stage pair is written once the MMAs have freed it
        // (empty[ss + 1] completes once the MMAs of both stages are done);
        // with LATE_EMPTY the loads and unpacking above overlap that wait
        if (LATE_EMPTY && !mbar_wait_bounded(&empty[ss + 1], s_par ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (active) {
          if (!is_a) {
            const uint32_t d = dst_row + ss * uint32_t(B_UN), e = d + uint32_t(B_UN);
            sts128(d + d0, o[0], o[1], o[2], o[3]);
            sts128(d + d1, o[4], o[5], o[6], o[7]);
            sts128(d + d2, o[8], o[9], o[10], o[11]);
            sts128(d + d3, o[12], o[13], o[14], o[15]);
            sts128(e + d0, o[16], o[17], o[18], o[19]);
            sts128(e + d1, o[20], o[21], o[22], o[23]);
            sts128(e + d2, o[24], o[25], o[26], o[27]);
            sts128(e + d3, o[28], o[29], o[30], o[31]);
          }
        }
        if (is_a) {
          QUAROT_TMEM_ST16(tmem_a_row + 32u * ss, o);
          QUAROT_TMEM_ST16(tmem_a_row + 32u * (ss + 1), (o + 16));
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          fence_before_sync();
        } else {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[ss + 1]);  // after the writes of both stages: covers the pair
          if constexpr (!EARLY_PK) mbar_arrive(&pk_empty[sp]);
        }
        sp += 2;
        if (sp == uint32_t(SP)) { sp = 0; pk_par ^= 1u; }
        ss += 2;
        if (ss == uint32_t(L::S)) { ss = 0; s_par ^= 1u; }
      }
      if (!ok) break;
      if constexpr (PRE) continue;  // the row sums are given
      const int a = ti & 1;
      if (!is_a) sum += __shfl_xor_sync(0xffffffffu, sum, 16);  // the row's other half
      if (!wait_cluster(&rs_empty[a], uint32_t((ti >> 1) & 1) ^ 1u, abort_flag)) break;
      if (is_a) {
        rsA[(2 * a + int(part)) * BM + r] = int(sum);
      } else if (part == 0 && r < BNH) {
        float* dst = rsB + a * BN_MAX + int(rank) * BNH + r;
        const float g = -8.0f * float(int(sum));  // exact: |8 sum| < 2^24
        *dst = g;
        st_cluster_s32(mapa(smem_u32(dst), rank ^ 1u), __float_as_int(g));
      }
      __syncwarp();
      if (lane == 0) {
        arrive_at(&rs_full[a], 0);
        arrive_at(&rs_full[a], 1);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - EPI_WARP0;  // 0..3
    const int q = warp & 3;          // TMEM lane quadrant of this warp
    const int r = 32 * q + lane;
    const int nchunks = BN / 32;
    const bool vec_ok = (N % 16) == 0 && (reinterpret_cast<uintptr_t>(y) & 31) == 0;
    int ti = 0;
    for (int tile = pair_id; tile < n_tiles && !*abort_flag; tile += n_pairs, ++ti) {
      const int a = ti & 1;
      const int m0 = (tile / n_tiles_n) * 2 * BM + int(rank) * BM, n0 = (tile % n_tiles_n) * BN;
      const int gm = m0 + r;
      // this warp's weight scales of the tile (warp-private, loaded before the
      // accumulator is ready; the warp's reads of the previous tile are done)
      float* sws_w = swS + e * BN_MAX;
      for (int c = 0; c < nchunks; ++c)
        sws_w[32 * c + lane] = n0 + 32 * c + lane < N ? __half2float(sw[n0 + 32 * c + lane]) : 0.f;
      const float sxr = gm < M ? __half2float(sx[gm]) : 0.f;
      float* rws_w = rwS + e * BN_MAX;  // PRE: -8 (sum_k w + 8 K) of the tile's columns
      float bias_r = 0.f;
      if constexpr (PRE) {
        for (int c = 0; c < nchunks; ++c) {
          const int n = n0 + 32 * c + lane;
          rws_w[32 * c + lane] = n < N ? -8.0f * float(w_rowsum[n] + 8 * K) : 0.f;
        }
        bias_r = gm < M ? -8.0f * float(a_rowsum[gm]) : 0.f;
      }
      __syncwarp();
      const int sa = DBL ? a : 0;
      const uint32_t use = DBL ? uint32_t(ti >> 1) : uint32_t(ti);
      if (!mbar_wait_bounded(&acc_full[sa], use & 1u, abort_flag) ||
          (!PRE && !wait_cluster(&rs_full[a], uint32_t((ti >> 1) & 1), abort_flag)))
        break;
      fence_after_sync();
      if constexpr (!PRE) bias_r = 64.0f * float(K) - 8.0f * float(rsA[2 * a * BM + r] + rsA[(2 * a + 1) * BM + r]);
      const float* rsb = PRE ? rws_w : rsB + a * BN_MAX;
      const uint32_t tmem_row = tmem_base + uint32_t(sa) * L::ACC_COLS + (uint32_t(32 * q) << 16);
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        const int c0 = 32 * c;
        const float* sws = sws_w + c0;  // sws[j]: scale of column n0 + c0 + j
        uint32_t v[32];
        __syncwarp();
        QUAROT_TMEM_LD32(tmem_row + uint32_t(c0), v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (c == nchunks - 1) {  // the accumulator is no longer needed by this warp
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[sa]);
        }
        const int gn = n0 + c0;
        if (gm < M && gn < N) {
          // exact integer accumulator, in place: acc = 2^18 * D - 8 * rowsum_w + bias_r
          const uint32_t rs_addr = smem_u32(rsb + c0), sw_addr = smem_u32(sws);
          // packed fp32x2 arithmetic: each lane of a pair rounds exactly as
          // the scalar fma + add would
          const float2 k18 = make_float2(262144.0f, 262144.0f), bias2 = make_float2(bias_r, bias_r);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const uint4 r4 = lds128(rs_addr + 4u * uint32_t(j));
            const float2 a01 = __fadd2_rn(__ffma2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), k18,
                                                     make_float2(__uint_as_float(r4.x), __uint_as_float(r4.y))), bias2);
            const float2 a23 = __fadd2_rn(__ffma2_rn(make_float2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])), k18,
                                                     make_float2(__uint_as_float(r4.z), __uint_as_float(r4.w))), bias2);
            v[j] = __float_as_uint(a01.x);
            v[j + 1] = __float_as_uint(a01.y);
            v[j + 2] = __float_as_uint(a23.x);
            v[j + 3] = __float_as_uint(a23.y);
          }
          __half* yrow = y + size_t(gm) * N + gn;
          if (vec_ok && gn + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j += 16) {
              uint32_t o[8];
#pragma unroll
              for (int t = 0; t < 8; t += 2) {
                const uint4 s4 = lds128(sw_addr + 4u * uint32_t(j + 2 * t));
                const float sv[4] = {__uint_as_float(s4.x), __uint_as_float(s4.y), __uint_as_float(s4.z),
                                     __uint_as_float(s4.w)};
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int jj = j + 2 * (t + u);
                  const float2 yv = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])),
                                                          make_float2(sxr, sxr)),
                                               make_float2(sv[2 * u], sv[2 * u + 1]));
                  const __half2 hv = __floats2half2_rn(yv.x, yv.y);
                  o[t + u] = *reinterpret_cast<const uint32_t*>(&hv);
                }
              }
              st_global_v8(yrow + j, o);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gn + j < N) yrow[j] = __float2half_rn(__fmul_rn(__fmul_rn(__uint_as_float(v[j]), sxr), sws[j]));
          }
          if (acc_out != nullptr) {
            int32_t* arow = acc_out + size_t(gm) * N + gn;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gn + j < N) arow[j] = __float2int_rn(__uint_as_float(v[j]));
          }
        }
      }
      __syncwarp();
      if (!PRE && lane == 0) {
        arrive_at(&rs_empty[a], 0);
        arrive_at(&rs_empty[a], 1);
      }
    }
  }

  fence_before_sync();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
  if (warp == 1) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}


// ===================================================================== A8 pair kernel
// The CTA-pair contraction with the activations already in tensor-core
// operand form (quarot_rotate_quant_a8): one byte per code, u = v + 8, in the
// K order the W converters produce, and each row's code sum sum_k v_k.  The A
// tile of a k-block (128 rows x 128 bytes per CTA) then needs no conversion:
// TMA writes it straight into a 128B-swizzled K-major stage that the MMA reads
// through a shared-memory descriptor.  Only the weights are converted (their
// nibbles stay packed in HBM, 4 bits per code), and tensor memory no longer
// holds A stages, so it holds two accumulators (columns [0, BN) and
// [256, 256 + BN)): the epilogue of tile i drains one while the MMAs of tile
// i + 1 fill the other.
//
//   warp 0          TMA producer of the packed W half rows (ring of SPW stages)
//   warp 1          TMEM allocator; MMA issuer in the leader, relay in the peer
//   warp 2          TMA producer of the A stages (ring of SA stages)
//   warps 3-10      W converters (packed -> e4m3 bytes -> shared memory)
//   warps 11-14     epilogue, one warp per TMEM lane quadrant
//
// Exact result: the MMA sums u_a u'_w 2^-18 (u'_w = w + 8, the weights'
// offset codes), so sum_k a_k w_k = 2^18 D - 8 sum_k u'_w - 8 sum_k a_k, the
// last term from the A row sums.
namespace a8 {

constexpr int SA = 6;             // operand stages: A bytes (TMA) + converted W half
constexpr int SPW = 4;            // packed W stages
constexpr int NBW8 = 8;           // W converter warps
constexpr int NEW8 = 4;           // epilogue warps
constexpr int CONV0 = 3;          // first converter warp
constexpr int EPI0 = CONV0 + NBW8;  // 11
constexpr int NT8 = 32 * (EPI0 + NEW8);  // 480
constexpr int A_UN = BM * BK;            // 16 KB
constexpr int W_PK = BNH_MAX * BKB;      // 7 KB
constexpr int W_UN = BNH_MAX * BK;       // 14 KB
constexpr int OFF_A = 0;
constexpr int OFF_WU = OFF_A + SA * A_UN;
constexpr int OFF_WP = OFF_WU + SA * W_UN;
constexpr int OFF_BAR8 = ((OFF_WP + SPW * W_PK) + 1023) / 1024 * 1024;
// barriers: pk_full[SPW] pk_empty[SPW] a_full[SA] full[SA] empty[SA]
//           acc_full[2] acc_empty[2] rs_full[2] rs_empty[2] drain
constexpr int NBAR8 = 2 * SPW + 3 * SA + 8 + 1;
constexpr int OFF_MISC8 = OFF_BAR8 + NBAR8 * 8;
constexpr int OFF_RSB8 = (OFF_MISC8 + 16 + 127) / 128 * 128;  // float [2][BN_MAX]: -8 x the tile's W row sums
constexpr int OFF_SW8 = OFF_RSB8 + 2 * BN_MAX * 4;            // float [NEW8][BN_MAX]: each epilogue warp's scales
constexpr int SMEM_BYTES8 = OFF_SW8 + NEW8 * BN_MAX * 4 + 1024;
constexpr uint32_t ACC_STRIDE = 256;  // tensor-memory columns between the two accumulators
static_assert(SMEM_BYTES8 <= 227 * 1024, "shared memory");
static_assert(SA % 2 == 0 && SPW % 2 == 0, "converters take stages in pairs");
static_assert(OFF_WU % 1024 == 0 && OFF_WP % 1024 == 0 && A_UN % 1024 == 0 && W_UN % 1024 == 0, "stage alignment");
static_assert(BN_MAX <= int(ACC_STRIDE) && 2 * ACC_STRIDE <= TMEM_COLS, "two accumulators in tensor memory");
static_assert(EPI0 % 4 == 3, "epilogue warps 11..14 cover the four TMEM lane quadrants");

__device__ __forceinline__ void mma2_ss(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__global__ void __launch_bounds__(NT8, 1)
w4a4_gemm_a8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __half* __restrict__ sx, const int32_t* __restrict__ rsx,
                         const __half* __restrict__ sw, int M, int N, int K, int BN, __half* __restrict__ y,
                         int32_t* __restrict__ acc_out) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR8);
  uint64_t* pk_full = bars;
  uint64_t* pk_empty = pk_full + SPW;
  uint64_t* a_full = pk_empty + SPW;
  uint64_t* full = a_full + SA;
  uint64_t* empty = full + SA;
  uint64_t* acc_full = empty + SA;  // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  uint64_t* rs_full = acc_empty + 2;   // [2]
  uint64_t* rs_empty = rs_full + 2;    // [2]
  uint64_t* drain = rs_empty + 2;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + OFF_MISC8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC8 + 4);
  float* rsB = reinterpret_cast<float*>(sm + OFF_RSB8);
  float* swS = reinterpret_cast<float*>(sm + OFF_SW8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair_id = int(blockIdx.x) >> 1, n_pairs = int(gridDim.x) >> 1;
  const int BNH = BN / 2;
  const int nkb = K / BK;
  const int n_tiles_n = (N + BN - 1) / BN;
  const int n_tiles = ((M + 2 * BM - 1) / (2 * BM)) * n_tiles_n;
  const uint32_t idesc = IDESC_BASE | (uint32_t(BN >> 3) << 17);

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int s = 0; s < SPW; ++s) {
      mbar_init(&pk_full[s], 1);
      mbar_init(&pk_empty[s], NBW8);
    }
    // the leader's full barriers count its own converter warps plus the relay
    for (int s = 0; s < SA; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&full[s], leader ? NBW8 + 1 : NBW8);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 2 * NEW8);  // every epilogue warp of the pair (used in the leader)
      mbar_init(&rs_full[s], 2 * NBW8);    // every converter warp of the pair
      mbar_init(&rs_empty[s], 2 * NEW8);   // every epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(const_cast<uint32_t*>(tmem_slot))),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival
  fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ W producer
    long issued = 0, it = 0;
    const int b_bytes = BNH * BKB;
    for (int tile = pair_id; tile < n_tiles && !warp_flag(abort_flag); tile += n_pairs) {
      const int n0 = (tile % n_tiles_n) * BN + int(rank) * BNH;
      for (int kb = 0; kb < nkb; kb += 2, it += 2) {
        // one 128-byte box per row covers k-blocks kb and kb + 1 (stages s, s + 1)
        const int s = int(it % SPW);
        if (!warp_wait(&pk_empty[s], uint32_t((it / SPW) & 1) ^ 1u, abort_flag)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&pk_full[s], 2 * b_bytes);
          tma_load_2d(smem_u32(sm + OFF_WP + s * W_PK), &tmB, kb * BKB, n0, &pk_full[s]);
        }
        __syncwarp();
        issued = it + 2;
      }
    }
    if (warp_flag(abort_flag) && lane == 0) {
      for (long j = (issued > SPW ? issued - SPW : 0); j < issued; j += 2)
        mbar_wait_bounded(&pk_full[j % SPW], uint32_t((j / SPW) & 1), nullptr);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ A producer
    long issued = 0, it = 0;
    for (int tile = pair_id; tile < n_tiles && !warp_flag(abort_flag); tile += n_pairs) {
      const int m0 = (tile / n_tiles_n) * 2 * BM + int(rank) * BM;
      // stage pairs, as the MMAs free them (the commit on the odd stage) and
      // behind one barrier (the odd stage's) for both k-blocks' loads
      for (int kb = 0; kb < nkb; kb += 2, it += 2) {
        const int s = int(it % SA);
        if (!warp_wait(&empty[s + 1], uint32_t((it / SA) & 1) ^ 1u, abort_flag)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&a_full[s + 1], 2 * A_UN);
          tma_load_2d(smem_u32(sm + OFF_A + s * A_UN), &tmA, kb * BK, m0, &a_full[s + 1]);
          tma_load_2d(smem_u32(sm + OFF_A + (s + 1) * A_UN), &tmA, (kb + 1) * BK, m0, &a_full[s + 1]);
        }
        __syncwarp();
        issued = it + 2;
      }
    }
    if (warp_flag(abort_flag) && lane == 0) {
      for (long j = (issued > SA ? issued - SA : 0); j < issued; j += 2)
        mbar_wait_bounded(&a_full[j % SA + 1], uint32_t((j / SA) & 1), nullptr);
    }
  } else if (warp == 1) {
    if (leader) {
      // ---------------------------------------------------------- MMA issuer
      long it = 0;
      int ti = 0;
      for (int tile = pair_id; tile < n_tiles && !warp_flag(abort_flag); tile += n_pairs, ++ti) {
        const int a = ti & 1;
        if (!warp_wait(&acc_empty[a], uint32_t((ti >> 1) & 1) ^ 1u, abort_flag)) break;
        fence_after_sync();
        const uint32_t tmem_d = tmem_base + uint32_t(a) * ACC_STRIDE;
        bool ok = true;
        // stages in pairs (the converters complete them in pairs; the pair's
        // two A loads complete one barrier)
        for (int kb = 0; kb < nkb; kb += 2, it += 2) {
          const int s = int(it % SA);
          const uint32_t par = uint32_t((it / SA) & 1);
          if (!warp_wait(&a_full[s + 1], par, abort_flag) || !warp_wait(&full[s + 1], par, abort_flag)) {
            ok = false;
            break;
          }
          fence_after_sync();
          if (lane == 0) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint64_t ad = sw128_desc(smem_u32(sm + OFF_A + (s + u) * A_UN));
              const uint64_t bd = sw128_desc(smem_u32(sm + OFF_WU + (s + u) * W_UN));
#pragma unroll
              for (int kk = 0; kk < BK / 32; ++kk)
                mma2_ss(tmem_d, ad + uint64_t(2 * kk), bd + uint64_t(2 * kk), idesc, ((kb + u) | kk) != 0);
            }
            // one commit frees the pair: it tracks every earlier MMA of this
            // thread, those of stage s included
            commit2(&empty[s + 1]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) commit2(&acc_full[a]);
        __syncwarp();
      }
      if (lane == 0) {
        commit2(drain);
        mbar_wait_bounded(drain, 0, nullptr);
      }
    } else {
      // ---------------------------------------------------------- relay
      // forward this CTA's completed stages (A landed, W converted) to the
      // leader, in the order the MMA issuer consumes them
      long it = 0;
      bool ok = true;
      for (int tile = pair_id; ok && tile < n_tiles && !warp_flag(abort_flag); tile += n_pairs) {
        for (int kb = 0; kb < nkb; kb += 2, it += 2) {
          const int s = int(it % SA);
          const uint32_t par = uint32_t((it / SA) & 1);
          if (!warp_wait(&a_full[s + 1], par, abort_flag) || !warp_wait(&full[s + 1], par, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            handoff_at(&full[s + 1], 0);  // the issuer waits on the pair's second stage only
          }
          __syncwarp();
        }
      }
    }
  } else if (warp < EPI0) {
    // ------------------------------------------------------------ W converters
    // row 16 * (warp - CONV0) + lane % 16 of this CTA's half of the weight
    // rows, half lane / 16 of it
    const int r = 16 * (warp - CONV0) + (lane & 15);
    const uint32_t part = uint32_t(lane) >> 4;
    const bool active = r < BNH;
    const uint32_t swz_dst = uint32_t(r) & 7u;
    // packed double stage: row r is 128 bytes (k-blocks kb, kb + 1), 128B swizzle
    const uint32_t src_row = smem_u32(sm + OFF_WP) + uint32_t(r) * 128u;
    const uint32_t src0 = src_row + (((2u * part) ^ swz_dst) << 4), src1 = src_row + (((2u * part + 1u) ^ swz_dst) << 4);
    const uint32_t src2 = src_row + (((2u * part + 4u) ^ swz_dst) << 4), src3 = src_row + (((2u * part + 5u) ^ swz_dst) << 4);
    const uint32_t dst_row = smem_u32(sm + OFF_WU) + uint32_t(r) * 128u;
    const uint32_t d0 = ((4u * part) ^ swz_dst) << 4, d1 = ((4u * part + 1u) ^ swz_dst) << 4;
    const uint32_t d2 = ((4u * part + 2u) ^ swz_dst) << 4, d3 = ((4u * part + 3u) ^ swz_dst) << 4;
    uint32_t sp = 0, pk_par = 0, ss = 0, s_par = 0;  // ring positions and phase parities
    int ti = 0;
    for (int tile = pair_id; tile < n_tiles && !*abort_flag; tile += n_pairs, ++ti) {
      uint32_t sum = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; kb += 2) {
        // empty[ss + 1] completes once the MMAs of both stages are done
        if (!mbar_wait_bounded(&pk_full[sp], pk_par, abort_flag) ||
            !mbar_wait_bounded(&empty[ss + 1], s_par ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (active) {
          uint32_t o[32];
          const uint32_t pk = sp * uint32_t(W_PK);
          const uint4 w0 = lds128(src0 + pk), w1 = lds128(src1 + pk);
          const uint4 w2 = lds128(src2 + pk), w3 = lds128(src3 + pk);
          unpack_word(w0.x, o[0], o[1]);
          unpack_word(w0.y, o[2], o[3]);
          unpack_word(w0.z, o[4], o[5]);
          unpack_word(w0.w, o[6], o[7]);
          unpack_word(w1.x, o[8], o[9]);
          unpack_word(w1.y, o[10], o[11]);
          unpack_word(w1.z, o[12], o[13]);
          unpack_word(w1.w, o[14], o[15]);
          unpack_word(w2.x, o[16], o[17]);
          unpack_word(w2.y, o[18], o[19]);
          unpack_word(w2.z, o[20], o[21]);
          unpack_word(w2.w, o[22], o[23]);
          unpack_word(w3.x, o[24], o[25]);
          unpack_word(w3.y, o[26], o[27]);
          unpack_word(w3.z, o[28], o[29]);
          unpack_word(w3.w, o[30], o[31]);
          // byte lanes of each 16-word sum stay below 16 * 15 = 240
          sum = __dp4a((((o[0] + o[1]) + (o[2] + o[3])) + ((o[4] + o[5]) + (o[6] + o[7]))) +
                           (((o[8] + o[9]) + (o[10] + o[11])) + ((o[12] + o[13]) + (o[14] + o[15]))),
                       0x01010101u, sum);
          sum = __dp4a((((o[16] + o[17]) + (o[18] + o[19])) + ((o[20] + o[21]) + (o[22] + o[23]))) +
                           (((o[24] + o[25]) + (o[26] + o[27])) + ((o[28] + o[29]) + (o[30] + o[31]))),
                       0x01010101u, sum);
          const uint32_t d = dst_row + ss * uint32_t(W_UN), e = d + uint32_t(W_UN);
          sts128(d + d0, o[0], o[1], o[2], o[3]);
          sts128(d + d1, o[4], o[5], o[6], o[7]);
          sts128(d + d2, o[8], o[9], o[10], o[11]);
          sts128(d + d3, o[12], o[13], o[14], o[15]);
          sts128(e + d0, o[16], o[17], o[18], o[19]);
          sts128(e + d1, o[20], o[21], o[22], o[23]);
          sts128(e + d2, o[24], o[25], o[26], o[27]);
          sts128(e + d3, o[28], o[29], o[30], o[31]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[ss + 1]);  // after the writes of both stages: covers the pair
          mbar_arrive(&pk_empty[sp]);
        }
        sp += 2;
        if (sp == uint32_t(SPW)) { sp = 0; pk_par ^= 1u; }
        ss += 2;
        if (ss == uint32_t(SA)) { ss = 0; s_par ^= 1u; }
      }
      if (!ok) break;
      const int a = ti & 1;
      sum += __shfl_xor_sync(0xffffffffu, sum, 16);  // the row's other half
      if (!wait_cluster(&rs_empty[a], uint32_t((ti >> 1) & 1) ^ 1u, abort_flag)) break;
      if (part == 0 && active) {
        float* dst = rsB + a * BN_MAX + int(rank) * BNH + r;
        const float g = -8.0f * float(int(sum));  // exact: |8 sum| < 2^24
        *dst = g;
        st_cluster_s32(mapa(smem_u32(dst), rank ^ 1u), __float_as_int(g));
      }
      __syncwarp();
      if (lane == 0) {
        arrive_at(&rs_full[a], 0);
        arrive_at(&rs_full[a], 1);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - EPI0;  // 0..3
    const int q = warp & 3;     // TMEM lane quadrant of this warp
    const int r = 32 * q + lane;
    const int nchunks = BN / 32;
    const bool vec_ok = (N % 16) == 0 && (reinterpret_cast<uintptr_t>(y) & 31) == 0;
    int ti = 0;
    for (int tile = pair_id; tile < n_tiles && !*abort_flag; tile += n_pairs, ++ti) {
      const int a = ti & 1;
      const int m0 = (tile / n_tiles_n) * 2 * BM + int(rank) * BM, n0 = (tile % n_tiles_n) * BN;
      const int gm = m0 + r;
      // this warp's weight scales of the tile (warp-private, loaded before the
      // accumulator is ready; the warp's reads of the previous tile are done)
      float* sws_w = swS + e * BN_MAX;
      for (int c = 0; c < nchunks; ++c)
        sws_w[32 * c + lane] = n0 + 32 * c + lane < N ? __half2float(sw[n0 + 32 * c + lane]) : 0.f;
      const float sxr = gm < M ? __half2float(sx[gm]) : 0.f;
      const float bias_r = gm < M ? -8.0f * float(rsx[gm]) : 0.f;  // exact: |8 sum| <= 2^22
      __syncwarp();
      if (!mbar_wait_bounded(&acc_full[a], uint32_t((ti >> 1) & 1), abort_flag) ||
          !wait_cluster(&rs_full[a], uint32_t((ti >> 1) & 1), abort_flag))
        break;
      fence_after_sync();
      const float* rsb = rsB + a * BN_MAX;
      const uint32_t tmem_row = tmem_base + uint32_t(a) * ACC_STRIDE + (uint32_t(32 * q) << 16);
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        const int c0 = 32 * c;
        const float* sws = sws_w + c0;  // sws[j]: scale of column n0 + c0 + j
        uint32_t v[32];
        __syncwarp();
        QUAROT_TMEM_LD32(tmem_row + uint32_t(c0), v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (c == nchunks - 1) {  // this warp no longer needs the accumulator
          fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(&acc_empty[a]);
            else handoff_at(&acc_empty[a], 0);
          }
        }
        const int gn = n0 + c0;
        if (gm < M && gn < N) {
          // exact integer accumulator, in place: acc = 2^18 D - 8 rowsum_w - 8 rowsum_a
          const uint32_t rs_addr = smem_u32(rsb + c0), sw_addr = smem_u32(sws);
          // packed fp32x2 arithmetic: each lane of a pair rounds exactly as
          // the scalar fma + add would
          const float2 k18 = make_float2(262144.0f, 262144.0f), bias2 = make_float2(bias_r, bias_r);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const uint4 r4 = lds128(rs_addr + 4u * uint32_t(j));
            const float2 a01 = __fadd2_rn(__ffma2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), k18,
                                                     make_float2(__uint_as_float(r4.x), __uint_as_float(r4.y))), bias2);
            const float2 a23 = __fadd2_rn(__ffma2_rn(make_float2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])), k18,
                                                     make_float2(__uint_as_float(r4.z), __uint_as_float(r4.w))), bias2);
            v[j] = __float_as_uint(a01.x);
            v[j + 1] = __float_as_uint(a01.y);
            v[j + 2] = __float_as_uint(a23.x);
            v[j + 3] = __float_as_uint(a23.y);
          }
          __half* yrow = y + size_t(gm) * N + gn;
          if (vec_ok && gn + 32 <= N) {
#pragma unroll
            for (int j = 0; j < 32; j += 16) {
              uint32_t o[8];
#pragma unroll
              for (int t = 0; t < 8; t += 2) {
                const uint4 s4 = lds128(sw_addr + 4u * uint32_t(j + 2 * t));
                const float sv[4] = {__uint_as_float(s4.x), __uint_as_float(s4.y), __uint_as_float(s4.z),
                                     __uint_as_float(s4.w)};
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int jj = j + 2 * (t + u);
                  const float2 yv = __fmul2_rn(__fmul2_rn(make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])),
                                                          make_float2(sxr, sxr)),
                                               make_float2(sv[2 * u], sv[2 * u + 1]));
                  const __half2 hv = __floats2half2_rn(yv.x, yv.y);
                  o[t + u] = *reinterpret_cast<const uint32_t*>(&hv);
                }
              }
              st_global_v8(yrow + j, o);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gn + j < N) yrow[j] = __float2half_rn(__fmul_rn(__fmul_rn(__uint_as_float(v[j]), sxr), sws[j]));
          }
          if (acc_out != nullptr) {
            int32_t* arow = acc_out + size_t(gm) * N + gn;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (gn + j < N) arow[j] = __float2int_rn(__uint_as_float(v[j]));
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        arrive_at(&rs_empty[a], 0);
        arrive_at(&rs_empty[a], 1);
      }
    }
  }

  fence_before_sync();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
  if (warp == 1) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace a8

}  // namespace pair

// ------------------------------------------------------------------ host
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static bool get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

static bool make_map(CUtensorMap* tm, const void* base, int64_t rows, int64_t K, int box_rows, bool two_kb = false) {
  cuuint64_t gdim[2] = {cuuint64_t(K / 2), cuuint64_t(rows)};
  cuuint64_t gstride[1] = {cuuint64_t(K / 2)};
  cuuint32_t box[2] = {cuuint32_t(two_kb ? 2 * BKB : BKB), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, two_kb ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activations in tensor-core operand form: [rows, K] bytes, 128-byte boxes
// (one k-block) in the 128B swizzle the MMA descriptor reads.
static bool make_map_a8(CUtensorMap* tm, const void* base, int64_t rows, int64_t K, int box_rows) {
  cuuint64_t gdim[2] = {cuuint64_t(K), cuuint64_t(rows)};
  cuuint64_t gstride[1] = {cuuint64_t(K)};
  cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile width for the N dimension: the candidate with the smallest per-SM
// makespan (tiles per SM x width), larger widths first on ties.
static int pick_bn(int64_t M, int64_t N, int sms) {
  const int cands[4] = {224, 192, 160, 128};
  int best = 224;
  int64_t best_cost = -1;
  const int64_t mt = (M + BM - 1) / BM;
  for (int bn : cands) {
    const int64_t tiles = mt * ((N + bn - 1) / bn);
    const int64_t cost = ((tiles + sms - 1) / sms) * bn;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// Pair kernel: the N-tile width and form with the smallest modelled time per
// pair.  The converters bound the pair and take about the same time per
// k-block at every width (~0.37-0.39 us on 152 SMs), so a tile costs its
// k-block count whatever its width.  With one accumulator every tile but the
// last also exposes its drain, which the next tile's MMAs must wait out
// (~2 us, about 5 k-blocks); two accumulators (widths up to 192, from three
// tiles per pair) hide it.  Ties go to the narrower tile, which gives each
// pair less work.  Fitted to the K = 4096 sweep and the 12288-deep shape:
// e.g. 8192 x 4096 x 4096 runs 112.3 us at 224 (8 tiles per pair, one
// accumulator), 122.3 at 192 and 130.4 at 160 (10 and 11 tiles, two).
// allow_dbl = false: a kernel with one accumulator only.
static void pick_pair_plan(int64_t M, int64_t N, int64_t K, int pairs, int* form, int* bn, bool allow_dbl = true) {
  constexpr int64_t kDrainKBlocks = 5;
  const int cands[4] = {128, 160, 192, 224};
  const int64_t mt = (M + 255) / 256, kb = K / BK;
  int64_t best_cost = -1;
  for (int w : cands) {
    const int64_t tiles = mt * ((N + w - 1) / w);
    const int64_t tpp = (tiles + pairs - 1) / pairs;
    const bool dbl = allow_dbl && w <= pair::Layout<2>::BN_LIMIT && tpp >= 3;
    const int64_t cost = tpp * kb + (dbl ? 0 : (tpp - 1) * kDrainKBlocks);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      *bn = w;
      *form = dbl ? 3 : 2;
    }
  }
}

// The launch plan of one GEMM on a GPU with `sms` SMs: for M > 128 with an
// even k-block count the CTA-pair kernel, else the one-SM kernel (form 1),
// and the N-tile width.  The pair kernel keeps one accumulator (form 2) or
// two (form 3), as pick_pair_plan models.
static void plan(int64_t M, int64_t N, int64_t K, int sms, int* form, int* bn) {
  if (M > BM && sms >= 2 && (K / BK) % 2 == 0) {
    pick_pair_plan(M, N, K, sms / 2, form, bn);
  } else {
    *form = 1;
    *bn = pick_bn(M, N, sms);
  }
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace gemm
}  // namespace quarot

using namespace quarot;

// Shared by quarot_w4a4_gemm (no row sums) and quarot_w4a4_gemm_rowsums
// (both code-sum vectors given: the CTA-pair forms skip the converters' sums).
static int w4a4_gemm_impl(const uint8_t* a_q, const void* a_scale, const int32_t* a_rowsum, const uint8_t* w_q,
                          const void* w_scale, const int32_t* w_rowsum, int64_t M, int64_t N, int64_t K, void* y,
                          int32_t* acc_out, void* stream) {
  using namespace quarot::gemm;
  if (M < 0 || N < 0 || K <= 0) return QUAROT_ERR_INVALID_ARG;
  if (K % BK != 0 || K > MAX_K) return QUAROT_ERR_UNSUPPORTED;
  if (M > (int64_t(1) << 31) - BM || N > (int64_t(1) << 31) - BN_MAX) return QUAROT_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return QUAROT_OK;
  if (!a_q || !a_scale || !w_q || !w_scale || !y) return QUAROT_ERR_INVALID_ARG;
  const bool pre = a_rowsum != nullptr && w_rowsum != nullptr;
  if ((reinterpret_cast<uintptr_t>(a_q) & 15) || (reinterpret_cast<uintptr_t>(w_q) & 15) ||
      (reinterpret_cast<uintptr_t>(a_scale) & 1) || (reinterpret_cast<uintptr_t>(w_scale) & 15) ||
      (reinterpret_cast<uintptr_t>(y) & 15) || (acc_out && (reinterpret_cast<uintptr_t>(acc_out) & 3)) ||
      (pre && ((reinterpret_cast<uintptr_t>(a_rowsum) & 3) || (reinterpret_cast<uintptr_t>(w_rowsum) & 3))))
    return QUAROT_ERR_ALIGNMENT;
  if (!get_encoder()) return QUAROT_ERR_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return QUAROT_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int form = 0, bn = 0;
  plan(M, N, K, sms, &form, &bn);
  if (form == 2 || form == 3) {
    // 2-SM path: clusters of two CTAs, one 256 x BN tile per pair (its
    // converters take k-blocks in pairs, so K % 256 == 0); form 3 keeps two
    // accumulators in tensor memory
    const int pairs = sms / 2;
    CUtensorMap ta, tb;
    if (!make_map(&ta, a_q, M, K, pair::BM, true) || !make_map(&tb, w_q, N, K, bn / 2, true)) return QUAROT_ERR_CUDA;
    // form 2: one accumulator; form 3: two, the width deciding the layout
    const int v = form == 2 ? 0 : (bn <= pair::Layout<1>::BN_LIMIT ? 1 : 2);
    using KernT = decltype(&pair::w4a4_gemm_pair_kernel<0, false>);
    const KernT kerns[3][2] = {{pair::w4a4_gemm_pair_kernel<0, false>, pair::w4a4_gemm_pair_kernel<0, true>},
                               {pair::w4a4_gemm_pair_kernel<1, false>, pair::w4a4_gemm_pair_kernel<1, true>},
                               {pair::w4a4_gemm_pair_kernel<2, false>, pair::w4a4_gemm_pair_kernel<2, true>}};
    const int smems[3] = {pair::Layout<0>::SMEM_BYTES, pair::Layout<1>::SMEM_BYTES, pair::Layout<2>::SMEM_BYTES};
    auto kern = kerns[v][pre ? 1 : 0];
    const int smem = smems[v];
    static quarot::AttrCache pattr[6];
    if (!smem_attr_once(kern, smem, pattr[2 * v + (pre ? 1 : 0)])) return QUAROT_ERR_LAUNCH;
    const int64_t tiles = ((M + 255) / 256) * ((N + bn - 1) / bn);
    const int64_t npairs = tiles < pairs ? tiles : pairs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * npairs));
    cfg.blockDim = dim3(pair::NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb,
                                             static_cast<const __half*>(a_scale), static_cast<const __half*>(w_scale),
                                             int(M), int(N), int(K), bn, static_cast<__half*>(y), acc_out,
                                             pre ? a_rowsum : nullptr, pre ? w_rowsum : nullptr);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? QUAROT_OK : QUAROT_ERR_LAUNCH;
  }
  CUtensorMap ta, tb;
  if (!make_map(&ta, a_q, M, K, BM) || !make_map(&tb, w_q, N, K, bn)) return QUAROT_ERR_CUDA;
  static quarot::AttrCache attr;
  if (!smem_attr_once(w4a4_gemm_kernel, SMEM_BYTES, attr)) return QUAROT_ERR_LAUNCH;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  const unsigned grid = unsigned(tiles < sms ? tiles : sms);
  w4a4_gemm_kernel<<<grid, NTHREADS, SMEM_BYTES, st>>>(
      ta, tb, static_cast<const __half*>(a_scale), static_cast<const __half*>(w_scale), int(M), int(N),
      int(K), bn, static_cast<__half*>(y), acc_out);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

extern "C" int quarot_w4a4_gemm(const uint8_t* a_q, const void* a_scale, const uint8_t* w_q,
                                const void* w_scale, int64_t M, int64_t N, int64_t K, void* y,
                                int32_t* acc_out, void* stream) {
  return w4a4_gemm_impl(a_q, a_scale, nullptr, w_q, w_scale, nullptr, M, N, K, y, acc_out, stream);
}

namespace quarot {
namespace gemm {
// Row code sums of a packed INT4 matrix (two's complement nibbles): one warp
// per row, 16 bytes (32 codes) per lane and step.  With u = v + 8 (the
// nibble with its sign bit flipped) the byte-wise sums of the low and high
// nibbles stay below 256, dp4a adds them, and sum v = sum u - 8 K.
__global__ void __launch_bounds__(256) int4_rowsum_kernel(const uint8_t* __restrict__ q, int64_t M, int64_t K,
                                                          int32_t* __restrict__ out) {
  const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const uint4* src = reinterpret_cast<const uint4*>(q + row * (K / 2));
  uint32_t acc = 0;
  for (int64_t c = lane; c < K / 32; c += 32) {
    const uint4 w = __ldg(src + c);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = ws[i] ^ 0x88888888u;
      acc = __dp4a((x & 0x0F0F0F0Fu) + ((x >> 4) & 0x0F0F0F0Fu), 0x01010101u, acc);
    }
  }
  acc = __reduce_add_sync(0xffffffffu, acc);
  if (lane == 0) out[row] = int32_t(int64_t(acc) - 8 * K);
}
}  // namespace gemm
}  // namespace quarot

extern "C" int quarot_int4_rowsum(const uint8_t* q, int64_t M, int64_t K, int32_t* rowsum_out, void* stream) {
  if (M < 0 || K <= 0 || K % 32 != 0 || K > (int64_t(1) << 24)) return QUAROT_ERR_INVALID_ARG;
  if (M == 0) return QUAROT_OK;
  if (q == nullptr || rowsum_out == nullptr) return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(rowsum_out) & 3))
    return QUAROT_ERR_ALIGNMENT;
  const int64_t blocks = (M + 7) / 8;
  if (blocks > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  quarot::gemm::int4_rowsum_kernel<<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(q, M, K,
                                                                                                   rowsum_out);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

extern "C" int quarot_w4a4_gemm_rowsums(const uint8_t* a_q, const void* a_scale, const int32_t* a_rowsum,
                                        const uint8_t* w_q, const void* w_scale, const int32_t* w_rowsum, int64_t M,
                                        int64_t N, int64_t K, void* y, int32_t* acc_out, void* stream) {
  if (M > 0 && N > 0 && (a_rowsum == nullptr || w_rowsum == nullptr)) return QUAROT_ERR_INVALID_ARG;
  return w4a4_gemm_impl(a_q, a_scale, a_rowsum, w_q, w_scale, w_rowsum, M, N, K, y, acc_out, stream);
}

extern "C" int quarot_w4a4_gemm_a8(const uint8_t* a8, const int32_t* a_rowsum, const void* a_scale,
                                   const uint8_t* w_q, const void* w_scale, int64_t M, int64_t N, int64_t K, void* y,
                                   int32_t* acc_out, void* stream) {
  using namespace quarot::gemm;
  if (M < 0 || N < 0 || K <= 0) return QUAROT_ERR_INVALID_ARG;
  if (K % (2 * BK) != 0 || K > MAX_K) return QUAROT_ERR_UNSUPPORTED;
  if (M > (int64_t(1) << 31) - 2 * BM || N > (int64_t(1) << 31) - BN_MAX) return QUAROT_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return QUAROT_OK;
  if (!a8 || !a_rowsum || !a_scale || !w_q || !w_scale || !y) return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a8) & 15) || (reinterpret_cast<uintptr_t>(w_q) & 15) ||
      (reinterpret_cast<uintptr_t>(a_rowsum) & 3) || (reinterpret_cast<uintptr_t>(a_scale) & 1) ||
      (reinterpret_cast<uintptr_t>(w_scale) & 15) || (reinterpret_cast<uintptr_t>(y) & 15) ||
      (acc_out && (reinterpret_cast<uintptr_t>(acc_out) & 3)))
    return QUAROT_ERR_ALIGNMENT;
  if (!get_encoder()) return QUAROT_ERR_CUDA;
  const int sms = sm_count();
  if (sms < 2) return sms <= 0 ? QUAROT_ERR_CUDA : QUAROT_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int pairs = sms / 2;
  int form_a8 = 0, bn = 0;
  pick_pair_plan(M, N, K, pairs, &form_a8, &bn, false);
  CUtensorMap ta, tb;
  if (!make_map_a8(&ta, a8, M, K, pair::BM) || !make_map(&tb, w_q, N, K, bn / 2, true)) return QUAROT_ERR_CUDA;
  static quarot::AttrCache attr8;
  if (!smem_attr_once(pair::a8::w4a4_gemm_a8_pair_kernel, pair::a8::SMEM_BYTES8, attr8)) return QUAROT_ERR_LAUNCH;
  const int64_t tiles = ((M + 255) / 256) * ((N + bn - 1) / bn);
  const int64_t npairs = tiles < pairs ? tiles : pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(2 * npairs));
  cfg.blockDim = dim3(pair::a8::NT8);
  cfg.dynamicSmemBytes = pair::a8::SMEM_BYTES8;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, pair::a8::w4a4_gemm_a8_pair_kernel, ta, tb,
                                           static_cast<const __half*>(a_scale), a_rowsum,
                                           static_cast<const __half*>(w_scale), int(M), int(N), int(K), bn,
                                           static_cast<__half*>(y), acc_out);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}

extern "C" int quarot_w4a4_gemm_plan(int64_t M, int64_t N, int64_t K, int sms, int* form, int* bn) {
  using namespace quarot::gemm;
  if (M <= 0 || N <= 0 || K <= 0 || sms <= 0 || form == nullptr || bn == nullptr) return QUAROT_ERR_INVALID_ARG;
  if (K % BK != 0 || K > MAX_K) return QUAROT_ERR_UNSUPPORTED;
  plan(M, N, K, sms, form, bn);
  return QUAROT_OK;
}
