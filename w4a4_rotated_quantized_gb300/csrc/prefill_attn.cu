// quarot_prefill_attn: the "Init" routine -- attention of a whole prompt over
// the INT4 KV cache, flash-attention style on the sm_103a tensor cores, with
// the keys and values dequantized as they are loaded.
//
// What it computes -- "QuaRot: Outlier-Free 4-Bit Inference in Rotated LLMs"
// (paper summary), "Kernel Implementation and Hardware Efficiency", quantized
// attention with KV cache, Init: during prefill every key and value is
// available at once, so they are dequantized and fed to a standard flash
// attention.  Stage 1d: the queries are rotated head-wise by H_d / sqrt(d)
// after RoPE, the keys in the cache carry the same rotation, so the scores are
// those of the unrotated attention.  For query token i of head h (KV head
// g = h / (Hq / Hkv)):
//   s_t = sm_scale * (q~_i . k^_t),  k^_t = k_s[t] * kcode_t,  t <= i (causal)
//   o_i = sum_t softmax(s)_t * v^_t, v^_t = v_s[t] * vcode_t   (rotated basis)
//
// Precision: the rotated query times sm_scale * log2(e) is split into fp16
// hi + lo halves, the keys enter the tensor cores as their exact integer codes
// and their scales multiply the fp32 scores, so the scores keep fp32-level
// precision; the dequantized values v^ = fp16(code * v_s) and the
// probabilities are fp16 (the pages' Init feeds fp16 dequantized values to
// flash attention); the products accumulate in fp32 in tensor memory.
//
// Design: one CTA per (128 query tokens, query head), 448 threads; with
// Hq / Hkv >= 2 the two query heads of a GQA group that read the same KV head
// run as a cluster of two CTAs (tcgen05 cta_group::2, M = 256): each CTA
// converts half of every key tile (64 keys) and half of every value tile (64
// dims), the two halves of the shared B operands, CTA 1 relays its operand
// barriers to CTA 0, and CTA 0 issues every MMA and multicasts completions.
// Per CTA, tensor
// memory (512 columns) holds the query halves (columns [0, 64) hi, [64, 128)
// lo, the A operand of S = Q K^T), two score buffers (columns 128 and 256) and
// the output O (columns 384 .. 511).  The tensor cores compute S(i+1) into one
// buffer while the softmax reads S(i) from the other; the fp16 probabilities
// P(i) overwrite the first 64 columns of their score buffer and are the A
// operand of O += P V (kind::f16, A from tensor memory).
//   warp 0      producer: the packed K/V codes of 128 keys by bulk copies,
//               their scales by plain loads, into a 4-stage ring
//   warp 1      tensor memory allocator and single-thread MMA issuer (in a
//               pair: CTA 0 issues, CTA 1 relays)
//   warps 2-5   converters: key codes -> exact fp16 codes, value codes ->
//               fp16 code * scale, in the 128-byte swizzled K-major layout
//               (keys row-wise; values transposed, the B operand of P V is
//               K-major along the keys); the key scales to fp32
//   warps 6-13  softmax, two warps per tensor memory lane quadrant: each
//               thread holds one half (64 scores) of its query row per key
//               tile (one tensor memory round trip), the pair exchanges row
//               maxima and sums through shared memory; the running max is
//               raised lazily (only when a tile exceeds it by more than 8 in
//               log2 units, so p < 2^8 stays in fp16 range), O rescaled in
//               tensor memory when it is; the warps also rotate the queries
// Every wait is bounded; an expired wait records QUAROT_ERR_TIMEOUT, the CTA
// drains its copies and MMAs, frees tensor memory and returns.
#include <math.h>

#include "common.cuh"

namespace quarot {
namespace prefill {

constexpr int HD = 128;    // head dim
constexpr int BQ = 128;    // query tokens per CTA (tensor memory lanes)
constexpr int BKV = 128;   // keys per tile
constexpr int SP = 4;      // packed stages
constexpr int SK = 2;      // converted key stages
constexpr int SV = 2;      // converted value stages
constexpr int NCW = 4;     // converter warps
constexpr int SM_W0 = 2 + NCW;
constexpr int TILE16 = 128 * HD * 2;                  // one 128 x 128 fp16 operand (two 16 KB swizzle atoms)
constexpr int PK_CODES = BKV * (HD / 2);              // 8 KB of codes per tensor
constexpr int PK_BYTES = 2 * PK_CODES + 2 * BKV * 2;  // K codes, V codes, K scales, V scales

constexpr int NSW = 8;     // softmax warps: two per tensor memory lane quadrant, one per half row
constexpr int NTHREADS = 32 * (SM_W0 + NSW);  // 448
// Shared memory of one CTA.  Converted stage s holds the keys at
// OFF_KV + 2 s STG and the values right after them.
//   single CTA: a stage is a whole 128 x 128 fp16 tile; before the first tile
//     the rotated queries are staged in fp32 in stage 1 (64 KB), which the
//     converters fill only after the queries have moved to tensor memory;
//   CTA pair (cta_group::2, M = 256): CTA r holds keys [64 r, 64 r + 64) of
//     each key tile and dims [64 r, 64 r + 64) of each value tile, the halves
//     of the B operands of S = Q K^T and O += P V; the query staging has its
//     own 64 KB.
template <bool PAIR>
struct Plan {
  static constexpr int ATOM = PAIR ? 8192 : 16384;  // 64 K-elements of every operand row, 128-byte swizzled
  static constexpr int STG = 2 * ATOM;              // one converted key or value stage
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_PK = OFF_KV + 2 * SK * STG;
  static constexpr int OFF_KSF = OFF_PK + SP * PK_BYTES;  // fp32 key scales [2][BKV], one per score buffer
  static constexpr int OFF_XCH = OFF_KSF + 2 * BKV * 4;    // fp32 [2 buffers][2 halves][BQ] row maxima, then [2 halves][BQ] row sums
  static constexpr int OFF_BAR = OFF_XCH + 3 * 2 * BQ * 4;
  // pk_full[SP] pk_empty[SP] k_full[SK] k_empty[SK] v_full[SV] v_empty[SV]
  // q_full s_full[2] p_full[2] ks_full[2] ks_empty[2] o_done drain xbar[4][2] lbar[4]
  static constexpr int NBAR = 2 * SP + 2 * SK + 2 * SV + 1 + 8 + 1 + 1 + 8 + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_QS = PAIR ? (OFF_MISC + 16 + 1023) / 1024 * 1024 : OFF_KV + 2 * STG;
  static constexpr int SMEM_BYTES = (PAIR ? OFF_QS + BQ * HD * 4 : OFF_MISC + 16) + 1024;  // + alignment slack
  static_assert(PAIR || (SK == SV && SK == 2 && BQ * HD * 4 == 2 * STG), "query staging fills stage 1");
  static_assert(OFF_PK % 16 == 0 && OFF_QS % 1024 == 0 && OFF_BAR % 8 == 0 && STG % 1024 == 0, "alignment");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_QHI = 0, COL_QLO = 64, COL_S = 128, COL_O = 384;  // S buffer b at COL_S + 128 b
// The queries are scaled by 2^8 before the hi/lo split (the lo halves stay in
// fp16's normal range); the key scales carry the 2^-8 back.
constexpr float QUP = 256.0f;

// kind::f16 instruction descriptor: D fp32, A and B fp16, both K-major,
// N = 128 (bits 17-22, N >> 3), M = 128 (bits 24-28, M >> 4).
constexpr uint32_t IDESC = (1u << 4) | (uint32_t(128 >> 3) << 17) | (uint32_t(128 >> 4) << 24);
// The same for a CTA pair: M = 256 (128 rows in each CTA's tensor memory).
constexpr uint32_t IDESC2 = (1u << 4) | (uint32_t(128 >> 3) << 17) | (uint32_t(256 >> 4) << 24);

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle
// layout: 128-byte rows, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFF) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(IDESC), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(IDESC), "r"(acc));
}
__device__ __forceinline__ void mma2_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(IDESC2), "r"(acc));
}
// Completion of the pair's MMAs, signalled on the barrier at this offset in both CTAs.
__device__ __forceinline__ void commit2(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(uint16_t(3))
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Arrival on the barrier at the same offset in CTA 0 of the pair (release at
// CTA scope: what the leader's MMAs read was published by its writers, shared
// memory by fence.proxy.async and tensor memory by tcgen05.wait::st).
__device__ __forceinline__ void handoff_to_leader(uint64_t* bar) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(smem_u32(bar)));
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t pack_f2h2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// INT4 codes are exact in fp16.  A nibble n holding v (two's complement)
// becomes 0x6400 | (n ^ 8) = 1024 + v + 8 (low nibble) or
// 0x6400 | ((n ^ 8) << 4) = 1024 + 16 (v + 8) (high nibble); one fused
// multiply-add per pair recovers v exactly.
// Byte p of w -> (code of its low nibble, code of its high nibble).
__device__ __forceinline__ uint32_t codes_of_byte(uint32_t w, int p) {
  const uint32_t x = prmt(w, 0u, uint32_t(p) | (4u << 4) | (uint32_t(p) << 8) | (4u << 12));
  return hfma2((x & 0x00F0000Fu) ^ 0x64806408u, 0x2C003C00u /* (1, 1/16) */, 0xD480E408u /* (-1032, -72) */);
}
// Byte p of wa and of wb -> (low nibble of a, low nibble of b) and (high of a, high of b).
__device__ __forceinline__ void codes_across(uint32_t wa, uint32_t wb, int p, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = prmt(wa, wb, uint32_t(p) | (uint32_t(p + 4) << 8));
  lo = hfma2((x & 0x000F000Fu) ^ 0x64086408u, 0x3C003C00u /* 1 */, 0xE408E408u /* -1032 */);
  hi = hfma2((x & 0x00F000F0u) ^ 0x64806480u, 0x2C002C00u /* 1/16 */, 0xD480D480u /* -72 */);
}

__device__ __forceinline__ bool warp_ok(bool ok) { return __all_sync(0xffffffffu, ok); }

template <bool PAIR>
__global__ void __launch_bounds__(NTHREADS, 1)
prefill_attn_kernel(const __half* __restrict__ q, const uint8_t* __restrict__ kq, const __half* __restrict__ ks,
                    const uint8_t* __restrict__ vq, const __half* __restrict__ vs, int B, int Hq, int Hkv, int T,
                    int T_max, float qscale, int causal, __half* __restrict__ out) {
  using PL = Plan<PAIR>;
  constexpr int OFF_KV = PL::OFF_KV, OFF_PK = PL::OFF_PK, OFF_QS = PL::OFF_QS, OFF_KSF = PL::OFF_KSF;
  constexpr int OFF_XCH = PL::OFF_XCH, OFF_BAR = PL::OFF_BAR, OFF_MISC = PL::OFF_MISC;
  constexpr int STG = PL::STG, ATOM = PL::ATOM;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* pk_full = bars;
  uint64_t* pk_empty = pk_full + SP;
  uint64_t* k_full = pk_empty + SP;
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* q_full = v_empty + SV;
  uint64_t* s_full = q_full + 1;     // [2] per score buffer
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* ks_full = p_full + 2;    // [2] key scales of the tile in score buffer b
  uint64_t* ks_empty = ks_full + 2;  // [2]
  uint64_t* o_done = ks_empty + 2;   // one phase per O += P V
  uint64_t* drain = o_done + 1;
  uint64_t* xbar = drain + 1;      // [4 quadrants][2 buffers]: the half-row pair's max exchange
  uint64_t* lbar = xbar + 8;       // [4 quadrants]: the pair's row-sum exchange
  float* ksf = reinterpret_cast<float*>(sm + OFF_KSF);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a pair serves two query heads of one GQA group (same KV head, same rows)
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int G = Hq / Hkv;
  const int n_qt = (T + BQ - 1) / BQ;
  const int unit = PAIR ? int(blockIdx.x) >> 1 : int(blockIdx.x);
  const int heads = PAIR ? Hq / 2 : Hq;  // head units per (prompt, query tile)
  const int per_qt = B * heads;
  const int qt = causal ? n_qt - 1 - unit / per_qt : unit / per_qt;  // longest rows first
  const int rem = unit % per_qt;
  const int h = PAIR ? 2 * (rem % heads) + int(rank) : rem % Hq, b = rem / heads;
  const int g = h / G;
  const int q0 = qt * BQ;
  const int nkt = causal ? qt + 1 : (T + BKV - 1) / BKV;
  const int64_t cache_row0 = (int64_t(b) * Hkv + g) * T_max;

  // The softmax threads load their half query row (64 fp16) first, so the
  // load latency overlaps the barrier and tensor-memory setup below.
  const bool is_sm = warp >= SM_W0;
  const int sm_r = 32 * (warp & 3) + lane, sm_hh = (warp - SM_W0) >> 2;
  const int sm_tok = q0 + sm_r;
  uint4 qraw[8];
  if (is_sm) {
    const uint4* src = reinterpret_cast<const uint4*>(q + ((int64_t(b) * T + sm_tok) * Hq + h) * HD + 64 * sm_hh);
#pragma unroll
    for (int m = 0; m < 8; ++m) qraw[m] = sm_tok < T ? __ldg(src + m) : make_uint4(0u, 0u, 0u, 0u);
  }

  if (threadIdx.x == 0) {
    // in the pair, the leader's operand barriers also count the peer's relay
    const int relay = (PAIR && leader) ? 1 : 0;
    for (int s = 0; s < SP; ++s) {
      mbar_init(&pk_full[s], 2);  // expect_tx arrival + the scales' arrival
      mbar_init(&pk_empty[s], NCW);
    }
    for (int s = 0; s < SK; ++s) {
      mbar_init(&k_full[s], NCW + relay);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&v_full[s], NCW + relay);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(q_full, NSW + relay);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], NSW + relay);
      mbar_init(&ks_full[s], NCW);
      mbar_init(&ks_empty[s], NSW);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    for (int k = 0; k < 8; ++k) mbar_init(&xbar[k], 2);
    for (int k = 0; k < 4; ++k) mbar_init(&lbar[k], 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(const_cast<uint32_t*>(tmem_slot))),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(const_cast<uint32_t*>(tmem_slot))),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote arrival
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    for (int i = 0; i < nkt; ++i) {
      const int sp = i % SP;
      if (!warp_ok(mbar_wait_bounded(&pk_empty[sp], uint32_t((i / SP) & 1) ^ 1u, abort_flag))) break;
      unsigned char* st = sm + OFF_PK + sp * PK_BYTES;
      const int t0 = i * BKV;
      const int nvalid = min(BKV, T - t0);
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&pk_full[sp], uint32_t(2 * nvalid * (HD / 2)));
        const uint8_t* ksrc = kq + (cache_row0 + t0) * (HD / 2);
        const uint8_t* vsrc = vq + (cache_row0 + t0) * (HD / 2);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_u32(st)),
                     "l"(ksrc), "r"(nvalid * (HD / 2)), "r"(smem_u32(&pk_full[sp]))
                     : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_u32(st + PK_CODES)),
                     "l"(vsrc), "r"(nvalid * (HD / 2)), "r"(smem_u32(&pk_full[sp]))
                     : "memory");
      }
      issued = i + 1;
      // scales of keys past T are zero, so their scores and values are zero
      __half* kss = reinterpret_cast<__half*>(st + 2 * PK_CODES);
      __half* vss = kss + BKV;
#pragma unroll
      for (int e = lane; e < BKV; e += 32) {
        const bool in = e < nvalid;
        kss[e] = in ? ks[cache_row0 + t0 + e] : __float2half(0.f);
        vss[e] = in ? vs[cache_row0 + t0 + e] : __float2half(0.f);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&pk_full[sp]);
    }
    if (*abort_flag && lane == 0) {
      for (int j = (issued > SP ? issued - SP : 0); j < issued; ++j)
        mbar_wait_bounded(&pk_full[j % SP], uint32_t((j / SP) & 1), nullptr);
    }
  } else if (warp == 1 && PAIR && !leader) {
    // ------------------------------------------------------------ relay (pair, CTA 1)
    // forward this CTA's completed operands to the leader's barriers, in the
    // order the leader's MMA issuer consumes them
    auto fwd = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (!warp_ok(mbar_wait_bounded(bar, parity, abort_flag))) return false;
      if (lane == 0) handoff_to_leader(bar);
      __syncwarp();
      return true;
    };
    bool ok = fwd(q_full, 0) && fwd(&k_full[0], 0);
    for (int i = 0; ok && i < nkt; ++i) {
      if (i + 1 < nkt) ok = fwd(&k_full[(i + 1) % SK], uint32_t(((i + 1) / SK) & 1));
      ok = ok && fwd(&v_full[i % SV], uint32_t((i / SV) & 1)) && fwd(&p_full[i & 1], uint32_t((i >> 1) & 1));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t kv_s = smem_u32(sm + OFF_KV);
      auto mma = [&](uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t acc) {
        if constexpr (PAIR) mma2_ts(d, a_tmem, bdesc, acc);
        else mma_ts(d, a_tmem, bdesc, acc);
      };
      auto done = [&](uint64_t* bar) {
        if constexpr (PAIR) commit2(bar);
        else commit(bar);
      };
      // S(i) into buffer i % 2: Q hi and Q lo (tensor memory) times the key codes
      auto issue_s = [&](int i) {
        const int kst = i % SK;
        const uint32_t d = tmem + COL_S + uint32_t(128 * (i & 1));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma(d, tmem + COL_QHI + uint32_t(8 * kk),
              sw128_desc(kv_s + uint32_t(2 * kst * STG + (kk >> 2) * ATOM + (kk & 3) * 32)), kk > 0);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          mma(d, tmem + COL_QLO + uint32_t(8 * kk),
              sw128_desc(kv_s + uint32_t(2 * kst * STG + (kk >> 2) * ATOM + (kk & 3) * 32)), 1u);
        done(&s_full[i & 1]);
        done(&k_empty[kst]);
      };
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag) && mbar_wait_bounded(&k_full[0], 0, abort_flag);
      if (ok) {
        fence_after();
        issue_s(0);
      }
      for (int i = 0; ok && i < nkt; ++i) {
        if (i + 1 < nkt) {
          // Buffer (i+1) % 2 holds P(i-1), the A operand of O += P(i-1) V.
          // The PTX ISA orders two tcgen05.mma of one thread only when they
          // share the accumulator and the shape; S(i+1) and O += P(i-1) V do
          // not, so S(i+1) waits for the commit of O += P(i-1) V (phase i-1
          // of o_done: the wait before S(i) made phase i-2 complete, so the
          // parity cannot alias an older phase).
          if (!mbar_wait_bounded(&k_full[(i + 1) % SK], uint32_t(((i + 1) / SK) & 1), abort_flag)) break;
          if (i > 0 && !mbar_wait_bounded(o_done, uint32_t((i - 1) & 1), abort_flag)) break;
          fence_after();
          issue_s(i + 1);
        }
        const int vst = i % SV;
        if (!mbar_wait_bounded(&v_full[vst], uint32_t((i / SV) & 1), abort_flag) ||
            !mbar_wait_bounded(&p_full[i & 1], uint32_t((i >> 1) & 1), abort_flag))
          break;
        fence_after();
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          mma(tmem + COL_O, tmem + COL_S + uint32_t(128 * (i & 1) + 8 * kk),
              sw128_desc(kv_s + uint32_t((2 * vst + 1) * STG + (kk >> 2) * ATOM + (kk & 3) * 32)),
              (i > 0 || kk > 0) ? 1u : 0u);
        done(o_done);
        done(&v_empty[vst]);
      }
      // every issued MMA completes before tensor memory is freed
      done(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else if (warp < SM_W0) {
    // ------------------------------------------------------------ converters
    const int cw = warp - 2;
    const int w = lane & 15, half = lane >> 4;
    for (int i = 0; i < nkt; ++i) {
      const int sp = i % SP, kst = i % SK, vst = i % SV;
      if (!warp_ok(mbar_wait_bounded(&pk_full[sp], uint32_t((i / SP) & 1), abort_flag))) break;
      if (!warp_ok(mbar_wait_bounded(&k_empty[kst], uint32_t((i / SK) & 1) ^ 1u, abort_flag))) break;
      // (single CTA) stage 1 held the queries
      if (!PAIR && i == 1 && !warp_ok(mbar_wait_bounded(q_full, 0, abort_flag))) break;
      const unsigned char* st = sm + OFF_PK + sp * PK_BYTES;
      const __half* kss = reinterpret_cast<const __half*>(st + 2 * PK_CODES);
      const uint32_t* vss2 = reinterpret_cast<const uint32_t*>(kss + BKV);  // value scales in pairs
      // keys: task (token t, word w) -> 16 bytes (dims 8w .. 8w+7) of row t,
      // exact codes; the lanes of one load cover 16 words x 2 tokens (all 32
      // banks), the 8 lanes of a quarter warp store 8 distinct 16-byte chunks.
      // Four words per step are loaded before any of their stores (the stores
      // may alias the loads as far as the compiler knows); the loop stays
      // rolled so the converters' code shares the instruction cache with the
      // softmax's.
      // (pair) this CTA's 64 keys start at key 64 r of the tile
      unsigned char* kdst = sm + OFF_KV + 2 * kst * STG;
      const unsigned char* ksrc = st + (PAIR ? 64 * int(rank) : 0) * (HD / 2);
#pragma unroll 1
      for (int it0 = 0; it0 < (PAIR ? BKV / 16 : BKV / 8); it0 += 4) {
        uint32_t words[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          words[u] = *reinterpret_cast<const uint32_t*>(ksrc + (2 * (cw + 4 * (it0 + u)) + half) * (HD / 2) + 4 * w);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = 2 * (cw + 4 * (it0 + u)) + half;
          *reinterpret_cast<uint4*>(kdst + (w >> 3) * ATOM + t * 128 + (((w & 7) ^ (t & 7)) << 4)) =
              make_uint4(codes_of_byte(words[u], 0), codes_of_byte(words[u], 1), codes_of_byte(words[u], 2),
                         codes_of_byte(words[u], 3));
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&k_full[kst]);
      // the key scales of tile i, for the softmax reading score buffer i % 2
      if (!warp_ok(mbar_wait_bounded(&ks_empty[i & 1], uint32_t((i >> 1) & 1) ^ 1u, abort_flag))) break;
      {
        const int t = 32 * cw + lane;
        ksf[(i & 1) * BKV + t] = __half2float(kss[t]) * (1.0f / QUP);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ks_full[i & 1]);

      if (!warp_ok(mbar_wait_bounded(&v_empty[vst], uint32_t((i / SV) & 1) ^ 1u, abort_flag))) break;
      // values, transposed: task (key chunk c of 8 tokens, word w) -> for each
      // of the 8 dims of word w, 16 bytes (the 8 tokens) of dim row 8w + e.
      // In one store the 8 lanes of a quarter warp hold 8 distinct chunks c.
      unsigned char* vdst = sm + OFF_KV + (2 * vst + 1) * STG;
      const unsigned char* vsrc = st + PK_CODES;
      // pair: 16 key chunks x this CTA's 8 words (dims 64 r .. 64 r + 63), one
      // task per thread; the 8 lanes of a quarter warp hold 8 distinct chunks
      const int wl = PAIR ? (lane & 7) : w;                  // word within this CTA's dims
      const int wsrc = PAIR ? 8 * int(rank) + wl : w;        // word within the packed row
#pragma unroll 1
      for (int pass = 0; pass < (PAIR ? 1 : 2); ++pass) {
        const int c = PAIR ? ((wl + cw + 4 * ((lane >> 3) & 1)) & 7) + 8 * (lane >> 4)
                           : ((w + cw + 4 * pass) & 7) + 8 * half;
        uint32_t W[8], s2[4];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
          W[jj] = *reinterpret_cast<const uint32_t*>(vsrc + (8 * c + jj) * (HD / 2) + 4 * wsrc);
#pragma unroll
        for (int u = 0; u < 4; ++u) s2[u] = vss2[4 * c + u];
        unsigned char* cbase = vdst + (c >> 3) * ATOM;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            codes_across(W[2 * u], W[2 * u + 1], p, lo[u], hi[u]);
            lo[u] = hmul2(lo[u], s2[u]);
            hi[u] = hmul2(hi[u], s2[u]);
          }
          const int n0 = 8 * wl + 2 * p, n1 = n0 + 1;
          *reinterpret_cast<uint4*>(cbase + n0 * 128 + (((c & 7) ^ (n0 & 7)) << 4)) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint4*>(cbase + n1 * 128 + (((c & 7) ^ (n1 & 7)) << 4)) =
              make_uint4(hi[0], hi[1], hi[2], hi[3]);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&v_full[vst]);
        mbar_arrive(&pk_empty[sp]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Two warps per tensor memory lane quadrant: warp v (0..7) serves rows
    // 32 qd .. 32 qd + 31 and columns 64 hh .. 64 hh + 63 of every tile; the
    // pair exchanges row maxima (per tile) and row sums (at the end) through
    // shared memory behind an mbarrier of the pair (bounded waits, so a pair
    // in which one warp gave up cannot hang the other).
    const int v8 = warp - SM_W0;
    const int qd = warp & 3;
    const int hh = v8 >> 2;
    float* xch = reinterpret_cast<float*>(sm + OFF_XCH);
    // publish this warp's values (written before the call), wait for the partner's
    auto pair_exchange = [&](uint64_t* bar, uint32_t parity) -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
      return warp_ok(mbar_wait_bounded(bar, parity, abort_flag));
    };
    // ---- q~ = q H / sqrt(d) (1/sqrt(d) rides in qsc): this thread's half row.
    // Natural-order FWHT, lower index a + b, upper a - b: spans 1 .. 32 in
    // registers, span 64 with the partner thread (same lane, other half)
    // through the fp32 staging area; a half row sits at [r][64 hh ..] in
    // 16-byte chunks, chunk m at m ^ (lane & 7).
    const int r = sm_r;
    const int tok = sm_tok;
    float* qs = reinterpret_cast<float*>(sm + OFF_QS);
    float x[64];
    {
      // xp[n] = elements (2n, 2n + 1): span 1 inside a pair, spans 2 .. 32
      // across pairs with packed fp32x2 add / subtract (same roundings as the
      // scalar butterflies: lower a + b, upper a - b)
      float2 xp[32];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t w4[4] = {qraw[m].x, qraw[m].y, qraw[m].z, qraw[m].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = h2_to_f2(w4[k]);
          xp[4 * m + k] = make_float2(f.x + f.y, f.x - f.y);
        }
      }
#pragma unroll
      for (int s = 1; s < 32; s <<= 1)
#pragma unroll
        for (int n = 0; n < 32; ++n)
          if ((n & s) == 0) {
            const float2 u0 = xp[n], u1 = xp[n + s];
            xp[n] = __fadd2_rn(u0, u1);
            xp[n + s] = __fadd2_rn(u0, make_float2(-u1.x, -u1.y));
          }
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        x[2 * n] = xp[n].x;
        x[2 * n + 1] = xp[n].y;
      }
    }
    float* my = qs + r * HD + 64 * hh;
#pragma unroll
    for (int m = 0; m < 16; ++m)
      *reinterpret_cast<float4*>(my + 4 * (m ^ (lane & 7))) = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
    asm volatile("bar.sync 5, %0;" ::"r"(32 * NSW) : "memory");  // both halves of every row are staged
    // ---- span 64 (both halves re-read from the staging area), then fp16 hi
    // and lo halves of q~ * scale -> tensor memory
    const float* other = qs + r * HD + 64 * (1 - hh);
    const uint32_t lane_off = uint32_t(32 * qd) << 16;
    const float qsc = qscale * QUP;
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      const int c = 2 * hh + c2;  // 32-dim chunk of the row
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int mm = 8 * c2 + m;  // 16-byte chunk within the half
        const float4 a4 = *reinterpret_cast<const float4*>(my + 4 * (mm ^ (lane & 7)));
        const float4 y4 = *reinterpret_cast<const float4*>(other + 4 * (mm ^ (lane & 7)));
        const float xa[4] = {a4.x, a4.y, a4.z, a4.w}, y[4] = {y4.x, y4.y, y4.z, y4.w};
        float xs[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) xs[e2] = (hh == 0 ? xa[e2] + y[e2] : y[e2] - xa[e2]) * qsc;
        float hv[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) hv[e2] = __half2float(__float2half_rn(xs[e2]));
        hi[2 * m] = pack_f2h2(hv[0], hv[1]);
        hi[2 * m + 1] = pack_f2h2(hv[2], hv[3]);
        lo[2 * m] = pack_f2h2(xs[0] - hv[0], xs[1] - hv[1]);
        lo[2 * m + 1] = pack_f2h2(xs[2] - hv[2], xs[3] - hv[3]);
      }
      tmem_st16(tmem + lane_off + COL_QHI + uint32_t(16 * c), hi);
      tmem_st16(tmem + lane_off + COL_QLO + uint32_t(16 * c), lo);
    }
    wait_st();
    fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);

    float m_run = -INFINITY, l_run = 0.f;  // l_run: this half's sum
    bool ok = true;
    for (int i = 0; i < nkt; ++i) {
      const int sb = i & 1;
      const uint32_t par = uint32_t((i >> 1) & 1);
      if (!warp_ok(mbar_wait_bounded(&s_full[sb], par, abort_flag) &&
                   mbar_wait_bounded(&ks_full[sb], par, abort_flag))) {
        ok = false;
        break;
      }
      fence_after();
      const uint32_t s_t = tmem + lane_off + COL_S + uint32_t(128 * sb);
      uint32_t v[64];
      tmem_ld32(s_t + uint32_t(64 * hh), v);
      tmem_ld32(s_t + uint32_t(64 * hh + 32), v + 32);
      wait_ld();
      // scores in log2 units: the fp32 product times the key's scale
      const uint32_t kf_s = smem_u32(ksf + sb * BKV + 64 * hh);
#pragma unroll
      for (int e8 = 0; e8 < 8; ++e8) {
        float kk[8];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(kk[4 * j]), "=f"(kk[4 * j + 1]), "=f"(kk[4 * j + 2]), "=f"(kk[4 * j + 3])
                       : "r"(kf_s + 32u * e8 + 16u * j));
#pragma unroll
        for (int u = 0; u < 8; u += 2) {
          const float2 sc = __fmul2_rn(make_float2(__uint_as_float(v[8 * e8 + u]), __uint_as_float(v[8 * e8 + u + 1])),
                                       make_float2(kk[u], kk[u + 1]));
          v[8 * e8 + u] = __float_as_uint(sc.x);
          v[8 * e8 + u + 1] = __float_as_uint(sc.y);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ks_empty[sb]);
      if (i == nkt - 1) {
        // the diagonal (causal) or ragged last tile: columns past this row's
        // last key are -inf
        const int lim = (causal ? min(tok, T - 1) - i * BKV : T - 1 - i * BKV) - 64 * hh;
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e > lim) v[e] = __float_as_uint(-INFINITY);
      }
      float mp[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mp[j] = __uint_as_float(v[j]);
#pragma unroll
      for (int e = 8; e < 64; e += 16)
#pragma unroll
        for (int j = 0; j < 8; ++j) mp[j] = max3f(mp[j], __uint_as_float(v[e + j]), __uint_as_float(v[e + 8 + j]));
      float mx = max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
      // the row max over both halves; after the barrier both halves' scores
      // are in registers, so the probabilities may overwrite the score columns
      xch[(sb * 2 + hh) * BQ + r] = mx;
      if (!pair_exchange(&xbar[qd * 2 + sb], par)) {
        ok = false;
        break;
      }
      mx = fmaxf(xch[(sb * 2) * BQ + r], xch[(sb * 2 + 1) * BQ + r]);
      // ---- lazy rescale: raise the running max only when the tile exceeds
      // it by more than 8 (log2 units); otherwise p <= 2^8
      const bool raise = mx > m_run + 8.0f;
      float alpha = 1.f;
      if (raise) {
        alpha = ex2(m_run - mx);  // 0 while m_run is -inf
        l_run *= alpha;
        m_run = mx;
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      // ---- p = 2^(s - m) -> fp16 pairs into columns [32 hh, 32 hh + 32) of the buffer
      // packed f32x2 subtract and sums: one instruction per two scores
      const float2 m_neg = make_float2(-m_use, -m_use);
      float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        const float2 d = __fadd2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), m_neg);
        const float p0 = ex2(d.x), p1 = ex2(d.y);
        ls[(e >> 1) & 1] = __fadd2_rn(ls[(e >> 1) & 1], make_float2(p0, p1));
        v[e >> 1] = pack_f2h2(p0, p1);
      }
      l_run += (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
      tmem_st32(s_t + uint32_t(32 * hh), v);
      if (i > 0 && __any_sync(0xffffffffu, raise)) {
        // O += P(i-1) V may still run: wait for it, then rescale this half of O
        // in place (before O += P(i) V, which the arrival below releases)
        if (!warp_ok(mbar_wait_bounded(o_done, uint32_t((i - 1) & 1), abort_flag))) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t o_t = tmem + lane_off + COL_O + uint32_t(64 * hh);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(o_t + uint32_t(32 * c), o);
          wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(o_t + uint32_t(32 * c), o);
        }
      }
      wait_st();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    // the row sum over both halves (own slots: the partner may still read
    // the last tile's maxima)
    float* xl = xch + 4 * BQ;
    xl[hh * BQ + r] = l_run;
    ok = ok && pair_exchange(&lbar[qd], 0);
    const float l_tot = xl[r] + xl[BQ + r];
    // The last O += P V is complete when the issuer's final commit (drain,
    // one phase per launch) is.  A parity wait on o_done could not tell: the
    // last score buffer this warp waited for was issued before O += P(nkt-2) V,
    // so o_done may still be two phases short, and its parity then reads as
    // phase nkt-1 complete.
    if (ok && warp_ok(mbar_wait_bounded(drain, 0u, abort_flag))) {
      fence_after();
      const float inv_l = 1.0f / l_tot;
      const uint32_t o_t = tmem + lane_off + COL_O + uint32_t(64 * hh);
      __half* orow = out + ((int64_t(b) * T + tok) * Hq + h) * HD + 64 * hh;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(o_t + uint32_t(32 * c), o);
        wait_ld();
        if (tok < T) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 u;
            u.x = pack_f2h2(__uint_as_float(o[e]) * inv_l, __uint_as_float(o[e + 1]) * inv_l);
            u.y = pack_f2h2(__uint_as_float(o[e + 2]) * inv_l, __uint_as_float(o[e + 3]) * inv_l);
            u.z = pack_f2h2(__uint_as_float(o[e + 4]) * inv_l, __uint_as_float(o[e + 5]) * inv_l);
            u.w = pack_f2h2(__uint_as_float(o[e + 6]) * inv_l, __uint_as_float(o[e + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + 32 * c + e) = u;
          }
        }
      }
    }
  }

  fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // no CTA leaves while its peer may still touch its memory
  if (warp == 1) {
    fence_after();
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

}  // namespace prefill
}  // namespace quarot

extern "C" int quarot_prefill_attn(const void* q, const uint8_t* k_q, const void* k_s, const uint8_t* v_q,
                                   const void* v_s, int64_t B, int64_t Hq, int64_t Hkv, int64_t d, int64_t T,
                                   int64_t T_max, float sm_scale, int causal, void* out, void* stream) {
  using namespace quarot::prefill;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || T < 0 || T_max < T || (Hq % Hkv) != 0) return QUAROT_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return QUAROT_ERR_INVALID_ARG;
  if (d != HD) return QUAROT_ERR_UNSUPPORTED;
  const int64_t G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return QUAROT_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return QUAROT_OK;
  if (B > 65535 || Hq > 1024 || T > (1 << 24) || T_max > (int64_t(1) << 30)) return QUAROT_ERR_UNSUPPORTED;
  if (q == nullptr || k_q == nullptr || k_s == nullptr || v_q == nullptr || v_s == nullptr || out == nullptr)
    return QUAROT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(k_q) & 15) ||
      (reinterpret_cast<uintptr_t>(v_q) & 15) || (reinterpret_cast<uintptr_t>(k_s) & 1) ||
      (reinterpret_cast<uintptr_t>(v_s) & 1) || (reinterpret_cast<uintptr_t>(out) & 15))
    return QUAROT_ERR_ALIGNMENT;
  const int64_t grid = ((T + BQ - 1) / BQ) * B * Hq;
  if (grid > 0x7fffffff) return QUAROT_ERR_UNSUPPORTED;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(float(HD));
  // q~ carries 1/sqrt(d) of the rotation, the softmax scale and log2(e)
  const float qscale = scale * 1.4426950408889634f / sqrtf(float(HD));
  const __half* qh = static_cast<const __half*>(q);
  const __half* ksh = static_cast<const __half*>(k_s);
  const __half* vsh = static_cast<const __half*>(v_s);
  __half* oh = static_cast<__half*>(out);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (G >= 2) {
    // CTA pairs: two query heads of a GQA group share each converted tile
    static quarot::AttrCache attr2;
    if (!quarot::smem_attr_once(prefill_attn_kernel<true>, Plan<true>::SMEM_BYTES, attr2)) return QUAROT_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));  // Hq is even (G >= 2): whole pairs
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = Plan<true>::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_attn_kernel<true>, qh, k_q, ksh, v_q, vsh, int(B),
                                             int(Hq), int(Hkv), int(T), int(T_max), qscale, causal, oh);
    return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? QUAROT_OK : QUAROT_ERR_LAUNCH;
  }
  static quarot::AttrCache attr1;
  if (!quarot::smem_attr_once(prefill_attn_kernel<false>, Plan<false>::SMEM_BYTES, attr1)) return QUAROT_ERR_LAUNCH;
  prefill_attn_kernel<false><<<dim3(unsigned(grid)), dim3(NTHREADS), Plan<false>::SMEM_BYTES, st>>>(
      qh, k_q, ksh, v_q, vsh, int(B), int(Hq), int(Hkv), int(T), int(T_max), qscale, causal, oh);
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}
