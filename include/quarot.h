/*
 * quarot.h -- C ABI of libquarot.so, the GB300 (sm_103a) hot path of QuaRot:
 * online randomized Hadamard rotation fused with per-token INT4 quantization,
 * a W4A4 GEMM with a scale-dequant epilogue, and the rotated INT4 KV cache
 * (append + one-token decode attention).
 *
 * Sources (page title, section):
 *   [S] "QuaRot: Outlier-Free 4-Bit Inference in Rotated LLMs" (paper summary),
 *       section 3 "Technical Approach" (Stages 1a-1d, 2a-2c, "Kernel
 *       Implementation and Hardware Efficiency").
 *   [G] "QuaRot Guide: Outlier-Free 4-Bit W4A4 LLM Quantization" (blog),
 *       sections on the RHT, the INT4 grid and the 4-bit rotated KV cache.
 *   [E] QuaRot paper-viz explainer: Sylvester for 2^n, Kronecker with a
 *       Paley-12 block for 12288.
 *
 * Conventions for every entry point:
 *   - Pointers to tensors are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them.  fp16 data is passed as void*
 *     (IEEE binary16).  All tensors are dense row-major (C order) unless a
 *     leading dimension is given.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream.
 *   - Arguments are validated on the host before any launch; a rejected call
 *     launches nothing and returns a nonzero status.  No exception crosses
 *     the ABI.
 *   - Kernels that wait on hardware barriers give up after a bounded time,
 *     record QUAROT_ERR_TIMEOUT in a device error word and return;
 *     quarot_check_error() reads (and clears) that word.
 *   - INT4 codes are two's complement in [-8, 7], two per byte, the even
 *     index in the low nibble.
 */
#ifndef QUAROT_H_
#define QUAROT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  QUAROT_OK = 0,
  QUAROT_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size */
  QUAROT_ERR_UNSUPPORTED = 2, /* size outside what the kernels implement     */
  QUAROT_ERR_ALIGNMENT = 3,   /* pointer or leading dimension misaligned      */
  QUAROT_ERR_LAUNCH = 4,      /* the CUDA launch itself failed                */
  QUAROT_ERR_TIMEOUT = 5,     /* a device-side bounded wait expired           */
  QUAROT_ERR_CUDA = 6         /* another CUDA runtime/driver error            */
};

/* Human-readable text for a status code (static storage, never NULL). */
const char* quarot_status_string(int status);

/* ABI version: (major << 16) | minor.  1.1 adds, with every 1.0 entry point
 * unchanged: quarot_w4a4_gemm_plan, quarot_legacy_imma_probe,
 * quarot_rotate_quant_a8, quarot_w4a4_gemm_a8, quarot_rotate_quant_rowsum,
 * quarot_int4_rowsum and quarot_w4a4_gemm_rowsums. */
int quarot_version(void);

/* Synchronizes `stream`, then returns and clears the device error word of the
 * current device (QUAROT_OK if no kernel recorded an error), or
 * QUAROT_ERR_CUDA if the synchronization itself failed. */
int quarot_check_error(void* stream);

/* Self-test of the bounded wait every kernel relies on: one device thread
 * waits on a hardware barrier that nothing completes, gives up after the
 * library's wait limit (one second), records QUAROT_ERR_TIMEOUT in the
 * device error word and returns.  The call itself returns QUAROT_OK (or
 * QUAROT_ERR_LAUNCH); the next quarot_check_error() on `stream` returns
 * QUAROT_ERR_TIMEOUT and clears the word; the context stays usable. */
int quarot_selftest_wait(void* stream);

/*
 * quarot_rotate_quant -- online randomized Hadamard rotation of each row
 * followed by per-token symmetric INT4 quantization and packing.
 * [S] Stage 1a (Q = H diag(s), Kronecker sizes), Stage 1b (online FWHT in
 * FP32), Stage 2b (per-token scale, clipping ratio), "Kernel Implementation"
 * (quantize, pack two INT4 per byte); [G] RHT and quantizer formulas.
 *
 * For each row i of x:
 *   r = (x_i * s) @ H_d / sqrt(d)          (fp32; s = 1 if signs == NULL)
 *   S = fp16(min(max(clip_ratio * max_j |r_j|, 1e-5) / 7, 65504))
 *   q_j = clamp(round_half_even(r_j / S), -8, 7), packed two per byte.
 * H_d is Sylvester for d = 2^n, and H12 (x) H_{d/12} (Paley I, q = 11) for
 * d = 12 * 2^n (row-vector convention, column index c * (d/12) + e).
 * The same call quantizes weight rows offline (per-output-channel RTN).
 *
 *   x         fp16 [M, ld_x], first d columns used (ld_x >= d, ld_x % 8 == 0,
 *             x 16-byte aligned)
 *   M         rows (>= 0; M == 0 is a no-op)
 *   d         row width: 2^n with 16 <= d <= 8192, or 12 * 2^n with
 *             3072 <= d <= 12288
 *   signs     int8 [d] of +1/-1 (read only), or NULL
 *   clip_ratio  in (0, 1]
 *   q_out     uint8 [M, d/2], 16-byte aligned
 *   scale_out fp16 [M]
 *   rot_out   fp32 [M, d] (the rotated values r, for testing), or NULL
 */
int quarot_rotate_quant(const void* x, int64_t M, int64_t d, int64_t ld_x, const int8_t* signs,
                        float clip_ratio, uint8_t* q_out, void* scale_out, float* rot_out,
                        void* stream);

/*
 * quarot_rotate_quant_fp16 -- quarot_rotate_quant with the rotation carried
 * out in fp16 arithmetic.  [S] "Kernel Implementation and Hardware
 * Efficiency", online Hadamard transforms: FP32 arithmetic is the default and
 * FP16 the tested alternative with nearly identical accuracy (Appendix A.7,
 * Table 10).  The pages fix no operation order; this library's:
 *   y = fp16(s * x * fp16(1/sqrt(d)))
 *   butterflies of span 1, 2, ..., P/2 (P the power-of-two factor of d),
 *   pairing i and i + h (i & h == 0) into (fp16(a + b), fp16(a - b))
 *   for d = 12 P: out[c P + j] = fp16 running sum over a = 0 .. 11 of
 *   H12[a][c] * y[a P + j], rounded after every term
 * then the quantizer of quarot_rotate_quant on the fp16 values (rot_out
 * receives them).  The sums stay below sqrt(d) max|x|, so inputs above
 * 65504 / sqrt(d) in magnitude may overflow to inf.  Arguments, widths and
 * errors as quarot_rotate_quant.
 */
int quarot_rotate_quant_fp16(const void* x, int64_t M, int64_t d, int64_t ld_x, const int8_t* signs,
                             float clip_ratio, uint8_t* q_out, void* scale_out, float* rot_out,
                             void* stream);

/*
 * quarot_rmsnorm_rotate_quant -- quarot_rotate_quant preceded by a scale-free
 * RMSNorm of each row, fused in the same kernel.  [G] "Deep Dive: The
 * End-to-End QuaRot Layer Lifecycle", 2 "Online Activation Rotation Fused into
 * RMSNorm" (RMSNorm(x) = x / sqrt(mean x^2 + eps), normalize, FWHT and quantize
 * in one kernel); [S] "Computational Invariance and Between-Block Rotation
 * (Stage 1a)": the learned RMSNorm scale is absorbed into the next weights, so
 * only the normalization stays online.
 *
 * For each row i of x:
 *   y = x_i / sqrt(mean_j x_ij^2 + eps)            (fp32)
 *   r = (y * s) @ H_d / sqrt(d), then S and q exactly as quarot_rotate_quant
 * (the rotation preserves the row norm, so the sum of squares is taken from
 * the input row).  Arguments as quarot_rotate_quant, plus:
 *   eps       > 0 (finite); otherwise QUAROT_ERR_INVALID_ARG
 *   rot_out   receives the normalized rotated values r, or NULL
 */
int quarot_rmsnorm_rotate_quant(const void* x, int64_t M, int64_t d, int64_t ld_x, float eps,
                                const int8_t* signs, float clip_ratio, uint8_t* q_out, void* scale_out,
                                float* rot_out, void* stream);

/*
 * quarot_crosshead_rotate_quant -- the online cross-head Hadamard applied to
 * the concatenated attention output before the output projection, fused with
 * per-token INT4 quantization.  [S] Stage 1c, "The online Hadamard heads
 * transform": H_{nh dh} = (I_nh (x) H_dh)(H_nh (x) I_dh); the head-wise factor
 * is carried by the rotated values (quarot_decode_attn with unrotate_out = 0),
 * the cross-head factor runs here; Stage 2b per-token quantizer.
 *
 * For each row i of z (d = nh * dh, element h * dh + j):
 *   r[k * dh + j] = sum_h z[h * dh + j] * H_nh[h][k] / sqrt(nh)   (fp32)
 *   S, q exactly as quarot_rotate_quant (clip_ratio).
 * A W_out prepared with quarot_rotate_quant(signs = NULL) at width d then
 * sees the fully rotated input (Sylvester H_d = H_nh (x) H_dh).
 *
 *   z         fp16 [M, ld_z], first nh * dh columns used, 2-byte aligned
 *   nh        power of two, 1 .. 64 (else QUAROT_ERR_UNSUPPORTED)
 *   dh        64 or 128
 *   q_out     uint8 [M, d/2], 4-byte aligned
 *   scale_out fp16 [M]
 *   rot_out   fp32 [M, d] (the rotated values), or NULL
 */
int quarot_crosshead_rotate_quant(const void* z, int64_t M, int64_t nh, int64_t dh, int64_t ld_z, float clip_ratio,
                                  uint8_t* q_out, void* scale_out, float* rot_out, void* stream);

/*
 * quarot_w4a4_gemm -- W4A4 GEMM with INT32-exact accumulation and the
 * per-token x per-output-channel dequantization epilogue.
 * [S] Stage 2b "dequantization step", "Kernel Implementation" (INT4 GEMM,
 * INT32 accumulator, scale by scale_x[i] * scale_w[j]); [G] "Pure INT4 Tensor
 * Core GEMM Execution".
 *
 *   acc[i, j] = sum_k a[i, k] * w[j, k]               (exact integer)
 *   y[i, j]   = fp16(fp32(fp32(acc) * sx[i]) * sw[j])
 *
 *   a_q       uint8 [M, K/2] packed activations (K-major), 16-byte aligned
 *   a_scale   fp16 [M], 2-byte aligned
 *   w_q       uint8 [N, K/2] packed weights (K-major, [out, in]), 16-byte aligned
 *   w_scale   fp16 [N], 16-byte aligned (the epilogue loads it in 16-byte vectors)
 *   M, N      >= 0 (ragged tails handled); K % 128 == 0, 128 <= K <= 65536
 *             (the bound keeps every partial sum exact in fp32 on the tensor cores)
 *   y         fp16 [M, N], 16-byte aligned
 *   acc_out   int32 [M, N] (the exact accumulator, for testing), or NULL; 4-byte aligned
 * Misaligned pointers return QUAROT_ERR_ALIGNMENT before any launch.
 */
int quarot_w4a4_gemm(const uint8_t* a_q, const void* a_scale, const uint8_t* w_q,
                     const void* w_scale, int64_t M, int64_t N, int64_t K, void* y,
                     int32_t* acc_out, void* stream);

/*
 * quarot_rotate_quant_a8 -- quarot_rotate_quant with the codes written in the
 * tensor-core operand form that quarot_w4a4_gemm_a8 reads, instead of packed
 * nibbles.  [S] Stage 2a (online Hadamard, per-token symmetric INT4
 * quantization): the same codes and scales as quarot_rotate_quant, bit for
 * bit.  The pages have no such format: sm_103a tensor cores take 8-bit
 * operands only, so every 4-bit code is widened to a byte before an MMA; this
 * entry point widens each activation code once, where it is produced, rather
 * than once per output-column tile inside the GEMM.
 *
 *   x, M, d, ld_x, signs, clip_ratio   as quarot_rotate_quant; d = 4096 or
 *                                      12288 (else QUAROT_ERR_UNSUPPORTED)
 *   a8_out      uint8 [M, d], 16-byte aligned: byte 8g + j holds u = v + 8
 *               (0..15) of code 8g + p(j), p = (0, 2, 4, 6, 1, 3, 5, 7); the
 *               e4m3 byte with that bit pattern has the value u * 2^-9
 *   scale_out   fp16 [M], 2-byte aligned
 *   rowsum_out  int32 [M], 4-byte aligned: sum over the row's codes v
 * Misaligned pointers return QUAROT_ERR_ALIGNMENT before any launch.
 */
int quarot_rotate_quant_a8(const void* x, int64_t M, int64_t d, int64_t ld_x, const int8_t* signs,
                           float clip_ratio, uint8_t* a8_out, void* scale_out, int32_t* rowsum_out,
                           void* stream);

/*
 * quarot_w4a4_gemm_a8 -- quarot_w4a4_gemm with the activations in the form
 * quarot_rotate_quant_a8 writes: the same exact accumulator and the same fp16
 * output, bit for bit.  [S] Stage 2b, "Kernel Implementation".  The weights
 * stay packed INT4 (4 bits per code in memory); only their conversion runs
 * inside the GEMM.
 *
 *   a8        uint8 [M, K] (quarot_rotate_quant_a8 layout), 16-byte aligned
 *   a_rowsum  int32 [M] code sums of the rows, 4-byte aligned
 *   a_scale, w_q, w_scale, y, acc_out   as quarot_w4a4_gemm
 *   M, N      >= 0; K % 256 == 0, 256 <= K <= 65536 (else QUAROT_ERR_UNSUPPORTED)
 * Runs on CTA pairs (thread-block clusters of two); a GPU with fewer than two
 * SMs gets QUAROT_ERR_UNSUPPORTED.  Misaligned pointers return
 * QUAROT_ERR_ALIGNMENT before any launch.
 */
int quarot_w4a4_gemm_a8(const uint8_t* a8, const int32_t* a_rowsum, const void* a_scale, const uint8_t* w_q,
                        const void* w_scale, int64_t M, int64_t N, int64_t K, void* y, int32_t* acc_out,
                        void* stream);

/*
 * quarot_rotate_quant_rowsum -- quarot_rotate_quant (same codes, scales and
 * errors) that also writes each row's code sum rowsum_out[i] = sum_k q[i, k]
 * (int32 [M], 4-byte aligned), the per-token offset correction of
 * quarot_w4a4_gemm_rowsums.  Supported widths: d = 4096 and 12288
 * (QUAROT_ERR_UNSUPPORTED otherwise; quarot_int4_rowsum serves any width).
 */
int quarot_rotate_quant_rowsum(const void* x, int64_t M, int64_t d, int64_t ld_x, const int8_t* signs,
                               float clip_ratio, uint8_t* q_out, void* scale_out, int32_t* rowsum_out,
                               void* stream);

/*
 * quarot_int4_rowsum -- code sums of the rows of a packed INT4 matrix q
 * (uint8 [M, K/2] in the quarot_rotate_quant format, 16-byte aligned):
 * rowsum_out[i] = sum_k q[i, k] (int32 [M], 4-byte aligned).  K % 32 == 0,
 * K <= 2^24.  For the weight rows this runs once, at weight preparation.
 */
int quarot_int4_rowsum(const uint8_t* q, int64_t M, int64_t K, int32_t* rowsum_out, void* stream);

/*
 * quarot_w4a4_gemm_rowsums -- quarot_w4a4_gemm with the row code sums of
 * both operands given: a_rowsum[i] = sum_k a[i, k] (int32 [M]) and
 * w_rowsum[j] = sum_k w[j, k] (int32 [N]), both 4-byte aligned, from
 * quarot_rotate_quant_rowsum / quarot_int4_rowsum.  The result is the same,
 * bit for bit (the exact accumulator and its dequantization); the CTA-pair
 * kernel then leaves the sums of its offset encoding to these inputs instead
 * of summing the codes it unpacks.  Sums that are not the codes' sums give
 * wrong results.  Other arguments and errors as quarot_w4a4_gemm; null sums
 * (M, N > 0) are QUAROT_ERR_INVALID_ARG.
 */
int quarot_w4a4_gemm_rowsums(const uint8_t* a_q, const void* a_scale, const int32_t* a_rowsum,
                             const uint8_t* w_q, const void* w_scale, const int32_t* w_rowsum, int64_t M, int64_t N,
                             int64_t K, void* y, int32_t* acc_out, void* stream);

/* quarot_w4a4_gemm_plan -- which kernel and N-tile width quarot_w4a4_gemm
 * launches for an M x N x K problem on a GPU with `sms` SMs (a host-only
 * query: it touches no device).  *form = 2 for the CTA-pair kernel (M > 128
 * and an even number of 128-wide k-blocks) with one tensor-memory
 * accumulator, 3 for the same kernel with two (possible at tile widths up to
 * 192 from three tiles per pair: one tile's drain overlaps the next tile's
 * MMAs), 1 for the one-SM kernel; *bn is the N-tile width, one of 128, 160,
 * 192, 224.  The pair kernel's width and form minimise a time model per pair
 * (a tile costs its k-block count, each drain that one accumulator exposes
 * about 5 k-blocks more, ties going to the narrower width).  Returns QUAROT_ERR_INVALID_ARG
 * for non-positive sizes or null outputs and QUAROT_ERR_UNSUPPORTED for a K
 * the GEMM rejects.  The pages have no counterpart: it lets tests and tools
 * see which tile configuration a shape exercises. */
int quarot_w4a4_gemm_plan(int64_t M, int64_t N, int64_t K, int sms, int* form, int* bn);

/*
 * quarot_kv_write -- "Append": rotate the new keys and values head-wise by
 * H_d / sqrt(d) (no random signs), quantize each (token, head) vector to
 * symmetric INT4 with an fp16 scale (clip 1.0, the formula of
 * quarot_rotate_quant) and store them at positions t_start .. t_start+T_new-1.
 * [S] Stage 1c/1d (head-wise H_dh on V and on post-RoPE K), Stage 2c (KV
 * cache procedure), "Append" routine; [G] "4-Bit Rotated KV Cache".
 *
 *   k, v      fp16 [B, T_new, Hkv, d], 16-byte aligned
 *   d         64, 128 or 256
 *   t_start   >= 0, t_start + T_new <= T_max
 *   k_q, v_q  uint8 [B, Hkv, T_max, d/2] caches, 16-byte aligned
 *   k_s, v_s  fp16 [B, Hkv, T_max] per-(token, head) scales
 */
int quarot_kv_write(const void* k, const void* v, int64_t B, int64_t T_new, int64_t Hkv,
                    int64_t d, int64_t t_start, int64_t T_max, uint8_t* k_q, void* k_s,
                    uint8_t* v_q, void* v_s, void* stream);

/*
 * quarot_decode_workspace_bytes -- bytes of scratch quarot_decode_attn needs
 * for these sizes (split-T partial softmax states).  0 on invalid sizes.
 */
size_t quarot_decode_workspace_bytes(int64_t B, int64_t Hq, int64_t d, int64_t T);

/*
 * quarot_decode_attn -- one-token GQA decode attention over the INT4 cache,
 * dequantizing on read.  [S] Stage 1d (rotate the query head-wise after
 * RoPE), Stage 2c (load, dequantize on the fly, dot products, softmax),
 * "Decode" routine.
 *
 *   q~ = q_h @ H_d / sqrt(d);  g = h / (Hq / Hkv)
 *   s_t = sm_scale * (q~ . (k_s[t] * kcode_t)),  p = softmax(s) over t < T
 *   o   = sum_t p_t * v_s[t] * vcode_t;  if unrotate_out: o <- o @ H_d / sqrt(d)
 *
 *   q         fp16 [B, Hq, d], 16-byte aligned
 *   k_q, k_s, v_q, v_s  caches as written by quarot_kv_write (capacity T_max)
 *   d         128; Hq % Hkv == 0 and Hq / Hkv in {1, 2, 4, 8}
 *   T         tokens to attend, 0 <= T <= T_max (T == 0 gives o = 0)
 *   sm_scale  softmax scale; <= 0 selects 1/sqrt(d)
 *   unrotate_out  0: o stays in the rotated basis (the rotation is absorbed
 *             by W_out, Stage 1c); 1: o is rotated back
 *   out       fp16 [B, Hq, d]
 *   workspace device scratch of ws_bytes >= quarot_decode_workspace_bytes(),
 *             256-byte aligned, owned by the caller; contents need no
 *             initialisation and are clobbered
 */
int quarot_decode_attn(const void* q, const uint8_t* k_q, const void* k_s, const uint8_t* v_q,
                       const void* v_s, int64_t B, int64_t Hq, int64_t Hkv, int64_t d, int64_t T,
                       int64_t T_max, float sm_scale, int unrotate_out, void* out, void* workspace,
                       size_t ws_bytes, void* stream);

/*
 * quarot_prefill_attn -- "Init": attention of a whole prompt over the INT4
 * cache, flash-attention style, dequantizing keys and values on load.
 * [S] "Kernel Implementation and Hardware Efficiency", quantized attention
 * with KV cache, Init (flash attention with dequantized keys and values, all
 * of them available at once during prefill); Stage 1d (the query is rotated
 * head-wise after RoPE, as the cached keys are).
 *
 * Query i of head h attends to cached tokens t < T (t <= i when causal):
 *   q~ = q[b, i, h] @ H_d / sqrt(d);  g = h / (Hq / Hkv)
 *   s_t = sm_scale * (q~ . (k_s[t] * kcode_t)),  p = softmax(s)
 *   out[b, i, h] = sum_t p_t * v_s[t] * vcode_t    (rotated basis, Stage 1c)
 * Arithmetic: q~ * sm_scale * log2(e), the dequantized keys and values and
 * the probabilities are fp16 (the pages' fp16 flash attention); products
 * accumulate in fp32 on the tensor cores; softmax is fp32.
 *
 *   q         fp16 [B, T, Hq, d] (prompt tokens 0 .. T-1), 16-byte aligned
 *   k_q, k_s, v_q, v_s  caches as written by quarot_kv_write (capacity
 *             T_max >= T, tokens 0 .. T-1 written); k_q, v_q 16-byte aligned
 *   d         128; Hq % Hkv == 0, Hq / Hkv in {1, 2, 4, 8}
 *   sm_scale  softmax scale; <= 0 selects 1/sqrt(d)
 *   causal    1: token i sees t <= i (prefill); 0: every token sees all T
 *   out       fp16 [B, T, Hq, d], 16-byte aligned
 * T == 0 or B == 0 is a no-op.
 */
int quarot_prefill_attn(const void* q, const uint8_t* k_q, const void* k_s, const uint8_t* v_q,
                        const void* v_s, int64_t B, int64_t Hq, int64_t Hkv, int64_t d, int64_t T,
                        int64_t T_max, float sm_scale, int causal, void* out, void* stream);

/*
 * quarot_kv_write_asym -- quarot_kv_write with the pages' own KV quantizer:
 * asymmetric per group of 128 with a zero point and a clipping ratio.
 * [S] Stage 2c "KV Cache Quantization (online, per-group asymmetric)": group
 * size 128 = one group per (token, head) vector at d = 128; s = (a_max -
 * a_min) / (2^4 - 1); z = round(a_min / s); a_min, a_max from a clipping ratio
 * (0.95 in the pages).  The page's formula mixes units; this library keeps
 * the zero point on the code grid:
 *   a = clip * (min, max) of the rotated vector,
 *   s = fp16(min(max(a_max - a_min, 1e-5) / 15, 65504)),
 *   z = clamp(rne(a_min / s), -32768, 32767),
 *   q = clamp(rne(x / s) - z, 0, 15), and x^ = s (q + z) on read.
 * The rotation is the head-wise H_d / sqrt(d) of quarot_kv_write.
 *
 *   k, v, B, T_new, Hkv, d, t_start, T_max   as quarot_kv_write
 *   clip_ratio  in (0, 1]
 *   k_q, v_q  uint8 [B, Hkv, T_max, d/2] unsigned codes (even dim in the low nibble)
 *   k_s, v_s  fp16 [B, Hkv, T_max] scales
 *   k_z, v_z  int16 [B, Hkv, T_max] zero points (2-byte aligned; 16-byte
 *             aligned with T_max % 8 == 0 for the decode's bulk-copy path)
 */
int quarot_kv_write_asym(const void* k, const void* v, int64_t B, int64_t T_new, int64_t Hkv, int64_t d,
                         int64_t t_start, int64_t T_max, float clip_ratio, uint8_t* k_q, void* k_s, int16_t* k_z,
                         uint8_t* v_q, void* v_s, int16_t* v_z, void* stream);

/*
 * quarot_decode_attn_asym -- quarot_decode_attn over caches written by
 * quarot_kv_write_asym: k^_t = k_s[t] (kcode_t + k_z[t]), v^_t likewise,
 * dequantized on read ([S] Stage 2c "Dequantizes each group on-the-fly").
 * Arguments as quarot_decode_attn plus the zero-point arrays; the same
 * workspace size (quarot_decode_workspace_bytes).
 */
int quarot_decode_attn_asym(const void* q, const uint8_t* k_q, const void* k_s, const int16_t* k_z,
                            const uint8_t* v_q, const void* v_s, const int16_t* v_z, int64_t B, int64_t Hq,
                            int64_t Hkv, int64_t d, int64_t T, int64_t T_max, float sm_scale, int unrotate_out,
                            void* out, void* workspace, size_t ws_bytes, void* stream);

/* quarot_legacy_imma_probe -- a measurement utility: one launch that issues
 * nothing but one legacy warp-level tensor-core instruction, mma.sync s8
 * m16n8k32 (bits = 8), s4 m16n8k64 (bits = 4) or f16 m16n8k16 with fp32
 * accumulators (bits = 16, the instruction of the decode and prefill
 * attention kernels), from registers, in eight independent chains per warp
 * on every SM.  [S] "Kernel
 * Implementation and Hardware Efficiency" runs its 4-bit GEMM on this
 * instruction class (CUTLASS INT4 on Ampere); the probe measures the rate it
 * reaches on this GPU, context for the tcgen05 GEMM's throughput.
 *
 *   bits     8, 4 or 16
 *   iters    loop trips per warp (> 0); each trip issues 8 instructions
 *   sink     int32 device word, 4-byte aligned (written only in a case that
 *            keeps the compiler from removing the arithmetic)
 *   ops      host int64: receives the operations the launch performs
 *            (2 per multiply-accumulate); time the launch with events on
 *            `stream` and divide
 * Returns QUAROT_ERR_INVALID_ARG for other widths, iters <= 0 or null
 * pointers.  The pages have no such entry point. */
int quarot_legacy_imma_probe(int bits, int iters, int32_t* sink, int64_t* ops, void* stream);

/*
 * quarot_decode_attn_static -- quarot_decode_attn for callers that cannot
 * allocate device memory when they run decode (a plain C host without an
 * allocator, a serving loop that forbids cudaMalloc/cudaFree after start-up
 * because they synchronise the device or may fail, a plug-in that only
 * receives its input and output buffers).  The QuaRot pages have no
 * counterpart: this is a deployment variant of the "Decode" entry above.
 *
 * Same arguments and result as quarot_decode_attn, without the workspace:
 * the split-T scratch is a fixed array of QUAROT_DECODE_STATIC_SCRATCH_BYTES
 * inside the library, present on every GPU that loads it until process exit.
 * The call allocates nothing.
 *   - Returns QUAROT_ERR_UNSUPPORTED, before touching the device, when
 *     quarot_decode_workspace_bytes(B, Hq, d, T) exceeds that maximum.
 *   - The first call in each CUDA context looks up the array's device
 *     address (with that device current) and caches it with the context's
 *     id; make that first call before any stream capture.  After a
 *     cudaDeviceReset (or any re-creation of the context) the library's
 *     module is loaded again and the array may move: the next call sees a
 *     new context id and looks the address up again, so the array's old
 *     contents are gone but no stale address is used.  A failed lookup
 *     returns QUAROT_ERR_CUDA.
 *   - Invalid arguments get the status quarot_decode_attn gives them, and
 *     nothing touches the device for a rejected request.
 *   - Every call on a device shares the one array.  No part of it needs to
 *     start at zero (each call writes every slot it later reads), but two
 *     calls whose executions overlap on the GPU (different streams, no
 *     ordering between them) race on it and give undefined results.
 */
#define QUAROT_DECODE_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

int quarot_decode_attn_static(const void* q, const uint8_t* k_q, const void* k_s, const uint8_t* v_q,
                              const void* v_s, int64_t B, int64_t Hq, int64_t Hkv, int64_t d, int64_t T,
                              int64_t T_max, float sm_scale, int unrotate_out, void* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QUAROT_H_ */
