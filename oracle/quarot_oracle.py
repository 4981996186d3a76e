"""CPU oracle for the QuaRot W4A4 hot path -- TEST INFRASTRUCTURE ONLY.

This module is the plain, slow, obviously-correct statement of what the hot
path computes.  It is used by the test-suite, by ``__graft_entry__.smoke()``
and by ``bench.py``'s CPU-baseline leg, and by nothing else: the product path
(``w4a4_rotated_quantized_gb300``) never imports, calls or links it, and this
module imports nothing from the product.  It shares no code with the CUDA
path; the only common module is ``workloads`` (seeded random inputs).

Arithmetic is numpy float64 with explicit dense Hadamard matrices, an exact
integer GEMM, and float32/float16 only where the method
fixes the storage precision (rotated values are compared as fp32, scales are
stored as fp16, the dequantised output is fp16).  ``rotate_fwht`` is a second,
O(d log d) mode of the same rotation (butterflies instead of the dense
product), pinned against the dense definition; it exists only so that the
host baseline can be timed with the fast transform as well.

Sources (page title, section):
  [S]  "QuaRot: Outlier-Free 4-Bit Inference in Rotated LLMs" (paper summary
       page), section 3 "Technical Approach": Stage 1a (randomized Hadamard,
       Kronecker sizes), Stage 1c/1d (head-wise H_dh on V, K and Q), Stage 2a/2b
       (symmetric per-channel / per-token quantizers, dequantisation), Stage 2c
       (KV decode procedure), "Kernel Implementation and Hardware Efficiency".
  [G]  "QuaRot Guide: Outlier-Free 4-Bit W4A4 LLM Quantization" (blog),
       sections "The Collapse of Naive W4A4" (INT4 grid -8..7), "Why Randomized
       Walsh-Hadamard Transforms (RHT) Disperse Outliers" (Sylvester doubling,
       x~_j = (1/sqrt d) sum_k D_kk H_jk x_k), "End-to-End Implementation" (abs-max
       floor 1e-5).
  [E]  QuaRot paper-viz explainer (romaanj.github.io): Sylvester for 2^n and a
       Kronecker product with a Paley-12 block for 12288.

Readings where the pages are silent or disagree (each also listed in the
design notes):
  * rotation is x~ = (x * s) @ H / sqrt(d), row-vector convention, signs first;
  * FP16 rotation variant: scale by fp16(1/sqrt(d)) first, then butterflies of
    span 1, 2, ..., P/2 and (for 12 * 2^n) the Paley-12 sums in index order,
    every result rounded to fp16;
  * H_12288 = H12 (+) H1024 (Kronecker, index k = a*1024 + b), H12 = Paley I
    with q = 11: Jacobsthal Q_ij = chi(j - i), S = [[0, 1^T], [-1, Q]], H = I + S;
  * activation scale S = max(clip * max|x~|, 1e-5) / 7, stored as fp16
    (saturating at 65504), codes = clamp(round_half_even(x~ / S_fp16), -8, 7);
  * two codes per byte, even index in the low nibble, two's complement;
  * dequant epilogue Y = fp16(fp32(fp32(acc) * sx_i) * sw_j);
  * cross-head transform: x~ = z (H_nh (x) I_dh) / sqrt(nh), index h * dh + j,
    no random signs (head counts a power of two);
  * RMSNorm is scale-free, x / sqrt(mean(x^2) + eps), applied before the
    rotation (they commute: the rotation preserves the row norm);
  * asymmetric KV mode: a = 0.95 * (min, max) of the group, s = fp16(range / 15),
    integer zero point z = rne(a_min / s) stored as int16, q = clamp(rne(x/s) - z,
    0, 15), x^ = s (q + z);
  * KV: head-wise H_128 without random signs, per-(token, head) symmetric INT4
    with an fp16 scale; decode softmax in full precision, GQA head h reads KV
    head h // (Hq / Hkv); output optionally rotated back by the same H_128;
  * prefill ("Init"): prompt token i attends to cached tokens t <= i (or to all
    T tokens without the mask), with the same rotated query, dequantized keys
    and values and full-precision softmax as the decode; the output stays in
    the rotated basis.
"""
from __future__ import annotations

import functools
import math

import numpy as np

FP16_MAX = 65504.0
SCALE_FLOOR = 1e-5  # abs-max floor of the guide's quantize_to_int4_symmetric
QMIN, QMAX = -8, 7  # INT4 grid, [G] "The Collapse of Naive W4A4"


# ---------------------------------------------------------------------------
# Hadamard matrices ([G] Sylvester doubling; [S] Stage 1a Kronecker sizes;
# [E] Paley-12 block)
# ---------------------------------------------------------------------------
@functools.lru_cache(maxsize=None)
def sylvester(n: int) -> np.ndarray:
    """Integer Sylvester Hadamard matrix of order n = 2^k: H_1 = [1],
    H_2m = [[H_m, H_m], [H_m, -H_m]]."""
    if n < 1 or n & (n - 1):
        raise ValueError(f"Sylvester order must be a power of two, got {n}")
    h = np.ones((1, 1), dtype=np.int8)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    h.setflags(write=False)
    return h


def legendre(a: int, q: int) -> int:
    """chi(a) for prime q: 0 if a = 0 mod q, +1 for a nonzero square, -1 otherwise."""
    a %= q
    if a == 0:
        return 0
    squares = {(x * x) % q for x in range(1, q)}
    return 1 if a in squares else -1


@functools.lru_cache(maxsize=None)
def paley12() -> np.ndarray:
    """Paley construction I of order q + 1 = 12 with q = 11 (q = 3 mod 4).

    Jacobsthal matrix Q_ij = chi(j - i) (antisymmetric for q = 3 mod 4),
    S = [[0, 1^T], [-1, Q]] and H = I + S.  Not symmetric.
    """
    q = 11
    Q = np.array([[legendre(j - i, q) for j in range(q)] for i in range(q)], dtype=np.int8)
    S = np.zeros((q + 1, q + 1), dtype=np.int8)
    S[0, 1:] = 1
    S[1:, 0] = -1
    S[1:, 1:] = Q
    H = (np.eye(q + 1, dtype=np.int8) + S).astype(np.int8)
    H.setflags(write=False)
    return H


@functools.lru_cache(maxsize=4)
def hadamard(d: int) -> np.ndarray:
    """Dense integer (+-1) Hadamard matrix of order d, as int8 [d, d].

    d = 2^n: Sylvester.  d = 12 * 2^n: H12 (Kronecker) H_{2^n}, entry
    [(a, b), (c, e)] = H12[a, c] * H_{2^n}[b, e] with row/col index a*2^n + b.
    """
    if d >= 1 and d & (d - 1) == 0:
        return sylvester(d)
    if d % 12 == 0 and (d // 12) & (d // 12 - 1) == 0:
        H = np.kron(paley12(), sylvester(d // 12)).astype(np.int8)
        H.setflags(write=False)
        return H
    raise ValueError(f"no Hadamard construction for d = {d} (need 2^n or 12*2^n)")


def _apply_dense(xs: np.ndarray, H: np.ndarray, block: int = 1024) -> np.ndarray:
    """xs @ H in float64, with H's columns converted to float64 a block at a time
    (bounds memory at d = 12288; the product itself is the plain dense one)."""
    d = H.shape[0]
    out = np.empty((xs.shape[0], d), dtype=np.float64)
    for j0 in range(0, d, block):
        out[:, j0:j0 + block] = xs @ H[:, j0:j0 + block].astype(np.float64)
    return out


# ---------------------------------------------------------------------------
# Online rotation ([S] Stage 1a, 1b; [G] RHT section)
# ---------------------------------------------------------------------------
def rotate(x: np.ndarray, signs: np.ndarray | None) -> np.ndarray:
    """x~ = (x * s) @ H_d / sqrt(d) for each row, exact in float64, returned as fp32.

    x: [..., d] (any float dtype, fp16 in the workloads).  signs: int8 [d] of
    +-1, or None for the plain (unsigned) Hadamard used on K, V and q.
    """
    x = np.asarray(x)
    d = x.shape[-1]
    xs = x.reshape(-1, d).astype(np.float64)
    if signs is not None:
        xs = xs * np.asarray(signs, dtype=np.float64)[None, :]
    r = _apply_dense(xs, hadamard(d)) / math.sqrt(d)
    return r.astype(np.float32).reshape(x.shape)


def rotate_f64(x: np.ndarray, signs: np.ndarray | None) -> np.ndarray:
    """Same map as ``rotate`` but left in float64 (for invariance checks)."""
    x = np.asarray(x)
    d = x.shape[-1]
    xs = x.reshape(-1, d).astype(np.float64)
    if signs is not None:
        xs = xs * np.asarray(signs, dtype=np.float64)[None, :]
    return (_apply_dense(xs, hadamard(d)) / math.sqrt(d)).reshape(x.shape)


def fwht_rows(xs: np.ndarray) -> np.ndarray:
    """The fast Walsh-Hadamard transform of every row, y = x @ H_{2^n} (Sylvester,
    unnormalized), in float64: n rounds of butterflies (a + b, a - b) over pairs
    at distance h = 1, 2, 4, ..., as in [G] "The Fast Walsh-Hadamard Transform".
    O(d log d) per row; the dense product ``_apply_dense`` is the definition."""
    y = np.array(xs, dtype=np.float64, copy=True)
    M, d = y.shape
    if d < 1 or d & (d - 1):
        raise ValueError(f"FWHT length must be a power of two, got {d}")
    h = 1
    while h < d:
        v = y.reshape(M, d // (2 * h), 2, h)
        a = v[:, :, 0, :].copy()
        b = v[:, :, 1, :]
        v[:, :, 0, :] = a + b
        v[:, :, 1, :] = a - b
        h *= 2
    return y


def rotate_fwht(x: np.ndarray, signs: np.ndarray | None) -> np.ndarray:
    """The same map as ``rotate`` computed with the fast transform (the oracle's
    O(d log d) mode, for timing on the host): signs, then the FWHT of each
    2^n block, then (for d = 12 * 2^n) the dense H12 across the 12 blocks,
    x~[a 2^n + b] = sum_c y[c 2^n + b] H12[c, a], scaled by 1/sqrt(d); float64,
    returned as fp32."""
    x = np.asarray(x)
    d = x.shape[-1]
    xs = x.reshape(-1, d).astype(np.float64)
    if signs is not None:
        xs = xs * np.asarray(signs, dtype=np.float64)[None, :]
    if d >= 1 and d & (d - 1) == 0:
        r = fwht_rows(xs)
    elif d % 12 == 0 and (d // 12) & (d // 12 - 1) == 0:
        p = d // 12
        y = fwht_rows(xs.reshape(-1, p)).reshape(xs.shape[0], 12, p)
        r = np.einsum("mcb,ca->mab", y, paley12().astype(np.float64)).reshape(xs.shape[0], d)
    else:
        raise ValueError(f"no Hadamard construction for d = {d} (need 2^n or 12*2^n)")
    return (r / math.sqrt(d)).astype(np.float32).reshape(x.shape)


# ---------------------------------------------------------------------------
# Symmetric INT4 quantizer ([S] Stage 2a/2b; [G] quantizer formula)
# ---------------------------------------------------------------------------
def quant_scale(absmax: np.ndarray, clip_ratio: float = 1.0) -> np.ndarray:
    """Per-row scale S = max(clip * absmax, 1e-5) / 7, rounded to fp16 (saturating)."""
    s = np.maximum(clip_ratio * np.asarray(absmax, dtype=np.float64), SCALE_FLOOR) / 7.0
    return np.minimum(s, FP16_MAX).astype(np.float16)


def round_half_even(y: np.ndarray) -> np.ndarray:
    """Round to nearest, ties to even (numpy's rint is IEEE roundTiesToEven)."""
    return np.rint(y)


def quantize_rows(xr: np.ndarray, clip_ratio: float = 1.0):
    """Per-row symmetric INT4: returns (codes int8 [..., d], scale fp16 [...]).

    The codes are computed with the stored fp16 scale:
    q = clamp(round_half_even(x~ / S), -8, 7), the division done in float64.
    """
    xr = np.asarray(xr, dtype=np.float32)
    absmax = np.max(np.abs(xr), axis=-1)
    S = quant_scale(absmax, clip_ratio)
    y = xr.astype(np.float64) / S.astype(np.float64)[..., None]
    q = np.clip(round_half_even(y), QMIN, QMAX).astype(np.int8)
    return q, S


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte: byte i = (q[2i] & 0xF) | ((q[2i+1] & 0xF) << 4)."""
    c = np.asarray(codes).astype(np.int16)
    if c.shape[-1] % 2:
        raise ValueError("last dimension must be even to pack two codes per byte")
    lo = c[..., 0::2] & 0xF
    hi = c[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Inverse of pack_int4: signed codes int8 [..., 2 * nbytes]."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    lo = p & 0xF
    hi = (p >> 4) & 0xF
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def rotate_quant(x: np.ndarray, signs: np.ndarray | None, clip_ratio: float = 1.0):
    """Rotation followed by per-row INT4 quantize-and-pack.

    Returns (packed uint8 [M, d/2], scale fp16 [M], rotated fp32 [M, d]).
    Applied to activations online ([S] Stage 1b/2b) and to weight rows offline
    for per-output-channel RTN ([S] Stage 2a; [G] "Offline Weight
    Transformation": W~ = W H^T, one scale per output row).
    """
    r = rotate(x, signs)
    q, S = quantize_rows(r, clip_ratio)
    return pack_int4(q), S, r


# ---------------------------------------------------------------------------
# FP16 online Hadamard ([S] "Kernel Implementation and Hardware Efficiency",
# online Hadamard transforms: FP32 arithmetic is the default, FP16 arithmetic
# the tested alternative with nearly identical accuracy, Appendix A.7 /
# Table 10)
# ---------------------------------------------------------------------------
def _f16(a) -> np.ndarray:
    """Round to the nearest fp16 value (ties to even), returned as float64."""
    return np.asarray(a, dtype=np.float64).astype(np.float16).astype(np.float64)


def rotate_fp16_arith(x: np.ndarray, signs: np.ndarray | None) -> np.ndarray:
    """The rotation x~ = (x * s) @ H_d / sqrt(d) computed in fp16 arithmetic.

    The pages name the variant but not its operation order; this library's
    reading (every step rounds to fp16, round-to-nearest-even):
      1. y = fp16(s * x * c) with c = fp16(1 / sqrt(d)) (the scaling comes first
         so no intermediate exceeds the row's l1 norm times c);
      2. the Sylvester part, d = NA * P with P a power of two: butterflies of
         span h = 1, 2, 4, ..., P/2 within each length-P segment, pairing
         indices i and i + h (i & h == 0) into (fp16(a + b), fp16(a - b));
      3. for d = 12 P, the Paley-12 part across the segments: for each column
         c and in-segment index j, acc = 0 then acc = fp16(acc + H12[a, c] *
         y[a P + j]) for a = 0, 1, ..., 11.
    Returns float64 [..., d] holding the fp16 values.
    """
    x = np.asarray(x)
    d = x.shape[-1]
    na = 12 if (d % 12 == 0 and (d // 12) & (d // 12 - 1) == 0) else 1
    P = d // na
    if P < 1 or P & (P - 1):
        raise ValueError(f"no Hadamard construction for d = {d} (need 2^n or 12*2^n)")
    xs = x.reshape(-1, d).astype(np.float64)
    if signs is not None:
        xs = xs * np.asarray(signs, dtype=np.float64)[None, :]
    c = float(np.float16(1.0 / math.sqrt(d)))
    y = _f16(xs * c).reshape(-1, na, P)
    h = 1
    while h < P:
        v = y.reshape(y.shape[0], na, P // (2 * h), 2, h)
        a, b = v[:, :, :, 0, :], v[:, :, :, 1, :]
        y = np.stack([_f16(a + b), _f16(a - b)], axis=3).reshape(y.shape[0], na, P)
        h *= 2
    if na == 12:
        H12 = paley12().astype(np.float64)
        out = np.empty_like(y)
        for col in range(12):
            acc = np.zeros((y.shape[0], P))
            for a in range(12):
                acc = _f16(acc + H12[a, col] * y[:, a, :])
            out[:, col, :] = acc
        y = out
    return y.reshape(x.shape)


def rotate_quant_fp16(x: np.ndarray, signs: np.ndarray | None, clip_ratio: float = 1.0):
    """The FP16-arithmetic rotation followed by the same per-row INT4
    quantize-and-pack as ``rotate_quant``.  Returns (packed, scale fp16, rotated
    fp32 holding fp16 values)."""
    r = rotate_fp16_arith(x, signs).astype(np.float32)
    q, S = quantize_rows(r, clip_ratio)
    return pack_int4(q), S, r


# ---------------------------------------------------------------------------
# Scale-free RMSNorm fused with the rotation and the quantizer ([G] "Deep Dive:
# The End-to-End QuaRot Layer Lifecycle", part 2 "Online Activation Rotation
# Fused into RMSNorm"; [S] "Computational Invariance and Between-Block
# Rotation (Stage 1a)": the learned RMSNorm scale is absorbed into the next
# weights, leaving a pure normalization)
# ---------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean_j x_j^2 + eps) for each row, in float64.

    Scale-free: the per-feature scale is folded into the following weights,
    so only the normalization remains.  ([S] writes it as division by the row
    norm; the guide's form with the 1/d mean and eps differs only by the
    constant sqrt(d), which the per-token quantizer scale absorbs.)
    """
    xs = np.asarray(x, dtype=np.float64)
    return xs / np.sqrt(np.mean(xs * xs, axis=-1, keepdims=True) + eps)


def rmsnorm_rotate_quant(x: np.ndarray, signs: np.ndarray | None, eps: float, clip_ratio: float = 1.0):
    """RMSNorm, then the rotation, then the per-row INT4 quantizer, in that order.

    Returns (packed uint8 [M, d/2], scale fp16 [M], rotated fp32 [M, d]); the
    rotated values are (rmsnorm(x) * s) @ H / sqrt(d), exact in float64 and
    rounded once to fp32.
    """
    r = rotate(rmsnorm(x, eps), signs)
    q, S = quantize_rows(r, clip_ratio)
    return pack_int4(q), S, r


# ---------------------------------------------------------------------------
# Cross-head Hadamard before the output projection ([S] Stage 1c "The online
# Hadamard heads transform": H_{nh dh} = (I_nh (x) H_dh)(H_nh (x) I_dh); the
# head-wise factor is in the rotated values, the cross-head factor
# Z <- Z (H_nh (x) I_dh) runs online, then the per-token quantizer feeds the
# W4A4 output projection)
# ---------------------------------------------------------------------------
def crosshead_rotate(z: np.ndarray, nh: int) -> np.ndarray:
    """x~ = z (H_nh (x) I_dh) / sqrt(nh) for each row of d = nh * dh, element
    index k = h * dh + j: x~[k, j] = sum_h z[h, j] H_nh[h, k] / sqrt(nh).
    Exact in float64, returned as fp32."""
    z = np.asarray(z)
    d = z.shape[-1]
    if d % nh:
        raise ValueError("d must be a multiple of nh")
    zs = z.reshape(-1, nh, d // nh).astype(np.float64)
    H = hadamard(nh).astype(np.float64)
    r = np.einsum("mhj,hk->mkj", zs, H) / math.sqrt(nh)
    return r.reshape(z.shape).astype(np.float32)


def crosshead_rotate_quant(z: np.ndarray, nh: int, clip_ratio: float = 1.0):
    """Cross-head rotation, then the per-row INT4 quantize-and-pack:
    (packed uint8 [M, d/2], scale fp16 [M], rotated fp32 [M, d])."""
    r = crosshead_rotate(z, nh)
    q, S = quantize_rows(r, clip_ratio)
    return pack_int4(q), S, r


# ---------------------------------------------------------------------------
# W4A4 GEMM + dequant epilogue ([S] Stage 2b "dequantization step",
# "Kernel Implementation"; [G] "Pure INT4 Tensor Core GEMM Execution")
# ---------------------------------------------------------------------------
def int_gemm(a_codes: np.ndarray, w_codes: np.ndarray) -> np.ndarray:
    """acc[i, j] = sum_k a[i, k] * w[j, k], exact integers (int64 result)."""
    a = np.asarray(a_codes, dtype=np.int64)
    w = np.asarray(w_codes, dtype=np.int64)
    return a @ w.T


def dequant(acc: np.ndarray, sx: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """Y = fp16(fp32(fp32(acc) * sx[i]) * sw[j]) -- exact integer to fp32, two
    fp32 products, one rounding to fp16."""
    acc = np.asarray(acc)
    if np.max(np.abs(acc), initial=0) > 2 ** 24:
        raise ValueError("accumulator outside the range fp32 holds exactly")
    a32 = acc.astype(np.float32)
    t = a32 * np.asarray(sx, dtype=np.float16).astype(np.float32)[:, None]
    t = t * np.asarray(sw, dtype=np.float16).astype(np.float32)[None, :]
    return t.astype(np.float16)


def w4a4_gemm(a_packed, a_scale, w_packed, w_scale):
    """Returns (acc int64 [M, N], y fp16 [M, N]) from packed operands."""
    acc = int_gemm(unpack_int4(a_packed), unpack_int4(w_packed))
    return acc, dequant(acc, a_scale, w_scale)


# ---------------------------------------------------------------------------
# Rotated INT4 KV cache ([S] Stage 1c/1d, Stage 2c "KV cache operation during
# decoding", "Append"/"Decode" routines)
# ---------------------------------------------------------------------------
def kv_quant(kv: np.ndarray):
    """Head-wise rotation x~ = x @ H_d / sqrt(d) (no signs) and per-(token, head)
    symmetric INT4.  kv: fp16 [B, T, Hkv, d] -> (packed [B, Hkv, T, d/2], scale fp16 [B, Hkv, T])."""
    kv = np.asarray(kv)
    B, T, H, d = kv.shape
    r = rotate(kv, None)  # [B, T, H, d] fp32
    q, S = quantize_rows(r, 1.0)
    packed = pack_int4(q)  # [B, T, H, d/2]
    return np.ascontiguousarray(packed.transpose(0, 2, 1, 3)), np.ascontiguousarray(S.transpose(0, 2, 1))


def kv_write(k, v, t_start, k_cache, k_scale, v_cache, v_scale):
    """Append: quantize T_new tokens of K and V and store them at positions
    t_start .. t_start + T_new - 1 of the caches (modified in place)."""
    T_new = np.asarray(k).shape[1]
    kq, ks = kv_quant(k)
    vq, vs = kv_quant(v)
    k_cache[:, :, t_start:t_start + T_new, :] = kq
    k_scale[:, :, t_start:t_start + T_new] = ks
    v_cache[:, :, t_start:t_start + T_new, :] = vq
    v_scale[:, :, t_start:t_start + T_new] = vs


def decode_attn(q, k_cache, k_scale, v_cache, v_scale, T: int, sm_scale: float | None = None,
                unrotate: bool = False) -> np.ndarray:
    """One-token GQA decode attention over the first T cached tokens, float64.

    q: fp16 [B, Hq, d].  Caches [B, Hkv, T_max, d/2] uint8 and [B, Hkv, T_max] fp16.
    q~ = q @ H / sqrt(d); for head h the KV head is g = h // (Hq / Hkv);
    k^_t = Ks[t] * codes_t, s_t = sm_scale * (q~ . k^_t), p = softmax(s),
    o = sum_t p_t * Vs[t] * vcodes_t; optionally o <- o @ H / sqrt(d).
    Returns float64 [B, Hq, d].
    """
    q = np.asarray(q)
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    grp = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if sm_scale is None or sm_scale <= 0 else float(sm_scale)
    qr = rotate_f64(q, None)  # [B, Hq, d]
    out = np.zeros((B, Hq, d), dtype=np.float64)
    if T == 0:
        return out
    for b in range(B):
        for g in range(Hkv):
            kd = unpack_int4(k_cache[b, g, :T]).astype(np.float64) * k_scale[b, g, :T].astype(np.float64)[:, None]
            vd = unpack_int4(v_cache[b, g, :T]).astype(np.float64) * v_scale[b, g, :T].astype(np.float64)[:, None]
            qs = qr[b, g * grp:(g + 1) * grp]  # [grp, d]
            s = scale * (qs @ kd.T)  # [grp, T]
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            out[b, g * grp:(g + 1) * grp] = p @ vd
    if unrotate:
        out = rotate_f64(out, None)
    return out


def prefill_attn(q, k_cache, k_scale, v_cache, v_scale, T: int, sm_scale: float | None = None,
                 causal: bool = True, unrotate: bool = False) -> np.ndarray:
    """Prefill ("Init") attention of T query tokens over the first T cached
    tokens ([S] "Quantized attention with KV cache", Init routine: attention
    over the whole prompt with dequantized keys and values), float64.

    q: fp16 [B, T, Hq, d]; query i sits at position i.  q~ = q @ H / sqrt(d)
    per head; head h reads KV head h // (Hq / Hkv); s[i, t] = sm_scale *
    (q~_i . k^_t) with k^_t = Ks[t] * codes_t, restricted to t <= i when
    causal; p = softmax over t; o_i = sum_t p[i, t] * Vs[t] * vcodes_t;
    optionally o <- o @ H / sqrt(d).  Returns float64 [B, T, Hq, d].
    """
    q = np.asarray(q)
    B, Tq, Hq, d = q.shape
    if Tq != T:
        raise ValueError("prefill takes T queries for T cached tokens")
    Hkv = k_cache.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    grp = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if sm_scale is None or sm_scale <= 0 else float(sm_scale)
    qr = rotate_f64(q, None)  # [B, T, Hq, d]
    out = np.zeros((B, T, Hq, d), dtype=np.float64)
    if T == 0:
        return out
    mask = np.tril(np.ones((T, T), dtype=bool)) if causal else np.ones((T, T), dtype=bool)
    for b in range(B):
        for g in range(Hkv):
            kd = unpack_int4(k_cache[b, g, :T]).astype(np.float64) * k_scale[b, g, :T].astype(np.float64)[:, None]
            vd = unpack_int4(v_cache[b, g, :T]).astype(np.float64) * v_scale[b, g, :T].astype(np.float64)[:, None]
            for h in range(g * grp, (g + 1) * grp):
                s = scale * (qr[b, :, h] @ kd.T)  # [T, T]
                s = np.where(mask, s, -np.inf)
                s = s - s.max(axis=1, keepdims=True)
                p = np.exp(s)
                p /= p.sum(axis=1, keepdims=True)
                out[b, :, h] = p @ vd
    if unrotate:
        out = rotate_f64(out, None)
    return out


# ---------------------------------------------------------------------------
# Asymmetric per-group KV quantizer ([S] Stage 2c "KV Cache Quantization --
# online, per-group asymmetric": group size 128, i.e. one group per (token,
# head) at head_dim 128; scale s = (a_max - a_min) / (2^b - 1); zero point
# z = round(a_min / s); a_min, a_max from a clipping ratio of 0.95; dequantize
# on the fly).  The page mixes units (z subtracted from v, "s v^ + z"); the
# reading here keeps z on the code grid: q = clamp(rne(x / s) - z, 0, 15),
# x^ = s (q + z).
# ---------------------------------------------------------------------------
ZP_MIN, ZP_MAX = -32768, 32767  # zero points are stored as int16


def quantize_asym_rows(xr: np.ndarray, clip_ratio: float = 0.95):
    """Per-row asymmetric 4-bit quantizer.

    a_max = clip * max_j x_j, a_min = clip * min_j x_j;
    s = fp16(min(max(a_max - a_min, 1e-5) / 15, 65504)) (quantization uses the
    stored fp16 value); z = clamp(rne(a_min / s), int16 range);
    q_j = clamp(rne(x_j / s) - z, 0, 15).
    Returns (codes uint8 [..., d], scale fp16 [...], zero int16 [...]).
    """
    x = np.asarray(xr, dtype=np.float32).astype(np.float64)
    a_max = clip_ratio * x.max(axis=-1)
    a_min = clip_ratio * x.min(axis=-1)
    s = np.minimum(np.maximum(a_max - a_min, SCALE_FLOOR) / 15.0, FP16_MAX).astype(np.float16)
    sf = s.astype(np.float64)
    z = np.clip(round_half_even(a_min / sf), ZP_MIN, ZP_MAX)
    q = np.clip(round_half_even(x / sf[..., None]) - z[..., None], 0, 15)
    return q.astype(np.uint8), s, z.astype(np.int16)


def unpack_uint4(packed: np.ndarray) -> np.ndarray:
    """Unsigned nibbles (0..15), even index in the low nibble: uint8 [..., 2 * nbytes]."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def dequant_asym(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """x^ = s (q + z), float64."""
    return scale.astype(np.float64)[..., None] * (codes.astype(np.float64) + zero.astype(np.float64)[..., None])


def kv_quant_asym(kv: np.ndarray, clip_ratio: float = 0.95):
    """Head-wise rotation x~ = x @ H_d / sqrt(d) (no signs), then the asymmetric
    quantizer per (token, head).  kv: fp16 [B, T, Hkv, d] ->
    (packed [B, Hkv, T, d/2], scale fp16 [B, Hkv, T], zero int16 [B, Hkv, T])."""
    r = rotate(np.asarray(kv), None)
    q, s, z = quantize_asym_rows(r, clip_ratio)
    packed = pack_int4(q.astype(np.int16))  # unsigned nibbles pack like two's complement ones
    tr = (0, 2, 1, 3)
    return (np.ascontiguousarray(packed.transpose(tr)), np.ascontiguousarray(s.transpose(0, 2, 1)),
            np.ascontiguousarray(z.transpose(0, 2, 1)))


def kv_write_asym(k, v, t_start, k_cache, k_scale, k_zero, v_cache, v_scale, v_zero, clip_ratio: float = 0.95):
    """Append with the asymmetric quantizer: positions t_start .. t_start + T_new - 1."""
    T_new = np.asarray(k).shape[1]
    sl = slice(t_start, t_start + T_new)
    kq, ks, kz = kv_quant_asym(k, clip_ratio)
    vq, vs, vz = kv_quant_asym(v, clip_ratio)
    k_cache[:, :, sl, :], k_scale[:, :, sl], k_zero[:, :, sl] = kq, ks, kz
    v_cache[:, :, sl, :], v_scale[:, :, sl], v_zero[:, :, sl] = vq, vs, vz


def decode_attn_asym(q, k_cache, k_scale, k_zero, v_cache, v_scale, v_zero, T: int,
                     sm_scale: float | None = None, unrotate: bool = False) -> np.ndarray:
    """decode_attn over the asymmetric cache: k^_t = Ks[t] (kcodes_t + Kz[t]),
    v^_t = Vs[t] (vcodes_t + Vz[t]); everything else as decode_attn.  float64 [B, Hq, d]."""
    q = np.asarray(q)
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    grp = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if sm_scale is None or sm_scale <= 0 else float(sm_scale)
    qr = rotate_f64(q, None)
    out = np.zeros((B, Hq, d), dtype=np.float64)
    if T == 0:
        return out
    for b in range(B):
        for g in range(Hkv):
            kd = dequant_asym(unpack_uint4(k_cache[b, g, :T]), k_scale[b, g, :T], k_zero[b, g, :T])
            vd = dequant_asym(unpack_uint4(v_cache[b, g, :T]), v_scale[b, g, :T], v_zero[b, g, :T])
            qs = qr[b, g * grp:(g + 1) * grp]
            s = scale * (qs @ kd.T)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(axis=1, keepdims=True)
            out[b, g * grp:(g + 1) * grp] = p @ vd
    if unrotate:
        out = rotate_f64(out, None)
    return out


# ---------------------------------------------------------------------------
# Tolerance helpers for parity (the bars stated for the hot path)
# ---------------------------------------------------------------------------
def boundary_mask(xr: np.ndarray, scale: np.ndarray, eps: float = 1e-4) -> np.ndarray:
    """True where |x~ / S| lies within eps of a .5 rounding boundary (codes may
    legitimately differ there between two correct implementations)."""
    y = np.abs(np.asarray(xr, dtype=np.float64) / np.asarray(scale, dtype=np.float16).astype(np.float64)[..., None])
    frac = y - np.floor(y)
    return np.abs(frac - 0.5) < eps


def rotation_error(r_test: np.ndarray, r_ref: np.ndarray) -> float:
    """max_j |r_test - r_ref| / max(|r_ref_j|, rms(row)), the relative bar for
    rotated values floored at the row RMS."""
    r_ref = np.asarray(r_ref, dtype=np.float64)
    r_test = np.asarray(r_test, dtype=np.float64)
    rms = np.sqrt(np.mean(r_ref ** 2, axis=-1, keepdims=True))
    den = np.maximum(np.abs(r_ref), np.maximum(rms, 1e-30))
    return float(np.max(np.abs(r_test - r_ref) / den)) if r_ref.size else 0.0


def rel_fro(test: np.ndarray, ref: np.ndarray) -> float:
    """||test - ref||_F / ||ref||_F in float64."""
    ref = np.asarray(ref, dtype=np.float64)
    test = np.asarray(test, dtype=np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(test - ref) / n) if n > 0 else float(np.linalg.norm(test))
