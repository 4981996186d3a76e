"""QuaRot W4A4 hot path on GB300 (sm_103a): Python binding of libquarot.so.

This module only marshals arguments: it checks devices/dtypes/shapes, allocates
outputs with torch when the caller does not pass them, and calls the C ABI
declared in ``include/quarot.h``.  Every step of the computation runs in the
CUDA kernels of ``csrc/``; there is no CPU fallback.  If the shared library is
missing the calls raise ``QuarotError``.

Functions (same names as the C entry points):
    quarot_rotate_quant, quarot_w4a4_gemm, quarot_kv_write,
    quarot_decode_attn, quarot_decode_workspace_bytes, quarot_check_error,
    and the tensor-core operand form of the layer: quarot_rotate_quant_a8,
    quarot_w4a4_gemm_a8

``QuarotLinear`` composes them into the W4A4 linear layer: weight rows
rotated and quantized once, then per call the tokens rotated and quantized
and the INT4 GEMM with its dequant epilogue.  ``QuarotKVCache`` holds the
rotated INT4 KV cache with its append, decode and prompt-attention calls.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libquarot.so")

QUAROT_OK = 0
QUAROT_ERR_TIMEOUT = 5
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported size", 3: "misaligned pointer or leading dimension",
          4: "kernel launch failed", 5: "device-side wait timed out", 6: "CUDA error"}

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SIGS = {
    "quarot_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "quarot_version": (ctypes.c_int, []),
    "quarot_check_error": (ctypes.c_int, [_P]),
    "quarot_selftest_wait": (ctypes.c_int, [_P]),
    "quarot_rotate_quant": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, ctypes.c_float, _P, _P, _P, _P]),
    "quarot_rotate_quant_fp16": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, ctypes.c_float, _P, _P, _P, _P]),
    "quarot_rmsnorm_rotate_quant": (ctypes.c_int, [_P, _I64, _I64, _I64, ctypes.c_float, _P, ctypes.c_float, _P, _P,
                                                   _P, _P]),
    "quarot_crosshead_rotate_quant": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, ctypes.c_float, _P, _P, _P, _P]),
    "quarot_w4a4_gemm": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P]),
    "quarot_rotate_quant_a8": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, ctypes.c_float, _P, _P, _P, _P]),
    "quarot_w4a4_gemm_a8": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P]),
    "quarot_rotate_quant_rowsum": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, ctypes.c_float, _P, _P, _P, _P]),
    "quarot_int4_rowsum": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "quarot_w4a4_gemm_rowsums": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P]),
    "quarot_w4a4_gemm_plan": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                             ctypes.POINTER(ctypes.c_int)]),
    "quarot_kv_write": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "quarot_decode_workspace_bytes": (ctypes.c_size_t, [_I64, _I64, _I64, _I64]),
    "quarot_decode_attn": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                          ctypes.c_float, ctypes.c_int, _P, _P, ctypes.c_size_t, _P]),
    "quarot_decode_attn_static": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                                 ctypes.c_float, ctypes.c_int, _P, _P]),
    "quarot_legacy_imma_probe": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _P, ctypes.POINTER(ctypes.c_int64), _P]),
    "quarot_prefill_attn": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                           ctypes.c_float, ctypes.c_int, _P, _P]),
    "quarot_kv_write_asym": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _I64, _I64, ctypes.c_float, _P, _P, _P,
                                            _P, _P, _P, _P]),
    "quarot_decode_attn_asym": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64,
                                               ctypes.c_float, ctypes.c_int, _P, _P, ctypes.c_size_t, _P]),
}
DECODE_STATIC_SCRATCH_BYTES = 8 * 1024 * 1024  # QUAROT_DECODE_STATIC_SCRATCH_BYTES
EXPORTED = tuple(_SIGS)


class QuarotError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, 'unknown status')} (status {status})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads libquarot.so (once) and declares the ABI signatures."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise QuarotError(6, f"libquarot.so not found at {p}; build it with "
                             "w4a4_rotated_quantized_gb300.build.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != QUAROT_OK:
        raise QuarotError(status, where)


def _stream(stream, dev):
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, dev=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise QuarotError(1, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise QuarotError(1, f"{name} must be {dtype}, got {t.dtype}")
    if dev is not None and t.device != dev:
        raise QuarotError(1, f"{name} is on {t.device}, expected {dev}")
    if not t.is_contiguous():
        raise QuarotError(1, f"{name} must be contiguous")


def _need_rows(t, dtype, name, dev=None) -> int:
    """A 2-D input read row by row: contiguous rows, any row stride >= the
    width (a column slice of a wider tensor).  Returns the row stride in
    elements, the entry points' ld argument."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise QuarotError(1, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise QuarotError(1, f"{name} must be {dtype}, got {t.dtype}")
    if dev is not None and t.device != dev:
        raise QuarotError(1, f"{name} is on {t.device}, expected {dev}")
    if t.dim() != 2:
        raise QuarotError(1, f"{name} must be 2-D")
    if t.shape[0] > 1 and (t.stride(1) != 1 or t.stride(0) < t.shape[1]):
        raise QuarotError(1, f"{name} must have contiguous rows")
    if t.shape[0] <= 1 and t.shape[1] > 1 and t.stride(1) != 1:
        raise QuarotError(1, f"{name} must have contiguous rows")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def quarot_version() -> int:
    return load().quarot_version()


def quarot_check_error(stream=None, device=None) -> None:
    """Synchronizes the stream and raises if a kernel recorded a device-side error."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(load().quarot_check_error(_stream(stream, dev)), "quarot_check_error")


def quarot_selftest_wait(stream=None, device=None) -> None:
    """Launches the bounded-wait self-test (one device thread, about one second);
    the next quarot_check_error() raises QuarotError with QUAROT_ERR_TIMEOUT."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(load().quarot_selftest_wait(_stream(stream, dev)), "quarot_selftest_wait")


def _rotate_quant_outputs(x, signs, q_out, scale_out, rot_out, want_rot):
    _need_rows(x, torch.float16, "x")
    dev = x.device
    M, d = x.shape
    if signs is not None:
        _need(signs, torch.int8, "signs", dev)
    if q_out is None:
        q_out = torch.empty((M, d // 2), dtype=torch.uint8, device=dev)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float16, device=dev)
    if rot_out is None and want_rot:
        rot_out = torch.empty((M, d), dtype=torch.float32, device=dev)
    _need(q_out, torch.uint8, "q_out", dev)
    _need(scale_out, torch.float16, "scale_out", dev)
    if rot_out is not None:
        _need(rot_out, torch.float32, "rot_out", dev)
    return q_out, scale_out, rot_out


def quarot_rmsnorm_rotate_quant(x, signs=None, eps: float = 1e-6, clip_ratio: float = 1.0, q_out=None,
                                scale_out=None, rot_out=None, stream=None, want_rot: bool = False):
    """x: fp16 [M, d] -> RMSNorm (scale-free), rotation and INT4 quantization in
    one kernel: (packed uint8 [M, d/2], scale fp16 [M], rotated fp32 [M, d] or None)."""
    q_out, scale_out, rot_out = _rotate_quant_outputs(x, signs, q_out, scale_out, rot_out, want_rot)
    M, d = x.shape
    st = load().quarot_rmsnorm_rotate_quant(_ptr(x), M, d, _need_rows(x, torch.float16, "x"), float(eps), _ptr(signs), float(clip_ratio),
                                            _ptr(q_out), _ptr(scale_out), _ptr(rot_out), _stream(stream, x.device))
    _check(st, "quarot_rmsnorm_rotate_quant")
    return q_out, scale_out, rot_out


def quarot_crosshead_rotate_quant(z, nh: int, clip_ratio: float = 1.0, q_out=None, scale_out=None, rot_out=None,
                                  stream=None, want_rot: bool = False):
    """z fp16 [M, nh * dh] (or [M, nh, dh]) -> cross-head Hadamard + INT4:
    (packed uint8 [M, d/2], scale fp16 [M], rotated fp32 [M, d] or None)."""
    if z.dim() == 3:
        z = z.reshape(z.shape[0], -1)
    q_out, scale_out, rot_out = _rotate_quant_outputs(z, None, q_out, scale_out, rot_out, want_rot)
    M, d = z.shape
    if d % nh:
        raise QuarotError(1, "row width is not a multiple of nh")
    st = load().quarot_crosshead_rotate_quant(_ptr(z), M, int(nh), d // int(nh), _need_rows(z, torch.float16, "z"), float(clip_ratio), _ptr(q_out),
                                              _ptr(scale_out), _ptr(rot_out), _stream(stream, z.device))
    _check(st, "quarot_crosshead_rotate_quant")
    return q_out, scale_out, rot_out


def quarot_rotate_quant(x, signs=None, clip_ratio: float = 1.0, q_out=None, scale_out=None, rot_out=None,
                        stream=None, want_rot: bool = False):
    """x: fp16 [M, d], rows contiguous (any row stride) -> (packed uint8 [M, d/2],
    scale fp16 [M], rotated fp32 [M, d] or None)."""
    ld = _need_rows(x, torch.float16, "x")
    dev = x.device
    M, d = x.shape
    if signs is not None:
        _need(signs, torch.int8, "signs", dev)
    if q_out is None:
        q_out = torch.empty((M, d // 2), dtype=torch.uint8, device=dev)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float16, device=dev)
    if rot_out is None and want_rot:
        rot_out = torch.empty((M, d), dtype=torch.float32, device=dev)
    _need(q_out, torch.uint8, "q_out", dev)
    _need(scale_out, torch.float16, "scale_out", dev)
    if rot_out is not None:
        _need(rot_out, torch.float32, "rot_out", dev)
    st = load().quarot_rotate_quant(_ptr(x), M, d, ld, _ptr(signs), float(clip_ratio), _ptr(q_out),
                                    _ptr(scale_out), _ptr(rot_out), _stream(stream, dev))
    _check(st, "quarot_rotate_quant")
    return q_out, scale_out, rot_out


def quarot_rotate_quant_fp16(x, signs=None, clip_ratio: float = 1.0, q_out=None, scale_out=None, rot_out=None,
                             stream=None, want_rot: bool = False):
    """quarot_rotate_quant with the rotation in fp16 arithmetic (the pages'
    FP16 online-Hadamard variant); rot_out receives the fp16 values as fp32."""
    q_out, scale_out, rot_out = _rotate_quant_outputs(x, signs, q_out, scale_out, rot_out, want_rot)
    M, d = x.shape
    st = load().quarot_rotate_quant_fp16(_ptr(x), M, d, _need_rows(x, torch.float16, "x"), _ptr(signs), float(clip_ratio), _ptr(q_out),
                                         _ptr(scale_out), _ptr(rot_out), _stream(stream, x.device))
    _check(st, "quarot_rotate_quant_fp16")
    return q_out, scale_out, rot_out


def quarot_w4a4_gemm(a_q, a_scale, w_q, w_scale, y=None, acc_out=None, stream=None, want_acc: bool = False):
    """a_q uint8 [M, K/2], w_q uint8 [N, K/2] -> (y fp16 [M, N], acc int32 [M, N] or None)."""
    _need(a_q, torch.uint8, "a_q")
    dev = a_q.device
    _need(w_q, torch.uint8, "w_q", dev)
    _need(a_scale, torch.float16, "a_scale", dev)
    _need(w_scale, torch.float16, "w_scale", dev)
    M, Kh = a_q.shape
    N, Kh2 = w_q.shape
    if Kh != Kh2:
        raise QuarotError(1, "a_q and w_q disagree on K")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
    if acc_out is None and want_acc:
        acc_out = torch.empty((M, N), dtype=torch.int32, device=dev)
    _need(y, torch.float16, "y", dev)
    if acc_out is not None:
        _need(acc_out, torch.int32, "acc_out", dev)
    st = load().quarot_w4a4_gemm(_ptr(a_q), _ptr(a_scale), _ptr(w_q), _ptr(w_scale), M, N, 2 * Kh, _ptr(y),
                                 _ptr(acc_out), _stream(stream, dev))
    _check(st, "quarot_w4a4_gemm")
    return y, acc_out


def quarot_rotate_quant_a8(x, signs=None, clip_ratio: float = 1.0, a8_out=None, scale_out=None, rowsum_out=None,
                           stream=None):
    """x: fp16 [M, d] (d = 4096 or 12288) -> the codes in tensor-core operand
    form: (uint8 [M, d] offset codes in the GEMM's K order, scale fp16 [M],
    row code sums int32 [M])."""
    ld = _need_rows(x, torch.float16, "x")
    dev = x.device
    M, d = x.shape
    if signs is not None:
        _need(signs, torch.int8, "signs", dev)
    if a8_out is None:
        a8_out = torch.empty((M, d), dtype=torch.uint8, device=dev)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float16, device=dev)
    if rowsum_out is None:
        rowsum_out = torch.empty((M,), dtype=torch.int32, device=dev)
    _need(a8_out, torch.uint8, "a8_out", dev)
    _need(scale_out, torch.float16, "scale_out", dev)
    _need(rowsum_out, torch.int32, "rowsum_out", dev)
    st = load().quarot_rotate_quant_a8(_ptr(x), M, d, ld, _ptr(signs), float(clip_ratio), _ptr(a8_out),
                                       _ptr(scale_out), _ptr(rowsum_out), _stream(stream, dev))
    _check(st, "quarot_rotate_quant_a8")
    return a8_out, scale_out, rowsum_out


def quarot_w4a4_gemm_a8(a8, a_rowsum, a_scale, w_q, w_scale, y=None, acc_out=None, stream=None,
                        want_acc: bool = False):
    """a8 uint8 [M, K] (quarot_rotate_quant_a8 form), w_q uint8 [N, K/2] ->
    (y fp16 [M, N], acc int32 [M, N] or None)."""
    _need(a8, torch.uint8, "a8")
    dev = a8.device
    _need(a_rowsum, torch.int32, "a_rowsum", dev)
    _need(w_q, torch.uint8, "w_q", dev)
    _need(a_scale, torch.float16, "a_scale", dev)
    _need(w_scale, torch.float16, "w_scale", dev)
    M, K = a8.shape
    N, Kh = w_q.shape
    if K != 2 * Kh:
        raise QuarotError(1, "a8 and w_q disagree on K")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
    if acc_out is None and want_acc:
        acc_out = torch.empty((M, N), dtype=torch.int32, device=dev)
    _need(y, torch.float16, "y", dev)
    if acc_out is not None:
        _need(acc_out, torch.int32, "acc_out", dev)
    st = load().quarot_w4a4_gemm_a8(_ptr(a8), _ptr(a_rowsum), _ptr(a_scale), _ptr(w_q), _ptr(w_scale), M, N, K,
                                    _ptr(y), _ptr(acc_out), _stream(stream, dev))
    _check(st, "quarot_w4a4_gemm_a8")
    return y, acc_out


def quarot_rotate_quant_rowsum(x, signs=None, clip_ratio: float = 1.0, q_out=None, scale_out=None, rowsum_out=None,
                               stream=None):
    """x: fp16 [M, d] (d = 4096 or 12288), rows contiguous -> (packed uint8
    [M, d/2], scale fp16 [M], row code sums int32 [M])."""
    ld = _need_rows(x, torch.float16, "x")
    dev = x.device
    M, d = x.shape
    if signs is not None:
        _need(signs, torch.int8, "signs", dev)
    if q_out is None:
        q_out = torch.empty((M, d // 2), dtype=torch.uint8, device=dev)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float16, device=dev)
    if rowsum_out is None:
        rowsum_out = torch.empty((M,), dtype=torch.int32, device=dev)
    _need(q_out, torch.uint8, "q_out", dev)
    _need(scale_out, torch.float16, "scale_out", dev)
    _need(rowsum_out, torch.int32, "rowsum_out", dev)
    st = load().quarot_rotate_quant_rowsum(_ptr(x), M, d, ld, _ptr(signs), float(clip_ratio), _ptr(q_out),
                                           _ptr(scale_out), _ptr(rowsum_out), _stream(stream, dev))
    _check(st, "quarot_rotate_quant_rowsum")
    return q_out, scale_out, rowsum_out


def quarot_int4_rowsum(q, rowsum_out=None, stream=None):
    """q: packed uint8 [M, K/2] -> row code sums int32 [M]."""
    _need(q, torch.uint8, "q")
    M, Kh = q.shape
    if rowsum_out is None:
        rowsum_out = torch.empty((M,), dtype=torch.int32, device=q.device)
    _need(rowsum_out, torch.int32, "rowsum_out", q.device)
    st = load().quarot_int4_rowsum(_ptr(q), M, 2 * Kh, _ptr(rowsum_out), _stream(stream, q.device))
    _check(st, "quarot_int4_rowsum")
    return rowsum_out


def quarot_w4a4_gemm_rowsums(a_q, a_scale, a_rowsum, w_q, w_scale, w_rowsum, y=None, acc_out=None, stream=None,
                             want_acc: bool = False):
    """quarot_w4a4_gemm with both operands' row code sums given (int32 [M]
    and [N]) -> (y fp16 [M, N], acc int32 [M, N] or None)."""
    _need(a_q, torch.uint8, "a_q")
    dev = a_q.device
    _need(w_q, torch.uint8, "w_q", dev)
    _need(a_scale, torch.float16, "a_scale", dev)
    _need(w_scale, torch.float16, "w_scale", dev)
    _need(a_rowsum, torch.int32, "a_rowsum", dev)
    _need(w_rowsum, torch.int32, "w_rowsum", dev)
    M, Kh = a_q.shape
    N, Kh2 = w_q.shape
    if Kh != Kh2:
        raise QuarotError(1, "a_q and w_q disagree on K")
    if a_rowsum.numel() != M or w_rowsum.numel() != N:
        raise QuarotError(1, "row sums must have M and N entries")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
    if acc_out is None and want_acc:
        acc_out = torch.empty((M, N), dtype=torch.int32, device=dev)
    _need(y, torch.float16, "y", dev)
    if acc_out is not None:
        _need(acc_out, torch.int32, "acc_out", dev)
    st = load().quarot_w4a4_gemm_rowsums(_ptr(a_q), _ptr(a_scale), _ptr(a_rowsum), _ptr(w_q), _ptr(w_scale),
                                         _ptr(w_rowsum), M, N, 2 * Kh, _ptr(y), _ptr(acc_out), _stream(stream, dev))
    _check(st, "quarot_w4a4_gemm_rowsums")
    return y, acc_out


def quarot_w4a4_gemm_plan(M: int, N: int, K: int, sms: int) -> tuple[int, int]:
    """(form, bn): the kernel quarot_w4a4_gemm launches for M x N x K on a GPU
    with `sms` SMs (2 = CTA pair, 1 = one SM) and its N-tile width."""
    form, bn = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().quarot_w4a4_gemm_plan(M, N, K, sms, ctypes.byref(form), ctypes.byref(bn)), "quarot_w4a4_gemm_plan")
    return form.value, bn.value


def quarot_legacy_imma_probe(bits: int, iters: int, sink, stream=None) -> int:
    """Launches the mma.sync integer-rate probe on `stream`; returns the integer
    operations the launch performs.  `sink` is an int32 CUDA tensor."""
    _need(sink, torch.int32, "sink")
    ops = ctypes.c_int64(0)
    _check(load().quarot_legacy_imma_probe(int(bits), int(iters), _ptr(sink), ctypes.byref(ops),
                                           _stream(stream, sink.device)), "quarot_legacy_imma_probe")
    return ops.value


def quarot_kv_write(k, v, t_start, k_q, k_s, v_q, v_s, stream=None):
    """k, v fp16 [B, T_new, Hkv, d] appended at t_start into caches [B, Hkv, T_max, d/2] (+ scales)."""
    _need(k, torch.float16, "k")
    dev = k.device
    _need(v, torch.float16, "v", dev)
    for t, n in ((k_q, "k_q"), (v_q, "v_q")):
        _need(t, torch.uint8, n, dev)
    for t, n in ((k_s, "k_s"), (v_s, "v_s")):
        _need(t, torch.float16, n, dev)
    B, T_new, Hkv, d = k.shape
    if tuple(v.shape) != tuple(k.shape):
        raise QuarotError(1, "k and v shapes differ")
    T_max = k_q.shape[2]
    st = load().quarot_kv_write(_ptr(k), _ptr(v), B, T_new, Hkv, d, int(t_start), T_max, _ptr(k_q), _ptr(k_s),
                                _ptr(v_q), _ptr(v_s), _stream(stream, dev))
    _check(st, "quarot_kv_write")


def quarot_decode_workspace_bytes(B: int, Hq: int, d: int, T: int) -> int:
    return int(load().quarot_decode_workspace_bytes(B, Hq, d, T))


def quarot_decode_attn(q, k_q, k_s, v_q, v_s, T: int, sm_scale: float = 0.0, unrotate_out: bool = False,
                       out=None, workspace=None, stream=None):
    """q fp16 [B, Hq, d] against the first T cached tokens -> out fp16 [B, Hq, d]."""
    _need(q, torch.float16, "q")
    dev = q.device
    for t, n in ((k_q, "k_q"), (v_q, "v_q")):
        _need(t, torch.uint8, n, dev)
    for t, n in ((k_s, "k_s"), (v_s, "v_s")):
        _need(t, torch.float16, n, dev)
    B, Hq, d = q.shape
    Hkv, T_max = k_q.shape[1], k_q.shape[2]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    _need(out, torch.float16, "out", dev)
    need = quarot_decode_workspace_bytes(B, Hq, d, T)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    st = load().quarot_decode_attn(_ptr(q), _ptr(k_q), _ptr(k_s), _ptr(v_q), _ptr(v_s), B, Hq, Hkv, d, int(T),
                                   T_max, float(sm_scale), int(bool(unrotate_out)), _ptr(out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check(st, "quarot_decode_attn")
    return out


def quarot_decode_attn_static(q, k_q, k_s, v_q, v_s, T: int, sm_scale: float = 0.0, unrotate_out: bool = False,
                              out=None, stream=None):
    """quarot_decode_attn without a workspace argument: the scratch is the
    library's fixed device array, so the call itself allocates nothing (pass
    ``out`` to avoid the only torch allocation here).  For callers that cannot
    allocate device memory when they run decode."""
    _need(q, torch.float16, "q")
    dev = q.device
    for t, n in ((k_q, "k_q"), (v_q, "v_q")):
        _need(t, torch.uint8, n, dev)
    for t, n in ((k_s, "k_s"), (v_s, "v_s")):
        _need(t, torch.float16, n, dev)
    B, Hq, d = q.shape
    Hkv, T_max = k_q.shape[1], k_q.shape[2]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    _need(out, torch.float16, "out", dev)
    st = load().quarot_decode_attn_static(_ptr(q), _ptr(k_q), _ptr(k_s), _ptr(v_q), _ptr(v_s), B, Hq, Hkv, d,
                                          int(T), T_max, float(sm_scale), int(bool(unrotate_out)), _ptr(out),
                                          _stream(stream, dev))
    _check(st, "quarot_decode_attn_static")
    return out


def quarot_prefill_attn(q, k_q, k_s, v_q, v_s, sm_scale: float = 0.0, causal: bool = True, out=None,
                        stream=None):
    """Prompt queries q fp16 [B, T, Hq, d] against cached tokens 0 .. T-1
    ("Init") -> out fp16 [B, T, Hq, d] in the rotated basis."""
    _need(q, torch.float16, "q")
    dev = q.device
    for t, n in ((k_q, "k_q"), (v_q, "v_q")):
        _need(t, torch.uint8, n, dev)
    for t, n in ((k_s, "k_s"), (v_s, "v_s")):
        _need(t, torch.float16, n, dev)
    B, T, Hq, d = q.shape
    Hkv, T_max = k_q.shape[1], k_q.shape[2]
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=torch.float16, device=dev)
    _need(out, torch.float16, "out", dev)
    st = load().quarot_prefill_attn(_ptr(q), _ptr(k_q), _ptr(k_s), _ptr(v_q), _ptr(v_s), B, Hq, Hkv, d, T, T_max,
                                    float(sm_scale), int(bool(causal)), _ptr(out), _stream(stream, dev))
    _check(st, "quarot_prefill_attn")
    return out


class QuarotLinear:
    """The QuaRot W4A4 linear layer, y = x W^T in the rotated INT4 domain
    ([G] "End-to-End Implementation", [S] Stages 1a, 2a, 2b): at
    construction the weight rows are rotated by diag(s) H / sqrt(K) and
    quantized per output channel (quarot_rotate_quant on the rows); each call
    rotates and quantizes the tokens the same way (per token) and runs
    quarot_w4a4_gemm.  weight: fp16 [N, K] on the GPU, K a supported rotation
    width; signs: int8 [K] of +-1 or None; x: fp16 [..., K] -> fp16 [..., N].
    No bias: the layer is the hot path's two kernels and nothing else."""

    def __init__(self, weight, signs=None, clip_ratio: float = 1.0, weight_clip_ratio: float = 1.0, stream=None):
        ld = _need_rows(weight, torch.float16, "weight")
        del ld
        self.out_features, self.in_features = weight.shape
        self.signs = signs
        self.clip_ratio = float(clip_ratio)
        self.w_q, self.w_scale, _ = quarot_rotate_quant(weight, signs, clip_ratio=weight_clip_ratio, stream=stream)
        # widths whose quantizer also writes the row code sums: the GEMM then
        # takes both operands' sums instead of forming them while unpacking
        self.rowsums = self.in_features in (4096, 12288)
        self.w_rowsum = quarot_int4_rowsum(self.w_q, stream=stream) if self.rowsums else None

    def __call__(self, x, y=None, stream=None):
        if x.shape[-1] != self.in_features:
            raise QuarotError(1, f"x has {x.shape[-1]} features, the layer {self.in_features}")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features)
        if y is not None:
            y = y.view(-1, self.out_features)
        if self.rowsums:
            a_q, a_scale, a_rs = quarot_rotate_quant_rowsum(x2, self.signs, clip_ratio=self.clip_ratio, stream=stream)
            y, _ = quarot_w4a4_gemm_rowsums(a_q, a_scale, a_rs, self.w_q, self.w_scale, self.w_rowsum, y=y,
                                            stream=stream)
        else:
            a_q, a_scale, _ = quarot_rotate_quant(x2, self.signs, clip_ratio=self.clip_ratio, stream=stream)
            y, _ = quarot_w4a4_gemm(a_q, a_scale, self.w_q, self.w_scale, y=y, stream=stream)
        return y.view(*lead, self.out_features)


class QuarotKVCache:
    """The rotated INT4 KV cache of B sequences, Hkv heads of width d, room
    for T_max tokens ([S] Stage 2c, Append / Decode / Init routines):
    ``append`` quantizes new tokens into positions length .. length + T_new - 1
    (quarot_kv_write, or quarot_kv_write_asym for the asymmetric cache);
    ``decode`` attends one query token per sequence over the cached tokens
    (quarot_decode_attn / _asym, with a workspace sized once for T_max);
    ``prefill`` runs the prompt attention of length query tokens over them
    (quarot_prefill_attn, symmetric cache).  Queries and outputs stay in the
    rotated head basis unless unrotate_out is set."""

    def __init__(self, B: int, Hkv: int, T_max: int, d: int = 128, device=None, asym: bool = False,
                 clip_ratio: float = 0.95):
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.B, self.Hkv, self.T_max, self.d = int(B), int(Hkv), int(T_max), int(d)
        self.asym, self.clip_ratio = bool(asym), float(clip_ratio)
        self.tensors = (new_kv_cache_asym if self.asym else new_kv_cache)(self.B, self.Hkv, self.T_max, self.d, device)
        self.length = 0
        self._ws = {}

    def append(self, k, v, stream=None) -> None:
        """k, v fp16 [B, T_new, Hkv, d]."""
        T_new = int(k.shape[1])
        if self.length + T_new > self.T_max:
            raise QuarotError(1, f"cache holds {self.T_max} tokens; {self.length} + {T_new} do not fit")
        if self.asym:
            quarot_kv_write_asym(k, v, self.length, *self.tensors, clip_ratio=self.clip_ratio, stream=stream)
        else:
            quarot_kv_write(k, v, self.length, *self.tensors, stream=stream)
        self.length += T_new

    def decode(self, q, sm_scale: float = 0.0, unrotate_out: bool = False, out=None, stream=None):
        """q fp16 [B, Hq, d] -> fp16 [B, Hq, d] over the length cached tokens."""
        Hq = int(q.shape[1])
        ws = self._ws.get(Hq)
        if ws is None:
            need = quarot_decode_workspace_bytes(self.B, Hq, self.d, self.T_max)
            ws = self._ws[Hq] = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
        fn = quarot_decode_attn_asym if self.asym else quarot_decode_attn
        return fn(q, *self.tensors, T=self.length, sm_scale=sm_scale, unrotate_out=unrotate_out, out=out,
                  workspace=ws, stream=stream)

    def prefill(self, q, sm_scale: float = 0.0, causal: bool = True, out=None, stream=None):
        """q fp16 [B, length, Hq, d] -> fp16 [B, length, Hq, d]."""
        if self.asym:
            raise QuarotError(2, "prompt attention reads the symmetric cache only")
        if int(q.shape[1]) != self.length:
            raise QuarotError(1, f"{q.shape[1]} query tokens for {self.length} cached tokens")
        return quarot_prefill_attn(q, *self.tensors, sm_scale=sm_scale, causal=causal, out=out, stream=stream)


def new_kv_cache(B: int, Hkv: int, T_max: int, d: int, device):
    """Zeroed caches (k_q, k_s, v_q, v_s) in the layout quarot_kv_write expects."""
    kq = torch.zeros((B, Hkv, T_max, d // 2), dtype=torch.uint8, device=device)
    vq = torch.zeros_like(kq)
    ks = torch.zeros((B, Hkv, T_max), dtype=torch.float16, device=device)
    vs = torch.zeros_like(ks)
    return kq, ks, vq, vs


def new_kv_cache_asym(B: int, Hkv: int, T_max: int, d: int, device):
    """Zeroed asymmetric caches (k_q, k_s, k_z, v_q, v_s, v_z): unsigned codes,
    fp16 scales, int16 zero points, in the layout quarot_kv_write_asym expects."""
    kq = torch.zeros((B, Hkv, T_max, d // 2), dtype=torch.uint8, device=device)
    ks = torch.zeros((B, Hkv, T_max), dtype=torch.float16, device=device)
    kz = torch.zeros((B, Hkv, T_max), dtype=torch.int16, device=device)
    return kq, ks, kz, torch.zeros_like(kq), torch.zeros_like(ks), torch.zeros_like(kz)


def quarot_kv_write_asym(k, v, t_start, k_q, k_s, k_z, v_q, v_s, v_z, clip_ratio: float = 0.95, stream=None):
    """Append with the asymmetric per-group quantizer (group = head vector)."""
    _need(k, torch.float16, "k")
    dev = k.device
    _need(v, torch.float16, "v", dev)
    for t_, n in ((k_q, "k_q"), (v_q, "v_q")):
        _need(t_, torch.uint8, n, dev)
    for t_, n in ((k_s, "k_s"), (v_s, "v_s")):
        _need(t_, torch.float16, n, dev)
    for t_, n in ((k_z, "k_z"), (v_z, "v_z")):
        _need(t_, torch.int16, n, dev)
    B, T_new, Hkv, d = k.shape
    if tuple(v.shape) != tuple(k.shape):
        raise QuarotError(1, "k and v shapes differ")
    T_max = k_q.shape[2]
    st = load().quarot_kv_write_asym(_ptr(k), _ptr(v), B, T_new, Hkv, d, int(t_start), T_max, float(clip_ratio),
                                     _ptr(k_q), _ptr(k_s), _ptr(k_z), _ptr(v_q), _ptr(v_s), _ptr(v_z),
                                     _stream(stream, dev))
    _check(st, "quarot_kv_write_asym")


def quarot_decode_attn_asym(q, k_q, k_s, k_z, v_q, v_s, v_z, T: int, sm_scale: float = 0.0,
                            unrotate_out: bool = False, out=None, workspace=None, stream=None):
    """quarot_decode_attn over the asymmetric cache -> out fp16 [B, Hq, d]."""
    _need(q, torch.float16, "q")
    dev = q.device
    for t_, n in ((k_q, "k_q"), (v_q, "v_q")):
        _need(t_, torch.uint8, n, dev)
    for t_, n in ((k_s, "k_s"), (v_s, "v_s")):
        _need(t_, torch.float16, n, dev)
    for t_, n in ((k_z, "k_z"), (v_z, "v_z")):
        _need(t_, torch.int16, n, dev)
    B, Hq, d = q.shape
    Hkv, T_max = k_q.shape[1], k_q.shape[2]
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    _need(out, torch.float16, "out", dev)
    need = quarot_decode_workspace_bytes(B, Hq, d, T)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    st = load().quarot_decode_attn_asym(_ptr(q), _ptr(k_q), _ptr(k_s), _ptr(k_z), _ptr(v_q), _ptr(v_s), _ptr(v_z),
                                        B, Hq, Hkv, d, int(T), T_max, float(sm_scale), int(bool(unrotate_out)),
                                        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream, dev))
    _check(st, "quarot_decode_attn_asym")
    return out
