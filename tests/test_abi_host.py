"""Host-side checks of the C ABI: the library builds, loads, exports every
function include/quarot.h declares, and rejects bad arguments before any
launch (no GPU is touched by these calls)."""
import ctypes
import os
import re

import pytest
import torch

import __graft_entry__
import w4a4_rotated_quantized_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return q.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "quarot.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(quarot_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert sorted(q.EXPORTED) == _declared()


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        s = lib.quarot_status_string(code)
        assert s and s.decode() == q.STATUS[code]
    assert lib.quarot_status_string(99) == b"unknown status"
    assert lib.quarot_version() >> 16 == 1 and lib.quarot_version() & 0xFFFF >= 1


P = ctypes.c_void_p
FAKE = P(0x10000)  # never dereferenced: every call below fails validation first


def test_rotate_quant_validation(lib):
    f = lib.quarot_rotate_quant
    assert f(FAKE, 0, 4096, 4096, None, 1.0, FAKE, FAKE, None, None) == 0  # M = 0 no-op
    assert f(FAKE, 4, 24, 24, None, 1.0, FAKE, FAKE, None, None) == 2  # no construction for 24
    assert f(FAKE, 4, 20, 20, None, 1.0, FAKE, FAKE, None, None) == 3  # ld % 8
    assert f(FAKE, -1, 4096, 4096, None, 1.0, FAKE, FAKE, None, None) == 1
    assert f(FAKE, 4, 4096, 4000, None, 1.0, FAKE, FAKE, None, None) == 1  # ld < d
    assert f(FAKE, 4, 4096, 4096, None, 0.0, FAKE, FAKE, None, None) == 1  # clip
    assert f(FAKE, 4, 4096, 4096, None, 1.5, FAKE, FAKE, None, None) == 1
    assert f(None, 4, 4096, 4096, None, 1.0, FAKE, FAKE, None, None) == 1
    assert f(P(0x10002), 4, 4096, 4096, None, 1.0, FAKE, FAKE, None, None) == 3  # misaligned x
    assert f(FAKE, 4, 4096, 4100, None, 1.0, FAKE, FAKE, None, None) == 3  # ld % 8
    assert f(FAKE, 4, 4104, 4104, None, 1.0, FAKE, FAKE, None, None) == 2  # no construction


def test_rotate_quant_fp16_validation(lib):
    f = lib.quarot_rotate_quant_fp16
    assert f(FAKE, 0, 4096, 4096, None, 1.0, FAKE, FAKE, None, None) == 0  # M = 0 no-op
    assert f(FAKE, 4, 24, 24, None, 1.0, FAKE, FAKE, None, None) == 2  # no construction for 24
    assert f(FAKE, 4, 4096, 4000, None, 1.0, FAKE, FAKE, None, None) == 1  # ld < d
    assert f(FAKE, 4, 4096, 4096, None, 0.0, FAKE, FAKE, None, None) == 1  # clip
    assert f(None, 4, 4096, 4096, None, 1.0, FAKE, FAKE, None, None) == 1
    assert f(P(0x10002), 4, 4096, 4096, None, 1.0, FAKE, FAKE, None, None) == 3  # misaligned x
    assert f(FAKE, 4, 4096, 4100, None, 1.0, FAKE, FAKE, None, None) == 3  # ld % 8


def test_rmsnorm_rotate_quant_validation(lib):
    f = lib.quarot_rmsnorm_rotate_quant
    assert f(FAKE, 0, 4096, 4096, 1e-6, None, 1.0, FAKE, FAKE, None, None) == 0  # M = 0 no-op
    assert f(FAKE, 4, 4096, 4096, 0.0, None, 1.0, FAKE, FAKE, None, None) == 1  # eps must be > 0
    assert f(FAKE, 4, 4096, 4096, -1.0, None, 1.0, FAKE, FAKE, None, None) == 1
    assert f(FAKE, 4, 4096, 4096, float("nan"), None, 1.0, FAKE, FAKE, None, None) == 1
    assert f(FAKE, 4, 4096, 4096, float("inf"), None, 1.0, FAKE, FAKE, None, None) == 1
    assert f(FAKE, 4, 24, 24, 1e-6, None, 1.0, FAKE, FAKE, None, None) == 2  # no construction for 24
    assert f(FAKE, 4, 4096, 4096, 1e-6, None, 1.5, FAKE, FAKE, None, None) == 1  # clip
    assert f(P(0x10002), 4, 4096, 4096, 1e-6, None, 1.0, FAKE, FAKE, None, None) == 3  # misaligned x


def test_gemm_validation(lib):
    f = lib.quarot_w4a4_gemm
    assert f(FAKE, FAKE, FAKE, FAKE, 0, 16, 256, FAKE, None, None) == 0
    assert f(FAKE, FAKE, FAKE, FAKE, 16, 16, 200, FAKE, None, None) == 2  # K % 128
    assert f(FAKE, FAKE, FAKE, FAKE, 16, 16, 131072, FAKE, None, None) == 2  # K too large for exact fp32
    assert f(FAKE, FAKE, FAKE, FAKE, -1, 16, 256, FAKE, None, None) == 1
    assert f(None, FAKE, FAKE, FAKE, 16, 16, 256, FAKE, None, None) == 1
    assert f(P(0x10008), FAKE, FAKE, FAKE, 16, 16, 256, FAKE, None, None) == 3


def test_kv_validation(lib):
    f = lib.quarot_kv_write
    assert f(FAKE, FAKE, 1, 4, 8, 128, 14, 16, FAKE, FAKE, FAKE, FAKE, None) == 1  # past T_max
    assert f(FAKE, FAKE, 1, 4, 8, 96, 0, 16, FAKE, FAKE, FAKE, FAKE, None) == 2
    assert f(FAKE, FAKE, 0, 4, 8, 128, 0, 16, FAKE, FAKE, FAKE, FAKE, None) == 0
    d = lib.quarot_decode_attn
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 64, 4, 8, 0.0, 0, FAKE, FAKE, 1 << 20, None) == 2
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 30, 8, 128, 4, 8, 0.0, 0, FAKE, FAKE, 1 << 20, None) == 1
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 128, 9, 8, 0.0, 0, FAKE, FAKE, 1 << 20, None) == 1
    assert d(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 128, 4, 8, 0.0, 0, FAKE, FAKE, 16, None) == 1  # small ws


def test_kv_asym_validation(lib):
    w = lib.quarot_kv_write_asym
    assert w(FAKE, FAKE, 0, 1, 8, 128, 0, 16, 0.95, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 0  # B = 0
    assert w(FAKE, FAKE, 1, 1, 8, 128, 0, 16, 0.0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1  # clip
    assert w(FAKE, FAKE, 1, 1, 8, 128, 0, 16, 1.5, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert w(FAKE, FAKE, 1, 1, 8, 96, 0, 16, 0.95, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 2  # d
    assert w(FAKE, FAKE, 1, 1, 8, 128, 0, 16, 0.95, FAKE, FAKE, None, FAKE, FAKE, FAKE, None) == 1  # no k_z
    assert w(FAKE, FAKE, 1, 1, 8, 128, 0, 16, 0.95, FAKE, FAKE, P(0x10001), FAKE, FAKE, FAKE, None) == 3
    assert w(FAKE, FAKE, 1, 4, 8, 128, 14, 16, 0.95, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1  # overflow
    a = lib.quarot_decode_attn_asym
    assert a(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 32, 8, 128, 16, 16, 0.0, 0, FAKE, FAKE, 0, None) == 0
    assert a(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 64, 16, 16, 0.0, 0, FAKE, FAKE, 1 << 20, None) == 2
    assert a(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 1, 32, 8, 128, 16, 16, 0.0, 0, FAKE, FAKE, 1 << 20,
             None) == 1  # no k_z
    assert a(FAKE, FAKE, FAKE, P(0x10001), FAKE, FAKE, FAKE, 1, 32, 8, 128, 16, 16, 0.0, 0, FAKE, P(0x10000),
             1 << 20, None) == 3  # misaligned k_z
    assert a(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 30, 8, 128, 16, 16, 0.0, 0, FAKE, FAKE, 1 << 20, None) == 1


def test_prefill_validation(lib):
    f = lib.quarot_prefill_attn
    args = [FAKE] * 5
    assert f(*args, 0, 32, 8, 128, 16, 16, 0.0, 1, FAKE, None) == 0  # B = 0 no-op
    assert f(*args, 1, 32, 8, 128, 0, 16, 0.0, 1, FAKE, None) == 0  # T = 0 no-op
    assert f(*args, 1, 32, 8, 64, 16, 16, 0.0, 1, FAKE, None) == 2  # d
    assert f(*args, 1, 48, 4, 128, 16, 16, 0.0, 1, FAKE, None) == 2  # group of 12
    assert f(*args, 1, 30, 8, 128, 16, 16, 0.0, 1, FAKE, None) == 1  # Hq % Hkv
    assert f(*args, 1, 32, 8, 128, 17, 16, 0.0, 1, FAKE, None) == 1  # T > T_max
    assert f(*args, 1, 32, 8, 128, 16, 16, 0.0, 2, FAKE, None) == 1  # causal flag
    assert f(*args, -1, 32, 8, 128, 16, 16, 0.0, 1, FAKE, None) == 1
    assert f(FAKE, FAKE, FAKE, None, FAKE, 1, 32, 8, 128, 16, 16, 0.0, 1, FAKE, None) == 1  # no v_q
    assert f(FAKE, P(0x10008), FAKE, FAKE, FAKE, 1, 32, 8, 128, 16, 16, 0.0, 1, FAKE, None) == 3  # k_q % 16
    assert f(P(0x10004), FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 128, 16, 16, 0.0, 1, FAKE, None) == 3  # q % 16
    assert f(*args, 1, 32, 8, 128, 16, 16, 0.0, 1, P(0x10008), None) == 3  # out % 16


def test_crosshead_validation(lib):
    f = lib.quarot_crosshead_rotate_quant
    assert f(FAKE, 0, 32, 128, 4096, 1.0, FAKE, FAKE, None, None) == 0  # M = 0 no-op
    assert f(FAKE, 4, 24, 128, 3072, 1.0, FAKE, FAKE, None, None) == 2  # nh not a power of two
    assert f(FAKE, 4, 128, 128, 16384, 1.0, FAKE, FAKE, None, None) == 2  # nh > 64
    assert f(FAKE, 4, 32, 96, 3072, 1.0, FAKE, FAKE, None, None) == 2  # dh
    assert f(FAKE, 4, 32, 128, 4000, 1.0, FAKE, FAKE, None, None) == 1  # ld < d
    assert f(FAKE, 4, 32, 128, 4096, 0.0, FAKE, FAKE, None, None) == 1  # clip
    assert f(None, 4, 32, 128, 4096, 1.0, FAKE, FAKE, None, None) == 1
    assert f(P(0x10001), 4, 32, 128, 4096, 1.0, FAKE, FAKE, None, None) == 3  # misaligned z
    assert f(FAKE, 4, 32, 128, 4096, 1.0, P(0x10002), FAKE, None, None) == 3  # misaligned q_out


def test_workspace_size(lib):
    assert q.quarot_decode_workspace_bytes(16, 32, 128, 4096) == 16 * 32 * 16 * 130 * 4
    assert q.quarot_decode_workspace_bytes(1, 1, 128, 1) == 768  # 130 floats rounded up to 256 B
    assert q.quarot_decode_workspace_bytes(1, 1, 64, 1) == 0


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(q, "_lib", None)
    with pytest.raises(q.QuarotError):
        q.load("/nonexistent/libquarot.so")


def test_gemm_plan_query(lib):
    """The launch plan (kernel form, N-tile width) as the host computes it for
    a 152-SM GB300: the pair kernel's width and accumulator count minimise
    its modelled time per pair (a tile costs its k-blocks, a drain exposed by
    the one-accumulator form about 5 more; ties go to the narrower width),
    small M takes the one-SM kernel, an odd k-block count the one-SM kernel at
    any M; bad sizes are rejected."""
    assert q.quarot_w4a4_gemm_plan(2048, 4096, 12288, 152) == (2, 224)
    assert q.quarot_w4a4_gemm_plan(8192, 4096, 4096, 152) == (2, 224)  # 8 tiles at 224 beat 10 and 11 narrower
    assert q.quarot_w4a4_gemm_plan(4000, 3000, 256, 152) == (3, 160)  # tied with 192: the narrower
    assert q.quarot_w4a4_gemm_plan(7000, 1000, 256, 152) == (3, 128)  # tied with 160 and 192
    assert q.quarot_w4a4_gemm_plan(1137, 7330, 512, 152) == (3, 192)
    assert q.quarot_w4a4_gemm_plan(2048, 2560, 1024, 152) == (2, 160)
    assert q.quarot_w4a4_gemm_plan(8192, 12288, 4096, 152) == (3, 192)  # 27 tiles per pair at 192
    assert q.quarot_w4a4_gemm_plan(2048, 12288, 4096, 152) == (2, 224)  # 6 x 32 + 5 drains < 7 x 32
    assert q.quarot_w4a4_gemm_plan(512, 12288, 4096, 152) == (2, 192)
    assert q.quarot_w4a4_gemm_plan(16, 256, 256, 152) == (1, 128)
    assert q.quarot_w4a4_gemm_plan(1156, 2888, 128, 152) == (1, 224)
    assert q.quarot_w4a4_gemm_plan(1030, 2568, 384, 152)[0] == 1
    form, bn = ctypes.c_int(0), ctypes.c_int(0)
    f = lib.quarot_w4a4_gemm_plan
    assert f(0, 8, 128, 152, ctypes.byref(form), ctypes.byref(bn)) == 1
    assert f(8, 8, 100, 152, ctypes.byref(form), ctypes.byref(bn)) == 2
    assert f(8, 8, 131072, 152, ctypes.byref(form), ctypes.byref(bn)) == 2
    assert f(8, 8, 128, 152, None, ctypes.byref(bn)) == 1


def test_legacy_probe_validation(lib):
    """The mma.sync rate probe accepts widths 8, 4 and 16 only, and rejects
    bad arguments before touching the device."""
    ops = ctypes.c_int64(0)
    f = lib.quarot_legacy_imma_probe
    for bits in (0, 2, 12, 32):
        assert f(bits, 8, FAKE, ctypes.byref(ops), None) == 1
    assert f(16, 0, FAKE, ctypes.byref(ops), None) == 1
    assert f(16, 8, None, ctypes.byref(ops), None) == 1
    assert f(16, 8, FAKE, None, None) == 1
    assert f(16, 8, P(0x10002), ctypes.byref(ops), None) == 3


def test_a8_validation(lib):
    """The tensor-core operand form of the layer rejects bad arguments before
    any launch: widths other than 4096 / 12288, K not a multiple of 256,
    null and misaligned pointers."""
    f = lib.quarot_rotate_quant_a8
    assert f(FAKE, 0, 4096, 4096, None, 1.0, FAKE, FAKE, FAKE, None) == 0  # M = 0 no-op
    assert f(FAKE, 4, 2048, 2048, None, 1.0, FAKE, FAKE, FAKE, None) == 2
    assert f(FAKE, 4, 4096, 4096, None, 0.0, FAKE, FAKE, FAKE, None) == 1
    assert f(FAKE, 4, 4096, 4096, None, 1.0, FAKE, FAKE, None, None) == 1
    assert f(FAKE, 4, 4096, 4096, None, 1.0, P(0x10008), FAKE, FAKE, None) == 3
    assert f(FAKE, 4, 4096, 4096, None, 1.0, FAKE, FAKE, P(0x10002), None) == 3
    g = lib.quarot_w4a4_gemm_a8
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, 256, FAKE, None, None) == 0  # M = 0 no-op
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 8, 128, FAKE, None, None) == 2  # K % 256
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 8, 131072, FAKE, None, None) == 2
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 8, 256, FAKE, None, None) == 1
    assert g(FAKE, None, FAKE, FAKE, FAKE, 8, 8, 256, FAKE, None, None) == 1
    assert g(FAKE, P(0x10002), FAKE, FAKE, FAKE, 8, 8, 256, FAKE, None, None) == 3
    assert g(P(0x10008), FAKE, FAKE, FAKE, FAKE, 8, 8, 256, FAKE, None, None) == 3


def test_row_strided_views_accepted_and_others_rejected():
    """The binding's row check: a column slice of a wider tensor passes with
    its row stride; a transposed view (non-contiguous rows) is rejected before
    any launch (host only: the check runs before the library is called)."""
    if not torch.cuda.is_available():
        # the check itself needs CUDA tensors; on a CPU-only host assert the
        # CPU-tensor rejection path instead
        with pytest.raises(q.QuarotError):
            q._need_rows(torch.zeros((4, 16), dtype=torch.float16), torch.float16, "x")
        return
    wide = torch.zeros((4, 40), dtype=torch.float16, device="cuda")
    assert q._need_rows(wide[:, 8:24], torch.float16, "x") == 40
    assert q._need_rows(wide[:1, 8:24], torch.float16, "x") == 16
    with pytest.raises(q.QuarotError):
        q._need_rows(wide.t(), torch.float16, "x")


def test_rowsum_entry_points_validate_on_host(lib):
    """The row-sum entry points reject bad arguments before any launch."""
    P = ctypes.c_void_p(16)
    f = lib.quarot_int4_rowsum
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    assert f(P, -1, 128, P, None) == 1
    assert f(P, 4, 100, P, None) == 1          # K % 32
    assert f(None, 4, 128, P, None) == 1
    assert f(ctypes.c_void_p(8), 4, 128, P, None) == 3
    assert f(P, 0, 128, P, None) == 0
    g = lib.quarot_rotate_quant_rowsum
    g.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert g(P, 4, 256, 256, None, 1.0, P, P, P, None) == 2   # width without the sum form
    assert g(P, 4, 4096, 4096, None, 1.0, P, P, None, None) == 1
    h = lib.quarot_w4a4_gemm_rowsums
    h.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 3
    assert h(P, P, None, P, P, P, 256, 256, 256, P, None, None) == 1
    assert h(P, P, P, P, P, ctypes.c_void_p(18), 256, 256, 256, P, None, None) == 3
