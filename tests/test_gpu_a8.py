"""GPU parity of the layer in tensor-core operand form: quarot_rotate_quant_a8
(each INT4 code widened to one byte, u = v + 8, with the row code sums) and
quarot_w4a4_gemm_a8 (activations from that form, weights packed INT4).

Bars: the bytes are the oracle's codes (up to the .5-boundary and fp16-scale
cases of check_quant, which the packed kernel shares) in the documented
order, bit-identical to the packed entry point's codes; the row sums are the
exact sums of those codes; the GEMM's INT32 accumulator is bit-exact against
the oracle's integer GEMM and its fp16 output bit-identical to the oracle's
dequantization (and to quarot_w4a4_gemm on the same codes).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from test_gpu_parity import DEV, OUT_TOL, _t, _tile_rows, check_quant, q  # noqa: F401  (q: fixture)

pytestmark = pytest.mark.gpu

PERM = np.array([0, 2, 4, 6, 1, 3, 5, 7])  # byte j of a group of 8 holds code PERM[j]


def a8_bytes(codes):
    """Natural-order INT4 codes [M, K] -> the operand bytes [M, K]."""
    M, K = codes.shape
    u = (codes.astype(np.int16) + 8).astype(np.uint8)
    return np.ascontiguousarray(u.reshape(M, K // 8, 8)[:, :, PERM].reshape(M, K))


def a8_codes(b):
    """Operand bytes [M, K] -> natural-order INT4 codes [M, K]."""
    M, K = b.shape
    inv = np.argsort(PERM)
    return (b.reshape(M, K // 8, 8)[:, :, inv].reshape(M, K).astype(np.int16) - 8).astype(np.int8)


def test_a8_byte_order_helpers_round_trip():
    c = W.int4_codes(3, 64, 5)
    b = a8_bytes(c)
    assert b.max() <= 15 and np.array_equal(a8_codes(b), c)
    # byte 1 of a group is code 2, byte 4 is code 1
    assert b[0, 1] == c[0, 2] + 8 and b[0, 4] == c[0, 1] + 8


def _check_a8(q, x, s, clip=1.0, rows=None):
    """quarot_rotate_quant_a8 against the oracle and against the packed entry point."""
    xt = _t(x)
    st = None if s is None else _t(s)
    b8, s8, rs = q.quarot_rotate_quant_a8(xt, st, clip_ratio=clip)
    gq, gs, grot = q.quarot_rotate_quant(xt, st, clip_ratio=clip, want_rot=True)
    q.quarot_check_error()
    # the same codes and scales as the packed form, bit for bit, on every row
    assert torch.equal(s8, gs)
    b8n = b8.cpu().numpy()
    codes = a8_codes(b8n)
    assert np.array_equal(codes, O.unpack_int4(gq.cpu().numpy()))
    assert np.array_equal(rs.cpu().numpy(), codes.astype(np.int64).sum(axis=1))
    assert b8n.max() <= 15
    # and the oracle's codes (sampled rows at full size)
    if rows is None:
        rows = np.arange(x.shape[0])
    check_quant(O.pack_int4(codes[rows]), s8.cpu().numpy()[rows], grot.cpu().numpy()[rows],
                O.rotate(x[rows], s), clip=clip)


@pytest.mark.parametrize("d", [4096, 12288])
@pytest.mark.parametrize("signed", [True, False])
def test_rotate_quant_a8_widths(q, d, signed):
    M = 37  # ragged for the two-row CTAs of the 4096 kernel
    x = W.activations(M, d, W.outlier_channels(d, max(1, d // 512), 5 + d), 100.0, 11 + d)
    _check_a8(q, x, W.random_signs(d, 21 + d) if signed else None)


@pytest.mark.parametrize("d", [4096, 12288])
def test_rotate_quant_a8_clip_09_and_one_row(q, d):
    x = W.activations(19, d, [1, 7], 50.0, 3)
    s = W.random_signs(d, 4)
    _check_a8(q, x, s, clip=0.9)
    _check_a8(q, x[:1], s)


def test_rotate_quant_a8_edge_rows(q):
    d = 4096
    x = np.zeros((5, d), dtype=np.float16)
    x[1, 3] = 1.0            # one-hot: every code +-7
    x[2] = 65504.0           # largest fp16: the scale saturates
    x[3, ::2] = -1.0
    x[4] = np.float16(6e-8)  # subnormal inputs
    _check_a8(q, x, None)
    b8, _, rs = q.quarot_rotate_quant_a8(_t(x), None)
    assert np.all(b8.cpu().numpy()[0] == 8) and int(rs[0]) == 0


def test_rotate_quant_a8_down_proj_full(q):
    """2048 x 12288 at full size (persistent CTAs, several rows each): every
    row bit-identical to the packed form, sampled rows against the oracle."""
    x, _, s = W.layer_inputs("down_proj", N=0)
    rows = np.random.default_rng(2).choice(x.shape[0], 32, replace=False)
    rows[:2] = [0, x.shape[0] - 1]
    _check_a8(q, x, s, rows=np.sort(rows))


def test_rotate_quant_a8_empty(q):
    x = torch.empty((0, 4096), dtype=torch.float16, device=DEV)
    b8, s8, rs = q.quarot_rotate_quant_a8(x)
    assert b8.shape == (0, 4096) and rs.shape == (0,)


# ---------------------------------------------------------------- GEMM
def _gemm_a8(q, a, w, sx, sw):
    b = a8_bytes(a)
    rs = a.astype(np.int64).sum(axis=1).astype(np.int32)
    y, acc = q.quarot_w4a4_gemm_a8(_t(b), _t(rs), _t(sx), _t(O.pack_int4(w)), _t(sw), want_acc=True)
    q.quarot_check_error()
    return y, acc


# every shape runs the CTA-pair kernel: ragged M and N tails in either CTA of
# a pair, M below one CTA's 128 rows, N below one tile, K from 256 to 12288
A8_SHAPES = [(1, 8, 256), (16, 256, 256), (200, 300, 256), (257, 513, 512), (256, 512, 4096),
             (130, 264, 12288), (385, 136, 768), (600, 1000, 1024)]


@pytest.mark.parametrize("M,N,K", A8_SHAPES)
def test_gemm_a8_bit_exact(q, M, N, K):
    seed = 500 + M + N + K
    a, w = W.int4_codes(M, K, seed), W.int4_codes(N, K, seed + 1)
    sx, sw = W.fp16_scales(M, seed + 2), W.fp16_scales(N, seed + 3)
    y, acc = _gemm_a8(q, a, w, sx, sw)
    ref = O.int_gemm(a, w)
    assert np.array_equal(acc.cpu().numpy(), ref)
    assert np.array_equal(y.cpu().numpy().view(np.uint16), O.dequant(ref, sx, sw).view(np.uint16))


def _gemm_a8_sampled(q, M, N, K, seed):
    a, w = W.int4_codes(M, K, seed), W.int4_codes(N, K, seed + 1)
    sx, sw = W.fp16_scales(M, seed + 2), W.fp16_scales(N, seed + 3)
    y, acc = _gemm_a8(q, a, w, sx, sw)
    # the packed entry point on the same codes gives the same bytes everywhere
    yp, _ = q.quarot_w4a4_gemm(_t(O.pack_int4(a)), _t(sx), _t(O.pack_int4(w)), _t(sw))
    assert torch.equal(y, yp)
    del yp
    rows = _tile_rows(M, 2, seed)
    ri = torch.from_numpy(rows).to(DEV)
    acc_s = acc.index_select(0, ri).cpu().numpy()
    y_s = y.index_select(0, ri).cpu().numpy()
    del y, acc
    ref = O.int_gemm(a[rows], w)
    assert np.array_equal(acc_s, ref)
    assert np.array_equal(y_s.view(np.uint16), O.dequant(ref, sx[rows], sw).view(np.uint16))


def test_gemm_a8_full_down_proj_sampled(q):
    """2048 x 4096 x 12288 at full size (the bench launch)."""
    _gemm_a8_sampled(q, 2048, 4096, 12288, 1900)


@pytest.mark.parametrize("M", [512, 2048, 8192])
@pytest.mark.parametrize("N", [4096, 12288])
def test_gemm_a8_sweep_shapes(q, M, N):
    """M x 4096 x N at full size: N-tile widths 160, 192 and 224 and many
    tiles per pair, so both accumulators are reused many times."""
    _gemm_a8_sampled(q, M, N, 4096, 5000 + M + N)


@pytest.mark.parametrize("K", [16384, 65536])
def test_gemm_a8_extremes_at_large_k(q, K):
    """All-extreme codes up to the largest K: the offset products and the
    row-sum corrections stay exact in fp32."""
    M, N = 200, 136
    a = np.full((M, K), 7, dtype=np.int8)
    a[1::3] = -8
    a[2::5, ::2] = -7
    w = np.full((N, K), 7, dtype=np.int8)
    w[1::4] = -8
    w[3::7, 1::3] = 6
    y, acc = _gemm_a8(q, a, w, W.fp16_scales(M, 1), W.fp16_scales(N, 2))
    acc = acc.cpu().numpy()
    assert np.array_equal(acc, O.int_gemm(a, w))
    assert acc[0, 0] == 49 * K and acc[1, 0] == -56 * K and acc[1, 1] == 64 * K


@pytest.mark.parametrize("config,M,N", [("tiny_a8", 64, 256), ("down_proj", 256, 512), ("sweep", 512, 4096)])
def test_layer_a8_end_to_end(q, config, M, N):
    """X -> quarot_rotate_quant_a8 -> quarot_w4a4_gemm_a8 against the oracle's
    layer, and bit-identical to the packed path."""
    x, w, s = W.layer_inputs("rotq4096" if config == "tiny_a8" else config, M=M, N=N)
    a8, asx, ars = q.quarot_rotate_quant_a8(_t(x), _t(s))
    wq, wsx, _ = q.quarot_rotate_quant(_t(w), _t(s))
    y, _ = q.quarot_w4a4_gemm_a8(a8, ars, asx, wq, wsx)
    aq, asx2, _ = q.quarot_rotate_quant(_t(x), _t(s))
    yp, _ = q.quarot_w4a4_gemm(aq, asx2, wq, wsx)
    assert torch.equal(y, yp)
    oa, osx, _ = O.rotate_quant(x, s)
    ow, osw, _ = O.rotate_quant(w, s)
    _, oy = O.w4a4_gemm(oa, osx, ow, osw)
    assert O.rel_fro(y.cpu().numpy(), oy) <= OUT_TOL
