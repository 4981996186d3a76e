"""GPU parity of the row-code-sum path: quarot_rotate_quant_rowsum (the packed
codes and scales of quarot_rotate_quant plus each row's code sum),
quarot_int4_rowsum (code sums of any packed INT4 matrix) and
quarot_w4a4_gemm_rowsums (the GEMM with both operands' sums given).

Bars: the codes and scales are bit-identical to quarot_rotate_quant's; every
sum is exact; the GEMM's INT32 accumulator and fp16 output are bit-identical
to quarot_w4a4_gemm's on the same codes (and so to the oracle's integer GEMM
and dequantization, which that entry point is held to), on every plan the
shapes reach.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from test_gpu_parity import DEV, GEMM_SHAPES, ONE_SM_WIDE, PAIR_FORMS, _t, q  # noqa: F401  (q: fixture)

pytestmark = pytest.mark.gpu


def _codes(gq):
    return O.unpack_int4(gq.cpu().numpy()).astype(np.int64)


@pytest.mark.parametrize("d", [4096, 12288])
@pytest.mark.parametrize("M", [1, 37, 2048])
def test_rotate_quant_rowsum(q, d, M):
    x = W.activations(M, d, W.outlier_channels(d, 6, 3 + d), 80.0, 17 + d + M)
    s = _t(W.random_signs(d, 9 + d))
    gq, gs, rs = q.quarot_rotate_quant_rowsum(_t(x), s)
    pq, ps, _ = q.quarot_rotate_quant(_t(x), s)
    q.quarot_check_error()
    assert torch.equal(gq, pq) and torch.equal(gs, ps)
    assert np.array_equal(rs.cpu().numpy(), _codes(gq).sum(axis=1))


def test_rotate_quant_rowsum_edge_rows_and_stride(q):
    d = 4096
    x = np.zeros((6, d), dtype=np.float16)
    x[1, 3] = 1.0
    x[2] = 65504.0
    x[3, ::2] = -1.0
    x[4] = np.float16(6e-8)
    x[5, 7::3] = -2.5
    wide = torch.zeros((6, d + 40), dtype=torch.float16, device=DEV)
    wide[:, 8:8 + d] = _t(x)
    for xin in (_t(x), wide[:, 8:8 + d]):
        gq, gs, rs = q.quarot_rotate_quant_rowsum(xin, None, clip_ratio=0.9)
        pq, ps, _ = q.quarot_rotate_quant(_t(x), None, clip_ratio=0.9)
        assert torch.equal(gq, pq) and torch.equal(gs, ps)
        assert np.array_equal(rs.cpu().numpy(), _codes(gq).sum(axis=1))
    assert int(rs[0]) == 0


@pytest.mark.parametrize("M,K", [(1, 32), (7, 128), (1000, 4096), (257, 12288), (3, 65536)])
def test_int4_rowsum(q, M, K):
    c = W.int4_codes(M, K, 40 + K)
    c[0, :] = -8 if M > 1 else c[0, :]
    rs = q.quarot_int4_rowsum(_t(O.pack_int4(c)))
    q.quarot_check_error()
    assert np.array_equal(rs.cpu().numpy(), c.astype(np.int64).sum(axis=1))


def _gemm_both(q, M, N, K, seed):
    a, w = W.int4_codes(M, K, seed), W.int4_codes(N, K, seed + 1)
    sx, sw = W.fp16_scales(M, seed + 2), W.fp16_scales(N, seed + 3)
    aq, wq = _t(O.pack_int4(a)), _t(O.pack_int4(w))
    ars, wrs = q.quarot_int4_rowsum(aq), q.quarot_int4_rowsum(wq)
    y1, acc1 = q.quarot_w4a4_gemm_rowsums(aq, _t(sx), ars, wq, _t(sw), wrs, want_acc=True)
    y0, acc0 = q.quarot_w4a4_gemm(aq, _t(sx), wq, _t(sw), want_acc=True)
    q.quarot_check_error()
    assert torch.equal(acc1, acc0) and torch.equal(y1, y0)
    return a, w, sx, sw, y1, acc1


@pytest.mark.parametrize("M,N,K", list(GEMM_SHAPES) + PAIR_FORMS + ONE_SM_WIDE)
def test_gemm_rowsums_matches_gemm(q, M, N, K):
    a, w, sx, sw, y, acc = _gemm_both(q, M, N, K, 700 + M + N + K)
    if M * N * K <= 2 ** 31:
        ref = O.int_gemm(a, w)
        assert np.array_equal(acc.cpu().numpy(), ref)
        assert np.array_equal(y.cpu().numpy().view(np.uint16), O.dequant(ref, sx, sw).view(np.uint16))


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 12288), (8192, 4096, 4096), (2048, 12288, 4096)])
def test_gemm_rowsums_full_size(q, M, N, K):
    """The bench shape and sweep shapes (one and two accumulators) at full
    size: the whole output equal to quarot_w4a4_gemm's."""
    _gemm_both(q, M, N, K, 800 + M + N)


@pytest.mark.parametrize("M,N,K,reps", [(2048, 4096, 12288, 100), (8192, 12288, 4096, 20), (4000, 3000, 256, 100)])
def test_gemm_repeatable(q, M, N, K, reps):
    """Back-to-back launches of both GEMM entry points on one set of codes give
    the same bits every time: the bench shape (one accumulator), a shape with
    two 192-wide accumulators and the four-stage ring, and one with two
    160-wide accumulators and one stage pair per tile.  A rare ordering slip
    between the converters, the relay, the MMA issuer and the epilogue would
    show as a launch that differs."""
    g = torch.Generator(device="cpu").manual_seed(M + N + K)
    aq = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, generator=g).to(DEV)
    wq = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, generator=g).to(DEV)
    sx = (torch.rand(M, generator=g) * 0.1 + 0.01).half().to(DEV)
    sw = (torch.rand(N, generator=g) * 0.01 + 0.001).half().to(DEV)
    ars, wrs = q.quarot_int4_rowsum(aq), q.quarot_int4_rowsum(wq)
    y0, acc0 = q.quarot_w4a4_gemm_rowsums(aq, sx, ars, wq, sw, wrs, want_acc=True)
    yp, accp = q.quarot_w4a4_gemm(aq, sx, wq, sw, want_acc=True)
    assert torch.equal(acc0, accp) and torch.equal(y0, yp)
    y = torch.empty_like(y0)
    acc = torch.empty_like(acc0)
    for i in range(reps):
        if i % 2 == 0:
            q.quarot_w4a4_gemm_rowsums(aq, sx, ars, wq, sw, wrs, y=y, acc_out=acc)
        else:
            q.quarot_w4a4_gemm(aq, sx, wq, sw, y=y, acc_out=acc)
        assert torch.equal(acc, acc0) and torch.equal(y, y0), i
    q.quarot_check_error()


def test_gemm_rowsums_extremes_large_k(q):
    M, N, K = 200, 136, 65536
    a = np.full((M, K), 7, dtype=np.int8)
    a[1::3] = -8
    w = np.full((N, K), -8, dtype=np.int8)
    w[1::4] = 7
    aq, wq = _t(O.pack_int4(a)), _t(O.pack_int4(w))
    y, acc = q.quarot_w4a4_gemm_rowsums(aq, _t(W.fp16_scales(M, 1)), q.quarot_int4_rowsum(aq), wq,
                                        _t(W.fp16_scales(N, 2)), q.quarot_int4_rowsum(wq), want_acc=True)
    assert np.array_equal(acc.cpu().numpy(), O.int_gemm(a, w))


def test_layer_rowsum_chain(q):
    """X -> quarot_rotate_quant_rowsum -> quarot_w4a4_gemm_rowsums equals the
    plain chain bit for bit (down_proj shape, 256 rows)."""
    x, w, s = W.layer_inputs("down_proj", M=256, N=512)
    st = _t(s)
    wq, ws, _ = q.quarot_rotate_quant(_t(w), st)
    aq, as_, ars = q.quarot_rotate_quant_rowsum(_t(x), st)
    y, _ = q.quarot_w4a4_gemm_rowsums(aq, as_, ars, wq, ws, q.quarot_int4_rowsum(wq))
    aq0, as0, _ = q.quarot_rotate_quant(_t(x), st)
    y0, _ = q.quarot_w4a4_gemm(aq0, as0, wq, ws)
    assert torch.equal(y, y0)
