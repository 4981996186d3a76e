"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars (stated for the hot path): INT32 accumulators bit-exact on identical
codes; rotated fp32 within 1e-5 relative (floored at the row RMS); INT4 codes
identical except where |x/S| is within 1e-4 of a .5 boundary, with fewer than
1e-4 of codes affected; scales within one fp16 ulp; dequantised outputs within
1e-3 relative Frobenius error.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

ROT_TOL = 1e-5
OUT_TOL = 1e-3


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import w4a4_rotated_quantized_gb300 as mod

    mod.load()
    torch.cuda.set_device(0)
    return mod


DEV = "cuda:0"


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _fp16_ulp(s):
    s = np.asarray(s, dtype=np.float16)
    with np.errstate(over="ignore"):
        return np.abs(np.spacing(s).astype(np.float64))


# rows checked by check_quant, and rows whose scale differs from the oracle's
# by one fp16 ulp (a rounding-boundary case), over the whole module
_SCALE_TALLY = {"rows": 0, "differ": 0}


def _own_scale(grot, clip):
    """The quantizer's fp16 scale of the GPU's own rotated values, in the
    kernel's precision (fp32 abs-max, fp32 clip product, floor, division by 7,
    saturation, one rounding to fp16)."""
    m = np.abs(grot.astype(np.float32)).max(axis=-1)
    s = np.maximum(np.float32(clip) * m, np.float32(1e-5)) / np.float32(7.0)
    return np.minimum(s, np.float32(65504.0)).astype(np.float16)


def check_quant(gq, gs, grot, r_ref, clip=1.0):
    """Compare GPU (packed, scale, rotated) with the oracle's rotated values."""
    assert O.rotation_error(grot, r_ref) <= ROT_TOL
    q_ref, s_ref = O.quantize_rows(r_ref, clip)
    ds = np.abs(gs.astype(np.float64) - s_ref.astype(np.float64))
    assert np.all(ds <= _fp16_ulp(s_ref) * 1.0001), float(ds.max())
    # the GPU's scale is the quantizer's scale of its own rotated values
    assert np.array_equal(gs.view(np.uint16), _own_scale(grot, clip).view(np.uint16))
    same_scale = gs == s_ref
    # a scale may differ only where the oracle's unrounded scale and the GPU's
    # lie on the two sides of an fp16 rounding midpoint, within the rotation
    # tolerance of each other
    if not same_scale.all():
        m_ref = np.abs(r_ref.astype(np.float64)).max(axis=-1)
        s32_ref = np.maximum(clip * m_ref, 1e-5) / 7.0
        s32_gpu = np.maximum(np.float32(clip) * np.abs(grot.astype(np.float32)).max(axis=-1),
                             np.float32(1e-5)).astype(np.float64) / 7.0
        lo = np.minimum(s_ref, gs).astype(np.float64)
        mid = lo + _fp16_ulp(lo) / 2
        dif = ~same_scale
        assert np.all(np.abs(s32_ref[dif] - s32_gpu[dif]) <= 2 * ROT_TOL * s32_ref[dif])
        assert np.all((np.minimum(s32_ref, s32_gpu)[dif] <= mid[dif] * (1 + 1e-7)) &
                      (np.maximum(s32_ref, s32_gpu)[dif] >= mid[dif] * (1 - 1e-7))), "scale off by one ulp away from a midpoint"
    rows = int(np.prod(gs.shape))
    _SCALE_TALLY["rows"] += rows
    _SCALE_TALLY["differ"] += int((~same_scale).sum())
    codes = O.unpack_int4(gq)
    diff = codes != q_ref
    # where the scales agree, codes may differ only at .5 boundaries
    bnd = O.boundary_mask(r_ref, s_ref)
    bad = diff & ~bnd & same_scale[..., None]
    assert not bad.any(), f"{int(bad.sum())} codes differ away from a rounding boundary"
    # where they differ, the codes are the oracle's rotated values quantized
    # with the GPU's scale (again up to .5 boundaries)
    if not same_scale.all():
        q_alt = np.clip(O.round_half_even(r_ref.astype(np.float64) / gs.astype(np.float64)[..., None]), -8, 7)
        bnd_alt = O.boundary_mask(r_ref, gs)
        bad = (codes != q_alt) & ~bnd_alt & ~same_scale[..., None]
        assert not bad.any(), f"{int(bad.sum())} codes differ from the oracle values quantized with the GPU scale"
    frac = diff[same_scale].mean() if same_scale.any() else 0.0
    assert frac < 1e-4, frac
    # codes must be the quantizer applied to the GPU's own rotated values with its own scale
    y = grot.astype(np.float64) / gs.astype(np.float64)[..., None]
    own = np.clip(np.rint(y), -8, 7)
    near = np.abs(np.abs(y - np.floor(y)) - 0.5) < 1e-5
    assert np.all((own == codes) | near)


# ---------------------------------------------------------------- bounded waits
def test_bounded_wait_expires_and_context_survives(q):
    """A device wait on a barrier that nothing completes gives up after the
    library's limit (one second), reports QUAROT_ERR_TIMEOUT once, and the
    context keeps running kernels correctly afterwards (no fault, no hang)."""
    import time

    q.quarot_check_error()  # start from a clear error word
    t0 = time.perf_counter()
    q.quarot_selftest_wait()
    with pytest.raises(q.QuarotError) as e:
        q.quarot_check_error()
    dt = time.perf_counter() - t0
    assert e.value.status == q.QUAROT_ERR_TIMEOUT
    assert 0.9 <= dt < 30.0, dt
    q.quarot_check_error()  # the word was cleared
    x, _, s = W.layer_inputs("tiny")
    gq, gs, grot = q.quarot_rotate_quant(_t(x), _t(s), want_rot=True)
    q.quarot_check_error()
    check_quant(gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy(), O.rotate(x, s))


# ---------------------------------------------------------------- rotate+quant
@pytest.mark.parametrize("d", [16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192, 3072, 6144, 12288])
@pytest.mark.parametrize("signed", [True, False])
def test_rotate_quant_widths(q, d, signed):
    M = 37  # ragged: not a multiple of the rows per CTA
    x = W.activations(M, d, W.outlier_channels(d, max(1, d // 512), 5 + d), 100.0, 11 + d)
    s = W.random_signs(d, 21 + d) if signed else None
    gq, gs, grot = q.quarot_rotate_quant(_t(x), None if s is None else _t(s), want_rot=True)
    r_ref = O.rotate(x, s)
    check_quant(gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy(), r_ref)


@pytest.mark.parametrize("d", [256, 4096, 12288])
def test_rotate_quant_clip_09(q, d):
    x = W.activations(19, d, [1, 7], 50.0, 3)
    s = W.random_signs(d, 4)
    gq, gs, grot = q.quarot_rotate_quant(_t(x), _t(s), clip_ratio=0.9, want_rot=True)
    check_quant(gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy(), O.rotate(x, s), clip=0.9)


def test_rotate_quant_edge_rows(q):
    d = 4096
    x = np.zeros((5, d), dtype=np.float16)
    x[1, 3] = 1.0            # one-hot: all |r| equal -> every code +-7
    x[2] = 65504.0           # largest fp16: scale saturates below fp16 max
    x[3, ::2] = -1.0
    x[4] = np.float16(6e-8)  # subnormal inputs
    gq, gs, grot = q.quarot_rotate_quant(_t(x), None, want_rot=True)
    gq, gs, grot = gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy()
    codes = O.unpack_int4(gq)
    assert np.all(codes[0] == 0) and float(gs[0]) == float(np.float16(1e-5 / 7))
    assert np.all(np.abs(codes[1]) == 7)
    assert np.isfinite(gs.astype(np.float32)).all()
    check_quant(gq, gs, grot, O.rotate(x, None))


def test_rotate_quant_empty(q):
    x = torch.empty((0, 4096), dtype=torch.float16, device=DEV)
    gq, gs, _ = q.quarot_rotate_quant(x)
    assert gq.shape == (0, 2048)


def test_rotate_quant_config_rotq4096_full(q):
    """2048 x 4096 at full size (the bench launch); oracle on sampled rows."""
    x, _, s = W.layer_inputs("rotq4096")
    gq, gs, grot = q.quarot_rotate_quant(_t(x), _t(s), want_rot=True)
    rows = np.random.default_rng(0).choice(x.shape[0], 192, replace=False)
    rows[:2] = [0, x.shape[0] - 1]
    check_quant(gq.cpu().numpy()[rows], gs.cpu().numpy()[rows], grot.cpu().numpy()[rows], O.rotate(x[rows], s))


def test_rotate_quant_config_down_proj_sampled(q):
    x, _, s = W.layer_inputs("down_proj", N=0)
    gq, gs, grot = q.quarot_rotate_quant(_t(x), _t(s), want_rot=True)
    rows = np.random.default_rng(1).choice(x.shape[0], 48, replace=False)
    check_quant(gq.cpu().numpy()[rows], gs.cpu().numpy()[rows], grot.cpu().numpy()[rows], O.rotate(x[rows], s))


# ---------------------------------------------------------------- fused RMSNorm + rotate + quant
# ---------------------------------------------------------------- FP16 online Hadamard (next row f4)
def _check_fp16_rotation(q, x, s, clip=1.0):
    gq, gs, grot = q.quarot_rotate_quant_fp16(_t(x), None if s is None else _t(s), clip_ratio=clip, want_rot=True)
    gq, gs, grot = gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy()
    r16 = O.rotate_fp16_arith(x, s).astype(np.float32)
    # every step is a correctly rounded fp16 operation in the same order:
    # the rotated values are bit-identical
    assert np.array_equal(grot, r16)
    check_quant(gq, gs, grot, r16, clip)
    return grot


@pytest.mark.parametrize("d", [16, 128, 256, 1024, 2048, 4096, 8192, 3072, 6144, 12288])
def test_rotate_quant_fp16_widths(q, d):
    M = 37  # ragged: not a multiple of the rows per CTA
    x = W.activations(M, d, W.outlier_channels(d, max(1, d // 512), 5 + d), 100.0, 11 + d)
    _check_fp16_rotation(q, x, W.random_signs(d, 21 + d))


def test_rotate_quant_fp16_no_signs_clip_and_close_to_fp32(q):
    x, _, s = W.layer_inputs("rotq4096", M=64)
    _check_fp16_rotation(q, x, None, clip=0.9)
    # the variant's rotation stays within its error bound of the exact one:
    # (log2 4096 + 2) * 2^-11 * |x|
    grot = _check_fp16_rotation(q, x, s)
    err = np.linalg.norm(grot.astype(np.float64) - O.rotate_f64(x, s), axis=1)
    assert np.all(err <= 14 * 2.0 ** -11 * np.linalg.norm(x.astype(np.float64), axis=1))


@pytest.mark.parametrize("d", [4096, 12288])
def test_rotate_quant_fp16_edge_rows(q, d):
    """Zero, one-hot (small and near the fp16 maximum), alternating, subnormal
    and smallest-normal rows through the persistent fp16 kernels."""
    x = np.zeros((7, d), dtype=np.float16)
    x[1, 3] = 1.0
    x[2, d - 1] = 60000.0
    x[3, ::2] = -1.0
    x[4] = np.float16(6e-8)
    x[5, 1::3] = 2.0 ** -14
    x[6, 5::7] = -3.5
    _check_fp16_rotation(q, x, W.random_signs(d, 3))
    gq, gs, _ = q.quarot_rotate_quant_fp16(_t(x), None)
    assert np.all(gq.cpu().numpy()[0] == 0)


@pytest.mark.parametrize("config", ["down_proj", "rotq4096"])
def test_rotate_quant_fp16_full(q, config):
    """2048 rows at full size (2048 x 12288 and 2048 x 4096): persistent CTAs
    take several rows each; rows sampled by the oracle, including rows of a
    CTA's second and later trips."""
    x, _, s = W.layer_inputs(config, N=0)
    gq, gs, grot = q.quarot_rotate_quant_fp16(_t(x), _t(s), want_rot=True)
    rows = [0, 1, 607, 777, 1216, 1520, 2047]
    r16 = O.rotate_fp16_arith(x[rows], s).astype(np.float32)
    grot = grot.cpu().numpy()[rows]
    assert np.array_equal(grot, r16)
    check_quant(gq.cpu().numpy()[rows], gs.cpu().numpy()[rows], grot, r16)


@pytest.mark.parametrize("d", [16, 256, 1024, 3072, 4096, 8192, 12288])
def test_rmsnorm_rotate_quant_widths(q, d):
    M = 37
    x = W.activations(M, d, W.outlier_channels(d, max(1, d // 512), 7 + d), 100.0, 13 + d)
    s = W.random_signs(d, 23 + d)
    gq, gs, grot = q.quarot_rmsnorm_rotate_quant(_t(x), _t(s), eps=1e-6, want_rot=True)
    _, _, r_ref = O.rmsnorm_rotate_quant(x, s, 1e-6)
    check_quant(gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy(), r_ref)


@pytest.mark.parametrize("d", [256, 4096, 12288])
def test_rmsnorm_rotate_quant_clip_eps_edge_rows(q, d):
    x = W.activations(9, d, [1, 5], 30.0, 41)
    x[0] = 0.0            # zero row: eps keeps it finite, codes 0 and the floor scale
    x[1] = 0.25           # constant row: mean square 1/16
    x[2] *= np.float16(1e-3)  # small row: eps visible in the normalization
    s = W.random_signs(d, 43)
    eps = 1e-4
    gq, gs, grot = q.quarot_rmsnorm_rotate_quant(_t(x), _t(s), eps=eps, clip_ratio=0.9, want_rot=True)
    _, _, r_ref = O.rmsnorm_rotate_quant(x, s, eps, 0.9)
    gq, gs, grot = gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy()
    assert np.all(O.unpack_int4(gq)[0] == 0) and float(gs[0]) == float(np.float16(1e-5 / 7))
    check_quant(gq, gs, grot, r_ref, clip=0.9)


def test_rmsnorm_rotate_quant_down_proj_sampled(q):
    """2048 x 12288: the persistent kernel takes several rows per CTA."""
    x, _, s = W.layer_inputs("down_proj", N=0)
    gq, gs, grot = q.quarot_rmsnorm_rotate_quant(_t(x), _t(s), eps=1e-6, want_rot=True)
    rows = np.random.default_rng(5).choice(x.shape[0], 40, replace=False)
    rows[:2] = [0, x.shape[0] - 1]
    _, _, r_ref = O.rmsnorm_rotate_quant(x[rows], s, 1e-6)
    check_quant(gq.cpu().numpy()[rows], gs.cpu().numpy()[rows], grot.cpu().numpy()[rows], r_ref)


# ---------------------------------------------------------------- cross-head Hadamard + quant (next row f3)
@pytest.mark.parametrize("nh,dh", [(1, 128), (2, 64), (8, 128), (32, 128), (64, 64)])
def test_crosshead_rotate_quant_parity(q, nh, dh):
    M = 37
    z = W.query(M, nh, dh, 70 + nh).reshape(M, nh * dh)
    z[3, min(dh + 5, nh * dh - 1)] = np.float16(60.0)  # an outlier in one head
    gq, gs, grot = q.quarot_crosshead_rotate_quant(_t(z), nh, want_rot=True)
    check_quant(gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy(), O.crosshead_rotate(z, nh))
    gq, gs, grot = q.quarot_crosshead_rotate_quant(_t(z), nh, clip_ratio=0.9, want_rot=True)
    check_quant(gq.cpu().numpy(), gs.cpu().numpy(), grot.cpu().numpy(), O.crosshead_rotate(z, nh), clip=0.9)


def test_attention_output_path_end_to_end(q):
    """Decode in the rotated basis -> cross-head Hadamard + INT4 -> W4A4 GEMM
    against W_out rows rotated by the full H_4096 (= H_32 (x) H_128)."""
    B, Hkv, G, d, T, N = 4, 8, 4, 128, 256, 512
    Hq = Hkv * G
    k = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 81)
    v = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 82)
    qq = W.query(B, Hq, d, 83)
    gc = q.new_kv_cache(B, Hkv, T, d, DEV)
    q.quarot_kv_write(_t(k), _t(v), 0, *gc)
    o_rot = q.quarot_decode_attn(_t(qq), *gc, T=T, unrotate_out=False)  # [B, Hq, d], rotated basis
    zq, zs, _ = q.quarot_crosshead_rotate_quant(o_rot, Hq)
    w_out = W.weights(N, Hq * d, 84)
    wq, ws, _ = q.quarot_rotate_quant(_t(w_out), None)
    y, _ = q.quarot_w4a4_gemm(zq, zs, wq, ws)
    y = y.cpu().numpy().astype(np.float64)
    # parity: the oracle's chain on the GPU's decode output
    oz, ozs, _ = O.crosshead_rotate_quant(o_rot.cpu().numpy().reshape(B, Hq * d), Hq)
    ow, ows, _ = O.rotate_quant(w_out, None)
    _, oy = O.w4a4_gemm(oz, ozs, ow, ows)
    assert O.rel_fro(y, oy) <= OUT_TOL
    # the rotations cancel: y approximates the un-rotated attention output times
    # W_out^T up to the W4A4 error (a wrong factor would be an O(1) error)
    gnp = [t.cpu().numpy() for t in gc]
    attn = O.decode_attn(qq, *gnp, T=T, unrotate=True).reshape(B, Hq * d)
    assert O.rel_fro(y, attn @ w_out.astype(np.float64).T) < 0.25


# ---------------------------------------------------------------- GEMM
def _gemm_case(q, M, N, K, seed, codes_a=None, codes_w=None):
    a = W.int4_codes(M, K, seed) if codes_a is None else codes_a
    w = W.int4_codes(N, K, seed + 1) if codes_w is None else codes_w
    sx = W.fp16_scales(M, seed + 2)
    sw = W.fp16_scales(N, seed + 3)
    ap, wp = O.pack_int4(a), O.pack_int4(w)
    y, acc = q.quarot_w4a4_gemm(_t(ap), _t(sx), _t(wp), _t(sw), want_acc=True)
    q.quarot_check_error()
    return a, w, sx, sw, y.cpu().numpy(), acc.cpu().numpy()


# M <= 128 runs the one-SM kernel; M > 128 with K % 256 == 0 the CTA-pair kernel
# (ragged M and N tails in either CTA of a pair); (257, 513, 384) has an odd
# k-block count and takes the one-SM kernel at M > 128
GEMM_SHAPES = [(16, 256, 256), (128, 256, 128), (200, 300, 256), (1, 8, 128), (257, 513, 384),
               (256, 512, 4096), (130, 264, 12288), (385, 136, 768), (600, 1000, 1024)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_bit_exact(q, M, N, K):
    a, w, sx, sw, y, acc = _gemm_case(q, M, N, K, 100 + M + N + K)
    ref = O.int_gemm(a, w)
    assert np.array_equal(acc, ref)
    assert np.array_equal(y.view(np.uint16), O.dequant(ref, sx, sw).view(np.uint16))


def test_gemm_adversarial_extremes(q):
    K = 12288
    a = np.full((130, K), -8, dtype=np.int8)
    a[1::2] = 7
    a[2, ::3] = -7
    w = np.full((260, K), -8, dtype=np.int8)
    w[::3] = 7
    _, _, _, _, y, acc = _gemm_case(q, 130, 260, K, 7, a, w)
    assert np.array_equal(acc, O.int_gemm(a, w))
    assert acc[0, 0] == -56 * K and acc[0, 1] == 64 * K and acc[1, 0] == 49 * K


def _tile_rows(M, form, salt):
    """One row in every TMEM lane quadrant of every M tile (256-row pair tiles
    for the CTA-pair kernel, 128-row tiles for the one-SM kernel), plus the
    last row."""
    rows = []
    for m0 in range(0, M, 128):
        for qd in range(4):
            r = m0 + 32 * qd + (7 * (m0 // 128) + 13 * qd + salt) % 32
            if r < M:
                rows.append(r)
    rows.append(M - 1)
    return np.unique(np.array(rows))


def _gemm_sampled(q, M, N, K, seed):
    """Full-size launch; exact INT32 accumulator and bit-identical fp16 output
    on _tile_rows, all N columns."""
    a = W.int4_codes(M, K, seed)
    w = W.int4_codes(N, K, seed + 1)
    sx = W.fp16_scales(M, seed + 2)
    sw = W.fp16_scales(N, seed + 3)
    y, acc = q.quarot_w4a4_gemm(_t(O.pack_int4(a)), _t(sx), _t(O.pack_int4(w)), _t(sw), want_acc=True)
    q.quarot_check_error()
    form, _ = q.quarot_w4a4_gemm_plan(M, N, K, torch.cuda.get_device_properties(0).multi_processor_count)
    rows = _tile_rows(M, form, seed)
    ri = torch.from_numpy(rows).to(DEV)
    acc_s = acc.index_select(0, ri).cpu().numpy()
    y_s = y.index_select(0, ri).cpu().numpy()
    del y, acc
    ref = O.int_gemm(a[rows], w)
    assert np.array_equal(acc_s, ref)
    assert np.array_equal(y_s.view(np.uint16), O.dequant(ref, sx[rows], sw).view(np.uint16))


def test_gemm_full_down_proj_sampled(q):
    """2048 x 4096 x 12288 at full size (the bench launch)."""
    _gemm_sampled(q, 2048, 4096, 12288, 900)


@pytest.mark.parametrize("M", [512, 2048, 8192])
@pytest.mark.parametrize("N", [4096, 12288])
def test_gemm_sweep_shapes(q, M, N):
    """The prefill GEMM sweep, M x 4096 x N, at full size: every pair tile and
    lane quadrant sampled (BN 128, 160, 192 and 224 among them)."""
    _gemm_sampled(q, M, N, 4096, 3000 + M + N)


# one-SM kernel (odd k-block count) at the widths the sweep does not reach
ONE_SM_WIDE = [(1156, 2888, 128), (1030, 2568, 384), (771, 2696, 128)]

# CTA-pair plans the sweep does not reach: one accumulator at BN 160, and two
# accumulators with ragged M and N tails at BN 128, 160 (six-stage ring) and
# 192 (four-stage ring), from one stage pair per tile to four
PAIR_FORMS = [(2048, 2560, 1024), (4000, 3000, 256), (1137, 7330, 512), (3100, 7000, 768), (1548, 5648, 768),
              (7000, 1000, 256)]


@pytest.mark.parametrize("M,N,K", PAIR_FORMS)
def test_gemm_pair_forms(q, M, N, K):
    _gemm_sampled(q, M, N, K, 4500 + M + N)


@pytest.mark.parametrize("M,N,K", ONE_SM_WIDE)
def test_gemm_one_sm_wide_tiles(q, M, N, K):
    _gemm_sampled(q, M, N, K, 4000 + M)


def test_gemm_parity_covers_every_tile_width(q):
    """The GEMM shapes of this module reach N-tile widths 128, 160, 192 and
    224 in both the one-SM and the single-accumulator CTA-pair kernel, and
    128, 160 and 192 in the two-accumulator CTA-pair kernel, on this GPU."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shapes = list(GEMM_SHAPES) + [(2048, 4096, 12288)] + [(M, N, 4096) for M in (512, 2048, 8192)
                                                         for N in (4096, 12288)] + ONE_SM_WIDE + PAIR_FORMS
    seen = {q.quarot_w4a4_gemm_plan(M, N, K, sms) for M, N, K in shapes}
    want = [(f, bn) for f in (1, 2) for bn in (128, 160, 192, 224)] + [(3, 128), (3, 160), (3, 192)]
    for p in want:
        assert p in seen, (p, sms)


@pytest.mark.parametrize("K", [16384, 32768, 65536])
@pytest.mark.parametrize("M", [64, 200])
def test_gemm_extremes_at_large_k(q, K, M):
    """All-extreme codes up to the largest K the ABI accepts (65536): every
    partial sum of the offset encoding stays an integer below 2^24 units, so
    the fp32 accumulation must stay exact.  M = 64 runs the one-SM kernel,
    M = 200 the CTA pair."""
    N = 136
    a = np.full((M, K), 7, dtype=np.int8)
    a[1::3] = -8
    a[2::5, ::2] = -7
    w = np.full((N, K), 7, dtype=np.int8)
    w[1::4] = -8
    w[3::7, 1::3] = 6
    _, _, _, _, y, acc = _gemm_case(q, M, N, K, 11 + K + M, a, w)
    assert np.array_equal(acc, O.int_gemm(a, w))
    assert acc[0, 0] == 49 * K and acc[1, 0] == -56 * K and acc[1, 1] == 64 * K


# ---------------------------------------------------------------- layer end to end
@pytest.mark.parametrize("config,M,N", [("tiny", None, None), ("down_proj", 256, 512), ("sweep", 512, 4096)])
def test_layer_end_to_end(q, config, M, N):
    x, w, s = W.layer_inputs(config, M=M, N=N)
    aq, asx, _ = q.quarot_rotate_quant(_t(x), _t(s))
    wq, wsx, _ = q.quarot_rotate_quant(_t(w), _t(s))
    y, _ = q.quarot_w4a4_gemm(aq, asx, wq, wsx)
    oa, osx, _ = O.rotate_quant(x, s)
    ow, osw, _ = O.rotate_quant(w, s)
    _, oy = O.w4a4_gemm(oa, osx, ow, osw)
    assert O.rel_fro(y.cpu().numpy(), oy) <= OUT_TOL


# ---------------------------------------------------------------- KV cache
def _caches(shape_like, T_max):
    B, _, H, d = shape_like
    return [np.zeros((B, H, T_max, d // 2), np.uint8), np.zeros((B, H, T_max), np.float16),
            np.zeros((B, H, T_max, d // 2), np.uint8), np.zeros((B, H, T_max), np.float16)]


@pytest.mark.parametrize("d", [64, 128, 256])
def test_kv_write_parity(q, d):
    B, T, H, T_max, t0 = 3, 37, 2, 64, 5
    k = W.kv_tensors(B, T, H, d, 2, 20.0, 31)
    v = W.kv_tensors(B, T, H, d, 2, 20.0, 32)
    gc = q.new_kv_cache(B, H, T_max, d, DEV)
    q.quarot_kv_write(_t(k), _t(v), t0, *gc)
    gk, gks, gv, gvs = [t.cpu().numpy() for t in gc]
    for src, codes, scales in ((k, gk, gks), (v, gv, gvs)):
        r = O.rotate(src, None)  # [B, T, H, d]
        q_ref, s_ref = O.quantize_rows(r, 1.0)
        s_gpu = scales[:, :, t0:t0 + T].transpose(0, 2, 1)
        c_gpu = O.unpack_int4(codes[:, :, t0:t0 + T].transpose(0, 2, 1, 3))
        assert np.all(np.abs(s_gpu.astype(np.float64) - s_ref.astype(np.float64)) <= _fp16_ulp(s_ref))
        diff = (c_gpu != q_ref) & ~O.boundary_mask(r, s_ref)
        assert not diff.any()
        assert np.all(codes[:, :, :t0] == 0) and np.all(codes[:, :, t0 + T:] == 0)


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("T", [1, 5, 256, 300, 1000])
def test_decode_parity(q, G, T):
    B, Hkv, d, T_max = 2, 2, 128, 1024
    k = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 41 + T)
    v = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 42 + T)
    qq = W.query(B, Hkv * G, d, 43 + T)
    oc = _caches(k.shape, T_max)
    O.kv_write(k, v, 0, *oc)
    for unrot in (False, True):
        out = q.quarot_decode_attn(_t(qq), *[_t(c) for c in oc], T=T, unrotate_out=unrot)
        ref = O.decode_attn(qq, *oc, T=T, unrotate=unrot)
        assert O.rel_fro(out.cpu().numpy(), ref) <= OUT_TOL
        _check_per_head(out.cpu().numpy(), ref)


def _check_per_head(out, ref):
    """Every (sequence, query head) on its own, against the typical output
    norm over the heads: a slip confined to one head or one split cannot hide
    under the whole tensor's Frobenius ratio."""
    o = out.astype(np.float64)
    num = np.sqrt(((o - ref) ** 2).sum(axis=-1))  # [B, Hq]
    den = np.sqrt((ref ** 2).sum(axis=-1))
    typ = np.sqrt((den ** 2).mean())
    assert np.all(num <= 4 * OUT_TOL * np.maximum(den, typ)), float((num / np.maximum(den, typ)).max())


def test_decode_single_sequence_long(q):
    """B = 1 at the kv4 context (T 4096, 8 KV heads x 4 query heads): eight
    (sequence, KV head) rows over 152 SMs, so the split-T path runs with its
    largest split count."""
    B, Hkv, G, d, T = 1, 8, 4, 128, 4096
    k = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 141)
    v = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 142)
    qq = W.query(B, Hkv * G, d, 143)
    oc = _caches(k.shape, T)
    O.kv_write(k, v, 0, *oc)
    for unrot in (False, True):
        out = q.quarot_decode_attn(_t(qq), *[_t(c) for c in oc], T=T, unrotate_out=unrot).cpu().numpy()
        ref = O.decode_attn(qq, *oc, T=T, unrotate=unrot)
        assert O.rel_fro(out, ref) <= OUT_TOL
        _check_per_head(out, ref)


@pytest.mark.parametrize("G", [1, 8])
@pytest.mark.parametrize("T", [2048, 2304])
def test_decode_split_counts(q, G, T):
    """One sequence, two KV heads: T 2048 runs 8 splits of 256 tokens per row
    and T 2304 runs 9, so the combine merges 8 and 9 partial states per head,
    for one query head per KV head and for eight."""
    B, Hkv, d = 1, 2, 128
    k = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 61 + T + G)
    v = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 62 + T + G)
    qq = W.query(B, Hkv * G, d, 63 + T + G)
    oc = _caches(k.shape, T)
    O.kv_write(k, v, 0, *oc)
    for unrot in (False, True):
        out = q.quarot_decode_attn(_t(qq), *[_t(c) for c in oc], T=T, unrotate_out=unrot).cpu().numpy()
        ref = O.decode_attn(qq, *oc, T=T, unrotate=unrot)
        assert O.rel_fro(out, ref) <= OUT_TOL
        _check_per_head(out, ref)


def test_decode_custom_scale_and_zero_T(q):
    B, Hkv, G, d, T = 1, 2, 4, 128, 77
    k = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 5)
    v = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 6)
    qq = W.query(B, Hkv * G, d, 7)
    oc = _caches(k.shape, 128)
    O.kv_write(k, v, 0, *oc)
    out = q.quarot_decode_attn(_t(qq), *[_t(c) for c in oc], T=T, sm_scale=0.05)
    assert O.rel_fro(out.cpu().numpy(), O.decode_attn(qq, *oc, T=T, sm_scale=0.05)) <= OUT_TOL
    out0 = q.quarot_decode_attn(_t(qq), *[_t(c) for c in oc], T=0)
    assert torch.all(out0 == 0)


def test_kv4_config_full(q):
    """B16 x T4096 x Hkv8 x Hq32: full-size append and decode; oracle on two sequences."""
    k, v, qq = W.kv_inputs("kv4")
    B, T, Hkv, d = k.shape
    gc = q.new_kv_cache(B, Hkv, T, d, DEV)
    q.quarot_kv_write(_t(k), _t(v), 0, *gc)
    out = q.quarot_decode_attn(_t(qq), *gc, T=T)
    q.quarot_check_error()
    out = out.cpu().numpy()
    gnp = [t.cpu().numpy() for t in gc]
    for b in (0, B - 1):
        oc = _caches(k[b:b + 1].shape, T)
        O.kv_write(k[b:b + 1], v[b:b + 1], 0, *oc)
        for name, g, o in (("k_s", gnp[1][b], oc[1][0]), ("v_s", gnp[3][b], oc[3][0])):
            assert np.all(np.abs(g.astype(np.float64) - o.astype(np.float64)) <= _fp16_ulp(o)), name
        ref = O.decode_attn(qq[b:b + 1], *oc, T=T)
        assert O.rel_fro(out[b:b + 1], ref) <= OUT_TOL
        _check_per_head(out[b:b + 1], ref)


# ---------------------------------------------------------------- prefill "Init" attention (next row f4)
def _prefill_case(B, T, Hkv, G, seed, T_max=None):
    k = W.kv_tensors(B, T, Hkv, 128, 2, 20.0, seed)
    v = W.kv_tensors(B, T, Hkv, 128, 2, 20.0, seed + 1)
    qq = W.prefill_query(B, T, Hkv * G, 128, seed + 2)
    oc = _caches(k.shape, T_max or T)
    O.kv_write(k, v, 0, *oc)
    return qq, oc


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("T", [1, 100, 128, 300, 520])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_parity(q, G, T, causal):
    qq, oc = _prefill_case(2, T, 2, G, 51 + T + G)
    out = q.quarot_prefill_attn(_t(qq), *[_t(c) for c in oc], causal=causal)
    q.quarot_check_error()
    ref = O.prefill_attn(qq, *oc, T=T, causal=causal)
    assert O.rel_fro(out.cpu().numpy(), ref) <= OUT_TOL
    # every query row on its own, against the typical output norm of its head
    # (fp16 rounding of v^ and p is relative to the values, not to a row whose
    # terms cancel)
    o = out.cpu().numpy().astype(np.float64)
    num = np.sqrt(((o - ref) ** 2).sum(axis=-1))  # [B, T, Hq]
    den = np.sqrt((ref ** 2).sum(axis=-1))
    typ = np.sqrt((den ** 2).mean(axis=1, keepdims=True))
    assert np.all(num <= 4 * OUT_TOL * np.maximum(den, typ))


def test_prefill_ignores_cache_past_T(q):
    """Tokens T .. T_max-1 of the cache hold garbage codes and inf/nan scales;
    the prompt attends to tokens < T only."""
    B, T, T_max, Hkv, G = 1, 200, 384, 2, 4
    qq, oc = _prefill_case(B, T, Hkv, G, 61, T_max=T_max)
    rng = np.random.default_rng(62)
    for c in (oc[0], oc[2]):
        c[:, :, T:] = rng.integers(0, 256, c[:, :, T:].shape, dtype=np.uint8)
    for s in (oc[1], oc[3]):
        s[:, :, T:] = np.array([np.inf, np.nan, 60000.0], np.float16)[rng.integers(0, 3, s[:, :, T:].shape)]
    for causal in (True, False):
        out = q.quarot_prefill_attn(_t(qq), *[_t(c) for c in oc], causal=causal)
        ref = O.prefill_attn(qq, *oc, T=T, causal=causal)
        assert np.isfinite(out.cpu().numpy()).all()
        assert O.rel_fro(out.cpu().numpy(), ref) <= OUT_TOL


def test_prefill_causal_rows_ignore_later_tokens(q):
    """Causal row i reads tokens 0..i: rewriting every cached token after t
    (codes and scales, finite) leaves rows 0..t bit-identical, since masked
    keys enter the diagonal tile with probability exactly 0."""
    B, T, Hkv, G, t = 2, 300, 2, 4, 150
    qq, oc = _prefill_case(B, T, Hkv, G, 91)
    base = q.quarot_prefill_attn(_t(qq), *[_t(c) for c in oc]).cpu().numpy()
    rng = np.random.default_rng(92)
    oc2 = [c.copy() for c in oc]
    for c in (oc2[0], oc2[2]):
        c[:, :, t + 1:] = rng.integers(0, 256, c[:, :, t + 1:].shape, dtype=np.uint8)
    oc2[1][:, :, t + 1:] *= np.float16(3.0)
    oc2[3][:, :, t + 1:] *= np.float16(0.5)
    assert np.isfinite(oc2[1]).all() and np.isfinite(oc2[3]).all()
    out = q.quarot_prefill_attn(_t(qq), *[_t(c) for c in oc2]).cpu().numpy()
    q.quarot_check_error()
    assert np.array_equal(out[:, :t + 1], base[:, :t + 1])
    assert not np.array_equal(out[:, T - 1], base[:, T - 1])


def test_prefill_custom_scale_and_empty(q):
    qq, oc = _prefill_case(1, 150, 2, 4, 71)
    out = q.quarot_prefill_attn(_t(qq), *[_t(c) for c in oc], sm_scale=0.05)
    assert O.rel_fro(out.cpu().numpy(), O.prefill_attn(qq, *oc, T=150, sm_scale=0.05)) <= OUT_TOL
    e = q.quarot_prefill_attn(_t(qq[:, :0]), *[_t(c) for c in oc])
    assert e.shape == (1, 0, 8, 128)


def test_prefill_last_row_is_decode(q):
    """The causal prefill's last row and the decode kernel answer the same question."""
    qq, oc = _prefill_case(2, 333, 2, 4, 81)
    g = [_t(c) for c in oc]
    out = q.quarot_prefill_attn(_t(qq), *g)
    dec = q.quarot_decode_attn(_t(np.ascontiguousarray(qq[:, -1])), *g, T=333)
    assert O.rel_fro(out[:, -1].cpu().numpy(), dec.cpu().numpy().astype(np.float64)) <= 2 * OUT_TOL


def test_prefill_long_context_g8(q):
    """One 4096-token prompt, 8 query heads on one KV head (32 key tiles for the
    last query tile): long causal rows, many lazy-rescale decisions."""
    qq, oc = _prefill_case(1, 4096, 1, 8, 91)
    out = q.quarot_prefill_attn(_t(qq), *[_t(c) for c in oc])
    q.quarot_check_error()
    ref = O.prefill_attn(qq, *oc, T=4096)
    assert O.rel_fro(out.cpu().numpy(), ref) <= OUT_TOL


def test_prefill_config_full(q):
    """B4 x T2048 x Hq32/Hkv8 at full size, over a cache the oracle wrote (the
    append kernel is pinned on its own); oracle on the first and last prompt
    (all heads, all rows)."""
    k, v, qq = W.prefill_inputs("prefill")
    B, T, Hkv, d = k.shape
    oc = _caches(k.shape, T)
    O.kv_write(k, v, 0, *oc)
    out = q.quarot_prefill_attn(_t(qq), *[_t(c) for c in oc])
    q.quarot_check_error()
    out = out.cpu().numpy()
    for b in (0, B - 1):
        ref = O.prefill_attn(qq[b:b + 1], *[c[b:b + 1] for c in oc], T=T)
        assert O.rel_fro(out[b:b + 1], ref) <= OUT_TOL


@pytest.mark.parametrize("case", ["pair_130", "bench_4x2048"])
def test_prefill_repeated_launches_bit_identical(q, case):
    """200 launches of the CTA-pair prefill give the same bits every time, and
    the first is within the bar of the oracle: the 130-token prompt with two
    query heads on one KV head (two query tiles, the second ragged) and the
    4 x 2048 bench prompt (32 query / 8 KV heads)."""
    if case == "pair_130":
        T = 130
        k = W.kv_tensors(1, T, 1, 128, 2, 20.0, 7)
        v = W.kv_tensors(1, T, 1, 128, 2, 20.0, 8)
        qq = W.prefill_query(1, T, 2, 128, 9)
    else:
        k, v, qq = W.prefill_inputs("prefill")
        T = k.shape[1]
    oc = _caches(k.shape, T)
    O.kv_write(k, v, 0, *oc)
    g = [_t(c) for c in oc]
    qt = _t(qq)
    first = q.quarot_prefill_attn(qt, *g)
    q.quarot_check_error()
    b = qq.shape[0] - 1
    ref = O.prefill_attn(qq[b:b + 1], *[c[b:b + 1] for c in oc], T=T)
    assert O.rel_fro(first[b:b + 1].cpu().numpy(), ref) <= OUT_TOL
    out = torch.empty_like(first)
    mismatches = 0
    for _ in range(200):
        out.fill_(float("nan"))
        q.quarot_prefill_attn(qt, *g, out=out)
        mismatches += int(not torch.equal(out, first))
    q.quarot_check_error()
    assert mismatches == 0


# ---------------------------------------------------------------- asymmetric KV (next row f1)
def _caches_asym(shape_like, T_max):
    B, _, H, d = shape_like
    c = [np.zeros((B, H, T_max, d // 2), np.uint8), np.zeros((B, H, T_max), np.float16),
         np.zeros((B, H, T_max), np.int16)]
    return c + [x.copy() for x in c]


def _check_asym_vectors(r, clip, codes, scales, zeros):
    """GPU (codes, scale, zero) of rotated vectors r against the oracle quantizer."""
    q_ref, s_ref, z_ref = O.quantize_asym_rows(r, clip)
    assert np.all(np.abs(scales.astype(np.float64) - s_ref.astype(np.float64)) <= _fp16_ulp(s_ref))
    same = (scales == s_ref)
    sf = s_ref.astype(np.float64)
    a_min = clip * r.astype(np.float64).min(axis=-1)
    zb = np.abs(np.abs(a_min / sf - np.floor(a_min / sf)) - 0.5) < 1e-4  # z on a rounding boundary
    dz = np.abs(zeros.astype(np.int64) - z_ref.astype(np.int64))
    assert np.all(dz[same] <= zb[same].astype(np.int64)), "zero points differ away from a boundary"
    ok = same & (zeros == z_ref)
    y = r.astype(np.float64) / sf[..., None]
    near = np.abs(np.abs(y - np.floor(y)) - 0.5) < 1e-4
    bad = (codes != q_ref) & ~near & ok[..., None]
    assert not bad.any(), f"{int(bad.sum())} codes differ away from a rounding boundary"


@pytest.mark.parametrize("d", [64, 128, 256])
def test_kv_write_asym_parity(q, d):
    B, T, H, T_max, t0, clip = 3, 37, 2, 64, 5, 0.95
    k = W.kv_tensors(B, T, H, d, 2, 20.0, 51)
    v = W.kv_tensors(B, T, H, d, 2, 20.0, 52)
    gc = q.new_kv_cache_asym(B, H, T_max, d, DEV)
    q.quarot_kv_write_asym(_t(k), _t(v), t0, *gc, clip_ratio=clip)
    gk, gks, gkz, gv, gvs, gvz = [t.cpu().numpy() for t in gc]
    for src, codes, scales, zeros in ((k, gk, gks, gkz), (v, gv, gvs, gvz)):
        r = O.rotate(src, None)  # [B, T, H, d]
        _check_asym_vectors(r, clip, O.unpack_uint4(codes[:, :, t0:t0 + T].transpose(0, 2, 1, 3)),
                            scales[:, :, t0:t0 + T].transpose(0, 2, 1), zeros[:, :, t0:t0 + T].transpose(0, 2, 1))
        assert np.all(codes[:, :, :t0] == 0) and np.all(codes[:, :, t0 + T:] == 0)
        assert np.all(zeros[:, :, :t0] == 0) and np.all(zeros[:, :, t0 + T:] == 0)


@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("T", [997, 1003])
def test_decode_unaligned_cache_rows(q, asym, T):
    """A cache capacity that is not a multiple of 8 tokens: the scale rows (and
    zero-point rows) of the (sequence, KV head) rows start off 16-byte
    boundaries, so bulk copies cannot fetch them and every tile takes the
    plain-load path; T 997 also ends on a ragged tile, T 1003 fills the cache."""
    B, Hkv, G, d, T_max = 2, 2, 4, 128, 1003
    k = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 71 + T)
    v = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 72 + T)
    qq = W.query(B, Hkv * G, d, 73 + T)
    if asym:
        oc = _caches_asym(k.shape, T_max)
        O.kv_write_asym(k, v, 0, *oc, clip_ratio=0.95)
    else:
        oc = _caches(k.shape, T_max)
        O.kv_write(k, v, 0, *oc)
    for unrot in (False, True):
        if asym:
            out = q.quarot_decode_attn_asym(_t(qq), *[_t(c) for c in oc], T=T, unrotate_out=unrot)
            ref = O.decode_attn_asym(qq, *oc, T=T, unrotate=unrot)
        else:
            out = q.quarot_decode_attn(_t(qq), *[_t(c) for c in oc], T=T, unrotate_out=unrot)
            ref = O.decode_attn(qq, *oc, T=T, unrotate=unrot)
        assert O.rel_fro(out.cpu().numpy(), ref) <= OUT_TOL
        _check_per_head(out.cpu().numpy(), ref)


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("T", [1, 17, 300, 1000])
def test_decode_asym_parity(q, G, T):
    B, Hkv, d, T_max = 2, 2, 128, 1024
    k = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 61 + T)
    v = W.kv_tensors(B, T, Hkv, d, 2, 20.0, 62 + T)
    qq = W.query(B, Hkv * G, d, 63 + T)
    oc = _caches_asym(k.shape, T_max)
    O.kv_write_asym(k, v, 0, *oc)
    for unrot in (False, True):
        out = q.quarot_decode_attn_asym(_t(qq), *[_t(c) for c in oc], T=T, unrotate_out=unrot)
        ref = O.decode_attn_asym(qq, *oc, T=T, unrotate=unrot)
        assert O.rel_fro(out.cpu().numpy(), ref) <= OUT_TOL


def test_kv4_config_full_asym(q):
    """B16 x T4096 x Hkv8 x Hq32 with the asymmetric cache: append and decode at
    full size; oracle on two sequences."""
    k, v, qq = W.kv_inputs("kv4")
    B, T, Hkv, d = k.shape
    gc = q.new_kv_cache_asym(B, Hkv, T, d, DEV)
    q.quarot_kv_write_asym(_t(k), _t(v), 0, *gc)
    out = q.quarot_decode_attn_asym(_t(qq), *gc, T=T)
    q.quarot_check_error()
    out = out.cpu().numpy()
    gnp = [t.cpu().numpy() for t in gc]
    for b in (0, B - 1):
        oc = _caches_asym(k[b:b + 1].shape, T)
        O.kv_write_asym(k[b:b + 1], v[b:b + 1], 0, *oc)
        for i, name in ((1, "k_s"), (4, "v_s")):
            g_, o_ = gnp[i][b], oc[i][0]
            assert np.all(np.abs(g_.astype(np.float64) - o_.astype(np.float64)) <= _fp16_ulp(o_)), name
        ref = O.decode_attn_asym(qq[b:b + 1], *oc, T=T)
        assert O.rel_fro(out[b:b + 1], ref) <= OUT_TOL


def test_zz_scale_differences_are_rare(q):
    """Over every check_quant call of this module (run last: pytest keeps file
    order), fewer than 1e-3 of the rows have a scale one fp16 ulp away from
    the oracle's."""
    t = _SCALE_TALLY
    if t["rows"] == 0:
        pytest.skip("no quantizer checks ran")
    assert t["differ"] < 1e-3 * t["rows"], t


# ---------------------------------------------------------------- row-strided inputs (ld_x > d)
@pytest.mark.parametrize("entry,d", [("rotate", 256), ("rotate", 3072), ("rotate", 4096), ("rotate", 12288),
                                     ("fp16", 1024), ("fp16", 4096), ("fp16", 12288),
                                     ("rmsnorm", 4096), ("rmsnorm", 12288),
                                     ("a8", 4096), ("a8", 12288), ("crosshead", 4096)])
def test_rotate_family_row_strided(q, entry, d):
    """A column slice of a wider tensor (row stride d + 72, column offset 8):
    the entry points read it through their ld argument and return exactly
    what they return for the same rows made contiguous -- every kernel form
    (generic, segment, staged persistent with bulk row copies)."""
    M = 300
    x = W.activations(M, d, W.outlier_channels(d, 4, 7 + d), 50.0, 13 + d)
    wide = torch.zeros((M, d + 72), dtype=torch.float16, device=DEV)
    wide[:, 8:8 + d] = _t(x)
    xs = wide[:, 8:8 + d]
    assert xs.stride(0) == d + 72 and not xs.is_contiguous()
    xc = xs.contiguous()
    s = _t(W.random_signs(d, 5 + d))
    if entry == "rotate":
        got, ref = q.quarot_rotate_quant(xs, s, want_rot=True), q.quarot_rotate_quant(xc, s, want_rot=True)
    elif entry == "fp16":
        got, ref = q.quarot_rotate_quant_fp16(xs, s, want_rot=True), q.quarot_rotate_quant_fp16(xc, s, want_rot=True)
    elif entry == "rmsnorm":
        got, ref = q.quarot_rmsnorm_rotate_quant(xs, s, want_rot=True), q.quarot_rmsnorm_rotate_quant(xc, s, want_rot=True)
    elif entry == "a8":
        got, ref = q.quarot_rotate_quant_a8(xs, s), q.quarot_rotate_quant_a8(xc, s)
    else:
        got, ref = q.quarot_crosshead_rotate_quant(xs, 32, want_rot=True), q.quarot_crosshead_rotate_quant(xc, 32, want_rot=True)
    q.quarot_check_error()
    for g, r in zip(got, ref):
        assert torch.equal(g, r)
    # the padding columns were not written and the contiguous path agrees with the oracle elsewhere
    assert torch.count_nonzero(wide[:, :8]) == 0 and torch.count_nonzero(wide[:, 8 + d:]) == 0


# 1024 CTAs of work each: more than any one wave (at most 8 CTAs of 256
# threads per SM, keys and values sharing it) on this GPU
@pytest.mark.parametrize("d,B,H,T", [(64, 4, 8, 4096), (128, 2, 8, 4096), (256, 2, 4, 4096)])
@pytest.mark.parametrize("asym", [False, True])
def test_kv_write_grid_stride(q, d, B, H, T, asym):
    """Appends large enough (more items than one wave of resident CTAs) that
    the KV write walks them with its grid stride and register prefetch; every
    vector against the oracle, with an offset and untouched slots around it."""
    T_max, t0 = T + 24, 16
    k = W.kv_tensors(B, T, H, d, 2, 20.0, 71 + d)
    v = W.kv_tensors(B, T, H, d, 2, 20.0, 72 + d)
    if asym:
        gc = q.new_kv_cache_asym(B, H, T_max, d, DEV)
        q.quarot_kv_write_asym(_t(k), _t(v), t0, *gc, clip_ratio=0.95)
        gk, gks, gkz, gv, gvs, gvz = [t.cpu().numpy() for t in gc]
        parts = ((k, gk, gks, gkz), (v, gv, gvs, gvz))
    else:
        gc = q.new_kv_cache(B, H, T_max, d, DEV)
        q.quarot_kv_write(_t(k), _t(v), t0, *gc)
        gk, gks, gv, gvs = [t.cpu().numpy() for t in gc]
        parts = ((k, gk, gks, None), (v, gv, gvs, None))
    for src, codes, scales, zeros in parts:
        r = O.rotate(src, None)  # [B, T, H, d]
        if asym:
            _check_asym_vectors(r, 0.95, O.unpack_uint4(codes[:, :, t0:t0 + T].transpose(0, 2, 1, 3)),
                                scales[:, :, t0:t0 + T].transpose(0, 2, 1), zeros[:, :, t0:t0 + T].transpose(0, 2, 1))
        else:
            q_ref, s_ref = O.quantize_rows(r, 1.0)
            s_gpu = scales[:, :, t0:t0 + T].transpose(0, 2, 1)
            c_gpu = O.unpack_int4(codes[:, :, t0:t0 + T].transpose(0, 2, 1, 3))
            assert np.all(np.abs(s_gpu.astype(np.float64) - s_ref.astype(np.float64)) <= _fp16_ulp(s_ref))
            assert not ((c_gpu != q_ref) & ~O.boundary_mask(r, s_ref)).any()
        assert np.all(codes[:, :, :t0] == 0) and np.all(codes[:, :, t0 + T:] == 0)
        assert np.all(scales[:, :, :t0] == 0) and np.all(scales[:, :, t0 + T:] == 0)


# ---------------------------------------------------------------- the layer object
@pytest.mark.parametrize("K,N", [(4096, 1024), (12288, 512), (256, 1000)])
def test_quarot_linear_layer(q, K, N):
    """QuarotLinear: the two-call chain (weights prepared once), against the
    oracle's layer and bit-identical to calling the entry points by hand;
    leading batch dimensions pass through."""
    x, w, s = W.layer_inputs("down_proj" if K == 12288 else ("rotq4096" if K == 4096 else "tiny"), M=96, N=N)
    x = x[:96, :K]
    w = w[:N, :K]
    s = s[:K]
    lin = q.QuarotLinear(_t(w), _t(s))
    y = lin(_t(x).view(2, 48, K))
    assert y.shape == (2, 48, N)
    wq, wsc, _ = q.quarot_rotate_quant(_t(w), _t(s))
    aq, asc, _ = q.quarot_rotate_quant(_t(x), _t(s))
    yh, _ = q.quarot_w4a4_gemm(aq, asc, wq, wsc)
    q.quarot_check_error()
    assert torch.equal(y.view(96, N), yh)
    oa, osx, _ = O.rotate_quant(x, s)
    ow, osw, _ = O.rotate_quant(w, s)
    _, oy = O.w4a4_gemm(oa, osx, ow, osw)
    assert O.rel_fro(y.view(96, N).cpu().numpy(), oy) <= OUT_TOL


@pytest.mark.parametrize("asym", [False, True])
def test_quarot_kv_cache_object(q, asym):
    """QuarotKVCache: a 300-token prompt appended in two chunks, its prompt
    attention (symmetric cache), then three one-token decode steps, each
    against the oracle's cache and attention at the same length."""
    B, Hkv, G, d, T_max = 2, 2, 4, 128, 512
    cache = q.QuarotKVCache(B, Hkv, T_max, d, DEV, asym=asym)
    oc = _caches_asym((B, 0, Hkv, d), T_max) if asym else _caches((B, 0, Hkv, d), T_max)
    owrite = (lambda k, v, t: O.kv_write_asym(k, v, t, *oc)) if asym else (lambda k, v, t: O.kv_write(k, v, t, *oc))
    k = W.kv_tensors(B, 300, Hkv, d, 2, 20.0, 91)
    v = W.kv_tensors(B, 300, Hkv, d, 2, 20.0, 92)
    for lo, hi in ((0, 180), (180, 300)):
        cache.append(_t(k[:, lo:hi]), _t(v[:, lo:hi]))
        owrite(k[:, lo:hi], v[:, lo:hi], lo)
    assert cache.length == 300
    if not asym:
        qp = W.prefill_query(B, 300, Hkv * G, d, 93)
        out = cache.prefill(_t(qp))
        assert O.rel_fro(out.cpu().numpy(), O.prefill_attn(qp, *oc, T=300)) <= OUT_TOL
    else:
        with pytest.raises(q.QuarotError):
            cache.prefill(_t(W.prefill_query(B, 300, Hkv * G, d, 93)))
    for step in range(3):
        kn = W.kv_tensors(B, 1, Hkv, d, 2, 20.0, 100 + step)
        vn = W.kv_tensors(B, 1, Hkv, d, 2, 20.0, 200 + step)
        cache.append(_t(kn), _t(vn))
        owrite(kn, vn, 300 + step)
        qq = W.query(B, Hkv * G, d, 300 + step)
        out = cache.decode(_t(qq))
        T = 301 + step
        ref = O.decode_attn_asym(qq, *oc, T=T) if asym else O.decode_attn(qq, *oc, T=T)
        assert O.rel_fro(out.cpu().numpy(), ref) <= OUT_TOL
    q.quarot_check_error()
    with pytest.raises(q.QuarotError):
        cache.append(_t(W.kv_tensors(B, 300, Hkv, d, 2, 20.0, 5)), _t(W.kv_tensors(B, 300, Hkv, d, 2, 20.0, 6)))
