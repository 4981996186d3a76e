"""Pins of the CPU oracle to what the QuaRot pages and mathematics fix.

Each test checks the oracle against something other than itself: a
hand-worked fixture, a closed form, an independent brute-force definition,
or an invariant the pages state.  A plausible slip in the oracle (a dropped
sign vector, a transposed Hadamard, the wrong Kronecker order, the wrong
rounding mode, a swapped nibble) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W


# ---------------------------------------------------------------- Hadamard
def _sylvester_entry(k, j):
    """Closed form of the Sylvester matrix: (-1)^popcount(k & j)."""
    return -1 if bin(k & j).count("1") % 2 else 1


def _euler_chi(a, q=11):
    """Legendre symbol by Euler's criterion a^((q-1)/2) mod q."""
    a %= q
    if a == 0:
        return 0
    return 1 if pow(a, (q - 1) // 2, q) == 1 else -1


def _paley_entry(i, j):
    """Paley I entry written from the definition H = I + S, S = [[0,1],[-1,Q]]."""
    if i == j:
        return 1
    if i == 0:
        return 1
    if j == 0:
        return -1
    return _euler_chi((j - 1) - (i - 1))


def test_sylvester_h4_golden(golden):
    g = golden("sylvester_h4.txt")["_rows"]
    assert np.array_equal(O.sylvester(4), np.array(g))


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 64, 256, 1024, 4096])
def test_sylvester_orthogonal_integer(n):
    # integer sums below 2^53 are exact in float64, so BLAS gives H H^T exactly
    H = O.sylvester(n)
    rows = np.arange(n) if n <= 1024 else np.random.default_rng(n).choice(n, 256, replace=False)
    sub = H[rows].astype(np.float64)
    prod = sub @ H.astype(np.float64).T
    ref = np.zeros((len(rows), n))
    ref[np.arange(len(rows)), rows] = n
    assert np.array_equal(prod, ref)
    assert np.array_equal(H, H.T)  # symmetric, so H H = n I as the pages use


@pytest.mark.parametrize("n", [2, 8, 32, 128])
def test_sylvester_closed_form(n):
    ref = np.array([[_sylvester_entry(k, j) for j in range(n)] for k in range(n)])
    assert np.array_equal(O.sylvester(n), ref)


def test_paley12_definition_and_orthogonality(golden):
    g = golden("paley12_column_sums.txt")
    H = O.paley12().astype(np.int64)
    ref = np.array([[_paley_entry(i, j) for j in range(12)] for i in range(12)])
    assert np.array_equal(H, ref)
    assert np.array_equal(H @ H.T, 12 * np.eye(12, dtype=np.int64))
    assert not np.array_equal(H, H.T)
    residues = sorted({(x * x) % 11 for x in range(1, 11)})
    assert residues == [int(v) for v in g["residues"]]
    assert [O.legendre(a, 11) for a in range(11)] == [_euler_chi(a) for a in range(11)]
    assert list(H.sum(axis=1)) == [int(v) for v in g["row_sums"]]
    assert list(H.sum(axis=0)) == [int(v) for v in g["col_sums"]]


def test_kronecker_factorisation_of_sylvester():
    # H_{n*d} = (I_n (x) H_d)(H_n (x) I_d) for powers of two (Stage 1c identity)
    n, d = 16, 64
    lhs = O.sylvester(n * d).astype(np.float64)
    a = np.kron(np.eye(n), O.sylvester(d).astype(np.float64))
    b = np.kron(O.sylvester(n).astype(np.float64), np.eye(d))
    assert np.array_equal(lhs, a @ b)


def test_hadamard_12288_rows_orthogonal_and_order():
    H = O.hadamard(12288)
    assert H.shape == (12288, 12288)
    rng = np.random.default_rng(0)
    rows = rng.choice(12288, 48, replace=False)
    sub = H[rows].astype(np.float64)
    assert np.array_equal(sub @ sub.T, 12288 * np.eye(48))
    # entry [(a,b),(c,e)] = H12[a,c] * H1024[b,e] with index a*1024 + b
    for (i, j) in [(0, 0), (1025, 3), (5000, 11000), (12287, 1024), (2047, 4095)]:
        a, b = divmod(i, 1024)
        c, e = divmod(j, 1024)
        assert H[i, j] == _paley_entry(a, c) * _sylvester_entry(b, e)


def test_hadamard_24_brute_force():
    H = O.hadamard(24)
    ref = np.array([[_paley_entry(i // 2, j // 2) * _sylvester_entry(i % 2, j % 2)
                     for j in range(24)] for i in range(24)])
    assert np.array_equal(H, ref)


def test_unsupported_width():
    with pytest.raises(ValueError):
        O.hadamard(20)


# ---------------------------------------------------------------- rotation
def _brute_rotate(x, s, entry):
    d = len(x)
    return [sum(s[k] * float(x[k]) * entry(k, j) for k in range(d)) / math.sqrt(d) for j in range(d)]


@pytest.mark.parametrize("d", [2, 4, 8, 16])
def test_rotation_brute_force_sylvester(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal(d).astype(np.float16)
    s = W.random_signs(d, 7 + d)
    got = O.rotate(x[None], s)[0]
    ref = np.array(_brute_rotate(x, s, _sylvester_entry), dtype=np.float32)
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-7)


def test_rotation_brute_force_kronecker_24():
    rng = np.random.default_rng(24)
    x = rng.standard_normal(24).astype(np.float16)
    s = W.random_signs(24, 31)
    got = O.rotate(x[None], s)[0]
    ref = np.array(_brute_rotate(x, s, lambda k, j: _paley_entry(k // 2, j // 2) * _sylvester_entry(k % 2, j % 2)),
                   dtype=np.float32)
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("d", [256, 4096, 12288])
def test_one_hot_spreads_to_plus_minus_inv_sqrt_d(d):
    # a single loud coordinate comes out at +-1/sqrt(d) everywhere (explainer)
    x = np.zeros((3, d), dtype=np.float16)
    x[0, 0] = 1.0
    x[1, d // 3] = 1.0
    x[2, d - 1] = -2.0
    r = O.rotate(x, None)
    assert np.allclose(np.abs(r[0]), 1 / math.sqrt(d), rtol=1e-6)
    assert np.allclose(r[0], 1 / math.sqrt(d), rtol=1e-6)  # row 0 of H is all ones
    assert np.allclose(np.abs(r[1]), 1 / math.sqrt(d), rtol=1e-6)
    assert np.allclose(np.abs(r[2]), 2 / math.sqrt(d), rtol=1e-6)


def test_signs_act_on_inputs_not_outputs():
    d = 256
    s = W.random_signs(d, 5)
    i = 17
    x = np.zeros((1, d), dtype=np.float16)
    x[0, i] = 1.0
    r = O.rotate(x, s)[0]
    row = np.array([_sylvester_entry(i, j) for j in range(d)], dtype=np.float64)
    assert np.allclose(r, s[i] * row / math.sqrt(d), rtol=1e-6)


def test_constant_vector_pins_convention_sylvester():
    d = 4096
    r = O.rotate(np.ones((1, d), dtype=np.float16), None)[0]
    ref = np.zeros(d)
    ref[0] = math.sqrt(d)
    assert np.allclose(r, ref, atol=1e-4)


def test_constant_vector_pins_convention_and_kron_order_12288(golden):
    # x @ (H12 (x) H1024) for x = 1: column sums of H12 times 1024 at b = 0
    g = golden("paley12_column_sums.txt")
    colsum = [int(v) for v in g["col_sums"]]
    d = 12288
    r = O.rotate(np.ones((1, d), dtype=np.float16), None)[0]
    ref = np.zeros(d)
    for c in range(12):
        ref[c * 1024] = colsum[c] * 1024 / math.sqrt(d)
    assert np.allclose(r, ref, atol=1e-3)


@pytest.mark.parametrize("d", [256, 4096, 12288])
def test_norm_preservation(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((4, d)).astype(np.float16)
    s = W.random_signs(d, 3)
    r = O.rotate_f64(x, s)
    assert np.allclose(np.linalg.norm(r, axis=1), np.linalg.norm(x.astype(np.float64), axis=1), rtol=1e-12)


@pytest.mark.parametrize("d", [4096, 12288])
def test_invariance_error_fp32_roundoff(d):
    # ||(XQ)(WQ)^T - XW^T|| / ||XW^T|| at fp32 round-off: "a few times 1e-7"
    x, w, s = W.layer_inputs("down_proj" if d == 12288 else "sweep", M=32, N=48)
    xr = O.rotate(x, s)
    wr = O.rotate(w, s)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    got32 = xr.astype(np.float32) @ wr.astype(np.float32).T
    err32 = np.linalg.norm(got32 - ref) / np.linalg.norm(ref)
    assert err32 < 2e-6
    got64 = O.rotate_f64(x, s) @ O.rotate_f64(w, s).T
    assert np.linalg.norm(got64 - ref) / np.linalg.norm(ref) < 1e-12


def _rmsnorm(x):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True))


@pytest.mark.parametrize("d", [256, 12288])
def test_rmsnorm_commutation(d):
    # RMSNorm(X) = RMSNorm(X Q^T) Q with Q = diag(s) H / sqrt(d)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, d))
    s = W.random_signs(d, 9).astype(np.float64)
    H = O.hadamard(d).astype(np.float64)
    xqt = (x @ H.T) / math.sqrt(d) * s[None, :]  # X Q^T = X H^T diag(s) / sqrt(d)
    lhs = O.rotate_f64(_rmsnorm(xqt), s.astype(np.int8))
    assert np.allclose(lhs, _rmsnorm(x), rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- fused RMSNorm + rotation + quant
def test_rmsnorm_rotate_quant_worked_example(golden):
    g = golden("rmsnorm_rotate_quant_worked.txt")
    x = np.array([[float(v) for v in g["x"]]], dtype=np.float16)
    eps = float(g["eps"][0])
    assert np.array_equal(O.rmsnorm(x, eps)[0], np.array([float(v) for v in g["y"]]))
    packed, S, r = O.rmsnorm_rotate_quant(x, None, eps)
    assert np.allclose(r[0], np.array([float(v) for v in g["rotated"]]), rtol=1e-7, atol=1e-7)
    assert float(S[0]) == float(g["scale"][0])
    assert np.array_equal(O.unpack_int4(packed)[0], np.array([int(v) for v in g["codes"]]))
    assert np.array_equal(packed[0], np.array([int(v) for v in g["packed"]], dtype=np.uint8))


def test_rmsnorm_eps_inside_the_root():
    # mean(x^2) = 1, eps = 3: 1 / sqrt(1 + 3) = 1/2 exactly
    assert np.array_equal(O.rmsnorm(np.ones((1, 4)), 3.0), np.full((1, 4), 0.5))


@pytest.mark.parametrize("d", [16, 4096])
def test_rmsnorm_unit_mean_square_and_scale_invariance(d):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, d)) * rng.uniform(0.1, 100.0, (5, 1))
    y = O.rmsnorm(x, 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-12)
    assert np.allclose(O.rmsnorm(7.5 * x, 0.0), y, rtol=1e-12)


def test_rmsnorm_commutes_with_the_rotation():
    # the pages' identity RMSNorm(X) = RMSNorm(X Q^T) Q, on the oracle's RMSNorm
    d = 4096
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, d))
    s = W.random_signs(d, 11)
    H = O.hadamard(d).astype(np.float64)
    xqt = (x @ H.T) / math.sqrt(d) * s.astype(np.float64)[None, :]
    assert np.allclose(O.rotate_f64(O.rmsnorm(xqt, 0.0), s), O.rmsnorm(x, 0.0), rtol=1e-10, atol=1e-12)


def test_rmsnorm_rotate_quant_zero_row_and_row_scale_freedom():
    packed, S, r = O.rmsnorm_rotate_quant(np.zeros((1, 256), np.float16), None, 1e-6)
    assert np.all(packed == 0) and np.all(r == 0)
    assert float(S[0]) == float(np.float16(1e-5 / 7))
    # a power-of-two factor on the row leaves the normalized row, hence every
    # output, unchanged (eps = 0)
    x, _, s = W.layer_inputs("tiny")
    a = O.rmsnorm_rotate_quant(x, s, 0.0)
    b = O.rmsnorm_rotate_quant((x.astype(np.float32) * 0.25).astype(np.float16), s, 0.0)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))


# ---------------------------------------------------------------- cross-head Hadamard (next row f3)
def test_crosshead_worked_example(golden):
    g = golden("crosshead_rotate_quant_worked.txt")
    z = np.array([[float(v) for v in g["z"]]], dtype=np.float16)
    packed, S, r = O.crosshead_rotate_quant(z, int(g["nh"][0]))
    assert np.allclose(r[0], np.array([float(v) for v in g["rotated"]]), rtol=1e-6)
    assert float(S[0]) == float(g["scale"][0])
    assert np.array_equal(O.unpack_int4(packed)[0], np.array([int(v) for v in g["codes"]]))
    assert np.array_equal(packed[0], np.array([int(v) for v in g["packed"]], dtype=np.uint8))


def test_crosshead_after_headwise_is_the_full_hadamard():
    # the pages' identity H_{nh dh} = (I_nh (x) H_dh)(H_nh (x) I_dh): the head-wise
    # rotation (already in the rotated values) followed by the cross-head one is
    # the full Sylvester rotation of the concatenated heads
    nh, dh = 32, 128
    rng = np.random.default_rng(12)
    z = rng.standard_normal((3, nh * dh))
    headwise = O.rotate_f64(z.reshape(3, nh, dh), None).reshape(3, nh * dh)
    assert np.allclose(O.crosshead_rotate(headwise, nh), O.rotate_f64(z, None), rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("nh", [1, 4, 32])
def test_crosshead_norm_and_identity(nh):
    rng = np.random.default_rng(13)
    z = rng.standard_normal((4, nh * 64)).astype(np.float32)
    r = O.crosshead_rotate(z, nh).astype(np.float64)
    assert np.allclose(np.linalg.norm(r, axis=1), np.linalg.norm(z.astype(np.float64), axis=1), rtol=1e-6)
    if nh == 1:
        assert np.array_equal(r, z.astype(np.float64))
    # within-head position j only mixes with the same j of other heads
    one = np.zeros((1, nh * 64), np.float32)
    one[0, 5] = 1.0
    nz = np.nonzero(O.crosshead_rotate(one, nh)[0])[0]
    assert np.array_equal(nz % 64, np.full(nh, 5)) and len(nz) == nh


# ---------------------------------------------------------------- quantizer
def _golden_quant(g):
    x = np.array([float(v) for v in g["x"]], dtype=np.float32)
    return (float(g["clip"][0]), x, float(g["scale"][0]), np.array([int(v) for v in g["codes"]]),
            np.array([int(v, 16) for v in g["bytes"]], dtype=np.uint8))


@pytest.mark.parametrize("name", ["quant_pack_worked.txt", "quant_clip09_worked.txt"])
def test_quantizer_worked_examples(golden, name):
    clip, x, scale, codes, byts = _golden_quant(golden(name))
    q, S = O.quantize_rows(x[None], clip)
    assert float(S[0]) == scale
    assert np.array_equal(q[0], codes)
    assert np.array_equal(O.pack_int4(q)[0], byts)
    assert np.array_equal(O.unpack_int4(byts[None])[0], codes)


def test_pack_nibble_order_and_twos_complement():
    assert O.pack_int4(np.array([[-8, 7]]))[0, 0] == 0x78
    assert O.pack_int4(np.array([[7, -8]]))[0, 0] == 0x87
    assert O.pack_int4(np.array([[-1, -1]]))[0, 0] == 0xFF
    assert O.pack_int4(np.array([[1, 0]]))[0, 0] == 0x01
    allc = np.array(np.meshgrid(np.arange(-8, 8), np.arange(-8, 8))).reshape(2, -1).T
    assert np.array_equal(O.unpack_int4(O.pack_int4(allc)), allc)


def test_zero_row_and_floor():
    q, S = O.quantize_rows(np.zeros((1, 64), dtype=np.float32))
    assert np.all(q == 0)
    assert float(S[0]) == float(np.float16(1e-5 / 7))


def test_quantizer_invariants_random():
    x, _, s = W.layer_inputs("tiny")
    r = O.rotate(x, s)
    q, S = O.quantize_rows(r, 1.0)
    assert q.min() >= -7 and q.max() <= 7  # -8 unreachable without clipping
    am = np.argmax(np.abs(r), axis=1)
    assert np.all(np.abs(q[np.arange(len(q)), am]) == 7)
    Sf = S.astype(np.float64)[:, None]
    err = np.abs(r.astype(np.float64) - Sf * q)
    assert np.all(err <= Sf / 2 * (1 + 1e-6) + 1e-12)
    q9, S9 = O.quantize_rows(r, 0.9)
    assert q9.min() >= -8 and q9.max() <= 7
    assert (q9 == -8).any() or (q9 == 7).any()


def test_rounding_is_half_even():
    x = np.array([[7.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.5, -6.5]], dtype=np.float32)
    q, S = O.quantize_rows(x)
    assert float(S[0]) == 1.0
    assert list(q[0]) == [7, 0, 2, 2, 0, -2, 4, -6]


# ---------------------------------------------------------------- GEMM
def test_int_gemm_brute_force():
    a = W.int4_codes(4, 32, 1)
    w = W.int4_codes(3, 32, 2)
    ref = [[sum(int(a[i, k]) * int(w[j, k]) for k in range(32)) for j in range(3)] for i in range(4)]
    assert np.array_equal(O.int_gemm(a, w), np.array(ref))


def test_int_gemm_adversarial_extremes():
    K = 12288
    a = np.full((2, K), -8, dtype=np.int8)
    w = np.stack([np.full(K, -8, dtype=np.int8), np.full(K, 7, dtype=np.int8)])
    acc = O.int_gemm(a, w)
    assert acc[0, 0] == 64 * K and acc[0, 1] == -56 * K


def test_packed_gemm_matches_unpacked():
    a = W.int4_codes(5, 64, 3)
    w = W.int4_codes(7, 64, 4)
    sx = W.fp16_scales(5, 5)
    sw = W.fp16_scales(7, 6)
    acc, y = O.w4a4_gemm(O.pack_int4(a), sx, O.pack_int4(w), sw)
    assert np.array_equal(acc, O.int_gemm(a, w))
    exact = acc * sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    assert np.all(np.abs(y.astype(np.float64) - exact) <= np.abs(exact) * 2.0 ** -10 + 1e-7)


def test_dequant_exact_cases():
    y = O.dequant(np.array([[100, -3]]), np.array([0.5], dtype=np.float16), np.array([0.25, 2.0], dtype=np.float16))
    assert y.dtype == np.float16 and list(y[0]) == [12.5, -3.0]


def test_method_effect_rotation_beats_naive():
    # rotated W4A4 error is well below naive W4A4 error on outlier inputs
    x, w, s = W.layer_inputs("tiny")
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    ap, asx, _ = O.rotate_quant(x, s)
    wp, wsx, _ = O.rotate_quant(w, s)
    _, y_rot = O.w4a4_gemm(ap, asx, wp, wsx)
    qa, sa = O.quantize_rows(x.astype(np.float32))
    qw, sw = O.quantize_rows(w.astype(np.float32))
    _, y_naive = O.w4a4_gemm(O.pack_int4(qa), sa, O.pack_int4(qw), sw)
    e_rot = O.rel_fro(y_rot, ref)
    e_naive = O.rel_fro(y_naive, ref)
    assert e_rot < 0.75 * e_naive, (e_rot, e_naive)


# ---------------------------------------------------------------- KV + decode
def test_kv_quant_one_hot_layout():
    B, T, H, d = 2, 3, 2, 128
    k = np.zeros((B, T, H, d), dtype=np.float16)
    k[1, 2, 1, 5] = 3.0
    packed, S = O.kv_quant(k)
    assert packed.shape == (B, H, T, d // 2) and S.shape == (B, H, T)
    codes = O.unpack_int4(packed[1, 1, 2])
    assert np.all(np.abs(codes) == 7)
    row = np.array([_sylvester_entry(5, j) for j in range(d)])
    assert np.array_equal(np.sign(codes), row)
    assert float(S[1, 1, 2]) == float(np.float16(3.0 / math.sqrt(d) / 7))
    assert np.all(O.unpack_int4(packed[0]) == 0)


def _fill_cache(k, v, T_max):
    B, T, H, d = k.shape
    kc = np.zeros((B, H, T_max, d // 2), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((B, H, T_max), np.float16)
    vs = np.zeros_like(ks)
    O.kv_write(k, v, 0, kc, ks, vc, vs)
    return kc, ks, vc, vs


def test_score_invariance():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((5, 128))
    k = rng.standard_normal((7, 128))
    assert np.allclose(O.rotate_f64(q, None) @ O.rotate_f64(k, None).T, q @ k.T, rtol=1e-12, atol=1e-12)


def test_decode_single_token_returns_dequantized_value():
    k, v, q = W.kv_inputs(B=2, T=1)
    kc, ks, vc, vs = _fill_cache(k, v, 4)
    out = O.decode_attn(q, kc, ks, vc, vs, T=1)
    Hq, Hkv = q.shape[1], k.shape[2]
    for h in range(Hq):
        g = h // (Hq // Hkv)
        vd = O.unpack_int4(vc[:, g, 0]).astype(np.float64) * vs[:, g, 0].astype(np.float64)[:, None]
        assert np.allclose(out[:, h], vd, rtol=1e-12, atol=1e-12)


def test_decode_identical_keys_average_values():
    B, T, H, d = 1, 5, 1, 128
    rng = np.random.default_rng(4)
    kk = np.repeat(rng.standard_normal((1, 1, 1, d)), T, axis=1).astype(np.float16)
    vv = rng.standard_normal((B, T, H, d)).astype(np.float16)
    kc, ks, vc, vs = _fill_cache(kk, vv, 8)
    q = rng.standard_normal((B, 2, d)).astype(np.float16)
    out = O.decode_attn(q, kc, ks, vc, vs, T=T)
    vd = O.unpack_int4(vc[0, 0, :T]).astype(np.float64) * vs[0, 0, :T].astype(np.float64)[:, None]
    assert np.allclose(out[0, 0], vd.mean(axis=0), rtol=1e-10, atol=1e-12)
    assert np.allclose(out[0, 1], vd.mean(axis=0), rtol=1e-10, atol=1e-12)


def test_decode_brute_force_tiny():
    # B=1, Hq=2, Hkv=1, d=4, T=3: softmax and weighted sum written with math.exp
    rng = np.random.default_rng(5)
    d, T = 4, 3
    k = rng.standard_normal((1, T, 1, d)).astype(np.float16)
    v = rng.standard_normal((1, T, 1, d)).astype(np.float16)
    q = rng.standard_normal((1, 2, d)).astype(np.float16)
    kc, ks, vc, vs = _fill_cache(k, v, T)
    out = O.decode_attn(q, kc, ks, vc, vs, T=T, unrotate=True)
    H4 = [[_sylvester_entry(i, j) for j in range(d)] for i in range(d)]
    kcodes = O.unpack_int4(kc[0, 0])
    vcodes = O.unpack_int4(vc[0, 0])
    for h in range(2):
        qr = [sum(float(q[0, h, i]) * H4[i][j] for i in range(d)) / 2.0 for j in range(d)]
        s = [sum(qr[j] * float(ks[0, 0, t]) * int(kcodes[t, j]) for j in range(d)) / 2.0 for t in range(T)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        p = [x / sum(e) for x in e]
        o = [sum(p[t] * float(vs[0, 0, t]) * int(vcodes[t, j]) for t in range(T)) for j in range(d)]
        o_un = [sum(o[i] * H4[i][j] for i in range(d)) / 2.0 for j in range(d)]
        assert np.allclose(out[0, h], o_un, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- FP16 online Hadamard (next row f4)
def test_fp16_hadamard_worked_example(golden):
    g = golden("fp16_hadamard_worked.txt")
    x = np.array([[float(v) for v in g["x"]]], dtype=np.float16)
    r = O.rotate_fp16_arith(x, None)
    assert np.array_equal(r[0], [float(v) for v in g["rot16"]])
    assert np.array_equal(O.rotate_f64(x, None)[0], [float(v) for v in g["exact"]])
    packed, S, rr = O.rotate_quant_fp16(x, None)
    assert float(S[0]) == float(g["scale"][0])
    assert O.quantize_rows(rr)[0][0].tolist() == [int(v) for v in g["codes"]]
    assert packed[0].tolist() == [int(v) for v in g["packed"]]


def test_fp16_hadamard_exact_when_representable():
    # small integers scaled by 1/4: every partial sum is an integer / 4 below 2^10
    rng = np.random.default_rng(31)
    x = (4 * rng.integers(-3, 4, (5, 16))).astype(np.float16)
    s = W.random_signs(16, 32)
    assert np.array_equal(O.rotate_fp16_arith(x, s), O.rotate_f64(x, s))


@pytest.mark.parametrize("d", [256, 4096, 3072])
def test_fp16_hadamard_error_bound(d):
    # after the fp16 scaling by c the row norm is |x| c sqrt(d) ~ |x|; each
    # butterfly stage is sqrt(2) times an orthogonal map plus a rounding of at
    # most u = 2^-11 relative per element, so ||r16 - r|| <= (log2 P + 2) u ||x||
    # (one more u for c itself); the Paley stage's 12 sequential sums add at
    # most 11 u sqrt(12) ||x||
    x, _, s = W.layer_inputs("rotq4096")
    x = x[:64, :d]
    s = s[:d]
    r16 = O.rotate_fp16_arith(x, s)
    r = O.rotate_f64(x, s)
    na = 12 if d % 12 == 0 else 1
    L = int(math.log2(d // na))
    u = 2.0 ** -11
    bound = (L + 2) * u + (11 * math.sqrt(12) * u if na == 12 else 0.0)
    err = np.linalg.norm(r16 - r, axis=1)
    nx = np.linalg.norm(x.astype(np.float64), axis=1)
    assert np.all(err <= bound * nx)
    # and it really is fp16 arithmetic, far above fp32 round-off
    assert np.median(err / nx) > 1e-5


def test_fp16_hadamard_brute_force_d8():
    # independent fp16 rounding through the IEEE binary16 codec of struct
    import struct

    def r16(v):
        return struct.unpack("<e", struct.pack("<e", v))[0]

    rng = np.random.default_rng(33)
    d = 8
    for _ in range(20):
        x = rng.standard_normal(d).astype(np.float16) * np.float16(300)
        s = rng.choice([-1, 1], d).astype(np.int8)
        c = r16(1.0 / math.sqrt(d))
        v = [r16(float(x[i]) * float(s[i]) * c) for i in range(d)]
        h = 1
        while h < d:
            for i in range(d):
                if i & h == 0:
                    a, b = v[i], v[i + h]
                    v[i], v[i + h] = r16(a + b), r16(a - b)
            h *= 2
        assert np.array_equal(O.rotate_fp16_arith(x[None, :], s)[0], v)


def test_fp16_hadamard_paley_sequence_d12():
    # d = 12 (P = 1): only the Paley-12 sums, accumulated in index order
    import struct

    def r16(v):
        return struct.unpack("<e", struct.pack("<e", v))[0]

    rng = np.random.default_rng(34)
    x = (rng.standard_normal(12) * 1000).astype(np.float16)
    c = r16(1.0 / math.sqrt(12))
    y = [r16(float(v) * c) for v in x]
    H = O.paley12()
    want = []
    for col in range(12):
        acc = 0.0
        for a in range(12):
            acc = r16(acc + int(H[a, col]) * y[a])
        want.append(acc)
    assert np.array_equal(O.rotate_fp16_arith(x[None, :], None)[0], want)


# ---------------------------------------------------------------- prefill attention (next row f4)
def _prefill_case(B, T, Hkv, G, d, seed):
    k = W.kv_tensors(B, T, Hkv, d, 2, 20.0, seed)
    v = W.kv_tensors(B, T, Hkv, d, 2, 20.0, seed + 1)
    qq = np.random.default_rng(seed + 2).standard_normal((B, T, Hkv * G, d)).astype(np.float16)
    kc, ks, vc, vs = _fill_cache(k, v, T)
    return qq, kc, ks, vc, vs


def test_prefill_rows_agree_with_decode():
    # the pinned decode is prefill's row: causal row i = decode of query i over
    # tokens 0..i; without the mask every row = decode over all T tokens
    B, T, Hkv, G, d = 1, 9, 2, 2, 128
    qq, kc, ks, vc, vs = _prefill_case(B, T, Hkv, G, d, 21)
    causal = O.prefill_attn(qq, kc, ks, vc, vs, T)
    full = O.prefill_attn(qq, kc, ks, vc, vs, T, causal=False, unrotate=True)
    for i in (0, 4, T - 1):
        assert np.allclose(causal[:, i], O.decode_attn(qq[:, i], kc, ks, vc, vs, T=i + 1), rtol=1e-12, atol=1e-12)
        assert np.allclose(full[:, i], O.decode_attn(qq[:, i], kc, ks, vc, vs, T=T, unrotate=True), rtol=1e-12,
                           atol=1e-12)
    # causal row 0 sees only token 0: its dequantized value
    v0 = O.unpack_int4(vc[:, :, 0]).astype(np.float64) * vs[:, :, 0].astype(np.float64)[..., None]
    assert np.allclose(causal[:, 0], np.repeat(v0, G, axis=1), rtol=1e-12, atol=1e-12)


def test_prefill_brute_force_tiny():
    # B=1, T=3, Hq=2, Hkv=1, d=4, causal: explicit loops and math.exp
    d, T = 4, 3
    rng = np.random.default_rng(22)
    k = rng.standard_normal((1, T, 1, d)).astype(np.float16)
    v = rng.standard_normal((1, T, 1, d)).astype(np.float16)
    q = rng.standard_normal((1, T, 2, d)).astype(np.float16)
    kc, ks, vc, vs = _fill_cache(k, v, T)
    out = O.prefill_attn(q, kc, ks, vc, vs, T)
    H4 = [[_sylvester_entry(i, j) for j in range(d)] for i in range(d)]
    kcodes, vcodes = O.unpack_int4(kc[0, 0]), O.unpack_int4(vc[0, 0])
    for h in range(2):
        for i in range(T):
            qr = [sum(float(q[0, i, h, a]) * H4[a][j] for a in range(d)) / 2.0 for j in range(d)]
            s = [sum(qr[j] * float(ks[0, 0, t]) * int(kcodes[t, j]) for j in range(d)) / 2.0 for t in range(i + 1)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            p = [x / sum(e) for x in e]
            o = [sum(p[t] * float(vs[0, 0, t]) * int(vcodes[t, j]) for t in range(i + 1)) for j in range(d)]
            assert np.allclose(out[0, i, h], o, rtol=1e-12, atol=1e-12)


def test_prefill_noncausal_is_invariant_to_key_order():
    # without the mask attention is a sum over keys: permuting the cached
    # tokens (codes and scales together) leaves every output row unchanged
    B, T, Hkv, G, d = 1, 11, 2, 2, 128
    qq, kc, ks, vc, vs = _prefill_case(B, T, Hkv, G, d, 23)
    perm = np.random.default_rng(24).permutation(T)
    base = O.prefill_attn(qq, kc, ks, vc, vs, T, causal=False)
    shuf = O.prefill_attn(qq, kc[:, :, perm], ks[:, :, perm], vc[:, :, perm], vs[:, :, perm], T, causal=False)
    assert np.allclose(shuf, base, rtol=1e-12, atol=1e-12)
    # the causal form is not: row 0 then sees the token that moved to slot 0
    caus = O.prefill_attn(qq, kc[:, :, perm], ks[:, :, perm], vc[:, :, perm], vs[:, :, perm], T)
    v_moved = O.unpack_int4(vc[:, :, perm[0]]).astype(np.float64) * vs[:, :, perm[0]].astype(np.float64)[..., None]
    assert np.allclose(caus[:, 0], np.repeat(v_moved, G, axis=1), rtol=1e-12, atol=1e-12)


def test_prefill_causal_rows_ignore_later_tokens():
    # causal row i reads tokens 0..i only: rewriting every token after t
    # leaves rows 0..t exactly as they were, and changes a later row
    B, T, Hkv, G, d, t = 1, 10, 1, 4, 128, 5
    qq, kc, ks, vc, vs = _prefill_case(B, T, Hkv, G, d, 25)
    base = O.prefill_attn(qq, kc, ks, vc, vs, T)
    rng = np.random.default_rng(26)
    kc2, vc2, ks2, vs2 = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    kc2[:, :, t + 1:] = rng.integers(0, 256, kc2[:, :, t + 1:].shape, dtype=np.uint8)
    vc2[:, :, t + 1:] = rng.integers(0, 256, vc2[:, :, t + 1:].shape, dtype=np.uint8)
    ks2[:, :, t + 1:] = ks2[:, :, t + 1:] * np.float16(3.0)
    vs2[:, :, t + 1:] = vs2[:, :, t + 1:] * np.float16(0.5)
    out = O.prefill_attn(qq, kc2, ks2, vc2, vs2, T)
    assert np.array_equal(out[:, :t + 1], base[:, :t + 1])
    assert not np.allclose(out[:, T - 1], base[:, T - 1])


# ---------------------------------------------------------------- asymmetric KV quantizer (next row f1)
@pytest.mark.parametrize("ex", ["A", "B"])
def test_kv_asym_quantizer_worked_examples(golden, ex):
    g = golden("kv_asym_quant_worked.txt")
    x = np.array([[float(v) for v in g[f"{ex}_x"]]], dtype=np.float32)
    q, s, z = O.quantize_asym_rows(x, float(g[f"{ex}_clip"][0]))
    assert float(s[0]) == float(g[f"{ex}_scale"][0])
    assert int(z[0]) == int(g[f"{ex}_zero"][0])
    assert np.array_equal(q[0], np.array([int(v) for v in g[f"{ex}_codes"]]))


def test_kv_asym_quantizer_invariants():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((200, 128)) * rng.uniform(0.01, 50.0, (200, 1))
         + rng.uniform(-20.0, 20.0, (200, 1))).astype(np.float32)
    q, s, z = O.quantize_asym_rows(x, 1.0)
    assert q.min() >= 0 and q.max() <= 15
    # the grid s (z + 0 .. 15) starts within s/2 of the row min and ends within
    # s/2 of the row max (plus the fp16 rounding of s): error at most one step
    err = np.abs(O.dequant_asym(q, s, z) - x.astype(np.float64))
    assert np.all(err <= 1.01 * s.astype(np.float64)[:, None])
    # codes are monotone in the input, and the row min / max sit at the grid ends
    order = np.argsort(x, axis=1)
    assert np.all(np.diff(np.take_along_axis(q.astype(int), order, axis=1), axis=1) >= 0)
    assert np.all(q.min(axis=1) == 0) and np.all(q.max(axis=1) >= 14)


def test_kv_asym_zero_row_and_unsigned_nibbles():
    q, s, z = O.quantize_asym_rows(np.zeros((1, 128), np.float32))
    assert np.all(q == 0) and int(z[0]) == 0
    assert float(s[0]) == float(np.float16(1e-5 / 15))
    allc = np.array(np.meshgrid(np.arange(16), np.arange(16))).reshape(2, -1).T
    assert np.array_equal(O.unpack_uint4(O.pack_int4(allc)), allc.astype(np.uint8))
    assert O.pack_int4(np.array([[15, 0]]))[0, 0] == 0x0F and O.pack_int4(np.array([[0, 15]]))[0, 0] == 0xF0


def _asym_cache(B, Hkv, T, d, seed):
    rng = np.random.default_rng(seed)
    c = [rng.integers(0, 256, (B, Hkv, T, d // 2), dtype=np.uint8) for _ in range(2)]
    s = [rng.uniform(0.05, 0.4, (B, Hkv, T)).astype(np.float16) for _ in range(2)]
    z = [rng.integers(-12, 4, (B, Hkv, T)).astype(np.int16) for _ in range(2)]
    return c[0], s[0], z[0], c[1], s[1], z[1]


def test_decode_asym_single_token_and_identical_keys():
    B, Hkv, Hq, d = 2, 2, 4, 128
    kc, ks, kz, vc, vs, vz = _asym_cache(B, Hkv, 5, d, 8)
    q = np.random.default_rng(9).standard_normal((B, Hq, d)).astype(np.float16)
    out = O.decode_attn_asym(q, kc, ks, kz, vc, vs, vz, T=1)
    v0 = O.dequant_asym(O.unpack_uint4(vc[:, :, 0]), vs[:, :, 0], vz[:, :, 0])  # [B, Hkv, d]
    assert np.allclose(out, np.repeat(v0, Hq // Hkv, axis=1), rtol=1e-12, atol=1e-12)
    kc[:, :, 1:5], ks[:, :, 1:5], kz[:, :, 1:5] = kc[:, :, :1], ks[:, :, :1], kz[:, :, :1]
    out = O.decode_attn_asym(q, kc, ks, kz, vc, vs, vz, T=5)
    vm = O.dequant_asym(O.unpack_uint4(vc[:, :, :5]), vs[:, :, :5], vz[:, :, :5]).mean(axis=2)
    assert np.allclose(out, np.repeat(vm, Hq // Hkv, axis=1), rtol=1e-10, atol=1e-12)


def test_decode_asym_brute_force_tiny():
    # B=1, Hq=2, Hkv=1, d=4, T=3, written with explicit loops and math.exp
    d, T = 4, 3
    kc, ks, kz, vc, vs, vz = _asym_cache(1, 1, T, d, 10)
    q = np.random.default_rng(11).standard_normal((1, 2, d)).astype(np.float16)
    out = O.decode_attn_asym(q, kc, ks, kz, vc, vs, vz, T=T)
    H4 = [[_sylvester_entry(i, j) for j in range(d)] for i in range(d)]
    kcode = [[(int(kc[0, 0, t, j // 2]) >> (4 * (j % 2))) & 15 for j in range(d)] for t in range(T)]
    vcode = [[(int(vc[0, 0, t, j // 2]) >> (4 * (j % 2))) & 15 for j in range(d)] for t in range(T)]
    for h in range(2):
        qr = [sum(float(q[0, h, i]) * H4[i][j] for i in range(d)) / 2.0 for j in range(d)]
        s = [sum(qr[j] * float(ks[0, 0, t]) * (kcode[t][j] + int(kz[0, 0, t])) for j in range(d)) / 2.0
             for t in range(T)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        p = [x / sum(e) for x in e]
        o = [sum(p[t] * float(vs[0, 0, t]) * (vcode[t][j] + int(vz[0, 0, t])) for t in range(T)) for j in range(d)]
        assert np.allclose(out[0, h], o, rtol=1e-12, atol=1e-12)


def test_decode_unrotated_close_to_float_attention():
    # informational sanity bound: INT4 KV attention stays near fp64 attention
    k, v, q = W.kv_inputs(B=1, T=64)
    kc, ks, vc, vs = _fill_cache(k, v, 64)
    out = O.decode_attn(q, kc, ks, vc, vs, T=64, unrotate=True)
    Hq, Hkv, d = q.shape[1], k.shape[2], q.shape[2]
    ref = np.zeros_like(out)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = (k[0, :, g].astype(np.float64) @ q[0, h].astype(np.float64)) / math.sqrt(d)
        p = np.exp(s - s.max())
        p /= p.sum()
        ref[0, h] = p @ v[0, :, g].astype(np.float64)
    assert O.rel_fro(out, ref) < 0.25


@pytest.mark.parametrize("d", [1, 2, 16, 256, 4096, 24, 96, 3072, 12288])
def test_fwht_mode_equals_dense_rotation(d):
    """The oracle's fast mode computes the dense definition: equal in float64
    to the dense product up to rounding (the two orders of the same sums), and
    bit-identical in fp32 except where the double rounding straddles a tie."""
    rng = np.random.default_rng(d)
    x = rng.standard_normal((5, d)).astype(np.float16)
    x[0, :] = 0
    x[0, d // 3] = 1.0  # one-hot: +-1/sqrt(d) everywhere
    s = W.random_signs(d, d + 1)
    dense = O.rotate_f64(x, s)
    fast = O.rotate_fwht(x, s).astype(np.float64)
    scale = np.abs(dense).max(axis=1, keepdims=True)
    assert np.all(np.abs(fast - dense) <= 2 ** -22 * scale)
    assert np.allclose(np.abs(fast[0]), 1 / np.sqrt(d), rtol=0, atol=1e-7)
    assert np.mean(fast.astype(np.float32) == O.rotate(x, s)) > 0.99


def test_fwht_rows_is_the_sylvester_product():
    """fwht_rows(x) = x @ H (unnormalized) for the Sylvester matrix, brute force."""
    rng = np.random.default_rng(3)
    for d in (1, 2, 4, 8, 64):
        x = rng.standard_normal((3, d))
        assert np.allclose(O.fwht_rows(x), x @ O.sylvester(d).astype(np.float64), atol=1e-12)
    with pytest.raises(ValueError):
        O.fwht_rows(np.ones((1, 12)))
