"""quarot_decode_attn_static: the decode entry point for callers that cannot
allocate device memory when they run decode (plain C hosts without an
allocator, serving loops that forbid cudaMalloc after start-up, plug-ins that
only receive their input and output buffers).  Its scratch is a fixed array
inside the library, so it takes no workspace argument.

The GPU test calls it through the C ABI twice in a row, with different sizes
and inputs, and checks each result against quarot_decode_attn given its own
caller-allocated workspace.  Both run the same kernels with the same split
count (the split count does not depend on the workspace size), so the
outputs must be bit-identical.  This file is collected last so that a
failure here cannot hide another test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

OUT_TOL = 1e-3


def _rel_fro(a, b):
    a = a.double()
    b = b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


def _cache(B, Hkv, T, d, seed, dev):
    rng = np.random.Generator(np.random.PCG64(seed))
    kq = torch.from_numpy(rng.integers(0, 256, size=(B, Hkv, T, d // 2), dtype=np.uint8)).to(dev)
    vq = torch.from_numpy(rng.integers(0, 256, size=(B, Hkv, T, d // 2), dtype=np.uint8)).to(dev)
    ks = torch.from_numpy(W.fp16_scales(B * Hkv * T, seed + 1, 0.05, 0.5).reshape(B, Hkv, T)).to(dev)
    vs = torch.from_numpy(W.fp16_scales(B * Hkv * T, seed + 2, 0.05, 0.5).reshape(B, Hkv, T)).to(dev)
    return kq, ks, vq, vs


def test_static_rejects_oversize_without_touching_the_device():
    import __graft_entry__

    __graft_entry__.build()
    import w4a4_rotated_quantized_gb300 as q

    lib = q.load()
    P = ctypes.c_void_p(0x10000)  # never dereferenced: the request is rejected first
    # 64 x 32 heads x 32 splits x 130 floats = 34 MB > the 8 MB array
    assert lib.quarot_decode_attn_static(P, P, P, P, P, 64, 32, 8, 128, 8192, 8192, 0.0, 0, P, None) == 2
    assert q.quarot_decode_workspace_bytes(64, 32, 128, 8192) > q.DECODE_STATIC_SCRATCH_BYTES


@pytest.mark.parametrize("B,Hq,Hkv,d,T,T_max", [
    (2, 32, 8, 64, 100, 128),    # head_dim other than 128: unsupported
    (2, 32, 8, 128, 200, 128),   # T beyond the cache: invalid
    (2, 32, 2, 128, 100, 128),   # 16 query heads per KV head: unsupported
    (2, 30, 8, 128, 100, 128),   # Hq not a multiple of Hkv: invalid
    (-1, 32, 8, 128, 100, 128),  # negative batch: invalid
])
def test_static_rejects_like_the_workspace_entry(B, Hq, Hkv, d, T, T_max):
    """Requests that quarot_decode_attn rejects get the same status from the
    static entry point, before it looks up its scratch (no GPU needed)."""
    import __graft_entry__

    __graft_entry__.build()
    import w4a4_rotated_quantized_gb300 as q

    lib = q.load()
    P = ctypes.c_void_p(0x10000)  # never dereferenced
    ws = ctypes.c_void_p(0x100000)
    want = lib.quarot_decode_attn(P, P, P, P, P, B, Hq, Hkv, d, T, T_max, 0.0, 0, P, ws, 1 << 30, None)
    got = lib.quarot_decode_attn_static(P, P, P, P, P, B, Hq, Hkv, d, T, T_max, 0.0, 0, P, None)
    assert want != 0 and got == want, (want, got)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import w4a4_rotated_quantized_gb300 as q

    lib = q.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    cases = [  # (B, Hkv, G, T, T_max, unrotate): the bench shape, then a smaller one
        (16, 8, 4, 4096, 4096, 0),
        (3, 2, 8, 700, 1024, 1),
    ]
    assert q.quarot_decode_workspace_bytes(16, 32, 128, 4096) <= q.DECODE_STATIC_SCRATCH_BYTES
    for i, (B, Hkv, G, T, T_max, unrot) in enumerate(cases):
        d = 128
        kq, ks, vq, vs = _cache(B, Hkv, T_max, d, 100 + i, dev)
        qq = torch.from_numpy(W.query(B, Hkv * G, d, 200 + i)).to(dev)
        ref = q.quarot_decode_attn(qq, kq, ks, vq, vs, T=T, unrotate_out=bool(unrot))
        out = torch.full((B, Hkv * G, d), float("nan"), dtype=torch.float16, device=dev)
        st = lib.quarot_decode_attn_static(
            ctypes.c_void_p(qq.data_ptr()), ctypes.c_void_p(kq.data_ptr()), ctypes.c_void_p(ks.data_ptr()),
            ctypes.c_void_p(vq.data_ptr()), ctypes.c_void_p(vs.data_ptr()), B, Hkv * G, Hkv, d, T, T_max, 0.0,
            unrot, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, q.STATUS.get(st)
        q.quarot_check_error(stream)
        assert torch.isfinite(out).all()
        assert _rel_fro(out, ref) <= OUT_TOL
        # same kernels, same split count: the same bits
        assert torch.equal(out, ref)
