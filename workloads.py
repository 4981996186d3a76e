"""Seeded synthetic inputs for the QuaRot hot path.

This module is the only code shared by the CPU oracle (``oracle/``) and the
CUDA path (``w4a4_rotated_quantized_gb300``).  It draws random numbers and
nothing else: no rotation, no quantization, no arithmetic of the method.

The shapes and value distributions follow the workloads of the QuaRot pages:
LLaMA/Qwen-like layer widths (hidden 4096, MLP 12288), N(0,1) activations with
a few coordinate-aligned outlier channels scaled up (the "Activation Outlier
Phenomenon" of "QuaRot Guide: Outlier-Free 4-Bit W4A4 LLM Quantization",
where roughly 0.1 % of channels carry values up to 100x the rest, always in
the same channel indices), N(0, 0.02^2) weights, and a LLaMA-2 GQA attention
shape for the KV cache (32 query heads, 8 KV heads, head_dim 128).  No dataset
and no trained weights are involved.

All generators use numpy's PCG64 so that the same seed gives the same bits on
x86 and Arm hosts.
"""
from __future__ import annotations

import numpy as np

# Seed layout: base + config index, then fixed offsets per tensor kind.
SEED_BASE = 1000
OFF_X, OFF_W, OFF_SIGNS, OFF_OUTLIER, OFF_K, OFF_V, OFF_Q = 0, 100, 200, 300, 400, 500, 600


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def random_signs(d: int, seed: int) -> np.ndarray:
    """The random +-1 diagonal s of the randomized Hadamard matrix, as int8 [d]."""
    bits = _rng(seed).integers(0, 2, size=d, dtype=np.int8)
    return (1 - 2 * bits).astype(np.int8)


def outlier_channels(d: int, n: int, seed: int) -> np.ndarray:
    """n distinct channel indices in [0, d), sorted."""
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(_rng(seed).choice(d, size=n, replace=False)).astype(np.int64)


def activations(M: int, d: int, channels, factor: float, seed: int) -> np.ndarray:
    """fp16 [M, d]: N(0,1) draws, the listed channels multiplied by ``factor``."""
    x = _rng(seed).standard_normal((M, d), dtype=np.float32)
    ch = np.asarray(channels, dtype=np.int64)
    if ch.size:
        x[:, ch] *= np.float32(factor)
    return x.astype(np.float16)


def weights(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    """fp16 [N, K] with N(0, std^2) entries ([out_features, in_features])."""
    w = _rng(seed).standard_normal((N, K), dtype=np.float32) * np.float32(std)
    return w.astype(np.float16)


def int4_codes(rows: int, cols: int, seed: int, low: int = -8, high: int = 7) -> np.ndarray:
    """Uniform integer codes in [low, high] as int8 [rows, cols] (GEMM operand tests)."""
    return _rng(seed).integers(low, high + 1, size=(rows, cols), dtype=np.int8)


def fp16_scales(n: int, seed: int, lo: float = 1e-3, hi: float = 2.0) -> np.ndarray:
    """Positive fp16 scales drawn log-uniformly in [lo, hi]."""
    u = _rng(seed).random(n)
    return np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo))).astype(np.float16)


def kv_tensors(B: int, T: int, Hkv: int, d: int, n_outlier: int, factor: float, seed: int) -> np.ndarray:
    """fp16 [B, T, Hkv, d]: N(0,1), with ``n_outlier`` seeded dims per head scaled by ``factor``."""
    rng = _rng(seed)
    x = rng.standard_normal((B, T, Hkv, d), dtype=np.float32)
    for h in range(Hkv):
        dims = np.sort(rng.choice(d, size=n_outlier, replace=False))
        x[:, :, h, dims] *= np.float32(factor)
    return x.astype(np.float16)


def query(B: int, Hq: int, d: int, seed: int) -> np.ndarray:
    """fp16 [B, Hq, d] with N(0,1) entries."""
    return _rng(seed).standard_normal((B, Hq, d), dtype=np.float32).astype(np.float16)


def prefill_query(B: int, T: int, Hq: int, d: int, seed: int) -> np.ndarray:
    """fp16 [B, T, Hq, d] prompt queries with N(0,1) entries."""
    return _rng(seed).standard_normal((B, T, Hq, d), dtype=np.float32).astype(np.float16)


# ---------------------------------------------------------------------------
# The five workloads.  Index i uses seeds SEED_BASE + i + offset.
# ---------------------------------------------------------------------------
CONFIGS = {
    "tiny": dict(index=0, kind="layer", M=16, K=256, N=256, outliers=[3, 77], factor=50.0),
    "rotq4096": dict(index=1, kind="rotq", M=2048, K=4096, n_outlier=8, factor=100.0),
    "down_proj": dict(index=2, kind="layer", M=2048, K=12288, N=4096, n_outlier=12, factor=100.0),
    "sweep": dict(index=3, kind="sweep", Ms=(512, 2048, 8192), K=4096, Ns=(4096, 12288),
                  n_outlier=8, factor=100.0),
    "kv4": dict(index=4, kind="kv", B=16, T=4096, Hkv=8, Hq=32, d=128, n_outlier=2, factor=20.0),
    # Init (prefill) attention over the same cache shape: 4 prompts of 2048
    # tokens (the pages' prefill length), 32 query / 8 KV heads, head_dim 128
    "prefill": dict(index=5, kind="prefill", B=4, T=2048, Hkv=8, Hq=32, d=128, n_outlier=2, factor=20.0),
}


def seed_of(config: str, offset: int) -> int:
    return SEED_BASE + CONFIGS[config]["index"] + offset


def layer_inputs(config: str, M: int | None = None, N: int | None = None):
    """(x fp16 [M,K], w fp16 [N,K] or None, signs int8 [K]) for a layer/rotq/sweep config.

    ``M``/``N`` override the config's sizes (the sweep has several); rows are
    drawn for the full M so a prefix of rows is the same for any M.
    """
    c = CONFIGS[config]
    K = c["K"]
    M = M if M is not None else c.get("M")
    if "outliers" in c:
        ch = c["outliers"]
    else:
        ch = outlier_channels(K, c["n_outlier"], seed_of(config, OFF_OUTLIER))
    x = activations(M, K, ch, c["factor"], seed_of(config, OFF_X))
    N = N if N is not None else c.get("N")
    w = weights(N, K, seed_of(config, OFF_W)) if N is not None else None
    s = random_signs(K, seed_of(config, OFF_SIGNS))
    return x, w, s


def kv_inputs(config: str = "kv4", B: int | None = None, T: int | None = None):
    """(k, v fp16 [B,T,Hkv,d], q fp16 [B,Hq,d]) for the KV decode config."""
    c = CONFIGS[config]
    B = B if B is not None else c["B"]
    T = T if T is not None else c["T"]
    k = kv_tensors(B, T, c["Hkv"], c["d"], c["n_outlier"], c["factor"], seed_of(config, OFF_K))
    v = kv_tensors(B, T, c["Hkv"], c["d"], c["n_outlier"], c["factor"], seed_of(config, OFF_V))
    q = query(B, c["Hq"], c["d"], seed_of(config, OFF_Q))
    return k, v, q


def prefill_inputs(config: str = "prefill", B: int | None = None, T: int | None = None):
    """(k, v fp16 [B,T,Hkv,d], q fp16 [B,T,Hq,d]) for the prefill attention config."""
    c = CONFIGS[config]
    B = B if B is not None else c["B"]
    T = T if T is not None else c["T"]
    k = kv_tensors(B, T, c["Hkv"], c["d"], c["n_outlier"], c["factor"], seed_of(config, OFF_K))
    v = kv_tensors(B, T, c["Hkv"], c["d"], c["n_outlier"], c["factor"], seed_of(config, OFF_V))
    q = prefill_query(B, T, c["Hq"], c["d"], seed_of(config, OFF_Q))
    return k, v, q
