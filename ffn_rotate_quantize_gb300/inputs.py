"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module holds no arithmetic of the method: it only draws random numbers
(numpy PCG64, ``default_rng(seed)``) in a fixed order and rounds them to
bf16 bit patterns.  Draw order: outlier channel indices -> x -> W (-> W_up,
W_down) -> bias -> dy.  Values are drawn in fp32 and rounded to bfloat16 with
round-to-nearest-even.  bf16 arrays are ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import numpy as np

# Workloads: the shapes and distributions of the rotated-INT8 linear, decode,
# prefill, SwiGLU FFN and backward-dx cases.  rot = (a, b, groups).
CONFIGS = {
    "tiny_linear": dict(M=16, K=256, N=256, n_outliers=4, outlier_scale=20.0,
                        w_std=0.02, bias_std=0.01, rot=(16, 16, 1)),
    "decode_gemv": dict(M=1, K=4096, N=4096, n_outliers=41, outlier_scale=30.0,
                        w_std=0.02, bias_std=None, rot=(64, 64, 1)),
    "prefill_linear": dict(M=1024, K=4096, N=14336, n_outliers=41, outlier_scale=30.0,
                           w_std=0.02, bias_std=0.01, rot=(64, 64, 1)),
    "swiglu_ffn": dict(M=1024, d=4096, H=16384, w_std=0.02,
                       rot_d=(64, 64, 1), rot_h=(128, 128, 1)),
    "backward_dx": dict(M=4096, N=16384, K=4096, dy_std=1e-3, w_std=0.02, rot=(64, 64, 1)),
}


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); return uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_to_float(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, std):
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)


def outlier_count(K: int, frac: float = 0.01) -> int:
    """Number of outlier channels for a fraction of K (1% of 4096 -> 41)."""
    return int(round(frac * K))


def linear_case(M, K, N, n_outliers=0, outlier_scale=1.0, w_std=0.02, bias_std=None, seed=0):
    """x bf16 [M,K] ~ N(0,1) with outlier channels scaled; W bf16 [N,K] ~ N(0,w_std); bias bf16 [N] or None."""
    rng = np.random.default_rng(seed)
    idx = rng.choice(K, size=n_outliers, replace=False) if n_outliers else np.zeros(0, np.int64)
    x = _normal(rng, (M, K), 1.0)
    if n_outliers:
        x[:, idx] *= np.float32(outlier_scale)
    w = _normal(rng, (N, K), w_std)
    bias = bf16_bits(_normal(rng, (N,), bias_std)) if bias_std else None
    return dict(x=bf16_bits(x), w=bf16_bits(w), bias=bias, outliers=np.sort(idx))


def ffn_case(M, d, H, w_std=0.02, seed=0, n_outliers=0, outlier_scale=1.0):
    """x bf16 [M,d] ~ N(0,1); W_gate, W_up bf16 [H,d]; W_down bf16 [d,H], all ~ N(0,w_std)."""
    rng = np.random.default_rng(seed)
    idx = rng.choice(d, size=n_outliers, replace=False) if n_outliers else np.zeros(0, np.int64)
    x = _normal(rng, (M, d), 1.0)
    if n_outliers:
        x[:, idx] *= np.float32(outlier_scale)
    wg = _normal(rng, (H, d), w_std)
    wu = _normal(rng, (H, d), w_std)
    wd = _normal(rng, (d, H), w_std)
    return dict(x=bf16_bits(x), wg=bf16_bits(wg), wu=bf16_bits(wu), wd=bf16_bits(wd))


def backward_case(M, N, K, dy_std=1e-3, w_std=0.02, seed=0):
    """W bf16 [N,K] ~ N(0,w_std) (to be int8-prepared) and dy bf16 [M,N] ~ N(0,dy_std)."""
    rng = np.random.default_rng(seed)
    w = _normal(rng, (N, K), w_std)
    dy = _normal(rng, (M, N), dy_std)
    return dict(w=bf16_bits(w), dy=bf16_bits(dy))


def config_case(name: str, seed: int = 0, **override):
    """Inputs of a named workload (sizes may be overridden for scaled-down parity cases)."""
    c = dict(CONFIGS[name])
    c.update(override)
    if name in ("tiny_linear", "decode_gemv", "prefill_linear"):
        case = linear_case(c["M"], c["K"], c["N"], c["n_outliers"], c["outlier_scale"],
                           c["w_std"], c["bias_std"], seed)
    elif name == "swiglu_ffn":
        case = ffn_case(c["M"], c["d"], c["H"], c["w_std"], seed)
    elif name == "backward_dx":
        case = backward_case(c["M"], c["N"], c["K"], c["dy_std"], c["w_std"], seed)
    else:
        raise KeyError(name)
    case["config"] = c
    return case
