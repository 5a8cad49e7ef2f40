"""CPU oracle for the rotated-INT8 linear / FFN path (numpy wrappers over oracle.c).

TEST INFRASTRUCTURE ONLY.  The product library never imports, links or runs
anything in this folder.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA path.

Every function follows the PyPI page "xpu-kernels 0.2.0"
(pypi.org/project/xpu-kernels/0.2.0); the section is named on each function.
Arrays holding bf16 values are ``numpy.uint16`` bit patterns.  Rotation
descriptors are ``(a, b, groups)`` with ``K = a * b * groups``.

Pins (tests/test_oracle.py) tie each function to something other than itself:
the printed H4, the page's index map for a 256-group, an explicit Kronecker
matrix, one-hot inputs, round-half-even ties, numpy/torch library routines
and error budgets the page states.  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_c_void_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build_oracle(force: bool = False) -> str:
    """Compile oracle.c into oracle/liboracle.so with gcc (OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.orc_hadamard.restype = _int
        lib.orc_rotate_rows.restype = _int
        lib.orc_gemm_s8.restype = _i64
        lib.orc_num_threads.restype = _int
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_c_void_p)


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().orc_num_threads())


# ---------------------------------------------------------------- bf16 helpers
def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().orc_bf16_to_f32(_p(h), _p(out), _i64(h.size))
    return out


def f32_to_bf16(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().orc_f32_to_bf16(_p(f), _p(out), _i64(f.size))
    return out


# ---------------------------------------------------------------- rotation
def hadamard(n: int) -> np.ndarray:
    """Integer factor H_n ("Algorithm: fused ConvRot rotation"; H2 on the top bit when 4 does not divide log-size)."""
    H = np.empty((n, n), np.int32)
    if _load().orc_hadamard(_int(n), _p(H)) != 0:
        raise ValueError(f"n={n} is not a power of two")
    return H


def rotate(x: np.ndarray, rot) -> np.ndarray:
    """v = (I_g (x) H_a (x) H_b) x / sqrt(ab) per row; fp64 sums, fp32 result."""
    a, b, g = rot
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    v = np.empty_like(x)
    if _load().orc_rotate_rows(_p(x), _p(v), _i64(M), _i64(K), _int(a), _int(b), _int(g)) != 0:
        raise ValueError(f"bad rotation descriptor {rot} for K={K}")
    return v


def rotation_matrix(rot) -> np.ndarray:
    """Explicit fp64 matrix I_g (x) H_a (x) H_b / sqrt(ab) (small K only)."""
    a, b, g = rot
    R = np.kron(hadamard(a).astype(np.float64), hadamard(b).astype(np.float64)) / np.sqrt(a * b)
    return np.kron(np.eye(g), R)


# ---------------------------------------------------------------- quantizer
def quantize(v: np.ndarray):
    """Per-row int8 quantizer ("API": int8 [M,K] + fp32 [M] row scales). Returns (q, s)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    M, K = v.shape
    q = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    _load().orc_quantize_rows(_p(v), _p(q), _p(s), _i64(M), _i64(K))
    return q, s


def rotate_quantize(x_bf16: np.ndarray, rot):
    """Fused ConvRot rotation + per-token INT8 quantization of bf16 rows ("Use from C")."""
    return quantize(rotate(bf16_to_f32(x_bf16), rot))


def prepare_weight(w_bf16: np.ndarray, rot):
    """W bf16 [N,K] -> (W8 int8 [N,K], s fp32 [N]); the rotation baked into the rows ("Use from Python")."""
    return rotate_quantize(w_bf16, rot)


# ---------------------------------------------------------------- GEMM + epilogue
def gemm_s8(q: np.ndarray, w8: np.ndarray) -> np.ndarray:
    """acc[m,n] = sum_k q[m,k] w8[n,k] in int64 (the page's int8 GEMM)."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    w8 = np.ascontiguousarray(w8, dtype=np.int8)
    M, K = q.shape
    N, K2 = w8.shape
    assert K == K2
    acc = np.empty((M, N), np.int64)
    bad = _load().orc_gemm_s8(_p(q), _p(w8), _p(acc), _i64(M), _i64(N), _i64(K))
    if bad:
        raise OverflowError(f"{bad} accumulators do not fit in int32")
    return acc


def dequant(acc: np.ndarray, xs: np.ndarray, ws: np.ndarray, bias_bf16=None) -> np.ndarray:
    """y = bf16(fmaf(fp32(acc) * xs[m], ws[n], bias[n])) ("API", dequant epilogue)."""
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    M, N = acc.shape
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    ws = np.ascontiguousarray(ws, dtype=np.float32)
    y = np.empty((M, N), np.uint16)
    if bias_bf16 is None:
        bptr = None
    else:
        bias = bf16_to_f32(bias_bf16)
        bptr = _p(bias)
    _load().orc_dequant(_p(acc), _i64(N), _p(xs), _p(ws), bptr, _p(y), _i64(N), _i64(M), _i64(N))
    return y


def linear_acc(x_bf16, w8, rot):
    """(acc int64 [M,N], x_scale fp32 [M]) -- "linear_acc" of "Use from Python"."""
    q, xs = rotate_quantize(x_bf16, rot)
    return gemm_s8(q, w8), xs


def linear(x_bf16, w8, ws, bias_bf16, rot):
    """bf16 [M,N] = dequant(linear_acc(x)) -- "linear" of "Use from Python"."""
    acc, xs = linear_acc(x_bf16, w8, rot)
    return dequant(acc, xs, ws, bias_bf16)


# ---------------------------------------------------------------- FFN
def silu_glu(g_bf16: np.ndarray, u_bf16: np.ndarray) -> np.ndarray:
    """h = silu(g) * u in fp32 from bf16 g, u."""
    g = np.ascontiguousarray(g_bf16, dtype=np.uint16)
    u = np.ascontiguousarray(u_bf16, dtype=np.uint16)
    h = np.empty(g.shape, np.float32)
    _load().orc_silu_glu(_p(g), _p(u), _p(h), _i64(g.size))
    return h


def ffn(x_bf16, wg8, sg, wu8, su, wd8, sd, rot_d, rot_h, keep=False):
    """SwiGLU FFN as the unfused chain: linear_acc -> dequant -> silu*up -> rotate+quantize -> down.

    The page's MLP pattern (gate GEMM, up GEMM, GLU/SwiGLU, down GEMM) with
    "dequant_act_quantize" as its middle ("Use from Python").  No biases.
    """
    qx, xs = rotate_quantize(x_bf16, rot_d)
    g = dequant(gemm_s8(qx, wg8), xs, sg)
    u = dequant(gemm_s8(qx, wu8), xs, su)
    h = silu_glu(g, u)
    qh, hs = quantize(rotate(h, rot_h))
    y = dequant(gemm_s8(qh, wd8), hs, sd)
    if keep:
        return y, dict(qx=qx, xs=xs, g=g, u=u, h=h, qh=qh, hs=hs)
    return y


# ---------------------------------------------------------------- backward
def dequant_weight(w8, s, rot) -> np.ndarray:
    """W_hat bf16 [N,K] = bf16((W8[n,:] * s[n]) R): recover W ("The backward"); reading R-7: un-rotate."""
    w8 = np.ascontiguousarray(w8, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    N, K = w8.shape
    w = np.empty((N, K), np.float32)
    _load().orc_scale_rows_s8(_p(w8), _p(s), _p(w), _i64(N), _i64(K))
    return f32_to_bf16(rotate(w, rot))


def linear_dx(dy_bf16, w_bf16) -> np.ndarray:
    """dx = dy @ W with bf16 inputs, fp64 sums, bf16 result ("The backward")."""
    dy = np.ascontiguousarray(dy_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    M, N = dy.shape
    N2, K = w.shape
    assert N == N2
    dx = np.empty((M, K), np.uint16)
    _load().orc_matmul_bf16_nn(_p(dy), _p(w), _p(dx), _i64(M), _i64(N), _i64(K))
    return dx


def linear_dx_int8(dy_bf16, w8, s, rot, keep=False):
    """dx via the int8 route ("The backward", linear_dx_int8).

    dy'[m,n] = dy[m,n] * s[n] (fp32); per-row quantize with no rotation
    (reading R-10); acc[m,k] = sum_n qd[m,n] W8[n,k] (int64);
    dx_rot = fp32(acc) * t[m]; dx = bf16(dx_rot R).
    """
    dy = np.ascontiguousarray(dy_bf16, dtype=np.uint16)
    w8 = np.ascontiguousarray(w8, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    M, N = dy.shape
    N2, K = w8.shape
    assert N == N2
    dyp = np.empty((M, N), np.float32)
    _load().orc_scale_cols_bf16(_p(dy), _p(s), _p(dyp), _i64(M), _i64(N))
    qd, t = quantize(dyp)
    acc = gemm_s8(qd, np.ascontiguousarray(w8.T))
    dxr = np.empty((M, K), np.float32)
    _load().orc_dequant_f32(_p(acc), _p(t), _p(dxr), _i64(M), _i64(K))
    dx = f32_to_bf16(rotate(dxr, rot))
    if keep:
        return dx, dict(dyp=dyp, qd=qd, t=t, acc=acc, dxr=dxr)
    return dx


def rotate_bf16(x_bf16, rot) -> np.ndarray:
    """Rotate-only bf16 path ("Use from C": the BF16 path needs only the rotation)."""
    return f32_to_bf16(rotate(bf16_to_f32(x_bf16), rot))


def linear_bf16(x_bf16, w_bf16, bias_bf16=None) -> np.ndarray:
    """y = bf16(x @ W^T + bias) with bf16 inputs, fp64 sums, one rounding to fp32 then bf16.

    The linear layer of the rotate-only BF16 path ("Use from C"): with x and W both rotated by the
    same R (R R^T = I) it computes the unrotated layer up to bf16 rounding."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    M, K = x.shape
    N, K2 = w.shape
    assert K == K2
    b = None if bias_bf16 is None else np.ascontiguousarray(bias_bf16, dtype=np.uint16)
    assert b is None or b.shape == (N,)
    y = np.empty((M, N), np.uint16)
    _load().orc_linear_bf16(_p(x), _p(w), None if b is None else _p(b), _p(y), _i64(M), _i64(N), _i64(K))
    return y
