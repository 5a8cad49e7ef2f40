"""Torch-facing binding of libgbq: argument marshalling only.

Every function allocates its outputs with torch (the C ABI itself never
allocates), passes ``data_ptr()``s and the current CUDA stream to the matching
``gbq_*`` entry point, and raises ``GbqError`` on a non-zero status.  All
compute happens in the library's CUDA kernels.  The operations follow the PyPI
page "xpu-kernels 0.2.0" ("Use from Python", "The backward: dL/dx, weight-only").
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import GbqError, Rot, check, lib  # noqa: F401

OP_LINEAR, OP_INT8_GEMM, OP_FFN, OP_LINEAR_DX_INT8 = 1, 2, 3, 4


def rot(a: int, b: int, groups: int = 1) -> Rot:
    return Rot(a, b, groups)


def _rot(r) -> Rot:
    return r if isinstance(r, Rot) else Rot(*r)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _req(t, dtype, name):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor, got {t.dtype} on {t.device}")


def _vec(t, n, dtype, name, optional=False):
    """A per-row / per-column vector argument: a contiguous CUDA tensor of n elements of dtype."""
    if t is None and optional:
        return
    if t is None:
        raise ValueError(f"{name}: required")
    _req(t, dtype, name)
    if t.numel() != n:
        raise ValueError(f"{name}: expected {n} elements, got {t.numel()}")


def _mat(t, shape, dtype, name):
    _req(t, dtype, name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _out(out, shape, dtype, device, name="out"):
    """A new output tensor, or the caller's after checking that it has exactly the expected shape and type
    (the C ABI takes raw pointers and writes shape-many elements)."""
    if out is None:
        return torch.empty(shape, dtype=dtype, device=device)
    _req(out, dtype, name)
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(out.shape)}")
    return out


def init() -> str:
    check(lib().gbq_init())
    return lib().gbq_device_name().decode()


def device_status(stream=None) -> int:
    st = ctypes.c_uint32(0)
    check(lib().gbq_device_status(_stream(stream), ctypes.byref(st)))
    return st.value


K_ROTATE, K_I8GEMM, K_BF16GEMM, K_GEMV, K_ELEMWISE = 0, 1, 2, 3, 4


def prof_enable(on: bool = True) -> None:
    """Bracket every library kernel launch with CUDA events (library-owned) from now on."""
    check(lib().gbq_prof_enable(1 if on else 0))


def prof_read(kind: int):
    """(launches, total ms) of the timed launches of one kernel class."""
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    check(lib().gbq_prof_read(kind, ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


def workspace_size(op: int, M: int, N: int = 0, K: int = 0, H: int = 0) -> int:
    return int(lib().gbq_workspace_size(op, M, N, K, H))


def _workspace(op, M, N, K, H, device, workspace=None):
    """(workspace, its size in bytes): a new one of the size the library asks for, or the caller's, whose
    actual size is passed on (the library rejects one that is too small)."""
    if workspace is None:
        n = workspace_size(op, M, N, K, H)
        return torch.empty(max(n, 1), dtype=torch.uint8, device=device), n
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace: expected a contiguous CUDA tensor")
    return workspace, workspace.numel() * workspace.element_size()


# ------------------------------------------------------------------ rotate + quantize
def quantize_act(x: torch.Tensor, r, stream=None):
    """bf16 [M,K] -> (int8 [M,K], fp32 [M]) = quantize(R x) per row."""
    _req(x, torch.bfloat16, "x")
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    s = torch.empty((M,), dtype=torch.float32, device=x.device)
    check(lib().gbq_quantize_act(_ptr(x), _ptr(q), _ptr(s), M, K, _rot(r), _stream(stream)))
    return q, s


def prepare_weight(w: torch.Tensor, r, stream=None):
    """bf16 W [N,K] -> (W8 int8 [N,K], s fp32 [N]), the rotation baked into the rows."""
    _req(w, torch.bfloat16, "w")
    N, K = w.shape
    w8 = torch.empty((N, K), dtype=torch.int8, device=w.device)
    s = torch.empty((N,), dtype=torch.float32, device=w.device)
    check(lib().gbq_prepare_weight(_ptr(w), _ptr(w8), _ptr(s), N, K, _rot(r), _stream(stream)))
    return w8, s


def quantize_act_glu(g: torch.Tensor, u: torch.Tensor, r, stream=None):
    """(bf16 g, bf16 u) [M,H] -> quantize(R (silu(g) * u))."""
    _req(g, torch.bfloat16, "g")
    M, H = g.shape
    _mat(u, (M, H), torch.bfloat16, "u")
    q = torch.empty((M, H), dtype=torch.int8, device=g.device)
    s = torch.empty((M,), dtype=torch.float32, device=g.device)
    check(lib().gbq_quantize_act_glu(_ptr(g), _ptr(u), _ptr(q), _ptr(s), M, H, _rot(r), _stream(stream)))
    return q, s


def dequant_act_quantize(acc_g, acc_u, x_scale, s_gate, s_up, r, stream=None):
    """int32 gate/up accumulators -> quantize(R (silu(dequant(acc_g)) * dequant(acc_u)))."""
    _req(acc_g, torch.int32, "acc_g")
    M, H = acc_g.shape
    _mat(acc_u, (M, H), torch.int32, "acc_u")
    _vec(x_scale, M, torch.float32, "x_scale")
    _vec(s_gate, H, torch.float32, "s_gate")
    _vec(s_up, H, torch.float32, "s_up")
    q = torch.empty((M, H), dtype=torch.int8, device=acc_g.device)
    s = torch.empty((M,), dtype=torch.float32, device=acc_g.device)
    check(lib().gbq_dequant_act_quantize(_ptr(acc_g), _ptr(acc_u), H, _ptr(x_scale), _ptr(s_gate), _ptr(s_up),
                                         _ptr(q), _ptr(s), M, H, _rot(r), _stream(stream)))
    return q, s


def rotate_bf16(x: torch.Tensor, r, stream=None, out=None):
    """bf16 [M,K] -> bf16(R x)."""
    _req(x, torch.bfloat16, "x")
    M, K = x.shape
    y = _out(out, x.shape, torch.bfloat16, x.device)
    check(lib().gbq_rotate_bf16(_ptr(x), _ptr(y), M, K, _rot(r), _stream(stream)))
    return y


def linear_bf16(x: torch.Tensor, w: torch.Tensor, bias=None, out=None, stream=None):
    """bf16 x [M,K] @ bf16 w[N,K]^T + bias [N] -> bf16 y [M,N] (the rotate-only path's linear)."""
    _req(x, torch.bfloat16, "x")
    M, K = x.shape
    N = w.shape[0]
    _mat(w, (N, K), torch.bfloat16, "w")
    _vec(bias, N, torch.bfloat16, "bias", optional=True)
    y = _out(out, (M, N), torch.bfloat16, x.device)
    check(lib().gbq_linear_bf16(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), M, N, K,
                                _stream(stream)))
    return y


# ------------------------------------------------------------------ linear
def int8_gemm(q: torch.Tensor, w8: torch.Tensor, workspace=None, stream=None):
    """int8 [M,K] x int8 [N,K] -> int32 [M,N], exact."""
    _req(q, torch.int8, "q")
    M, K = q.shape
    N = w8.shape[0]
    _mat(w8, (N, K), torch.int8, "w8")
    acc = torch.empty((M, N), dtype=torch.int32, device=q.device)
    ws, n = _workspace(OP_INT8_GEMM, M, N, K, 0, q.device, workspace)
    check(lib().gbq_int8_gemm(_ptr(q), _ptr(w8), _ptr(acc), N, M, N, K, _ptr(ws), n, _stream(stream)))
    return acc


def linear_acc(x: torch.Tensor, w8: torch.Tensor, r, workspace=None, stream=None):
    """bf16 x [M,K] -> (int32 acc [M,N], fp32 x_scale [M])."""
    _req(x, torch.bfloat16, "x")
    M, K = x.shape
    N = w8.shape[0]
    _mat(w8, (N, K), torch.int8, "w8")
    acc = torch.empty((M, N), dtype=torch.int32, device=x.device)
    xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    ws, n = _workspace(OP_LINEAR, M, N, K, 0, x.device, workspace)
    check(lib().gbq_linear_acc(_ptr(x), _ptr(w8), _ptr(acc), N, _ptr(xs), M, N, K, _rot(r), _ptr(ws), n,
                               _stream(stream)))
    return acc, xs


def dequant(acc: torch.Tensor, x_scale, w_scale, bias=None, out=None, stream=None):
    """int32 acc [M,N] (a strided column slice is allowed) -> bf16 [M,N]."""
    if acc.dtype != torch.int32 or acc.stride(1) != 1:
        raise ValueError("acc must be int32 with unit column stride")
    M, N = acc.shape
    _vec(x_scale, M, torch.float32, "x_scale")
    _vec(w_scale, N, torch.float32, "w_scale")
    _vec(bias, N, torch.bfloat16, "bias", optional=True)
    y = _out(out, (M, N), torch.bfloat16, acc.device)
    check(lib().gbq_dequant(_ptr(acc), acc.stride(0), _ptr(x_scale), _ptr(w_scale), _ptr(bias), _ptr(y),
                            y.stride(0), M, N, _stream(stream)))
    return y


def linear(x: torch.Tensor, w8: torch.Tensor, w_scale, bias, r, workspace=None, out=None, stream=None):
    """bf16 x [M,K] -> bf16 y [M,N] = dequant(linear_acc(x))."""
    _req(x, torch.bfloat16, "x")
    M, K = x.shape
    N = w8.shape[0]
    _mat(w8, (N, K), torch.int8, "w8")
    _vec(w_scale, N, torch.float32, "w_scale")
    _vec(bias, N, torch.bfloat16, "bias", optional=True)
    y = _out(out, (M, N), torch.bfloat16, x.device)
    ws, n = _workspace(OP_LINEAR, M, N, K, 0, x.device, workspace)
    check(lib().gbq_linear(_ptr(x), _ptr(w8), _ptr(w_scale), _ptr(bias), _ptr(y), M, N, K, _rot(r), _ptr(ws), n,
                           _stream(stream)))
    return y


def linear_noalloc(x: torch.Tensor, w8: torch.Tensor, w_scale, bias, r, out=None, stream=None):
    """linear() without a workspace: the library's static device scratch is used (see include/gbq.h)."""
    _req(x, torch.bfloat16, "x")
    M, K = x.shape
    N = w8.shape[0]
    _mat(w8, (N, K), torch.int8, "w8")
    _vec(w_scale, N, torch.float32, "w_scale")
    _vec(bias, N, torch.bfloat16, "bias", optional=True)
    y = _out(out, (M, N), torch.bfloat16, x.device)
    check(lib().gbq_linear_noalloc(_ptr(x), _ptr(w8), _ptr(w_scale), _ptr(bias), _ptr(y), M, N, K, _rot(r),
                                   _stream(stream)))
    return y


# ------------------------------------------------------------------ FFN
def ffn_fused(x, wg8, s_gate, wu8, s_up, wd8, s_down, rot_d, rot_h, workspace=None, out=None, stream=None):
    """bf16 x [M,d] -> bf16 y [M,d] = down(quantize(R_h(silu(gate(x)) * up(x))))."""
    _req(x, torch.bfloat16, "x")
    M, d = x.shape
    H = wg8.shape[0]
    _mat(wg8, (H, d), torch.int8, "wg8")
    _mat(wu8, (H, d), torch.int8, "wu8")
    _mat(wd8, (d, H), torch.int8, "wd8")
    _vec(s_gate, H, torch.float32, "s_gate")
    _vec(s_up, H, torch.float32, "s_up")
    _vec(s_down, d, torch.float32, "s_down")
    y = _out(out, (M, d), torch.bfloat16, x.device)
    ws, n = _workspace(OP_FFN, M, 0, d, H, x.device, workspace)
    check(lib().gbq_ffn_fused(_ptr(x), _ptr(wg8), _ptr(s_gate), _ptr(wu8), _ptr(s_up), _ptr(wd8), _ptr(s_down),
                              _ptr(y), M, d, H, _rot(rot_d), _rot(rot_h), _ptr(ws), n, _stream(stream)))
    return y


# ------------------------------------------------------------------ backward
def dequant_weight(w8: torch.Tensor, w_scale, r, stream=None):
    """int8 W8 [N,K] + fp32 s [N] -> bf16 W [N,K], un-rotated."""
    _req(w8, torch.int8, "w8")
    N, K = w8.shape
    _vec(w_scale, N, torch.float32, "w_scale")
    w = torch.empty((N, K), dtype=torch.bfloat16, device=w8.device)
    check(lib().gbq_dequant_weight(_ptr(w8), _ptr(w_scale), _ptr(w), N, K, _rot(r), _stream(stream)))
    return w


def linear_dx(dy: torch.Tensor, w: torch.Tensor, out=None, stream=None):
    """bf16 dy [M,N] @ bf16 W [N,K] -> bf16 dx [M,K]."""
    _req(dy, torch.bfloat16, "dy")
    M, N = dy.shape
    K = w.shape[1]
    _mat(w, (N, K), torch.bfloat16, "w")
    dx = _out(out, (M, K), torch.bfloat16, dy.device)
    check(lib().gbq_linear_dx(_ptr(dy), _ptr(w), _ptr(dx), M, N, K, _stream(stream)))
    return dx


def linear_dx_int8(dy: torch.Tensor, w8: torch.Tensor, w_scale, r, workspace=None, out=None, stream=None):
    """dx through the int8 route: quantize dy*s, int8 GEMM against W8, rotate back."""
    _req(dy, torch.bfloat16, "dy")
    M, N = dy.shape
    K = w8.shape[1]
    _mat(w8, (N, K), torch.int8, "w8")
    _vec(w_scale, N, torch.float32, "w_scale")
    dx = _out(out, (M, K), torch.bfloat16, dy.device)
    ws, n = _workspace(OP_LINEAR_DX_INT8, M, N, K, 0, dy.device, workspace)
    check(lib().gbq_linear_dx_int8(_ptr(dy), _ptr(w8), _ptr(w_scale), _ptr(dx), M, N, K, _rot(r), _ptr(ws), n,
                                   _stream(stream)))
    return dx
