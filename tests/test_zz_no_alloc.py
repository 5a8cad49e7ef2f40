"""gbq_linear_noalloc: the linear layer for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc where they run the layer -- a plugin inside a
framework that owns all device memory, or a latency-critical loop that cannot
afford cudaMalloc's implicit synchronisation -- so they cannot provide the
workspace gbq_linear needs.  gbq_linear_noalloc takes its scratch from a static
device array inside the library.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import _lib as L
from ffn_rotate_quantize_gb300 import inputs as I
from parity import assert_bf16_parity, bf16_dev, bf16_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ffn_rotate_quantize_gb300 import ops as G
    G.init()
    return G


def _call_noalloc(x, w8, ws, bias, y, rot):
    M, K = x.shape
    N = w8.shape[0]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = L.lib().gbq_linear_noalloc(p(x), p(w8), p(ws), p(bias), p(y), M, N, K, L.Rot(*rot),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("M,K,N,rot,with_bias", [(300, 4096, 392, (64, 64, 1), True),
                                                  (1, 4096, 4096, (64, 64, 1), False)])
def test_noalloc_matches_linear_on_two_calls(ops, M, K, N, rot, with_bias):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    for call in range(2):  # a second call with other inputs: no state may leak through the shared scratch
        c = I.linear_case(M, K, N, n_outliers=max(1, K // 100), outlier_scale=30.0, bias_std=0.01, seed=100 + call)
        w8, ws = O.prepare_weight(c["w"], rot)
        x = bf16_dev(c["x"])
        bias = bf16_dev(c["bias"]) if with_bias else None
        y_ref = ops.linear(x, d(w8), d(ws), bias, rot)
        y = torch.empty_like(y_ref)
        rc = _call_noalloc(x, d(w8), d(ws), bias, y, rot)
        assert rc == 0, L.lib().gbq_last_error().decode()
        torch.cuda.synchronize()
        assert_bf16_parity(bf16_np(y), bf16_np(y_ref))
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert ops.device_status() == 0


def _linear_pair(ops, M, K, N, rot, seed, with_bias=True):
    """(noalloc output, gbq_linear output on a caller workspace) for one seeded case."""
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    c = I.linear_case(M, K, N, n_outliers=max(1, K // 100), outlier_scale=30.0, bias_std=0.01, seed=seed)
    w8, ws = O.prepare_weight(c["w"], rot)
    x = bf16_dev(c["x"])
    bias = bf16_dev(c["bias"]) if with_bias else None
    y_ref = ops.linear(x, d(w8), d(ws), bias, rot)
    y = torch.empty_like(y_ref)
    rc = _call_noalloc(x, d(w8), d(ws), bias, y, rot)
    assert rc == 0, L.lib().gbq_last_error().decode()
    torch.cuda.synchronize()
    return y, y_ref


def test_noalloc_large_call_then_smaller_calls(ops):
    """A call that fills most of the scratch, then smaller ones (whose scratch is a prefix of what the large
    call wrote), then a non-square rotation, then the few-token GEMV over codes in the scratch: every result
    equals gbq_linear on a workspace, bit for bit, so nothing left in the shared array by an earlier call
    reaches a later one."""
    cases = [(1500, 4096, 256, (64, 64, 1)), (37, 4096, 300, (64, 64, 1)), (2, 4096, 520, (64, 64, 1)),
             (129, 2048, 200, (32, 64, 1)), (8, 4096, 300, (64, 64, 1)), (1, 2048, 200, (32, 64, 1))]
    for i, (M, K, N, rot) in enumerate(cases):
        y, y_ref = _linear_pair(ops, M, K, N, rot, seed=300 + i)
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), (M, K, N, rot)
    assert ops.device_status() == 0


def test_noalloc_at_its_limit(ops):
    """M = 2047, K = 4096: codes and scales take exactly the 16 MiB, so the optional per-block code sums
    do not fit and the GEMM runs its default exact chunks; still bit-identical to gbq_linear with the
    full workspace (which has room for the sums)."""
    M, K, N, rot = 2047, 4096, 256, (64, 64, 1)
    assert M * K * 2 + (M * 4 + 255) // 256 * 256 == 16 << 20
    y, y_ref = _linear_pair(ops, M, K, N, rot, seed=400, with_bias=False)
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert ops.device_status() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(ops):
    M, K, N = 2048, 8192, 256  # 32 MiB of codes > the 16 MiB static scratch
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w8 = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    ws = torch.ones(N, dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rc = _call_noalloc(x, w8, ws, None, y, (64, 64, 2))
    assert rc == -28
    assert "static scratch" in L.lib().gbq_last_error().decode()
