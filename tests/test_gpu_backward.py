"""GPU parity of the dx backward: dequant_weight + linear_dx, and linear_dx_int8."""
import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I
from parity import assert_bf16_parity, assert_int8_parity, bf16_dev, bf16_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ffn_rotate_quantize_gb300 import ops as G
    G.init()
    return G


@pytest.fixture(autouse=True)
def _device_status_clean(ops):
    yield
    assert ops.device_status() == 0


def d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


DX_CASES = [(200, 2048, 1024, (32, 32, 1)), (64, 16384, 256, (16, 16, 1)), (129, 1024, 4096, (64, 64, 1))]


@pytest.mark.parametrize("M,N,K,rot", DX_CASES)
def test_linear_dx(ops, M, N, K, rot):
    c = I.backward_case(M, N, K, seed=M + N)
    w8, s = O.prepare_weight(c["w"], rot)
    what = O.dequant_weight(w8, s, rot)
    dx = ops.linear_dx(bf16_dev(c["dy"]), bf16_dev(what))
    assert_bf16_parity(bf16_np(dx), O.linear_dx(c["dy"], what), acc_len=N)


@pytest.mark.parametrize("M,N,K,rot", DX_CASES)
def test_linear_dx_int8(ops, M, N, K, rot):
    c = I.backward_case(M, N, K, seed=M + N + 1)
    w8, s = O.prepare_weight(c["w"], rot)
    dx = ops.linear_dx_int8(bf16_dev(c["dy"]), d(w8), d(s), rot)
    dx_r, mid = O.linear_dx_int8(c["dy"], w8, s, rot, keep=True)
    assert_bf16_parity(bf16_np(dx), dx_r)


def test_linear_dx_int8_gemm_exact(ops):
    """The contraction over W8's rows is exact given identical codes (dy on the int grid, s = 1)."""
    rng = np.random.default_rng(21)
    M, N, K = 130, 2048, 256
    qd = rng.integers(-127, 128, (M, N))
    qd[:, 0] = 127
    dy = I.bf16_bits(qd.astype(np.float32) * np.float32(2.0 ** -7))
    w8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s = np.ones(N, np.float32)
    dx = ops.linear_dx_int8(bf16_dev(dy), d(w8), d(s), (16, 16, 1))
    assert_bf16_parity(bf16_np(dx), O.linear_dx_int8(dy, w8, s, (16, 16, 1)))


def test_linear_dx_int8_large_accumulators(ops):
    """Accumulators past 2^22 (dy rows of ones against +127 weight rows) beside small ones in
    the same tile: the fp32 row-scale epilogue converts both ranges exactly."""
    rng = np.random.default_rng(23)
    M, N, K = 130, 1024, 256
    dy = rng.standard_normal((M, N)).astype(np.float32)
    dy[::3] = 1.0
    dy = I.bf16_bits(dy)
    w8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
    w8[:, :40] = 127
    s = np.ones(N, np.float32)
    dx = ops.linear_dx_int8(bf16_dev(dy), d(w8), d(s), (16, 16, 1))
    assert_bf16_parity(bf16_np(dx), O.linear_dx_int8(dy, w8, s, (16, 16, 1)))
