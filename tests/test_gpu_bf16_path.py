"""GPU parity of the rotate-only BF16 path ("Use from C" on the PyPI page "xpu-kernels 0.2.0"):
gbq_rotate_bf16 on the activation, then gbq_linear_bf16 against the weight stored pre-rotated in bf16."""
import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I
from parity import acc_error_usage, assert_bf16_parity, bf16_dev, bf16_np, f32

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


# Several 128 x 256 tiles, ragged M and N tails, N not a multiple of 8 (element-wise epilogue),
# one contraction block (K = 64) and long ones.
SHAPES = [(300, 392, 4096), (1, 128, 64), (129, 131, 1088), (257, 1000, 1024), (64, 520, 16384)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("with_bias", [True, False])
def test_linear_bf16(ops, M, N, K, with_bias):
    rng = np.random.default_rng(M + N + K + with_bias)
    x = I.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = I.bf16_bits(rng.standard_normal((N, K)).astype(np.float32) * np.float32(0.02))
    b = I.bf16_bits(rng.standard_normal(N).astype(np.float32) * np.float32(0.05)) if with_bias else None
    y = ops.linear_bf16(bf16_dev(x), bf16_dev(w), bf16_dev(b) if with_bias else None)
    assert_bf16_parity(bf16_np(y), O.linear_bf16(x, w, b), acc_len=K)
    exact = f32(x).astype(np.float64) @ f32(w).astype(np.float64).T
    if with_bias:
        exact = exact + f32(b).astype(np.float64)[None, :]
    usage = acc_error_usage(bf16_np(y), exact, K)
    print(f"linear_bf16 {M}x{N}x{K}: accumulation error uses {usage:.3g} of E*rms")
    assert usage <= 0.5


def test_linear_bf16_exact_on_small_integers(ops):
    """Small-integer operands: every fp32 partial sum is an exact integer, so the only rounding is the
    final one to bf16 and the result is bit-exact."""
    rng = np.random.default_rng(5)
    M, N, K = 130, 300, 1024
    xb = I.bf16_bits(rng.integers(-4, 5, (M, K)).astype(np.float32))
    wb = I.bf16_bits(rng.integers(-4, 5, (N, K)).astype(np.float32))
    bb = I.bf16_bits(rng.integers(-100, 101, N).astype(np.float32))
    y = ops.linear_bf16(bf16_dev(xb), bf16_dev(wb), bf16_dev(bb))
    assert np.array_equal(bf16_np(y), O.linear_bf16(xb, wb, bb))


@pytest.mark.parametrize("M,K,N,rot", [(300, 4096, 392, (64, 64, 1)), (40, 3072, 128, (16, 16, 12)),
                                       (129, 16384, 256, (128, 128, 1))])
def test_rotated_bf16_layer(ops, M, K, N, rot):
    """The comparator chain: GPU rotation of x, then the bf16 linear against bf16(W R)."""
    c = I.linear_case(M, K, N, n_outliers=max(1, K // 100), outlier_scale=30.0, bias_std=0.01, seed=M + K)
    wr = O.rotate_bf16(c["w"], rot)  # one-time weight preparation of the bf16 path
    xr = ops.rotate_bf16(bf16_dev(c["x"]), rot)
    y = ops.linear_bf16(xr, bf16_dev(wr), bf16_dev(c["bias"]))
    xr_ref = O.rotate_bf16(c["x"], rot)
    assert_bf16_parity(bf16_np(xr), xr_ref, what="x R")
    # An element of x R whose fp32 sum sits at a bf16 rounding boundary may round the other way than
    # the oracle's fp64 sum; the linear is checked element by element on the GPU's own rotated x,
    # the whole chain normwise against the oracle's chain.
    assert_bf16_parity(bf16_np(y), O.linear_bf16(bf16_np(xr), wr, c["bias"]), acc_len=K)
    assert_bf16_parity(bf16_np(y), O.linear_bf16(xr_ref, wr, c["bias"]), maxrel=np.inf)


def test_rotated_bf16_prefill_sampled(ops):
    """The full prefill shape (x [1024,4096], W [14336,4096], R = H64 (x) H64 / 64, bias) in the launch
    configuration the benchmark times; the oracle checks 12 sampled rows."""
    rot, M, K, N = (64, 64, 1), 1024, 4096, 14336
    c = I.linear_case(M, K, N, n_outliers=I.outlier_count(K), outlier_scale=30.0, bias_std=0.01, seed=0)
    wr_d = ops.rotate_bf16(bf16_dev(c["w"]), rot)
    xr_d = ops.rotate_bf16(bf16_dev(c["x"]), rot)
    y = ops.linear_bf16(xr_d, wr_d, bf16_dev(c["bias"]))
    rows = np.random.default_rng(1).choice(M, 12, replace=False)
    rows[0], rows[1] = 0, M - 1
    xr = bf16_np(xr_d)[rows]
    wr = bf16_np(wr_d)
    assert_bf16_parity(bf16_np(y)[rows], O.linear_bf16(xr, wr, c["bias"]), acc_len=K)


def test_linear_bf16_rejects_bad_args(ops):
    x = torch.zeros((4, 96), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        ops.linear_bf16(x, w)  # K = 96 is not a multiple of 64
    y = ops.linear_bf16(torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((8, 128), dtype=torch.bfloat16, device="cuda"))
    assert y.shape == (0, 8)
