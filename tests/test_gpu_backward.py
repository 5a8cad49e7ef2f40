"""GPU parity of the dx backward: dequant_weight + linear_dx, and linear_dx_int8."""
import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I
from parity import acc_error_usage, assert_bf16_parity, assert_int8_parity, bf16_dev, bf16_np, bf16_half_ulp, f32

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


DX_CASES = [(200, 2048, 1024, (32, 32, 1)), (64, 16384, 256, (16, 16, 1)), (129, 1024, 4096, (64, 64, 1)),
            (700, 16384, 256, (16, 16, 1)), (160, 12288, 512, (16, 16, 2))]


@pytest.mark.parametrize("M,N,K,rot", DX_CASES)
def test_linear_dx(ops, M, N, K, rot):
    c = I.backward_case(M, N, K, seed=M + N)
    w8, s = O.prepare_weight(c["w"], rot)
    what = O.dequant_weight(w8, s, rot)
    dx = ops.linear_dx(bf16_dev(c["dy"]), bf16_dev(what))
    assert_bf16_parity(bf16_np(dx), O.linear_dx(c["dy"], what), acc_len=N)
    # The max-rel floor rests on a bound E * rms of the fp32 accumulation error: show how much of it is used.
    exact = f32(c["dy"]).astype(np.float64) @ f32(what).astype(np.float64)
    usage = acc_error_usage(bf16_np(dx), exact, N)
    print(f"linear_dx {M}x{N}x{K}: accumulation error uses {usage:.3g} of E*rms")
    assert usage <= 0.5


@pytest.mark.parametrize("M,N,K,rot", DX_CASES)
def test_linear_dx_int8(ops, M, N, K, rot):
    c = I.backward_case(M, N, K, seed=M + N + 1)
    w8, s = O.prepare_weight(c["w"], rot)
    dx = ops.linear_dx_int8(bf16_dev(c["dy"]), d(w8), d(s), rot)
    dx_r, mid = O.linear_dx_int8(c["dy"], w8, s, rot, keep=True)
    assert_bf16_parity(bf16_np(dx), dx_r)


@pytest.mark.parametrize("N,K,groups", [(300, 4096, 1), (64, 8192, 2), (1000, 4096, 1)])
def test_dequant_weight_at_its_rounding_bound(ops, N, K, groups):
    """dequant_weight for H64 (x) H64 transforms the codes exactly and rounds once, W_hat = bf16(fl((W8 s) R));
    the oracle rounds W8 s to fp32 first and sums in fp64 (reading R-17).  So every element is within one
    bf16 unit of the oracle's plus the residue of its fp32 roundings, 64 * 127 * s[n] * 2^-24, and not
    merely within the generic bf16 tolerance."""
    rot = (64, 64, groups)
    c = I.backward_case(8, N, K, seed=N + K)
    w8, s = O.prepare_weight(c["w"], rot)
    w = f32(bf16_np(ops.dequant_weight(d(w8), d(s), rot))).astype(np.float64)
    r = f32(O.dequant_weight(w8, s, rot)).astype(np.float64)
    bound = 2.0 * bf16_half_ulp(np.maximum(np.abs(w), np.abs(r))) + 64 * 127 * s.astype(np.float64)[:, None] * 2.0 ** -24
    err = np.abs(w - r)
    assert np.all(err <= bound), f"worst {np.max(err / bound):.3f} of the bound"
    print(f"dequant_weight {N}x{K}: {np.count_nonzero(err)} of {err.size} elements differ, worst "
          f"{np.max(err / bound):.3f} of the bound")


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


def _a256(v):
    return (v + 255) // 256 * 256


def test_linear_dx_int8_chunk_plan(ops):
    """With the preferred workspace the dy quantizer also writes each row's sum of |code| over every
    1024-long block of N, and the int8 GEMM accumulates longer exact fp32 chunks for token tiles whose
    sums allow it.  The result must equal, bit for bit, the one from the minimum workspace (1024-long
    chunks), here with a tile of all-(+127) rows against all-(+127) weight columns (partial sums up to
    127^2 * 1024 per block, so that tile must keep 1024-long chunks) beside Gaussian tiles."""
    rng = np.random.default_rng(23)
    M, N, K, rot = 300, 16384, 1024, (32, 32, 1)
    dy = rng.standard_normal((M, N)).astype(np.float32) * np.float32(1e-3)
    dy[:128] = np.float32(2e-3)  # codes +127 everywhere
    dy_b = I.bf16_bits(dy)
    w8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
    w8[:, :8] = 127
    s = np.ones(N, np.float32)
    dyd, w8d, sd = bf16_dev(dy_b), d(w8), d(s)
    pref = ops.workspace_size(ops.OP_LINEAR_DX_INT8, M, N, K)
    minimum = _a256(M * N * 2) + _a256(M * 4) + _a256(M * K * 4)
    assert pref == minimum + _a256(M * 4 * (N // 1024))
    ws_p = torch.zeros(pref, dtype=torch.uint8, device="cuda")
    ws_m = torch.zeros(minimum, dtype=torch.uint8, device="cuda")
    dx_p = ops.linear_dx_int8(dyd, w8d, sd, rot, ws_p)
    dx_m = ops.linear_dx_int8(dyd, w8d, sd, rot, ws_m)
    torch.cuda.synchronize()
    assert torch.equal(dx_p.view(torch.int16), dx_m.view(torch.int16))
    # the block sums written by the quantizer match its own codes
    codes = ws_p[:M * N * 2].view(torch.float16).view(M, N).float().cpu().numpy().astype(np.int64)
    l1 = ws_p[minimum:minimum + M * 4 * 16].view(torch.int32).view(M, 16).cpu().numpy()
    assert np.array_equal(l1, np.abs(codes).reshape(M, 16, 1024).sum(axis=2))
    assert l1[:128].min() == 127 * 1024 and l1[128:].max() < 2 ** 17 // 4  # tile 0: 1-block chunks only
    assert_bf16_parity(bf16_np(dx_p), O.linear_dx_int8(dy_b, w8, s, rot))


def test_linear_dx_int8_dy_codes_long_run(ops):
    """The dy quantizer's codes, row scales and block sums with more rows than SMs times row stages (each
    persistent CTA of the long-row quantizer reuses its shared-memory stages), a zero row among them: equal,
    bit for bit, to the oracle's per-row quantization of dy * s (R = I, so no rotation rounding)."""
    rng = np.random.default_rng(29)
    M, N, K, rot = 1500, 16384, 256, (16, 16, 1)
    dy_b = I.bf16_bits(rng.standard_normal((M, N)).astype(np.float32) * np.float32(1e-3))
    dy_b[5] = 0
    w8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s = rng.random(N).astype(np.float32) * np.float32(0.01) + np.float32(1e-3)
    pref = ops.workspace_size(ops.OP_LINEAR_DX_INT8, M, N, K)
    minimum = _a256(M * N * 2) + _a256(M * 4) + _a256(M * K * 4)
    ws_p = torch.zeros(pref, dtype=torch.uint8, device="cuda")
    dx = ops.linear_dx_int8(bf16_dev(dy_b), d(w8), d(s), rot, ws_p)
    torch.cuda.synchronize()
    dx_r, mid = O.linear_dx_int8(dy_b, w8, s, rot, keep=True)
    codes = ws_p[:M * N * 2].view(torch.float16).view(M, N).float().cpu().numpy().astype(np.int64)
    t = ws_p[_a256(M * N * 2):_a256(M * N * 2) + M * 4].view(torch.float32).cpu().numpy()
    assert t[5] == 0 and not codes[5].any()
    assert np.array_equal(t, mid["t"])
    assert np.array_equal(codes, mid["qd"].astype(np.int64))
    l1 = ws_p[minimum:minimum + M * 4 * 16].view(torch.int32).view(M, 16).cpu().numpy()
    assert np.array_equal(l1, np.abs(codes).reshape(M, 16, 1024).sum(axis=2))
    assert_bf16_parity(bf16_np(dx), dx_r)
