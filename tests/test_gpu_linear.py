"""GPU parity of the int8 GEMM, dequant epilogue, linear_acc and linear (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I
from parity import assert_bf16_parity, assert_int8_parity, assert_rows_explained, bf16_dev, bf16_np

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


# Shapes span several 128x128 tiles, ragged tails in M and N, K below, at and above
# one 1024-long exact chunk, and the K of the down projection.
GEMM_SHAPES = [(300, 392, 4096), (1, 128, 64), (129, 130, 1088), (64, 256, 16384), (257, 384, 1024)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_int8_gemm_bit_exact(ops, M, N, K):
    rng = np.random.default_rng(M + N + K)
    q = rng.integers(-127, 128, (M, K)).astype(np.int8)
    w = rng.integers(-127, 128, (N, K)).astype(np.int8)
    acc = ops.int8_gemm(d(q), d(w)).cpu().numpy()
    assert np.array_equal(acc.astype(np.int64), O.gemm_s8(q, w))


@pytest.mark.parametrize("K", [1024, 4096, 16384])
def test_int8_gemm_extreme_magnitudes(ops, K):
    """All-|127| operands: partial sums reach 127^2*K, far past 2^24 in fp32."""
    M, N = 130, 256
    rng = np.random.default_rng(K)
    q = np.where(rng.random((M, K)) < 0.5, 127, -127).astype(np.int8)
    q[:3] = 127
    w = np.where(rng.random((N, K)) < 0.5, 127, -127).astype(np.int8)
    w[:3] = 127
    w[3:6] = -127
    acc = ops.int8_gemm(d(q), d(w)).cpu().numpy()
    assert np.array_equal(acc.astype(np.int64), O.gemm_s8(q, w))
    assert acc[0, 0] == 127 * 127 * K and acc[0, 3] == -127 * 127 * K


def test_int8_gemm_one_hot_rows(ops):
    """Rotated one-hot rows quantize to +-127 patterns whose products reach 127^2*K."""
    rot, K = (64, 64, 1), 4096
    x = np.zeros((8, K), np.float32)
    for r in range(8):
        x[r, 37 * r] = 1.0
    q, _ = O.rotate_quantize(I.bf16_bits(x), rot)
    acc = ops.int8_gemm(d(q), d(q)).cpu().numpy().astype(np.int64)
    assert np.array_equal(acc, np.diag(np.full(8, 127 * 127 * K)))


def _case(M, K, N, seed, rot, outliers=True):
    c = I.linear_case(M, K, N, n_outliers=max(1, K // 100) if outliers else 0, outlier_scale=30.0,
                      bias_std=0.01, seed=seed)
    w8, ws = O.prepare_weight(c["w"], rot)
    return c, w8, ws


LINEAR_CASES = [(300, 4096, 392, (64, 64, 1)), (16, 256, 256, (16, 16, 1)), (129, 1024, 200, (32, 32, 1)),
                (64, 16384, 256, (128, 128, 1)), (40, 3072, 128, (16, 16, 12)),
                # N*2 bytes not a multiple of 16: rows too ragged for the tensor-store epilogue
                (130, 1024, 131, (32, 32, 1))]


@pytest.mark.parametrize("M,K,N,rot", LINEAR_CASES)
def test_linear_and_linear_acc(ops, M, K, N, rot):
    c, w8, ws = _case(M, K, N, seed=M + K, rot=rot)
    x, bias = bf16_dev(c["x"]), bf16_dev(c["bias"])
    acc, xs = ops.linear_acc(x, d(w8), rot)
    y = ops.linear(x, d(w8), d(ws), bias, rot)
    torch.cuda.synchronize()
    qr, sr = O.rotate_quantize(c["x"], rot)
    acc_r = O.gemm_s8(qr, w8)
    y_r = O.dequant(acc_r, sr, ws, c["bias"])
    # The GPU's own quantized x: rows whose codes match the oracle's must give the exact accumulator.
    qg, _ = ops.quantize_act(x, rot)
    assert_int8_parity(qg.cpu().numpy(), qr)
    same = np.all(qg.cpu().numpy() == qr, axis=1)
    assert np.array_equal(acc.cpu().numpy()[same].astype(np.int64), acc_r[same])
    assert_rows_explained(bf16_np(y), y_r, same)
    # dequant(linear_acc(x)) == linear(x), bit for bit ("Use from Python").
    y2 = ops.dequant(acc, xs, d(ws), bias)
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))


def test_tiny_config_exact(ops):
    """x [16,256], W [256,256], R = H16 (x) H16 / 16, bias."""
    c = I.config_case("tiny_linear")
    rot = c["config"]["rot"]
    w8g, wsg = ops.prepare_weight(bf16_dev(c["w"]), rot)
    w8, ws = O.prepare_weight(c["w"], rot)
    assert_int8_parity(w8g.cpu().numpy(), w8)
    y = ops.linear(bf16_dev(c["x"]), w8g, wsg, bf16_dev(c["bias"]), rot)
    assert_bf16_parity(bf16_np(y), O.linear(c["x"], w8, ws, c["bias"], rot))


def test_dequant_standalone_and_slice(ops):
    rng = np.random.default_rng(9)
    M, N = 77, 520
    acc = rng.integers(-2 ** 27, 2 ** 27, (M, N)).astype(np.int32)
    xs = (rng.random(M) * 1e-4).astype(np.float32)
    ws = (rng.random(N) * 1e-3).astype(np.float32)
    bias = I.bf16_bits(rng.standard_normal(N).astype(np.float32) * 0.01)
    y = ops.dequant(d(acc), d(xs), d(ws), bf16_dev(bias))
    ref = O.dequant(acc.astype(np.int64), xs, ws, bias)
    assert np.array_equal(bf16_np(y), ref)  # identical fp32 operations -> identical bits
    # a strided column slice of a wider accumulator (the page's dequant_slice)
    s0, s1 = 128, 392
    ys = ops.dequant(d(acc)[:, s0:s1], d(xs), d(ws[s0:s1]), bf16_dev(bias[s0:s1]))
    assert np.array_equal(bf16_np(ys), ref[:, s0:s1])
    yn = ops.dequant(d(acc), d(xs), d(ws), None)
    assert np.array_equal(bf16_np(yn), O.dequant(acc.astype(np.int64), xs, ws, None))


# M <= 4 runs a decode GEMV (weight streaming) inside gbq_linear (the rotation inside for the square shapes
# it covers, else the codes GEMV); linear_acc stays on the GEMM.
DECODE_CASES = [(1, 4096, 4096, (64, 64, 1), False), (2, 1024, 520, (32, 32, 1), True),
                (4, 256, 1000, (16, 16, 1), True), (3, 4096, 300, (16, 16, 16), False), (1, 4096, 7, (64, 64, 1), True),
                (4, 4096, 1500, (64, 64, 1), True), (3, 8192, 333, (64, 64, 2), False),
                # K = 4096 register-streaming kernel (one or two tokens): three rows per warp with slice rows
                # 16.. staged in shared memory (N = 3000: 20 rows per CTA); 32 rows per CTA; three and four
                # tokens (the codes GEMV) with a ragged last slice (N = 4100: 27 rows per CTA, the last CTA 23)
                (2, 4096, 3000, (64, 64, 1), True), (3, 4096, 4100, (64, 64, 1), False),
                (4, 4096, 4864, (64, 64, 1), True), (1, 4096, 4864, (64, 64, 1), True),
                (2, 4096, 4864, (64, 64, 1), False),
                # the ring kernel with the rotation inside (one or two tokens, K <= 4096): n = 16, n = 16 in
                # sixteen groups, n = 64 past the register-streaming kernel's 32 rows per CTA
                (1, 256, 1000, (16, 16, 1), True), (2, 4096, 300, (16, 16, 16), False),
                (1, 4096, 6000, (64, 64, 1), True)]


@pytest.mark.parametrize("M,K,N,rot,with_bias", DECODE_CASES)
def test_decode_gemv(ops, M, K, N, rot, with_bias):
    c, w8, ws = _case(M, K, N, seed=M * 3 + K + N, rot=rot)
    x = bf16_dev(c["x"])
    bias = bf16_dev(c["bias"]) if with_bias else None
    bias_np = c["bias"] if with_bias else None
    y = ops.linear(x, d(w8), d(ws), bias, rot)
    acc, xs = ops.linear_acc(x, d(w8), rot)
    y2 = ops.dequant(acc, xs, d(ws), bias)
    # the GEMV path and the GEMM path + dequant give the same bits
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    qr, sr = O.rotate_quantize(c["x"], rot)
    qg, _ = ops.quantize_act(x, rot)
    assert_int8_parity(qg.cpu().numpy(), qr)
    same = np.all(qg.cpu().numpy() == qr, axis=1)
    assert_rows_explained(bf16_np(y), O.dequant(O.gemm_s8(qr, w8), sr, ws, bias_np), same)


def test_linear_large_accumulators_exact(ops):
    """One-hot x and W rows rotate to +-127 code patterns, so matching rows accumulate 127^2*K
    (far past 2^22) next to zeros: the bf16 epilogue must convert both exactly."""
    rot, M, K, N = (64, 64, 1), 8, 4096, 256
    x = np.zeros((M, K), np.float32)
    w = np.zeros((N, K), np.float32)
    for r in range(M):
        x[r, 37 * r] = 1.0 + r
    for n in range(N):
        w[n, (37 * n) % K] = 0.5
    xb, wb = I.bf16_bits(x), I.bf16_bits(w)
    bias = I.bf16_bits(np.linspace(-1, 1, N).astype(np.float32))
    w8, ws = O.prepare_weight(wb, rot)
    y = ops.linear(bf16_dev(xb), d(w8), d(ws), bf16_dev(bias), rot)
    y_r = O.linear(xb, w8, ws, bias, rot)
    assert np.array_equal(bf16_np(y), y_r)
    assert np.abs(O.linear_acc(xb, w8, rot)[0]).max() == 127 * 127 * K


def test_linear_acc_extended_chunk_at_its_bound(ops):
    """The tightest case of the chunk plan: every token's codes are positive and each aligned pair of
    1024-long blocks sums to just under 2^17, so the tile takes 2048-long exact chunks whose partial sums
    against all-(+127) weight rows reach 127 * sum|q| ~ 0.99 * 2^24 (a 4096-long chunk would pass 2^24 and
    round).  x = R v for target codes v (R is symmetric and orthogonal, so x rotates back to v up to the
    bf16 rounding of x); the accumulators must equal the int64 product of the GPU's own codes."""
    rot, M, K, N = (64, 64, 1), 300, 4096, 256
    rng = np.random.default_rng(53)
    v = rng.integers(51, 79, (M, K)).astype(np.float64)
    v[:, 0] = 127.0
    for m in range(M):  # each 2048-long half sums to at most 130300 (a margin for the bf16 rounding of x)
        for h in range(2):
            seg = v[m, 2048 * h:2048 * (h + 1)]
            extra = int(seg.sum() - 130300)
            if extra > 0:
                np.subtract.at(seg, rng.integers(1, 2048, extra), 1.0)
    x = I.bf16_bits(O.rotate(v.astype(np.float32), rot))  # R v (fp64 sums, rounded), then bf16
    w8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
    w8[:8] = 127
    w8[8:16] = np.where(np.arange(K) % 2 == 0, 127, -127)
    acc, _ = ops.linear_acc(bf16_dev(x), d(w8), rot)
    q = ops.quantize_act(bf16_dev(x), rot)[0].cpu().numpy().astype(np.int64)
    assert q.min() >= 0
    blk = np.abs(q).reshape(M, 4, 1024).sum(axis=2)
    pairs = blk[:, 0::2] + blk[:, 1::2]
    assert pairs.max() <= 2 ** 17 and pairs.min() > 2 ** 17 - 2000, (pairs.min(), pairs.max())
    assert blk.sum(axis=1).min() > 2 ** 17  # a 4096-long chunk would not be exact
    assert 127 * pairs.max() > 0.98 * 2 ** 24
    acc_r = O.gemm_s8(q.astype(np.int8), w8)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_r)
    assert acc_r[:, :8].min() > 1.9 * 2 ** 24  # totals far past 2^24, from exact 2048-long chunks


def test_linear_acc_chunk_plans_exact(ops):
    """Token tiles whose codes have small sums of |q| over their 1024-long K blocks accumulate
    longer exact fp32 chunks, tiles with large ones (one-hot rows rotate to all-|127| codes) take
    1024-long chunks: both must give
    the exact int32 accumulator of the GPU's own codes, here against weights that include all-|127|
    rows (the largest partial sums the bound allows)."""
    rot, M, K, N = (64, 64, 1), 600, 4096, 300
    rng = np.random.default_rng(41)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[256:512] = 0.0
    for r in range(256, 512):
        x[r, (13 * r) % K] = 1.0 + (r % 7)  # one-hot: codes +-127 everywhere, sum |q| = 127 K
    xb = I.bf16_bits(x)
    w8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
    w8[:8] = 127
    w8[8:16] = np.where(rng.random((8, K)) < 0.5, 127, -127)
    acc, _ = ops.linear_acc(bf16_dev(xb), d(w8), rot)
    qg, _ = ops.quantize_act(bf16_dev(xb), rot)
    q = qg.cpu().numpy()
    blk = np.abs(q.astype(np.int64)).reshape(M, 4, 1024).sum(axis=2)  # |q| sums of the 1024-long blocks
    pairs = blk[:, 0::2] + blk[:, 1::2]
    assert pairs[:256].max() <= 2 ** 17 and pairs[256:512].min() > 2 ** 17  # longer and default chunks
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), O.gemm_s8(q, w8))
    # and through the FFN-sized contraction (K = 16384, rot128): large L1 -> default chunks
    rot2, K2 = (128, 128, 1), 16384
    x2 = I.bf16_bits(rng.standard_normal((130, K2)).astype(np.float32))
    w2 = rng.integers(-127, 128, (64, K2)).astype(np.int8)
    acc2, _ = ops.linear_acc(bf16_dev(x2), d(w2), rot2)
    q2, _ = ops.quantize_act(bf16_dev(x2), rot2)
    assert np.array_equal(acc2.cpu().numpy().astype(np.int64), O.gemm_s8(q2.cpu().numpy(), w2))


@pytest.mark.parametrize("M,N,with_bias", [(70000, 16, True), (33, 100, True), (5, 2051, False), (300, 14336, True)])
def test_dequant_shapes(ops, M, N, with_bias):
    """The 8-column path (including rows striding past the grid's rows), ragged last column groups and the
    element-by-element path (N not a multiple of 8, so rows are not 16-byte aligned) compute the oracle's
    fp32 operations: identical bits."""
    rng = np.random.default_rng(M + N)
    acc = rng.integers(-2 ** 27, 2 ** 27, (M, N)).astype(np.int32)
    xs = (rng.random(M) * 1e-4).astype(np.float32)
    ws = (rng.random(N) * 1e-3).astype(np.float32)
    bias = I.bf16_bits(rng.standard_normal(N).astype(np.float32) * 0.01) if with_bias else None
    y = ops.dequant(d(acc), d(xs), d(ws), bf16_dev(bias) if with_bias else None)
    assert np.array_equal(bf16_np(y), O.dequant(acc.astype(np.int64), xs, ws, bias))


def test_binding_rejects_wrong_output_shape(ops):
    """The binding checks a caller's output tensor before the C call writes M x N elements through it."""
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    w8 = torch.zeros((64, 256), dtype=torch.int8, device="cuda")
    s = torch.ones((64,), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        ops.linear(x, w8, s, None, (16, 16, 1), out=torch.empty((2, 32), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        ops.linear(x, w8, s, None, (16, 16, 1), out=torch.empty((2, 64), dtype=torch.float32, device="cuda"))
    y = ops.linear(x, w8, s, None, (16, 16, 1), out=torch.empty((2, 64), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert y.shape == (2, 64) and bool((y.float() == 0).all())
    # inputs: a weight of the wrong width, a scale or bias vector of the wrong length
    with pytest.raises(ValueError):
        ops.linear(x, torch.zeros((64, 128), dtype=torch.int8, device="cuda"), s, None, (16, 16, 1))
    with pytest.raises(ValueError):
        ops.linear(x, w8, torch.ones((32,), dtype=torch.float32, device="cuda"), None, (16, 16, 1))
    with pytest.raises(ValueError):
        ops.linear(x, w8, s, torch.zeros((65,), dtype=torch.bfloat16, device="cuda"), (16, 16, 1))
    # a caller's workspace is passed with its real size: one too small is refused by the library
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(Exception, match="workspace"):
        ops.linear(x, w8, s, None, (16, 16, 1), workspace=small)


@pytest.mark.parametrize("M", [1, 8, 300])
def test_linear_into_pinned_host_memory(ops, M):
    """y in pinned host memory: the GEMM (plain stores instead of TMA) and the GEMVs write it directly; the
    result equals the device-resident one bit for bit."""
    from ffn_rotate_quantize_gb300 import _lib as L
    K, N, rot = 4096, 520, (64, 64, 1)
    c = I.linear_case(M, K, N, n_outliers=41, outlier_scale=30.0, bias_std=0.01, seed=500 + M)
    w8, ws = O.prepare_weight(c["w"], rot)
    x, bias = bf16_dev(c["x"]), bf16_dev(c["bias"])
    w8d, wsd = d(w8), d(ws)
    y_dev = ops.linear(x, w8d, wsd, bias, rot)
    y_host = torch.zeros((M, N), dtype=torch.bfloat16).pin_memory()
    work = torch.empty(ops.workspace_size(ops.OP_LINEAR, M, N, K), dtype=torch.uint8, device="cuda")
    L.check(L.lib().gbq_linear(x.data_ptr(), w8d.data_ptr(), wsd.data_ptr(), bias.data_ptr(), y_host.data_ptr(),
                               M, N, K, ops._rot(rot), work.data_ptr(), work.numel(),
                               torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
