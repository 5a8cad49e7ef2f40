"""GPU parity for every shape of the rotation descriptor: a != b, small factors, odd total log2 (one
unnormalised H2 level, scaled by fl(sqrt(1/2))), many groups, and the identity on outputs that used to
need a rotation.  The descriptor is R = I_groups (x) (H_a (x) H_b) / sqrt(a*b) with any powers of two
(PyPI page "xpu-kernels 0.2.0", "Algorithm: fused ConvRot rotation": the transform is a Kronecker
product of Hadamard factors; the page's own instance is H4^(x)4 per 256-group).  Everything is checked
against the CPU oracle, whose rotation is the explicit Kronecker definition summed in fp64."""
import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I
from parity import (assert_bf16_parity, assert_int8_parity, assert_rows_explained, assert_scale_parity,
                    bf16_dev, bf16_np)

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


def _x(M, K, seed, outliers=0, scale=30.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outliers:
        idx = rng.choice(K, outliers, replace=False)
        x[:, idx] *= scale
    if M > 2:
        x[1] = 0.0          # an all-zero row
        x[2] *= 1e4         # a large-magnitude row
    return I.bf16_bits(x)


def _oracle_q(xb, rot):
    v = O.rotate(O.bf16_to_f32(xb), rot)
    q, s = O.quantize(v)
    with np.errstate(divide="ignore", invalid="ignore"):
        vs = np.where(s[:, None] > 0, v / s[:, None], 0).astype(np.float32)
    return q, s, vs


# K = 2048 and 8192 as non-square full-width factors (common hidden sizes), small factors, odd total
# log2, the identity factor on one side, factors above 128, grouped non-square forms.
NONSQUARE = [(32, 64, 1), (64, 32, 1), (64, 128, 1), (128, 64, 1), (16, 32, 1), (32, 16, 3), (2, 32, 1),
             (8, 8, 1), (4, 16, 4), (16, 4, 1), (2, 2, 16), (1, 64, 1), (64, 1, 2), (256, 8, 1), (8, 256, 1),
             (2, 1, 8), (128, 256, 1), (4, 4, 3)]


@pytest.mark.parametrize("rot", NONSQUARE)
@pytest.mark.parametrize("M", [1, 7, 130])
def test_quantize_act_any_descriptor(ops, rot, M):
    K = rot[0] * rot[1] * rot[2]
    xb = _x(M, K, seed=M * 11 + K + rot[0], outliers=max(1, K // 100))
    q, s = ops.quantize_act(bf16_dev(xb), rot)
    torch.cuda.synchronize()
    qr, sr, vs = _oracle_q(xb, rot)
    assert_scale_parity(s.cpu().numpy(), sr)
    assert_int8_parity(q.cpu().numpy(), qr, vs)


@pytest.mark.parametrize("rot", [(32, 64, 1), (64, 128, 1), (2, 1, 8), (8, 256, 1)])
def test_one_hot_closed_form_any_descriptor(ops, rot):
    """A one-hot row rotates to +-1/sqrt(a*b) on its group (exact for even log2(a*b); one rounding of
    fl(sqrt(1/2)) otherwise): every code is +-127 in the sign pattern of R's column, other groups 0."""
    K = rot[0] * rot[1] * rot[2]
    ks = [0, 1, K // 3, K - 1]
    x = np.zeros((len(ks), K), np.float32)
    for r, k in enumerate(ks):
        x[r, k] = 1.0
    q, _ = ops.quantize_act(bf16_dev(I.bf16_bits(x)), rot)
    R = O.rotation_matrix(rot)
    qn = q.cpu().numpy().astype(np.int64)
    for r, k in enumerate(ks):
        assert np.array_equal(qn[r], (127 * np.sign(R[:, k])).astype(np.int64))


@pytest.mark.parametrize("rot", [(32, 64, 1), (128, 64, 1), (2, 32, 1), (8, 256, 1)])
def test_rotate_bf16_any_descriptor(ops, rot):
    K = rot[0] * rot[1] * rot[2]
    xb = _x(65, K, seed=K + 3, outliers=3)
    xr = ops.rotate_bf16(bf16_dev(xb), rot)
    assert_bf16_parity(bf16_np(xr), O.rotate_bf16(xb, rot))


# Square descriptors with more groups than one CTA of the square kernels holds run the generic kernel;
# its values must equal the square kernels' bit for bit (same levels, order and fp32 operations).
# A group's rotated values do not depend on the other groups, so a row of G groups rotated at once must
# equal the same G groups rotated as G rows of one group.
@pytest.mark.parametrize("rot", [(16, 16, 128), (32, 32, 40), (64, 64, 9), (128, 128, 3)])
def test_generic_kernel_equals_square_kernels(ops, rot):
    a, b, G = rot
    n = a * b
    xb = _x(24, n * G, seed=n + G, outliers=5)
    wide = ops.rotate_bf16(bf16_dev(xb), rot)                               # generic (many groups)
    per_group = ops.rotate_bf16(bf16_dev(xb.reshape(24 * G, n)), (a, b, 1))  # square kernels
    assert torch.equal(wide.view(torch.int16).reshape(-1), per_group.view(torch.int16).reshape(-1))
    assert_bf16_parity(bf16_np(wide), O.rotate_bf16(xb, rot))


@pytest.mark.parametrize("rot", [(128, 64, 1), (32, 64, 1), (16, 32, 4)])
def test_prepare_weight_any_descriptor(ops, rot):
    K = rot[0] * rot[1] * rot[2]
    rng = np.random.default_rng(K)
    wb = I.bf16_bits(rng.standard_normal((300, K)).astype(np.float32) * 0.02)
    w8, ws = ops.prepare_weight(bf16_dev(wb), rot)
    w8r, wsr = O.prepare_weight(wb, rot)
    v = O.rotate(O.bf16_to_f32(wb), rot)
    assert_scale_parity(ws.cpu().numpy(), wsr)
    assert_int8_parity(w8.cpu().numpy(), w8r, (v / wsr[:, None]).astype(np.float32))


# M <= 16 runs a GEMV: with the generic rotation inside for M K <= 8192, else over codes from the rotation
# kernels (the square in-kernel rotations do not cover these descriptors); larger M the GEMM.  Every route
# gives the same bits as dequant(linear_acc).
# (16, 16, 128) is square but has too many groups for the in-kernel rotation of the decode GEMV; the
# square (64, 64, 1) at M = 5, 8 and 16 takes the codes GEMV as a small batch.
@pytest.mark.parametrize("M,K,N,rot", [(130, 2048, 392, (32, 64, 1)), (1, 2048, 512, (64, 32, 1)),
                                       (64, 8192, 256, (64, 128, 1)), (3, 8192, 300, (128, 64, 1)),
                                       (40, 1024, 200, (8, 8, 16)), (2, 2048, 1000, (32, 64, 1)),
                                       (4, 8192, 777, (64, 128, 1)), (4, 1024, 200, (8, 8, 16)),
                                       (1, 2048, 300, (1, 1, 2048)), (3, 1536, 152, (32, 16, 3)),
                                       (1, 32768, 160, (16, 16, 128)), (4, 16384, 4096, (128, 128, 1)),
                                       (5, 4096, 1000, (64, 64, 1)), (8, 4096, 4096, (64, 64, 1)),
                                       (16, 4096, 700, (64, 64, 1)), (11, 8192, 300, (64, 128, 1)),
                                       (16, 2048, 2000, (32, 64, 1)), (7, 1024, 200, (8, 8, 16)),
                                       # edges of the codes GEMV: fewer weight rows than warps or SMs, one
                                       # row per ring stage at K = 32768, and past its shared-memory limit
                                       (16, 64, 1, (8, 8, 1)), (3, 64, 5, (2, 32, 1)),
                                       (2, 32768, 100, (128, 256, 1)), (4, 32768, 100, (128, 256, 1)),
                                       # the GEMV with the generic rotation inside (M K <= 8192): grouped,
                                       # two tokens, the largest K, factor 2, odd log2, a tiny row
                                       (1, 1024, 200, (8, 8, 16)), (2, 4096, 300, (32, 128, 1)),
                                       (1, 8192, 152, (64, 128, 1)), (1, 4096, 100, (2, 2048, 1)),
                                       (1, 512, 7, (2, 256, 1)), (1, 64, 1, (8, 8, 1))])
def test_linear_any_descriptor(ops, M, K, N, rot):
    c = I.linear_case(M, K, N, n_outliers=max(1, K // 100), outlier_scale=30.0, bias_std=0.01, seed=M + K + N)
    w8, ws = O.prepare_weight(c["w"], rot)
    x, bias = bf16_dev(c["x"]), bf16_dev(c["bias"])
    acc, xs = ops.linear_acc(x, d(w8), rot)
    y = ops.linear(x, d(w8), d(ws), bias, rot)
    torch.cuda.synchronize()
    qr, sr = O.rotate_quantize(c["x"], rot)
    acc_r = O.gemm_s8(qr, w8)
    qg, _ = ops.quantize_act(x, rot)
    assert_int8_parity(qg.cpu().numpy(), qr)
    same = np.all(qg.cpu().numpy() == qr, axis=1)
    assert np.array_equal(acc.cpu().numpy()[same].astype(np.int64), acc_r[same])
    assert_rows_explained(bf16_np(y), O.dequant(acc_r, sr, ws, c["bias"]), same)
    y2 = ops.dequant(acc, xs, d(ws), bias)
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("M,dm,H,rd,rh", [(64, 2048, 8192, (32, 64, 1), (64, 128, 1)),
                                          (40, 1024, 2048, (1, 1, 1024), (1, 1, 2048)),
                                          (33, 512, 1024, (16, 32, 1), (8, 8, 16)),
                                          # the GEMV route (M <= 16)
                                          (1, 2048, 8192, (32, 64, 1), (64, 128, 1)),
                                          (4, 1024, 2048, (1, 1, 1024), (1, 1, 2048)),
                                          (3, 512, 1024, (16, 32, 1), (8, 8, 16))])
def test_ffn_any_descriptor(ops, M, dm, H, rd, rh):
    c = I.ffn_case(M, dm, H, seed=M + dm + H)
    wg8, sg = O.prepare_weight(c["wg"], rd)
    wu8, su = O.prepare_weight(c["wu"], rd)
    wd8, sd = O.prepare_weight(c["wd"], rh)
    x = bf16_dev(c["x"])
    y = ops.ffn_fused(x, d(wg8), d(sg), d(wu8), d(su), d(wd8), d(sd), rd, rh)
    accg, xs = ops.linear_acc(x, d(wg8), rd)
    accu, _ = ops.linear_acc(x, d(wu8), rd)
    g = ops.dequant(accg, xs, d(sg))
    u = ops.dequant(accu, xs, d(su))
    qh, hs = ops.quantize_act_glu(g, u, rh)
    qh2, hs2 = ops.dequant_act_quantize(accg, accu, xs, d(sg), d(su), rh)
    assert torch.equal(qh, qh2) and torch.equal(hs, hs2)
    y_chain = ops.dequant(ops.int8_gemm(qh, d(wd8)), hs, d(sd))
    assert torch.equal(y.view(torch.int16), y_chain.view(torch.int16)), "fused FFN != unfused chain"
    y_r, mid = O.ffn(c["x"], wg8, sg, wu8, su, wd8, sd, rd, rh, keep=True)
    # Each stage against the oracle on the GPU's own inputs to that stage: x codes; g, u on rows whose x
    # codes and scale bits equal the oracle's; the hidden codes from the GPU's g, u; y from the GPU's codes.
    qx, xs_q = ops.quantize_act(x, rd)
    assert_int8_parity(qx.cpu().numpy(), mid["qx"], what="qx")
    same_x = np.all(qx.cpu().numpy() == mid["qx"], axis=1) & (xs_q.cpu().numpy() == mid["xs"])
    assert np.array_equal(bf16_np(g)[same_x], mid["g"][same_x])
    assert np.array_equal(bf16_np(u)[same_x], mid["u"][same_x])
    vh = O.rotate(O.silu_glu(bf16_np(g), bf16_np(u)), rh)
    qhr, hsr = O.quantize(vh)
    assert_scale_parity(hs.cpu().numpy(), hsr)
    with np.errstate(divide="ignore", invalid="ignore"):
        vs = np.where(hsr[:, None] > 0, vh / hsr[:, None], 0).astype(np.float32)
    assert_int8_parity(qh.cpu().numpy(), qhr, vs, what="qh")
    y_own = O.dequant(O.gemm_s8(qh.cpu().numpy(), wd8), hs.cpu().numpy(), sd)
    assert np.array_equal(bf16_np(y), y_own)
    same = same_x & np.all(qh.cpu().numpy() == mid["qh"], axis=1)
    assert_rows_explained(bf16_np(y), y_r, same)


@pytest.mark.parametrize("rot", [(32, 64, 1), (64, 32, 1), (2, 1024, 1), (16, 32, 4)])
def test_dequant_weight_any_descriptor(ops, rot):
    K = rot[0] * rot[1] * rot[2]
    c = I.backward_case(8, 300, K, seed=K + rot[0])
    w8, s = O.prepare_weight(c["w"], rot)
    w = ops.dequant_weight(d(w8), d(s), rot)
    assert_bf16_parity(bf16_np(w), O.dequant_weight(w8, s, rot))


# N >= 8192 takes the split contraction (two half-N GEMMs, int32 reduce-add), below it one GEMM.
@pytest.mark.parametrize("M,N,K,rot", [(130, 8192, 2048, (64, 32, 1)), (200, 2048, 2048, (32, 64, 1)),
                                       (64, 1024, 8192, (128, 64, 1)), (70, 1024, 512, (1, 1, 512))])
def test_linear_dx_int8_any_descriptor(ops, M, N, K, rot):
    c = I.backward_case(M, N, K, seed=M + N + K)
    w8, s = O.prepare_weight(c["w"], rot)
    dx = ops.linear_dx_int8(bf16_dev(c["dy"]), d(w8), d(s), rot)
    assert_bf16_parity(bf16_np(dx), O.linear_dx_int8(c["dy"], w8, s, rot))


@pytest.mark.parametrize("rot", [(64, 128, 1), (1, 1, 1024), (32, 16, 2)])
def test_activation_quantizers_any_descriptor(ops, rot):
    """quantize_act_glu against the oracle's fp32 SiLU-GLU + rotation + quantizer, and
    dequant_act_quantize (from int32 accumulators) equal to dequant + quantize_act_glu bit for bit."""
    H = rot[0] * rot[1] * rot[2]
    M = 50
    rng = np.random.default_rng(H + rot[0])
    accg = rng.integers(-2 ** 20, 2 ** 20, (M, H)).astype(np.int32)
    accu = rng.integers(-2 ** 20, 2 ** 20, (M, H)).astype(np.int32)
    xs = (rng.random(M) * 1e-4 + 1e-6).astype(np.float32)
    sg = (rng.random(H) * 1e-3 + 1e-5).astype(np.float32)
    su = (rng.random(H) * 1e-3 + 1e-5).astype(np.float32)
    g = ops.dequant(d(accg), d(xs), d(sg))
    u = ops.dequant(d(accu), d(xs), d(su))
    q1, h1 = ops.quantize_act_glu(g, u, rot)
    q2, h2 = ops.dequant_act_quantize(d(accg), d(accu), d(xs), d(sg), d(su), rot)
    assert torch.equal(q1, q2) and torch.equal(h1, h2)
    v = O.rotate(O.silu_glu(bf16_np(g), bf16_np(u)), rot)
    qr, sr = O.quantize(v)
    assert_scale_parity(h1.cpu().numpy(), sr)
    assert_int8_parity(q1.cpu().numpy(), qr, (v / np.where(sr > 0, sr, 1)[:, None]).astype(np.float32))


@pytest.mark.parametrize("rot", [(32, 64, 1), (64, 64, 1), (64, 128, 1), (128, 128, 1), (16, 16, 16), (1, 1, 4096),
                                 (8, 8, 16)])
def test_linear_routes_agree_across_token_counts(ops, rot):
    """Every token count from 1 to 17 -- the GEMVs with the rotation inside (square and generic), the codes
    GEMV and the GEMM -- gives linear == dequant(linear_acc) bit for bit, with bias, on one weight."""
    K = rot[0] * rot[1] * rot[2]
    N = 136
    c = I.linear_case(17, K, N, n_outliers=max(1, K // 100), outlier_scale=30.0, bias_std=0.01, seed=K + rot[0])
    w8, ws = O.prepare_weight(c["w"], rot)
    w8d, wsd, bias = d(w8), d(ws), bf16_dev(c["bias"])
    for M in (1, 2, 3, 4, 5, 8, 15, 16, 17):
        x = bf16_dev(c["x"][:M])
        y = ops.linear(x, w8d, wsd, bias, rot)
        acc, xs = ops.linear_acc(x, w8d, rot)
        y2 = ops.dequant(acc, xs, wsd, bias)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), (rot, M)


@pytest.mark.parametrize("M,N,K", [(1, 19456, 1024), (2, 14592, 1024), (4, 7296, 1024), (3, 7296, 2048)])
def test_codes_gemv_wide_stages(ops, M, N, K):
    """The codes GEMV with many weight rows per stage (up to 64 / MP, padded to a power of two: 64 at one
    token, 32 at two, 16 at four), on the identity descriptor that sends even one token through it: the same
    bits as dequant(linear_acc), with bias."""
    rot = (1, 1, K)
    c = I.linear_case(M, K, N, n_outliers=max(1, K // 100), outlier_scale=30.0, bias_std=0.01, seed=N + M)
    w8, ws = O.prepare_weight(c["w"], rot)
    x, bias = bf16_dev(c["x"]), bf16_dev(c["bias"])
    y = ops.linear(x, d(w8), d(ws), bias, rot)
    acc, xs = ops.linear_acc(x, d(w8), rot)
    y2 = ops.dequant(acc, xs, d(ws), bias)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
