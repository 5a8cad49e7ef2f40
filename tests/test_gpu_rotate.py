"""GPU parity of the rotate(+quantize) kernels against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I
from parity import (assert_bf16_parity, assert_int8_parity, assert_scale_parity, bf16_dev, bf16_np)

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


ROTS = [(16, 16, 1), (32, 32, 1), (64, 64, 1), (128, 128, 1), (16, 16, 12), (64, 64, 2), (1, 1, 4096)]


@pytest.mark.parametrize("rot", ROTS)
@pytest.mark.parametrize("M", [1, 7, 130])
def test_quantize_act(ops, rot, M):
    K = rot[0] * rot[1] * rot[2]
    xb = _x(M, K, seed=M * 7 + K, outliers=max(1, K // 100))
    q, s = ops.quantize_act(bf16_dev(xb), rot)
    torch.cuda.synchronize()
    qr, sr, vs = _oracle_q(xb, rot)
    assert_scale_parity(s.cpu().numpy(), sr)
    assert_int8_parity(q.cpu().numpy(), qr, vs)


@pytest.mark.parametrize("rot", [(16, 16, 1), (64, 64, 1), (128, 128, 1)])
def test_one_hot_closed_form(ops, rot):
    K = rot[0] * rot[1]
    ks = [0, 1, K // 3, K - 1]
    x = np.zeros((len(ks), K), np.float32)
    for r, k in enumerate(ks):
        x[r, k] = 1.0
    q, s = ops.quantize_act(bf16_dev(I.bf16_bits(x)), rot)
    inv = np.float32(1.0 / np.sqrt(K))
    assert np.all(s.cpu().numpy() == np.float32(inv / np.float32(127)))
    H = O.rotation_matrix(rot)
    qn = q.cpu().numpy().astype(np.int64)
    for r, k in enumerate(ks):
        assert np.array_equal(qn[r], (127 * np.sign(H[:, k])).astype(np.int64))


@pytest.mark.parametrize("rot", [(16, 16, 1), (64, 64, 1), (128, 128, 1), (16, 16, 3)])
def test_prepare_weight(ops, rot):
    K = rot[0] * rot[1] * rot[2]
    wb = I.bf16_bits(np.random.default_rng(3).standard_normal((200, K), dtype=np.float32) * np.float32(0.02))
    w8, s = ops.prepare_weight(bf16_dev(wb), rot)
    qr, sr, vs = _oracle_q(wb, rot)
    assert_scale_parity(s.cpu().numpy(), sr)
    assert_int8_parity(w8.cpu().numpy(), qr, vs)


@pytest.mark.parametrize("rot", [(16, 16, 1), (32, 32, 1), (64, 64, 1), (128, 128, 1), (16, 16, 5)])
def test_rotate_bf16(ops, rot):
    K = rot[0] * rot[1] * rot[2]
    xb = _x(33, K, seed=K)
    y = ops.rotate_bf16(bf16_dev(xb), rot)
    assert_bf16_parity(bf16_np(y), O.rotate_bf16(xb, rot))


@pytest.mark.parametrize("rot", [(16, 16, 1), (64, 64, 1), (128, 128, 1), (1, 1, 4096)])
def test_dequant_weight(ops, rot):
    K = rot[0] * rot[1] * rot[2]
    wb = I.bf16_bits(np.random.default_rng(4).standard_normal((150, K), dtype=np.float32) * np.float32(0.02))
    w8, s = O.prepare_weight(wb, rot)
    w = ops.dequant_weight(torch.from_numpy(w8).cuda(), torch.from_numpy(s).cuda(), rot)
    assert_bf16_parity(bf16_np(w), O.dequant_weight(w8, s, rot))


@pytest.mark.parametrize("rot", [(16, 16, 1), (64, 64, 1), (128, 128, 1)])
def test_quantize_act_glu(ops, rot):
    H = rot[0] * rot[1]
    rng = np.random.default_rng(5)
    g = I.bf16_bits(rng.standard_normal((70, H), dtype=np.float32) * np.float32(3))
    u = I.bf16_bits(rng.standard_normal((70, H), dtype=np.float32))
    q, s = ops.quantize_act_glu(bf16_dev(g), bf16_dev(u), rot)
    v = O.rotate(O.silu_glu(g, u), rot)
    qr, sr = O.quantize(v)
    assert_scale_parity(s.cpu().numpy(), sr)
    assert_int8_parity(q.cpu().numpy(), qr, (v / sr[:, None]).astype(np.float32))


@pytest.mark.parametrize("rot", [(16, 16, 1), (64, 64, 1)])
def test_dequant_act_quantize_matches_chain(ops, rot):
    """dequant_act_quantize == dequant -> quantize_act_glu, bit for bit ("Use from Python")."""
    H = rot[0] * rot[1]
    rng = np.random.default_rng(6)
    M = 40
    acc_g = rng.integers(-200000, 200000, (M, H)).astype(np.int32)
    acc_u = rng.integers(-200000, 200000, (M, H)).astype(np.int32)
    xs = (rng.random(M) * 1e-4 + 1e-5).astype(np.float32)
    sg = (rng.random(H) * 1e-4 + 1e-5).astype(np.float32)
    su = (rng.random(H) * 1e-4 + 1e-5).astype(np.float32)
    d = lambda a: torch.from_numpy(a).cuda()
    q, s = ops.dequant_act_quantize(d(acc_g), d(acc_u), d(xs), d(sg), d(su), rot)
    g = ops.dequant(d(acc_g), d(xs), d(sg))
    u = ops.dequant(d(acc_u), d(xs), d(su))
    q2, s2 = ops.quantize_act_glu(g, u, rot)
    assert torch.equal(q, q2) and torch.equal(s, s2)
    # and the chain against the oracle
    gr = O.dequant(acc_g.astype(np.int64), xs, sg)
    ur = O.dequant(acc_u.astype(np.int64), xs, su)
    v = O.rotate(O.silu_glu(gr, ur), rot)
    qr, sr = O.quantize(v)
    assert_int8_parity(q.cpu().numpy(), qr, (v / sr[:, None]).astype(np.float32))


@pytest.mark.parametrize("rot,M", [((64, 64, 1), 3001), ((16, 16, 1), 2999), ((32, 32, 1), 2001),
                                   ((16, 16, 5), 1999), ((64, 64, 2), 1201)])
def test_quantize_act_many_rows(ops, rot, M):
    """Many rows per persistent team: every input stage is refilled several times and the
    last row unit is ragged."""
    K = rot[0] * rot[1] * rot[2]
    xb = _x(M, K, seed=M + K, outliers=max(1, K // 100))
    q, s = ops.quantize_act(bf16_dev(xb), rot)
    torch.cuda.synchronize()
    qr, sr, vs = _oracle_q(xb, rot)
    assert_scale_parity(s.cpu().numpy(), sr)
    assert_int8_parity(q.cpu().numpy(), qr, vs)


def test_quantize_act_glu_many_rows(ops):
    rot, M = (128, 128, 1), 1500
    H = rot[0] * rot[1]
    rng = np.random.default_rng(15)
    g = I.bf16_bits(rng.standard_normal((M, H), dtype=np.float32) * np.float32(3))
    u = I.bf16_bits(rng.standard_normal((M, H), dtype=np.float32))
    q, s = ops.quantize_act_glu(bf16_dev(g), bf16_dev(u), rot)
    v = O.rotate(O.silu_glu(g, u), rot)
    qr, sr = O.quantize(v)
    assert_scale_parity(s.cpu().numpy(), sr)
    assert_int8_parity(q.cpu().numpy(), qr, (v / sr[:, None]).astype(np.float32))


@pytest.mark.parametrize("rot,N", [((64, 64, 1), 2500), ((32, 32, 1), 1999)])
def test_dequant_weight_many_rows(ops, rot, N):
    K = rot[0] * rot[1] * rot[2]
    wb = I.bf16_bits(np.random.default_rng(14).standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
    w8, s = O.prepare_weight(wb, rot)
    w = ops.dequant_weight(torch.from_numpy(w8).cuda(), torch.from_numpy(s).cuda(), rot)
    assert_bf16_parity(bf16_np(w), O.dequant_weight(w8, s, rot))


@pytest.mark.parametrize("rot,N", [((64, 64, 1), 1), ((64, 64, 1), 3041), ((64, 64, 3), 77)])
def test_dequant_weight_power_of_two_scales_exact(ops, rot, N):
    """With power-of-two row scales, (W8 s) R is exact in fp64 and in the integer transform, so the
    bf16 result is the one rounding of the same exact value on both sides: identical bits."""
    K = rot[0] * rot[1] * rot[2]
    rng = np.random.default_rng(N + K)
    w8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
    w8[0, :7] = 127
    s = np.ldexp(np.float32(1.0), rng.integers(-14, -4, N)).astype(np.float32)
    w = ops.dequant_weight(torch.from_numpy(w8).cuda(), torch.from_numpy(s).cuda(), rot)
    assert np.array_equal(bf16_np(w), O.dequant_weight(w8, s, rot))


@pytest.mark.parametrize("rot", [(64, 64, 2), (64, 64, 5)])
def test_dequant_weight_grouped(ops, rot):
    K = rot[0] * rot[1] * rot[2]
    wb = I.bf16_bits(np.random.default_rng(K).standard_normal((61, K), dtype=np.float32) * np.float32(0.02))
    w8, s = O.prepare_weight(wb, rot)
    w = ops.dequant_weight(torch.from_numpy(w8).cuda(), torch.from_numpy(s).cuda(), rot)
    assert_bf16_parity(bf16_np(w), O.dequant_weight(w8, s, rot))


@pytest.mark.parametrize("K,M", [(16384, 1000), (10000, 157), (8200, 3)])
def test_quantize_act_identity_long_rows_exact(ops, K, M):
    """R = I on long rows (one CTA of 256 or 512 threads per row, the row held in registers): the values
    are the bf16 inputs themselves, so scales and codes equal the oracle's exactly, including a zero row
    and a row of tiny values."""
    xb = _x(M, K, seed=M + K, outliers=max(1, K // 100))
    xb[0] = 0
    if M > 2:
        xb[2] = I.bf16_bits(np.full(K, 1e-30, np.float32) * np.sign(np.random.default_rng(K).standard_normal(K)))
    q, s = ops.quantize_act(bf16_dev(xb), (1, 1, K))
    qr, sr, _ = _oracle_q(xb, (1, 1, K))
    assert np.array_equal(s.cpu().numpy(), sr)
    assert np.array_equal(q.cpu().numpy(), qr)
