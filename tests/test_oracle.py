"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources: the PyPI page "xpu-kernels 0.2.0" (printed H4 and the 256-group index
map of "Algorithm: fused ConvRot rotation"; error budgets of "Verification" and
"The backward: dL/dx, weight-only"), closed forms (one-hot inputs, orthogonality,
round-half-even ties) and library routines (numpy matmul, torch bf16 casts).
"""
import os

import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(t) for t in line.split()])
    return np.array(rows, dtype=np.int64)


H4P = _load_table("h4_printed.txt")


def _digit_hadamard(n_digits):
    """H4^(x)n built entry by entry from base-4 digits and the printed H4."""
    n = 4 ** n_digits
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    H = np.ones((n, n), np.int64)
    for d in range(n_digits):
        H *= H4P[(i >> (2 * d)) & 3, (j >> (2 * d)) & 3]
    return H


def _ulp_diff_f32(a, b):
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(a - b)


# ------------------------------------------------------------------ rotation
def test_h4_is_the_printed_matrix():
    assert np.array_equal(O.hadamard(4), H4P)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_factors_orthogonal_symmetric(n):
    H = O.hadamard(n).astype(np.int64)
    assert set(np.unique(H)) <= {-1, 1}
    assert np.array_equal(H, H.T)
    assert np.array_equal(H @ H.T, n * np.eye(n, dtype=np.int64))


def test_group256_matches_page_index_map():
    # The fixture's digit columns must follow the page's formulas ...
    t = _load_table("index_map_256.txt")
    i, w, q = t[:, 0], t[:, 1], t[:, 2]
    assert np.array_equal(i, 16 * w + q)
    assert np.array_equal(t[:, 3], q & 3)
    assert np.array_equal(t[:, 4], (q >> 2) & 3)
    assert np.array_equal(t[:, 5], w & 3)
    assert np.array_equal(t[:, 6], w >> 2)
    # ... and the 256-point transform is the product of one printed H4 per digit.
    idx = np.arange(256)
    w_, q_ = idx >> 4, idx & 15
    dig = np.stack([q_ & 3, (q_ >> 2) & 3, w_ & 3, w_ >> 2])  # [4, 256]
    H = np.ones((256, 256), np.int64)
    for d in range(4):
        H *= H4P[dig[d][:, None], dig[d][None, :]]
    R = O.rotation_matrix((16, 16, 1))
    assert np.array_equal(R * 16.0, H.astype(np.float64))
    # (H4/2)^4 = 1/16 = 1/sqrt(256): every entry of R is +-1/16.
    assert np.all(np.abs(R) == 1.0 / 16.0)


def test_h128_reading_h2_on_top_bit():
    H64 = _digit_hadamard(3)
    H2 = np.array([[1, 1], [1, -1]])
    i = np.arange(128)[:, None]
    j = np.arange(128)[None, :]
    expected = H2[i >> 6, j >> 6] * H64[i & 63, j & 63]
    assert np.array_equal(O.hadamard(128).astype(np.int64), expected)
    assert np.array_equal(O.hadamard(64).astype(np.int64), H64)


@pytest.mark.parametrize("rot", [(16, 16, 1), (64, 64, 1), (4, 16, 1), (16, 16, 3), (1, 1, 1)])
def test_rotation_orthonormal_exact(rot):
    R = O.rotation_matrix(rot)
    assert np.array_equal(R, R.T)
    assert np.array_equal(R @ R.T, np.eye(R.shape[0]))


def test_rotation_orthonormal_non_power_of_four():
    R = O.rotation_matrix((2, 4, 1))
    np.testing.assert_allclose(R @ R.T, np.eye(8), atol=1e-15)


@pytest.mark.parametrize("rot", [(1, 4, 1), (4, 4, 1), (16, 16, 1), (16, 32, 1), (2, 8, 1),
                                 (64, 64, 1), (16, 16, 4), (8, 128, 1)])
def test_rotate_matches_explicit_kronecker(rot):
    a, b, g = rot
    K = a * b * g
    rng = np.random.default_rng(1)
    x = I.bf16_to_float(I.bf16_bits(rng.standard_normal((5, K), dtype=np.float32)))
    x[1, :] *= 100.0
    x[2, ::7] *= 30.0
    v = O.rotate(x, rot)
    ref = (O.rotation_matrix(rot) @ x.astype(np.float64).T).T.astype(np.float32)
    assert _ulp_diff_f32(v, ref).max() <= 1


def _digit_hadamard_any(n):
    """H_n for a power of two n: the printed H4 on every base-4 digit, and an unnormalised H2 on the most
    significant index bit when log2 n is odd (the reading of the H128 case taken for every odd size)."""
    logn = int(np.log2(n))
    H = _digit_hadamard(logn // 2)
    if logn % 2:
        H = np.kron(np.array([[1, 1], [1, -1]], np.int64), H)  # the first factor sits on the top bit
    return H


@pytest.mark.parametrize("rot", [(32, 64, 1), (64, 128, 1), (16, 32, 1), (2, 8, 1), (128, 64, 1)])
def test_one_hot_rotates_to_pm_inv_sqrt_k_non_square(rot):
    """a != b, including an odd total log2 (1 / sqrt(K) irrational): a one-hot row rotates to
    fl32(+-1 / sqrt(K)) in the sign pattern of column k of H_a (x) H_b, built here from base-4 digits."""
    a, b, _ = rot
    K = a * b
    Hfull = np.kron(_digit_hadamard_any(a), _digit_hadamard_any(b))
    inv = np.float32(1.0 / np.sqrt(np.float64(K)))
    for k in (0, 1, K // 3, K - 1):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        v = O.rotate(x, rot)
        assert np.all(np.abs(v) == inv)
        assert np.array_equal(np.sign(v[0]).astype(np.int64), Hfull[:, k])


@pytest.mark.parametrize("rot", [(16, 16, 3), (8, 8, 16), (32, 64, 2), (2, 32, 5)])
def test_grouped_rotation_acts_on_each_group_alone(rot):
    """groups = G is the block-diagonal I_G (x) R: each a*b-long group of a row is rotated by itself, as a
    row of its own would be (the page's groupsize), and the quantizer then takes one scale over the row."""
    a, b, g = rot
    n = a * b
    rng = np.random.default_rng(3)
    x = I.bf16_to_float(I.bf16_bits(rng.standard_normal((3, n * g), dtype=np.float32)))
    x[:, :n] *= 50.0  # groups of very different magnitude
    v = O.rotate(x, rot)
    for k in range(g):
        assert np.array_equal(v[:, k * n:(k + 1) * n], O.rotate(np.ascontiguousarray(x[:, k * n:(k + 1) * n]),
                                                                 (a, b, 1)))
    q, s = O.quantize(v)
    assert np.array_equal(s, (np.abs(v).max(axis=1) / np.float32(127.0)).astype(np.float32))


@pytest.mark.parametrize("rot", [(16, 16, 1), (64, 64, 1), (128, 128, 1)])
def test_one_hot_rotates_to_pm_inv_sqrt_k(rot):
    a, b, _ = rot
    K = a * b
    Ha = _digit_hadamard(int(np.log2(a)) // 2) if a in (16, 64) else \
        np.array([[1, 1], [1, -1]])[np.arange(a)[:, None] >> 6, np.arange(a)[None, :] >> 6] * \
        _digit_hadamard(3)[np.arange(a)[:, None] & 63, np.arange(a)[None, :] & 63]
    Hfull = np.kron(Ha, Ha)
    for k in (0, 1, K // 3, K - 1):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        v = O.rotate(x, rot)
        inv = np.float32(1.0 / np.sqrt(K))
        assert np.all(np.abs(v) == inv)
        assert np.array_equal(np.sign(v[0]).astype(np.int64), Hfull[:, k])
        q, s = O.quantize(v)
        assert s[0] == np.float32(inv / np.float32(127.0))
        assert np.array_equal(q[0].astype(np.int64), 127 * Hfull[:, k])


# ------------------------------------------------------------------ quantizer
def test_quantize_round_half_even_and_edges():
    v = np.array([[127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -127.0, 126.5, 0.49999997]], np.float32)
    q, s = O.quantize(v)
    assert s[0] == 1.0
    assert q[0].tolist() == [127, 2, 4, -2, 0, 0, 2, -127, 126, 0]
    v2 = np.array([[254.0, 3.0, 5.0, 7.0, -5.0]], np.float32)  # s = 2: 1.5, 2.5, 3.5, -2.5
    q2, s2 = O.quantize(v2)
    assert s2[0] == 2.0 and q2[0].tolist() == [127, 2, 2, 4, -2]
    z, sz = O.quantize(np.zeros((2, 64), np.float32))
    assert np.all(z == 0) and np.all(sz == 0)
    tiny = np.zeros((1, 8), np.float32)
    tiny[0, 3] = np.float32(1e-44)  # amax/127 underflows to 0 -> s = 0, q = 0
    qt, st = O.quantize(tiny)
    assert st[0] == 0 and np.all(qt == 0)


def test_quantize_error_bound_and_range():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 1024)).astype(np.float32)
    v[:, ::50] *= 25.0
    q, s = O.quantize(v)
    assert np.all(np.abs(q.astype(np.int64)).max(axis=1) == 127)
    assert q.min() >= -127
    err = np.abs(v.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-5))
    amax = np.abs(v).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(127.0)).astype(np.float32))


def test_quantize_sign_symmetry():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((16, 512)).astype(np.float32)
    q, s = O.quantize(v)
    qn, sn = O.quantize(-v)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)


# ------------------------------------------------------------------ GEMM / epilogue
def test_gemm_matches_numpy_int64():
    rng = np.random.default_rng(4)
    q = rng.integers(-127, 128, (9, 300), dtype=np.int64).astype(np.int8)
    w = rng.integers(-127, 128, (37, 300), dtype=np.int64).astype(np.int8)
    acc = O.gemm_s8(q, w)
    assert np.array_equal(acc, q.astype(np.int64) @ w.astype(np.int64).T)


def test_gemm_extremes_fit_int32():
    K = 16384
    q = np.full((2, K), 127, np.int8)
    w = np.full((3, K), -127, np.int8)
    acc = O.gemm_s8(q, w)
    assert np.all(acc == -127 * 127 * K)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    f = rng.standard_normal(4096).astype(np.float32) * np.float32(1e3)
    ties = (np.arange(1, 64, dtype=np.uint32) << 16 | 0x8000).view(np.float32) * 1.0
    f = np.concatenate([f, ties, -ties, np.array([0.0, -0.0, 1e-40, 3.4e38], np.float32)])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16(f), want)
    assert np.array_equal(I.bf16_bits(f), want)
    assert np.array_equal(O.bf16_to_f32(want), torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_dequant_hand_values():
    acc = np.array([[0, 3, 2 ** 24 + 1, -5]], np.int64)
    xs = np.array([0.5], np.float32)
    ws = np.array([1.0, 4.0, 2.0, 0.25], np.float32)
    bias = I.bf16_bits(np.array([0.125, 0.25, 0.0, -1.0], np.float32))
    y = O.bf16_to_f32(O.dequant(acc, xs, ws, bias))[0]
    # 0*.5*1+.125 ; 3*.5*4+.25 ; fp32(2^24+1)=2^24 (nearest even) -> 2^24 ; -5*.5*.25-1
    assert y.tolist() == [0.125, 6.25, float(2 ** 24), -1.625]
    y0 = O.dequant(np.zeros((2, 4), np.int64), np.ones(2, np.float32), ws, None)
    assert np.all(y0 == 0)


def test_dequant_within_one_bf16_ulp_of_exact():
    rng = np.random.default_rng(6)
    acc = rng.integers(-2 ** 26, 2 ** 26, (32, 64))
    xs = (rng.random(32) * 1e-3 + 1e-5).astype(np.float32)
    ws = (rng.random(64) * 1e-3 + 1e-5).astype(np.float32)
    bias = I.bf16_bits(rng.standard_normal(64).astype(np.float32) * 0.01)
    y = O.bf16_to_f32(O.dequant(acc, xs, ws, bias)).astype(np.float64)
    exact = acc * xs[:, None].astype(np.float64) * ws[None, :] + I.bf16_to_float(bias)[None, :]
    assert np.all(np.abs(y - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-30)


def test_linear_accuracy_vs_fp64():
    """End-to-end error budget ("Verification": about 0.9% relative L2 vs fp64)."""
    c = I.config_case("tiny_linear")
    rot = c["config"]["rot"]
    w8, ws = O.prepare_weight(c["w"], rot)
    y = O.bf16_to_f32(O.linear(c["x"], w8, ws, c["bias"], rot)).astype(np.float64)
    x = I.bf16_to_float(c["x"]).astype(np.float64)
    w = I.bf16_to_float(c["w"]).astype(np.float64)
    ref = x @ w.T + I.bf16_to_float(c["bias"])[None, :]
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert 0.002 < rel < 0.03, rel
    # dequant(linear_acc) == linear, bit for bit (page "Use from Python").
    acc, xs = O.linear_acc(c["x"], w8, rot)
    assert np.array_equal(O.dequant(acc, xs, ws, c["bias"]), O.linear(c["x"], w8, ws, c["bias"], rot))


def test_rotation_removes_outlier_damage():
    """Without a shared rotation the outlier channels blow up the per-token scale."""
    c = I.linear_case(32, 1024, 64, n_outliers=10, outlier_scale=30.0, seed=7)
    x = I.bf16_to_float(c["x"]).astype(np.float64)
    w = I.bf16_to_float(c["w"]).astype(np.float64)
    ref = x @ w.T
    errs = {}
    for rot in [(1, 1, 1024), (32, 32, 1)]:  # identity vs full-width rotation
        w8, ws = O.prepare_weight(c["w"], rot)
        y = O.bf16_to_f32(O.linear(c["x"], w8, ws, None, rot)).astype(np.float64)
        errs[rot] = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert errs[(32, 32, 1)] < 0.5 * errs[(1, 1, 1024)]


# ------------------------------------------------------------------ FFN
def test_silu_glu_vs_fp64():
    rng = np.random.default_rng(8)
    g = I.bf16_bits(rng.standard_normal(5000).astype(np.float32) * 4)
    u = I.bf16_bits(rng.standard_normal(5000).astype(np.float32))
    h = O.silu_glu(g, u).astype(np.float64)
    gf = I.bf16_to_float(g).astype(np.float64)
    uf = I.bf16_to_float(u).astype(np.float64)
    ref = gf / (1 + np.exp(-gf)) * uf
    assert np.all(np.abs(h - ref) <= np.abs(ref) * 4e-7 + 1e-38)
    assert O.silu_glu(I.bf16_bits(np.zeros(1, np.float32)), I.bf16_bits(np.ones(1, np.float32)))[0] == 0.0


def test_ffn_accuracy_vs_fp64():
    c = I.ffn_case(8, 256, 512, seed=9)
    rd, rh = (16, 16, 1), (16, 32, 1)
    wg8, sg = O.prepare_weight(c["wg"], rd)
    wu8, su = O.prepare_weight(c["wu"], rd)
    wd8, sd = O.prepare_weight(c["wd"], rh)
    y = O.bf16_to_f32(O.ffn(c["x"], wg8, sg, wu8, su, wd8, sd, rd, rh)).astype(np.float64)
    x = I.bf16_to_float(c["x"]).astype(np.float64)
    g = x @ I.bf16_to_float(c["wg"]).astype(np.float64).T
    u = x @ I.bf16_to_float(c["wu"]).astype(np.float64).T
    ref = (g / (1 + np.exp(-g)) * u) @ I.bf16_to_float(c["wd"]).astype(np.float64).T
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert 0.003 < rel < 0.06, rel


# ------------------------------------------------------------------ backward
def test_dequant_weight_recovers_w():
    """Page, "The backward": the recovered weight is ~0.9% off (0.90% int8 + 0.17% bf16)."""
    c = I.backward_case(4, 64, 4096, seed=10)
    rot = (64, 64, 1)
    w8, s = O.prepare_weight(c["w"], rot)
    what = O.bf16_to_f32(O.dequant_weight(w8, s, rot)).astype(np.float64)
    w = I.bf16_to_float(c["w"]).astype(np.float64)
    rel = np.linalg.norm(what - w) / np.linalg.norm(w)
    assert 0.007 < rel < 0.011, rel
    # Literal reading (identity rotation) leaves the weight in the rotated basis.
    lit = O.bf16_to_f32(O.dequant_weight(w8, s, (1, 1, 4096))).astype(np.float64)
    wr = (O.rotation_matrix(rot) @ w.T).T
    assert np.linalg.norm(lit - wr) / np.linalg.norm(wr) < 0.011


def test_dequant_weight_against_exact_integer_transform():
    """(W8 s) R has a closed form: s / 64 times the integer row W8 H (H = H64 (x) H64 built here from the
    printed H4 by digits; |W8 H| < 127 * 4096 < 2^24, so fp64 holds it exactly).  The oracle, which rounds
    W8 s to fp32 before its fp64 sum, lies within one bf16 unit of it plus the residue of those roundings
    (at most 64 * 127 * s * 2^-24), and equals bf16 of it exactly when s is a power of two."""
    g = np.random.default_rng(12)
    N, K, rot = 48, 4096, (64, 64, 1)
    w8 = g.integers(-127, 128, (N, K)).astype(np.int8)
    w8[0] = 0
    w8[1] = 127
    H = _digit_hadamard(6)
    v = w8.astype(np.int64) @ H
    for s in ((g.random(N) * 1e-3 + 1e-5).astype(np.float32),
              np.ldexp(np.float32(1), g.integers(-14, -4, N)).astype(np.float32)):
        exact = s[:, None].astype(np.float64) * v.astype(np.float64) / 64.0
        got = O.dequant_weight(w8, s, rot)
        o = O.bf16_to_f32(got).astype(np.float64)
        resid = 64.0 * 127.0 * s[:, None].astype(np.float64) * 2.0 ** -24
        mag = np.abs(exact) + resid
        ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 1e-38))) - 7)
        assert np.all(np.abs(o - exact) <= resid + ulp)
    assert np.array_equal(got, O.f32_to_bf16(exact.astype(np.float32)))  # power-of-two scales: exact


def test_linear_dx_matches_numpy():
    rng = np.random.default_rng(11)
    dy = I.bf16_bits(rng.standard_normal((8, 96)).astype(np.float32))
    w = I.bf16_bits(rng.standard_normal((96, 40)).astype(np.float32))
    dx = O.linear_dx(dy, w)
    ref = I.bf16_to_float(dy).astype(np.float64) @ I.bf16_to_float(w).astype(np.float64)
    want = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.mean(dx == want) > 0.99
    assert np.all(np.abs(O.bf16_to_f32(dx) - O.bf16_to_f32(want)) <= np.abs(O.bf16_to_f32(want)) * 2 ** -7 + 1e-30)


def test_linear_dx_int8_noise_vs_bf16_route():
    """Page, "The backward": the int8 dx route is noisier than the bf16 route (~40%)."""
    c = I.backward_case(64, 2048, 256, seed=12)
    rot = (16, 16, 1)
    w8, s = O.prepare_weight(c["w"], rot)
    dy = I.bf16_to_float(c["dy"]).astype(np.float64)
    ref = dy @ I.bf16_to_float(c["w"]).astype(np.float64)
    d16 = O.bf16_to_f32(O.linear_dx(c["dy"], O.dequant_weight(w8, s, rot))).astype(np.float64)
    d8 = O.bf16_to_f32(O.linear_dx_int8(c["dy"], w8, s, rot)).astype(np.float64)
    e16 = np.linalg.norm(d16 - ref) / np.linalg.norm(ref)
    e8 = np.linalg.norm(d8 - ref) / np.linalg.norm(ref)
    assert 0.004 < e16 < 0.02
    assert 1.05 * e16 < e8 < 3.0 * e16, (e16, e8)


def test_linear_dx_int8_exact_when_dy_is_on_the_grid():
    """With s = 1, dy' already on a per-row int grid and an identity rotation the route is exact."""
    rng = np.random.default_rng(13)
    qd = rng.integers(-127, 128, (6, 64))
    qd[:, 0] = 127
    step = np.float32(2.0 ** -7)
    dy = I.bf16_bits(qd.astype(np.float32) * step)
    w8 = rng.integers(-127, 128, (64, 16)).astype(np.int8)
    s = np.ones(64, np.float32)
    dx = O.bf16_to_f32(O.linear_dx_int8(dy, w8, s, (1, 1, 16))).astype(np.float64)
    exact = (qd @ w8.astype(np.int64)).astype(np.float64) * float(step)
    want = O.bf16_to_f32(O.f32_to_bf16(exact.astype(np.float32)))
    assert np.array_equal(dx, want)


# ------------------------------------------------------------------ rotate-only bf16 path
def test_linear_bf16_integer_brute_force():
    """Small-integer operands: the exact sum (Python integers, loop over k) rounded once to bf16.
    Non-square shapes, so a transposed operand or a dropped bias fails."""
    rng = np.random.default_rng(31)
    M, N, K = 3, 5, 64
    xi = rng.integers(-8, 9, (M, K))
    wi = rng.integers(-8, 9, (N, K))
    bi = rng.integers(-50, 51, N)
    xb = I.bf16_bits(xi.astype(np.float32))
    wb = I.bf16_bits(wi.astype(np.float32))
    bb = I.bf16_bits(bi.astype(np.float32))
    for bias in (None, bb):
        y = O.linear_bf16(xb, wb, bias)
        for m in range(M):
            for n in range(N):
                exact = sum(int(xi[m, k]) * int(wi[n, k]) for k in range(K)) + (0 if bias is None else int(bi[n]))
                assert y[m, n] == I.bf16_bits(np.array([exact], np.float32))[0], (m, n)


def test_linear_bf16_rotated_pair_is_the_unrotated_layer():
    """"Use from C": the BF16 path rotates the activation and multiplies by the pre-rotated weight;
    R orthogonal makes that the original layer up to the bf16 roundings of the rotated operands."""
    rng = np.random.default_rng(32)
    M, K, N, rot = 16, 256, 48, (16, 16, 1)
    x = I.bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = I.bf16_bits(rng.standard_normal((N, K)).astype(np.float32) * np.float32(0.02))
    b = I.bf16_bits(rng.standard_normal(N).astype(np.float32) * np.float32(0.01))
    y = O.bf16_to_f32(O.linear_bf16(O.rotate_bf16(x, rot), O.rotate_bf16(w, rot), b)).astype(np.float64)
    ref = (I.bf16_to_float(x).astype(np.float64) @ I.bf16_to_float(w).astype(np.float64).T
           + I.bf16_to_float(b).astype(np.float64))
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < 6e-3, rel
    # and the rotation is not the identity on this data: the rotated operands differ from the inputs
    assert not np.array_equal(O.rotate_bf16(x, rot), x)
