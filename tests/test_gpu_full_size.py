"""GPU parity at the benchmark's full sizes, with its inputs and through the calls it times; the oracle
checks sampled rows (each output row depends only on its own token row and the whole weight).

  prefill linear  x [1024, 4096] (1% outlier channels x30), W [14336, 4096], bias, R = H64 (x) H64 / 64
  SwiGLU FFN      x [1024, 4096], W_gate / W_up [16384, 4096], W_down [4096, 16384], R_d = H64 (x) H64,
                  R_h = H128 (x) H128
  backward        dy [4096, 16384], W [16384, 4096]: dequant_weight, linear_dx, linear_dx_int8
"""
import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I
from parity import (assert_bf16_parity, assert_int8_parity, assert_rows_explained, assert_scale_parity, bf16_dev,
                    bf16_np)

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


def _rows(n, k, seed):
    r = np.random.default_rng(seed).choice(n, k, replace=False)
    r[0], r[1] = 0, n - 1
    return np.sort(r)


def test_prefill_full_size_sampled(ops):
    rot, M, K, N = (64, 64, 1), 1024, 4096, 14336
    c = I.linear_case(M, K, N, n_outliers=I.outlier_count(K), outlier_scale=30.0, bias_std=0.01, seed=0)
    w8_d, s_d = ops.prepare_weight(bf16_dev(c["w"]), rot)
    x = bf16_dev(c["x"])
    y = bf16_np(ops.linear(x, w8_d, s_d, bf16_dev(c["bias"]), rot))
    acc, xs = ops.linear_acc(x, w8_d, rot)
    q, _ = ops.quantize_act(x, rot)
    w8, s = w8_d.cpu().numpy(), s_d.cpu().numpy()
    # weight preparation on sampled weight rows
    wr = _rows(N, 64, 1)
    w8_r, s_r = O.prepare_weight(c["w"][wr], rot)
    assert_scale_parity(s[wr], s_r, what="w_scale")
    assert_int8_parity(w8[wr], w8_r, what="w8")
    # activation codes, exact accumulators on the GPU's own codes, the epilogue bit for bit
    rows = _rows(M, 12, 2)
    q_r, xs_r = O.rotate_quantize(c["x"][rows], rot)
    qg, xsg = q.cpu().numpy()[rows], xs.cpu().numpy()[rows]
    assert_scale_parity(xsg, xs_r, what="x_scale")
    assert_int8_parity(qg, q_r)
    acc_r = O.gemm_s8(qg, w8)
    assert np.array_equal(acc.cpu().numpy()[rows].astype(np.int64), acc_r)
    assert np.array_equal(y[rows], O.dequant(acc_r, xsg, s, c["bias"]))
    # and the whole chain from x against the oracle's
    same = np.all(qg == q_r, axis=1)
    assert_rows_explained(y[rows], O.linear(c["x"][rows], w8, s, c["bias"], rot), same)
    # the few-token routes on this weight (ring GEMV with the rotation inside for one or two tokens, the
    # rotation kernel + codes GEMV up to 16): per row the same codes, sums and epilogue as the GEMM route
    for m in (1, 2, 7, 16):
        ym = bf16_np(ops.linear(x[:m], w8_d, s_d, bf16_dev(c["bias"]), rot))
        assert np.array_equal(ym.view(np.uint16), y[:m].view(np.uint16)), f"{m}-token route != GEMM route"


def test_ffn_full_size_sampled(ops):
    M, dm, H, rd, rh = 1024, 4096, 16384, (64, 64, 1), (128, 128, 1)
    c = I.ffn_case(M, dm, H, seed=0)
    wg8, sg = ops.prepare_weight(bf16_dev(c["wg"]), rd)
    wu8, su = ops.prepare_weight(bf16_dev(c["wu"]), rd)
    wd8, sd = ops.prepare_weight(bf16_dev(c["wd"]), rh)
    x = bf16_dev(c["x"])
    y = ops.ffn_fused(x, wg8, sg, wu8, su, wd8, sd, rd, rh)
    # the fused call equals the unfused chain of public calls, bit for bit, at full size
    accg, xs = ops.linear_acc(x, wg8, rd)
    accu, _ = ops.linear_acc(x, wu8, rd)
    qh, hs = ops.dequant_act_quantize(accg, accu, xs, sg, su, rh)
    y_chain = ops.dequant(ops.int8_gemm(qh, wd8), hs, sd)
    assert torch.equal(y.view(torch.int16), y_chain.view(torch.int16)), "fused FFN != unfused chain"
    del accu, y_chain
    # sampled rows against the oracle's chain
    rows = _rows(M, 8, 3)
    n = lambda t: t.cpu().numpy()
    y_r, mid = O.ffn(c["x"][rows], n(wg8), n(sg), n(wu8), n(su), n(wd8), n(sd), rd, rh, keep=True)
    qx, _ = ops.quantize_act(x, rd)
    qx = n(qx)[rows]
    assert_int8_parity(qx, mid["qx"], what="qx")
    same_x = np.all(qx == mid["qx"], axis=1)
    assert np.array_equal(n(accg)[rows][same_x].astype(np.int64), O.gemm_s8(mid["qx"][same_x], n(wg8)))
    qh = n(qh)[rows]
    assert_int8_parity(qh[same_x], mid["qh"][same_x], what="qh")
    same = same_x & np.all(qh == mid["qh"], axis=1)
    assert_rows_explained(bf16_np(y)[rows], y_r, same)
    # the few-token route (int8 codes, gate|up GEMV over [W_gate; W_up], hidden codes, down GEMV) at the
    # same sizes: per row the same codes, sums and epilogues, so the rows of the GEMM route's output
    for m in (1, 2, 5):
        ym = ops.ffn_fused(x[:m], wg8, sg, wu8, su, wd8, sd, rd, rh)
        assert torch.equal(ym.view(torch.int16), y[:m].view(torch.int16)), f"{m}-token FFN != GEMM route"


def test_backward_full_size_sampled(ops):
    M, N, K, rot = 4096, 16384, 4096, (64, 64, 1)
    c = I.backward_case(M, N, K, seed=0)
    w8_d, s_d = ops.prepare_weight(bf16_dev(c["w"]), rot)
    dy = bf16_dev(c["dy"])
    w8, s = w8_d.cpu().numpy(), s_d.cpu().numpy()
    what = ops.dequant_weight(w8_d, s_d, rot)
    wr = _rows(N, 64, 4)
    assert_bf16_parity(bf16_np(what)[wr], O.dequant_weight(w8[wr], s[wr], rot), what="W_hat")
    rows = _rows(M, 8, 5)
    dx = ops.linear_dx(dy, what)
    assert_bf16_parity(bf16_np(dx)[rows], O.linear_dx(c["dy"][rows], bf16_np(what)), what="dx", acc_len=N)
    dx8 = ops.linear_dx_int8(dy, w8_d, s_d, rot)
    assert_bf16_parity(bf16_np(dx8)[rows], O.linear_dx_int8(c["dy"][rows], w8, s, rot), what="dx_int8")
