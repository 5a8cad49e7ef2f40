"""GPU parity of the fused SwiGLU FFN: fused == unfused chain bit for bit, and both vs the oracle."""
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


# M <= 16 (while the codes fit in shared memory) runs the GEMV route, larger M the GEMMs.
FFN_CASES = [(200, 1024, 4096, (32, 32, 1), (64, 64, 1)), (16, 256, 1024, (16, 16, 1), (32, 32, 1)),
             (130, 256, 16384, (16, 16, 1), (128, 128, 1)), (1, 1024, 4096, (32, 32, 1), (64, 64, 1)),
             (5, 1024, 16384, (32, 32, 1), (128, 128, 1))]


@pytest.mark.parametrize("M,dm,H,rd,rh", FFN_CASES)
def test_ffn_fused_vs_chain_and_oracle(ops, M, dm, H, rd, rh):
    c = I.ffn_case(M, dm, H, seed=M + H)
    wg8, sg = O.prepare_weight(c["wg"], rd)
    wu8, su = O.prepare_weight(c["wu"], rd)
    wd8, sd = O.prepare_weight(c["wd"], rh)
    x = bf16_dev(c["x"])
    y = ops.ffn_fused(x, d(wg8), d(sg), d(wu8), d(su), d(wd8), d(sd), rd, rh)
    # unfused chain through the public entry points
    accg, xs = ops.linear_acc(x, d(wg8), rd)
    accu, _ = ops.linear_acc(x, d(wu8), rd)
    g = ops.dequant(accg, xs, d(sg))
    u = ops.dequant(accu, xs, d(su))
    qh, hs = ops.quantize_act_glu(g, u, rh)
    qh2, hs2 = ops.dequant_act_quantize(accg, accu, xs, d(sg), d(su), rh)
    assert torch.equal(qh, qh2) and torch.equal(hs, hs2)
    accd = ops.int8_gemm(qh, d(wd8))
    y_chain = ops.dequant(accd, hs, d(sd))
    assert torch.equal(y.view(torch.int16), y_chain.view(torch.int16)), "fused FFN != unfused chain"
    # oracle
    y_r, mid = O.ffn(c["x"], wg8, sg, wu8, su, wd8, sd, rd, rh, keep=True)
    qx, _ = ops.quantize_act(x, rd)
    same_x = np.all(qx.cpu().numpy() == mid["qx"], axis=1)
    # identical x codes -> identical accumulators and epilogue arithmetic -> identical g, u bits
    assert np.array_equal(bf16_np(g)[same_x], mid["g"][same_x])
    assert np.array_equal(bf16_np(u)[same_x], mid["u"][same_x])
    assert_int8_parity(qh.cpu().numpy()[same_x], mid["qh"][same_x], what="qh")
    same = same_x & np.all(qh.cpu().numpy() == mid["qh"], axis=1)
    assert_rows_explained(bf16_np(y), y_r, same)
