"""The hot-path calls captured in a CUDA graph and replayed give the eager results bit for bit
(decode GEMV, prefill linear with its quantizer-to-GEMM overlap, the fused FFN, dx_int8)."""
import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300 import inputs as I
from parity import bf16_dev

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


def _capture_and_compare(ops, calls):
    """calls: list of (fn(out), out tensor).  Eager run, then the same calls captured in one graph
    (first-launch set-up happened in the eager run) and replayed twice into fresh outputs."""
    eager = []
    for fn, out in calls:
        fn(out)
        eager.append(out.clone())
    torch.cuda.synchronize()
    for _, out in calls:
        out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for fn, out in calls:
            fn(out)
    for _ in range(2):
        for _, out in calls:
            out.zero_()
        g.replay()
        torch.cuda.synchronize()
        for (_, out), ref in zip(calls, eager):
            assert torch.equal(out.view(torch.int16) if out.dtype == torch.bfloat16 else out,
                               ref.view(torch.int16) if ref.dtype == torch.bfloat16 else ref)


def test_graph_decode_and_prefill(ops):
    rot = (64, 64, 1)
    rng = np.random.default_rng(77)
    w = I.bf16_bits(rng.standard_normal((1500, 4096)).astype(np.float32) * np.float32(0.02))
    w8, ws = O.prepare_weight(w, rot)
    w8d, wsd = d(w8), d(ws)
    bias = bf16_dev(I.bf16_bits(rng.standard_normal(1500).astype(np.float32) * np.float32(0.01)))
    x1 = bf16_dev(I.bf16_bits(rng.standard_normal((1, 4096)).astype(np.float32)))
    x2 = bf16_dev(I.bf16_bits(rng.standard_normal((300, 4096)).astype(np.float32)))
    ws1 = torch.empty(ops.workspace_size(ops.OP_LINEAR, 1, 1500, 4096), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(ops.workspace_size(ops.OP_LINEAR, 300, 1500, 4096), dtype=torch.uint8, device="cuda")
    y1 = torch.empty((1, 1500), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((300, 1500), dtype=torch.bfloat16, device="cuda")
    _capture_and_compare(ops, [
        (lambda out: ops.linear(x1, w8d, wsd, None, rot, ws1, out=out), y1),
        (lambda out: ops.linear(x2, w8d, wsd, bias, rot, ws2, out=out), y2),
    ])


@pytest.mark.parametrize("M", [1, 64])
def test_graph_ffn_and_dx_int8(ops, M):
    """The fused FFN (decode and prefill token counts) and dx_int8 against the down projection."""
    rd, rh = (32, 32, 1), (64, 64, 1)
    c = I.ffn_case(M, 1024, 4096, seed=78 + M)
    wg8, sg = O.prepare_weight(c["wg"], rd)
    wu8, su = O.prepare_weight(c["wu"], rd)
    wd8, sd = O.prepare_weight(c["wd"], rh)
    x = bf16_dev(c["x"])
    t = [d(a) for a in (wg8, sg, wu8, su, wd8, sd)]
    wsf = torch.empty(ops.workspace_size(ops.OP_FFN, M, 0, 1024, 4096), dtype=torch.uint8, device="cuda")
    yf = torch.empty((M, 1024), dtype=torch.bfloat16, device="cuda")
    # dy [130, d] against W_down [d, H] (rotated over H): dx [130, H]
    dy = bf16_dev(I.bf16_bits(np.random.default_rng(79).standard_normal((130, 1024)).astype(np.float32)
                              * np.float32(1e-3)))
    wsx = torch.empty(ops.workspace_size(ops.OP_LINEAR_DX_INT8, 130, 1024, 4096), dtype=torch.uint8,
                      device="cuda")
    dx = torch.empty((130, 4096), dtype=torch.bfloat16, device="cuda")
    _capture_and_compare(ops, [
        (lambda out: ops.ffn_fused(x, *t, rd, rh, wsf, out=out), yf),
        (lambda out: ops.linear_dx_int8(dy, t[4], t[5], rh, wsx, out=out), dx),
    ])


def test_linear_dx_int8_two_stream_split_graph(ops):
    """linear_dx_int8 over a long contraction (N = 8192: two GEMM halves on the library's second stream and
    the caller's, summed exactly into one accumulator) captured in a graph replays the eager bits, which
    match the oracle."""
    M, N, K, rot = 200, 8192, 1024, (32, 32, 1)
    c = I.backward_case(M, N, K, seed=81)
    w8, s = O.prepare_weight(c["w"], rot)
    dy, w8d, sd = bf16_dev(c["dy"]), d(w8), d(s)
    ws = torch.empty(ops.workspace_size(ops.OP_LINEAR_DX_INT8, M, N, K), dtype=torch.uint8, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    _capture_and_compare(ops, [(lambda out: ops.linear_dx_int8(dy, w8d, sd, rot, ws, out=out), dx)])
    from parity import assert_bf16_parity, bf16_np
    assert_bf16_parity(bf16_np(dx), O.linear_dx_int8(c["dy"], w8, s, rot))


# The last three run the rotation kernels + codes GEMV (programmatic dependent launch after the quantizer).
@pytest.mark.parametrize("M,K,rot", [(1, 4096, (64, 64, 1)), (3, 4096, (64, 64, 1)), (2, 1024, (32, 32, 1)),
                                     (8, 4096, (64, 64, 1)), (1, 2048, (32, 64, 1)), (4, 8192, (64, 64, 2))])
def test_decode_chain_back_to_back(ops, M, K, rot):
    """Stacked decode layers, each reading the previous layer's output as its x, launched back to
    back (the GEMV waits for the kernel before it while the next call's weight prefetch runs beside
    it) give the bits of the same calls with a device synchronisation after each, and of a graph
    replay of the chain."""
    L, NW = 12, 4
    ws_, w8s = [], []
    for k in range(NW):
        c = I.linear_case(M, K, K, n_outliers=I.outlier_count(K), outlier_scale=30.0, seed=100 + k)
        w8, s = ops.prepare_weight(bf16_dev(c["w"]), rot)
        w8s.append(w8)
        ws_.append(s)
    x0 = bf16_dev(I.linear_case(M, K, 8, n_outliers=I.outlier_count(K), outlier_scale=30.0, seed=7)["x"])
    work = torch.empty(max(ops.workspace_size(ops.OP_LINEAR, M, K, K), 256), dtype=torch.uint8, device="cuda")

    def run(sync):
        bufs = [x0] + [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        for i in range(L):
            ops.linear(bufs[i], w8s[i % NW], ws_[i % NW], None, rot, workspace=work, out=bufs[i + 1])
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return bufs

    ref = run(True)
    got = run(False)
    for i in range(1, L + 1):
        assert torch.equal(ref[i].view(torch.int16), got[i].view(torch.int16)), f"layer {i}"
    assert torch.isfinite(ref[L].float()).all()
    bufs = [x0] + [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(L):
            ops.linear(bufs[i], w8s[i % NW], ws_[i % NW], None, rot, workspace=work, out=bufs[i + 1])
    for _ in range(2):
        for b in bufs[1:]:
            b.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        for i in range(1, L + 1):
            assert torch.equal(ref[i].view(torch.int16), bufs[i].view(torch.int16)), f"graph layer {i}"
