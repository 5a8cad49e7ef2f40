"""Self-test on this machine: `python -m ffn_rotate_quantize_gb300`.

The page's package ships the same kind of command ("Use from Python": a self-test of the library and of every
kernel gate on the machine at hand). This one loads libgbq.so, reports the device and runs every entry point
once on a small case, checking a property that holds without any reference implementation:

  * closed forms: a one-hot row rotates to +-1/sqrt(K) in the sign pattern of the Hadamard column, so its
    codes are +-127 and its scale fl(fl(1/sqrt K)/127) (n = 16, 64 and 128 factors);
  * exactness: the int8 contraction equals an int64 matrix product; the identity-rotation dequant_weight
    equals one fp32 multiply rounded to bf16;
  * bit identities between routes: linear == dequant(linear_acc) (the GEMM, the decode GEMV and the codes
    GEMV), linear_noalloc == linear, the fused FFN (GEMV and GEMM routes) == its chain of public calls;
  * loose bounds: R R = I through the rotate-only path, dequant_weight(prepare_weight(W)) within 2% of W,
    linear_dx against an fp32 product, the int8 dx route within 5% of the bf16 one;
  * a clean device status word afterwards.

A check that cannot run (no GPU) is reported SKIPPED and never counts as passed. Exit status: 0 when every
check ran and passed, 1 when one failed, 2 when a check was skipped.
"""
import sys
import traceback

import numpy as np
import torch


def hadamard_sign(n: int, p: np.ndarray, q: int) -> np.ndarray:
    """Sign of H_n[p, q] for n = 4^j (H4^(x)j) or n = 2 * 4^j (H2 (x) H4^(x)j, H2 on the top index bit).

    H4 = J - 2 * antidiag, so H4[u, v] = -1 exactly when u + v == 3; H2[u, v] = -1 when u == v == 1; a
    Kronecker product multiplies the factors' entries digit by digit."""
    j = (n.bit_length() - 1) // 2
    sign = np.ones_like(p)
    for d in range(j):
        u, v = (p >> (2 * d)) & 3, (q >> (2 * d)) & 3
        sign = np.where(u + v == 3, -sign, sign)
    if n != 4 ** j:  # the H2 factor on bit 2j
        sign = np.where(((p >> (2 * j)) & 1) & ((q >> (2 * j)) & 1) == 1, -sign, sign)
    return sign


def rotation_sign(a: int, b: int, i: np.ndarray, k: int) -> np.ndarray:
    """Sign of (H_a (x) H_b)[i, k] with the index convention (A (x) B)[i b + i', k b + k'] = A[i, k] B[i', k']."""
    return hadamard_sign(a, i // b, k // b) * hadamard_sign(b, i % b, k % b)


def _bf16(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(torch.bfloat16)


def _rel(a: torch.Tensor, r: torch.Tensor) -> float:
    a, r = a.double(), r.double()
    return float(torch.linalg.vector_norm(a - r) / torch.linalg.vector_norm(r))


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def check_onehot(G, dev):
    out = []
    for rot in [(16, 16, 1), (64, 64, 1), (128, 128, 1)]:
        a, b, _ = rot
        K = a * b
        ks = np.array([0, 1, K // 3, K - 1])
        x = np.zeros((len(ks), K), np.float32)
        x[np.arange(len(ks)), ks] = 1.0
        q, s = G.quantize_act(_bf16(x, dev), rot)
        q, s = q.cpu().numpy(), s.cpu().numpy()
        s_ref = np.float32(np.float32(1.0 / np.sqrt(K)) / np.float32(127.0))
        i = np.arange(K)
        for r, k in enumerate(ks):
            if s[r] != s_ref or not np.array_equal(q[r].astype(np.int64), 127 * rotation_sign(a, b, i, int(k))):
                return False, f"K={K} one-hot column {k}: scale {s[r]!r} (expected {s_ref!r}) or codes differ"
        out.append(f"K={K}")
    return True, "codes +-127 in the Hadamard sign pattern, exact scales: " + ", ".join(out)


def check_int8_gemm(G, dev):
    g = np.random.default_rng(1)
    M, N, K = 130, 256, 1088
    q = g.integers(-127, 128, (M, K)).astype(np.int8)
    w = g.integers(-127, 128, (N, K)).astype(np.int8)
    q[0], w[0] = 127, 127  # one output at 127^2 K
    acc = G.int8_gemm(torch.from_numpy(q).to(dev), torch.from_numpy(w).to(dev)).cpu()
    ref = torch.from_numpy(q).long() @ torch.from_numpy(w).long().T
    return torch.equal(acc.long(), ref), f"{M}x{N}x{K} against an int64 product"


def _layer(G, dev, M, K, N, rot, seed):
    g = np.random.default_rng(seed)
    x = g.standard_normal((M, K)).astype(np.float32)
    x[:, g.choice(K, max(1, K // 100), replace=False)] *= 30.0  # outlier channels
    w = g.standard_normal((N, K)).astype(np.float32) * 0.02
    bias = g.standard_normal(N).astype(np.float32) * 0.01
    w8, s = G.prepare_weight(_bf16(w, dev), rot)
    return _bf16(x, dev), w8, s, _bf16(bias, dev)


def check_linear_routes(G, dev):
    # the GEMM route, the decode GEMV with the rotation inside, the codes GEMV (a small batch) and the GEMV
    # with the generic rotation inside (one token with a non-square descriptor)
    for M, K, rot in ((64, 4096, (64, 64, 1)), (1, 4096, (64, 64, 1)), (8, 4096, (64, 64, 1)),
                      (1, 2048, (32, 64, 1))):
        x, w8, s, bias = _layer(G, dev, M, K, 512, rot, seed=M + K)
        y = G.linear(x, w8, s, bias, rot)
        acc, xs = G.linear_acc(x, w8, rot)
        if not _same_bits(y, G.dequant(acc, xs, s, bias)):
            return False, f"M={M} {rot}: linear != dequant(linear_acc)"
        if not _same_bits(y, G.linear_noalloc(x, w8, s, bias, rot)):
            return False, f"M={M} {rot}: linear_noalloc != linear"
    return True, ("linear == dequant(linear_acc) == linear_noalloc, bit for bit: GEMM (M = 64), decode GEMV "
                  "(M = 1), codes GEMV (M = 8), GEMV with the generic rotation inside (M = 1 with 32 x 64)")


def check_ffn_chain(G, dev):
    d, H, rd, rh = 256, 1024, (16, 16, 1), (32, 32, 1)
    for M in (16, 64):  # the GEMV route (few tokens) and the GEMM route
        g = np.random.default_rng(3 + M)
        x = _bf16(g.standard_normal((M, d)), dev)
        wg8, sg = G.prepare_weight(_bf16(g.standard_normal((H, d)) * 0.02, dev), rd)
        wu8, su = G.prepare_weight(_bf16(g.standard_normal((H, d)) * 0.02, dev), rd)
        wd8, sd = G.prepare_weight(_bf16(g.standard_normal((d, H)) * 0.02, dev), rh)
        y = G.ffn_fused(x, wg8, sg, wu8, su, wd8, sd, rd, rh)
        accg, xs = G.linear_acc(x, wg8, rd)
        accu, _ = G.linear_acc(x, wu8, rd)
        qh, hs = G.dequant_act_quantize(accg, accu, xs, sg, su, rh)
        y_chain = G.dequant(G.int8_gemm(qh, wd8), hs, sd)
        if not _same_bits(y, y_chain):
            return False, f"M={M}: ffn_fused != chain of public calls"
    return True, f"ffn_fused == chain of public calls (GEMM-only), {d}x{H}, M = 16 (GEMVs) and 64 (GEMMs)"


def check_rotation_involution(G, dev):
    rot = (64, 64, 1)
    x = _bf16(np.random.default_rng(4).standard_normal((8, 4096)), dev)
    e = _rel(G.rotate_bf16(G.rotate_bf16(x, rot), rot), x)
    return e < 1e-2, f"|R R x - x| / |x| = {e:.2e} (two bf16 roundings)"


def check_dequant_weight(G, dev):
    g = np.random.default_rng(5)
    N, K = 96, 4096
    w8 = torch.from_numpy(g.integers(-127, 128, (N, K)).astype(np.int8)).to(dev)
    s = torch.from_numpy((g.random(N) * 1e-3 + 1e-4).astype(np.float32)).to(dev)
    if not _same_bits(G.dequant_weight(w8, s, (1, 1, K)), (w8.float() * s[:, None]).to(torch.bfloat16)):
        return False, "identity rotation: W8 * s differs from one fp32 multiply rounded to bf16"
    w = _bf16(g.standard_normal((N, K)) * 0.02, dev)
    rot = (64, 64, 1)
    e = _rel(G.dequant_weight(*G.prepare_weight(w, rot), rot), w)
    return e < 0.02, f"identity rotation exact; recovered W within {100 * e:.2f}% of W"


def check_backward(G, dev):
    g = np.random.default_rng(6)
    M, N, K, rot = 130, 2048, 1024, (32, 32, 1)
    dy = _bf16(g.standard_normal((M, N)) * 1e-3, dev)
    w8, s = G.prepare_weight(_bf16(g.standard_normal((N, K)) * 0.02, dev), rot)
    what = G.dequant_weight(w8, s, rot)
    dx = G.linear_dx(dy, what)
    e = _rel(dx, dy.float() @ what.float())
    if e > 4e-3:
        return False, f"linear_dx vs fp32 product: {e:.2e}"
    e8 = _rel(G.linear_dx_int8(dy, w8, s, rot), dx)
    return e8 < 0.05, f"linear_dx within {e:.1e} of an fp32 product; int8 route within {100 * e8:.2f}% of it"


CHECKS = [
    ("rotate+quantize one-hot rows", check_onehot),
    ("int8 GEMM exact", check_int8_gemm),
    ("linear routes bit-identical", check_linear_routes),
    ("fused FFN == chain", check_ffn_chain),
    ("rotate-only R R = I", check_rotation_involution),
    ("dequant_weight", check_dequant_weight),
    ("linear_dx / linear_dx_int8", check_backward),
]


def main() -> int:
    from . import _lib
    try:
        _lib.lib()
    except Exception as e:  # the library is the product: without it nothing runs
        print(f"library: unavailable ({e})")
        return 1
    print(f"library: {_lib.LIB_PATH}")
    if not torch.cuda.is_available():
        for name, _ in CHECKS:
            print(f"SKIPPED  {name}: no CUDA device")
        return 2
    from . import ops as G
    print(f"device: {G.init()}")
    dev = torch.device("cuda")
    failed = 0
    for name, fn in CHECKS:
        try:
            ok, detail = fn(G, dev)
            torch.cuda.synchronize()
        except Exception:
            ok, detail = False, traceback.format_exc(limit=2).strip().splitlines()[-1]
        failed += not ok
        print(f"{'PASS' if ok else 'FAIL':8s} {name}: {detail}")
    status = G.device_status()
    if status:
        failed += 1
    print(f"{'PASS' if not status else 'FAIL':8s} device status word: {status:#x}")
    return 1 if failed else 0


if __name__ == "__main__":
    sys.exit(main())
