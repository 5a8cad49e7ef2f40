"""Comparison helpers for GPU-vs-oracle parity (tolerances from the method's contract).

- int8 codes: bit-exact, except elements on a rounding boundary, which may
  differ by +-1 in at most 1e-4 of the values (fp32 rotation order differs
  from the oracle's fp64 sums).
- int32 accumulators computed from identical int8 operands: bit-exact.
- fp32 scales: amax of an fp32 butterfly differs from the fp64-rounded one by a
  few ulps: relative 2e-6.
- bf16 outputs: max relative error 1e-2 and normwise relative error 2e-3.  The
  max-rel denominator is max(|ref|, floor) with floor = max(1e-3, 100*E)*rms(ref),
  where E bounds the absolute accumulation error of a float dot product of
  length n run on the tensor cores relative to rms(ref): each MMA step adds 16
  products into an fp32 partial sum and may drop one unit of its last place,
  partial sums stay within ~4 rms, so E = (n/16) * 2^-23 * 4 = (n/16) * 2^-21.
  Integer paths (exact accumulators) use n = 0, i.e. the 1e-3 floor.
"""
import numpy as np
import torch

INT8_BUDGET = 1e-4
SCALE_RTOL = 2e-6
BF16_MAXREL = 1e-2
BF16_NORMREL = 2e-3


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def f32(a: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def assert_int8_parity(q_gpu, q_ref, v_over_s_ref=None, budget=INT8_BUDGET, what="q"):
    q_gpu = np.asarray(q_gpu).astype(np.int64)
    q_ref = np.asarray(q_ref).astype(np.int64)
    assert q_gpu.shape == q_ref.shape, (q_gpu.shape, q_ref.shape)
    d = q_gpu - q_ref
    bad = np.flatnonzero(d)
    assert np.abs(d).max(initial=0) <= 1, f"{what}: |diff| up to {np.abs(d).max()}"
    assert bad.size <= budget * q_ref.size, f"{what}: {bad.size} of {q_ref.size} codes differ"
    if v_over_s_ref is not None and bad.size:
        frac = np.abs(np.abs(np.asarray(v_over_s_ref).ravel()[bad]) % 1.0 - 0.5)
        assert np.all(frac < 1e-3), f"{what}: mismatches not on a rounding boundary: {frac.max()}"
    return bad.size


def assert_scale_parity(s_gpu, s_ref, what="scale"):
    s_gpu = np.asarray(s_gpu, np.float64)
    s_ref = np.asarray(s_ref, np.float64)
    err = np.abs(s_gpu - s_ref)
    assert np.all(err <= SCALE_RTOL * np.abs(s_ref)), f"{what}: max rel err {np.max(err / np.maximum(s_ref, 1e-38))}"


def float_acc_floor(n: int) -> float:
    """Max-rel floor (in units of rms(ref)) for a tensor-core fp32 dot product of length n."""
    return max(1e-3, 100.0 * (n / 16.0) * 2.0 ** -21)


def assert_bf16_parity(y_gpu_bits, y_ref_bits, what="y", maxrel=BF16_MAXREL, normrel=BF16_NORMREL, acc_len=0):
    y = f32(y_gpu_bits).astype(np.float64)
    r = f32(y_ref_bits).astype(np.float64)
    assert y.shape == r.shape
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
    floor = max(float_acc_floor(acc_len) * rms, 1e-30)
    mr = np.max(np.abs(y - r) / np.maximum(np.abs(r), floor)) if r.size else 0.0
    nr = np.linalg.norm(y - r) / max(np.linalg.norm(r), 1e-30)
    assert mr <= maxrel, f"{what}: max-rel {mr:.3e} > {maxrel}"
    assert nr <= normrel, f"{what}: norm-rel {nr:.3e} > {normrel}"
    return mr, nr


def assert_rows_explained(y_gpu_bits, y_ref_bits, same_rows, what="y"):
    """Strict bf16 parity on rows whose int8 codes match the oracle's; on the other
    rows (codes that legitimately differ by +-1 at a rounding boundary) only the
    normwise bound of the whole output applies."""
    same_rows = np.asarray(same_rows, bool)
    mr = None
    if same_rows.any():
        mr, _ = assert_bf16_parity(np.asarray(y_gpu_bits)[same_rows], np.asarray(y_ref_bits)[same_rows], what=what)
    y = f32(y_gpu_bits).astype(np.float64)
    r = f32(y_ref_bits).astype(np.float64)
    nr = np.linalg.norm(y - r) / max(np.linalg.norm(r), 1e-30)
    assert nr <= BF16_NORMREL, f"{what}: norm-rel {nr:.3e} > {BF16_NORMREL}"
    return mr, nr


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |v| (8 significant bits): the largest error of rounding v to bf16."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def acc_error_usage(y_gpu_bits, exact, n: int) -> float:
    """How much of the derived accumulation-error bound E*rms (E = (n/16) * 2^-21, the max-rel floor's
    premise) a tensor-core float dot product of length n used: the largest excess of |y - exact| over the
    bf16 rounding (half a bf16 unit at the larger of |y|, |exact|), in units of E*rms(exact).  `exact` is the dot
    product in fp64 (no rounding)."""
    y = f32(y_gpu_bits).astype(np.float64)
    x = np.asarray(exact, np.float64)
    rms = np.sqrt(np.mean(x * x))
    excess = np.maximum(np.abs(y - x) - bf16_half_ulp(np.maximum(np.abs(x), np.abs(y))), 0.0)
    return float(excess.max() / ((n / 16.0) * 2.0 ** -21 * rms))
