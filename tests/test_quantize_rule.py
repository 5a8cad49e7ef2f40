"""The kernels' quantize rule, checked on the CPU in IEEE fp32 (numpy float32 arithmetic rounds to nearest
even, as the kernels' __fmul_rn / __fadd_rn / __frcp_rn do).

The kernels compute r = fl(1/s), t = fl(v r) and read the code out of the low byte of m = fl(t + 1.5 * 2^23);
they keep it when |t - (m - 1.5 * 2^23)| <= 0.4999 and otherwise recompute with IEEE division. The claim that
makes the codes identical to the definition clamp(rne(fl(v / s))): every kept code equals it. Inputs span row
maxima from 1e-30 to 1e4, uniform values, the row maximum itself, and values placed a few ulp around the
half-integer multiples of s, where the two roundings can part."""
import numpy as np
import pytest

MAGIC = np.float32(12582912.0)  # 1.5 * 2^23


def _kernel_codes(v, s):
    with np.errstate(over="ignore", invalid="ignore"):
        r = np.float32(1.0) / s
        t = (v * r).astype(np.float32)
        m = (t + MAGIC).astype(np.float32)
        d = np.abs(t - (m - MAGIC)).astype(np.float32)
    code = (m.view(np.uint32) & 0xFF).astype(np.uint8).view(np.int8).astype(np.int64)
    return code, (d <= np.float32(0.4999)) & (s >= np.float32(1e-30))  # tiny scales: always division


def _definition(v, s):
    return np.clip(np.rint((v / s).astype(np.float32)), -127, 127).astype(np.int64)


@pytest.mark.parametrize("seed", range(4))
def test_kept_codes_equal_the_definition(seed):
    g = np.random.default_rng(seed)
    rows, n = 400, 2048
    amax = np.exp(g.uniform(np.log(1e-30), np.log(1e4), rows)).astype(np.float32)
    s = (amax / np.float32(127.0)).astype(np.float32)
    v = (g.uniform(-1, 1, (rows, n)) * amax[:, None]).astype(np.float32)
    v[:, 0] = amax
    v[:, 1] = -amax
    # near the half-integer multiples of s: (k + 1/2) s nudged by up to 3 ulp either way
    k = g.integers(-127, 127, (rows, n // 4))
    half = ((k + 0.5) * s[:, None]).astype(np.float32)
    v[:, 2:2 + n // 4] = np.nextafter(half, np.where(g.random(half.shape) < 0.5, np.inf, -np.inf)).astype(np.float32)
    for _ in range(2):
        v[:, 2:2 + n // 4] = np.where(g.random(half.shape) < 0.5, v[:, 2:2 + n // 4],
                                      np.nextafter(v[:, 2:2 + n // 4], np.float32(np.inf)))
    v = np.clip(v, -amax[:, None], amax[:, None])
    code, kept = _kernel_codes(v, s[:, None])
    ref = _definition(v, s[:, None])
    assert kept[s >= np.float32(1e-30)][:, 2 + n // 4:].mean() > 0.999  # the filter is rare off the boundaries
    assert np.array_equal(code[kept], ref[kept])


def test_the_filter_catches_every_disagreement():
    """Where the reciprocal path's code differs from the definition's, the filter always sends the value to
    the division path (so a disagreement can never reach the output)."""
    g = np.random.default_rng(11)
    s = g.uniform(1e-3, 1e-1, 50000).astype(np.float32)
    k = g.integers(-127, 127, s.shape)
    v = ((k + 0.5) * s).astype(np.float32)
    for nudge in range(3):  # the fp32 value nearest each half-integer multiple, then 1 and 2 ulp above it
        code, kept = _kernel_codes(v, s)
        differ = code != _definition(v, s)
        assert differ.any() or nudge == 2  # the two roundings do part here
        assert not np.any(differ & kept)
        v = np.nextafter(v, np.float32(np.inf)).astype(np.float32)
