"""The seeded input recipe: the generators draw the stated shapes and distributions (x ~ N(0,1) with 1% of
channels scaled, weights ~ N(0,0.02), bias ~ N(0,0.01), dy ~ N(0,1e-3)), in a fixed order per seed, rounded to
bf16 with round-to-nearest-even (checked against torch's cast)."""
import numpy as np
import pytest
import torch

from ffn_rotate_quantize_gb300 import inputs as I


def test_bf16_bits_matches_torch():
    g = np.random.default_rng(0)
    a = np.concatenate([g.standard_normal(100000).astype(np.float32) * np.float32(10.0) ** g.integers(-30, 30, 100000),
                        np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.3895314e38], np.float32)])
    a = a.astype(np.float32)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(I.bf16_bits(a), ref)
    assert np.array_equal(I.bf16_to_float(ref), torch.from_numpy(a).to(torch.bfloat16).float().numpy())
    nan = I.bf16_bits(np.array([np.nan], np.float32))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


def test_outlier_count():
    assert I.outlier_count(4096) == 41 and I.outlier_count(256) == 3 and I.outlier_count(16384) == 164


def test_linear_case_distributions():
    c = I.linear_case(256, 4096, 2048, n_outliers=41, outlier_scale=30.0, bias_std=0.01, seed=0)
    x = I.bf16_to_float(c["x"]).astype(np.float64)
    w = I.bf16_to_float(c["w"]).astype(np.float64)
    b = I.bf16_to_float(c["bias"]).astype(np.float64)
    idx = c["outliers"]
    assert len(idx) == 41 and len(np.unique(idx)) == 41
    rest = np.setdiff1d(np.arange(4096), idx)
    assert abs(x[:, rest].std() - 1.0) < 0.01 and abs(x[:, rest].mean()) < 0.01
    assert abs(x[:, idx].std() - 30.0) < 1.0
    col_rms = np.sqrt((x ** 2).mean(axis=0))
    assert set(np.argsort(col_rms)[-41:]) == set(idx)  # the scaled channels are the loud ones
    assert abs(w.std() - 0.02) < 2e-4 and abs(b.std() - 0.01) < 1.5e-3


def test_recipe_is_seeded_and_ordered():
    a = I.linear_case(8, 256, 16, n_outliers=3, outlier_scale=20.0, bias_std=0.01, seed=5)
    b = I.linear_case(8, 256, 16, n_outliers=3, outlier_scale=20.0, bias_std=0.01, seed=5)
    c = I.linear_case(8, 256, 16, n_outliers=3, outlier_scale=20.0, bias_std=0.01, seed=6)
    for k in ("x", "w", "bias", "outliers"):
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(a["x"], c["x"])
    # draw order: outlier indices, then x, then W, then bias
    rng = np.random.default_rng(5)
    idx = rng.choice(256, size=3, replace=False)
    x = rng.standard_normal((8, 256), dtype=np.float32)
    x[:, idx] *= np.float32(20.0)
    w = rng.standard_normal((16, 256), dtype=np.float32) * np.float32(0.02)
    assert np.array_equal(a["x"], I.bf16_bits(x)) and np.array_equal(a["w"], I.bf16_bits(w))


@pytest.mark.parametrize("name", ["tiny_linear", "decode_gemv", "prefill_linear", "swiglu_ffn", "backward_dx"])
def test_named_workloads_shapes(name):
    small = {"tiny_linear": {}, "decode_gemv": dict(N=64), "prefill_linear": dict(M=4, N=64),
             "swiglu_ffn": dict(M=4, H=256, d=512), "backward_dx": dict(M=4, N=64, K=256)}[name]
    c = I.config_case(name, **small)
    cfg = c["config"]
    if name == "swiglu_ffn":
        assert c["x"].shape == (cfg["M"], cfg["d"]) and c["wg"].shape == (cfg["H"], cfg["d"])
        assert c["wd"].shape == (cfg["d"], cfg["H"])
    elif name == "backward_dx":
        assert c["dy"].shape == (cfg["M"], cfg["N"]) and c["w"].shape == (cfg["N"], cfg["K"])
        assert abs(I.bf16_to_float(c["dy"]).std() - 1e-3) < 1e-4
    else:
        assert c["x"].shape == (cfg["M"], cfg["K"]) and c["w"].shape == (cfg["N"], cfg["K"])
        assert (c["bias"] is None) == (cfg["bias_std"] is None)
        assert len(c["outliers"]) == cfg["n_outliers"]
