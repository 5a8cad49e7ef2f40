"""The self-test command (`python -m ffn_rotate_quantize_gb300`): its closed-form Hadamard signs against the
oracle's explicit Kronecker matrices, its behaviour without a GPU (every check SKIPPED, exit status 2, never a
pass), and on a GPU every check passing."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle as O
from ffn_rotate_quantize_gb300.selftest import hadamard_sign, rotation_sign

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("n", [4, 8, 16, 32, 64, 128])
def test_hadamard_sign_matches_oracle(n):
    H = O.hadamard(n)
    p = np.arange(n)
    for q in range(n):
        assert np.array_equal(hadamard_sign(n, p, q), H[:, q])


@pytest.mark.parametrize("rot", [(16, 16, 1), (64, 64, 1), (32, 32, 1)])
def test_rotation_sign_matches_oracle(rot):
    a, b, _ = rot
    R = O.rotation_matrix(rot) * np.sqrt(a * b)
    i = np.arange(a * b)
    for k in (0, 1, a * b // 3, a * b - 1):
        assert np.array_equal(rotation_sign(a, b, i, k), np.rint(R[:, k]).astype(np.int64))


def _run():
    return subprocess.run([sys.executable, "-m", "ffn_rotate_quantize_gb300"], cwd=ROOT, capture_output=True,
                          text=True, timeout=600)


@pytest.mark.skipif(torch.cuda.is_available(), reason="the no-GPU behaviour")
def test_selftest_without_gpu_skips():
    from ffn_rotate_quantize_gb300 import _lib as L
    if not os.path.exists(L.LIB_PATH):
        from ffn_rotate_quantize_gb300.build import build_lib
        build_lib()
    r = _run()
    assert r.returncode == 2, r.stdout + r.stderr
    lines = r.stdout.strip().splitlines()
    assert lines[0].startswith("library: ")
    assert all(l.startswith("SKIPPED") for l in lines[1:]) and len(lines) > 1
    assert "PASS" not in r.stdout


@pytest.mark.gpu
def test_selftest_on_gpu_passes():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    r = _run()
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout and "SKIPPED" not in r.stdout
