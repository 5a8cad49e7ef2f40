"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments with a code and a message before
touching the GPU."""
import ctypes
import os
import subprocess

import pytest

from ffn_rotate_quantize_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from ffn_rotate_quantize_gb300.build import build_lib
        build_lib()
    return L.lib()


def test_exports_every_declared_symbol(lib):
    declared = L.header_symbols()
    assert len(declared) >= 19
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    assert set(L.SIGNATURES) == set(declared), set(L.SIGNATURES) ^ set(declared)


R = L.Rot


def _err(lib):
    return lib.gbq_last_error().decode()


def test_bad_rotation_rejected(lib):
    p = ctypes.c_void_p(16)
    rc = lib.gbq_quantize_act(p, p, p, 4, 256, R(16, 8, 2), None)
    assert rc == -95 and "supported factors" in _err(lib)
    rc = lib.gbq_quantize_act(p, p, p, 4, 256, R(16, 16, 2), None)
    assert rc == -22 and "!= K" in _err(lib)
    rc = lib.gbq_quantize_act(p, p, p, 4, 256, R(3, 16, 1), None)
    assert rc == -22 and "powers of two" in _err(lib)


def test_bad_sizes_and_pointers_rejected(lib):
    p = ctypes.c_void_p(16)
    assert lib.gbq_linear(p, p, p, None, p, 8, 64, 100, R(1, 1, 100), p, 1 << 20, None) == -22
    assert "multiple of 64" in _err(lib)
    assert lib.gbq_quantize_act(ctypes.c_void_p(18), p, p, 4, 256, R(16, 16, 1), None) == -22
    assert "16-byte aligned" in _err(lib)
    assert lib.gbq_quantize_act(None, p, p, 4, 256, R(16, 16, 1), None) == -22
    assert lib.gbq_ffn_fused(p, p, p, p, p, p, p, p, 4, 256, 200, R(16, 16, 1), R(16, 16, 1), p, 0, None) == -22


def test_workspace_too_small_rejected(lib):
    """gbq_workspace_size reports the preferred size (with the per-row code L1 norms that let the
    GEMM run whole tiles as one exact chunk); calls accept anything down to the minimum, codes and
    scales: M*K*2 + M*4, each rounded up to 256 bytes, and reject less."""
    p = ctypes.c_void_p(256)
    need = lib.gbq_workspace_size(1, 300, 512, 1024, 0)
    a256 = lambda v: (v + 255) // 256 * 256
    minimum = a256(300 * 1024 * 2) + a256(300 * 4)
    assert need == minimum + a256(300 * 4)
    rc = lib.gbq_linear(p, p, p, None, p, 300, 512, 1024, R(32, 32, 1), p, minimum - 1, None)
    assert rc == -28 and "workspace" in _err(lib)


def test_empty_input_is_a_noop(lib):
    p = ctypes.c_void_p(16)
    assert lib.gbq_quantize_act(p, p, p, 0, 256, R(16, 16, 1), None) == 0
    assert lib.gbq_linear(p, p, p, None, p, 0, 64, 256, R(16, 16, 1), None, 0, None) == 0


def test_no_device_reported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = ctypes.c_void_p(256)
    rc = lib.gbq_quantize_act(p, p, p, 4, 256, R(16, 16, 1), None)
    assert rc == -19 and _err(lib)
