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


def test_every_entry_point_accepts_empty_inputs(lib):
    """An empty batch (M = 0, or N = 0 for the weight calls) is valid for every entry point: it returns 0
    and launches nothing, before any device work (so it holds on a machine without a GPU too), with
    valid-looking or null pointers (an empty tensor may report a null data pointer)."""
    for p in (ctypes.c_void_p(256), None):
        _check_empty_calls(lib, p)


def _check_empty_calls(lib, p):
    r1, r2 = R(16, 16, 1), R(64, 64, 1)
    calls = {
        "quantize_act": lambda: lib.gbq_quantize_act(p, p, p, 0, 256, r1, None),
        "quantize_act_glu": lambda: lib.gbq_quantize_act_glu(p, p, p, p, 0, 256, r1, None),
        "dequant_act_quantize": lambda: lib.gbq_dequant_act_quantize(p, p, 256, p, p, p, p, p, 0, 256, r1, None),
        "prepare_weight": lambda: lib.gbq_prepare_weight(p, p, p, 0, 256, r1, None),
        "int8_gemm": lambda: lib.gbq_int8_gemm(p, p, p, 64, 0, 64, 256, p, 1 << 20, None),
        "linear_acc": lambda: lib.gbq_linear_acc(p, p, p, 64, p, 0, 64, 256, r1, p, 1 << 20, None),
        "dequant": lambda: lib.gbq_dequant(p, 64, p, p, None, p, 64, 0, 64, None),
        "linear": lambda: lib.gbq_linear(p, p, p, None, p, 0, 64, 256, r1, None, 0, None),
        "ffn_fused": lambda: lib.gbq_ffn_fused(p, p, p, p, p, p, p, p, 0, 4096, 4096, r2, r2, None, 0, None),
        "dequant_weight": lambda: lib.gbq_dequant_weight(p, p, p, 0, 256, r1, None),
        "linear_dx": lambda: lib.gbq_linear_dx(p, p, p, 0, 256, 256, None),
        "linear_bf16": lambda: lib.gbq_linear_bf16(p, p, None, p, 0, 64, 256, None),
        "linear_dx_int8": lambda: lib.gbq_linear_dx_int8(p, p, p, p, 0, 1024, 256, r1, None, 0, None),
        "rotate_bf16": lambda: lib.gbq_rotate_bf16(p, p, 0, 256, r1, None),
        "linear_noalloc": lambda: lib.gbq_linear_noalloc(p, p, p, None, p, 0, 64, 256, r1, None),
    }
    failed = {name: (rc, _err(lib)) for name, call in calls.items() if (rc := call()) != 0}
    assert not failed, failed
