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
    rc = lib.gbq_quantize_act(p, p, p, 4, 8, R(2, 4, 1), None)  # valid, but rows of 8 values
    assert rc == -95 and "K % 16 == 0" in _err(lib)
    rc = lib.gbq_quantize_act(p, p, p, 4, 65536, R(128, 512, 1), None)  # valid, but beyond the generic kernel
    assert rc == -95 and "K <= 49152" in _err(lib)
    rc = lib.gbq_quantize_act(p, p, p, 4, 256, R(16, 16, 2), None)
    assert rc == -22 and "!= K" in _err(lib)
    rc = lib.gbq_quantize_act(p, p, p, 4, 256, R(3, 16, 1), None)
    assert rc == -22 and "powers of two" in _err(lib)


# Every power-of-two factor pair of the rotation descriptor (a != b, small factors, many groups) is
# accepted by every rotation entry point; M = 0 runs the full argument check and launches nothing.
ACCEPTED = [(32, 64, 1), (64, 32, 1), (64, 128, 1), (128, 64, 1), (16, 32, 1), (32, 16, 2), (2, 32, 1),
            (8, 8, 1), (4, 16, 4), (16, 4, 1), (2, 2, 16), (1, 64, 1), (64, 1, 2), (256, 8, 1), (16, 16, 128),
            (64, 64, 9), (128, 128, 3)]


@pytest.mark.parametrize("rot", ACCEPTED)
def test_every_descriptor_accepted(lib, rot):
    p = ctypes.c_void_p(256)
    K = rot[0] * rot[1] * rot[2]
    r = R(*rot)
    calls = {
        "quantize_act": lambda: lib.gbq_quantize_act(p, p, p, 0, K, r, None),
        "quantize_act_glu": lambda: lib.gbq_quantize_act_glu(p, p, p, p, 0, K, r, None),
        "dequant_act_quantize": lambda: lib.gbq_dequant_act_quantize(p, p, K, p, p, p, p, p, 0, K, r, None),
        "prepare_weight": lambda: lib.gbq_prepare_weight(p, p, p, 0, K, r, None),
        "rotate_bf16": lambda: lib.gbq_rotate_bf16(p, p, 0, K, r, None),
        "dequant_weight": lambda: lib.gbq_dequant_weight(p, p, p, 0, K, r, None),
    }
    if K % 64 == 0:
        calls.update({
            "linear_acc": lambda: lib.gbq_linear_acc(p, p, p, 64, p, 0, 64, K, r, p, 1 << 20, None),
            "linear": lambda: lib.gbq_linear(p, p, p, None, p, 0, 64, K, r, None, 0, None),
            "linear_noalloc": lambda: lib.gbq_linear_noalloc(p, p, p, None, p, 0, 64, K, r, None),
            "linear_dx_int8": lambda: lib.gbq_linear_dx_int8(p, p, p, p, 0, 1024, K, r, None, 0, None),
        })
    if K % 128 == 0:
        calls["ffn_fused (rot_h)"] = lambda: lib.gbq_ffn_fused(p, p, p, p, p, p, p, p, 0, 256, K, R(16, 16, 1), r,
                                                               None, 0, None)
        calls["ffn_fused (rot_d)"] = lambda: lib.gbq_ffn_fused(p, p, p, p, p, p, p, p, 0, K, 256, r, R(16, 16, 1),
                                                               None, 0, None)
    failed = {name: (rc, _err(lib)) for name, call in calls.items() if (rc := call()) != 0}
    assert not failed, failed


def test_identity_accepted_where_it_was_refused(lib):
    """The identity descriptor on the outputs that used to need a rotation (dx, the FFN hidden, the fused
    dequant-activation-quantize): accepted like every other descriptor."""
    p = ctypes.c_void_p(256)
    ident = lambda k: R(1, 1, k)
    assert lib.gbq_linear_dx_int8(p, p, p, p, 0, 1024, 256, ident(256), None, 0, None) == 0, _err(lib)
    assert lib.gbq_ffn_fused(p, p, p, p, p, p, p, p, 0, 256, 1024, R(16, 16, 1), ident(1024), None, 0, None) == 0
    assert lib.gbq_dequant_act_quantize(p, p, 256, p, p, p, p, p, 0, 256, ident(256), None) == 0


def test_noalloc_checks_arguments_before_its_scratch(lib):
    """gbq_linear_noalloc runs gbq_linear's size and rotation checks first: a K that is not a multiple of 64
    is GBQ_EINVAL even when M is far beyond the static scratch, and a bad rotation is reported as such."""
    p = ctypes.c_void_p(256)
    assert lib.gbq_linear_noalloc(p, p, p, None, p, 1 << 20, 64, 100, R(1, 1, 100), None) == -22
    assert "multiple of 64" in _err(lib)
    assert lib.gbq_linear_noalloc(p, p, p, None, p, 1 << 20, 64, 4096, R(64, 64, 2), None) == -22
    assert "!= K" in _err(lib)


def test_noalloc_without_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = ctypes.c_void_p(256)
    # valid sizes: the device set-up comes next and reports the missing device (not a scratch error)
    assert lib.gbq_linear_noalloc(p, p, p, None, p, 1 << 20, 64, 4096, R(64, 64, 1), None) == -19


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
