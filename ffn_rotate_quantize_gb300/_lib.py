"""ctypes loader for libgbq.so and the C signatures of include/gbq.h.

The library is required: if it is missing or cannot load, every call raises.
There is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(_HERE), "include", "gbq.h")
LIB_PATH = os.environ.get("GBQ_LIB", os.path.join(_HERE, "libgbq.so"))

c_i64 = ctypes.c_int64
c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p
c_sz = ctypes.c_size_t


class Rot(ctypes.Structure):
    """gbq_rot: R = I_groups (x) (H_a (x) H_b) / sqrt(a*b)."""
    _fields_ = [("a", c_i32), ("b", c_i32), ("groups", c_i32)]


# name -> argtypes (restype int unless listed in _RESTYPES)
SIGNATURES = {
    "gbq_init": [],
    "gbq_device_name": [],
    "gbq_last_error": [],
    "gbq_device_status": [c_vp, ctypes.POINTER(ctypes.c_uint32)],
    "gbq_sync": [c_vp],
    "gbq_workspace_size": [ctypes.c_int, c_i64, c_i64, c_i64, c_i64],
    "gbq_quantize_act": [c_vp, c_vp, c_vp, c_i64, c_i64, Rot, c_vp],
    "gbq_quantize_act_glu": [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, Rot, c_vp],
    "gbq_dequant_act_quantize": [c_vp, c_vp, c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, Rot, c_vp],
    "gbq_prepare_weight": [c_vp, c_vp, c_vp, c_i64, c_i64, Rot, c_vp],
    "gbq_int8_gemm": [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i64, c_vp, c_sz, c_vp],
    "gbq_linear_acc": [c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, c_i64, c_i64, Rot, c_vp, c_sz, c_vp],
    "gbq_dequant": [c_vp, c_i64, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp],
    "gbq_linear": [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, Rot, c_vp, c_sz, c_vp],
    "gbq_ffn_fused": [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, Rot, Rot, c_vp, c_sz,
                      c_vp],
    "gbq_dequant_weight": [c_vp, c_vp, c_vp, c_i64, c_i64, Rot, c_vp],
    "gbq_linear_dx": [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp],
    "gbq_linear_bf16": [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp],
    "gbq_linear_dx_int8": [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, Rot, c_vp, c_sz, c_vp],
    "gbq_rotate_bf16": [c_vp, c_vp, c_i64, c_i64, Rot, c_vp],
    "gbq_linear_noalloc": [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, Rot, c_vp],
    "gbq_prof_enable": [ctypes.c_int],
    "gbq_prof_read": [ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)],
}
_RESTYPES = {"gbq_device_name": ctypes.c_char_p, "gbq_last_error": ctypes.c_char_p, "gbq_workspace_size": c_sz}

_lib = None


class GbqError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libgbq error {code}: {msg}")
        self.code = code


def header_symbols() -> list[str]:
    """Every function name declared in include/gbq.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(gbq_[a-z0-9_]+)\s*\(", text)))


def lib():
    """Load libgbq.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with `python -m ffn_rotate_quantize_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _RESTYPES.get(name, ctypes.c_int)
        _lib = L
    return _lib


def check(rc: int) -> None:
    if rc != 0:
        raise GbqError(rc, lib().gbq_last_error().decode())
