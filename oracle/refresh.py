"""ctypes loader for the C oracle of the compressed-residual refresh (test infrastructure only).

``build()`` compiles ``refresh.c`` into ``oracle/_build/liboracle_refresh.so`` with
gcc -O2 -ffp-contract=off (and OpenMP), so no fused multiply-add other than the
explicit ``fmaf`` of the refresh rule is formed.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "refresh.c")
_OUT = os.path.join(_HERE, "_build", "liboracle_refresh.so")
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        tmp = _OUT + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_refresh_residual.restype = ctypes.c_int
        lib.oracle_refresh_residual.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
        lib.oracle_apply_residual.restype = ctypes.c_int
        lib.oracle_apply_residual.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_int]
        _lib = lib
    return _lib


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Exact bit patterns of values that are already bf16 (fp64 holding bf16 values)."""
    f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("values are not bf16-representable")
    return (u >> 16).astype(np.uint16)


def refresh_residual(fresh, stale, dtype: str):
    """Returns (new_stale fp64, codes int8, scales fp32) for flat buffers ``fresh``, ``stale``."""
    lib = _load()
    n = int(np.asarray(fresh).size)
    if dtype == "bf16":
        f = _bf16_bits(np.asarray(fresh).reshape(-1))
        s = _bf16_bits(np.asarray(stale).reshape(-1)).copy()
        code = 1
    elif dtype == "f32":
        f = np.ascontiguousarray(np.asarray(fresh).reshape(-1), dtype=np.float32)
        s = np.ascontiguousarray(np.asarray(stale).reshape(-1), dtype=np.float32).copy()
        code = 0
    else:
        raise ValueError(dtype)
    codes = np.zeros(n, dtype=np.int8)
    scales = np.zeros((n + 127) // 128, dtype=np.float32)
    rc = lib.oracle_refresh_residual(f.ctypes.data, s.ctypes.data, codes.ctypes.data,
                                     scales.ctypes.data, n, code)
    if rc:
        raise ValueError("oracle_refresh_residual: bad arguments")
    if dtype == "bf16":
        new = (s.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        new = s.astype(np.float64)
    return new, codes, scales


def apply_residual(stale, codes, scales, dtype: str):
    """Receiver side: new stale (fp64) = store(fmaf(code, scale, stale)) per element."""
    lib = _load()
    n = int(np.asarray(stale).size)
    if dtype == "bf16":
        s = _bf16_bits(np.asarray(stale).reshape(-1)).copy()
        code = 1
    elif dtype == "f32":
        s = np.ascontiguousarray(np.asarray(stale).reshape(-1), dtype=np.float32).copy()
        code = 0
    else:
        raise ValueError(dtype)
    c = np.ascontiguousarray(codes, dtype=np.int8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    if c.size != n or sc.size != (n + 127) // 128:
        raise ValueError("message size mismatch")
    if lib.oracle_apply_residual(s.ctypes.data, c.ctypes.data, sc.ctypes.data, n, code):
        raise ValueError("oracle_apply_residual: bad arguments")
    if dtype == "bf16":
        return (s.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return s.astype(np.float64)
