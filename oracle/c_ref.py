"""ctypes wrapper and build step for the plain-C Newton–Schulz cross-check
(``ns_ref.c``).  TEST INFRASTRUCTURE ONLY: only ``tests/`` use it."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ns_ref.c")
_LIB = os.path.join(_HERE, "_build", "libns_ref.so")


def build(force: bool = False) -> str:
    """Compile ns_ref.c with gcc into oracle/_build/libns_ref.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.ns_ref_iterate.restype = ctypes.c_int
        _lib.ns_ref_iterate.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p]
    return _lib


def ns_iterate_c(X, coeffs, normalize: bool = True) -> np.ndarray:
    """Run ns_ref_iterate on a float64 copy of X; coeffs is a list of (a, b, c)."""
    lib = _load()
    X = np.ascontiguousarray(X, dtype=np.float64)
    co = np.ascontiguousarray(np.asarray(coeffs, dtype=np.float64).reshape(-1, 3))
    out = np.empty_like(X)
    rc = lib.ns_ref_iterate(X.ctypes.data, X.shape[0], X.shape[1], co.ctypes.data, co.shape[0],
                            int(bool(normalize)), out.ctypes.data)
    if rc != 0:
        raise RuntimeError("ns_ref_iterate failed")
    return out
