"""Builds and loads the oracle's C loops (moe_oracle.c) with gcc.

Test infrastructure only (see oracle/__init__.py).  The shared object is
built next to the source, from this file alone, with no flag that relaxes
IEEE arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so (if stale) and return its path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i64 = ctypes.c_int64
            vp = ctypes.c_void_p
            L.oracle_num_threads.restype = ctypes.c_int
            L.oracle_set_num_threads.argtypes = [ctypes.c_int]
            L.oracle_gate_logits.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            L.oracle_matmul_fp8.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            L.oracle_matmul_bf16.argtypes = [i64, i64, i64, vp, vp, vp]
            _lib = L
    return _lib


def ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))
