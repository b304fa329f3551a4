"""ORACLE -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never loads it and has no
CPU fallback.

* ``seqsum_oracle.c`` -- the literal sequential loop, built strict-fp.
* ``bigint_sim.py``   -- an exact integer simulation of each binary64 add,
  which pins the C loop.

Parity unpinned: NaN payloads only (x86-64, aarch64 and the GPU may return
different NaN bits; results are then compared as "both NaN").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "seqsum_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liboracle.so")

# Strict floating point: every add kept, in order, unfused, not vectorised.
CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fno-tree-vectorize",
          "-fno-associative-math", "-fno-reciprocal-math", "-frounding-math",
          "-fno-unsafe-math-optimizations", "-fPIC", "-shared", "-std=c11"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, strict fp)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            L.oracle_seqsum.restype = ctypes.c_double
            L.oracle_seqsum.argtypes = [dp, ctypes.c_int64, ctypes.c_double]
            L.oracle_seqsum_batched.restype = None
            L.oracle_seqsum_batched.argtypes = [dp, ip, ctypes.c_int32, dp, dp]
            L.oracle_seqsum_trace.restype = None
            L.oracle_seqsum_trace.argtypes = [dp, ctypes.c_int64, ctypes.c_double, dp]
            L.oracle_seqsum_strided.restype = None
            L.oracle_seqsum_strided.argtypes = [dp, ctypes.c_int64, ctypes.c_int32, dp, dp,
                                                ctypes.POINTER(ctypes.c_float)]
            L.oracle_env_check.restype = ctypes.c_int
            L.oracle_env_check.argtypes = []
            bad = L.oracle_env_check()
            if bad:
                raise RuntimeError(f"host FPU not in round-to-nearest / no-FTZ state (code {bad})")
            _lib = L
        return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def seqsum(x: np.ndarray, s0: float = 0.0) -> float:
    """s = s0; for i: s += x[i]  (binary64, round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    return lib().oracle_seqsum(_dptr(x), len(x), float(s0))


def seqsum_batched(x: np.ndarray, offsets: np.ndarray, s0s: np.ndarray) -> np.ndarray:
    """Independent sequential sums over x[offsets[k]:offsets[k+1]]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    s0s = np.ascontiguousarray(s0s, dtype=np.float64)
    n = len(offsets) - 1
    out = np.empty(n, dtype=np.float64)
    lib().oracle_seqsum_batched(_dptr(x), offsets.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                n, _dptr(s0s), _dptr(out))
    return out


def seqsum_strided(x: np.ndarray, stride: int, s0s: np.ndarray):
    """stride interleaved sums (term i of sum k at x[i*stride + k]), one
    accumulator each, and their float means (float)(sum / n).  Returns
    (sums, means)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    s0s = np.ascontiguousarray(s0s, dtype=np.float64)
    n = len(x) // stride
    outs = np.empty(stride, dtype=np.float64)
    means = np.empty(stride, dtype=np.float32)
    lib().oracle_seqsum_strided(_dptr(x), n, int(stride), _dptr(s0s), _dptr(outs),
                                means.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return outs, means


def seqsum_trace(x: np.ndarray, s0: float = 0.0) -> np.ndarray:
    """Running sum after every add."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(len(x), dtype=np.float64)
    lib().oracle_seqsum_trace(_dptr(x), len(x), float(s0), _dptr(out))
    return out


def same_bits(a: float, b: float) -> bool:
    """Bit equality, except that any two NaNs compare equal (the one case the
    oracle leaves unpinned)."""
    a, b = float(a), float(b)
    if a != a and b != b:
        return True
    return np.float64(a).view(np.uint64) == np.float64(b).view(np.uint64)
