"""ctypes front end of ``oracle.c`` -- TEST INFRASTRUCTURE ONLY.

Builds ``liboracle.so`` with the host C compiler (gcc, OpenMP) and exposes
the plain fp64 definition of y = x.W^T (+ residual) to numpy.  All array
arguments are numpy ``uint16`` arrays holding raw bfloat16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile ``src`` into the shared object ``out`` (gcc -O2 -fopenmp).

    Portable C only: the same source builds on x86_64 and aarch64.  No
    -march=native and no -ffast-math, so fp64 arithmetic follows IEEE.
    """
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *extra_flags,
           src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _bind(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_decode.restype = ctypes.c_double
    lib.oracle_bf16_round.argtypes = [ctypes.c_double]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_ulp_bf16.argtypes = [ctypes.c_double]
    lib.oracle_ulp_bf16.restype = ctypes.c_double
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_linear.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                  u16p, u16p, u16p, f64p, f64p, u16p, ctypes.c_int]
    lib.oracle_linear.restype = ctypes.c_int
    lib.oracle_linear_points.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         u16p, u16p, u16p, ctypes.c_int64, i64p, i64p,
                                         f64p, f64p, ctypes.c_int]
    lib.oracle_linear_points.restype = ctypes.c_int
    lib.oracle_bf16_decode_array.argtypes = [ctypes.c_int64, u16p, f64p]
    lib.oracle_bf16_decode_array.restype = None
    lib.oracle_bf16_round_array.argtypes = [ctypes.c_int64, f64p, u16p]
    lib.oracle_bf16_round_array.restype = None
    lib.oracle_ulp_bf16_array.argtypes = [ctypes.c_int64, f64p, f64p]
    lib.oracle_ulp_bf16_array.restype = None
    return lib


def load(path: str | None = None):
    """Load (building first if missing or stale) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            if (not os.path.exists(_LIB)
                    or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
                build()
            _lib = _bind(ctypes.CDLL(_LIB))
        return _lib


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as uint16 bit patterns")
    return a


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def bf16_decode(bits, lib=None) -> np.ndarray:
    """bf16 bit patterns -> fp64 values."""
    lib = lib or load()
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_bf16_decode_array(b.size, _ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double))
    return out


def bf16_round(values, lib=None) -> np.ndarray:
    """fp64 values -> bf16 bit patterns, round to nearest even."""
    lib = lib or load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib.oracle_bf16_round_array(v.size, _ptr(v, ctypes.c_double), _ptr(out, ctypes.c_uint16))
    return out


def ulp_bf16(values, lib=None) -> np.ndarray:
    """Spacing of bf16 values at |v| (2^-133 for zero and subnormals)."""
    lib = lib or load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    lib.oracle_ulp_bf16_array(v.size, _ptr(v, ctypes.c_double), _ptr(out, ctypes.c_double))
    return out


def max_threads(lib=None) -> int:
    return int((lib or load()).oracle_max_threads())


def linear(x, W, res=None, nthreads: int = 0, lib=None):
    """Return (y_ref fp64 [M,N], s1 fp64 [M,N], y_bf16 uint16 [M,N])."""
    lib = lib or load()
    x, W = _u16(x), _u16(W)
    M, K = x.shape
    N, K2 = W.shape
    if K2 != K:
        raise ValueError("x and W disagree on K")
    r = None
    if res is not None:
        r = _u16(res)
        if r.shape != (M, N):
            raise ValueError("residual must be [M,N]")
    y = np.empty((M, N), dtype=np.float64)
    s1 = np.empty((M, N), dtype=np.float64)
    yb = np.empty((M, N), dtype=np.uint16)
    rc = lib.oracle_linear(M, N, K, _ptr(x, ctypes.c_uint16), _ptr(W, ctypes.c_uint16),
                           _ptr(r, ctypes.c_uint16), _ptr(y, ctypes.c_double),
                           _ptr(s1, ctypes.c_double), _ptr(yb, ctypes.c_uint16),
                           int(nthreads))
    if rc != 0:
        raise ValueError("oracle_linear rejected its arguments")
    return y, s1, yb


def linear_points(x, W, ms, ns, res=None, nthreads: int = 0, lib=None):
    """The definition at output points (ms[j], ns[j]): returns (y_ref, s1)."""
    lib = lib or load()
    x, W = _u16(x), _u16(W)
    M, K = x.shape
    N, _ = W.shape
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    r = None if res is None else _u16(res)
    y = np.empty(ms.shape, dtype=np.float64)
    s1 = np.empty(ms.shape, dtype=np.float64)
    rc = lib.oracle_linear_points(M, N, K, _ptr(x, ctypes.c_uint16), _ptr(W, ctypes.c_uint16),
                                  _ptr(r, ctypes.c_uint16), ms.size,
                                  _ptr(ms, ctypes.c_int64), _ptr(ns, ctypes.c_int64),
                                  _ptr(y, ctypes.c_double), _ptr(s1, ctypes.c_double),
                                  int(nthreads))
    if rc != 0:
        raise ValueError("oracle_linear_points rejected its arguments")
    return y, s1
