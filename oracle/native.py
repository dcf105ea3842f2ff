"""Build and load the plain-C float64 oracle (oracle/ssm_oracle.c) with gcc.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libssm_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no -march) if it is missing or stale."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        i64, fp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
        _lib.ssm_oracle_ssd.argtypes = [fp] * 7 + [dp, dp] + [i64] * 6 + [fp, i64, ctypes.c_int]
        _lib.ssm_oracle_ssd.restype = ctypes.c_int
        _lib.ssm_oracle_linscan.argtypes = [fp, fp, dp, i64, i64, fp, i64, ctypes.c_int]
        _lib.ssm_oracle_linscan.restype = ctypes.c_int
        _lib.ssm_oracle_max_threads.restype = ctypes.c_int
    return _lib


def max_threads() -> int:
    return int(lib().ssm_oracle_max_threads())


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def ssd_fwd(x, dt, A, B, C, D, h0=None, units=None, threads: int = 0):
    """C oracle of the SSD forward on the selected (batch, head) units.

    Shapes as oracle.ssd.ssd_fwd.  ``units`` lists u = batch_index * nheads +
    head (default: all).  Returns (y [n_units, L, H], h_final [n_units, H, S])
    in float64.
    """
    x, dt, A, B, C, D = map(_f32, (x, dt, A, B, C, D))
    h0 = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64)
    batch, L, nh, H = x.shape
    G, S = B.shape[2], B.shape[3]
    if units is None:
        units = np.arange(batch * nh, dtype=np.int64)
    units = np.ascontiguousarray(units, dtype=np.int64)
    y = np.empty((len(units), L, H))
    hf = np.empty((len(units), H, S))
    rc = lib().ssm_oracle_ssd(_ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0),
                              _ptr(y), _ptr(hf), batch, L, nh, H, S, G, _ptr(units), len(units), threads)
    if rc != 0:
        raise ValueError(f"ssm_oracle_ssd returned {rc}")
    return y, hf


def linscan(a, b, rows=None, threads: int = 0):
    """C oracle of the scalar scan on the selected rows of [rows, L] inputs; float64 [n_sel, L]."""
    a, b = _f32(a), _f32(b)
    if a.shape != b.shape or a.ndim != 2:
        raise ValueError("a, b must be [rows, L] and equal")
    if rows is None:
        rows = np.arange(a.shape[0], dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    h = np.empty((len(rows), a.shape[1]))
    rc = lib().ssm_oracle_linscan(_ptr(a), _ptr(b), _ptr(h), a.shape[0], a.shape[1], _ptr(rows), len(rows),
                                  threads)
    if rc != 0:
        raise ValueError(f"ssm_oracle_linscan returned {rc}")
    return h
