"""Double-precision CPU oracle for exact attention, forward and VJP.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product path (the CUDA
library and its Python binding) never imports this package, and this package
imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (plain C, OpenMP over independent
heads / KV groups); this module only compiles it and marshals numpy float64
arrays. Every function is the plain definition of attention (see the C file's
header for the formulas and the page passages they follow).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc -O3 -fopenmp a C file into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    return compile_source(_SRC, _LIB)


def load_library(path: str):
    """Bind another build of the oracle's C interface (used by the tests that
    plant mistakes in a copy of the oracle to show the pins catch them)."""
    return _bind(path)


SOURCE = _SRC


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i,
                                    ctypes.c_double, i, i, i, i]
    lib.oracle_attn_fwd.restype = None
    lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                    i, i, i, i, i, i, ctypes.c_double,
                                    i, i, i, i]
    lib.oracle_attn_bwd.restype = None
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _as_f64(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return np.ascontiguousarray(a)


def _dims(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, T, D]")
    B, Hq, Tq, D = q.shape
    Bk, Hkv, Tkv, Dk = k.shape
    if k.shape != v.shape or Bk != B or Dk != D or Hq % Hkv:
        raise ValueError(f"incompatible shapes q{q.shape} k{k.shape} v{v.shape}")
    return B, Hq, Hkv, Tq, Tkv, D


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def attn_fwd(q, k, v, scale: float, causal: bool = False, window: int = 0,
             row_lo: int = 0, row_hi: int | None = None, lib=None):
    """Return (O, LSE) in float64. Rows outside [row_lo, row_hi) are NaN."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, Hq, Hkv, Tq, Tkv, D = _dims(q, k, v)
    row_hi = Tq if row_hi is None else row_hi
    o = np.full((B, Hq, Tq, D), np.nan)
    lse = np.full((B, Hq, Tq), np.nan)
    (lib or _load()).oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                            B, Hq, Hkv, Tq, Tkv, D, float(scale), int(bool(causal)),
                            int(window), int(row_lo), int(row_hi))
    return o, lse


def attn_bwd(q, k, v, dout, scale: float, causal: bool = False, window: int = 0,
             row_lo: int = 0, row_hi: int | None = None, lib=None):
    """Return a dict with dq, dk, dv, o, lse, dvec (float64).

    dq/o/lse/dvec rows outside [row_lo, row_hi) are NaN; dk/dv are the sums
    over the covered query rows (the full gradient when the range is [0, Tq)).
    """
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, Hq, Hkv, Tq, Tkv, D = _dims(q, k, v)
    if dout.shape != q.shape:
        raise ValueError("dO must have the shape of Q")
    row_hi = Tq if row_hi is None else row_hi
    dq = np.full(q.shape, np.nan)
    dk = np.empty(k.shape)
    dv = np.empty(v.shape)
    o = np.full(q.shape, np.nan)
    lse = np.full((B, Hq, Tq), np.nan)
    dvec = np.full((B, Hq, Tq), np.nan)
    (lib or _load()).oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(o), _ptr(lse), _ptr(dvec),
                            B, Hq, Hkv, Tq, Tkv, D, float(scale), int(bool(causal)),
                            int(window), int(row_lo), int(row_hi))
    return {"dq": dq, "dk": dk, "dv": dv, "o": o, "lse": lse, "dvec": dvec}
