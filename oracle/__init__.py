"""fp64 CPU oracle for attention forward and the FlashAttention-2 backward.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg, never by the library.  It shares no code with
the CUDA path; both sides only share the seeded input generators.

The arithmetic lives in ``fa_ref.c`` (plain C loops in double precision, see
its header for the definitions and the pages they follow).  This module
compiles it with gcc on first use and exposes numpy wrappers.

Functions (all take / return float64 numpy arrays, layouts [B, H, S, d];
``window`` is the sliding-window size, 0 for none):
    ref_fwd(Q, K, V, scale, causal, window=0)              -> (O, LSE)
    ref_preprocess(dO, O)                                  -> D
    ref_bwd(dO, Q, K, V, O, LSE, scale, causal, window=0)  -> (dQ, dK, dV, D)
    ref_dq_rows(..., rows, scale, causal, window=0)        -> dQ rows
    ref_dkv_rows(..., rows, scale, causal, window=0)       -> (dK rows, dV rows)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libfa_ref.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fa_ref.c into a shared library (gcc, OpenMP, -O2, no -march)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def open_library(path: str):
    """ctypes handle on a compiled fa_ref.c with its argument types declared."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    Dbl = ctypes.c_double
    lib.fa_ref_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, Dbl, I, I]
    lib.fa_ref_preprocess.argtypes = [P, P, P, ctypes.c_long, I]
    lib.fa_ref_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, Dbl, I, I]
    lib.fa_ref_dq_rows.argtypes = [P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, Dbl, I, I]
    lib.fa_ref_dkv_rows.argtypes = [P, P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, Dbl, I, I]
    lib.fa_ref_num_threads.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def num_threads() -> int:
    return int(_load().fa_ref_num_threads())


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float64:
        a = a.astype(np.float64)
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _window(window) -> int:
    w = int(window)
    if w < 0:
        raise ValueError(f"window must be >= 0, got {w}")
    return w


def _dims(Q, K):
    B, H, S_q, d = Q.shape
    Bk, H_kv, S_k, dk = K.shape
    if Bk != B or dk != d or H % H_kv != 0:
        raise ValueError(f"incompatible shapes Q{Q.shape} K{K.shape}")
    return B, H, H_kv, S_q, S_k, d


def ref_fwd(Q, K, V, scale: float, causal: bool, window: int = 0):
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, H_kv, S_q, S_k, d = _dims(Q, K)
    O = np.empty((B, H, S_q, d))
    LSE = np.empty((B, H, S_q))
    _load().fa_ref_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                       B, H, H_kv, S_q, S_k, d, float(scale), int(bool(causal)), _window(window))
    return O, LSE


def ref_preprocess(dO, O):
    dO, O = _f64(dO), _f64(O)
    d = dO.shape[-1]
    D = np.empty(dO.shape[:-1])
    _load().fa_ref_preprocess(_ptr(dO), _ptr(O), _ptr(D), int(D.size), d)
    return D


def ref_bwd(dO, Q, K, V, O, LSE, scale: float, causal: bool, window: int = 0):
    dO, Q, K, V, O, LSE = (_f64(x) for x in (dO, Q, K, V, O, LSE))
    B, H, H_kv, S_q, S_k, d = _dims(Q, K)
    dQ = np.empty_like(Q)
    dK = np.empty_like(K)
    dV = np.empty_like(V)
    D = np.empty((B, H, S_q))
    _load().fa_ref_bwd(_ptr(dO), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                       _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(D),
                       B, H, H_kv, S_q, S_k, d, float(scale), int(bool(causal)), _window(window))
    return dQ, dK, dV, D


def ref_dq_rows(dO, Q, K, V, O, LSE, rows, scale: float, causal: bool, window: int = 0):
    """dQ for flat query rows (b*H + h)*S_q + i."""
    dO, Q, K, V, O, LSE = (_f64(x) for x in (dO, Q, K, V, O, LSE))
    B, H, H_kv, S_q, S_k, d = _dims(Q, K)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.size, d))
    _load().fa_ref_dq_rows(_ptr(dO), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                           _ptr(rows), int(rows.size), _ptr(out),
                           B, H, H_kv, S_q, S_k, d, float(scale), int(bool(causal)),
                           _window(window))
    return out


def ref_dkv_rows(dO, Q, K, V, O, LSE, rows, scale: float, causal: bool, window: int = 0):
    """dK, dV for flat key rows (b*H_kv + hk)*S_k + j (summed over the group)."""
    dO, Q, K, V, O, LSE = (_f64(x) for x in (dO, Q, K, V, O, LSE))
    B, H, H_kv, S_q, S_k, d = _dims(Q, K)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dk = np.empty((rows.size, d))
    dv = np.empty((rows.size, d))
    _load().fa_ref_dkv_rows(_ptr(dO), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                            _ptr(rows), int(rows.size), _ptr(dk), _ptr(dv),
                            B, H, H_kv, S_q, S_k, d, float(scale), int(bool(causal)),
                            _window(window))
    return dk, dv
