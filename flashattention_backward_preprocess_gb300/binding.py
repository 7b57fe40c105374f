"""ctypes binding of include/fa.h.  Argument marshalling only.

Each function mirrors the C entry point of the same name: shapes are read
from the tensors, pointers and the current CUDA stream are passed through,
and a non-zero status raises FaError carrying fa_last_error().  Output
tensors may be passed in (written in place) or are allocated with
torch.empty (device memory is PyTorch's job; the library never allocates
outputs).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

FA_F32, FA_F16, FA_BF16 = 0, 1, 2
_STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
           4: "FA_ERR_TIMEOUT", 5: "FA_ERR_NOMEM"}
_DT = {torch.float32: FA_F32, torch.float16: FA_F16, torch.bfloat16: FA_BF16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libfa.so")
_lock = threading.Lock()
_lib = None

#: every symbol include/fa.h declares
EXPORTS = ("fa_bwd", "fa_bwd_ex", "fa_bwd_noalloc", "fa_bwd_preprocess", "fa_fwd", "fa_fwd_ex", "fa_bwd_host",
           "fa_bwd_workspace_bytes",
           "fa_check_device", "fa_profile", "fa_profile_read", "fa_selftest_timeout",
           "fa_last_error", "fa_shutdown", "fa_version")


class FaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load libfa.so (built by flashattention_backward_preprocess_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise FaError(3, f"CUDA library not built: {p} (run flashattention_backward_preprocess_gb300.build.build())")
        lib = ctypes.CDLL(p)
        V, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        big = [V] * 9 + [I] * 6 + [F, I, I, V]
        lib.fa_bwd.argtypes = big
        lib.fa_bwd.restype = I
        lib.fa_bwd_noalloc.argtypes = big
        lib.fa_bwd_noalloc.restype = I
        lib.fa_bwd_host.argtypes = big
        lib.fa_bwd_host.restype = I
        lib.fa_bwd_preprocess.argtypes = [V, V, V, I, I, I, I, I, V]
        lib.fa_bwd_preprocess.restype = I
        lib.fa_fwd.argtypes = [V, V, V, V, V, I, I, I, I, I, I, F, I, I, V]
        lib.fa_fwd.restype = I
        lib.fa_bwd_ex.argtypes = [V] * 9 + [I] * 6 + [F, I, I, I, I, V]
        lib.fa_bwd_ex.restype = I
        lib.fa_fwd_ex.argtypes = [V, V, V, V, V, I, I, I, I, I, I, F, I, I, I, V]
        lib.fa_fwd_ex.restype = I
        lib.fa_bwd_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_check_device.argtypes = [V]
        lib.fa_check_device.restype = I
        lib.fa_profile.argtypes = [I]
        lib.fa_profile.restype = I
        lib.fa_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]
        lib.fa_profile_read.restype = I
        lib.fa_selftest_timeout.argtypes = [ctypes.c_ulonglong, V]
        lib.fa_selftest_timeout.restype = I
        lib.fa_last_error.restype = ctypes.c_char_p
        lib.fa_version.restype = ctypes.c_char_p
        lib.fa_shutdown.restype = None
        if path is None:
            _lib = lib
        return lib


def fa_last_error() -> str:
    return load_library().fa_last_error().decode()


def fa_version() -> str:
    return load_library().fa_version().decode()


def fa_shutdown() -> None:
    load_library().fa_shutdown()


def fa_bwd_workspace_bytes(B: int, H: int, S_q: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, S_q, d))


def _check(rc: int):
    if rc != 0:
        raise FaError(rc, fa_last_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise FaError(1, f"dtype: unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _shape4(name: str, t: torch.Tensor):
    if t.dim() != 4:
        raise FaError(1, f"{name}: must be 4-D [B, H, S, d], got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise FaError(1, f"{name}: must be contiguous")
    return tuple(t.shape)


def _on_device(tensors, want_cuda: bool = True):
    """All tensors on one CUDA device (or all on the host for the *_host call)."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise FaError(1, f"tensors: expected one device, got {sorted(map(str, devs))}")
    dev = devs.pop()
    if want_cuda and dev.type != "cuda":
        raise FaError(1, f"tensors: device pointers required, got {dev}")
    if not want_cuda and dev.type != "cpu":
        raise FaError(1, f"tensors: host tensors required, got {dev}")
    return dev


def _dims(Q, K):
    B, H, S_q, d = _shape4("Q", Q)
    Bk, H_kv, S_k, dk = _shape4("K", K)
    if Bk != B or dk != d:
        raise FaError(1, f"K: shape {tuple(K.shape)} incompatible with Q {tuple(Q.shape)}")
    return B, H, H_kv, S_q, S_k, d


def fa_bwd(dO, Q, K, V, O, LSE, scale: float | None = None, causal: bool = False,
           dQ=None, dK=None, dV=None, stream=None, window_size: int = 0, deterministic: bool = False):
    """dQ, dK, dV of attention; see include/fa.h (fa_bwd, and fa_bwd_ex when a
    sliding window or the deterministic mode is asked for)."""
    B, H, H_kv, S_q, S_k, d = _dims(Q, K)
    for name, t, shp in (("dO", dO, Q.shape), ("O", O, Q.shape), ("V", V, K.shape)):
        if tuple(t.shape) != tuple(shp):
            raise FaError(1, f"{name}: expected shape {tuple(shp)}, got {tuple(t.shape)}")
    if tuple(LSE.shape) != (B, H, S_q) or LSE.dtype != torch.float32:
        raise FaError(1, f"LSE: expected float32 shape {(B, H, S_q)}, got {LSE.dtype} {tuple(LSE.shape)}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dev = _on_device((dO, Q, K, V, O, LSE, dQ, dK, dV))
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    for name, t, ref in (("dQ", dQ, Q), ("dK", dK, K), ("dV", dV, V)):
        if t.shape != ref.shape or t.dtype != ref.dtype or not t.is_contiguous():
            raise FaError(1, f"{name}: must be contiguous {ref.dtype} {tuple(ref.shape)}")
    lib = load_library()
    args = (_ptr(dO), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(dQ), _ptr(dK), _ptr(dV),
            B, H, H_kv, S_q, S_k, d, scale, int(bool(causal)))
    with torch.cuda.device(dev):
        if int(window_size) == 0 and not deterministic:
            _check(lib.fa_bwd(*args, _dtype(Q), _stream(stream)))
        else:
            _check(lib.fa_bwd_ex(*args, int(window_size), int(bool(deterministic)), _dtype(Q),
                                 _stream(stream)))
    return dQ, dK, dV


def fa_bwd_noalloc(dO, Q, K, V, O, LSE, dQ, dK, dV, scale: float | None = None,
                   causal: bool = False, stream=None):
    """fa_bwd without any device allocation by the library (fixed 32 MiB scratch);
    outputs must be passed in.  See include/fa.h (fa_bwd_noalloc)."""
    B, H, H_kv, S_q, S_k, d = _dims(Q, K)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dev = _on_device((dO, Q, K, V, O, LSE, dQ, dK, dV))
    with torch.cuda.device(dev):
        _check(load_library().fa_bwd_noalloc(_ptr(dO), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                                             _ptr(dQ), _ptr(dK), _ptr(dV), B, H, H_kv, S_q, S_k, d,
                                             scale, int(bool(causal)), _dtype(Q), _stream(stream)))
    return dQ, dK, dV


def fa_bwd_host(dO, Q, K, V, O, LSE, scale: float | None = None, causal: bool = False,
                dQ=None, dK=None, dV=None, stream=None):
    """fa_bwd on host (CPU, ideally pinned) tensors; copies inside the call."""
    B, H, H_kv, S_q, S_k, d = _dims(Q, K)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _on_device((dO, Q, K, V, O, LSE, dQ, dK, dV), want_cuda=False)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    _check(load_library().fa_bwd_host(_ptr(dO), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                                      _ptr(dQ), _ptr(dK), _ptr(dV), B, H, H_kv, S_q, S_k, d, scale,
                                      int(bool(causal)), _dtype(Q), _stream(stream)))
    return dQ, dK, dV


def fa_bwd_preprocess(dO, O, D=None, stream=None):
    """D = rowsum(dO * O) in fp32, shape [B, H, S_q]."""
    B, H, S_q, d = _shape4("dO", dO)
    if tuple(O.shape) != (B, H, S_q, d):
        raise FaError(1, f"O: expected shape {(B, H, S_q, d)}, got {tuple(O.shape)}")
    dev = _on_device((dO, O, D))
    D = torch.empty((B, H, S_q), dtype=torch.float32, device=dev) if D is None else D
    if tuple(D.shape) != (B, H, S_q) or D.dtype != torch.float32 or not D.is_contiguous():
        raise FaError(1, f"D: must be contiguous float32 {(B, H, S_q)}")
    with torch.cuda.device(dev):
        _check(load_library().fa_bwd_preprocess(_ptr(dO), _ptr(O), _ptr(D), B, H, S_q, d,
                                                _dtype(dO), _stream(stream)))
    return D


def fa_fwd(Q, K, V, scale: float | None = None, causal: bool = False, O=None, LSE=None,
           stream=None, window_size: int = 0):
    """(O, LSE) of attention; see include/fa.h (fa_fwd, fa_fwd_ex for a sliding window)."""
    B, H, H_kv, S_q, S_k, d = _dims(Q, K)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dev = _on_device((Q, K, V, O, LSE))
    O = torch.empty_like(Q) if O is None else O
    LSE = torch.empty((B, H, S_q), dtype=torch.float32, device=dev) if LSE is None else LSE
    lib = load_library()
    args = (_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, H_kv, S_q, S_k, d, scale,
            int(bool(causal)))
    with torch.cuda.device(dev):
        if int(window_size) == 0:
            _check(lib.fa_fwd(*args, _dtype(Q), _stream(stream)))
        else:
            _check(lib.fa_fwd_ex(*args, int(window_size), _dtype(Q), _stream(stream)))
    return O, LSE


def fa_profile(enable: bool) -> None:
    """Start (clearing the record) or stop per-kernel event timing of fa_bwd."""
    _check(load_library().fa_profile(int(bool(enable))))


def fa_profile_read():
    """(ms_preprocess, ms_main, ms_finalize, calls) summed over recorded fa_bwd calls."""
    ms = (ctypes.c_float * 3)()
    n = ctypes.c_int()
    _check(load_library().fa_profile_read(ms, ctypes.byref(n)))
    return float(ms[0]), float(ms[1]), float(ms[2]), int(n.value)


def fa_selftest_timeout(limit_ns: int = 1_000_000, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait that must run out after limit_ns)."""
    _check(load_library().fa_selftest_timeout(int(limit_ns), _stream(stream)))


def fa_check_device(stream=None) -> None:
    """Raise FaError(FA_ERR_TIMEOUT) if a kernel on `stream` recorded a timeout."""
    _check(load_library().fa_check_device(_stream(stream)))
