"""Exact scaled-dot-product attention for training on GB300 (sm_103a).

Thin Python binding over the C ABI of ``libfa_gb300.so`` (declared in
``include/fa.h``): it only turns torch tensors into pointers and sizes, calls
the C function, and raises ``FaError`` on a non-zero status. Every step of the
computation runs in the library's CUDA kernels; there is no fallback. If the
library has not been built, every call raises.

    import attention_fa_fwd_03_gb300 as fa
    fa.fa_fwd(q, k, v, o, lse, scale, causal=True)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, Hq, Tq), dtype=torch.uint8, device="cuda")
    fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, causal=True, workspace=ws)
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["FA_FP16", "FA_BF16", "FaError", "fa_fwd", "fa_bwd", "fa_bwd_preprocess", "fa_bwd_dkv",
           "fa_bwd_dq", "fa_bwd_workspace_size",
           "fa_status_string", "fa_device_status", "fa_abi_version", "fa_selftest_wait_timeout",
           "fa_set_wait_limit_cycles", "library", "library_path"]

FA_FP16 = 0
FA_BF16 = 1
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED_HEAD_DIM",
                3: "FA_ERR_UNSUPPORTED_DTYPE", 4: "FA_ERR_MISALIGNED", 5: "FA_ERR_LAUNCH",
                6: "FA_ERR_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({_status_text(status)})")


def library_path() -> str:
    return os.path.join(_HERE, "libfa_gb300.so")


def library():
    """The loaded C library (ctypes), with argument types declared."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing "
                               "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i,
                               vp, sz, vp]
        lib.fa_bwd.restype = i
        lib.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
        lib.fa_bwd_preprocess.restype = i
        lib.fa_bwd_dkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i,
                                   vp]
        lib.fa_bwd_dkv.restype = i
        lib.fa_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i, vp]
        lib.fa_bwd_dq.restype = i
        lib.fa_bwd_workspace_size.argtypes = [i, i, i]
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i, vp]
        lib.fa_device_status.restype = i
        lib.fa_abi_version.argtypes = []
        lib.fa_abi_version.restype = i
        lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        lib.fa_selftest_wait_timeout.restype = i
        lib.fa_set_wait_limit_cycles.argtypes = [ctypes.c_ulonglong]
        lib.fa_set_wait_limit_cycles.restype = i
        _lib = lib
        return lib


def _status_text(st: int) -> str:
    try:
        return library().fa_status_string(st).decode()
    except Exception:  # library missing while formatting an error
        return "?"


def _check(st: int, what: str) -> None:
    if st != 0:
        raise FaError(st, what)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise FaError(3, f"dtype {t.dtype}")


def _ptr(t) -> int:
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous (row-major [B, H, T, D])")
    return t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fa_abi_version() -> int:
    return library().fa_abi_version()


def fa_status_string(st: int) -> str:
    return library().fa_status_string(st).decode()


def fa_bwd_workspace_size(B: int, Hq: int, Tq: int) -> int:
    return int(library().fa_bwd_workspace_size(B, Hq, Tq))


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool = False, window: int = 0,
           stream=None) -> None:
    """O and LSE for q [B,Hq,Tq,D], k/v [B,Hkv,Tkv,D] (fp16 or bf16, contiguous,
    on the GPU); o [B,Hq,Tq,D] same dtype, lse [B,Hq,Tq] fp32 are written."""
    B, Hq, Tq, D = q.shape
    Hkv, Tkv = k.shape[1], k.shape[2]
    st = library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Tq, Tkv, D,
                          float(scale), int(bool(causal)), int(window), _dtype_code(q),
                          _stream(stream))
    _check(st, "fa_fwd")


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale: float, causal: bool = False,
           window: int = 0, workspace=None, stream=None) -> None:
    """dQ, dK, dV for the forward that produced o and lse. ``workspace`` is a
    device tensor of at least fa_bwd_workspace_size(B, Hq, Tq) bytes."""
    B, Hq, Tq, D = q.shape
    Hkv, Tkv = k.shape[1], k.shape[2]
    if workspace is None:
        raise ValueError("fa_bwd needs a workspace tensor (the library never allocates)")
    nbytes = workspace.numel() * workspace.element_size()
    st = library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                          _ptr(dk), _ptr(dv), B, Hq, Hkv, Tq, Tkv, D, float(scale),
                          int(bool(causal)), int(window), _dtype_code(q), _ptr(workspace),
                          nbytes, _stream(stream))
    _check(st, "fa_bwd")


def _ws_ptr(workspace) -> int:
    if workspace is None:
        raise ValueError("a D-vector workspace tensor is required (the library never allocates)")
    return _ptr(workspace)


def fa_bwd_preprocess(o, do, workspace, stream=None) -> None:
    """D-vector rowsum(dO * O) into ``workspace`` (fp32 [B, Hq, Tq])."""
    B, Hq, Tq, D = o.shape
    st = library().fa_bwd_preprocess(_ptr(o), _ptr(do), _ws_ptr(workspace), B, Hq, Tq, D,
                                     _dtype_code(o), _stream(stream))
    _check(st, "fa_bwd_preprocess")


def fa_bwd_dkv(q, k, v, do, lse, workspace, dk, dv, scale: float, causal: bool = False,
               window: int = 0, stream=None) -> None:
    """dK, dV given the D-vector already in ``workspace``."""
    B, Hq, Tq, D = q.shape
    Hkv, Tkv = k.shape[1], k.shape[2]
    st = library().fa_bwd_dkv(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ws_ptr(workspace),
                              _ptr(dk), _ptr(dv), B, Hq, Hkv, Tq, Tkv, D, float(scale),
                              int(bool(causal)), int(window), _dtype_code(q), _stream(stream))
    _check(st, "fa_bwd_dkv")


def fa_bwd_dq(q, k, v, do, lse, workspace, dq, scale: float, causal: bool = False,
              window: int = 0, stream=None) -> None:
    """dQ given the D-vector already in ``workspace``."""
    B, Hq, Tq, D = q.shape
    Hkv, Tkv = k.shape[1], k.shape[2]
    st = library().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ws_ptr(workspace),
                             _ptr(dq), B, Hq, Hkv, Tq, Tkv, D, float(scale), int(bool(causal)),
                             int(window), _dtype_code(q), _stream(stream))
    _check(st, "fa_bwd_dq")


def fa_selftest_wait_timeout(timeout_ms: int, stream=None) -> None:
    """Launch the library's bounded-wait self-test (see include/fa.h): a wait
    that can never complete gives up after ``timeout_ms``; read the result
    with fa_device_status()."""
    _check(library().fa_selftest_wait_timeout(int(timeout_ms), _stream(stream)),
           "fa_selftest_wait_timeout")


def fa_set_wait_limit_cycles(cycles: int) -> None:
    """Bound (SM clock cycles) of the kernels' ordinary waits for every later
    launch in this process; 0 restores the default. A diagnostic for tests of
    the give-up path (see include/fa.h)."""
    _check(library().fa_set_wait_limit_cycles(int(cycles)), "fa_set_wait_limit_cycles")


def fa_device_status(clear: bool = True, stream=None) -> int:
    """Synchronise ``stream`` and return the device status word (0 = no bounded
    wait gave up). Raises nothing; the caller inspects the bits."""
    bits = ctypes.c_uint(0)
    library().fa_device_status(ctypes.byref(bits), int(bool(clear)), _stream(stream))
    return int(bits.value)
