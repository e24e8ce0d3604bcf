"""GB300 (sm_103a) exact attention, FlashAttention-style: Python binding of ``libfa.so``.

The functions ``fa_fwd``, ``fa_bwd``, ``fa_bwd_workspace_bytes``, ``fa_get_device_status``,
``fa_set_wait_timeout_ns``, ``fa_selftest_wait_timeout`` and ``fa_status_string`` mirror the C
ABI in ``include/fa.h`` one to one: they only marshal arguments (device pointers, sizes,
stream handle).  Every step of the computation runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback, and loading fails loudly when the library has not been built.

``forward`` / ``backward`` / ``attention`` are conveniences over the same calls for torch
tensors of shape [B, H, L, D] (memory allocation and the current CUDA stream come from torch).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = ["FaError", "load_library", "library_path", "fa_fwd", "fa_bwd",
           "fa_bwd_workspace_bytes", "fa_get_device_status", "fa_set_wait_timeout_ns",
           "fa_selftest_wait_timeout", "fa_trace_next_call", "fa_launch_count", "fa_status_string",
           "fa_bwd_noalloc", "forward", "backward", "attention",
           "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
           "FA_BF16", "FA_FP16"]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_BF16, FA_FP16 = 0, 1

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libfa.so")
_lib = None
_lock = threading.Lock()

EXPORTED = ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_get_device_status",
            "fa_set_wait_timeout_ns", "fa_selftest_wait_timeout", "fa_trace_next_call",
            "fa_launch_count", "fa_status_string", "fa_bwd_noalloc")


class FaError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} failed: {fa_status_string(status)} ({status})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Loads the in-tree libfa.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libfa.so not built ({_LIB_PATH}); run "
                               "`python -m tiled_attention_08_gb300.build` first")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_bytes.restype = sz
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, i, vp]
        lib.fa_bwd.restype = i
        lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i,
                                       vp]
        lib.fa_bwd_noalloc.restype = i
        lib.fa_get_device_status.argtypes = [vp]
        lib.fa_get_device_status.restype = i
        lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.fa_set_wait_timeout_ns.restype = i
        lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.fa_selftest_wait_timeout.restype = i
        lib.fa_trace_next_call.argtypes = [ctypes.POINTER(ctypes.c_void_p), i]
        lib.fa_trace_next_call.restype = i
        lib.fa_launch_count.argtypes = []
        lib.fa_launch_count.restype = ctypes.c_uint64
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


# ---------------------------------------------------------------------------------------
# One-to-one wrappers of the C ABI (raw pointers as ints, stream as an int handle).
# ---------------------------------------------------------------------------------------
def fa_fwd(q, k, v, o, lse, B, H, L, D, scale, causal, dtype, stream) -> int:
    return load_library().fa_fwd(q, k, v, o, lse, B, H, L, D, scale, int(causal), dtype, stream)


def fa_bwd_workspace_bytes(B, H, L, D) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, L, D))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, L, D, scale,
           causal, dtype, stream) -> int:
    return load_library().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                                 B, H, L, D, scale, int(causal), dtype, stream)


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, L, D, scale, causal, dtype,
                   stream) -> int:
    """fa_bwd without a caller workspace, for callers that cannot allocate device memory: the
    scratch comes from a fixed 16 MiB array compiled into the library (see include/fa.h)."""
    return load_library().fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, L, D, scale,
                                         int(causal), dtype, stream)


def fa_get_device_status(stream) -> int:
    return load_library().fa_get_device_status(stream)


def fa_set_wait_timeout_ns(ns: int) -> int:
    return load_library().fa_set_wait_timeout_ns(int(ns))


def fa_selftest_wait_timeout(ns: int, stream) -> int:
    return load_library().fa_selftest_wait_timeout(int(ns), stream)


def fa_trace_next_call(events, n_pairs: int) -> int:
    """``events``: sequence of 2*n_pairs raw cudaEvent_t handles (ints)."""
    arr = (ctypes.c_void_p * max(1, len(events)))(*[ctypes.c_void_p(int(e)) for e in events])
    return load_library().fa_trace_next_call(arr, n_pairs)


def fa_launch_count() -> int:
    return int(load_library().fa_launch_count())


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


# ---------------------------------------------------------------------------------------
# torch conveniences
# ---------------------------------------------------------------------------------------
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"unsupported dtype {t.dtype}; expected bfloat16 or float16")


def _check(t, name, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous [B,H,L,D]")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream_handle(device) -> int:
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None):
    """O, LSE = attention(q, k, v) for contiguous CUDA tensors [B,H,L,D] (bf16 or fp16)."""
    import torch
    _check(q, "q")
    _check(k, "k", q.shape)
    _check(v, "v", q.shape)
    B, H, L, D = q.shape
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else torch.empty((B, H, L), device=q.device, dtype=torch.float32)
    st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, L, D,
                float(scale), causal, dt, _stream_handle(q.device))
    if st != FA_OK:
        raise FaError("fa_fwd", st)
    return o, l


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
             workspace=None):
    """dQ, dK, dV for the forward above (same shapes and dtype as q)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check(t, name, q.shape)
    B, H, L, D = q.shape
    _check(lse, "lse", (B, H, L))
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ws_bytes = fa_bwd_workspace_bytes(B, H, L, D)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=q.device, dtype=torch.uint8)
    dq = torch.empty_like(q)
    dk = torch.empty_like(q)
    dv = torch.empty_like(q)
    st = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                workspace.numel() * workspace.element_size(), B, H, L, D, float(scale), causal, dt,
                _stream_handle(q.device))
    if st != FA_OK:
        raise FaError("fa_bwd", st)
    return dq, dk, dv


def attention(q, k, v, causal: bool = False, scale: float | None = None):
    """Differentiable attention for torch autograd (forward and backward run in libfa)."""
    import torch

    class _Attention(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q_, k_, v_):
            o_, lse_ = forward(q_, k_, v_, causal, scale)
            ctx.save_for_backward(q_, k_, v_, o_, lse_)
            return o_

        @staticmethod
        def backward(ctx, do_):
            q_, k_, v_, o_, lse_ = ctx.saved_tensors
            return backward(q_, k_, v_, o_, lse_, do_.contiguous(), causal, scale)

    return _Attention.apply(q, k, v)
