"""GB300 (sm_103a) exact attention, FlashAttention-style: Python binding of ``libfa.so``.

The functions ``fa_fwd``, ``fa_fwd_ex``, ``fa_bwd``, ``fa_bwd_ex``, ``fa_bwd_workspace_bytes``,
``fa_get_device_status``, ``fa_set_wait_timeout_ns``, ``fa_selftest_wait_timeout`` and
``fa_status_string`` mirror the C ABI in ``include/fa.h`` one to one: they only marshal
arguments (device pointers, strides, sizes, stream handle).  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and loading fails loudly
when the library has not been built.

``forward`` / ``backward`` / ``attention`` are conveniences over the same calls for torch
tensors viewed as [B, H, L, D] with a contiguous last dimension and any other strides (memory
allocation and the current CUDA stream come from torch); queries and keys may differ in length.
``attention_blhd`` takes [B, L, H, D] tensors and ``attention_qkvpacked`` one [B, L, 3, H, D]
tensor, the layouts of the flash_attn_func and flash_attn_qkvpacked_func interfaces the pages
use ("FlashAttention data-flow optimisation", section 4.1, step 3; "AIInfra notes 01: from
TFLOPS to FlashAttention", sections 4.2-4.3).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = ["FaError", "load_library", "library_path", "fa_fwd", "fa_fwd_ex", "fa_bwd", "fa_bwd_ex",
           "fa_bwd_workspace_bytes", "fa_bwd_workspace_bytes_ex", "fa_set_forward_pair",
           "fa_get_device_status",
           "fa_set_wait_timeout_ns",
           "fa_selftest_wait_timeout", "fa_trace_next_call", "fa_launch_count", "fa_status_string",
           "fa_bwd_noalloc", "forward", "backward", "attention", "attention_blhd",
           "attention_qkvpacked", "FaStrides", "fa_decode_paged", "fa_decode_workspace_bytes",
           "decode_paged", "FA_PAGE_TOKENS",
           "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
           "FA_BF16", "FA_FP16"]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_BF16, FA_FP16 = 0, 1
FA_PAGE_TOKENS = 16

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libfa.so")
_lib = None
_lock = threading.Lock()

EXPORTED = ("fa_fwd", "fa_fwd_ex", "fa_bwd", "fa_bwd_ex", "fa_bwd_workspace_bytes",
            "fa_bwd_workspace_bytes_ex", "fa_set_forward_pair", "fa_get_device_status",
            "fa_set_wait_timeout_ns", "fa_selftest_wait_timeout", "fa_trace_next_call",
            "fa_launch_count", "fa_status_string", "fa_bwd_noalloc", "fa_decode_paged",
            "fa_decode_workspace_bytes")


class FaStrides(ctypes.Structure):
    """fa_strides: element strides (batch, head, row) of a [B, H, L, D] operand."""
    _fields_ = [("batch", ctypes.c_int64), ("head", ctypes.c_int64), ("row", ctypes.c_int64)]


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
        d64, u64 = ctypes.c_double, ctypes.c_uint64
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_bytes.restype = sz
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, i, vp]
        lib.fa_bwd.restype = i
        sp = ctypes.POINTER(FaStrides)
        lib.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, sp, i, i, i, i, i, f, i, d64, u64, i, vp]
        lib.fa_fwd_ex.restype = i
        lib.fa_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, sp, i, i, i, i, i, f,
                                  i, d64, u64, i, i, vp]
        lib.fa_bwd_workspace_bytes_ex.argtypes = [i, i, i, i, i]
        lib.fa_bwd_workspace_bytes_ex.restype = sz
        lib.fa_bwd_ex.restype = i
        lib.fa_decode_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_decode_workspace_bytes.restype = sz
        lib.fa_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
        lib.fa_decode_paged.restype = i
        lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i,
                                       vp]
        lib.fa_bwd_noalloc.restype = i
        lib.fa_get_device_status.argtypes = [vp]
        lib.fa_get_device_status.restype = i
        lib.fa_set_forward_pair.argtypes = [i]
        lib.fa_set_forward_pair.restype = i
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


def _strides_array(strides):
    """Sequence of (batch, head, row) element strides -> ctypes array of fa_strides."""
    return (FaStrides * len(strides))(*[FaStrides(*map(int, t)) for t in strides])


def fa_fwd_ex(q, k, v, o, lse, strides, B, H, Lq, Lk, D, scale, causal, dropout_p, seed, dtype,
              stream) -> int:
    """``strides``: four (batch, head, row) tuples for q, k, v, o."""
    return load_library().fa_fwd_ex(q, k, v, o, lse, _strides_array(strides), B, H, Lq, Lk, D,
                                    scale, int(causal), float(dropout_p),
                                    int(seed) & 0xFFFFFFFFFFFFFFFF, dtype, stream)


def fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, strides, B, H, Lq,
              Lk, D, scale, causal, dropout_p, seed, deterministic, dtype, stream) -> int:
    """``strides``: eight (batch, head, row) tuples for q, k, v, o, dout, dq, dk, dv."""
    return load_library().fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace,
                                    workspace_bytes, _strides_array(strides), B, H, Lq, Lk, D,
                                    scale, int(causal), float(dropout_p),
                                    int(seed) & 0xFFFFFFFFFFFFFFFF, int(deterministic), dtype,
                                    stream)


def fa_bwd_workspace_bytes_ex(B, H, Lq, D, deterministic) -> int:
    return int(load_library().fa_bwd_workspace_bytes_ex(B, H, Lq, D, int(deterministic)))


def fa_decode_workspace_bytes(B, H, D, max_pages) -> int:
    return int(load_library().fa_decode_workspace_bytes(B, H, D, max_pages))


def fa_decode_paged(q, k_cache, v_cache, block_tables, seq_lens, o, lse, workspace,
                    workspace_bytes, B, H, D, num_pages, max_pages, scale, dtype, stream) -> int:
    return load_library().fa_decode_paged(q, k_cache, v_cache, block_tables, seq_lens, o, lse,
                                          workspace, workspace_bytes, B, H, D, num_pages,
                                          max_pages, scale, dtype, stream)


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


def fa_set_forward_pair(mode: int) -> int:
    return int(load_library().fa_set_forward_pair(int(mode)))


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


def _view_strides(t, name, shape=None):
    """(batch, head, row) element strides of a CUDA tensor viewed as [B, H, L, D]."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 4:
        raise ValueError(f"{name} must be a [B, H, L, D] view")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.stride(3) != 1:
        raise ValueError(f"{name}: the last (D) dimension must be contiguous")
    return (t.stride(0), t.stride(1), t.stride(2))


def _stream_handle(device) -> int:
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
            dropout_p: float = 0.0, seed: int = 0):
    """O, LSE = attention(q, k, v) for CUDA tensors viewed as [B, H, Lq, D] (q) and
    [B, H, Lk, D] (k, v), bf16 or fp16, with a contiguous last dimension.  O has q's shape (and,
    where torch can keep them, q's strides); LSE is contiguous [B, H, Lq] fp32.  ``dropout_p``
    drops entries of P with the counter-based mask of ``seed`` (``fa_fwd_ex`` in fa.h)."""
    import torch
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    st = [_view_strides(q, "q"), _view_strides(k, "k", (B, H, Lk, D)),
          _view_strides(v, "v", (B, H, Lk, D))]
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty_like(q)
    st.append(_view_strides(o, "out", q.shape))
    l = lse if lse is not None else torch.empty((B, H, Lq), device=q.device, dtype=torch.float32)
    if not l.is_contiguous() or tuple(l.shape) != (B, H, Lq):
        raise ValueError("lse must be a contiguous [B, H, Lq] tensor")
    status = fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), st,
                       B, H, Lq, Lk, D, float(scale), causal, dropout_p, seed, dt,
                       _stream_handle(q.device))
    if status != FA_OK:
        raise FaError("fa_fwd_ex", status)
    return o, l


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
             workspace=None, grads=None, dropout_p: float = 0.0, seed: int = 0,
             deterministic: bool = True):
    """dQ, dK, dV for the forward above (with that forward's ``dropout_p`` and ``seed``).
    ``grads`` optionally gives the three output views (for example the parts of one packed
    gradient tensor); by default they are allocated like q, k, v.  ``deterministic=False``
    lets the library reduce dQ inside the dK/dV pass (D = 64, no dropout; see fa_bwd_ex)."""
    import torch
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    st = [_view_strides(q, "q"), _view_strides(k, "k", (B, H, Lk, D)),
          _view_strides(v, "v", (B, H, Lk, D)), _view_strides(o, "o", q.shape),
          _view_strides(dout, "dout", q.shape)]
    if tuple(lse.shape) != (B, H, Lq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [B, H, Lq] tensor")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ws_bytes = fa_bwd_workspace_bytes_ex(B, H, Lq, D, deterministic)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=q.device, dtype=torch.uint8)
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = grads
    st += [_view_strides(dq, "dq", q.shape), _view_strides(dk, "dk", k.shape),
           _view_strides(dv, "dv", k.shape)]
    status = fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                       workspace.data_ptr(), workspace.numel() * workspace.element_size(), st,
                       B, H, Lq, Lk, D, float(scale), causal, dropout_p, seed, deterministic,
                       dt, _stream_handle(q.device))
    if status != FA_OK:
        raise FaError("fa_bwd_ex", status)
    return dq, dk, dv


def _dropout_seed(dropout_p: float, seed: int | None) -> int:
    """The caller's seed, or for dropout without one a fresh 64-bit seed from torch's default
    generator (the mask itself is drawn on the device from the seed)."""
    if seed is not None or dropout_p == 0.0:
        return 0 if seed is None else int(seed)
    import torch
    return int(torch.randint(0, 2**62, (1,)).item())


def attention(q, k, v, causal: bool = False, scale: float | None = None, dropout_p: float = 0.0,
              seed: int | None = None, deterministic: bool = True):
    """Differentiable attention for torch autograd (forward and backward run in libfa) over
    [B, H, L, D] views (Lq may differ from Lk).  With ``dropout_p`` > 0 the forward and the
    backward regenerate the same dropout mask from ``seed`` (drawn from torch's generator when
    None)."""
    import torch
    seed_ = _dropout_seed(dropout_p, seed)

    class _Attention(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q_, k_, v_):
            o_, lse_ = forward(q_, k_, v_, causal, scale, dropout_p=dropout_p, seed=seed_)
            ctx.save_for_backward(q_, k_, v_, o_, lse_)
            return o_

        @staticmethod
        def backward(ctx, do_):
            q_, k_, v_, o_, lse_ = ctx.saved_tensors
            if do_.stride(-1) != 1:
                do_ = do_.contiguous()
            return backward(q_, k_, v_, o_, lse_, do_, causal, scale, dropout_p=dropout_p,
                            seed=seed_, deterministic=deterministic)

    return _Attention.apply(q, k, v)


def attention_blhd(q, k, v, causal: bool = False, scale: float | None = None,
                   dropout_p: float = 0.0, seed: int | None = None):
    """attention() for [B, L, H, D] tensors (the flash_attn_func layout); returns O as
    [B, Lq, H, D].  No copy: the kernels read and write the [B, L, H, D] memory directly."""
    return attention(q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), causal,
                     scale, dropout_p, seed).transpose(1, 2)


def attention_qkvpacked(qkv, causal: bool = False, scale: float | None = None):
    """attention() for one packed [B, L, 3, H, D] tensor (the flash_attn_qkvpacked_func layout);
    returns O as [B, L, H, D].  Q, K and V are read in place, and the backward writes dQ, dK, dV
    into the three interleaved parts of one packed [B, L, 3, H, D] gradient."""
    import torch

    class _Packed(torch.autograd.Function):
        @staticmethod
        def forward(ctx, qkv_):
            q_, k_, v_ = (qkv_[:, :, i].transpose(1, 2) for i in range(3))
            B, H, L, D = q_.shape
            o_ = torch.empty((B, L, H, D), device=qkv_.device, dtype=qkv_.dtype).transpose(1, 2)
            o_, lse_ = forward(q_, k_, v_, causal, scale, out=o_)
            ctx.save_for_backward(qkv_, o_, lse_)
            return o_.transpose(1, 2)

        @staticmethod
        def backward(ctx, do_):
            qkv_, o_, lse_ = ctx.saved_tensors
            q_, k_, v_ = (qkv_[:, :, i].transpose(1, 2) for i in range(3))
            if do_.stride(-1) != 1:
                do_ = do_.contiguous()
            dqkv = torch.empty_like(qkv_)
            parts = tuple(dqkv[:, :, i].transpose(1, 2) for i in range(3))
            backward(q_, k_, v_, o_, lse_, do_.transpose(1, 2), causal, scale, grads=parts)
            return dqkv

    return _Packed.apply(qkv)


def decode_paged(q, k_cache, v_cache, block_tables, seq_lens, scale: float | None = None,
                 out=None, lse=None, workspace=None):
    """One decode step over a paged cache: q [B, H, D]; k_cache, v_cache
    [num_pages, H, FA_PAGE_TOKENS, D] (bf16 or fp16, contiguous); block_tables [B, max_pages] and
    seq_lens [B] int32 CUDA tensors.  Returns O [B, H, D] and LSE [B, H] (fp32)."""
    import torch
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("seq_lens", seq_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_tables and seq_lens must be int32")
    B, H, D = q.shape
    num_pages = k_cache.shape[0]
    if tuple(k_cache.shape) != (num_pages, H, FA_PAGE_TOKENS, D) or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [num_pages, H, FA_PAGE_TOKENS, D]")
    max_pages = block_tables.shape[1] if block_tables.dim() == 2 else 0
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else torch.empty((B, H), device=q.device, dtype=torch.float32)
    ws_bytes = fa_decode_workspace_bytes(B, H, D, max_pages)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=q.device, dtype=torch.uint8)
    status = fa_decode_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                             block_tables.data_ptr(), seq_lens.data_ptr(), o.data_ptr(),
                             l.data_ptr(), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), B, H, D, num_pages,
                             max_pages, float(scale), dt, _stream_handle(q.device))
    if status != FA_OK:
        raise FaError("fa_decode_paged", status)
    return o, l
