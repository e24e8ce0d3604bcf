"""fp64 CPU oracle for exact scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package; the product path (``tiled_attention_08_gb300``)
never does, and shares no code with it.

* ``forward`` / ``backward`` call the plain C definition in ``oracle.c`` (materialised S
  and P in fp64; see the header of that file for the formulas and their sources).
* ``probs`` returns the full probability matrix of one head.
* ``decode_paged`` is one decode step over a paged key/value cache (one new query row per
  sequence attending to its cached tokens, gathered through the block table).
* ``online_forward`` is a second, independent fp64 routine in numpy that runs the
  streaming recurrence the pages describe ("FlashAttention data-flow optimisation: MI50
  memory and bandwidth bottlenecks", section 2.2, first layer: Q split into row blocks
  and K/V into column blocks; second layer: a running row max and running sum of
  exponentials updated as each column block arrives, the partial output rescaled when the
  max grows, and the row normalised once every block has been seen).  It is used only to
  check that the streaming recurrence equals the two-pass definition on tiny inputs.

Parity pins: every function here is pinned in ``tests/test_oracle_pins.py`` against closed
forms, invariants, finite differences and an independent library implementation; no
function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (-O2 -fopenmp) into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            dp = ctypes.POINTER(ctypes.c_double)
            L = ctypes.c_long
            u64 = ctypes.c_ulonglong
            lib.oracle_fwd_f64.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, ctypes.c_double,
                                           ctypes.c_int, L, ctypes.c_double, u64]
            lib.oracle_fwd_f64.restype = ctypes.c_int
            lib.oracle_bwd_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, L, L, L, L, L,
                                           ctypes.c_double, ctypes.c_int, L, ctypes.c_double,
                                           u64]
            u32p = ctypes.POINTER(ctypes.c_uint)
            lib.oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_bwd_f64.restype = ctypes.c_int
            lib.oracle_probs_f64.argtypes = [dp, dp, dp, L, L, L, ctypes.c_double,
                                             ctypes.c_int]
            lib.oracle_probs_f64.restype = ctypes.c_int
            ip = ctypes.POINTER(ctypes.c_int)
            lib.oracle_decode_paged_f64.argtypes = [dp, dp, dp, ip, ip, dp, dp, L, L, L, L, L, L,
                                                    ctypes.c_double]
            lib.oracle_decode_paged_f64.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (``OMP_NUM_THREADS`` or all cores)."""
    return int(_load().oracle_num_threads())


def _f64(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _as4d(a: np.ndarray) -> tuple[np.ndarray, bool]:
    if a.ndim == 2:
        return a[None, None], True
    if a.ndim != 4:
        raise ValueError("expected [B,H,L,D] or [L,D]")
    return a, False


def _check_qkv(q, k, v, extra=()):
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Lq,D] and k, v [B,H,Lk,D] must agree in B, H and D")
    for a in extra:
        if a.shape != q.shape:
            raise ValueError("dO must have the shape of q")


def forward(q, k, v, scale: float, causal: bool, block_doubles: int = 0, dropout_p: float = 0.0,
            seed: int = 0):
    """O [B,H,Lq,D] and LSE [B,H,Lq] (natural log) in fp64 for q [B,H,Lq,D] and k, v
    [B,H,Lk,D] (Lq may differ from Lk; causal rows are aligned to the end of the keys).  Also
    accepts [L,D] inputs.  ``dropout_p`` > 0 drops entries of P (Philox-4x32-10 keyed by
    ``seed``; see oracle.c)."""
    q, sq = _as4d(_f64(q))
    k, _ = _as4d(_f64(k))
    v, _ = _as4d(_f64(v))
    _check_qkv(q, k, v)
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    o = np.empty_like(q)
    lse = np.empty((B, H, Lq), dtype=np.float64)
    rc = _load().oracle_fwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Lq, Lk, D,
                                float(scale), int(bool(causal)), int(block_doubles),
                                float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF)
    if rc != 0:
        raise RuntimeError(f"oracle_fwd_f64 failed with code {rc}")
    if sq:
        return o[0, 0], lse[0, 0]
    return o, lse


def backward(q, k, v, do, scale: float, causal: bool, block_doubles: int = 0,
             dropout_p: float = 0.0, seed: int = 0):
    """dQ [B,H,Lq,D], dK, dV [B,H,Lk,D] and Delta [B,H,Lq] in fp64.  Also accepts [L,D]
    inputs."""
    q, sq = _as4d(_f64(q))
    k, _ = _as4d(_f64(k))
    v, _ = _as4d(_f64(v))
    do, _ = _as4d(_f64(do))
    _check_qkv(q, k, v, (do,))
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(k)
    delta = np.empty((B, H, Lq), dtype=np.float64)
    rc = _load().oracle_bwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(delta), B, H, Lq, Lk, D, float(scale), int(bool(causal)),
                                int(block_doubles), float(dropout_p),
                                int(seed) & 0xFFFFFFFFFFFFFFFF)
    if rc != 0:
        raise RuntimeError(f"oracle_bwd_f64 failed with code {rc}")
    if sq:
        return dq[0, 0], dk[0, 0], dv[0, 0], delta[0, 0]
    return dq, dk, dv, delta


def probs(q, k, scale: float, causal: bool) -> np.ndarray:
    """The probability matrix P [Lq,Lk] of one head (q: [Lq,D], k: [Lk,D])."""
    q = _f64(q)
    k = _f64(k)
    Lq, D = q.shape
    Lk = k.shape[0]
    p = np.empty((Lq, Lk), dtype=np.float64)
    rc = _load().oracle_probs_f64(_ptr(q), _ptr(k), _ptr(p), Lq, Lk, D, float(scale),
                                  int(bool(causal)))
    if rc != 0:
        raise RuntimeError(f"oracle_probs_f64 failed with code {rc}")
    return p


def online_forward(q, k, v, scale: float, causal: bool, block_q: int, block_k: int):
    """Streaming-softmax forward of one head in fp64, block by block (tiny inputs only).

    Follows the data-flow page's section 2.2: for every row block of Q, the column blocks
    of K/V arrive one at a time; each row keeps a running max ``m`` and a running sum
    ``l`` of exponentials, and the partial output is rescaled by exp(m_old - m_new)
    whenever the max grows.  Rows are normalised once all column blocks have been seen.
    Returns (O [L,D], LSE [L]).
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    L, D = q.shape
    o = np.zeros((L, D))
    lse = np.zeros(L)
    for r0 in range(0, L, block_q):
        r1 = min(L, r0 + block_q)
        rows = r1 - r0
        m = np.full(rows, -np.inf)
        l = np.zeros(rows)
        acc = np.zeros((rows, D))
        for c0 in range(0, L, block_k):
            c1 = min(L, c0 + block_k)
            s = scale * (q[r0:r1] @ k[c0:c1].T)
            if causal:
                qi = np.arange(r0, r1)[:, None]
                kj = np.arange(c0, c1)[None, :]
                s = np.where(kj > qi, -np.inf, s)
            blk_max = s.max(axis=1)
            m_new = np.maximum(m, blk_max)
            # A row that has seen no visible key yet keeps m = -inf; its factors are 0.
            safe = np.where(np.isneginf(m_new), 0.0, m_new)
            p = np.exp(s - safe[:, None])
            alpha = np.where(np.isneginf(m), 0.0, np.exp(m - safe))
            l = alpha * l + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ v[c0:c1]
            m = m_new
        o[r0:r1] = acc / l[:, None]
        lse[r0:r1] = m + np.log(l)
    return o, lse


def decode_paged(q, k_cache, v_cache, block_tables, seq_lens, scale: float):
    """O [B,H,D] and LSE [B,H] of one decode step over a paged cache, in fp64.

    q: [B,H,D]; k_cache, v_cache: [num_pages, H, page, D]; block_tables: [B, max_pages] ints;
    seq_lens: [B] ints (cached tokens per sequence, the newest included)."""
    q = _f64(q)
    kc = _f64(k_cache)
    vc = _f64(v_cache)
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    B, H, D = q.shape
    num_pages, Hc, page, Dc = kc.shape
    if Hc != H or Dc != D or vc.shape != kc.shape or bt.shape[0] != B or sl.shape != (B,):
        raise ValueError("shapes of q, the caches, the block table and seq_lens disagree")
    o = np.empty_like(q)
    lse = np.empty((B, H), dtype=np.float64)
    ip = ctypes.POINTER(ctypes.c_int)
    rc = _load().oracle_decode_paged_f64(_ptr(q), _ptr(kc), _ptr(vc), bt.ctypes.data_as(ip),
                                         sl.ctypes.data_as(ip), _ptr(o), _ptr(lse), B, H, D,
                                         num_pages, page, bt.shape[1], float(scale))
    if rc != 0:
        raise RuntimeError(f"oracle_decode_paged_f64 failed with code {rc}")
    return o, lse


def philox4x32_10(counter, key):
    """The four 32-bit output words of Philox-4x32-10 for a 4-word counter and 2-word key."""
    c = (ctypes.c_uint * 4)(*[int(x) & 0xFFFFFFFF for x in counter])
    k = (ctypes.c_uint * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    out = (ctypes.c_uint * 4)()
    _load().oracle_philox4x32_10(c, k, out)
    return [int(x) for x in out]
