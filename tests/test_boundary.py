"""The C-ABI boundary on the host: symbols, argument checks, status strings (no GPU work).

Every call below is rejected (or is empty) before the library touches the CUDA runtime, so
these run on a machine without a GPU.
"""
import ctypes
import os
import re

import pytest

import tiled_attention_08_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")
A = 0x100000  # fake, 16-byte aligned device addresses: never dereferenced by these calls
MB = 1 << 20


@pytest.fixture(scope="module")
def lib():
    from tiled_attention_08_gb300 import build
    build.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_fwd_ex", "fa_bwd_ex", "fa_bwd_workspace_bytes",
              "fa_get_device_status", "fa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libfa.so does not export {name}"
    assert set(declared_functions()) == set(fa.EXPORTED)


def test_status_strings(lib):
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(1) == "FA_ERR_INVALID_ARG"
    assert fa.fa_status_string(2) == "FA_ERR_UNSUPPORTED"
    assert fa.fa_status_string(3) == "FA_ERR_CUDA"
    assert fa.fa_status_string(4) == "FA_ERR_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


def _fwd(B=1, H=2, L=256, D=64, scale=0.125, causal=0, dtype=0, q=A, k=A + MB, v=A + 2 * MB,
         o=A + 3 * MB, lse=A + 4 * MB):
    return fa.fa_fwd(q, k, v, o, lse, B, H, L, D, scale, causal, dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=2), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(B=-1), fa.FA_ERR_INVALID_ARG),
    (dict(L=-5), fa.FA_ERR_INVALID_ARG),
    (dict(D=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(D=256), fa.FA_ERR_UNSUPPORTED),
    (dict(B=1 << 20, H=1 << 12), fa.FA_ERR_UNSUPPORTED),
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(v=A + 2 * MB + 8), fa.FA_ERR_INVALID_ARG),       # misaligned
    (dict(o=A + MB + 64), fa.FA_ERR_INVALID_ARG),          # o overlaps k
    (dict(lse=A + 3 * MB + 32), fa.FA_ERR_INVALID_ARG),    # lse overlaps o
    (dict(L=0), fa.FA_OK),                                 # empty: nothing to do
    (dict(B=0), fa.FA_OK),
    (dict(L=0, q=0, k=0, v=0, o=0, lse=0), fa.FA_OK),
], ids=lambda x: str(x))
def test_forward_argument_checks(lib, kw, status):
    assert _fwd(**kw) == status


def test_workspace_size(lib):
    # two fp32 vectors per head, padded to whole 128-row tiles, and 16 bytes of work counters
    assert fa.fa_bwd_workspace_bytes(2, 3, 200, 64) == 2 * 6 * 256 * 4 + 16
    assert fa.fa_bwd_workspace_bytes(1, 1, 128, 128) == 2 * 128 * 4 + 16
    assert fa.fa_bwd_workspace_bytes(1, 1, 0, 128) == 0
    assert fa.fa_bwd_workspace_bytes(1, 1, 128, 96) == 0
    assert fa.fa_bwd_workspace_bytes(-1, 1, 128, 64) == 0


def _bwd(B=1, H=2, L=256, D=64, causal=1, dtype=0, ws_bytes=None, **ptrs):
    p = dict(q=A, k=A + MB, v=A + 2 * MB, o=A + 3 * MB, do=A + 4 * MB, lse=A + 5 * MB,
             dq=A + 6 * MB, dk=A + 7 * MB, dv=A + 8 * MB, ws=A + 9 * MB)
    p.update(ptrs)
    if ws_bytes is None:
        ws_bytes = fa.fa_bwd_workspace_bytes(B, H, L, D)
    return fa.fa_bwd(p["q"], p["k"], p["v"], p["o"], p["do"], p["lse"], p["dq"], p["dk"], p["dv"],
                     p["ws"], ws_bytes, B, H, L, D, 0.125, causal, dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=5), fa.FA_ERR_INVALID_ARG),
    (dict(D=32), fa.FA_ERR_UNSUPPORTED),
    (dict(ws_bytes=16), fa.FA_ERR_INVALID_ARG),
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),
    (dict(do=0), fa.FA_ERR_INVALID_ARG),
    (dict(dq=A + 6 * MB + 4), fa.FA_ERR_INVALID_ARG),      # misaligned
    (dict(dk=A + 6 * MB + 4096), fa.FA_ERR_INVALID_ARG),   # dk overlaps dq
    (dict(dv=A + 16), fa.FA_ERR_INVALID_ARG),              # dv overlaps q
    (dict(ws=A + 5 * MB), fa.FA_ERR_INVALID_ARG),          # workspace overlaps lse
    (dict(L=0), fa.FA_OK),
], ids=lambda x: str(x))
def test_backward_argument_checks(lib, kw, status):
    assert _bwd(**kw) == status


def _fwd_ex(strides=None, B=1, H=2, Lq=256, Lk=256, D=64, dropout_p=0.0, **ptrs):
    p = dict(q=A, k=A + MB, v=A + 2 * MB, o=A + 3 * MB, lse=A + 4 * MB)
    p.update(ptrs)
    c = (H * Lq * D, Lq * D, D)
    ck = (H * Lk * D, Lk * D, D)
    st = strides or [c, ck, ck, c]
    return fa.fa_fwd_ex(p["q"], p["k"], p["v"], p["o"], p["lse"], st, B, H, Lq, Lk, D, 0.125, 1,
                        dropout_p, 7, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(strides=[(512 * 64, 256 * 64, 60)] + [(512 * 64, 256 * 64, 64)] * 3),
     fa.FA_ERR_INVALID_ARG),                                           # row stride not 8k
    (dict(strides=[(512 * 64, 0, 64)] * 4), fa.FA_ERR_INVALID_ARG),    # zero head stride, H = 2
    (dict(strides=[(-8, 256 * 64, 64)] * 4), fa.FA_ERR_INVALID_ARG),   # negative stride
    (dict(Lk=0), fa.FA_ERR_UNSUPPORTED),                               # queries, no key
    (dict(Lq=0), fa.FA_OK),                                            # no query: nothing to do
    (dict(o=A + 2 * MB + 4096), fa.FA_ERR_INVALID_ARG),               # o inside v's extent
    # [B,L,H,D] views whose extents overlap: o would be read as k
    (dict(strides=[(256 * 2 * 64, 64, 2 * 64)] * 4, o=A + MB), fa.FA_ERR_INVALID_ARG),
    (dict(dropout_p=1.0), fa.FA_ERR_INVALID_ARG),                      # nothing would be kept
    (dict(dropout_p=-0.25), fa.FA_ERR_INVALID_ARG),
    (dict(dropout_p=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(dropout_p=0.5, Lq=0), fa.FA_OK),                             # valid p, empty problem
], ids=lambda x: str(x)[:60])
def test_forward_ex_argument_checks(lib, kw, status):
    assert _fwd_ex(**kw) == status


def test_backward_ex_refuses_one_sided_empty_and_overlapping_outputs(lib):
    B, H, L, D = 1, 2, 256, 64
    c = (H * L * D, L * D, D)
    p = [A + i * MB for i in range(10)]
    ws = fa.fa_bwd_workspace_bytes(B, H, L, D)

    def call(strides, Lq=L, Lk=L, dropout_p=0.0, deterministic=1, **kw):
        q = dict(zip(("q", "k", "v", "o", "do", "lse", "dq", "dk", "dv", "ws"), p))
        q.update(kw)
        return fa.fa_bwd_ex(q["q"], q["k"], q["v"], q["o"], q["do"], q["lse"], q["dq"], q["dk"],
                            q["dv"], q["ws"], ws, strides, B, H, Lq, Lk, D, 0.125, 1, dropout_p,
                            7, deterministic, 0, None)

    assert call([c] * 8, Lq=0, Lk=0) == fa.FA_OK
    assert call([c] * 8, dropout_p=1.0) == fa.FA_ERR_INVALID_ARG
    assert call([c] * 8, dropout_p=float("inf")) == fa.FA_ERR_INVALID_ARG
    assert call([c] * 8, deterministic=2) == fa.FA_ERR_INVALID_ARG
    # dQ by reduction needs the accumulator: the deterministic-size workspace is too small
    assert call([c] * 8, deterministic=0) == fa.FA_ERR_INVALID_ARG
    assert call([c] * 8, Lq=0) == fa.FA_ERR_UNSUPPORTED
    assert call([c] * 8, Lk=0) == fa.FA_ERR_UNSUPPORTED
    # dk inside dq's extent with contiguous strides: not the interleaved parts of a packed tensor
    assert call([c] * 8, dk=p[6] + 4096) == fa.FA_ERR_INVALID_ARG
    # packed [B,L,3,H,D] strides but dk placed on top of dq's heads: overlapping elements
    pk = (L * 3 * H * D, D, 3 * H * D)
    assert call([c] * 5 + [pk] * 3, dk=p[6] + 64 * 2) == fa.FA_ERR_INVALID_ARG


def test_decode_workspace_and_argument_checks(lib):
    # Enough (sequence, head) pairs: one CTA each, no workspace.  Few: splits need one.
    assert fa.fa_decode_workspace_bytes(256, 32, 128, 256) == 0
    assert fa.fa_decode_workspace_bytes(1, 2, 128, 188) == 1 * 2 * 188 * (128 + 1) * 4
    assert fa.fa_decode_workspace_bytes(1, 2, 96, 10) == 0  # unsupported head size
    p = [A + i * MB for i in range(8)]

    def call(B=2, H=2, D=64, num_pages=10, max_pages=4, dtype=0, ws_bytes=1 << 20, **kw):
        q = dict(zip(("q", "kc", "vc", "bt", "sl", "o", "lse", "ws"), p))
        q.update(kw)
        return fa.fa_decode_paged(q["q"], q["kc"], q["vc"], q["bt"], q["sl"], q["o"], q["lse"],
                                  q["ws"], ws_bytes, B, H, D, num_pages, max_pages, 0.125, dtype,
                                  None)

    assert call(dtype=3) == fa.FA_ERR_INVALID_ARG
    assert call(D=96) == fa.FA_ERR_UNSUPPORTED
    assert call(B=70000) == fa.FA_ERR_UNSUPPORTED
    assert call(B=0) == fa.FA_OK
    assert call(q=0) == fa.FA_ERR_INVALID_ARG
    assert call(bt=0) == fa.FA_ERR_INVALID_ARG
    assert call(o=A + 8) == fa.FA_ERR_INVALID_ARG             # o overlaps q, misaligned
    assert call(o=p[1] + 64) == fa.FA_ERR_INVALID_ARG         # o inside the key cache
    assert call(lse=p[5] + 16) == fa.FA_ERR_INVALID_ARG       # lse overlaps o
    assert call(B=1, H=1, max_pages=64, ws_bytes=16) == fa.FA_ERR_INVALID_ARG  # workspace short


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "_LIB_PATH", str(tmp_path / "missing" / "libfa.so"))
    with pytest.raises(RuntimeError, match="not built"):
        fa.load_library()


def test_product_package_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "tiled_attention_08_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "liboracle" not in text and "oracle.c" not in text, f


def test_backward_workspace_sizes(lib):
    B, H, L = 2, 3, 300
    Lp = 384
    counters = 16  # work counters of the persistent passes, at the end
    for D in (64, 128):
        assert fa.fa_bwd_workspace_bytes(B, H, L, D) == 2 * B * H * Lp * 4 + counters
        assert fa.fa_bwd_workspace_bytes_ex(B, H, L, D, 1) == 2 * B * H * Lp * 4 + counters
    # dQ by reduction (D = 64 only): the fp32 accumulator [B*H, Lqpad, D] follows the vectors
    assert (fa.fa_bwd_workspace_bytes_ex(B, H, L, 64, 0) ==
            2 * B * H * Lp * 4 + B * H * Lp * 64 * 4 + counters)
    assert fa.fa_bwd_workspace_bytes_ex(B, H, L, 128, 0) == 2 * B * H * Lp * 4 + counters
    assert fa.fa_bwd_workspace_bytes_ex(B, H, L, 64, 2) == 0
    assert fa.fa_bwd_workspace_bytes_ex(B, H, 0, 64, 0) == 0
