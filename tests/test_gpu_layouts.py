"""CUDA path vs the fp64 oracle for general layouts and lengths, through fa_fwd_ex / fa_bwd_ex.

* [B, L, H, D] tensors (the flash_attn_func layout) and one packed [B, L, 3, H, D] tensor (the
  flash_attn_qkvpacked_func layout), read and written in place through strides, with autograd;
* queries and keys of different lengths, causal rows aligned to the end of the keys (query i
  sees key j iff j <= i + Lk - Lq), including query tiles in which no row, or only some rows,
  see a key (O = 0, LSE = -inf, dQ = 0 there).
"""
import math

import numpy as np
import pytest
import torch

import gpu_helpers as gh
import tiled_attention_08_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gh.require_gpu()


def _draw(shape, gen, dtype):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def _compare_head(oracle, q, k, v, do, o, lse, dq, dk, dv, scale, causal, dtype, raw_o):
    """One head: q, do, o, dq [Lq, D]; k, v, dk, dv [Lk, D]; lse [Lq] (float64 numpy)."""
    o_ref, lse_ref = oracle.forward(q, k, v, scale, causal)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), "rows with LSE = -inf differ"
    assert np.all(o[empty] == 0.0), "O of a row that sees no key"
    err = gh.o_errors(o, o_ref, dtype)
    o_max, o_mean = ((err["o_raw_max"], err["o_raw_mean"]) if raw_o
                     else (err["o_max"], err["o_mean"]))
    assert o_max <= gh.O_MAX_ABS and o_mean <= gh.O_MEAN_ABS, err
    if (~empty).any():
        assert np.max(np.abs(lse[~empty] - lse_ref[~empty])) <= gh.LSE_MAX_ABS
    dq_ref, dk_ref, dv_ref, _ = oracle.backward(q, k, v, do, scale, causal)
    assert np.all(dq[empty] == 0.0), "dQ of a row that sees no key"
    for name, got, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        nrm = np.linalg.norm(ref)
        if nrm < 1e-9:
            assert np.max(np.abs(got)) <= gh.O_MAX_ABS, name
        else:
            assert np.linalg.norm(got - ref) / nrm <= gh.GRAD_REL_FRO, (name, np.linalg.norm(got - ref) / nrm)


RECT = [(Lq, Lk, D, causal, dt)
        for (Lq, Lk) in ((128, 384), (200, 700), (384, 128), (700, 200), (300, 250), (1, 300),
                         (300, 1), (129, 1000))
        for D in (64, 128)
        for causal in (False, True)
        for dt in (torch.bfloat16,)] + \
       [(200, 700, 64, True, torch.float16), (700, 200, 128, True, torch.float16)]


@pytest.mark.parametrize("Lq,Lk,D,causal,dtype", RECT, ids=lambda x: str(x).replace("torch.", ""))
def test_rectangular_lengths(oracle_mod, Lq, Lk, D, causal, dtype):
    """Lq != Lk, contiguous [B,H,L,D], every head in full: several query and key tiles, ragged
    tails, and (Lq > Lk, causal) query tiles with no visible key or only some rows seeing one."""
    B, H = 2, 2
    g = torch.Generator().manual_seed(Lq * 31 + Lk * 7 + D + int(causal))
    q, do = _draw((B, H, Lq, D), g, dtype), _draw((B, H, Lq, D), g, dtype)
    k, v = _draw((B, H, Lk, D), g, dtype), _draw((B, H, Lk, D), g, dtype)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.forward(qd, kd, vd, causal, scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    for b in range(B):
        for h in range(H):
            _compare_head(oracle_mod, *(gh.f64(t[b, h]) for t in (q, k, v, do, o, lse, dq, dk, dv)),
                          scale, causal, dtype, raw_o=False)


@pytest.mark.parametrize("L,D,causal", [(384, 128, True), (300, 64, False), (1000, 64, True)])
def test_blhd_layout_autograd(oracle_mod, L, D, causal):
    """[B, L, H, D] tensors through attention_blhd and torch autograd: the kernels read q, k, v
    and write O, dQ, dK, dV in that layout (strides), no copies."""
    B, H = 2, 3
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(L + D)
    q, k, v, do = (_draw((B, L, H, D), g, torch.bfloat16) for _ in range(4))
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    o = fa.attention_blhd(qd, kd, vd, causal)
    assert o.shape == (B, L, H, D)
    o.backward(do.to(dev))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        for h in range(H):
            f = [gh.f64(t[b, :, h]) for t in (q, k, v, do)]
            _, lse_ref = oracle_mod.forward(f[0], f[1], f[2], scale, causal)  # (LSE: not returned)
            _compare_head(oracle_mod, *f, gh.f64(o[b, :, h]), lse_ref,
                          gh.f64(qd.grad[b, :, h]), gh.f64(kd.grad[b, :, h]),
                          gh.f64(vd.grad[b, :, h]), scale, causal, torch.bfloat16,
                          raw_o=L >= 128)


@pytest.mark.parametrize("L,D,causal,dtype", [(384, 128, True, torch.bfloat16),
                                              (257, 64, False, torch.float16),
                                              (2048, 128, True, torch.bfloat16)])
def test_qkvpacked_layout_autograd(oracle_mod, L, D, causal, dtype):
    """One packed [B, L, 3, H, D] tensor through attention_qkvpacked: Q, K, V read in place and
    dQ, dK, dV written into the three interleaved parts of one packed gradient tensor."""
    B, H = 1, 4
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(L * 3 + D)
    qkv = _draw((B, L, 3, H, D), g, dtype)
    do = _draw((B, L, H, D), g, dtype)
    x = qkv.to(dev).requires_grad_(True)
    o = fa.attention_qkvpacked(x, causal)
    assert o.shape == (B, L, H, D)
    o.backward(do.to(dev))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    assert x.grad.shape == qkv.shape
    scale = 1.0 / math.sqrt(D)
    for h in range(H):
        q, k, v = (gh.f64(qkv[0, :, i, h]) for i in range(3))
        _, lse_ref = oracle_mod.forward(q, k, v, scale, causal)
        _compare_head(oracle_mod, q, k, v, gh.f64(do[0, :, h]), gh.f64(o[0, :, h]), lse_ref,
                      *(gh.f64(x.grad[0, :, i, h]) for i in range(3)), scale, causal, dtype,
                      raw_o=True)


def test_blhd_matches_contiguous_bitwise():
    """The same problem in [B,H,L,D] and in [B,L,H,D] gives the same bits: strides change only
    where the tiles are read and written."""
    B, H, L, D = 2, 4, 640, 128
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(77)
    q, k, v, do = (_draw((B, L, H, D), g, torch.bfloat16).to(dev) for _ in range(4))
    a = fa.forward(*(t.transpose(1, 2) for t in (q, k, v)), True)
    ga = fa.backward(*(t.transpose(1, 2) for t in (q, k, v)), a[0], a[1], do.transpose(1, 2), True)
    c = [t.transpose(1, 2).contiguous() for t in (q, k, v, do)]
    b = fa.forward(c[0], c[1], c[2], True)
    gb = fa.backward(c[0], c[1], c[2], b[0], b[1], c[3], True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for x, y in zip(ga, gb):
        assert torch.equal(x, y)


def test_calls_from_new_host_threads(oracle_mod):
    """Forward and backward issued from a host thread that has made no CUDA call of its own (as
    torch's autograd engine issues the backward from its worker thread, which need not have a
    current context) launch and give the same bits as from the main thread.  The thread touches
    nothing but the C ABI: buffers and the stream handle come from the main thread."""
    import threading

    B, H, L, D = 1, 2, 300, 128
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(5)
    q, k, v, do = (_draw((B, H, L, D), g, torch.bfloat16).to(dev) for _ in range(4))
    ref_o, ref_lse = fa.forward(q, k, v, True)
    ref = fa.backward(q, k, v, ref_o, ref_lse, do, True)
    outs = [torch.empty_like(q) for _ in range(4)]  # o, dq, dk, dv
    lse = torch.empty_like(ref_lse)
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, L, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    torch.cuda.synchronize()
    status = []

    def work():
        scale = 1.0 / math.sqrt(D)
        status.append(fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), outs[0].data_ptr(),
                                lse.data_ptr(), B, H, L, D, scale, 1, fa.FA_BF16, stream))
        status.append(fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), outs[0].data_ptr(),
                                do.data_ptr(), lse.data_ptr(), outs[1].data_ptr(),
                                outs[2].data_ptr(), outs[3].data_ptr(), ws.data_ptr(), ws_bytes,
                                B, H, L, D, scale, 1, fa.FA_BF16, stream))

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert status == [fa.FA_OK, fa.FA_OK], [fa.fa_status_string(x) for x in status]
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(stream) == fa.FA_OK
    for a, b in zip([outs[0], lse] + outs[1:], [ref_o, ref_lse] + list(ref)):
        assert torch.equal(a, b)
