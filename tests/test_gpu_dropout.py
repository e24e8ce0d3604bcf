"""CUDA path vs the fp64 oracle under dropout on P (flash_attn_func's dropout_p, "FlashAttention
data-flow optimisation", section 4.1, step 3), through fa_fwd_ex / fa_bwd_ex.

Both sides draw the mask from the same counter-based generator (Philox-4x32-10, Salmon et al.,
SC 2011): entry (i, j) of head bh = b*H + h is kept iff word j % 4 of the block at counter
(j / 4, i, bh, 0) under the 64-bit seed is at least floor(p * 2^32).  So the comparison is exact
in the mask and within the usual tolerances in the values:

* the mask itself, bit for bit: with V = I (Lk = D) the forward's O is P o Z, zero exactly where
  an entry is dropped, and with dO = I (Lq = D) the backward's dV is (P o Z)^T, which exposes
  the dK/dV kernel's transposed mask the same way;
* O, LSE, dQ, dK, dV over whole [B, H, L, D] problems (the mask depends on the head index),
  several tiles, ragged tails, causal and not, Lq != Lk with rows that see no key;
* a tiny p runs the dropout kernels with nothing dropped and a keep factor that rounds to 1:
  bit for bit the result of the kernels without dropout;
* the same seed gives the same bits, another seed another mask, and autograd carries the seed
  from the forward to the backward.
"""
import math

import numpy as np
import pytest
import torch

import gpu_helpers as gh
import tiled_attention_08_gb300 as fa

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gh.require_gpu()


def _draw(shape, gen, dtype):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def _status_ok():
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK


def _eye(B, H, n, D, dtype):
    return torch.eye(n, D, dtype=dtype).expand(B, H, n, D).contiguous()


@pytest.mark.parametrize("Lq,causal", [(300, False), (257, True)])
def test_forward_mask_bit_exact(oracle_mod, Lq, causal):
    """V = I (Lk = D): O = (P o Z) V = P o Z, zero exactly at the dropped (and the masked)
    entries, since a visible entry has P > 0 here.  The zero pattern is compared with the
    oracle's element by element; with Lq > Lk under the causal mask, rows see no key at all."""
    B, H, D, p, seed = 2, 3, 128, 0.3, 0x1234_5678_9ABC_DEF0
    Lk = D
    g = torch.Generator().manual_seed(11)
    q = _draw((B, H, Lq, D), g, torch.bfloat16)
    k = _draw((B, H, Lk, D), g, torch.bfloat16)
    v = _eye(B, H, Lk, D, torch.bfloat16)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal, dropout_p=p, seed=seed)
    _status_ok()
    o_ref, lse_ref = oracle_mod.forward(gh.f64(q), gh.f64(k), gh.f64(v), 1.0 / math.sqrt(D),
                                        causal, dropout_p=p, seed=seed)
    got, ref = gh.f64(o), o_ref
    visible = np.ones((Lq, Lk), dtype=bool)
    if causal:
        visible = np.tril(visible, Lk - Lq)
    ref_zero = ref == 0.0
    assert np.array_equal(got == 0.0, ref_zero)
    kept = ~ref_zero[..., visible]
    assert abs(kept.mean() - (1.0 - p)) < 0.01, kept.mean()
    # LSE is that of P itself, not of the kept entries
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(gh.f64(lse)), empty)
    assert np.max(np.abs(gh.f64(lse)[~empty] - lse_ref[~empty])) <= gh.LSE_MAX_ABS


@pytest.mark.parametrize("Lk,causal", [(300, False), (400, True)])
def test_backward_mask_bit_exact(oracle_mod, Lk, causal):
    """dO = I (Lq = D): dV = (P o Z)^T dO = (P o Z)^T, zero exactly at the dropped entries, so
    the transposed mask that the dK/dV kernel builds across lanes is compared bit for bit."""
    B, H, D, p, seed = 2, 2, 128, 0.5, 987654321
    Lq = D
    g = torch.Generator().manual_seed(12)
    q = _draw((B, H, Lq, D), g, torch.bfloat16)
    k = _draw((B, H, Lk, D), g, torch.bfloat16)
    v = _draw((B, H, Lk, D), g, torch.bfloat16)
    do = _eye(B, H, Lq, D, torch.bfloat16)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = fa.forward(qd, kd, vd, causal, dropout_p=p, seed=seed)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, do.to(DEV), causal, dropout_p=p, seed=seed)
    _status_ok()
    _, _, dv_ref, _ = oracle_mod.backward(gh.f64(q), gh.f64(k), gh.f64(v), gh.f64(do),
                                          1.0 / math.sqrt(D), causal, dropout_p=p, seed=seed)
    assert np.array_equal(gh.f64(dv) == 0.0, dv_ref == 0.0)
    nz = dv_ref != 0.0
    rel = np.linalg.norm(gh.f64(dv)[nz] - dv_ref[nz]) / np.linalg.norm(dv_ref[nz])
    assert rel <= gh.GRAD_REL_FRO, rel


CASES = [
    # B, H, Lq, Lk, D, causal, p, dtype
    (2, 2, 300, 300, 64, True, 0.17, torch.bfloat16),
    (1, 3, 256, 384, 128, False, 0.5, torch.bfloat16),
    (2, 1, 700, 200, 64, True, 0.1, torch.bfloat16),     # Lq > Lk: rows that see no key
    (1, 2, 200, 700, 128, True, 0.3, torch.float16),
    (1, 2, 129, 129, 128, False, 0.9, torch.bfloat16),   # heavy dropout, ragged tiles
    (3, 2, 1000, 1000, 64, False, 0.25, torch.float16),
]


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal,p,dtype", CASES,
                         ids=lambda x: str(x).replace("torch.", ""))
def test_parity_with_dropout(oracle_mod, B, H, Lq, Lk, D, causal, p, dtype):
    seed = (B * 1000003 + Lq * 131 + Lk) * 2654435761 % 2**64
    g = torch.Generator().manual_seed(Lq + Lk + D)
    q, do = _draw((B, H, Lq, D), g, dtype), _draw((B, H, Lq, D), g, dtype)
    k, v = _draw((B, H, Lk, D), g, dtype), _draw((B, H, Lk, D), g, dtype)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.forward(qd, kd, vd, causal, scale, dropout_p=p, seed=seed)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, do.to(DEV), causal, scale, dropout_p=p,
                             seed=seed)
    _status_ok()
    f = [gh.f64(t) for t in (q, k, v, do)]
    o_ref, lse_ref = oracle_mod.forward(f[0], f[1], f[2], scale, causal, dropout_p=p, seed=seed)
    dq_ref, dk_ref, dv_ref, _ = oracle_mod.backward(*f, scale, causal, dropout_p=p, seed=seed)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(gh.f64(lse)), empty)
    if (~empty).any():
        assert np.max(np.abs(gh.f64(lse)[~empty] - lse_ref[~empty])) <= gh.LSE_MAX_ABS
    # Kept entries carry 1/(1-p): |O| grows with p, so the bound is the one beyond the 16-bit
    # rounding of the exact result.
    err = gh.o_errors(gh.f64(o), o_ref, dtype)
    assert err["o_max"] <= gh.O_MAX_ABS and err["o_mean"] <= gh.O_MEAN_ABS, err
    for name, got, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        rel = np.linalg.norm(gh.f64(got) - ref) / np.linalg.norm(ref)
        assert rel <= gh.GRAD_REL_FRO, (name, rel)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_tiny_p_equals_no_dropout_bitwise(D, causal):
    """p = 1e-12: the threshold floor(p * 2^32) is 0, so the dropout kernels keep every entry
    and the keep factor 1/(1-p) rounds to 1.0f: O, LSE, dQ, dK, dV equal those of the kernels
    without dropout bit for bit (the same arithmetic, only the mask code around it).  Sizes run
    the persistent kernels on the path without dropout."""
    B, H, L = 8, 16, 512
    g = torch.Generator().manual_seed(D + causal)
    q, k, v, do = (_draw((B, H, L, D), g, torch.bfloat16).to(DEV) for _ in range(4))
    a = fa.forward(q, k, v, causal)
    ga = fa.backward(q, k, v, a[0], a[1], do, causal)
    b = fa.forward(q, k, v, causal, dropout_p=1e-12, seed=3)
    gb = fa.backward(q, k, v, b[0], b[1], do, causal, dropout_p=1e-12, seed=3)
    _status_ok()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for x, y in zip(ga, gb):
        assert torch.equal(x, y)


def test_seed_determinism_and_autograd(oracle_mod):
    """The same seed twice: the same bits; another seed: another mask.  attention() with an
    explicit seed carries it to the backward (checked against the oracle)."""
    B, H, L, D, p = 1, 2, 384, 64, 0.2
    g = torch.Generator().manual_seed(21)
    q, k, v, do = (_draw((B, H, L, D), g, torch.bfloat16) for _ in range(4))
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o1, _ = fa.forward(qd, kd, vd, True, dropout_p=p, seed=5)
    o2, _ = fa.forward(qd, kd, vd, True, dropout_p=p, seed=5)
    o3, _ = fa.forward(qd, kd, vd, True, dropout_p=p, seed=6)
    _status_ok()
    assert torch.equal(o1, o2)
    assert not torch.equal(o1, o3)
    x = [t.to(DEV).requires_grad_(True) for t in (q, k, v)]
    o = fa.attention(*x, causal=True, dropout_p=p, seed=5)
    assert torch.equal(o.detach(), o1)
    o.backward(do.to(DEV))
    _status_ok()
    f = [gh.f64(t) for t in (q, k, v, do)]
    refs = oracle_mod.backward(*f, 1.0 / math.sqrt(D), True, dropout_p=p, seed=5)[:3]
    for t, ref in zip(x, refs):
        rel = np.linalg.norm(gh.f64(t.grad) - ref) / np.linalg.norm(ref)
        assert rel <= gh.GRAD_REL_FRO, rel
    # without a seed, attention() draws one per call: two calls drop differently
    a = fa.attention(qd, kd, vd, causal=True, dropout_p=p)
    b = fa.attention(qd, kd, vd, causal=True, dropout_p=p)
    assert not torch.equal(a, b)
