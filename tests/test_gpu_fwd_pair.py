"""The forward on CTA pairs (fa_set_forward_pair(1): D = 128, one tensor-core contraction of 256
query rows over two SMs) against the fp64 oracle and against the single-CTA forward, whose
per-row arithmetic it repeats (bit for bit equal O and LSE): causal and not, Lq != Lk with rows
that see no key, ragged tails and query tiles past the last row, fp16, a negative scale."""
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
    yield
    fa.fa_set_forward_pair(0)


def _draw(shape, gen, dtype):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def _both(q, k, v, causal, scale):
    out = []
    for mode in (1, 0):
        assert fa.fa_set_forward_pair(mode) == fa.FA_OK
        out.append(fa.forward(q, k, v, causal, scale))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    return out


CASES = [
    # B, H, Lq, Lk, causal, dtype, scale (None: 1/sqrt(D))
    (1, 2, 512, 512, True, torch.bfloat16, None),
    (2, 2, 300, 300, False, torch.bfloat16, None),
    (1, 3, 700, 200, True, torch.bfloat16, None),    # Lq > Lk: rows that see no key
    (1, 2, 200, 700, True, torch.float16, None),
    (1, 2, 129, 129, False, torch.bfloat16, None),   # one tile and a 1-row tail: three absent
    (2, 2, 640, 640, True, torch.bfloat16, -0.125),  # negative scale
    (1, 2, 384, 1000, False, torch.float16, 0.3),
]


@pytest.mark.parametrize("B,H,Lq,Lk,causal,dtype,scale", CASES,
                         ids=lambda x: str(x).replace("torch.", ""))
def test_pair_forward_parity(oracle_mod, B, H, Lq, Lk, causal, dtype, scale):
    D = 128
    g = torch.Generator().manual_seed(Lq * 7 + Lk + int(causal))
    q = _draw((B, H, Lq, D), g, dtype)
    k, v = _draw((B, H, Lk, D), g, dtype), _draw((B, H, Lk, D), g, dtype)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    (o2, l2), (o1, l1) = _both(q.to(DEV), k.to(DEV), v.to(DEV), causal, sc)
    assert torch.equal(o2, o1) and torch.equal(l2, l1)
    o_ref, lse_ref = oracle_mod.forward(gh.f64(q), gh.f64(k), gh.f64(v), sc, causal)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(gh.f64(l2)), empty)
    if (~empty).any():
        assert np.max(np.abs(gh.f64(l2)[~empty] - lse_ref[~empty])) <= gh.LSE_MAX_ABS
    err = gh.o_errors(gh.f64(o2), o_ref, dtype)
    assert err["o_max"] <= gh.O_MAX_ABS and err["o_mean"] <= gh.O_MEAN_ABS, err


def test_pair_forward_full_size_equals_single_cta():
    """B8 H32 L4096 D128 causal (the batched training shape) and B1 H16 L16384 at D = 128:
    the two forms give the same bits."""
    for (B, H, L) in ((8, 32, 4096), (1, 16, 16384)):
        g = torch.Generator().manual_seed(L)
        q, k, v = (_draw((B, H, L, 128), g, torch.bfloat16).to(DEV) for _ in range(3))
        (o2, l2), (o1, l1) = _both(q, k, v, True, None)
        assert torch.equal(o2, o1) and torch.equal(l2, l1)


def test_mode_argument():
    assert fa.fa_set_forward_pair(2) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_forward_pair(-1) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_set_forward_pair(0) == fa.FA_OK
