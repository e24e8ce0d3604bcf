"""dQ by reduction (fa_bwd_ex with deterministic = 0): at D = 64 the dK/dV pass also computes
dS K for every (key tile, query tile) pair and adds it into an fp32 accumulator, and a third
kernel converts it to dQ.  Checked against the fp64 oracle like the deterministic path (dQ,
dK, dV within the relative Frobenius bound; rows that see no key exactly zero), and against the
deterministic path itself: dK and dV come from the same arithmetic (bit for bit), dQ differs
only by the order of fp32 additions.  At D = 128, and with dropout, deterministic = 0 takes the
deterministic path (bit for bit)."""
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


CASES = [
    # B, H, Lq, Lk, causal, dtype
    (2, 2, 300, 300, True, torch.bfloat16),
    (1, 3, 256, 384, False, torch.bfloat16),
    (2, 1, 700, 200, True, torch.bfloat16),   # Lq > Lk: rows that see no key
    (1, 2, 200, 700, True, torch.float16),
    (1, 2, 129, 129, False, torch.float16),
    (1, 4, 1024, 1024, True, torch.bfloat16),
]


@pytest.mark.parametrize("B,H,Lq,Lk,causal,dtype", CASES,
                         ids=lambda x: str(x).replace("torch.", ""))
def test_parity_dq_by_reduction(oracle_mod, B, H, Lq, Lk, causal, dtype):
    D = 64
    g = torch.Generator().manual_seed(Lq * 3 + Lk + int(causal))
    q, do = _draw((B, H, Lq, D), g, dtype), _draw((B, H, Lq, D), g, dtype)
    k, v = _draw((B, H, Lk, D), g, dtype), _draw((B, H, Lk, D), g, dtype)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.forward(qd, kd, vd, causal, scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal, scale, deterministic=False)
    ref = fa.backward(qd, kd, vd, o, lse, dod, causal, scale)
    _status_ok()
    # dK, dV: the same kernels' arithmetic; dQ: fp32 sums in another order
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    diff = (dq.float() - ref[0].float()).norm() / ref[0].float().norm().clamp_min(1e-30)
    assert diff <= 5e-3, float(diff)
    f = [gh.f64(t) for t in (q, k, v, do)]
    dq_ref, dk_ref, dv_ref, _ = oracle_mod.backward(*f, scale, causal)
    empty = np.isneginf(oracle_mod.forward(f[0], f[1], f[2], scale, causal)[1])
    assert np.all(gh.f64(dq)[empty] == 0.0), "dQ of a row that sees no key"
    for name, got, r in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        rel = np.linalg.norm(gh.f64(got) - r) / np.linalg.norm(r)
        assert rel <= gh.GRAD_REL_FRO, (name, rel)


def test_full_size_long_sequence_sampled(oracle_mod):
    """B1 H16 L16384 D64 causal (the long-sequence workload) with dQ by reduction: whole heads
    are too slow for the oracle, so sampled query rows' dQ is checked against the oracle on the
    causal prefix that ends at that row (a complete sub-problem for those rows), and the whole
    dQ against the deterministic path."""
    B, H, L, D = 1, 16, 16384, 64
    g = torch.Generator().manual_seed(99)
    q, k, v, do = (_draw((B, H, L, D), g, torch.bfloat16) for _ in range(4))
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, True)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, True, deterministic=False)
    ref = fa.backward(qd, kd, vd, o, lse, dod, True)
    _status_ok()
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    diff = (dq.float() - ref[0].float()).norm() / ref[0].float().norm()
    assert diff <= 5e-3, float(diff)
    scale = 1.0 / math.sqrt(D)
    for h, n in ((0, 1000), (7, 4097), (15, 6000)):
        rows = slice(n - 8, n)
        f = [gh.f64(t[0, h, :n]) for t in (q, k, v, do)]
        dq_ref = oracle_mod.backward(*f, scale, True)[0]
        got = gh.f64(dq[0, h, rows])
        rel = np.linalg.norm(got - dq_ref[rows]) / np.linalg.norm(dq_ref[rows])
        assert rel <= gh.GRAD_REL_FRO, (h, n, rel)


@pytest.mark.parametrize("D,p", [(128, 0.0), (64, 0.2)])
def test_other_cases_take_the_deterministic_path(D, p):
    """deterministic = 0 at D = 128 or with dropout: the separate dQ pass, bit for bit."""
    B, H, L = 1, 4, 512
    g = torch.Generator().manual_seed(D)
    q, k, v, do = (_draw((B, H, L, D), g, torch.bfloat16).to(DEV) for _ in range(4))
    o, lse = fa.forward(q, k, v, True, dropout_p=p, seed=1)
    a = fa.backward(q, k, v, o, lse, do, True, dropout_p=p, seed=1, deterministic=False)
    b = fa.backward(q, k, v, o, lse, do, True, dropout_p=p, seed=1)
    _status_ok()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
