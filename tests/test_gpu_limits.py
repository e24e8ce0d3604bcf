"""Edge sizes on the GPU: the longest sequences and the most heads the kernels are built for,
checked against the fp64 oracle where it can answer one row at a time.

* L = 262144 (one head, causal): whole heads are far beyond the oracle, but query row i of a
  causal problem depends only on keys 0..i, so the last rows of the prefix [0, n) form a
  complete sub-problem: O, LSE and dQ of sampled rows are compared with the oracle on
  (q[n-8:n], k[:n], v[:n]) (queries aligned to the end of the keys).
* B*H = 70000 heads (more than the 65535 a grid's y dimension holds, and head offsets past
  2^32 bytes): every output of sampled heads, including ones past index 65535, against the
  oracle.
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


@pytest.mark.parametrize("L,D", [(262144, 64), (131072, 128)])
def test_longest_sequence_sampled_rows(oracle_mod, L, D):
    g = torch.Generator().manual_seed(L + D)
    q, k, v, do = (_draw((1, 1, L, D), g, torch.bfloat16) for _ in range(4))
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, True)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, True)
    _status_ok()
    scale = 1.0 / math.sqrt(D)
    for n in (129, 70001, L):
        rows = slice(n - 8, n)
        qs, dos = gh.f64(q[0, 0, rows]), gh.f64(do[0, 0, rows])
        ks, vs = gh.f64(k[0, 0, :n]), gh.f64(v[0, 0, :n])
        o_ref, lse_ref = oracle_mod.forward(qs, ks, vs, scale, True)
        err = gh.o_errors(gh.f64(o[0, 0, rows]), o_ref, torch.bfloat16)
        assert err["o_raw_max"] <= gh.O_MAX_ABS and err["o_raw_mean"] <= gh.O_MEAN_ABS, (n, err)
        assert np.max(np.abs(gh.f64(lse[0, 0, rows]) - lse_ref)) <= gh.LSE_MAX_ABS, n
        # dQ of these rows needs the forward's O of these rows (Delta = rowsum(dO o O)): the
        # oracle recomputes it from the same sub-problem.
        dq_ref = oracle_mod.backward(qs, ks, vs, dos, scale, True)[0]
        got = gh.f64(dq[0, 0, rows])
        rel = np.linalg.norm(got - dq_ref) / np.linalg.norm(dq_ref)
        assert rel <= gh.GRAD_REL_FRO, (n, rel)
    assert torch.isfinite(dk.float()).all() and torch.isfinite(dv.float()).all()


def test_more_heads_than_a_grid_column(oracle_mod):
    B, H, L, D = 2, 35000, 130, 64
    g = torch.Generator().manual_seed(7)
    q, k, v, do = (_draw((B, H, L, D), g, torch.bfloat16) for _ in range(4))
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, False)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, False)
    _status_ok()
    scale = 1.0 / math.sqrt(D)
    for bh in (0, 65534, 65535, 65536, B * H - 1):
        b, h = divmod(bh, H)
        f = [gh.f64(t[b, h]) for t in (q, k, v, do)]
        o_ref, lse_ref = oracle_mod.forward(f[0], f[1], f[2], scale, False)
        err = gh.o_errors(gh.f64(o[b, h]), o_ref, torch.bfloat16)
        assert err["o_raw_max"] <= gh.O_MAX_ABS and err["o_raw_mean"] <= gh.O_MEAN_ABS, (bh, err)
        assert np.max(np.abs(gh.f64(lse[b, h]) - lse_ref)) <= gh.LSE_MAX_ABS, bh
        refs = oracle_mod.backward(*f, scale, False)[:3]
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            rel = np.linalg.norm(gh.f64(got[b, h]) - ref) / np.linalg.norm(ref)
            assert rel <= gh.GRAD_REL_FRO, (bh, name, rel)
