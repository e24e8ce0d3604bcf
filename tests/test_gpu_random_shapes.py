"""Seeded random sweep of the CUDA path against the fp64 oracle: shapes drawn from sizes around
the 64- and 128-row tile edges (1 to 1024 queries, 1 to 1024 keys, Lq != Lk with the causal
rows aligned to the end of the keys), both head sizes and 16-bit types, causal and not, scales
other than 1/sqrt(D) (negative included), dropout on P, [B, L, H, D] strided views, the CTA-pair
forward and dQ by reduction; and, with many heads, the persistent grids (more items than SMs),
whose first, last and two seeded heads are compared.  Every case is held to the same bounds as
the fixed parity tests: O beyond half a 16-bit ulp <= 1e-2 (max) and 1e-3 (mean), LSE <= 1e-3,
dQ / dK / dV relative Frobenius error <= 2e-2 (an absolute bound where the exact gradient is 0;
under dropout that bound follows the rounding of the stored O, see the comment in _run).
"""
import math
import random

import numpy as np
import pytest
import torch

import gpu_helpers as gh
import tiled_attention_08_gb300 as fa

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SMALL_L = [1, 2, 7, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 383, 384, 385, 511, 640, 700,
           1000]
SMALL_LK = [1, 5, 64, 100, 128, 129, 250, 256, 300, 511, 512, 700, 1024]
BIG_L = [128, 250, 256, 384, 511, 512, 640, 1024]
BIG_LK = [128, 256, 300, 512, 1024]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gh.require_gpu()
    yield
    fa.fa_set_forward_pair(0)


def _case(rng, many_heads):
    D = rng.choice([64, 128])
    if many_heads:
        B, H = rng.choice([2, 4, 8]), rng.choice([24, 40, 64])
        Lq = rng.choice(BIG_L)
        Lk = Lq if rng.random() < 0.6 else rng.choice(BIG_LK)
    else:
        B, H = rng.choice([1, 1, 2, 3]), rng.choice([1, 2, 3, 5])
        Lq = rng.choice(SMALL_L)
        Lk = Lq if rng.random() < 0.5 else rng.choice(SMALL_LK)
    return dict(B=B, H=H, Lq=Lq, Lk=Lk, D=D, causal=rng.random() < 0.5,
                dtype=rng.choice([torch.bfloat16, torch.float16]),
                scale=rng.choice([None, None, None, 0.3, -0.125, 1.0 / 64]),
                drop=0.0 if many_heads else rng.choice([0.0, 0.0, 0.0, 0.15]),
                blhd=rng.random() < 0.3, det=rng.random() < 0.7,
                pair=D == 128 and rng.random() < 0.3)


def _run(oracle_mod, c, case, rng):
    B, H, Lq, Lk, D, dtype = c["B"], c["H"], c["Lq"], c["Lk"], c["D"], c["dtype"]
    pair = c["pair"] and c["drop"] == 0.0
    sc = 1.0 / math.sqrt(D) if c["scale"] is None else c["scale"]
    g = torch.Generator().manual_seed(case * 7919 + 13)
    q = torch.randn((B, H, Lq, D), generator=g).to(dtype)
    k = torch.randn((B, H, Lk, D), generator=g).to(dtype)
    v = torch.randn((B, H, Lk, D), generator=g).to(dtype)
    do = torch.randn((B, H, Lq, D), generator=g).to(dtype)
    seed = case * 31 + 7
    assert fa.fa_set_forward_pair(1 if pair else 0) == fa.FA_OK
    if c["blhd"]:
        qd, kd, vd, dod = (t.transpose(1, 2).contiguous().to(DEV).transpose(1, 2)
                           for t in (q, k, v, do))
    else:
        qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, c["causal"], sc, dropout_p=c["drop"], seed=seed)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, c["causal"], sc, dropout_p=c["drop"],
                             seed=seed, deterministic=c["det"])
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    if B * H > 16:  # first, last and two seeded heads (no dropout: its mask names the head)
        heads = sorted({0, B * H - 1, rng.randrange(B * H), rng.randrange(B * H)})
        sel = lambda t: t.reshape(B * H, *t.shape[2:])[heads].unsqueeze(0)  # noqa: E731
        q, k, v, do = (sel(t) for t in (q, k, v, do))
        o, lse, dq, dk, dv = (sel(t) for t in (o, lse, dq, dk, dv))
    o_ref, lse_ref = oracle_mod.forward(gh.f64(q), gh.f64(k), gh.f64(v), sc, c["causal"],
                                        dropout_p=c["drop"], seed=seed)
    refs = oracle_mod.backward(gh.f64(q), gh.f64(k), gh.f64(v), gh.f64(do), sc, c["causal"],
                               dropout_p=c["drop"], seed=seed)[:3]
    err = gh.o_errors(gh.f64(o), o_ref, dtype)
    bad = []
    if err["o_max"] > gh.O_MAX_ABS or err["o_mean"] > gh.O_MEAN_ABS:
        bad.append(("o", err))
    empty = np.isneginf(lse_ref)
    lse_g = gh.f64(lse)
    if not np.array_equal(np.isneginf(lse_g), empty):
        bad.append(("lse -inf rows", None))
    elif (~empty).any():
        e = float(np.max(np.abs(lse_g[~empty] - lse_ref[~empty])))
        if e > gh.LSE_MAX_ABS:
            bad.append(("lse", e))
    zero_bounds = {"dq": gh.O_MAX_ABS, "dk": gh.O_MAX_ABS, "dv": gh.O_MAX_ABS}
    if c["drop"] > 0.0:
        # With dropout the stored O = (P o Z) V / (1 - p) is rounded to 16 bits, and the
        # backward's Delta_i = rowsum(dO_i o O_i) uses it while dP uses V itself: in rows where
        # the exact dS cancels to 0 (a single visible key) the difference, about one 16-bit
        # rounding of dO_i . O_i, is what remains.  Bound it per row by 2^-m |dO_i| |O_i| (m
        # mantissa bits) and carry it through dQ = scale dS K and dK = scale dS^T Q.
        m = 8 if dtype == torch.bfloat16 else 11
        dsb = 2.0 ** -m * np.linalg.norm(gh.f64(do), axis=-1) * np.linalg.norm(o_ref, axis=-1)
        zero_bounds["dq"] = max(gh.O_MAX_ABS, 2 * abs(sc) * dsb.max() * np.abs(gh.f64(k)).max())
        zero_bounds["dk"] = max(gh.O_MAX_ABS, 2 * abs(sc) * dsb.sum(axis=-1).max()
                                * np.abs(gh.f64(q)).max())
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        got = gh.f64(got)
        norm = float(np.linalg.norm(ref))
        if norm < 1e-9:
            e = float(np.max(np.abs(got))) if got.size else 0.0
            if e > zero_bounds[name]:
                bad.append((name + " (exact 0)", e, zero_bounds[name]))
        else:
            e = float(np.linalg.norm(got - ref) / norm)
            if e > gh.GRAD_REL_FRO:
                bad.append((name, e))
    return bad


@pytest.mark.parametrize("seed,n,many_heads", [(11, 120, False), (12, 25, True)])
def test_random_shapes(oracle_mod, seed, n, many_heads):
    rng = random.Random(seed)
    failures = []
    for case in range(n):
        c = _case(rng, many_heads)
        bad = _run(oracle_mod, c, case + 1000 * seed, rng)
        if bad:
            failures.append((c, bad))
    assert not failures, failures
