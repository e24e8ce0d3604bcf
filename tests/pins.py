"""Pins for the fp64 attention oracle: facts fixed by the mathematics, not by the oracle.

Every pin takes an implementation object with
    forward(q, k, v, scale, causal)        -> (O [L,D], LSE [L])
    backward(q, k, v, do, scale, causal)   -> (dQ, dK, dV, Delta)
    probs(q, k, scale, causal)             -> P [L,L]
(one head, fp64 numpy arrays) and raises AssertionError when the implementation violates
the fact.  ``tests/test_oracle_pins.py`` runs them on the oracle;
``tests/test_oracle_mutants.py`` plants plausible mistakes in a copy of the method and checks
that each mistake trips at least one pin.

What the facts rest on:
* softmax rows are probability vectors (the definition of softmax);
* closed forms: a single key, identical keys, causal row 0, zero queries, a dominant key
  ("FlashAttention principles and engineering practice", section 2.1: attn = softmax(q k^T
  scale) v);
* shift invariance of softmax in the keys;
* the backward pass is the gradient of sum(O * dO): central finite differences, and the
  invariants sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i that follow from shift invariance and
  from rows of P summing to one;
* an independent library implementation of the same operation (torch's CPU
  scaled_dot_product_attention in fp64, with autograd), for random heads;
* queries and keys of different lengths (Lq != Lk, the flash_attn_func interface of "FlashAttention
  data-flow optimisation", section 4.1, step 3): with the causal mask the queries are read as the
  last Lq positions of the key sequence, so a suffix of the queries of a square causal problem
  must reproduce that problem's rows and gradients exactly; rows that see no key (Lq > Lk) give
  O = 0, LSE = -inf and dQ = 0.
"""
from __future__ import annotations

import math

import numpy as np

TIGHT = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


def pin_probs_are_distributions(impl):
    r = _rng(1)
    for causal in (False, True):
        L, D = 37, 5
        q, k = r.standard_normal((L, D)), r.standard_normal((L, D))
        p = impl.probs(q, k, 0.7, causal)
        assert np.all(p >= 0.0), "P has negative entries"
        _close(p.sum(axis=1), np.ones(L), TIGHT, "row sums of P")
        if causal:
            assert np.all(np.triu(p, 1) == 0.0), "causal P has weight above the diagonal"
            assert np.all(np.diag(p) > 0.0), "causal P drops the diagonal key"
        else:
            assert np.all(p > 0.0), "non-causal P has a zero entry"


def pin_single_key(impl):
    r = _rng(2)
    for D in (1, 4, 64):
        q, k, v = (r.standard_normal((1, D)) for _ in range(3))
        for causal in (False, True):
            o, lse = impl.forward(q, k, v, 0.3, causal)
            _close(o, v, TIGHT, "O for a single key")
            _close(lse, [0.3 * float(q[0] @ k[0])], TIGHT, "LSE for a single key")


def pin_identical_keys(impl):
    r = _rng(3)
    L, D = 19, 6
    q, v = r.standard_normal((L, D)), r.standard_normal((L, D))
    kappa = r.standard_normal(D)
    k = np.tile(kappa, (L, 1))
    o, lse = impl.forward(q, k, v, 0.45, False)
    _close(o, np.tile(v.mean(axis=0), (L, 1)), TIGHT, "O with identical keys")
    _close(lse, 0.45 * (q @ kappa) + math.log(L), TIGHT, "LSE with identical keys")
    # Causal: row i averages the first i+1 values.
    o, lse = impl.forward(q, k, v, 0.45, True)
    want = np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None]
    _close(o, want, TIGHT, "causal O with identical keys")
    _close(lse, 0.45 * (q @ kappa) + np.log(np.arange(1, L + 1)), TIGHT,
           "causal LSE with identical keys")


def pin_causal_row0(impl):
    r = _rng(4)
    L, D = 23, 8
    q, k, v = (r.standard_normal((L, D)) for _ in range(3))
    o, lse = impl.forward(q, k, v, 0.9, True)
    _close(o[0], v[0], TIGHT, "causal O row 0")
    _close(lse[0], 0.9 * float(q[0] @ k[0]), TIGHT, "causal LSE row 0")


def pin_zero_queries(impl):
    r = _rng(5)
    L, D = 17, 3
    q = np.zeros((L, D))
    k, v = r.standard_normal((L, D)), r.standard_normal((L, D))
    o, lse = impl.forward(q, k, v, 1.0, True)
    _close(o, np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None], TIGHT, "O for Q=0, causal")
    _close(lse, np.log(np.arange(1, L + 1)), TIGHT, "LSE for Q=0, causal")
    o, lse = impl.forward(q, k, v, 1.0, False)
    _close(o, np.tile(v.mean(axis=0), (L, 1)), TIGHT, "O for Q=0")
    _close(lse, np.full(L, math.log(L)), TIGHT, "LSE for Q=0")


def pin_key_shift(impl):
    r = _rng(6)
    L, D = 21, 5
    q, k, v = (r.standard_normal((L, D)) for _ in range(3))
    c = r.standard_normal(D)
    for causal in (False, True):
        o0, lse0 = impl.forward(q, k, v, 0.6, causal)
        o1, lse1 = impl.forward(q, k + c, v, 0.6, causal)
        _close(o1, o0, 1e-11, "O under a key shift")
        _close(lse1 - lse0, 0.6 * (q @ c), 1e-11, "LSE shift under a key shift")


def pin_dominant_key(impl):
    r = _rng(7)
    L, D = 12, 4
    u = r.standard_normal(D)
    q = np.tile(u, (L, 1))
    k = 0.01 * r.standard_normal((L, D))
    jstar = 3
    k[jstar] = 40.0 * u / float(u @ u)
    v = r.standard_normal((L, D))
    o, _ = impl.forward(q, k, v, 1.0, False)
    # Every other key carries weight below exp(-39); the residue is far under 1e-13.
    _close(o, np.tile(v[jstar], (L, 1)), 1e-13, "O with a dominant key")


def _loss(impl, q, k, v, do, scale, causal):
    o, _ = impl.forward(q, k, v, scale, causal)
    return float(np.sum(o * do))


def pin_finite_differences(impl):
    r = _rng(8)
    h = 1e-6
    for (L, D, causal) in ((5, 3, False), (8, 4, True), (6, 2, True)):
        q, k, v, do = (r.standard_normal((L, D)) for _ in range(4))
        scale = 0.8
        dq, dk, dv, _ = impl.backward(q, k, v, do, scale, causal)
        for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy()
                xm = x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                key = {"dQ": "q", "dK": "k", "dV": "v"}[name]
                args_p[key] = xp
                args_m[key] = xm
                fp = _loss(impl, args_p["q"], args_p["k"], args_p["v"], do, scale, causal)
                fm = _loss(impl, args_m["q"], args_m["k"], args_m["v"], do, scale, causal)
                num[idx] = (fp - fm) / (2 * h)
            rel = np.linalg.norm(g - num) / max(np.linalg.norm(num), 1e-30)
            assert rel <= 1e-6, f"{name} vs finite differences (L={L},D={D},causal={causal}): rel {rel:.2e}"


def pin_gradient_invariants(impl):
    r = _rng(9)
    L, D = 29, 7
    q, k, v, do = (r.standard_normal((L, D)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv, delta = impl.backward(q, k, v, do, 0.5, causal)
        _close(dk.sum(axis=0), np.zeros(D), 1e-11, "sum_j dK_j")
        _close(dv.sum(axis=0), do.sum(axis=0), 1e-11, "sum_j dV_j vs sum_i dO_i")
        o, _ = impl.forward(q, k, v, 0.5, causal)
        _close(delta, np.sum(do * o, axis=1), 1e-11, "Delta vs rowsum(dO * O)")


def pin_zero_queries_backward(impl):
    r = _rng(10)
    L, D = 13, 3
    q = np.zeros((L, D))
    k, v, do = (r.standard_normal((L, D)) for _ in range(3))
    _, _, dv, _ = impl.backward(q, k, v, do, 1.0, True)
    w = do / np.arange(1, L + 1)[:, None]
    want = np.cumsum(w[::-1], axis=0)[::-1]  # sum over i >= j of dO_i / (i+1)
    _close(dv, want, TIGHT, "dV for Q=0, causal")
    _, _, dv, _ = impl.backward(q, k, v, do, 1.0, False)
    _close(dv, np.tile(do.sum(axis=0) / L, (L, 1)), TIGHT, "dV for Q=0")


def pin_library_sdpa(impl):
    """Random heads against torch's fp64 CPU scaled_dot_product_attention and its autograd."""
    import torch
    import torch.nn.functional as F

    r = _rng(11)
    for (L, D, causal, scale) in ((33, 16, False, 0.25), (47, 8, True, 0.35), (64, 64, True, 0.125)):
        q, k, v, do = (r.standard_normal((L, D)) for _ in range(4))
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        to = F.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                            is_causal=causal, scale=scale)[0, 0]
        to.backward(torch.tensor(do, dtype=torch.float64))
        o, _ = impl.forward(q, k, v, scale, causal)
        _close(o, to.detach().numpy(), 1e-12, "O vs torch sdpa")
        dq, dk, dv, _ = impl.backward(q, k, v, do, scale, causal)
        _close(dq, tq.grad.numpy(), 1e-12, "dQ vs torch sdpa autograd")
        _close(dk, tk.grad.numpy(), 1e-12, "dK vs torch sdpa autograd")
        _close(dv, tv.grad.numpy(), 1e-12, "dV vs torch sdpa autograd")


def _zero_early_rows(a, n):
    b = a.copy()
    b[:n] = 0.0
    return b


def pin_suffix_queries(impl):
    """Bottom-right causal alignment: the last Lq queries against all Lk keys are rows
    [Lk-Lq, Lk) of the square causal problem, and so are their gradients (the early rows of the
    square problem then carry dO = 0)."""
    r = _rng(14)
    Lk, D, scale = 13, 5, 0.55
    q, k, v, do = (r.standard_normal((Lk, D)) for _ in range(4))
    for Lq in (1, 4, Lk - 1, Lk):
        n0 = Lk - Lq
        for causal in (True, False):
            o, lse = impl.forward(q[n0:], k, v, scale, causal)
            o_sq, lse_sq = impl.forward(q, k, v, scale, causal)
            _close(o, o_sq[n0:], 1e-12, f"O of the last {Lq} queries (causal={causal})")
            _close(lse, lse_sq[n0:], 1e-12, f"LSE of the last {Lq} queries (causal={causal})")
            dq, dk, dv, _ = impl.backward(q[n0:], k, v, do[n0:], scale, causal)
            dq_sq, dk_sq, dv_sq, _ = impl.backward(q, k, v, _zero_early_rows(do, n0), scale, causal)
            _close(dq, dq_sq[n0:], 1e-12, f"dQ of the last {Lq} queries (causal={causal})")
            _close(dk, dk_sq, 1e-12, f"dK with only the last {Lq} queries (causal={causal})")
            _close(dv, dv_sq, 1e-12, f"dV with only the last {Lq} queries (causal={causal})")


def pin_more_queries_than_keys(impl):
    """Lq > Lk, causal: the first Lq - Lk queries see no key (O = 0, LSE = -inf, dQ = 0, no
    contribution to dK, dV); the last Lk are the square causal problem."""
    r = _rng(15)
    Lq, Lk, D, scale = 11, 4, 3, 0.7
    q, do = r.standard_normal((Lq, D)), r.standard_normal((Lq, D))
    k, v = r.standard_normal((Lk, D)), r.standard_normal((Lk, D))
    n0 = Lq - Lk
    o, lse = impl.forward(q, k, v, scale, True)
    assert np.all(o[:n0] == 0.0), "O of a row that sees no key"
    assert np.all(np.isneginf(lse[:n0])), "LSE of a row that sees no key"
    o_sq, lse_sq = impl.forward(q[n0:], k, v, scale, True)
    _close(o[n0:], o_sq, 1e-12, "O of the rows that see keys")
    _close(lse[n0:], lse_sq, 1e-12, "LSE of the rows that see keys")
    dq, dk, dv, _ = impl.backward(q, k, v, do, scale, True)
    assert np.all(dq[:n0] == 0.0), "dQ of a row that sees no key"
    dq_sq, dk_sq, dv_sq, _ = impl.backward(q[n0:], k, v, do[n0:], scale, True)
    _close(dq[n0:], dq_sq, 1e-12, "dQ of the rows that see keys")
    _close(dk, dk_sq, 1e-12, "dK with rows that see no key")
    _close(dv, dv_sq, 1e-12, "dV with rows that see no key")
    # Non-causal: every row sees every key, whatever the lengths; rows are independent.
    o, lse = impl.forward(q, k, v, scale, False)
    for i in (0, n0, Lq - 1):
        o1, lse1 = impl.forward(q[i:i + 1], k, v, scale, False)
        _close(o[i:i + 1], o1, 1e-12, "non-causal O row vs a one-row problem")
        _close(lse[i:i + 1], lse1, 1e-12, "non-causal LSE row vs a one-row problem")


def pin_library_sdpa_rect(impl):
    """Lq != Lk against torch's fp64 CPU scaled_dot_product_attention and its autograd, with the
    causal mask built explicitly (query i sees key j iff j <= i + Lk - Lq)."""
    import torch
    import torch.nn.functional as F

    r = _rng(16)
    for (Lq, Lk, D, causal, scale) in ((9, 23, 8, True, 0.3), (23, 9, 8, False, 0.3),
                                       (5, 40, 16, True, 0.2), (17, 17, 4, True, 0.5)):
        q, do = r.standard_normal((Lq, D)), r.standard_normal((Lq, D))
        k, v = r.standard_normal((Lk, D)), r.standard_normal((Lk, D))
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        mask = None
        if causal:
            mask = torch.tensor(np.arange(Lk)[None, :] <= np.arange(Lq)[:, None] + (Lk - Lq))
        to = F.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                            attn_mask=mask, scale=scale)[0, 0]
        to.backward(torch.tensor(do, dtype=torch.float64))
        o, _ = impl.forward(q, k, v, scale, causal)
        _close(o, to.detach().numpy(), 1e-12, f"O vs torch sdpa (Lq={Lq}, Lk={Lk})")
        dq, dk, dv, _ = impl.backward(q, k, v, do, scale, causal)
        _close(dq, tq.grad.numpy(), 1e-12, f"dQ vs torch sdpa (Lq={Lq}, Lk={Lk})")
        _close(dk, tk.grad.numpy(), 1e-12, f"dK vs torch sdpa (Lq={Lq}, Lk={Lk})")
        _close(dv, tv.grad.numpy(), 1e-12, f"dV vs torch sdpa (Lq={Lq}, Lk={Lk})")


def pin_finite_differences_rect(impl):
    """Central differences of sum(O * dO) with Lq != Lk, including rows that see no key."""
    r = _rng(17)
    h = 1e-6
    for (Lq, Lk, D, causal) in ((3, 6, 2, True), (6, 3, 2, True), (4, 7, 3, False)):
        q, do = r.standard_normal((Lq, D)), r.standard_normal((Lq, D))
        k, v = r.standard_normal((Lk, D)), r.standard_normal((Lk, D))
        scale = 0.9
        dq, dk, dv, _ = impl.backward(q, k, v, do, scale, causal)
        for name, g in (("q", dq), ("k", dk), ("v", dv)):
            x = {"q": q, "k": k, "v": v}[name]
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                args = [{"q": q, "k": k, "v": v}, {"q": q, "k": k, "v": v}]
                for sgn, a in zip((1.0, -1.0), args):
                    xs = x.copy()
                    xs[idx] += sgn * h
                    a[name] = xs
                fp = _loss(impl, args[0]["q"], args[0]["k"], args[0]["v"], do, scale, causal)
                fm = _loss(impl, args[1]["q"], args[1]["k"], args[1]["v"], do, scale, causal)
                num[idx] = (fp - fm) / (2 * h)
            err = np.linalg.norm(g - num)
            assert err <= 1e-6 * max(np.linalg.norm(num), 1.0), \
                f"d{name} vs finite differences (Lq={Lq}, Lk={Lk}, causal={causal}): {err:.2e}"


ALL_PINS = [
    pin_probs_are_distributions,
    pin_single_key,
    pin_identical_keys,
    pin_causal_row0,
    pin_zero_queries,
    pin_key_shift,
    pin_dominant_key,
    pin_finite_differences,
    pin_gradient_invariants,
    pin_zero_queries_backward,
    pin_library_sdpa,
    pin_suffix_queries,
    pin_more_queries_than_keys,
    pin_library_sdpa_rect,
    pin_finite_differences_rect,
]
