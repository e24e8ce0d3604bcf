"""Pins for dropout on P in the fp64 oracle (CPU only).

The keep mask comes from Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011).  What fixes it:
* the generator reproduces the published known-answer vectors of Philox-4x32-10;
* with V the identity, O = P o Z exposes every factor Z_ij, which must equal what an independent
  Python restatement of the generator (itself checked on the same vectors) gives for the stated
  counter layout: word j % 4 of counter (j / 4, i, bh, 0), key = the seed, dropped iff the word is
  below floor(p * 2^32), kept entries scaled by 1/(1-p);
* p = 0 is the plain attention;
* dropout is unbiased: the mean of O over many seeds tends to the plain O;
* the backward is the gradient of sum(O * dO) for a fixed mask (central finite differences), and
  Delta = rowsum(dO o O) holds with the dropped O.
Planted mistakes (mask on S instead of P, no 1/(1-p), the wrong output word, the mask transposed in
the backward) must each trip a pin.
"""
import math

import numpy as np
import pytest

MASK = 0xFFFFFFFF
KAT = [((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
       ((MASK,) * 4, (MASK, MASK), (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
       ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
        (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1))]


def py_philox(ctr, key):
    """Philox-4x32-10 from its published definition (independent of the oracle's C code)."""
    c = list(ctr)
    k0, k1 = key
    for r in range(10):
        if r:
            k0, k1 = (k0 + 0x9E3779B9) & MASK, (k1 + 0xBB67AE85) & MASK
        p0, p1 = 0xD2511F53 * c[0], 0xCD9E8D57 * c[2]
        c = [(p1 >> 32) ^ c[1] ^ k0, p1 & MASK, (p0 >> 32) ^ c[3] ^ k1, p0 & MASK]
    return c


def py_factors(bh, Lq, Lk, p, seed):
    """Z [Lq, Lk] for head bh, from the stated counter layout."""
    thr = math.floor(p * 2 ** 32)
    key = (seed & MASK, seed >> 32)
    z = np.ones((Lq, Lk))
    if thr == 0:
        return z
    for i in range(Lq):
        for j4 in range(0, Lk, 4):
            w = py_philox((j4 >> 2, i, bh, 0), key)
            for jj in range(j4, min(Lk, j4 + 4)):
                z[i, jj] = 0.0 if w[jj & 3] < thr else 1.0 / (1.0 - p)
    return z


def test_philox_known_answers(oracle_mod):
    for ctr, key, want in KAT:
        assert py_philox(ctr, key) == list(want)
        assert oracle_mod.philox4x32_10(ctr, key) == list(want)


class OracleDrop:
    def __init__(self, mod):
        self.mod = mod

    def forward(self, q, k, v, scale, causal, p, seed):
        return self.mod.forward(q, k, v, scale, causal, dropout_p=p, seed=seed)

    def backward(self, q, k, v, do, scale, causal, p, seed):
        return self.mod.backward(q, k, v, do, scale, causal, dropout_p=p, seed=seed)


def pin_mask_layout(impl, oracle):
    """V = I exposes Z: O_ij = P_ij Z_ij, on several heads, causal and not, Lq != Lk."""
    r = np.random.default_rng(50)
    B, H, Lq, Lk = 1, 3, 7, 11
    D = Lk  # V = I needs V's width to be Lk, and q, k, v share D
    for causal, p, seed in ((False, 0.3, 12345), (True, 0.5, (7 << 32) | 99)):
        q = r.standard_normal((B, H, Lq, D))
        k = r.standard_normal((B, H, Lk, D))
        v = np.tile(np.eye(Lk), (B, H, 1, 1))
        o, _ = impl.forward(q, k, v, 0.8, causal, p, seed)
        for h in range(H):
            P = oracle.probs(q[0, h], k[0, h], 0.8, causal)
            Z = py_factors(h, Lq, Lk, p, seed)
            assert np.max(np.abs(o[0, h] - P * Z)) <= 1e-12, (h, causal)


def pin_zero_rate(impl, oracle):
    r = np.random.default_rng(51)
    q, k, v, do = (r.standard_normal((1, 2, 9, 4)) for _ in range(4))
    o0, l0 = oracle.forward(q, k, v, 0.5, True)
    o1, l1 = impl.forward(q, k, v, 0.5, True, 0.0, 77)
    assert np.max(np.abs(o0 - o1)) <= 1e-12 and np.max(np.abs(l0 - l1)) <= 1e-12
    g0 = oracle.backward(q, k, v, do, 0.5, True)
    g1 = impl.backward(q, k, v, do, 0.5, True, 0.0, 77)
    for a, b in zip(g0, g1):
        assert np.max(np.abs(a - b)) <= 1e-12


def pin_unbiased(impl, oracle):
    """Mean of O over 400 seeds against the plain O: each entry's error stays within 5 standard
    errors of the per-seed spread."""
    r = np.random.default_rng(52)
    q, k, v = (r.standard_normal((1, 1, 6, 3)) for _ in range(3))
    o_plain, lse_plain = oracle.forward(q, k, v, 0.7, False)
    outs = []
    for s in range(400):
        o, lse = impl.forward(q, k, v, 0.7, False, 0.25, 1000 + s)
        assert np.array_equal(lse, lse_plain), "the LSE is that of P, not of P o Z"
        outs.append(o)
    outs = np.array(outs)
    se = outs.std(axis=0) / math.sqrt(len(outs)) + 1e-12
    assert np.all(np.abs(outs.mean(axis=0) - o_plain) <= 5 * se + 1e-9)


def pin_gradients_with_dropout(impl, oracle):
    r = np.random.default_rng(53)
    h = 1e-6
    for (Lq, Lk, causal) in ((5, 5, True), (4, 7, False)):
        q, do = r.standard_normal((1, 2, Lq, 3)), r.standard_normal((1, 2, Lq, 3))
        k, v = r.standard_normal((1, 2, Lk, 3)), r.standard_normal((1, 2, Lk, 3))
        p, seed = 0.4, 2024
        dq, dk, dv, delta = impl.backward(q, k, v, do, 0.6, causal, p, seed)
        o, _ = impl.forward(q, k, v, 0.6, causal, p, seed)
        assert np.max(np.abs(delta - np.sum(do * o, axis=-1))) <= 1e-11, "Delta = rowsum(dO o O)"

        def loss(qq, kk, vv):
            return float(np.sum(impl.forward(qq, kk, vv, 0.6, causal, p, seed)[0] * do))

        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                a = {"q": q, "k": k, "v": v}
                b = dict(a)
                a[name], b[name] = xp, xm
                num[idx] = (loss(a["q"], a["k"], a["v"]) - loss(b["q"], b["k"], b["v"])) / (2 * h)
            assert np.linalg.norm(g - num) <= 1e-6 * max(np.linalg.norm(num), 1.0), name


PINS = [pin_mask_layout, pin_zero_rate, pin_unbiased, pin_gradients_with_dropout]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_dropout_pin(oracle_mod, pin):
    pin(OracleDrop(oracle_mod), oracle_mod)


class NumpyDrop:
    """numpy restatement of attention with dropout (test-side Philox), with planted mistakes."""

    def __init__(self, mutation=None):
        self.m = mutation

    def _z(self, bh, Lq, Lk, p, seed):
        z = py_factors(bh, Lq, Lk, p, seed)
        if self.m == "no_rescale":
            z = (z > 0).astype(float)
        if self.m == "wrong_word":
            z = py_factors(bh, Lk, Lq, p, seed).T if Lq == Lk else z[:, ::-1]
        return z

    def _probs(self, q, k, scale, causal):
        s = scale * (q @ k.T)
        Lq, Lk = s.shape
        if causal:
            s = np.where(np.arange(Lk)[None] > np.arange(Lq)[:, None] + Lk - Lq, -np.inf, s)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        return e / e.sum(axis=1, keepdims=True), (m[:, 0] + np.log(e.sum(axis=1)))

    def forward(self, q, k, v, scale, causal, p, seed):
        B, H, Lq, D = q.shape
        o = np.zeros_like(q)
        lse = np.zeros((B, H, Lq))
        for b in range(B):
            for h in range(H):
                P, l = self._probs(q[b, h], k[b, h], scale, causal)
                Z = self._z(b * H + h, Lq, k.shape[2], p, seed)
                if self.m == "mask_on_s":
                    P = P * (Z > 0)
                    P = P / P.sum(axis=1, keepdims=True).clip(1e-300)
                    o[b, h] = P @ v[b, h]
                else:
                    o[b, h] = (P * Z) @ v[b, h]
                lse[b, h] = l
        return o, lse

    def backward(self, q, k, v, do, scale, causal, p, seed):
        B, H, Lq, D = q.shape
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        delta = np.zeros((B, H, Lq))
        for b in range(B):
            for h in range(H):
                P, _ = self._probs(q[b, h], k[b, h], scale, causal)
                Z = self._z(b * H + h, Lq, k.shape[2], p, seed)
                Zb = Z.T.T if self.m != "backward_transposed" or Lq != k.shape[2] else Z.T
                dv[b, h] = (P * Z).T @ do[b, h]
                dP = (do[b, h] @ v[b, h].T) * Zb
                dl = (P * dP).sum(axis=1)
                dS = P * (dP - dl[:, None])
                dq[b, h] = scale * dS @ k[b, h]
                dk[b, h] = scale * dS.T @ q[b, h]
                delta[b, h] = dl
        return dq, dk, dv, delta


def test_numpy_copy_passes_every_pin(oracle_mod):
    for pin in PINS:
        pin(NumpyDrop(), oracle_mod)


@pytest.mark.parametrize("mutation", ["mask_on_s", "no_rescale", "wrong_word",
                                      "backward_transposed"])
def test_pins_catch_dropout_mutation(oracle_mod, mutation):
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(NumpyDrop(mutation), oracle_mod)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught '{mutation}'"
