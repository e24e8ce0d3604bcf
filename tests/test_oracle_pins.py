"""The fp64 oracle against facts fixed by the mathematics (CPU only)."""
import numpy as np
import pytest

import pins


class OracleImpl:
    """Adapts the oracle to the one-head interface the pins use."""

    def __init__(self, mod, block_doubles=0):
        self.mod = mod
        self.block_doubles = block_doubles

    def forward(self, q, k, v, scale, causal):
        return self.mod.forward(q, k, v, scale, causal, block_doubles=self.block_doubles)

    def backward(self, q, k, v, do, scale, causal):
        return self.mod.backward(q, k, v, do, scale, causal, block_doubles=self.block_doubles)

    def probs(self, q, k, scale, causal):
        return self.mod.probs(q, k, scale, causal)


@pytest.mark.parametrize("block_doubles", [0, 40], ids=["whole_head", "row_blocks"])
@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_mod, pin, block_doubles):
    pin(OracleImpl(oracle_mod, block_doubles))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", list(range(1, 34)))
def test_online_recurrence_matches_two_pass(oracle_mod, L, causal):
    """The streaming recurrence (running max/sum, rescaled partial O) equals the
    materialised two-pass softmax for every tile shape, tail tiles included."""
    r = np.random.default_rng(100 + L)
    D = 5
    q, k, v = (r.standard_normal((L, D)) * 2.0 for _ in range(3))
    o_ref, lse_ref = oracle_mod.forward(q, k, v, 0.6, causal)
    for bq in (1, 2, 4, 7):
        for bk in (1, 2, 4, 7):
            o, lse = oracle_mod.online_forward(q, k, v, 0.6, causal, bq, bk)
            np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_heads_are_independent(oracle_mod):
    """A [B,H,L,D] call equals per-head calls: head strides are honoured."""
    r = np.random.default_rng(12)
    B, H, L, D = 2, 3, 11, 4
    q, k, v, do = (r.standard_normal((B, H, L, D)) for _ in range(4))
    o, lse = oracle_mod.forward(q, k, v, 0.5, True)
    dq, dk, dv, delta = oracle_mod.backward(q, k, v, do, 0.5, True)
    for b in range(B):
        for h in range(H):
            o1, l1 = oracle_mod.forward(q[b, h], k[b, h], v[b, h], 0.5, True)
            g1 = oracle_mod.backward(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, True)
            np.testing.assert_array_equal(o[b, h], o1)
            np.testing.assert_array_equal(lse[b, h], l1)
            for a, c in zip((dq, dk, dv, delta), g1):
                np.testing.assert_array_equal(a[b, h], c)


def test_multihead_against_library(oracle_mod):
    """Batched heads against torch's fp64 CPU attention (an independent implementation)."""
    import torch
    import torch.nn.functional as F

    r = np.random.default_rng(13)
    B, H, L, D = 2, 3, 40, 16
    q, k, v, do = (r.standard_normal((B, H, L, D)) for _ in range(4))
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
        to = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.25)
        to.backward(torch.tensor(do))
        o, _ = oracle_mod.forward(q, k, v, 0.25, causal)
        dq, dk, dv, _ = oracle_mod.backward(q, k, v, do, 0.25, causal)
        np.testing.assert_allclose(o, to.detach().numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


def test_empty_sequence(oracle_mod):
    """L = 0 is a valid, empty problem."""
    z = np.zeros((1, 2, 0, 8))
    o, lse = oracle_mod.forward(z, z, z, 1.0, True)
    assert o.shape == (1, 2, 0, 8) and lse.shape == (1, 2, 0)


@pytest.mark.parametrize("block_doubles", [0, 40], ids=["whole_head", "row_blocks"])
def test_queries_without_keys(oracle_mod, block_doubles):
    """Lk = 0: every query row's softmax is over an empty set (O = 0, LSE = -inf, dQ = 0), in both
    the whole-head and the row-block paths."""
    r = np.random.default_rng(14)
    q, do = r.standard_normal((5, 3)), r.standard_normal((5, 3))
    k = np.zeros((0, 3))
    for causal in (False, True):
        o, lse = oracle_mod.forward(q, k, k, 0.5, causal, block_doubles=block_doubles)
        assert np.all(o == 0.0) and np.all(np.isneginf(lse))
        dq, dk, dv, _ = oracle_mod.backward(q, k, k, do, 0.5, causal, block_doubles=block_doubles)
        assert np.all(dq == 0.0) and dk.shape == (0, 3) and dv.shape == (0, 3)
