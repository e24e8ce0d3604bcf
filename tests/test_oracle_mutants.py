"""Plants plausible mistakes in a CPU copy of the method and checks the pins catch each.

The copy below is a small numpy restatement of the same definition the oracle follows; each
mutant changes one detail (a dropped term, a wrong sign or index, a transposed operand).  If
a pin set let one of these through, it would not be pinning the oracle.
"""
import math

import numpy as np
import pytest

import pins


class NumpyAttention:
    def __init__(self, mutation=None):
        self.m = mutation

    def _logits(self, q, k, scale, causal):
        s = (q @ k.T) * (1.0 if self.m == "drop_scale" else scale)
        if causal:
            L = q.shape[0]
            off = 1 if self.m == "mask_off_by_one" else 0
            mask = np.arange(L)[None, :] > np.arange(L)[:, None] + off
            if self.m == "mask_transposed":
                mask = mask.T
            s = np.where(mask, -np.inf, s)
        return s

    def probs(self, q, k, scale, causal):
        s = self._logits(q, k, scale, causal)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        if self.m == "normalise_columns":
            return e / e.sum(axis=0, keepdims=True)
        return e / e.sum(axis=1, keepdims=True)

    def forward(self, q, k, v, scale, causal):
        s = self._logits(q, k, scale, causal)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        p = self.probs(q, k, scale, causal)
        o = p @ (k if self.m == "swap_kv" else v)
        if self.m == "lse_log2":
            lse = m + np.log2(e.sum(axis=1))
        elif self.m == "lse_drop_max":
            lse = np.log(e.sum(axis=1))
        else:
            lse = m + np.log(e.sum(axis=1))
        return o, lse

    def backward(self, q, k, v, do, scale, causal):
        p = self.probs(q, k, scale, causal)
        dv = (p @ do) if self.m == "dv_untransposed" else p.T @ do
        dp = do @ v.T
        delta = (p * dp).sum(axis=1)
        if self.m == "ds_drop_delta":
            ds = p * dp
        elif self.m == "ds_sign":
            ds = p * (delta[:, None] - dp)
        else:
            ds = p * (dp - delta[:, None])
        dq = scale * (ds.T @ k if self.m == "dq_transposed" else ds @ k)
        dk = (1.0 if self.m == "dk_drop_scale" else scale) * (ds.T @ q)
        if self.m == "dk_uses_k":
            dk = scale * (ds.T @ k)
        return dq, dk, dv, delta


MUTATIONS = ["drop_scale", "mask_off_by_one", "mask_transposed", "normalise_columns", "swap_kv",
             "lse_log2", "lse_drop_max", "dv_untransposed", "ds_drop_delta", "ds_sign",
             "dq_transposed", "dk_drop_scale", "dk_uses_k"]


def _failing_pins(impl):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes_every_pin():
    assert _failing_pins(NumpyAttention()) == []


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_pins_catch_mutation(mutation):
    failed = _failing_pins(NumpyAttention(mutation))
    assert failed, f"no pin caught the planted mistake '{mutation}'"
