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
            Lq, Lk = q.shape[0], k.shape[0]
            off = 1 if self.m == "mask_off_by_one" else 0
            shift = 0 if self.m == "mask_top_left" else Lk - Lq
            mask = np.arange(Lk)[None, :] > np.arange(Lq)[:, None] + shift + off
            if self.m == "mask_transposed":
                mask = mask.T if Lq == Lk else mask[::-1, ::-1]
            s = np.where(mask, -np.inf, s)
        return s

    @staticmethod
    def _exp_rows(s):
        """exp(s - rowmax) with rows that see no key left at zero; returns (e, rowmax)."""
        m = s.max(axis=1)
        safe = np.where(np.isneginf(m), 0.0, m)
        return np.exp(s - safe[:, None]), m

    def probs(self, q, k, scale, causal):
        e, _ = self._exp_rows(self._logits(q, k, scale, causal))
        if self.m == "normalise_columns":
            den = e.sum(axis=0, keepdims=True)
        else:
            den = e.sum(axis=1, keepdims=True)
        return np.divide(e, den, out=np.zeros_like(e), where=den > 0)

    def forward(self, q, k, v, scale, causal):
        e, m = self._exp_rows(self._logits(q, k, scale, causal))
        p = self.probs(q, k, scale, causal)
        o = p @ (k if self.m == "swap_kv" else v)
        with np.errstate(divide="ignore"):
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
             "dq_transposed", "dk_drop_scale", "dk_uses_k", "mask_top_left"]


def _failing_pins(impl):
    """Names of the pins the implementation violates (a wrong value, or a shape error that a
    transposed operand raises once Lq != Lk)."""
    failed = []
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes_every_pin():
    assert _failing_pins(NumpyAttention()) == []


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_pins_catch_mutation(mutation):
    failed = _failing_pins(NumpyAttention(mutation))
    assert failed, f"no pin caught the planted mistake '{mutation}'"
