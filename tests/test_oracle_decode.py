"""Pins for the oracle's decode step over a paged key/value cache (CPU only).

A decode step is one new query row per sequence attending to all of that sequence's cached
tokens ("FlashAttention principles and engineering practice", section 4.2: served with
PagedAttention, block_size 16).  What fixes it, independently of the oracle's own gather:
* it is the LAST row of the causal attention over the whole sequence (the newest token sees every
  earlier one), which the prefill oracle computes and is itself pinned;
* where the pages sit in the cache is irrelevant: permuting the physical pages (and the block
  table with them) changes nothing, bit for bit;
* closed forms: an empty cache (O = 0, LSE = -inf) and a single cached token (O = V, LSE = scale q.k).
Planted mistakes in a numpy copy of the gather (wrong page, wrong slot, a dropped partial page, the
wrong head) must each trip a pin.
"""
import numpy as np
import pytest

PAGE = 16


def make_paged(rng, lens, H, D, extra_pages=5):
    """Random per-sequence K/V stored in shuffled physical pages; returns the dense copies."""
    B = len(lens)
    max_pages = max(1, max((n + PAGE - 1) // PAGE for n in lens))
    need = sum((n + PAGE - 1) // PAGE for n in lens)
    num_pages = need + extra_pages
    kc = rng.standard_normal((num_pages, H, PAGE, D))  # unused pages hold garbage
    vc = rng.standard_normal((num_pages, H, PAGE, D))
    order = rng.permutation(num_pages)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    dense_k, dense_v = [], []
    nxt = 0
    for b, n in enumerate(lens):
        k = rng.standard_normal((H, n, D))
        v = rng.standard_normal((H, n, D))
        for pg in range((n + PAGE - 1) // PAGE):
            phys = order[nxt]
            nxt += 1
            table[b, pg] = phys
            cnt = min(PAGE, n - pg * PAGE)
            kc[phys, :, :cnt] = k[:, pg * PAGE:pg * PAGE + cnt]
            vc[phys, :, :cnt] = v[:, pg * PAGE:pg * PAGE + cnt]
        dense_k.append(k)
        dense_v.append(v)
    table[table < 0] = 0  # entries past a sequence's pages are never read
    return kc, vc, table, dense_k, dense_v


def pin_last_row_of_prefill(decode, oracle):
    rng = np.random.default_rng(40)
    H, D, scale = 3, 8, 0.4
    lens = [1, 15, 16, 17, 40, 64, 5]
    kc, vc, table, dk, dv = make_paged(rng, lens, H, D)
    qfull = [rng.standard_normal((H, n, D)) for n in lens]
    q = np.stack([qf[:, -1] for qf in qfull])
    o, lse = decode(q, kc, vc, table, np.array(lens), scale)
    for b, n in enumerate(lens):
        for h in range(H):
            o_ref, lse_ref = oracle.forward(qfull[b][h], dk[b][h], dv[b][h], scale, True)
            assert np.max(np.abs(o[b, h] - o_ref[-1])) <= 1e-12, (b, h)
            assert abs(lse[b, h] - lse_ref[-1]) <= 1e-12, (b, h)


def pin_page_permutation(decode, oracle):
    rng = np.random.default_rng(41)
    H, D, scale = 2, 4, 0.7
    lens = [33, 1, 48, 20]
    kc, vc, table, _, _ = make_paged(rng, lens, H, D)
    q = rng.standard_normal((len(lens), H, D))
    o, lse = decode(q, kc, vc, table, np.array(lens), scale)
    perm = rng.permutation(kc.shape[0])       # physical page p moves to slot inv[p]
    inv = np.argsort(perm)
    o2, lse2 = decode(q, kc[perm], vc[perm], inv[table].astype(np.int32), np.array(lens), scale)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def pin_empty_and_single(decode, oracle):
    rng = np.random.default_rng(42)
    H, D, scale = 2, 4, 0.9
    kc, vc, table, dk, dv = make_paged(rng, [0, 1], H, D)
    q = rng.standard_normal((2, H, D))
    o, lse = decode(q, kc, vc, table, np.array([0, 1]), scale)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    for h in range(H):
        assert np.max(np.abs(o[1, h] - dv[1][h][0])) <= 1e-14
        assert abs(lse[1, h] - scale * float(q[1, h] @ dk[1][h][0])) <= 1e-14


PINS = [pin_last_row_of_prefill, pin_page_permutation, pin_empty_and_single]


class NumpyDecode:
    """A numpy restatement of the gather + one-row softmax, with optional planted mistakes."""

    def __init__(self, mutation=None):
        self.m = mutation

    def __call__(self, q, kc, vc, table, lens, scale):
        B, H, D = q.shape
        o = np.zeros((B, H, D))
        lse = np.full((B, H), -np.inf)
        for b in range(B):
            n = int(lens[b])
            if self.m == "drop_partial_page":
                n = (n // PAGE) * PAGE
            if n == 0:
                continue
            t = np.arange(n)
            pg = t // PAGE + (1 if self.m == "page_off_by_one" else 0)
            slot = (PAGE - 1 - t % PAGE) if self.m == "slot_reversed" else t % PAGE
            phys = table[b, np.minimum(pg, table.shape[1] - 1)]
            for h in range(H):
                hh = 0 if self.m == "head_zero" else h
                k = kc[phys, hh, slot]
                v = vc[phys, hh, slot]
                s = scale * (k @ q[b, h])
                mx = s.max()
                e = np.exp(s - mx)
                o[b, h] = (e @ v) / e.sum()
                lse[b, h] = mx + np.log(e.sum())
        return o, lse


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_decode_pin(oracle_mod, pin):
    pin(oracle_mod.decode_paged, oracle_mod)


def test_numpy_copy_passes_every_pin(oracle_mod):
    for pin in PINS:
        pin(NumpyDecode(), oracle_mod)


@pytest.mark.parametrize("mutation", ["page_off_by_one", "slot_reversed", "drop_partial_page",
                                      "head_zero"])
def test_pins_catch_decode_mutation(oracle_mod, mutation):
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(NumpyDecode(mutation), oracle_mod)
        except (AssertionError, IndexError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught '{mutation}'"


def test_oracle_decode_refuses_bad_pages(oracle_mod):
    rng = np.random.default_rng(43)
    kc, vc, table, _, _ = make_paged(rng, [20], 1, 4)
    q = rng.standard_normal((1, 1, 4))
    bad = table.copy()
    bad[0, 1] = kc.shape[0]  # past the last page
    with pytest.raises(RuntimeError):
        oracle_mod.decode_paged(q, kc, vc, bad, np.array([20]), 0.5)
    with pytest.raises(RuntimeError):
        oracle_mod.decode_paged(q, kc, vc, table, np.array([40]), 0.5)  # longer than the table
