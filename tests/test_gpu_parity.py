"""CUDA path vs the fp64 oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import gpu_helpers as gh
import tiled_attention_08_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gh.require_gpu()


SMALL = [(L, D, causal, dt)
         for D in (64, 128)
         for dt in (torch.bfloat16, torch.float16)
         for causal in (False, True)
         for L in (1, 3, 127, 129, 200, 384)]


@pytest.mark.parametrize("L,D,causal,dtype", SMALL,
                         ids=lambda x: str(x).replace("torch.", ""))
def test_small_shapes_full_tensors(oracle_mod, L, D, causal, dtype):
    """Every head, every row: several tiles, ragged tails, both masks, both dtypes."""
    w = workloads.custom(2, 3, L, D, causal, dtype)
    inp = workloads.make_inputs(w, seed=L * 7 + D)
    out = gh.run_gpu(w, inp, backward=True)
    for b in range(w.B):
        for h in range(w.H):
            gh.check_head(oracle_mod, w, inp, out, b, h, backward=True)


@pytest.mark.parametrize("L,D,causal", [(L, D, c) for L in (377, 384) for D in (64, 128)
                                         for c in (False, True)])
def test_persistent_rounds(oracle_mod, L, D, causal):
    """More work items than SMs (2 x 40 heads x 3 query or key tiles, 2 x 40 x 2 query-tile
    pairs) with short rows: the forward, the dK/dV pass and the dQ pass all run their persistent
    forms, each CTA taking items in more than one round; the item order gives every head items
    in several rounds, so each sampled head crosses the hand-offs between items."""
    n_tiles = (L + 127) // 128
    total = 2 * 40 * n_tiles
    assert total > torch.cuda.get_device_properties(0).multi_processor_count
    assert (n_tiles + 1 if causal else 2 * n_tiles) <= 64  # mean key tiles <= 32: persistent
    w = workloads.custom(2, 40, L, D, causal, torch.bfloat16)
    inp = workloads.make_inputs(w, seed=L + D + int(causal))
    out = gh.run_gpu(w, inp, backward=True)
    for b, h in gh.sample_heads(w.B, w.H):
        gh.check_head(oracle_mod, w, inp, out, b, h, backward=True)


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_workload_full_size(oracle_mod, name):
    """Each workload at its full size in the benchmark's launch configuration; heads are
    compared in full for the two smallest workloads, else on a sampled set of heads."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, seed=0, with_do=w.backward)
    out = gh.run_gpu(w, inp, backward=w.backward)
    heads = ([(b, h) for b in range(w.B) for h in range(w.H)] if w.B * w.H * w.L <= 32 * 2048
             else gh.sample_heads(w.B, w.H))
    for b, h in heads:
        gh.check_head(oracle_mod, w, inp, out, b, h, backward=w.backward)
    # Properties that hold at any size, checked on every head.
    o = out["o"].float()
    assert torch.isfinite(o).all() and torch.isfinite(out["lse"]).all()
    if w.backward:
        # Every head: sum_j dV_j = sum_i dO_i (rows of P sum to one), up to the 16-bit
        # rounding of P and of the stored dV.
        do = inp["do"].to("cuda", torch.float32)
        dv_sum = out["dv"].float().sum(dim=2)
        assert torch.allclose(dv_sum, do.sum(dim=2), atol=0.05 * np.sqrt(w.L), rtol=2e-2)
        for t in ("dq", "dk", "dv"):
            assert torch.isfinite(out[t].float()).all(), t


def test_deterministic(oracle_mod):
    """Forward and backward are bit-reproducible (no atomics anywhere)."""
    w = workloads.custom(2, 4, 700, 128, True, torch.bfloat16)
    inp = workloads.make_inputs(w, seed=5)
    a = gh.run_gpu(w, inp)
    b = gh.run_gpu(w, inp)
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_row_scaled_extremes(oracle_mod):
    """Large logits (Q rows scaled up to x4, keys stretched up to x3 along the sequence, scale
    1/sqrt(64)): the running max moves by far more than the rescale threshold across tiles,
    exercising the O rescale path."""
    w = workloads.Workload("row_scaled_unit_scale", 1, 2, 640, 64, False, torch.bfloat16,
                           row_scaled=True)
    inp = workloads.make_inputs(w, seed=9)
    # Sort keys so that later tiles carry larger logits for positive queries.
    inp["k"] = inp["k"] * torch.linspace(0.2, 3.0, w.L).reshape(1, 1, -1, 1).to(inp["k"].dtype)
    out = gh.run_gpu(w, inp)
    for b, h in [(0, 0), (0, 1)]:
        gh.check_head(oracle_mod, w, inp, out, b, h)


@pytest.mark.parametrize("scale", (1.0, 0.3, -0.125, 0.0))
@pytest.mark.parametrize("D,dtype", ((64, torch.float16), (128, torch.bfloat16)),
                         ids=("D64-fp16", "D128-bf16"))
@pytest.mark.parametrize("causal", (False, True))
def test_scale_argument(oracle_mod, scale, D, dtype, causal):
    """The scale multiplies Q K^T before the mask and the softmax for any finite value: larger
    than 1/sqrt(D) (a peaked softmax), negative (the row maximum of the logits is then taken
    where Q K^T is smallest) and zero (a uniform softmax).  Row-scaled queries widen the logit
    range; three query tiles with a ragged tail."""
    w = workloads.custom(1, 2, 300, D, causal, dtype, row_scaled=True, scale=scale)
    inp = workloads.make_inputs(w, seed=31 + D)
    out = gh.run_gpu(w, inp, backward=True)
    for h in range(w.H):
        gh.check_head(oracle_mod, w, inp, out, 0, h, backward=True)


def test_timeout_reported_and_context_survives(oracle_mod):
    """A device wait that nothing completes gives up after its limit, the status word reports
    FA_ERR_TIMEOUT, and the next call still works."""
    s = torch.cuda.current_stream().cuda_stream
    assert fa.fa_get_device_status(s) == fa.FA_OK
    assert fa.fa_selftest_wait_timeout(50_000_000, s) == fa.FA_OK  # 50 ms
    assert fa.fa_get_device_status(s) == fa.FA_ERR_TIMEOUT
    assert fa.fa_get_device_status(s) == fa.FA_OK  # read-and-clear
    w = workloads.custom(1, 2, 256, 64, True, torch.float16)
    inp = workloads.make_inputs(w, seed=3)
    out = gh.run_gpu(w, inp)
    gh.check_head(oracle_mod, w, inp, out, 0, 1)
