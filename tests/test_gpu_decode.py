"""CUDA decode step over a paged key/value cache vs the fp64 oracle, through fa_decode_paged.

One new query row per sequence attends to all of its cached tokens, stored in 16-token pages
through a block table ("FlashAttention principles and engineering practice", section 4.2).  The
cases cover empty and one-token sequences, partial last pages, pages in shuffled physical order
with noise in the unused slots, the split-and-combine path (few sequences, many pages), both
head sizes and dtypes, the full Llama-2-7B-shaped batch on sampled sequences, and out-of-range
device data (reported as an argument error, never copied from).
"""
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


def _check_sequence(oracle, w, inp, out_o, out_lse, b, heads=None):
    """Sequence b of the GPU result against the oracle on that sequence's pages only."""
    n = int(inp["seq_lens"][b])
    n_pages = (n + workloads.PAGE_TOKENS - 1) // workloads.PAGE_TOKENS
    pages = inp["block_tables"][b, :n_pages].long().cpu()
    kc = gh.f64(inp["k_cache"].index_select(0, pages.to(inp["k_cache"].device)))
    vc = gh.f64(inp["v_cache"].index_select(0, pages.to(inp["v_cache"].device)))
    table = np.arange(max(n_pages, 1), dtype=np.int32)[None]
    if kc.shape[0] == 0:  # an empty sequence reads no page; give the oracle one of noise
        kc = np.zeros((1,) + tuple(inp["k_cache"].shape[1:]))
        vc = kc
    o_ref, lse_ref = oracle.decode_paged(gh.f64(inp["q"][b:b + 1]), kc, vc, table,
                                         np.array([n]), w.scale)
    o = gh.f64(out_o[b])
    lse = gh.f64(out_lse[b])
    for h in (heads if heads is not None else range(w.H)):
        if n == 0:
            assert np.all(o[h] == 0.0) and np.isneginf(lse[h]), (b, h)
            continue
        err = gh.o_errors(o[h], o_ref[0, h], w.dtype)
        assert err["o_max"] <= gh.O_MAX_ABS and err["o_mean"] <= gh.O_MEAN_ABS, (b, h, err)
        assert abs(lse[h] - lse_ref[0, h]) <= gh.LSE_MAX_ABS, (b, h, lse[h], lse_ref[0, h])


def _run(w, inp):
    o, lse = fa.decode_paged(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                             inp["seq_lens"], w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("D,dtype", [(64, torch.float16), (128, torch.bfloat16),
                                     (64, torch.bfloat16), (128, torch.float16)],
                         ids=lambda x: str(x).replace("torch.", ""))
def test_decode_mixed_lengths(oracle_mod, D, dtype):
    lens = [0, 1, 15, 16, 17, 129, 300, 1000]
    w = workloads.DecodeWorkload("decode_small", len(lens), 3, D, dtype, 0, 0, extra_pages=7)
    inp = workloads.make_decode_inputs(w, seed=D, device="cuda", lens=lens)
    o, lse = _run(w, inp)
    for b in range(w.B):
        _check_sequence(oracle_mod, w, inp, o, lse, b)


@pytest.mark.parametrize("lens,H", [([3000], 2), ([2000, 0], 4), ([17, 4096, 1], 1)])
def test_decode_split_and_combine(oracle_mod, lens, H):
    """Few (sequence, head) pairs and many pages: the page range is split across CTAs and the
    splits' results are merged (splits past a short sequence's pages weigh nothing)."""
    w = workloads.DecodeWorkload("decode_splits", len(lens), H, 128, torch.bfloat16, 0, 0)
    assert fa.fa_decode_workspace_bytes(w.B, w.H, w.D, (max(lens) + 15) // 16) > 0
    inp = workloads.make_decode_inputs(w, seed=len(lens), device="cuda", lens=lens)
    o, lse = _run(w, inp)
    for b in range(w.B):
        _check_sequence(oracle_mod, w, inp, o, lse, b)


def test_decode_full_size(oracle_mod):
    """The Llama-2-7B decode batch (256 sequences of U[1, 4096] tokens, 32 heads of 128) in the
    benchmark's launch configuration; sequences compared on a sample, every head of each."""
    w = workloads.DECODE_WORKLOADS["decode_llama2_7b_B256"]
    inp = workloads.make_decode_inputs(w, seed=0, device="cuda")
    o, lse = _run(w, inp)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(3)
    for b in sorted({0, w.B - 1, *rng.integers(0, w.B, 2).tolist()}):
        _check_sequence(oracle_mod, w, inp, o, lse, b)


def test_decode_rejects_bad_device_data(oracle_mod):
    """A page index outside the cache or a length past the table is found by the kernel before
    any copy, reported as FA_ERR_INVALID_ARG, and leaves the context usable."""
    w = workloads.DecodeWorkload("decode_bad", 2, 2, 64, torch.bfloat16, 0, 0, extra_pages=2)
    inp = workloads.make_decode_inputs(w, seed=9, device="cuda", lens=[40, 20])
    s = torch.cuda.current_stream().cuda_stream
    assert fa.fa_get_device_status(s) == fa.FA_OK
    bad = dict(inp)
    bad["block_tables"] = inp["block_tables"].clone()
    bad["block_tables"][0, 1] = inp["k_cache"].shape[0]  # one past the last page
    fa.decode_paged(bad["q"], bad["k_cache"], bad["v_cache"], bad["block_tables"],
                    bad["seq_lens"], w.scale)
    assert fa.fa_get_device_status(s) == fa.FA_ERR_INVALID_ARG
    bad = dict(inp)
    bad["seq_lens"] = torch.tensor([40, 16 * inp["block_tables"].shape[1] + 1], dtype=torch.int32,
                                   device="cuda")
    fa.decode_paged(bad["q"], bad["k_cache"], bad["v_cache"], bad["block_tables"],
                    bad["seq_lens"], w.scale)
    assert fa.fa_get_device_status(s) == fa.FA_ERR_INVALID_ARG
    o, lse = _run(w, inp)  # the context still works
    for b in range(w.B):
        _check_sequence(oracle_mod, w, inp, o, lse, b)
