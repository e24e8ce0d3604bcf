"""Seeded synthetic inputs for the attention workloads (shared by tests and the benchmark).

This module holds no attention arithmetic: it only names the workload shapes and draws
i.i.d. N(0,1) tensors from a seeded torch CPU generator.  Draw order is q, k, v, dO, then
(for the row-scaled variant) one U(0.5, 4) factor per query row.  Values are drawn in fp32
and rounded to nearest-even into the workload's 16-bit dtype; the row factor multiplies the
fp32 draw of Q before that rounding, so every consumer sees the same 16-bit values.

The shapes stand in for the pages' workloads: the Llama-2-7B attention layer at sequence
2048 (32 heads of dimension 128), a batched training shape, a long sequence, a
short-sequence batch sweep and the single-head 128 x 64 case the data-flow page profiles
("FlashAttention data-flow optimisation: MI50 memory and bandwidth bottlenecks",
sections 2.1 and 3.1).  No dataset or model weights are involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    D: int
    causal: bool
    dtype: torch.dtype
    backward: bool = True
    row_scaled: bool = False
    scale_value: float | None = None  # None: the usual 1/sqrt(D)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D) if self.scale_value is None else float(self.scale_value)

    @property
    def plain_inputs(self) -> bool:
        """True for i.i.d. N(0,1) inputs at the usual 1/sqrt(D) scale: the setting the stated
        O error bounds are quoted for."""
        return not self.row_scaled and self.scale_value is None

    @property
    def dtype_name(self) -> str:
        return {torch.bfloat16: "bf16", torch.float16: "fp16"}[self.dtype]

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "L": self.L, "D": self.D,
                "causal": self.causal, "dtype": self.dtype_name, "row_scaled": self.row_scaled}


# The five workload families (the short-sequence sweep expands into four shapes).
WORKLOADS = {
    "single_head_L128_D64": Workload("single_head_L128_D64", 1, 1, 128, 64, False,
                                     torch.float16, backward=False),
    "llama2_7b_L2048": Workload("llama2_7b_L2048", 1, 32, 2048, 128, True, torch.bfloat16),
    "train_B8_L4096": Workload("train_B8_L4096", 8, 32, 4096, 128, True, torch.bfloat16),
    "train_B8_L4096_rowscaled": Workload("train_B8_L4096_rowscaled", 8, 32, 4096, 128, True,
                                         torch.bfloat16, row_scaled=True),
    "long_L16384_D64": Workload("long_L16384_D64", 1, 16, 16384, 64, True, torch.bfloat16),
    "short_L512_D64": Workload("short_L512_D64", 16, 32, 512, 64, False, torch.float16),
    "short_L512_D128": Workload("short_L512_D128", 16, 32, 512, 128, False, torch.float16),
    "short_L1024_D64": Workload("short_L1024_D64", 16, 32, 1024, 64, False, torch.float16),
    "short_L1024_D128": Workload("short_L1024_D128", 16, 32, 1024, 128, False, torch.float16),
}


def custom(B: int, H: int, L: int, D: int, causal: bool, dtype: torch.dtype,
           row_scaled: bool = False, scale: float | None = None) -> Workload:
    return Workload(f"custom_B{B}_H{H}_L{L}_D{D}", B, H, L, D, causal, dtype,
                    row_scaled=row_scaled, scale_value=scale)


def shrink(w: Workload, B: int | None = None, H: int | None = None,
           L: int | None = None) -> Workload:
    """Same workload family with fewer heads / shorter sequence (for quick checks)."""
    return replace(w, name=w.name + "_small", B=B or w.B, H=H or w.H, L=L or w.L)


def make_inputs(w: Workload, seed: int = 0, with_do: bool = True):
    """Returns dict of CPU tensors q, k, v (and do) of shape [B,H,L,D] in ``w.dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (w.B, w.H, w.L, w.D)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.row_scaled:
        f = torch.rand((w.B, w.H, w.L, 1), generator=g, dtype=torch.float32) * 3.5 + 0.5
        q = q * f
    out = {"q": q.to(w.dtype), "k": k.to(w.dtype), "v": v.to(w.dtype)}
    if with_do:
        out["do"] = do.to(w.dtype)
    return out


# ---------------------------------------------------------------------------------------
# Decode over a paged key/value cache ("FlashAttention principles and engineering practice",
# section 4.2: Llama-2-7B served with PagedAttention, block_size 16, up to 256 sequences in a
# continuous batch).  Synthetic stand-in: N(0,1) queries and cache, sequence lengths drawn
# uniformly, pages assigned in a shuffled order with spare pages left holding noise.
# ---------------------------------------------------------------------------------------
PAGE_TOKENS = 16


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    D: int
    dtype: torch.dtype
    min_len: int
    max_len: int
    extra_pages: int = 64

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def dtype_name(self) -> str:
        return {torch.bfloat16: "bf16", torch.float16: "fp16"}[self.dtype]

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "D": self.D,
                "page_tokens": PAGE_TOKENS, "seq_len": f"U[{self.min_len}, {self.max_len}]",
                "dtype": self.dtype_name}


DECODE_WORKLOADS = {
    "decode_llama2_7b_B256": DecodeWorkload("decode_llama2_7b_B256", 256, 32, 128,
                                            torch.bfloat16, 1, 4096),
}


def make_decode_inputs(w: DecodeWorkload, seed: int = 0, device="cpu", lens=None):
    """Returns dict q [B,H,D], k_cache, v_cache [num_pages,H,16,D] (w.dtype), block_tables
    [B,max_pages] int32, seq_lens [B] int32, all on `device`.  Draw order: lengths (unless
    given), page order, q, k_cache, v_cache.  Table entries past a sequence's pages are 0."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    if lens is None:
        lens = torch.randint(w.min_len, w.max_len + 1, (w.B,), generator=g)
    lens = torch.as_tensor(lens, dtype=torch.int64)
    pages = (lens + PAGE_TOKENS - 1) // PAGE_TOKENS
    max_pages = max(1, int(pages.max()) if len(pages) else 1)
    num_pages = int(pages.sum()) + w.extra_pages
    order = torch.randperm(num_pages, generator=g)
    table = torch.zeros((w.B, max_pages), dtype=torch.int32)
    nxt = 0
    for b in range(w.B):
        n = int(pages[b])
        table[b, :n] = order[nxt:nxt + n].to(torch.int32)
        nxt += n
    gd = torch.Generator(device=device)
    gd.manual_seed(int(seed) + 1)
    q = torch.randn((w.B, w.H, w.D), generator=gd, device=device, dtype=torch.float32)
    kc = torch.randn((num_pages, w.H, PAGE_TOKENS, w.D), generator=gd, device=device,
                     dtype=torch.float32)
    vc = torch.randn((num_pages, w.H, PAGE_TOKENS, w.D), generator=gd, device=device,
                     dtype=torch.float32)
    return {"q": q.to(w.dtype), "k_cache": kc.to(w.dtype), "v_cache": vc.to(w.dtype),
            "block_tables": table.to(device), "seq_lens": lens.to(torch.int32).to(device)}
