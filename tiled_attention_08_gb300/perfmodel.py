"""FLOP and byte model used to turn measured times into TFLOP/s and GB/s.

FLOPs ("AIInfra notes 01: from TFLOPS to FlashAttention", section 3.1, first gate): per head the
forward's contractions are QK^T (2*L*D*L) and PV (2*L*D*L), 4*L^2*D in all; the softmax's
exp/sum/divide work is not counted.  The causal mask halves it.  The backward is counted as
2.5 times the forward (five L x L x D contractions: the recomputed S, dP, dV, dK, dQ).

Algorithmic bytes: each 16-bit tensor element crosses HBM once (Q, K, V, O, dO read; O, dQ, dK,
dV written) plus the fp32 per-row vectors.  The data-flow page ("FlashAttention data-flow
optimisation: MI50 memory and bandwidth bottlenecks", section 2.1) counts the unfused forward
of one 128 x 64 fp32 head the same way (Q, K, V read, output written, plus the two L x L
intermediates S and P the fused kernel never stores); ``naive_forward_bytes`` restates that
count so the model can be checked against the page's figures.
"""
from __future__ import annotations

TILE = 128


def _heads(B: int, H: int) -> int:
    return B * H


def flops_fwd(B: int, H: int, L: int, D: int, causal: bool) -> float:
    f = 4.0 * _heads(B, H) * L * L * D
    return f * 0.5 if causal else f


def flops_bwd(B: int, H: int, L: int, D: int, causal: bool) -> float:
    return 2.5 * flops_fwd(B, H, L, D, causal)


def flops_kernel(kernel: str, B: int, H: int, L: int, D: int, causal: bool) -> float:
    """Algorithmic FLOPs one launch of each library kernel carries.

    fa_fwd: the forward (S and PV).  bwd_dkdv: 4 of the backward's 5 contractions (S, dP, dV,
    dK).  bwd_dq: the dQ contraction only; its recomputation of S and dP is repeated work and
    is not counted.  bwd_pre: no contraction.
    """
    f = flops_fwd(B, H, L, D, causal)
    return {"fa_fwd": f, "bwd_dkdv": 2.0 * f, "bwd_dq": 0.5 * f, "bwd_pre": 0.0}[kernel]


def _lpad(L: int) -> int:
    return ((L + TILE - 1) // TILE) * TILE


def bytes_kernel(kernel: str, B: int, H: int, L: int, D: int, elem: int = 2) -> float:
    """Algorithmic HBM bytes of one launch (each operand element read or written once)."""
    n = _heads(B, H)
    t = L * D * elem  # one [L, D] tensor of one head
    if kernel == "fa_fwd":
        per = 4 * t + 4 * L                     # Q, K, V in; O out; LSE out
    elif kernel == "bwd_pre":
        per = 2 * t + 4 * L + 8 * _lpad(L)      # O, dO, LSE in; two padded fp32 vectors out
    elif kernel == "bwd_dkdv":
        per = 6 * t + 8 * _lpad(L)              # K, V, Q, dO in; dK, dV out; vectors in
    elif kernel == "bwd_dq":
        per = 5 * t + 8 * _lpad(L)              # Q, dO, K, V in; dQ out; vectors in
    else:
        raise KeyError(kernel)
    return float(n * per)


def bytes_fwd(B: int, H: int, L: int, D: int, elem: int = 2) -> float:
    """Minimum HBM bytes of the forward: 8*L*D + 4*L per head for 16-bit tensors."""
    return bytes_kernel("fa_fwd", B, H, L, D, elem)


def bytes_bwd(B: int, H: int, L: int, D: int, elem: int = 2) -> float:
    """Minimum HBM bytes of the backward: Q, K, V, O, dO read and dQ, dK, dV written (eight
    [L, D] tensors, 16*L*D bytes for 16-bit), LSE read, Delta written and read back (12*L)."""
    return float(_heads(B, H) * (8 * L * D * elem + 12 * L))


def naive_forward_bytes(L: int, D: int, elem: int = 4) -> dict:
    """HBM bytes of the unfused forward of one head that stores S and P: the data-flow page's
    own accounting (section 2.1)."""
    qkv = 3 * L * D * elem
    s = L * L * elem
    p = L * L * elem
    out = L * D * elem
    return {"qkv": qkv, "s": s, "p": p, "out": out, "total": qkv + s + p + out}
