"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a plugin whose host framework owns all device memory, a running loop that must
not call cudaMalloc) cannot hand fa_bwd a workspace; fa_bwd_noalloc takes its scratch from a
fixed 16 MiB array inside the library instead.  This file is collected last on purpose: a
failure here must not stop a fail-fast run before every other test has run.
"""
import pytest
import torch

import tiled_attention_08_gb300 as fa
import workloads


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_attention_08_gb300 import build
    build.build()
    fa.load_library()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream

    # Sizes beyond the fixed scratch are refused before anything is enqueued:
    # 8 bytes x 4096 heads x 1024 rows = 32 MiB > 16 MiB.
    A = 0x100000
    big = fa.fa_bwd_noalloc(A, A + (1 << 30), A + (2 << 30), A + (3 << 30), A + (4 << 30),
                            A + (5 << 30), A + (6 << 30), A + (7 << 30), A + (8 << 30),
                            64, 64, 1024, 64, 0.125, 1, fa.FA_BF16, stream)
    assert big == fa.FA_ERR_UNSUPPORTED
    # fa_bwd's own argument checks come first: null pointers are an argument error at any size.
    assert fa.fa_bwd_noalloc(0, 0, 0, 0, 0, 0, 0, 0, 0, 64, 64, 1024, 64, 0.125, 1, fa.FA_BF16,
                             stream) == fa.FA_ERR_INVALID_ARG

    # The backward is deterministic (no atomics), so both entry points give the same bits.  The
    # third shape has more query tiles (2 x 40 x 3) than SMs: its dQ pass runs persistent CTAs,
    # which read their per-row vectors from the scratch array over several rounds.
    for (B, H, L, D, causal, dtype) in ((2, 4, 700, 128, True, torch.bfloat16),
                                        (1, 3, 300, 64, False, torch.float16),
                                        (2, 40, 384, 128, False, torch.bfloat16)):
        w = workloads.custom(B, H, L, D, causal, dtype)
        inp = workloads.make_inputs(w, seed=21)
        q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
        o, lse = fa.forward(q, k, v, causal, w.scale)
        ref = fa.backward(q, k, v, o, lse, do, causal, w.scale)  # workspace entry point
        dt = fa.FA_BF16 if dtype == torch.bfloat16 else fa.FA_FP16
        for _ in range(2):  # two calls in a row share (and reuse) the scratch array
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            st = fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, H, L, D, w.scale, int(causal), dt, stream)
            assert st == fa.FA_OK, fa.fa_status_string(st)
            torch.cuda.synchronize(dev)
            assert fa.fa_get_device_status(stream) == fa.FA_OK
            for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
                assert torch.equal(got, want), (B, H, L, D, name)
