"""The FLOP/byte model that converts times into TFLOP/s and GB/s, pinned to the pages."""
import os

import pytest

from tiled_attention_08_gb300 import perfmodel as pm

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_figures.txt")


def figures():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, value, unit, _src = (x.strip() for x in line.split("|", 3))
        out[key] = (float(value), unit)
    return out


def _matches_printed(nbytes, printed, unit):
    """The page prints KB both as 1000 and as 1024 bytes, rounded to its last digit."""
    if unit == "B":
        return nbytes == printed
    digits = 0 if float(printed).is_integer() else 1
    tol = 0.5 * 10 ** (-digits)
    return any(abs(nbytes / base - printed) <= tol for base in (1000.0, 1024.0))


def test_naive_forward_traffic_matches_page():
    f = figures()
    n = pm.naive_forward_bytes(128, 64, elem=4)
    assert _matches_printed(n["qkv"], *f["naive_qkv_bytes"])
    assert _matches_printed(n["s"], *f["naive_s_bytes"])
    assert _matches_printed(n["p"], *f["naive_p_bytes"])
    assert _matches_printed(n["out"], *f["naive_out_bytes"])
    # "about 260 KB" in total
    assert abs(n["total"] / 1000.0 - f["naive_total_bytes"][0]) < 5.0


def test_fused_forward_drops_the_two_LxL_intermediates():
    n = pm.naive_forward_bytes(128, 64, elem=4)
    fused = pm.bytes_fwd(1, 1, 128, 64, elem=4)
    # fused = Q, K, V in + O out + one fp32 LSE per row; no S, no P
    assert fused == n["qkv"] + n["out"] + 128 * 4
    assert fused < n["total"] - n["s"] - n["p"] + 1024


def test_row_stats_size_matches_page():
    f = figures()
    assert 128 * 4 == f["row_stats_bytes"][0]


def test_flop_model_matches_page_formula():
    f = figures()
    L, D = 2048, 64
    assert pm.flops_fwd(1, 1, L, D, False) == f["qkt_flops_L2048_D64"][0] + f["pv_flops_L2048_D64"][0]
    assert pm.flops_fwd(1, 1, L, D, True) == 0.5 * pm.flops_fwd(1, 1, L, D, False)
    assert pm.flops_bwd(2, 3, L, D, True) == 2.5 * pm.flops_fwd(2, 3, L, D, True)


def test_kernel_flops_add_up_to_the_pass_totals():
    args = (8, 32, 4096, 128, True)
    fwd = pm.flops_kernel("fa_fwd", *args)
    bwd = sum(pm.flops_kernel(k, *args) for k in ("bwd_pre", "bwd_dkdv", "bwd_dq"))
    assert fwd == pm.flops_fwd(*args)
    assert bwd == pytest.approx(pm.flops_bwd(*args))


def test_workload_sizes():
    # Llama-2-7B layer: 32 heads, L=2048, D=128, causal -> 34.4 GFLOP forward
    assert pm.flops_fwd(1, 32, 2048, 128, True) == pytest.approx(34.36e9, rel=1e-3)
    assert pm.bytes_fwd(1, 32, 2048, 128) == 32 * (8 * 2048 * 128 + 4 * 2048)
