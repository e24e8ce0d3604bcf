"""bench.py's DRAM-traffic record: keyed on the kernel source and the files shared by every
kernel, and ignored (reported as null) once any of them has changed since the capture."""
import importlib.util
import json
import os
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHARED = ("fa_internal.h", "fa_ptx.cuh", "fa_api.cu")


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture()
def bench_copy(tmp_path):
    """bench module whose ROOT is a scratch copy holding the kernel sources and a record."""
    bench = load_bench()
    csrc = tmp_path / "tiled_attention_08_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src_dir = os.path.join(ROOT, "tiled_attention_08_gb300", "csrc")
    headers = {n for n in os.listdir(src_dir) if n.endswith((".h", ".cuh"))}
    for name in set(bench.KERNEL_SOURCES.values()) | set(SHARED) | headers:
        shutil.copy(os.path.join(src_dir, name), csrc / name)
    (tmp_path / "profiles").mkdir()
    bench.ROOT = str(tmp_path)
    return bench, tmp_path


def write_record(tmp_path, kernel, sha, nbytes=123456789):
    rec = {kernel: {"train_B8_L4096": {"dram_bytes_per_launch": nbytes, "source_sha": sha,
                                       "note": "test"}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))


def test_sha_is_stable_and_distinct_per_kernel(bench_copy):
    bench, _ = bench_copy
    shas = {k: bench.kernel_sha(k) for k in bench.KERNEL_SOURCES}
    assert all(len(v) == 16 and int(v, 16) >= 0 for v in shas.values())
    assert len(set(shas.values())) == len(shas)
    assert shas == {k: bench.kernel_sha(k) for k in bench.KERNEL_SOURCES}


@pytest.mark.parametrize("edited", ["kernel"] + list(SHARED))
def test_sha_covers_kernel_and_shared_files(bench_copy, edited):
    bench, tmp = bench_copy
    kernel = "bwd_dkdv"
    before = bench.kernel_sha(kernel)
    name = bench.KERNEL_SOURCES[kernel] if edited == "kernel" else edited
    path = tmp / "tiled_attention_08_gb300" / "csrc" / name
    path.write_text(path.read_text() + "\n// edited\n")
    assert bench.kernel_sha(kernel) != before


def test_sha_covers_headers_the_kernel_includes(bench_copy):
    bench, tmp = bench_copy
    # The three attention passes include the persistent-schedule header; the preprocess
    # kernel does not.
    before = {k: bench.kernel_sha(k) for k in bench.KERNEL_SOURCES}
    path = tmp / "tiled_attention_08_gb300" / "csrc" / "fa_sched.h"
    path.write_text(path.read_text() + "\n// edited\n")
    after = {k: bench.kernel_sha(k) for k in bench.KERNEL_SOURCES}
    for k in ("fa_fwd", "bwd_dkdv", "bwd_dq"):
        assert after[k] != before[k], k
    assert after["bwd_pre"] == before["bwd_pre"]


def test_record_used_only_while_sources_match(bench_copy):
    bench, tmp = bench_copy
    kernel = "bwd_dkdv"
    write_record(tmp, kernel, bench.kernel_sha(kernel))
    value, note = bench.profiled_traffic(kernel, "train_B8_L4096")
    assert value == 123456789.0 and note == "test"
    src = tmp / "tiled_attention_08_gb300" / "csrc" / "fa_ptx.cuh"
    src.write_text(src.read_text() + "\n")
    value, note = bench.profiled_traffic(kernel, "train_B8_L4096")
    assert value is None and "changed" in note


def test_missing_record_or_workload_gives_null(bench_copy):
    bench, tmp = bench_copy
    assert bench.profiled_traffic("bwd_dkdv", "train_B8_L4096")[0] is None  # no file
    write_record(tmp, "fa_fwd", bench.kernel_sha("fa_fwd"))
    assert bench.profiled_traffic("bwd_dkdv", "train_B8_L4096")[0] is None  # other kernel
    assert bench.profiled_traffic("fa_fwd", "long_L16384_D64")[0] is None   # other workload


def test_committed_record_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    bench = load_bench()
    for kernel, per_wl in rec.items():
        assert kernel in bench.KERNEL_SOURCES
        for wl, r in per_wl.items():
            assert r["dram_bytes_per_launch"] > 0
            assert len(r["source_sha"]) == 16
            assert r.get("note")
