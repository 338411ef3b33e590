"""Host logic of bench.py (no GPU): the algorithmic work model against the
figures the configurations are planned with, the launch count against the
library's host loop, and the guard that drops stale DRAM traffic."""
import os
import shutil

import numpy as np
import pytest

import bench
from long_context_sparse_gb300 import synth


def test_work_model_at_131072_tokens():
    wl = synth.WORKLOADS["glm_chunked_s128k"]
    wm = bench.work_model(wl)
    # indexer: sum_t n_full(t) * H_I * 2 * D_I = 17.6 TFLOP
    assert wm["indexer_flops"] == pytest.approx(17.59e12, rel=1e-3)
    # 2048 keys for every query past the first 2047 (then fewer)
    assert wm["keys"] == pytest.approx(131072 * 2048, rel=0.02)
    # gathered K/V rows: 508 GiB (the 524 GiB forward figure adds streaming
    # Q and O, 8 GiB each)
    assert wm["fwd_gather_bytes"] / 2**30 == pytest.approx(508, rel=0.01)
    assert wm["bwd_scatter_bytes"] / 2**30 == pytest.approx(1016, rel=0.02)
    assert wm["fwd_flops"] == pytest.approx(34.9e12, rel=0.01)
    kv = bench.work_model(wl, kv=True)
    assert kv["fwd_gather_bytes"] == pytest.approx(wm["fwd_gather_bytes"] / 2)
    assert kv["bwd_scatter_bytes"] == pytest.approx(wm["bwd_scatter_bytes"] / 2)


def test_keys_of_row_matches_the_model():
    for name in ("glm_s16k", "padded2051_s64k"):
        wl = synth.scaled(synth.WORKLOADS[name], 3001)
        total = sum(bench.keys_of_row(wl, t) for t in range(wl.S))
        assert total == bench.work_model(wl)["keys"]
    wl = synth.scaled(synth.WORKLOADS["padded2051_s64k"], 100)
    assert bench.keys_of_row(wl, 0) == 1            # only the query itself
    assert bench.keys_of_row(wl, 10) == 11          # full budget: every token


def test_launch_count_mirrors_the_chunk_loop():
    wl = synth.WORKLOADS["glm_chunked_s128k"]
    # pool + 504 indexer chunks (the first 8 chunks hold <= K_p pools per
    # row) + 512 top-k chunks + forward + 6 backward launches
    assert bench.launches_per_step(wl) == 1 + 504 + 512 + 1 + 6
    assert bench.launches_per_step(wl, kv=True) == 1 + 504 + 512 + 1 + 4
    assert bench.launches_per_step(wl, streaming=True) == 1 + 1 + 1 + 6
    tiny = synth.WORKLOADS["tiny_fwd_s1k"]           # forward only, K_p = 64:
    # the first 256-query chunk holds <= 64 pools per row (no indexer launch)
    assert bench.launches_per_step(tiny) == 1 + 3 + 4 + 1


def test_traffic_guard_drops_stale_figures(tmp_path, monkeypatch):
    """A stored DRAM-traffic figure is reported only for the workload, the
    default variant and the kernel sources it was captured with."""
    wl = synth.WORKLOADS["glm_chunked_s128k"]
    csrc = os.path.join(bench.ROOT, "long_context_sparse_gb300", "csrc")
    fake = tmp_path / "long_context_sparse_gb300" / "csrc"
    fake.mkdir(parents=True)
    for f in ("attn_bwd_tc.cu", "attn_fwd_tc.cu", "attn_common.cuh", "dsa_common.cuh"):
        shutil.copy(os.path.join(csrc, f), fake / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the table as if captured on these sources
    table = {k: dict(e, sha256_16=bench.sources_hash(e["sources"]))
             for k, e in bench.MEASURED_TRAFFIC.items()}
    monkeypatch.setattr(bench, "MEASURED_TRAFFIC", table)
    for kernel, e in table.items():
        assert bench.measured_traffic(kernel, wl) == e["bytes"]    # sources as captured
        assert bench.measured_traffic(kernel, wl, "kv") is None    # another variant
        assert bench.measured_traffic(kernel, synth.WORKLOADS["glm_s16k"]) is None
    # a changed kernel source invalidates the figure
    with open(fake / "attn_bwd_tc.cu", "a") as fh:
        fh.write("\n// changed\n")
    assert bench.measured_traffic("attn_bwd_tc", wl) is None
    assert bench.measured_traffic("attn_fwd_tc", wl) is not None
