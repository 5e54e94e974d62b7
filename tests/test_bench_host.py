"""Host-side logic of bench.py (no GPU): percentiles, the FMA bound, the
recorded-traffic hash check and the oracle sample's accounting."""
import os
import types

import numpy as np

import bench
from int4_block_quantized_mnb_gb300.synth import WORKLOADS, make_inputs


def test_percentiles_are_nearest_rank():
    v = sorted([5.0, 1.0, 3.0, 2.0, 4.0])
    assert [bench.pct(v, q) for q in (0, 10, 50, 90, 100)] == [1.0, 1.0, 3.0, 5.0, 5.0]


def test_fma_bound_counts_m_n_k():
    w = WORKLOADS["small-batch-m8-k8192-n8192"]
    props = types.SimpleNamespace(multi_processor_count=152)
    b = bench.fma_bound(w, props, {"sm_max_mhz": 2000.0})
    assert b["fmas_per_launch"] == 8 * 8192 * 8192
    assert abs(b["tfma_per_s"] - 152 * 128 * 2e9 / 1e12) < 1e-9
    assert abs(b["us"] - 8 * 8192 * 8192 / (152 * 128 * 2e9) * 1e6) < 1e-9


def test_recorded_traffic_needs_the_current_kernel_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "gemv_dram_traffic.txt").write_text(
        "# comment\nkernel_source_sha256 = deadbeef\nattn-proj-m1-k4096-n4096 = 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "deadbeef")
    assert bench.recorded_traffic("attn-proj-m1-k4096-n4096") == 123
    assert bench.recorded_traffic("lm-head-m1-k4096-n151936") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "other")
    assert bench.recorded_traffic("attn-proj-m1-k4096-n4096") is None


def test_committed_traffic_record_is_parseable():
    path = os.path.join(bench.ROOT, "profiles", "gemv_dram_traffic.txt")
    lines = [l for l in open(path) if "=" in l and not l.lstrip().startswith("#")]
    keys = {l.split("=", 1)[0].strip() for l in lines}
    assert "kernel_source_sha256" in keys and "attn-proj-m1-k4096-n4096" in keys


def test_oracle_sample_accounts_whole_passes():
    w = WORKLOADS["tiny-m1-k256-n256"]
    inp = make_inputs(w.M, w.N, w.K, seed=0)
    gbs, desc, dt = bench.oracle_sample(w, inp, 0.2, 2)
    assert gbs > 0 and dt > 0 and "passes over all 256 output columns" in desc


def test_prefill_workload_names_and_rows():
    base = WORKLOADS["attn-proj-m1-k4096-n4096"]
    w = bench.FormatWorkload(base, 32, False, 512)
    assert (w.M, w.N, w.K) == (512, 4096, 4096) and w.name == "prefill-m512-k4096-n4096"
    w = bench.FormatWorkload(base, 64, True, 0)
    assert w.M == 1 and w.name == "attn-proj-m1-k4096-n4096-b64-sym"


def test_tensor_roofline_counts_two_m_n_k(tmp_path, monkeypatch):
    w = bench.FormatWorkload(WORKLOADS["attn-proj-m1-k4096-n4096"], 32, False, 2048)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))                 # no peaks file here
    r = bench.tensor_roofline(w, 100e-6, 150.0, 6000.0)
    flops = 2.0 * 2048 * 4096 * 4096
    assert r["bound"] == "tensor" and r["flops_per_launch"] == flops
    assert abs(r["achieved"] - flops / 100e-6 / 1e12) < 1e-9
    assert r["peak"] == bench.FALLBACK_BF16_TFLOPS and r["peak_kind"].startswith("fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"bf16_tflops": 2000.0}')
    assert bench.measured_tensor_peak() == (2000.0, "measured")


def test_prefill_options_parse(monkeypatch):
    monkeypatch.setattr("sys.argv", ["bench.py", "--m", "512", "--prefill-mma-sync", "--block", "64"])
    a = bench.parse()
    assert a.m == 512 and a.prefill_mma_sync and a.block == 64 and not a.tensor_cores
