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


def test_default_workload_is_the_lm_head_projection():
    assert bench.DEFAULT_WORKLOAD == "lm-head-m1-k4096-n151936"
    assert bench.DEFAULT_WORKLOAD in WORKLOADS


def test_graph_steps_give_about_ten_replays_of_whole_rotations():
    # the full test run: 20 steps of lm-head (2 weight copies, one launch a
    # step) run as one graph; long runs as about ten replays of whole rotations
    assert bench.graph_steps(20, 2) == 20
    assert bench.graph_steps(200, 2) == 200
    G = bench.graph_steps(2000, 2)
    assert G == 200 and divmod(2000, G) == (10, 0)
    assert bench.graph_steps(1000, 28) == 112          # four rotations of 28 steps
    assert bench.graph_steps(3, 1) == 3
    for steps in (1, 7, 20, 99, 201, 2000):
        for rot in (1, 2, 3, 28):
            g = bench.graph_steps(steps, rot)
            assert 1 <= g <= steps and (g % rot == 0 or g == steps)


def test_config_records_cover_the_five_configurations():
    cfgs = {c for c, _, _ in bench.CONFIG_RECORDS}
    assert cfgs == {0, 1, 2, 3, 4}
    names = [(n, o) for _, n, o in bench.CONFIG_RECORDS]
    assert ("attn-proj-m1-k4096-n4096", "f16") in names and ("attn-proj-m1-k4096-n4096", "bf16") in names
    assert {n for n, _ in names if n.startswith("small-batch")} == {
        "small-batch-m2-k8192-n8192", "small-batch-m4-k8192-n8192", "small-batch-m8-k8192-n8192"}
    for _, n, o in bench.CONFIG_RECORDS:
        assert o in WORKLOADS[n].out_dtypes


def test_pages_context_quotes_the_a100_figures():
    c = bench.PAGES_CONTEXT
    assert c["gate_up_gemv"]["us_per_call"] == 26.69 and c["gate_up_gemv"]["dram_tb_per_s"] == 2.267
    assert c["decode_64_tokens_bf16"]["cast_half_launches"] == [3024, 2398]


def test_cpulist_and_gpu_numa_lookup():
    """The e2e arm's host-buffer placement: sysfs cpulists parse, and a
    device without a UUID (or a host without nvidia-smi) gives no placement."""
    import types
    import bench
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("") == set()
    assert bench.gpu_local_cpus(types.SimpleNamespace(uuid="")) is None
