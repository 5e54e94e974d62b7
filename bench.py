#!/usr/bin/env python3
"""Benchmark of the int4 block-quantized MatMulNBits decode GEMV on GB300.

One step = one pass of the hot path over one input batch: the GEMV of the
chosen workload once per output dtype the workload names.  The default
workload is the M=1 lm_head-sized projection (K=4096, N=151936, fp16 output),
the largest single-GPU decode configuration; the 4096x4096 attention
projection runs an fp16-output and a bf16-output launch per step.

  value      algorithmic HBM bytes of the step's GEMV calls / device time per
             step, with inputs resident in HBM.  Weight copies rotate over more
             than 4x the L2 size so every launch streams its weights from HBM.
             The K timed steps run as replays of a CUDA graph of captured
             library launches (the kernel launches are the library's own).
  e2e        the same metric through the public API with host buffers: each step
             copies x, qweight, scales and zero-points from pinned host memory,
             runs the GEMV(s) and copies y back.
  roofline   the GEMV kernel's achieved bandwidth against the measured HBM peak.
  cpu_baseline  the CPU oracle timed on a bounded sample on this host's cores.
  configs    one sub-record per decode configuration (tiny 256x256, attention
             projection in fp16 and bf16, fused gate_up, lm_head, small batch
             M = 2, 4, 8): per-call time spread, GB/s, roofline fractions, the
             kernel's registers and theoretical occupancy, committed DRAM
             traffic.

``--impl reference`` times the CPU oracle alone (the reference arm).  With
torchrun and N > 1 every rank runs an independent replica (the path has no
exchange step) and rank 0 prints the line; value sums all ranks' bytes over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import shutil
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode GEMV µs/call and achieved HBM GB/s (% of GB300 peak) at M=1"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "lm-head-m1-k4096-n151936"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["mnb", "reference"], default="mnb")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--split-k", type=int, default=0,
                    help="0 = the library's choice (as a user calling with split_k=0 gets)")
    ap.add_argument("--tensor-cores", action="store_true",
                    help="permit the decode step kernel's tensor-core math (MNB_FLAG_TENSOR_CORES)")
    ap.add_argument("--prefill-mma-sync", action="store_true",
                    help="M > 8: the mma.sync form of the prefill GEMM instead of its tcgen05 form "
                         "(MNB_FLAG_PREFILL_MMA_SYNC)")
    ap.add_argument("--ab-staged", action="store_true",
                    help="time a synthetic decode step of bf16 GEMVs: fp16 GEMV + separate "
                         "narrowing launch (staged route) against the direct bf16 store")
    ap.add_argument("--block", type=int, default=32, choices=[16, 32, 64, 128],
                    help="quantization block size of the synthetic weights")
    ap.add_argument("--symmetric", action="store_true",
                    help="weights without zero-points (every zero-point 8)")
    ap.add_argument("--m", type=int, default=0,
                    help="activation rows instead of the workload's (M > 8: the prefill GEMM)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration sub-records (configs 0-4)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU seconds for the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


DATASHEET_HBM_GBS = 8000.0      # GB300 HBM3e, ~8 TB/s (the datasheet figure used here)


def pct(sorted_vals, q):
    """Nearest-rank percentile of an ascending list."""
    i = min(len(sorted_vals) - 1, max(0, int(round(q / 100.0 * (len(sorted_vals) - 1)))))
    return sorted_vals[i]


def fma_bound(w, props, clk):
    """The non-tensor FP32 FMA bound of an M > 1 call: M*N*K FMAs at SMs x 128
    FP32 lanes x the maximum SM clock seen (derived, not measured)."""
    mhz = (clk or {}).get("sm_max_mhz") or 2070.0
    rate = props.multi_processor_count * 128 * mhz * 1e6          # FMA/s
    fmas = w.M * w.N * w.K
    return {"fmas_per_launch": fmas, "tfma_per_s": rate / 1e12, "us": fmas / rate * 1e6,
            "rate_source": f"{props.multi_processor_count} SMs x 128 FP32 lanes x {mhz:.0f} MHz"}


FALLBACK_BF16_TFLOPS = 1900.0


def measured_tensor_peak():
    """Dense bf16 tensor TFLOP/s (burst) from MEASURED_PEAKS.json; fp16 runs at
    the same nominal rate."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def tensor_roofline(w, per_launch_s, gbs, hbm_peak):
    """The prefill GEMM (M > 8) against the dense tensor peak: 2 M N K flops per
    launch over its average duration; the HBM fraction beside it."""
    flops = 2.0 * w.M * w.N * w.K
    tf = flops / per_launch_s / 1e12
    peak, kind = measured_tensor_peak()
    return {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
            "peak_kind": kind + " bf16 (fp16 operands run at the same nominal rate)",
            "traffic": None, "flops_per_launch": flops,
            "hbm_achieved_gbs": gbs, "hbm_frac": gbs / hbm_peak}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = ("int4_block_quantized_mnb_gb300/csrc/mnb_gemv.cu",
                  "int4_block_quantized_mnb_gb300/csrc/mnb_dequant.cuh",
                  "int4_block_quantized_mnb_gb300/csrc/mnb_narrow.cuh",
                  "int4_block_quantized_mnb_gb300/csrc/mnb_general.cu",
                  "int4_block_quantized_mnb_gb300/csrc/mnb_prefill.cu",
                  "int4_block_quantized_mnb_gb300/csrc/mnb_prefill_tc.cu",
                  "int4_block_quantized_mnb_gb300/csrc/mnb_launch.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "gemv_dram_traffic.txt")
    try:
        with open(path) as f:
            entries = dict(line.split("=", 1) for line in f
                           if "=" in line and not line.lstrip().startswith("#"))
    except OSError:
        return None
    entries = {k.strip(): v.strip() for k, v in entries.items()}
    if entries.get("kernel_source_sha256") != kernel_source_hash():
        return None
    v = entries.get(workload)
    return int(v) if v else None


def parse_cpulist(text):
    """The CPU set of a sysfs cpulist ("0-3,8,10-11")."""
    cpus = set()
    for part in text.strip().split(","):
        if part:
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def gpu_local_cpus(props):
    """The host CPUs of the NUMA node the GPU is attached to (sysfs, by the
    PCI bus id nvidia-smi reports for the device's UUID), or None.  Pinned
    host buffers allocated from those CPUs land in that node's memory, next
    to the GPU's link."""
    exe = shutil.which("nvidia-smi")
    uuid = str(getattr(props, "uuid", "") or "")
    if exe is None or not uuid:
        return None
    if not uuid.startswith("GPU-"):
        uuid = "GPU-" + uuid
    try:
        bus = subprocess.run([exe, "--query-gpu=pci.bus_id", "--format=csv,noheader", "-i", uuid],
                             capture_output=True, text=True, timeout=20).stdout.strip()
        dom, rest = bus.split(":", 1)
        dev = f"{int(dom, 16):04x}:{rest}".lower()
        node = int(open(f"/sys/bus/pci/devices/{dev}/numa_node").read().strip())
        if node < 0:
            return None
        cpus = parse_cpulist(open(f"/sys/devices/system/node/node{node}/cpulist").read())
        return (node, cpus) if cpus else None
    except (OSError, ValueError, subprocess.SubprocessError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.reader = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if exe is None:
            return
        self.proc = subprocess.Popen(
            [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
             "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- CPU oracle --

def cpu_model():
    """Host CPU description from /proc/cpuinfo (model name, or the Arm part)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.machine()
    fields = {}
    for line in info:
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    parts = [f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part") if k in fields]
    return f"{platform.machine()} ({', '.join(parts)})" if parts else platform.machine()


class FormatWorkload:
    """A workload's shape with another weight format: block size and whether
    zero-points are stored (the symmetric format moves none)."""

    def __init__(self, base, block, symmetric, M=0):
        self.M, self.N, self.K, self.out_dtypes = base.M, base.N, base.K, base.out_dtypes
        self.block, self.symmetric = block, symmetric
        name = base.name
        if M:
            self.M = M
            name = f"{'prefill' if M > 8 else 'batch'}-m{M}-k{self.K}-n{self.N}"
        self.name = name + (f"-b{block}" if block != 32 else "") + ("-sym" if symmetric else "")

    def algorithmic_bytes(self) -> int:
        from int4_block_quantized_mnb_gb300.synth import bytes_per_call
        zp = self.N * ((self.K // self.block + 1) // 2) if self.symmetric else 0
        return bytes_per_call(self.M, self.N, self.K, self.block) - zp


def w_block(w):
    return getattr(w, "block", 32)


def w_zp(w, inp):
    return None if getattr(w, "symmetric", False) else inp.zp


def oracle_sample(w, inp, seconds, threads):
    """Times the CPU oracle on about `seconds` of work: a sample of output
    columns of the workload.  Returns (GB/s, description, threads used)."""
    from oracle import Oracle
    o = Oracle()
    n_calls = len(w.out_dtypes)      # one oracle pass yields every output dtype
    rng = np.random.default_rng(0)
    probe = rng.choice(w.N, size=min(w.N, max(threads, 16)), replace=False).astype(np.int64)
    t0 = time.perf_counter()
    o.gemv(inp.x, inp.qweight, inp.scales, w_zp(w, inp), w.M, w.N, w.K, block=w_block(w), cols=probe, threads=threads)
    rate = probe.size / max(time.perf_counter() - t0, 1e-6)          # columns per second
    ncols = int(max(threads, min(w.N, rate * seconds)))
    cols = rng.choice(w.N, size=ncols, replace=False).astype(np.int64)
    # whole passes over the sample until about `seconds` have elapsed
    passes = 0
    t0 = time.perf_counter()
    while True:
        o.gemv(inp.x, inp.qweight, inp.scales, w_zp(w, inp), w.M, w.N, w.K, block=w_block(w), cols=cols, threads=threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= 0.9 * seconds:
            break
    gbs = w.algorithmic_bytes() * n_calls * passes * (ncols / w.N) / dt / 1e9
    what = (f"{passes} passes over all {w.N} output columns" if passes > 1 else
            f"{ncols} of {w.N} output columns")
    desc = (f"{what} (all {w.M} rows, full K={w.K}), each pass producing the fp16 and bf16 "
            f"results, {dt:.1f} s on {threads} threads")
    return gbs, desc, dt


def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from int4_block_quantized_mnb_gb300.synth import make_inputs
    from oracle import Oracle
    inp = make_inputs(w.M, w.N, w.K, seed=0, block=w_block(w))
    o = Oracle()
    threads = os.cpu_count() or 1
    n_calls = len(w.out_dtypes)
    rng = np.random.default_rng(0)
    # calibrate: columns per second on all host threads
    probe = rng.choice(w.N, size=min(w.N, max(threads, 16)), replace=False).astype(np.int64)
    t0 = time.perf_counter()
    o.gemv(inp.x, inp.qweight, inp.scales, w_zp(w, inp), w.M, w.N, w.K, block=w_block(w), cols=probe, threads=threads)
    rate = probe.size / max(time.perf_counter() - t0, 1e-6)
    budget = 120.0
    per_step = int(max(1, min(w.N, rate * budget / max(1, args.steps + args.warmup))))
    cols = [rng.choice(w.N, size=per_step, replace=False).astype(np.int64)
            for _ in range(min(args.steps + args.warmup, 64))]
    for i in range(args.warmup):
        o.gemv(inp.x, inp.qweight, inp.scales, w_zp(w, inp), w.M, w.N, w.K, block=w_block(w), cols=cols[i % len(cols)],
               threads=threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        o.gemv(inp.x, inp.qweight, inp.scales, w_zp(w, inp), w.M, w.N, w.K, block=w_block(w), cols=cols[i % len(cols)],
               threads=threads)
    dt = time.perf_counter() - t0
    step_bytes = w.algorithmic_bytes() * n_calls * per_step / w.N
    value = step_bytes * args.steps / dt / 1e9
    sample = (f"each step: {per_step} of {w.N} output columns (all {w.M} rows, full K={w.K}) of "
              f"{w.name}, one oracle pass producing the fp16 and bf16 results")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N,
                   "out_dtypes": list(w.out_dtypes)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- GPU arm --

# A synthetic decoder layer at hidden size 4096 (q, k, v, o, fused gate_up,
# down; grouped k/v of 1024; intermediate 12288), M = 1: the GEMVs of one
# decode step of a bf16 model, for the staged-route A/B.
AB_LAYERS = 4
AB_LAYER = [("q", 4096, 4096), ("k", 4096, 1024), ("v", 4096, 1024), ("o", 4096, 4096),
            ("gate_up", 4096, 24576), ("down", 12288, 4096)]


def run_ab_staged(args):
    """The staged route (fp16 GEMV into a staging buffer, then the separate
    narrowing launch) against the GEMV's direct bf16 store, over the GEMVs of
    AB_LAYERS synthetic decoder layers, each route captured in one CUDA graph."""
    rank, local_rank, world = dist_env()
    if rank != 0:
        return 0
    import torch
    import int4_block_quantized_mnb_gb300 as mnb
    from int4_block_quantized_mnb_gb300.synth import make_inputs
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    mnb.load()

    def to_dev(a, dtype):
        return torch.from_numpy(a.view(np.int16).copy() if a.dtype == np.uint16 else a).view(
            dtype).to(dev)

    gemvs = []
    wbytes = 0
    for layer in range(AB_LAYERS):
        for i, (name, K, N) in enumerate(AB_LAYER):
            inp = make_inputs(1, N, K, seed=1000 * layer + i)
            g = dict(name=f"{name}{layer}", K=K, N=N, x=to_dev(inp.x, torch.float16),
                     q=to_dev(inp.qweight, torch.uint8), s=to_dev(inp.scales, torch.float16),
                     z=to_dev(inp.zp, torch.uint8),
                     y16=torch.empty((1, N), dtype=torch.float16, device=dev),
                     ybf=torch.empty((1, N), dtype=torch.bfloat16, device=dev))
            wbytes += g["q"].numel() + 2 * g["s"].numel() + g["z"].numel()
            gemvs.append(g)
    stream = torch.cuda.Stream(dev)
    tc = bool(args.tensor_cores)

    def staged():
        for g in gemvs:
            mnb.gemv(g["x"], g["q"], g["s"], g["z"], "f16", y=g["y16"], stream=stream,
                     weights_ready=True, tensor_cores=tc)
            mnb.cast_f16_to_bf16(g["y16"], g["ybf"], stream=stream)

    def direct():
        for g in gemvs:
            mnb.gemv(g["x"], g["q"], g["s"], g["z"], "bf16", y=g["ybf"], stream=stream,
                     weights_ready=True, tensor_cores=tc)

    def casts():
        for g in gemvs:
            mnb.cast_f16_to_bf16(g["y16"], g["ybf"], stream=stream)

    def timed(fn, reps):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                fn()
        graph.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / reps

    reps = max(20, args.steps if args.steps < 100000 else 200)
    us_direct = timed(direct, reps)
    us_staged = timed(staged, reps)
    us_casts = timed(casts, reps)
    # the staged route's bits equal the direct store's
    staged()
    torch.cuda.synchronize(dev)
    same = all(torch.equal(g["ybf"].view(torch.int16), mnb.cast_f16_to_bf16(g["y16"]).view(
        torch.int16)) for g in gemvs)
    n = len(gemvs)
    line = {
        "metric": "decode step us: staged fp16 GEMV + narrowing launch vs direct bf16 store",
        "unit": "us", "higher_is_better": False, "data": "synthetic", "n_gpus": 1,
        "config": {"workload": f"decode-step-{AB_LAYERS}x-h4096-kv1024-i12288-m1",
                   "gemvs_per_step": n, "weight_bytes": wbytes, "tensor_cores": tc,
                   "timing": f"CUDA events around {reps} replays of one graph per route"},
        "direct": {"us_per_step": us_direct, "launches_per_step": n},
        "staged": {"us_per_step": us_staged, "launches_per_step": 2 * n},
        "narrowing_launches_alone_us_per_step": us_casts,
        "saved_us_per_step": us_staged - us_direct,
        "saved_pct": 100.0 * (us_staged - us_direct) / us_staged,
        "staged_bits_equal_direct": bool(same),
    }
    print(json.dumps(line), flush=True)
    return 0


# The pages' own figures, quoted beside the GB300 numbers (other hardware:
# context, not the target).
PAGES_CONTEXT = {
    "hardware": "A100-class GPU (the pages' \"GPU 6\")",
    "gate_up_gemv": {"us_per_call": 26.69, "dram_tb_per_s": 2.267, "registers_per_thread": 64,
                     "achieved_occupancy_pct": 41.17,
                     "source": "PORT-1 (offline bias+interleave) -- measured NO-GO on the "
                               "multicol asymmetric-zp GEMV (onnx-genai PR 1002), ncu table"},
    "decode_64_tokens_bf16": {"cast_half_launches": [3024, 2398], "kernel_ms": [22.5, 21.3],
                              "source": "perf(cuda): let the split-K decode GEMV store bf16 "
                                        "directly (onnx-genai PR 1550), results"},
}

# The five decode configurations the GEMV is measured on; the attention
# projection is timed once per output dtype.
CONFIG_RECORDS = [
    (0, "tiny-m1-k256-n256", "f16"),
    (1, "attn-proj-m1-k4096-n4096", "f16"),
    (1, "attn-proj-m1-k4096-n4096", "bf16"),
    (2, "gate-up-m1-k5120-n27648", "bf16"),
    (3, "lm-head-m1-k4096-n151936", "f16"),
    (4, "small-batch-m2-k8192-n8192", "bf16"),
    (4, "small-batch-m4-k8192-n8192", "bf16"),
    (4, "small-batch-m8-k8192-n8192", "bf16"),
]


def to_device(a, dtype, dev):
    import torch
    return torch.from_numpy(a.view(np.int16).copy() if a.dtype == np.uint16 else a).view(
        dtype).to(dev)


class DeviceWorkload:
    """One workload's inputs on the device: the activations, R copies of the
    weights (R such that the copies together exceed 4x the L2 size, so a
    launch that follows the rotation finds none of its weights in L2) and one
    output buffer per output dtype."""

    def __init__(self, w, inp, dev, l2_bytes, zero_points=True, multiple=1):
        import torch
        self.w, self.dev = w, dev
        self.x = to_device(inp.x, torch.float16, dev)
        q0 = to_device(inp.qweight, torch.uint8, dev)
        s0 = to_device(inp.scales, torch.float16, dev)
        z0 = to_device(inp.zp, torch.uint8, dev) if zero_points else None
        self.wbytes = q0.numel() + 2 * s0.numel() + (0 if z0 is None else z0.numel())
        self.R = math.ceil(max(1, math.ceil(4 * l2_bytes / self.wbytes)) / multiple) * multiple
        self.copies = [(q0, s0, z0)] + [(q0.clone(), s0.clone(), None if z0 is None else z0.clone())
                                        for _ in range(self.R - 1)]
        self.ys = {o: torch.empty((w.M, w.N), dtype=torch.float16 if o == "f16" else torch.bfloat16,
                                  device=dev) for o in w.out_dtypes}

    def l2_note(self, l2_bytes):
        return (f"inputs larger than L2: {self.R} rotating weight copies, "
                f"{self.R * self.wbytes / 2**20:.0f} MiB vs L2 {l2_bytes / 2**20:.0f} MiB")


def graph_steps(steps, rotation):
    """Steps per captured graph for the K timed steps.  Up to 200 steps: all K
    in one graph (a graph boundary costs the overlap of two launches, about
    3.5 us, which at a few steps per graph would be measured as several
    percent of the call).  Beyond that: a whole number of weight rotations
    (`rotation` steps each) near K / 10, so about ten replays give the
    per-call spread.  Never more than K."""
    if steps <= 200:
        return steps
    return min(steps, rotation * max(1, round(steps / 10 / rotation)))


def graph_replays(launch, n_launches, replays, warm, stream, dev):
    """Captures `n_launches` calls launch(i) in one CUDA graph, replays it
    `warm` times untimed, then `replays` times with a CUDA event recorded
    between consecutive replays on the launching stream.  Returns the
    per-replay times in ms."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_launches):
                launch(i)
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize(dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(replays):
            g.replay()
            evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(replays)]


def traffic_entry(name, bytes_call, tc):
    """The committed ncu DRAM bytes of one launch of `name`'s kernel, or why
    there is none."""
    key = name + ("+tensor-cores" if tc else "")
    t = recorded_traffic(key)
    if t is None:
        return {"bytes": None, "why": "no committed ncu capture for the current kernel sources"}
    return {"bytes": t, "ratio_to_algorithmic": t / bytes_call}


def launch_record(mnb, w, out, tc, block=32, symmetric=False, pm=False):
    info = mnb.launch_info(w.M, w.N, w.K, block=block, out_dtype=out, symmetric=symmetric,
                           tensor_cores=tc, prefill_mma_sync=pm)
    return info


def config_record(mnb, cfg, name, out, dev, stream, l2, peak, props, clk_hint, tc):
    """One configuration's sub-record: per-call time spread over 20 graph
    replays of at least 40 launches each (weights rotating over > 4x L2),
    bandwidth, roofline fractions, the kernel's registers and theoretical
    occupancy, and its committed DRAM traffic."""
    import torch
    from int4_block_quantized_mnb_gb300.synth import WORKLOADS, make_inputs
    w = WORKLOADS[name]
    inp = make_inputs(w.M, w.N, w.K, seed=0)
    d = DeviceWorkload(w, inp, dev, l2)
    n = d.R * max(1, math.ceil(40 / d.R))

    def launch(i):
        q, s, z = d.copies[i % d.R]
        mnb.gemv(d.x, q, s, z, out_dtype=out, y=d.ys[out], stream=stream, weights_ready=True,
                 tensor_cores=tc)

    with torch.cuda.stream(stream):
        for i in range(3):
            launch(i)
    ms = graph_replays(launch, n, 20, 3, stream, dev)
    per = sorted(m * 1e3 / n for m in ms)
    p10, p50, p90 = (pct(per, q) for q in (10, 50, 90))
    b = w.algorithmic_bytes()
    gbs = b / (p50 * 1e-6) / 1e9
    info = launch_record(mnb, w, out, tc)
    rec = {"config": cfg, "workload": name, "M": w.M, "K": w.K, "N": w.N, "out": out,
           "bytes_per_call": b, "us_per_call": p50, "us_p10_p50_p90": [p10, p50, p90],
           "gbs": gbs, "frac_hbm": gbs / peak, "frac_datasheet": gbs / DATASHEET_HBM_GBS,
           "fma_bound": None, "kernel": info["kernel"],
           "registers_per_thread": info["registers_per_thread"],
           "theoretical_occupancy": info["theoretical_occupancy"],
           "grid": info["grid"], "threads": info["threads"], "dynamic_smem": info["dynamic_smem"],
           "traffic": traffic_entry(name, b, tc),
           "timing": f"median of 20 replays of a {n}-launch graph (3 untimed before); "
                     + d.l2_note(l2)}
    if w.M > 1:
        fb = fma_bound(w, props, clk_hint)
        rec["fma_bound"] = {"us": fb["us"], "frac": fb["us"] / p50, "rate_source": fb["rate_source"]}
    del d
    return rec


def main():
    args = parse()
    if args.ab_staged:
        return run_ab_staged(args)
    from int4_block_quantized_mnb_gb300.synth import WORKLOADS, make_inputs
    if args.workload not in WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {list(WORKLOADS)}")
    w = WORKLOADS[args.workload]
    formats = args.block != 32 or args.symmetric or args.m
    if formats:
        w = FormatWorkload(w, args.block, args.symmetric, args.m)
    if args.impl == "reference":
        return run_reference(args, w)

    rank, local_rank, world = dist_env()
    # The CPU oracle's thread pool is created before the first GPU call.
    inp = make_inputs(w.M, w.N, w.K, seed=0, block=w_block(w))
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        gbs, desc, _ = oracle_sample(w, inp, args.cpu_seconds, threads)
        gbs1, desc1, _ = oracle_sample(w, inp, args.cpu_seconds / 2, 1)
        cpu = {"value": gbs, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
               "single_thread": {"value": gbs1, "sample": desc1}, "cpu_model": cpu_model()}

    import torch
    import int4_block_quantized_mnb_gb300 as mnb
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    mnb.load()

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    outs = list(w.out_dtypes)
    L = len(outs)
    d = DeviceWorkload(w, inp, dev, l2, zero_points=w_zp(w, inp) is not None, multiple=L)
    R = d.R
    l2_note = d.l2_note(l2)
    x, copies, ys = d.x, d.copies, d.ys
    z0 = copies[0][2]
    split_k = args.split_k
    tc = bool(args.tensor_cores)
    pm = bool(args.prefill_mma_sync)
    stream = torch.cuda.Stream(dev)

    def step(j):
        # one step: every output dtype of the workload, each on its own weight copy
        for i, o in enumerate(outs):
            q, s, z = copies[(j * L + i) % R]
            mnb.gemv(x, q, s, z, out_dtype=o, split_k=split_k, y=ys[o], stream=stream,
                     weights_ready=True, tensor_cores=tc, block=w_block(w), prefill_mma_sync=pm)

    # Warm-up: W eager steps.
    with torch.cuda.stream(stream):
        for j in range(args.warmup):
            step(j)
    torch.cuda.synchronize(dev)

    # The K timed steps: replays of a graph of G steps (graph_steps); a shorter
    # graph takes the remainder.  Three untimed replays of each graph come
    # first.
    G = graph_steps(args.steps, R // L)
    full, rem = divmod(args.steps, G)

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for j in range(nsteps):
                    step(j)
        return g

    g_main = capture(G) if full else None
    g_rem = capture(rem) if rem else None
    for g in (g_main, g_rem):
        if g is not None:
            for _ in range(3):
                g.replay()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local_rank)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    # one event between consecutive replays: the spread of per-call times
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(full + 1)]
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(full):
            g_main.replay()
            evs[i + 1].record(stream)
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_ms = evs[0].elapsed_time(ev1)
    per_call_us = sorted(evs[i].elapsed_time(evs[i + 1]) * 1e3 / (G * L) for i in range(full))
    clk = clocks.stop()
    if world > 1:
        t = torch.tensor([t_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        t_ms = float(t.item())

    bytes_call = w.algorithmic_bytes()
    launches = args.steps * L
    per_launch_s = t_ms / 1e3 / launches
    value = bytes_call * launches * world / (t_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    achieved = bytes_call / per_launch_s / 1e9
    info = launch_record(mnb, w, outs[0], tc, w_block(w), w_zp(w, inp) is None, pm)

    # End to end through the public API with pinned host buffers, allocated
    # and touched from the CPUs of the GPU's own NUMA node.
    e2e = None
    if not args.no_e2e:
        local = gpu_local_cpus(props)
        saved_affinity = None
        if local is not None and hasattr(os, "sched_setaffinity"):
            try:
                saved_affinity = os.sched_getaffinity(0)
                os.sched_setaffinity(0, local[1])
            except OSError:
                saved_affinity = None
        hx = torch.from_numpy(inp.x.view(np.int16).copy()).view(torch.float16).pin_memory()
        hq = torch.from_numpy(inp.qweight).pin_memory()
        hs = torch.from_numpy(inp.scales.view(np.int16).copy()).view(torch.float16).pin_memory()
        hz = None if z0 is None else torch.from_numpy(inp.zp).pin_memory()
        hy = {o: torch.empty(ys[o].shape, dtype=ys[o].dtype).pin_memory() for o in outs}
        q0, s0 = copies[0][0], copies[0][1]
        dq, ds, dx = torch.empty_like(q0), torch.empty_like(s0), torch.empty_like(x)
        dz = None if z0 is None else torch.empty_like(z0)
        h2d = hx.numel() * 2 + hq.numel() + hs.numel() * 2 + (0 if hz is None else hz.numel())
        d2h = sum(hy[o].numel() * 2 for o in outs)
        E = max(3, min(args.steps, int(4e9 / h2d)))

        def e2e_step():
            dx.copy_(hx, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
            ds.copy_(hs, non_blocking=True)
            if dz is not None:
                dz.copy_(hz, non_blocking=True)
            for o in outs:
                mnb.gemv(dx, dq, ds, dz, out_dtype=o, split_k=split_k, y=ys[o], stream=stream,
                         tensor_cores=tc, block=w_block(w), prefill_mma_sync=pm)
                hy[o].copy_(ys[o], non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e_step()
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(E):
                e2e_step()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        te = e0.elapsed_time(e1) / 1e3
        if saved_affinity is not None:
            os.sched_setaffinity(0, saved_affinity)
        e2e = {"value": bytes_call * L * E / te / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": E,
               "host_numa_node": None if local is None else local[0]}
        del dq, ds, dx, dz

    # One sub-record per decode configuration (default format only).
    records = None
    if rank == 0 and not args.no_configs and not formats:
        del d, copies, ys, g_main, g_rem
        torch.cuda.empty_cache()
        records = []
        for cfg, name, out in CONFIG_RECORDS:
            records.append(config_record(mnb, cfg, name, out, dev, stream, l2, peak, props, clk,
                                         tc))
            torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    # per-call spread: from the timed replays when there are several, else from
    # the configuration sub-record of the same workload (20 replays)
    spread, spread_source = None, None
    if len(per_call_us) > 1:
        spread = [pct(per_call_us, q) for q in (10, 50, 90)]
        spread_source = f"{full} timed replays"
    else:
        for r in records or []:
            if r["workload"] == w.name and r["out"] == outs[0]:
                spread, spread_source = r["us_p10_p50_p90"], "configs sub-record of this workload"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "us_per_call": per_launch_s * 1e6,
        "us_per_call_p10_p50_p90": spread,
        "us_per_call_spread_source": spread_source,
        "pct_of_hbm_peak": 100.0 * achieved / peak,
        "config": {"workload": w.name, "M": w.M, "K": w.K, "N": w.N, "out_dtypes": outs,
                   "block": w_block(w), "zero_points": w_zp(w, inp) is not None,
                   "split_k": split_k if split_k else "auto", "tensor_cores": tc,
                   **({"prefill_form": "mma.sync" if pm else "tcgen05"} if w.M > 8 else {}),
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": l2_note,
                   "timing": f"CUDA events around {full} replays of a {G}-step graph"
                             + (f" + 1 replay of a {rem}-step graph" if rem else "")
                             + "; warm-up: W eager steps, then three untimed replays per graph"},
        "roofline": ({"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                      "frac": achieved / peak, "peak_kind": peak_kind,
                      "traffic": recorded_traffic(w.name + ("+tensor-cores" if tc else "")),
                      "algorithmic_bytes_per_launch": bytes_call,
                      "peak_datasheet": DATASHEET_HBM_GBS,
                      "frac_datasheet": achieved / DATASHEET_HBM_GBS,
                      "fma_bound": fma_bound(w, props, clk) if w.M > 1 else None}
                     if w.M <= 8 else dict(tensor_roofline(w, per_launch_s, achieved, peak),
                                           traffic=recorded_traffic(
                                               w.name + ("+mma-sync" if pm else "")))),
        "launch": info,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
        "context_pages_a100": PAGES_CONTEXT,
        "configs": records,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
