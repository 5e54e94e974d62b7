"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
library through its C ABI, and compare with the CPU oracle.

Bound (per element, fp16 arm):  |y - y_ref| <= 2^-10 |y_ref| + 1e-4 sum_k |x_k w_k|
with y_ref the oracle's fp16 result.  bf16 arm: bit-identical to the RNE bf16
narrowing of the same launch configuration's fp16 output, and within the same
bound of the oracle's bf16 value except where the fp16 arm itself differs from
the oracle's fp16 value (one fp16 ulp, a legal accumulation-order effect); there
the two bf16 values may be one bf16 ulp apart.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import int4_block_quantized_mnb_gb300 as mnb
from oracle import Oracle

REL = 2.0 ** -10
ABS = 1e-4

_oracle = None


def oracle() -> Oracle:
    global _oracle
    if _oracle is None:
        _oracle = Oracle()
    return _oracle


def to_device(inp, device="cuda", symmetric=False):
    """(x, qweight, scales, zp) on the device; zp is None for the symmetric format."""
    x = torch.from_numpy(inp.x.view(np.int16).copy()).view(torch.float16).to(device)
    q = torch.from_numpy(inp.qweight).to(device)
    s = torch.from_numpy(inp.scales.view(np.int16).copy()).view(torch.float16).to(device)
    z = None if symmetric else torch.from_numpy(inp.zp).to(device)
    return x, q, s, z


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def sentinel(M, N, out, device="cuda") -> torch.Tensor:
    """An output buffer filled with NaN so unwritten elements are detectable."""
    dt = torch.float16 if out == "f16" else torch.bfloat16
    return torch.full((M, N), float("nan"), dtype=dt, device=device)


def run(dev, out="f16", split_k=0, y=None, tensor_cores=False, block=32, prefill_mma_sync=False):
    x, q, s, z = dev
    M, N = x.shape[0], q.shape[0]
    if y is None:
        y = sentinel(M, N, out, x.device)
    mnb.gemv(x, q, s, z, out_dtype=out, split_k=split_k, y=y, tensor_cores=tensor_cores,
             block=block, prefill_mma_sync=prefill_mma_sync)
    torch.cuda.synchronize()
    return y


def compare(inp, y16_bits, ybf_bits=None, cols=None, threads=None, symmetric=False):
    """Assert the bound and the bf16 invariant on columns ``cols`` (all if None,
    the default everywhere: every one of the M*N outputs is compared); the
    oracle runs at the inputs' block size, without zero-points when
    ``symmetric``, on all host threads unless ``threads`` says otherwise."""
    threads = threads or os.cpu_count() or 1
    o = oracle()
    M, N, K = inp.M, inp.N, inp.K
    ref = o.gemv(inp.x, inp.qweight, inp.scales, None if symmetric else inp.zp, M, N, K,
                 block=inp.block, cols=cols, threads=threads)
    if cols is not None:
        y16_bits = y16_bits[:, cols]
        ybf_bits = None if ybf_bits is None else ybf_bits[:, cols]
    y = o.f16_to_f64(y16_bits)
    yr = o.f16_to_f64(ref["y_f16"])
    bound = REL * np.abs(yr) + ABS * ref["abs_sum"]
    err = np.abs(y - yr)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{bad.sum()} fp16 outputs outside the bound; first at "
                           f"{np.argwhere(bad)[:3].tolist()}: got {y[bad][:3]} want {yr[bad][:3]}")
    stats = dict(n=y.size, f16_mismatch=int((y16_bits != ref["y_f16"]).sum()),
                 max_err_over_bound=float((err / np.maximum(bound, 1e-30)).max()))
    if ybf_bits is not None:
        narrowed = o.f16_to_bf16(y16_bits)
        assert np.array_equal(ybf_bits, narrowed), \
            f"bf16 arm differs from bf16(fp16 arm) at {np.argwhere(ybf_bits != narrowed)[:3].tolist()}"
        yb = o.bf16_to_f64(ybf_bits)
        ybr = o.bf16_to_f64(ref["y_bf16"])
        ok = np.abs(yb - ybr) <= REL * np.abs(ybr) + ABS * ref["abs_sum"]
        f16_differs = y16_bits != ref["y_f16"]
        adjacent = np.abs(ybf_bits.astype(np.int32) - ref["y_bf16"].astype(np.int32)) <= 1
        assert np.all(ok | (f16_differs & adjacent)), "bf16 outputs outside the bound"
        stats["bf16_ulp_off"] = int((~ok).sum())
    return stats
