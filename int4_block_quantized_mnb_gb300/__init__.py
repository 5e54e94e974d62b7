"""int4 block-quantized MatMulNBits decode GEMV for GB300 (sm_103a).

``gemv`` computes y[m,n] = sum_k x[m,k] * (q[n,k] - zp[n,k/32]) * s[n,k/32]
for M <= 8 decode rows in one launch of the library's CUDA kernel, rounds to
fp16 and optionally narrows to bf16.  This module only marshals torch tensors
into the C ABI of ``libmnb.so`` (include/mnb.h); every arithmetic step runs in
the CUDA kernel.
"""
from __future__ import annotations

import ctypes

from ._native import (BLOCK, FLAG_PREFILL_MMA_SYNC, FLAG_TENSOR_CORES, FLAG_WEIGHTS_READY, MAX_M,
                      MAX_SPLIT_K, NUM_COUNTERS, OUT_BF16, OUT_F16, LaunchInfo, MnbError, check,
                      load)

__all__ = ["gemv", "gemv_ptr", "launch_info", "cast_f16_to_bf16", "split_k_auto", "min_split_k",
           "max_split_k", "counters", "reset_counters", "device_error", "MnbError", "OUT_F16", "OUT_BF16", "BLOCK",
           "MAX_M", "MAX_SPLIT_K", "FLAG_WEIGHTS_READY", "FLAG_TENSOR_CORES",
           "FLAG_PREFILL_MMA_SYNC"]

_DTYPES = {"f16": OUT_F16, "float16": OUT_F16, "bf16": OUT_BF16, "bfloat16": OUT_BF16}


def _out_code(out_dtype) -> int:
    import torch
    if out_dtype in (torch.float16,):
        return OUT_F16
    if out_dtype in (torch.bfloat16,):
        return OUT_BF16
    if isinstance(out_dtype, str) and out_dtype in _DTYPES:
        return _DTYPES[out_dtype]
    if out_dtype in (OUT_F16, OUT_BF16):
        return int(out_dtype)
    raise ValueError(f"out_dtype must be f16 or bf16, got {out_dtype!r}")


def gemv_ptr(x: int, qweight: int, scales: int, zp: int, y: int, M: int, N: int, K: int,
             block: int = BLOCK, out_dtype: int = OUT_F16, split_k: int = 0,
             stream: int = 0, flags: int = 0) -> None:
    """Raw C-ABI call with integer device pointers; raises MnbError on failure."""
    lib = load()
    if flags:
        check(lib.mnb_gemv_flags(x, qweight, scales, zp, y, M, N, K, block, out_dtype, split_k,
                                 flags, stream))
    else:
        check(lib.mnb_gemv(x, qweight, scales, zp, y, M, N, K, block, out_dtype, split_k, stream))


def gemv(x, qweight, scales, zp, out_dtype="f16", split_k: int = 0, y=None, stream=None,
         weights_ready: bool = False, tensor_cores: bool = False, block: int = BLOCK,
         prefill_mma_sync: bool = False):
    """y = MatMulNBits(x, qweight, scales, zp) on the current CUDA device.

    x [M][K] float16, qweight [N][K/2] uint8, scales [N][K/block] float16,
    zp [N][ceil(K/block/2)] uint8 or None (symmetric: every zero-point 8), all
    contiguous CUDA tensors; block is 16, 32, 64 or 128.  Returns y [M][N]
    float16 or bfloat16 (or writes the given ``y``).  ``weights_ready=True``
    promises that the kernel launched just before on the stream does not
    write qweight, scales or zp (static weights), so the call may start
    streaming them before that kernel completes.  ``tensor_cores=True``
    permits the decode step kernel's tensor-core math where it applies
    (MNB_FLAG_TENSOR_CORES).  ``prefill_mma_sync=True`` runs the mma.sync form
    of the prefill GEMM (M > 8) instead of its tcgen05 form
    (MNB_FLAG_PREFILL_MMA_SYNC).
    """
    import torch
    code = _out_code(out_dtype)
    if x.dim() != 2 or qweight.dim() != 2 or scales.dim() != 2 or (zp is not None and zp.dim() != 2):
        raise ValueError("x, qweight, scales and zp must be 2-D")
    M, K = x.shape
    N = qweight.shape[0]
    if block <= 0 or K % block != 0:
        raise ValueError("K must be a multiple of the block size")
    blocks = K // block
    if qweight.shape[1] * 2 != K or scales.shape != (N, blocks) or \
            (zp is not None and zp.shape != (N, (blocks + 1) // 2)):
        raise ValueError("shapes do not match x [M][K], qweight [N][K/2], scales [N][K/block], "
                         "zp [N][ceil(K/block/2)]")
    if x.dtype != torch.float16 or scales.dtype != torch.float16 or \
            qweight.dtype != torch.uint8 or (zp is not None and zp.dtype != torch.uint8):
        raise TypeError("x and scales must be float16; qweight and zp uint8")
    for t in (x, qweight, scales) + (() if zp is None else (zp,)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    ydt = torch.float16 if code == OUT_F16 else torch.bfloat16
    if y is None:
        y = torch.empty((M, N), dtype=ydt, device=x.device)
    elif y.shape != (M, N) or y.dtype != ydt or not y.is_contiguous() or not y.is_cuda:
        raise ValueError("y must be a contiguous [M][N] CUDA tensor of the output dtype")
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        gemv_ptr(x.data_ptr(), qweight.data_ptr(), scales.data_ptr(),
                 0 if zp is None else zp.data_ptr(), y.data_ptr(), M, N, K, int(block), code,
                 int(split_k), stream.cuda_stream,
                 (FLAG_WEIGHTS_READY if weights_ready else 0) |
                 (FLAG_TENSOR_CORES if tensor_cores else 0) |
                 (FLAG_PREFILL_MMA_SYNC if prefill_mma_sync else 0))
    return y


def launch_info(M: int, N: int, K: int, block: int = BLOCK, out_dtype="f16", split_k: int = 0,
                symmetric: bool = False, tensor_cores: bool = False,
                prefill_mma_sync: bool = False, x_aligned: bool = True) -> dict:
    """What ``gemv`` would launch for this shape on the current device
    (mnb_gemv_launch_info): kernel family, grid, threads, cluster, shared
    memory, registers per thread, resident CTAs per SM and theoretical
    occupancy.  The call only inspects pointers for alignment, so stand-in
    addresses with torch's allocation alignment are passed; nothing runs."""
    base = 1 << 40                     # 256-byte aligned stand-ins, far apart
    span = 1 << 36
    x = base + (0 if x_aligned else 2)
    info = LaunchInfo()
    flags = ((FLAG_TENSOR_CORES if tensor_cores else 0) |
             (FLAG_PREFILL_MMA_SYNC if prefill_mma_sync else 0))
    check(load().mnb_gemv_launch_info(x, base + span, base + 2 * span,
                                      0 if symmetric else base + 3 * span, base + 4 * span,
                                      M, N, K, int(block), _out_code(out_dtype), int(split_k),
                                      flags, ctypes.byref(info)))
    return {"kernel": info.kernel.decode(), "counter": info.counter, "grid": info.grid,
            "threads": info.threads, "cluster": info.cluster,
            "dynamic_smem": info.dynamic_smem, "static_smem": info.static_smem,
            "registers_per_thread": info.registers_per_thread,
            "ctas_per_sm": info.ctas_per_sm, "max_threads_per_sm": info.max_threads_per_sm,
            "theoretical_occupancy": info.theoretical_occupancy}


def cast_f16_to_bf16(src, dst=None, stream=None):
    """bf16(src) for a contiguous CUDA float16 tensor, as its own launch (the
    staged route's narrowing kernel); writes ``dst`` (bfloat16, same shape)
    when given, else returns a new tensor."""
    import torch
    if src.dtype != torch.float16 or not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA float16 tensor")
    if dst is None:
        dst = torch.empty(src.shape, dtype=torch.bfloat16, device=src.device)
    elif (dst.dtype != torch.bfloat16 or dst.shape != src.shape or not dst.is_contiguous()
          or not dst.is_cuda):
        raise ValueError("dst must be a contiguous CUDA bfloat16 tensor of src's shape")
    if stream is None:
        stream = torch.cuda.current_stream(src.device)
    with torch.cuda.device(src.device):
        check(load().mnb_cast_f16_to_bf16(src.data_ptr(), dst.data_ptr(), src.numel(),
                                          stream.cuda_stream))
    return dst


def split_k_auto(M: int, N: int, K: int) -> int:
    out = ctypes.c_int(0)
    check(load().mnb_split_k_auto(M, N, K, ctypes.byref(out)))
    return out.value


def min_split_k(M: int, K: int) -> int:
    out = ctypes.c_int(0)
    check(load().mnb_min_split_k(M, K, ctypes.byref(out)))
    return out.value


def max_split_k(K: int) -> int:
    out = ctypes.c_int(0)
    check(load().mnb_max_split_k(K, ctypes.byref(out)))
    return out.value


def counters() -> list:
    buf = (ctypes.c_uint64 * NUM_COUNTERS)()
    n = load().mnb_debug_counters(buf, NUM_COUNTERS)
    return [int(buf[i]) for i in range(n)]


def reset_counters() -> None:
    load().mnb_debug_counters_reset()


def device_error(stream=None, clear: bool = True) -> int:
    import torch
    s = (stream or torch.cuda.current_stream()).cuda_stream
    code = ctypes.c_uint(0)
    check(load().mnb_device_error(s, ctypes.byref(code), 1 if clear else 0))
    return code.value
