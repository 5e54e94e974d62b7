"""ctypes view of libmnb.so, declared from include/mnb.h.

Loading fails loudly when the library is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "libmnb.so")

# Names and values from include/mnb.h.
OUT_F16 = 0
OUT_BF16 = 1
STATUS = {0: "MNB_OK", 1: "MNB_ERR_NULL", 2: "MNB_ERR_SHAPE", 3: "MNB_ERR_BLOCK",
          4: "MNB_ERR_DTYPE", 5: "MNB_ERR_SPLITK", 6: "MNB_ERR_ALIGN", 7: "MNB_ERR_CUDA",
          8: "MNB_ERR_ALIAS", 9: "MNB_ERR_DEVICE", 10: "MNB_ERR_FLAGS"}
ABI_VERSION = 2
FLAG_WEIGHTS_READY = 1
FLAG_TENSOR_CORES = 2
FLAG_PREFILL_MMA_SYNC = 4
MAX_M = 8
MAX_PREFILL_M = 4194240
BLOCK = 32
MAX_SPLIT_K = 8
NUM_COUNTERS = 18


class LaunchInfo(ctypes.Structure):
    """struct mnb_launch_info."""
    _fields_ = [("kernel", ctypes.c_char * 64), ("counter", ctypes.c_int), ("grid", ctypes.c_int),
                ("threads", ctypes.c_int), ("cluster", ctypes.c_int),
                ("dynamic_smem", ctypes.c_int), ("static_smem", ctypes.c_int),
                ("registers_per_thread", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("max_threads_per_sm", ctypes.c_int), ("theoretical_occupancy", ctypes.c_double)]


# Every symbol the header declares, with (restype, argtypes).
_vp, _u8p, _ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "mnb_cast_f16_to_bf16": (ctypes.c_int, [_vp, _vp, ctypes.c_size_t, _vp]),
    "mnb_gemv": (ctypes.c_int, [_vp, _u8p, _vp, _u8p, _vp, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp]),
    "mnb_gemv_flags": (ctypes.c_int, [_vp, _u8p, _vp, _u8p, _vp, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_uint, _vp]),
    "mnb_split_k_auto": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip]),
    "mnb_min_split_k": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _ip]),
    "mnb_max_split_k": (ctypes.c_int, [ctypes.c_int, _ip]),
    "mnb_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mnb_last_error_detail": (ctypes.c_char_p, []),
    "mnb_last_cuda_error": (ctypes.c_char_p, []),
    "mnb_gemv_launch_info": (ctypes.c_int, [_vp, _u8p, _vp, _u8p, _vp, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_uint,
                                            ctypes.POINTER(LaunchInfo)]),
    "mnb_device_error": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint), ctypes.c_int]),
    "mnb_debug_counters": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int]),
    "mnb_debug_counters_reset": (None, []),
    "mnb_abi_version": (ctypes.c_int, []),
}

_lib = None


class MnbError(RuntimeError):
    """A non-OK status from libmnb."""

    def __init__(self, status: int, detail: str = ""):
        self.status = status
        name = STATUS.get(status, f"status {status}")
        super().__init__(f"{name}: {detail}" if detail else name)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmnb.so (built by ``int4_block_quantized_mnb_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIBRARY
    if not os.path.exists(p):
        raise RuntimeError(f"libmnb.so not found at {p}; build it with "
                           "`python -m int4_block_quantized_mnb_gb300.build`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.mnb_abi_version() != ABI_VERSION:
        raise RuntimeError("libmnb.so ABI version mismatch")
    if path is None:
        _lib = lib
    return lib


def check(status: int) -> None:
    if status != 0:
        detail = load().mnb_last_error_detail()
        raise MnbError(status, detail.decode() if detail else "")
