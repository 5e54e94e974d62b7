"""CPU oracle for the int4 block-quantized MatMulNBits decode GEMV.

TEST INFRASTRUCTURE ONLY.  This package wraps ``mnb_oracle.c`` (plain C,
f64 arithmetic) through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline arm of ``bench.py`` may import it; the product library
and its Python binding never do, and the two share no code.

The C source is compiled on first use (or by ``build()``) with gcc into
``oracle/_build/``; floating-point contraction is disabled so the result is the
same on x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mnb_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libmnb_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]

_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source file into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if force or not os.path.exists(LIBRARY) or \
            os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, LIBRARY)
    return LIBRARY


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    u16p = ctypes.POINTER(ctypes.c_uint16)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.mnbo_f16_to_f64.restype = ctypes.c_double
    lib.mnbo_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.mnbo_bf16_to_f64.restype = ctypes.c_double
    lib.mnbo_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.mnbo_f64_to_f16.restype = ctypes.c_uint16
    lib.mnbo_f64_to_f16.argtypes = [ctypes.c_double]
    lib.mnbo_f16_to_bf16.restype = ctypes.c_uint16
    lib.mnbo_f16_to_bf16.argtypes = [ctypes.c_uint16]
    for name, a, b in (("mnbo_f16_to_f64_array", u16p, f64p),
                       ("mnbo_bf16_to_f64_array", u16p, f64p),
                       ("mnbo_f64_to_f16_array", f64p, u16p),
                       ("mnbo_f16_to_bf16_array", u16p, u16p)):
        fn = getattr(lib, name)
        fn.restype = None
        fn.argtypes = [a, b, ctypes.c_size_t]
    lib.mnbo_q_at.restype = ctypes.c_int
    lib.mnbo_q_at.argtypes = [u8p, ctypes.c_int, ctypes.c_int64, ctypes.c_int]
    lib.mnbo_zp_at.restype = ctypes.c_int
    lib.mnbo_zp_at.argtypes = [u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int]
    lib.mnbo_gemv_cols.restype = ctypes.c_int
    lib.mnbo_gemv_cols.argtypes = [u16p, u8p, u16p, u8p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int64,
                                   f64p, f64p, u16p, u16p]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first when ``path`` is None)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """Array-level calls into one loaded oracle library (the default build,
    or a test's deliberately mutated copy)."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    # -- conversions -------------------------------------------------------
    def f16_to_f64(self, bits) -> np.ndarray:
        a = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(a.shape, dtype=np.float64)
        self.lib.mnbo_f16_to_f64_array(_ptr(a, ctypes.c_uint16), _ptr(out, ctypes.c_double), a.size)
        return out

    def bf16_to_f64(self, bits) -> np.ndarray:
        a = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(a.shape, dtype=np.float64)
        self.lib.mnbo_bf16_to_f64_array(_ptr(a, ctypes.c_uint16), _ptr(out, ctypes.c_double), a.size)
        return out

    def f64_to_f16(self, values) -> np.ndarray:
        a = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.mnbo_f64_to_f16_array(_ptr(a, ctypes.c_double), _ptr(out, ctypes.c_uint16), a.size)
        return out

    def f16_to_bf16(self, bits) -> np.ndarray:
        a = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.mnbo_f16_to_bf16_array(_ptr(a, ctypes.c_uint16), _ptr(out, ctypes.c_uint16), a.size)
        return out

    # -- packed format -----------------------------------------------------
    def q_at(self, qweight: np.ndarray, K: int, n: int, k: int) -> int:
        q = np.ascontiguousarray(qweight, dtype=np.uint8)
        return self.lib.mnbo_q_at(_ptr(q, ctypes.c_uint8), K, n, k)

    def zp_at(self, zp: np.ndarray | None, K: int, block: int, n: int, b: int) -> int:
        if zp is None:
            return self.lib.mnbo_zp_at(None, K, block, n, b)
        z = np.ascontiguousarray(zp, dtype=np.uint8)
        return self.lib.mnbo_zp_at(_ptr(z, ctypes.c_uint8), K, block, n, b)

    # -- the GEMV ----------------------------------------------------------
    def gemv(self, x_bits, qweight, scale_bits, zp, M: int, N: int, K: int,
             block: int = 32, cols=None, threads: int = 1) -> dict:
        """Reference outputs for columns ``cols`` (default: all N) of all M rows.

        Returns a dict of [M][ncols] arrays: ``y_exact`` (f64), ``abs_sum``
        (f64, sum of |x*w|), ``y_f16`` and ``y_bf16`` (uint16 bit patterns).
        ``threads`` > 1 splits the columns over host threads (ctypes releases
        the GIL during each call); the arithmetic per column is unchanged.
        """
        x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1)
        q = np.ascontiguousarray(qweight, dtype=np.uint8).reshape(-1)
        s = np.ascontiguousarray(scale_bits, dtype=np.uint16).reshape(-1)
        z = None if zp is None else np.ascontiguousarray(zp, dtype=np.uint8).reshape(-1)
        if cols is None:
            cols = np.arange(N, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64).reshape(-1)
        nc = cols.size
        y_exact = np.zeros((M, nc), dtype=np.float64)
        abs_sum = np.zeros((M, nc), dtype=np.float64)
        y_f16 = np.zeros((M, nc), dtype=np.uint16)
        y_bf16 = np.zeros((M, nc), dtype=np.uint16)
        if nc == 0:
            return dict(y_exact=y_exact, abs_sum=abs_sum, y_f16=y_f16, y_bf16=y_bf16)

        def run(c0: int, c1: int) -> None:
            sub = np.ascontiguousarray(cols[c0:c1])
            ye = np.zeros((M, c1 - c0), dtype=np.float64)
            ya = np.zeros((M, c1 - c0), dtype=np.float64)
            yh = np.zeros((M, c1 - c0), dtype=np.uint16)
            yb = np.zeros((M, c1 - c0), dtype=np.uint16)
            rc = self.lib.mnbo_gemv_cols(
                _ptr(x, ctypes.c_uint16), _ptr(q, ctypes.c_uint8), _ptr(s, ctypes.c_uint16),
                None if z is None else _ptr(z, ctypes.c_uint8),
                M, N, K, block, _ptr(sub, ctypes.c_int64), sub.size,
                _ptr(ye, ctypes.c_double), _ptr(ya, ctypes.c_double),
                _ptr(yh, ctypes.c_uint16), _ptr(yb, ctypes.c_uint16))
            if rc != 0:
                raise ValueError(f"oracle rejected the shape M={M} N={N} K={K} block={block}")
            y_exact[:, c0:c1] = ye
            abs_sum[:, c0:c1] = ya
            y_f16[:, c0:c1] = yh
            y_bf16[:, c0:c1] = yb

        threads = max(1, min(int(threads), nc))
        if threads == 1:
            run(0, nc)
        else:
            edges = np.linspace(0, nc, threads + 1).astype(np.int64)
            with ThreadPoolExecutor(max_workers=threads) as ex:
                list(ex.map(lambda i: run(int(edges[i]), int(edges[i + 1])), range(threads)))
        return dict(y_exact=y_exact, abs_sum=abs_sum, y_f16=y_f16, y_bf16=y_bf16)


def default() -> Oracle:
    return Oracle(load())
