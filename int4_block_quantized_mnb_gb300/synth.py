"""Seeded synthetic inputs for the MatMulNBits decode GEMV.

This module only draws random inputs in the packed layout; it holds none of
the method's arithmetic (no dequantization, no dot product, no rounding of
results).  The GPU path, the CPU oracle, the tests and the benchmark all take
their inputs from here.

Distributions (one seed, numpy's PCG64 stream, drawn in this order):
  x       [M][K]        standard normal, rounded to binary16
  qweight [N][K/2]      uint8 uniform on [0, 256): both nibbles uniform on [0, 16)
  scales  [N][K/32]     uniform on [0.002, 0.02], rounded to binary16
  zp      [N][ceil(K/64)] uint8 uniform on [0, 256): both nibbles uniform on
                        [0, 16); when K/32 is odd the last high nibble of each
                        row is padding and is left random on purpose
Drawing whole bytes is the same distribution as drawing the two 4-bit codes
independently and packing them low-nibble-first.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BLOCK = 32


@dataclass(frozen=True)
class Workload:
    """One decode-GEMV shape: M activation rows, K inputs, N outputs."""
    name: str
    M: int
    K: int
    N: int
    out_dtypes: tuple

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move once per call: packed weights, scales,
        zero-points, activations and outputs (2-byte outputs)."""
        return bytes_per_call(self.M, self.N, self.K)


def bytes_per_call(M: int, N: int, K: int, block: int = BLOCK) -> int:
    blocks = K // block
    return (N * K // 2) + N * blocks * 2 + N * ((blocks + 1) // 2) + M * K * 2 + M * N * 2


# The decode-layer shapes this GEMV is measured on.
WORKLOADS = {
    w.name: w for w in (
        Workload("tiny-m1-k256-n256", 1, 256, 256, ("f16",)),
        Workload("attn-proj-m1-k4096-n4096", 1, 4096, 4096, ("f16", "bf16")),
        Workload("gate-up-m1-k5120-n27648", 1, 5120, 27648, ("bf16",)),
        Workload("lm-head-m1-k4096-n151936", 1, 4096, 151936, ("f16",)),
        Workload("small-batch-m2-k8192-n8192", 2, 8192, 8192, ("bf16",)),
        Workload("small-batch-m4-k8192-n8192", 4, 8192, 8192, ("bf16",)),
        Workload("small-batch-m8-k8192-n8192", 8, 8192, 8192, ("bf16",)),
    )
}


@dataclass
class Inputs:
    """Host arrays in the packed layout (binary16 values as uint16 bits)."""
    M: int
    N: int
    K: int
    x: np.ndarray        # uint16 [M][K]
    qweight: np.ndarray  # uint8  [N][K/2]
    scales: np.ndarray   # uint16 [N][K/32]
    zp: np.ndarray       # uint8  [N][ceil(K/64)]
    block: int = BLOCK


def make_inputs(M: int, N: int, K: int, seed: int = 0, block: int = BLOCK) -> Inputs:
    """Draw one seeded input set of the given shape."""
    if K % block != 0 or K % 2 != 0:
        raise ValueError("K must be a multiple of the block size")
    blocks = K // block
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K)).astype(np.float16).view(np.uint16)
    qweight = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.uniform(0.002, 0.02, size=(N, blocks)).astype(np.float16).view(np.uint16)
    zp = rng.integers(0, 256, size=(N, (blocks + 1) // 2), dtype=np.uint8)
    return Inputs(M, N, K, np.ascontiguousarray(x), qweight,
                  np.ascontiguousarray(scales), zp, block)
