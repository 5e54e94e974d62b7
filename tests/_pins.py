"""Pins that tie the CPU oracle to facts fixed outside itself.

Each ``check_*`` function raises AssertionError when the given oracle build
disagrees with:
  * the IEEE 754 binary16 / bfloat16 definitions as implemented by numpy and
    torch (independent library routines),
  * hand-derived worked examples stored in ``tests/golden/hand_cases.json``,
  * closed forms (all-equal weights reduce the GEMV to a scaled sum of x),
  * a dense numpy f64 matmul over weights dequantized by code written here,
  * exact invariants (linearity in the scales, permutation of blocks,
    the symmetric zp = 8 special case).
They are used directly by ``test_oracle_pins.py`` and against deliberately
mutated oracle builds by ``test_oracle_mutants.py``.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import torch

from int4_block_quantized_mnb_gb300.synth import make_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_cases.json")


# ---------------------------------------------------------------- helpers --

def all_f16_bits() -> np.ndarray:
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def numpy_f16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bits.view(np.float16).astype(np.float64)


def torch_f16_to_bf16_bits(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(bits.astype(np.uint16).view(np.int16).copy()).view(torch.float16)
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def same_bits_or_both_nan(a_bits, b_bits, to_f64) -> np.ndarray:
    a = to_f64(a_bits)
    b = to_f64(b_bits)
    return (a_bits == b_bits) | (np.isnan(a) & np.isnan(b))


def dense_codes(qweight: np.ndarray, K: int) -> np.ndarray:
    """[N][K] weight codes from packed bytes (low nibble = even k)."""
    N = qweight.shape[0]
    codes = np.empty((N, K), dtype=np.int64)
    codes[:, 0::2] = qweight & 0x0F
    codes[:, 1::2] = qweight >> 4
    return codes


def dense_zero_points(zp, N: int, blocks: int) -> np.ndarray:
    if zp is None:
        return np.full((N, blocks), 8, dtype=np.int64)
    z = np.empty((N, 2 * zp.shape[1]), dtype=np.int64)
    z[:, 0::2] = zp & 0x0F
    z[:, 1::2] = zp >> 4
    return z[:, :blocks]


def numpy_reference(inp, block=32, zp="inputs"):
    """f64 dense reference: dequantize with numpy, then one matmul."""
    K, N = inp.K, inp.N
    blocks = K // block
    z = inp.zp if isinstance(zp, str) else zp
    w = (dense_codes(inp.qweight, K) - np.repeat(dense_zero_points(z, N, blocks), block, axis=1)) \
        * np.repeat(numpy_f16_to_f64(inp.scales), block, axis=1)
    x = numpy_f16_to_f64(inp.x)
    return x @ w.T, np.abs(x) @ np.abs(w).T


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def golden_arrays(case):
    M, N, K, B = case["M"], case["N"], case["K"], case["block"]
    x = np.zeros((M, K), dtype=np.float64)
    for m, k, v in case["x"]:
        x[m, k] = v
    xh = x.astype(np.float16)
    assert np.array_equal(xh.astype(np.float64), x), "fixture x not exact in binary16"
    q = np.zeros((N, K // 2), dtype=np.uint8)
    for n, i, h in case["q_bytes"]:
        q[n, i] = int(h, 16)
    zp = np.zeros((N, (K // B + 1) // 2), dtype=np.uint8)
    for n, i, h in case["zp_bytes"]:
        zp[n, i] = int(h, 16)
    s = np.array(case["scales"], dtype=np.float64)
    sh = s.astype(np.float16)
    assert np.array_equal(sh.astype(np.float64), s), "fixture scale not exact in binary16"
    return xh.view(np.uint16), q, sh.view(np.uint16), (None if case.get("symmetric") else zp)


# ------------------------------------------------------------ conversions --

def check_f16_to_f64(o) -> None:
    bits = all_f16_bits()
    got = o.f16_to_f64(bits)
    want = numpy_f16_to_f64(bits)
    ok = (got == want) | (np.isnan(got) & np.isnan(want))
    assert ok.all(), f"f16->f64 differs at {np.flatnonzero(~ok)[:5]}"
    # signed zero
    assert np.signbit(o.f16_to_f64(np.array([0x8000], np.uint16)))[0]


def check_bf16_to_f64(o) -> None:
    bits = all_f16_bits()  # every bf16 pattern too
    got = o.bf16_to_f64(bits)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    want = t.to(torch.float64).numpy()
    ok = (got == want) | (np.isnan(got) & np.isnan(want))
    assert ok.all(), f"bf16->f64 differs at {np.flatnonzero(~ok)[:5]}"


def f64_probe_values(seed: int = 7) -> np.ndarray:
    """Doubles that exercise every rounding decision of double -> binary16."""
    finite = numpy_f16_to_f64(all_f16_bits())
    finite = np.unique(finite[np.isfinite(finite) & (finite >= 0)])
    mids = (finite[:-1] + finite[1:]) / 2.0                       # exact ties
    above = np.nextafter(mids, np.inf)
    below = np.nextafter(mids, -np.inf)
    rng = np.random.default_rng(seed)
    mags = np.exp2(rng.uniform(-30.0, 17.0, size=200_000))
    extra = np.array([0.0, 65504.0, 65519.99, 65520.0, 65520.000001, 1e6, 2.0**-24, 2.0**-25,
                      3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, 1.0 + 2.0**-11,
                      1.0 + 3 * 2.0**-11, np.inf])
    v = np.concatenate([finite, mids, above, below, mags, extra])
    return np.concatenate([v, -v, [np.nan]])


def check_f64_to_f16(o) -> None:
    v = f64_probe_values()
    got = o.f64_to_f16(v)
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).view(np.uint16)
    ok = same_bits_or_both_nan(got, want, numpy_f16_to_f64)
    assert ok.all(), f"f64->f16 differs for {v[~ok][:5]}"


def check_f16_to_bf16(o) -> None:
    bits = all_f16_bits()
    got = o.f16_to_bf16(bits)
    want = torch_f16_to_bf16_bits(bits)
    ok = same_bits_or_both_nan(got, want, o.bf16_to_f64)
    assert ok.all(), f"f16->bf16 differs at {bits[~ok][:5]}"


# -------------------------------------------------------- packed accessors --

def check_unpack(o) -> None:
    K = 64
    q = np.zeros((2, K // 2), dtype=np.uint8)
    q[0, 0] = 0x21      # k0 = 1, k1 = 2
    q[1, 31] = 0xA7     # row 1: k62 = 7, k63 = 10
    assert o.q_at(q, K, 0, 0) == 1 and o.q_at(q, K, 0, 1) == 2
    assert o.q_at(q, K, 1, 62) == 7 and o.q_at(q, K, 1, 63) == 10
    assert o.q_at(q, K, 1, 0) == 0
    # zp rows are ceil(K/32/2) bytes: K = 96 -> 3 blocks -> 2 bytes per row
    zp = np.array([[0x21, 0xF3], [0x54, 0x06]], dtype=np.uint8)
    assert [o.zp_at(zp, 96, 32, 0, b) for b in range(3)] == [1, 2, 3]
    assert [o.zp_at(zp, 96, 32, 1, b) for b in range(3)] == [4, 5, 6]
    assert o.zp_at(None, 96, 32, 1, 2) == 8


# -------------------------------------------------------------- the GEMV --

def check_golden(o) -> None:
    for case in load_golden():
        x, q, s, zp = golden_arrays(case)
        r = o.gemv(x, q, s, zp, case["M"], case["N"], case["K"], case["block"])
        want = np.array(case["y_exact"], dtype=np.float64)
        assert np.array_equal(r["y_exact"], want), (case["name"], r["y_exact"], want)
        f16 = np.array([[int(h, 16) for h in row] for row in case["y_f16"]], dtype=np.uint16)
        bf = np.array([[int(h, 16) for h in row] for row in case["y_bf16"]], dtype=np.uint16)
        assert np.array_equal(r["y_f16"], f16), (case["name"], r["y_f16"], f16)
        assert np.array_equal(r["y_bf16"], bf), (case["name"], r["y_bf16"], bf)


def check_closed_form(o) -> None:
    """All-equal codes, zero-points and scales: y = (q - zp) * s * sum_k x."""
    for (M, N, K, qc, zc, sv, seed) in ((2, 3, 256, 11, 4, 0.01, 1), (1, 2, 96, 0, 15, 0.0078125, 2),
                                        (3, 1, 64, 9, 9, 0.02, 3)):
        inp = make_inputs(M, N, K, seed=seed)
        q = np.full_like(inp.qweight, qc | (qc << 4))
        zp = np.full_like(inp.zp, zc | (zc << 4))
        sh = np.float16(sv)
        s = np.full(inp.scales.shape, sh).view(np.uint16)
        r = o.gemv(inp.x, q, s, zp, M, N, K)
        xs = numpy_f16_to_f64(inp.x)
        for m in range(M):
            exact = Fraction(qc - zc) * Fraction(float(sh)) * sum(Fraction(float(v)) for v in xs[m])
            want = float(exact)
            assert float(Fraction(want)) == exact, "closed form not exact in f64"
            assert np.all(r["y_exact"][m] == want), (m, r["y_exact"][m], want)
            assert np.all(r["y_f16"][m] == np.float16(want).view(np.uint16))


def check_numpy_dense(o) -> None:
    """Random inputs from the generator against a dense f64 numpy matmul."""
    for (M, N, K, seed) in ((1, 7, 96, 11), (3, 5, 256, 12), (8, 9, 64, 13), (2, 4, 1024, 14)):
        inp = make_inputs(M, N, K, seed=seed)
        r = o.gemv(inp.x, inp.qweight, inp.scales, inp.zp, M, N, K)
        y, a = numpy_reference(inp)
        assert np.allclose(r["y_exact"], y, rtol=0, atol=1e-12 * (1 + a.max()))
        assert np.allclose(r["abs_sum"], a, rtol=1e-12, atol=0)
        f16 = y.astype(np.float16).view(np.uint16)
        # compare the fp16 rounding except where numpy's own f64 sum sits within
        # 1e-9 of a rounding tie (its summation order is not exact)
        v = numpy_f16_to_f64(r["y_f16"])
        near_tie = np.zeros_like(v, dtype=bool)
        for d in (np.nextafter(v.astype(np.float16), np.float16(np.inf)),
                  np.nextafter(v.astype(np.float16), np.float16(-np.inf))):
            mid = (v + d.astype(np.float64)) / 2
            near_tie |= np.abs(y - mid) < 1e-9 * (1 + a)
        assert np.all((r["y_f16"] == f16) | near_tie)


def check_invariants(o) -> None:
    M, N, K = 2, 6, 256
    inp = make_inputs(M, N, K, seed=21)
    base = o.gemv(inp.x, inp.qweight, inp.scales, inp.zp, M, N, K)
    # linearity: doubling every scale doubles the exact sum
    s2 = (numpy_f16_to_f64(inp.scales) * 2).astype(np.float16).view(np.uint16)
    r2 = o.gemv(inp.x, inp.qweight, s2, inp.zp, M, N, K)
    assert np.array_equal(r2["y_exact"], 2 * base["y_exact"])
    # permuting whole blocks of k consistently in x, weights, scales and zp
    blocks = K // 32
    perm = np.array([3, 0, 7, 5, 1, 6, 2, 4])
    xk = inp.x.reshape(M, blocks, 32)[:, perm].reshape(M, K)
    qk = inp.qweight.reshape(N, blocks, 16)[:, perm].reshape(N, K // 2)
    sk = inp.scales[:, perm]
    zc = dense_zero_points(inp.zp, N, blocks)[:, perm]
    zk = (zc[:, 0::2] | (zc[:, 1::2] << 4)).astype(np.uint8)
    rp = o.gemv(xk, qk, np.ascontiguousarray(sk), zk, M, N, K)
    assert np.array_equal(rp["y_exact"], base["y_exact"])
    # symmetric special case: no zero-point array == every zero-point 8
    r8 = o.gemv(inp.x, inp.qweight, inp.scales, np.full_like(inp.zp, 0x88), M, N, K)
    rn = o.gemv(inp.x, inp.qweight, inp.scales, None, M, N, K)
    assert np.array_equal(r8["y_exact"], rn["y_exact"])
    # column selection and threading do not change values
    cols = np.array([5, 0, 3])
    rc = o.gemv(inp.x, inp.qweight, inp.scales, inp.zp, M, N, K, cols=cols, threads=2)
    assert np.array_equal(rc["y_exact"], base["y_exact"][:, cols])


def check_brute_force_tiny(o) -> None:
    """Exhaustive over one weight code and one zero-point: K = 32, one active k."""
    K = 32
    x = np.zeros((1, K), dtype=np.float16)
    x[0, 5] = np.float16(1.5)
    s = np.array([[np.float16(0.25)]]).view(np.uint16)
    for qc in range(16):
        for zc in range(16):
            q = np.zeros((1, 16), dtype=np.uint8)
            q[0, 2] = qc << 4            # k = 5 is the high nibble of byte 2
            zp = np.array([[zc]], dtype=np.uint8)
            r = o.gemv(x.view(np.uint16), q, s, zp, 1, 1, K)
            assert r["y_exact"][0, 0] == 1.5 * (qc - zc) * 0.25


def check_block_sizes_numpy_dense(o) -> None:
    """Block sizes 16, 64 and 128, with and without zero-points, against the
    dense f64 numpy matmul of the same definition."""
    for (M, N, K, B, seed) in ((1, 5, 256, 16, 31), (2, 3, 256, 64, 32), (3, 4, 512, 128, 33),
                               (1, 6, 96, 16, 34), (2, 2, 384, 128, 35)):
        inp = make_inputs(M, N, K, seed=seed, block=B)
        for zp in (inp.zp, None):
            r = o.gemv(inp.x, inp.qweight, inp.scales, zp, M, N, K, block=B)
            y, a = numpy_reference(inp, block=B, zp=zp)
            assert np.allclose(r["y_exact"], y, rtol=0, atol=1e-12 * (1 + a.max())), (B, zp is None)
            assert np.allclose(r["abs_sum"], a, rtol=1e-12, atol=0), (B, zp is None)


def check_block_refinement(o) -> None:
    """A block of B is two blocks of B/2 with the same scale and zero-point:
    the exact sums are equal (same products, same order)."""
    for (M, N, K, B, seed) in ((2, 3, 256, 32, 41), (1, 4, 256, 64, 42), (2, 2, 512, 128, 43)):
        inp = make_inputs(M, N, K, seed=seed, block=B)
        blocks = K // B
        s_half = np.ascontiguousarray(np.repeat(inp.scales, 2, axis=1))
        z = dense_zero_points(inp.zp, N, blocks)
        z2 = np.repeat(z, 2, axis=1)
        zp_half = (z2[:, 0::2] | (z2[:, 1::2] << 4)).astype(np.uint8)
        for zp, zp2 in ((inp.zp, zp_half), (None, None)):
            r = o.gemv(inp.x, inp.qweight, inp.scales, zp, M, N, K, block=B)
            r2 = o.gemv(inp.x, inp.qweight, s_half, zp2, M, N, K, block=B // 2)
            assert np.array_equal(r["y_exact"], r2["y_exact"]), (B, zp is None)
            assert np.array_equal(r["y_f16"], r2["y_f16"])


def check_closed_form_block_sizes(o) -> None:
    """All-equal codes, zero-points and scales give (q - zp) * s * sum_k x at
    every block size; without zero-points zp is 8."""
    for (M, N, K, B, qc, zc, seed) in ((1, 3, 256, 16, 13, 2, 51), (2, 2, 256, 64, 1, 9, 52),
                                       (1, 2, 512, 128, 6, None, 53), (2, 1, 64, 16, 15, None, 54)):
        inp = make_inputs(M, N, K, seed=seed, block=B)
        q = np.full_like(inp.qweight, qc | (qc << 4))
        zp = None if zc is None else np.full_like(inp.zp, zc | (zc << 4))
        sh = np.float16(0.015625)
        s = np.full(inp.scales.shape, sh).view(np.uint16)
        r = o.gemv(inp.x, q, s, zp, M, N, K, block=B)
        xs = numpy_f16_to_f64(inp.x)
        z = 8 if zc is None else zc
        for m in range(M):
            exact = Fraction(qc - z) * Fraction(float(sh)) * sum(Fraction(float(v)) for v in xs[m])
            assert float(Fraction(float(exact))) == exact, "closed form not exact in f64"
            assert np.all(r["y_exact"][m] == float(exact)), (B, m)


ALL_CHECKS = (check_f16_to_f64, check_bf16_to_f64, check_f64_to_f16, check_f16_to_bf16,
              check_unpack, check_golden, check_closed_form, check_numpy_dense,
              check_invariants, check_brute_force_tiny, check_block_sizes_numpy_dense,
              check_block_refinement, check_closed_form_block_sizes)
