"""Plants plausible mistakes in a copy of the oracle's C source and checks that
at least one pin catches each of them.  Everything runs on the CPU; the
committed oracle source is never modified."""
import os

import pytest

import _pins
import oracle as oracle_pkg
from oracle import Oracle

# (name, text in mnb_oracle.c, replacement)
MUTANTS = [
    ("weight-nibbles-swapped", "return (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);",
     "return (k % 2 == 0) ? (byte >> 4) : (byte & 0xF);"),
    ("zp-nibbles-swapped", "return (b % 2 == 0) ? (byte & 0xF) : (byte >> 4);",
     "return (b % 2 == 0) ? (byte >> 4) : (byte & 0xF);"),
    ("zp-byte-index", "(size_t)(b / 2)];", "(size_t)(b / 2) * 0];"),
    ("zp-dropped", "double w = (double)(q - z) * s;", "double w = (double)(q) * s; (void)z;"),
    ("zp-sign", "double w = (double)(q - z) * s;", "double w = (double)(z - q) * s;"),
    ("scale-block-index", "scales[(size_t)n * (size_t)blocks + (size_t)b]",
     "scales[(size_t)n * (size_t)blocks + (size_t)(k / 64)]"),
    ("scale-row-index", "scales[(size_t)n * (size_t)blocks + (size_t)b]", "scales[(size_t)b]"),
    ("x-transposed", "x[(size_t)m * (size_t)K + (size_t)k]", "x[(size_t)k * (size_t)M + (size_t)m]"),
    ("weight-row-stride", "qweight[(size_t)n * (size_t)(K / 2) + (size_t)(k / 2)]",
     "qweight[(size_t)n * (size_t)(K / 4) + (size_t)(k / 2)]"),
    ("f16-truncates", "double m = round_half_even(ldexp(a, 10 - E));", "double m = floor(ldexp(a, 10 - E));"),
    ("ties-away", "return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    ("bf16-single-rounding", "uint16_t h = mnbo_f64_to_f16(acc);\n",
     "uint16_t h = mnbo_f64_to_f16(acc); double acc_direct = acc;\n"),
    ("f16-subnormal-as-normal", "v = ldexp((double)f, -24);", "v = ldexp((double)(1024 + f), -25);"),
    ("f16-overflow-late", "if (E > 15)", "if (E > 16)"),
    ("abs-sum-signed", "aacc += fabs(xv * w);", "aacc += xv * w;"),
    ("zp-row-stride", "int stride = (blocks + 1) / 2;", "int stride = blocks / 2;"),
    ("bf16-significand", "double m = round_half_even(ldexp(a, 7 - E));",
     "double m = round_half_even(ldexp(a, 8 - E)) / 2.0;"),
    ("block-fixed-at-32", "int b = k / block;", "int b = k / 32;"),
    ("zp-stride-fixed-at-32", "int blocks = K / block;\n    int stride", "int blocks = K / 32;\n    int stride"),
    ("symmetric-zero-point-0", "return 8;", "return 0;"),
    ("scale-stride-fixed-at-32", "scales[(size_t)n * (size_t)blocks + (size_t)b]",
     "scales[(size_t)n * (size_t)(K / 32) + (size_t)b]"),
]

# The bf16 single-rounding mutant needs its narrowing to read the unrounded sum.
EXTRA = {
    "bf16-single-rounding": ("y_bf16[o] = mnbo_f16_to_bf16(h);",
                             "y_bf16[o] = mnbo_f16_to_bf16(h) * 0 + bf16_direct(acc_direct);"),
}
BF16_DIRECT = r"""
static uint16_t bf16_direct(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e2; frexp(a, &e2); int E = e2 - 1;
    double m = round_half_even(ldexp(a, 7 - E));
    if (m == 256.0) { m = 128.0; E += 1; }
    return sign | (uint16_t)((E + 127) << 7) | (uint16_t)(m - 128.0);
}
"""


def _abs_sum_check(o):
    # the abs-sum output feeds the tolerance; pin it against numpy
    from int4_block_quantized_mnb_gb300.synth import make_inputs
    import numpy as np
    inp = make_inputs(2, 3, 64, seed=5)
    r = o.gemv(inp.x, inp.qweight, inp.scales, inp.zp, 2, 3, 64)
    _, a = _pins.numpy_reference(inp)
    assert np.allclose(r["abs_sum"], a, rtol=1e-12, atol=0)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    with open(oracle_pkg.SOURCE) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor for {name} no longer in the oracle source"
    mutated = src.replace(old, new)
    if name in EXTRA:
        o2, n2 = EXTRA[name]
        assert o2 in mutated
        mutated = mutated.replace(o2, n2)
        mutated = mutated.replace("/* ---- packed-format accessors", BF16_DIRECT + "\n/* ---- packed-format accessors")
    path = tmp_path / f"mutant_{name}.c"
    path.write_text(mutated)
    lib = oracle_pkg.compile_source(str(path), str(tmp_path / f"libmutant_{name}.so"))
    o = Oracle(oracle_pkg.load(lib))
    caught = []
    for check in _pins.ALL_CHECKS + (_abs_sum_check,):
        try:
            check(o)
        except AssertionError:
            caught.append(check.__name__)
        except Exception:  # a crash-free but nonsensical build also counts as caught
            caught.append(check.__name__ + "(error)")
    assert caught, f"no pin catches mutant {name}"
