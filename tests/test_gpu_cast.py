"""The staged route's narrowing kernel (mnb_cast_f16_to_bf16) against the
oracle's fp16 -> bf16 rounding, and the staged route against the direct bf16
store of the GEMV."""
import numpy as np
import pytest
import torch

import _gpu
import int4_block_quantized_mnb_gb300 as mnb
from int4_block_quantized_mnb_gb300.synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from int4_block_quantized_mnb_gb300 import build
    build.build()
    mnb.load()


def test_every_fp16_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    src = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.float16)
    before = mnb.counters()[14]
    got = mnb.cast_f16_to_bf16(src).view(torch.int16).cpu().numpy().view(np.uint16)
    assert mnb.counters()[14] - before == 1
    # bit for bit, NaNs included (the quiet NaN 0x7FC0 with the input's sign)
    assert np.array_equal(got, _gpu.oracle().f16_to_bf16(bits))


@pytest.mark.parametrize("n,soff,doff", [(1, 0, 0), (7, 0, 0), (8, 0, 0), (9, 0, 0),
                                          (1000, 1, 1), (65539, 0, 0), (65539, 3, 1),
                                          (65539, 0, 8), ((1 << 20) + 5, 8, 0)])
def test_sizes_and_alignment(n, soff, doff):
    """16-byte vectors with a scalar tail when both arrays are 16-byte aligned
    (element offsets 0 and 8), element by element otherwise."""
    rng = np.random.default_rng(n + soff + doff)
    bits = rng.integers(0, 0x7C00, size=n + soff, dtype=np.uint16)  # finite values
    buf = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.float16)
    src = buf[soff:]
    dst_buf = torch.full((n + doff + 4,), float("nan"), dtype=torch.bfloat16, device="cuda")
    dst = dst_buf[doff:doff + n]
    mnb.cast_f16_to_bf16(src, dst)
    got = dst.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, _gpu.oracle().f16_to_bf16(bits[soff:]))
    # nothing outside dst written
    assert torch.isnan(dst_buf[:doff]).all() and torch.isnan(dst_buf[doff + n:]).all()


def test_in_place():
    bits = np.arange(0, 0x7C00, 3, dtype=np.uint16)
    t = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.float16)
    out = mnb.cast_f16_to_bf16(t, t.view(torch.bfloat16))
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, _gpu.oracle().f16_to_bf16(bits))


@pytest.mark.parametrize("name", ["attn-proj-m1-k4096-n4096", "small-batch-m2-k8192-n8192"])
@pytest.mark.parametrize("tc", [False, True], ids=["default", "tensor_cores"])
def test_staged_route_equals_direct_store(name, tc):
    """GEMV to an fp16 staging buffer + the narrowing launch gives the bits of
    the GEMV's direct bf16 store."""
    w = WORKLOADS[name]
    inp = make_inputs(w.M, w.N, w.K, seed=5)
    x, q, s, z = _gpu.to_device(inp)
    staged = mnb.cast_f16_to_bf16(mnb.gemv(x, q, s, z, "f16", tensor_cores=tc))
    direct = mnb.gemv(x, q, s, z, "bf16", tensor_cores=tc)
    torch.cuda.synchronize()
    assert torch.equal(staged.view(torch.int16), direct.view(torch.int16))
