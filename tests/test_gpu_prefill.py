"""GPU parity of the prefill path (M > 8: the tensor-core GEMM with the decode
GEMV's epilogue) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import _gpu
import int4_block_quantized_mnb_gb300 as mnb
from int4_block_quantized_mnb_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu

FORMATS = [(32, False), (32, True), (64, False), (128, True)]
FORMAT_IDS = [f"b{b}-{'sym' if s else 'zp'}" for b, s in FORMATS]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    mnb.load()


def _run_both(inp, symmetric, tc=True):
    """Both output dtypes on the tcgen05 form (the default) or, with tc=False,
    the mma.sync form; checks which form ran and the oracle bound."""
    dev = _gpu.to_device(inp, symmetric=symmetric)
    c0 = mnb.counters()
    y16 = _gpu.bits(_gpu.run(dev, "f16", 0, block=inp.block, prefill_mma_sync=not tc))
    ybf = _gpu.bits(_gpu.run(dev, "bf16", 0, block=inp.block, prefill_mma_sync=not tc))
    c1 = mnb.counters()
    assert c1[16] - c0[16] == 2
    assert c1[17] - c0[17] == (2 if tc else 0)
    assert c1[12] == c0[12]                                     # decode tensor-core math only
    return _gpu.compare(inp, y16, ybf, symmetric=symmetric)


@pytest.mark.parametrize("block,symmetric", FORMATS, ids=FORMAT_IDS)
@pytest.mark.parametrize("M", [9, 16, 33, 64, 65, 130])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (130, 1024), (257, 384)])
def test_small_shapes(block, symmetric, M, N, K):
    if K % block:
        pytest.skip("K not a multiple of the block size")
    inp = make_inputs(M, N, K, seed=M * 11 + N + K + block, block=block)
    _run_both(inp, symmetric, tc=False)


@pytest.mark.parametrize("M,N,K,block,symmetric", [
    (512, 4096, 4096, 32, False), (128, 27648, 5120, 32, False), (257, 4096, 4096, 64, True),
    (1000, 1024, 8192, 128, False),
])
def test_full_size(M, N, K, block, symmetric):
    """Prefill-sized layers on the mma.sync form, every output element compared
    with the oracle."""
    inp = make_inputs(M, N, K, seed=M + N + block, block=block)
    _run_both(inp, symmetric, tc=False)


@pytest.mark.parametrize("block,symmetric", FORMATS, ids=FORMAT_IDS)
@pytest.mark.parametrize("M", [9, 64, 65, 100, 128, 130, 257])
@pytest.mark.parametrize("N,K", [(1, 128), (33, 96), (130, 1024), (257, 384)])
def test_tensor_core_small_shapes(block, symmetric, M, N, K):
    """The tcgen05 form (the default): each weight split exactly into two fp16
    parts, fp32 accumulators in tensor memory; same bound."""
    if K % block:
        pytest.skip("K not a multiple of the block size")
    inp = make_inputs(M, N, K, seed=M * 13 + N + K + block, block=block)
    _run_both(inp, symmetric, tc=True)


@pytest.mark.parametrize("M,N,K,block,symmetric", [
    (512, 4096, 4096, 32, False), (300, 27648, 5120, 64, True), (1000, 1024, 8192, 128, False),
    (300, 19456, 256, 32, False), (2100, 19456, 512, 64, True),
    (16, 27648, 5120, 32, False), (100, 27648, 5120, 64, True),
])
def test_tensor_core_full_size(M, N, K, block, symmetric):
    """Prefill-sized layers on the tcgen05 form (128- and 256-row activation
    tiles), every output element compared with the oracle."""
    inp = make_inputs(M, N, K, seed=M + N + block + 1, block=block)
    _run_both(inp, symmetric, tc=True)


@pytest.mark.parametrize("tc", [False, True], ids=["mma", "tcgen05"])
@pytest.mark.parametrize("M,N,K,block,symmetric", [
    (130, 257, 1024, 32, False), (300, 520, 2048, 64, True), (40, 1000, 512, 128, False),
])
def test_scale_ranges(M, N, K, block, symmetric, tc):
    """Scales above 2 (the tcgen05 form's fp32 split), exactly 2 and just above,
    and subnormal ones, mixed with the usual range within one warp's rows."""
    inp = make_inputs(M, N, K, seed=M + N + 3, block=block)
    sc = inp.scales.view(np.float16).astype(np.float32)
    r = np.arange(N)
    sc[r % 5 == 0] *= 900.0                              # up to 18
    sc[r % 7 == 0] = 2.0
    sc[r % 9 == 0] = np.float32(np.float16(2.0) + np.float16(2.0 ** -9))
    sc[r % 11 == 0] = 2.0 ** -18                        # subnormal
    sc[(r % 13 == 0)[:, None] & (np.arange(sc.shape[1]) % 3 == 0)[None, :]] *= -1.0
    inp.scales[...] = sc.astype(np.float16).view(np.uint16)
    _run_both(inp, symmetric, tc=tc)


@pytest.mark.parametrize("tc", [False, True], ids=["mma", "tcgen05"])
@pytest.mark.parametrize("M,N,K,block,symmetric", [
    (16, 512, 4096, 32, False), (9, 300, 8192, 64, True), (64, 4096, 4096, 128, False),
    (33, 1000, 2048, 32, True), (300, 1024, 4096, 32, False), (200, 2000, 2048, 64, True),
    (100, 200, 8192, 32, False), (128, 300, 4096, 64, True),
])
def test_k_split_over_a_cluster(M, N, K, block, symmetric, tc):
    """Small grids split K over a thread-block cluster (up to 8 CTAs, partial
    tiles summed in rank order through distributed shared memory), in both
    forms: within the bound, and the same bits on every run."""
    inp = make_inputs(M, N, K, seed=M + K + block, block=block)
    _run_both(inp, symmetric, tc=tc)
    dev = _gpu.to_device(inp, symmetric=symmetric)
    a = _gpu.bits(_gpu.run(dev, "f16", 0, block=block, prefill_mma_sync=not tc))
    b = _gpu.bits(_gpu.run(dev, "f16", 0, block=block, prefill_mma_sync=not tc))
    assert np.array_equal(a, b)


def test_exact_zero_rows():
    """Codes equal to their zero-points give exact zeros on the prefill path."""
    M, N, K = 40, 48, 512
    inp = make_inputs(M, N, K, seed=5)
    q = inp.qweight.copy()
    z = inp.zp.copy()
    q[::5] = 0x77
    z[::5] = 0x77
    x, _, s, _ = _gpu.to_device(inp)
    y = _gpu.bits(mnb.gemv(x, torch.from_numpy(q).cuda(), s, torch.from_numpy(z).cuda(), "f16"))
    assert np.all(y[:, ::5] == 0)
    y2 = _gpu.bits(mnb.gemv(x, torch.from_numpy(np.full_like(q, 0x88)).cuda(), s, None, "bf16"))
    assert np.all(y2 == 0)


@pytest.mark.parametrize("tc", [False, True], ids=["mma", "tcgen05"])
@pytest.mark.parametrize("M,N,K,block,symmetric", [
    (20, 96, 256, 32, False), (130, 300, 512, 64, True), (40, 200, 1024, 128, False),
])
def test_large_scales_stay_finite(M, N, K, block, symmetric, tc):
    """Scales of 8192 and 30000 (so (q - zp) s lies far outside the fp16
    range) with small activations (|x| <= 2^-9): the exact sums are finite,
    and both forms must give them within the bound, every element."""
    inp = make_inputs(M, N, K, seed=31 + M, block=block)
    rng = np.random.default_rng(31 + M)
    inp.x = rng.uniform(-2.0 ** -9, 2.0 ** -9, size=(M, K)).astype(np.float16).view(np.uint16)
    sc = np.empty((N, K // block), dtype=np.float32)
    sc[0::2] = 8192.0
    sc[1::2] = 30000.0
    sc[(np.arange(N) % 5 == 0)] *= -1.0
    inp.scales[...] = sc.astype(np.float16).view(np.uint16)
    ref = _gpu.oracle().gemv(inp.x, inp.qweight, inp.scales, None if symmetric else inp.zp,
                             M, N, K, block=block)
    r = _gpu.oracle().f16_to_f64(ref["y_f16"])
    assert np.isfinite(r).all() and (np.abs(r) > 65504 / 15).mean() > 0.01
    _run_both(inp, symmetric, tc=tc)
    dev = _gpu.to_device(inp, symmetric=symmetric)
    y = _gpu.oracle().f16_to_f64(_gpu.bits(_gpu.run(dev, "f16", 0, block=block,
                                                    prefill_mma_sync=not tc)))
    assert np.isfinite(y).all()


@pytest.mark.parametrize("tc", [False, True], ids=["mma", "tcgen05"])
def test_non_finite_inputs_follow_ieee(tc):
    """+inf meeting nonzero weights gives the exact form's +-inf (the tcgen05
    form must not add its low part, whose lo' is often 0 there); +inf meeting
    a code equal to its zero-point gives NaN; -inf and NaN propagate."""
    M, N, K = 20, 70, 512
    inp = make_inputs(M, N, K, seed=12)
    xs = inp.x.copy()
    xs[0, 3] = 0x7C00                    # +inf
    xs[5, 100] = 0xFC00                  # -inf
    xs[7, 200] = 0x7E00                  # NaN
    inp.x = xs
    qw = inp.qweight.copy()
    z0 = int(inp.zp[0, 0]) & 0xF
    qw[0, 1] = (qw[0, 1] & 0x0F) | (z0 << 4)          # row 0, k = 3: q = zp
    inp.qweight = qw
    dev = _gpu.to_device(inp)
    y16 = _gpu.bits(_gpu.run(dev, "f16", 0, prefill_mma_sync=not tc))
    ybf = _gpu.bits(_gpu.run(dev, "bf16", 0, prefill_mma_sync=not tc))
    o = _gpu.oracle()
    ref = o.gemv(inp.x, inp.qweight, inp.scales, inp.zp, M, N, K)
    g, r = o.f16_to_f64(y16), o.f16_to_f64(ref["y_f16"])
    assert np.isnan(r[0, 0]) and np.isinf(r[0]).sum() > 0 and np.isinf(r[5]).sum() > 0
    assert np.array_equal(np.isnan(g), np.isnan(r))
    assert np.array_equal(g[np.isinf(r)], r[np.isinf(r)])
    fin = np.isfinite(r)
    bound = _gpu.REL * np.abs(r[fin]) + _gpu.ABS * ref["abs_sum"][fin]
    assert np.all(np.abs(g[fin] - r[fin]) <= bound)
    assert np.array_equal(ybf, o.f16_to_bf16(y16))


@pytest.mark.parametrize("tc", [False, True], ids=["mma", "tcgen05"])
def test_exact_sums_with_rounded_weights(tc):
    """Small integer activations and one scale per weight row: on even rows a
    small normal one with a full 11-bit significand (1e-4 .. 4e-4), so fp16(w)
    rounds for many weights and the tcgen05 form's low parts are nonzero; on
    odd rows a subnormal one (k 2^-24), so its high parts are subnormal fp16
    operands.  Every sum is exact in fp32 (s times an integer below 2^13), so
    both forms must give the oracle's fp16 bits exactly."""
    M, N, K = 16, 64, 128
    inp = make_inputs(M, N, K, seed=21)
    rng = np.random.default_rng(21)
    inp.x = rng.integers(-3, 4, size=(M, K)).astype(np.float16).view(np.uint16)
    sc = rng.uniform(1e-4, 4e-4, size=N).astype(np.float16)
    sc[1::2] = (rng.integers(1, 1024, size=N // 2) * 2.0 ** -24).astype(np.float16)
    assert np.all(sc[0::2].astype(np.float64) >= 2.0 ** -14)          # normal
    assert np.all(sc[1::2].astype(np.float64) < 2.0 ** -14)           # subnormal
    inp.scales[...] = np.repeat(sc[:, None], inp.scales.shape[1], axis=1).view(np.uint16)
    dev = _gpu.to_device(inp)
    y16 = _gpu.bits(_gpu.run(dev, "f16", 0, prefill_mma_sync=not tc))
    ref = _gpu.oracle().gemv(inp.x, inp.qweight, inp.scales, inp.zp, M, N, K)
    assert np.array_equal(y16, ref["y_f16"]), int((y16 != ref["y_f16"]).sum())


def test_misaligned_activations():
    M, N, K = 20, 70, 512
    inp = make_inputs(M, N, K, seed=8)
    x, q, s, z = _gpu.to_device(inp)
    buf = torch.empty(M * K + 8, dtype=torch.float16, device="cuda")
    xm = buf[1:1 + M * K].view(M, K)
    xm.copy_(x)
    assert xm.data_ptr() % 16 != 0
    # unaligned activations take the synchronous mma.sync form: the bits of
    # the pipelined mma.sync form on aligned activations, never the tcgen05 form
    a = _gpu.bits(mnb.gemv(x, q, s, z, "f16", prefill_mma_sync=True))
    c0 = mnb.counters()
    b = _gpu.bits(mnb.gemv(xm, q, s, z, "f16"))
    assert mnb.counters()[17] == c0[17]
    assert np.array_equal(a, b)
    _gpu.compare(inp, b, None)


def test_weights_ready_chain_matches_plain_calls():
    """Prefill layers back to back, each reading the previous output, with the
    early-weights promise give the bits of plain calls."""
    M = 96
    layers = [(2048, 2048, 32, False), (1024, 2048, 64, True), (2048, 1024, 128, False)]
    devs = [_gpu.to_device(make_inputs(M, N, K, seed=70 + i, block=b), symmetric=sym)
            for i, (N, K, b, sym) in enumerate(layers)]
    x = devs[0][0]
    ref, got = [x], [x]
    for (_, _, b, _), (_, q, s, z) in zip(layers, devs):
        ref.append(mnb.gemv(ref[-1], q, s, z, "f16", block=b))
    torch.cuda.synchronize()
    for (_, _, b, _), (_, q, s, z) in zip(layers, devs):
        got.append(mnb.gemv(got[-1], q, s, z, "f16", block=b, weights_ready=True))
    torch.cuda.synchronize()
    for a, c in zip(ref[1:], got[1:]):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
        assert torch.isfinite(a.float()).all()


def test_decode_batches_keep_their_kernels():
    """M <= 8 never takes the prefill path."""
    inp = make_inputs(8, 300, 8192, seed=2)
    dev = _gpu.to_device(inp)
    c0 = mnb.counters()
    _gpu.run(dev, "f16", 0)
    assert mnb.counters()[16] == c0[16]


def test_no_device_error_recorded():
    assert mnb.device_error() == 0
