"""Parity of the sm_103a GEMV (through the C ABI) with the CPU oracle."""
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


SMALL = [(1, 32), (7, 64), (33, 96), (257, 1024), (130, 4096), (19, 8192)]


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", SMALL)
@pytest.mark.parametrize("split", ["auto", 1, "max"])
def test_small_shapes(M, N, K, split):
    inp = make_inputs(M, N, K, seed=100 + M * 7 + N + K)
    lo, hi = mnb.min_split_k(M, K), mnb.max_split_k(K)
    sk = {"auto": 0, 1: lo, "max": hi}[split]
    dev = _gpu.to_device(inp)
    y16 = _gpu.bits(_gpu.run(dev, "f16", sk))
    ybf = _gpu.bits(_gpu.run(dev, "bf16", sk))
    _gpu.compare(inp, y16, ybf)


@pytest.mark.parametrize("M", [1, 4])
def test_every_split_k(M):
    N, K = 300, 512
    inp = make_inputs(M, N, K, seed=5)
    dev = _gpu.to_device(inp)
    for sk in range(mnb.min_split_k(M, K), mnb.max_split_k(K) + 1):
        y16 = _gpu.bits(_gpu.run(dev, "f16", sk))
        ybf = _gpu.bits(_gpu.run(dev, "bf16", sk))
        _gpu.compare(inp, y16, ybf)


@pytest.mark.parametrize("tc", [False, True], ids=["default", "tensor_cores"])
@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_full_size(name, tc):
    w = WORKLOADS[name]
    inp = make_inputs(w.M, w.N, w.K, seed=0)
    dev = _gpu.to_device(inp)
    y16 = _gpu.bits(_gpu.run(dev, "f16", tensor_cores=tc))
    ybf = _gpu.bits(_gpu.run(dev, "bf16", tensor_cores=tc))
    # every element written (the NaN sentinel is gone) in both arms
    o = _gpu.oracle()
    assert not np.isnan(o.f16_to_f64(y16)).any()
    assert not np.isnan(o.bf16_to_f64(ybf)).any()
    # the bf16 arm is the narrowed fp16 arm everywhere, not only where sampled
    assert np.array_equal(ybf, o.f16_to_bf16(y16))
    # every output element against the oracle
    _gpu.compare(inp, y16, ybf)


@pytest.mark.parametrize("M", [2, 4, 8])
def test_small_batch_every_row_written(M):
    """A launch owns all M*N outputs: no row is left at the sentinel."""
    N, K = 8192, 8192
    inp = make_inputs(M, N, K, seed=M)
    dev = _gpu.to_device(inp)
    y = _gpu.run(dev, "bf16")
    ybits = _gpu.bits(y)
    assert not np.isnan(_gpu.oracle().bf16_to_f64(ybits)).any()
    rows = np.arange(M)
    # rows are distinct computations: no row is a copy of row 0
    for m in rows[1:]:
        assert not np.array_equal(ybits[m], ybits[0])
    y16 = _gpu.bits(_gpu.run(dev, "f16"))
    _gpu.compare(inp, y16, ybits)


def test_counters_prove_the_kernel_ran():
    inp = make_inputs(2, 64, 256, seed=3)
    dev = _gpu.to_device(inp)
    before = mnb.counters()
    _gpu.run(dev, "f16", 1)
    _gpu.run(dev, "bf16", 2)
    after = mnb.counters()
    d = [a - b for a, b in zip(after, before)]
    assert d[0] == 2 and d[1] == 1 and d[2] == 1 and d[3] == 1 and d[4 + 2 - 1] == 2


def test_tensor_core_kernel_only_on_request():
    """The tensor-core kernel runs only with the tensor_cores flag, and then
    only where it applies (no K split, K a multiple of 1024); every launch
    meets the bound."""
    for M, N, K, split, tc, want in ((4, 130, 4096, 1, True, 1), (2, 4096, 4096, 1, True, 1),
                                     (1, 130, 4096, 1, True, 1), (8, 130, 4096, 1, True, 1),
                                     (4, 130, 4096, 2, True, 0), (2, 130, 4096, 1, False, 0),
                                     (1, 4096, 4096, 0, False, 0), (2, 75, 288, 1, True, 0)):
        inp = make_inputs(M, N, K, seed=M + split + K)
        dev = _gpu.to_device(inp)
        before = mnb.counters()[12]
        y16 = _gpu.bits(_gpu.run(dev, "f16", split, tensor_cores=tc))
        ybf = _gpu.bits(_gpu.run(dev, "bf16", split, tensor_cores=tc))
        assert mnb.counters()[12] - before == 2 * want, (M, N, K, split, tc)
        _gpu.compare(inp, y16, ybf)


def test_mixed_shape_chain_matches_plain_calls():
    """A chain of differently shaped launches, each reading the previous
    output, with the early-weights promise gives the bits of plain calls."""
    shapes = [(4096, 4096), (24576, 4096), (4096, 24576), (1024, 4096)]
    layers = [_gpu.to_device(make_inputs(1, N, K, seed=40 + i))[1:]
              for i, (N, K) in enumerate(shapes)]
    x = _gpu.to_device(make_inputs(1, 4096, 4096, seed=39))[0]
    ref = [x]
    for q, sc, z in layers:
        ref.append(mnb.gemv(ref[-1], q, sc, z, "f16"))
    torch.cuda.synchronize()
    got = [x]
    for q, sc, z in layers:
        got.append(mnb.gemv(got[-1], q, sc, z, "f16", weights_ready=True))
    torch.cuda.synchronize()
    for a, b in zip(ref[1:], got[1:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.isfinite(a.float()).all()


def test_step_kernel_takes_default_launches():
    """Without a K split, with K a multiple of 1024 and activations that fit,
    launches run the step kernel (TMA tensor copies, CUDA-core math: four rows
    per lane for M = 2 and 3, two rows per lane for M = 1 and M >= 4); other
    launches run the row-tile kernel.  No default launch uses tensor-core
    math."""
    for M, N, K, split, want in ((1, 4096, 4096, 0, 1), (2, 300, 8192, 1, 1), (4, 130, 4096, 0, 1),
                                 (3, 77, 1024, 1, 1), (5, 130, 4096, 0, 1), (8, 300, 8192, 0, 1),
                                 (7, 40, 2048, 1, 1), (2, 130, 4096, 2, 0), (1, 75, 288, 0, 0)):
        inp = make_inputs(M, N, K, seed=M * 3 + split + K)
        dev = _gpu.to_device(inp)
        c0 = mnb.counters()
        y16 = _gpu.bits(_gpu.run(dev, "f16", split))
        ybf = _gpu.bits(_gpu.run(dev, "bf16", split))
        c1 = mnb.counters()
        assert c1[13] - c0[13] == 2 * want, (M, N, K, split)
        assert c1[12] == c0[12]
        if want:
            assert mnb.split_k_auto(M, N, K) == 1
            layout = "four rows per lane" if M in (2, 3) else "two rows per lane"
            assert layout in mnb.launch_info(M, N, K, split_k=split)["kernel"], (M, N, K)
        _gpu.compare(inp, y16, ybf)


@pytest.mark.parametrize("M,K_fit", [(1, 55296), (2, 30720), (3, 20480), (5, 12288), (8, 8192)])
def test_step_kernel_activation_limit(M, K_fit):
    """Staged activations take K/32 * (64 M + 16) bytes of shared memory, at
    most 136 KiB: the largest K (a multiple of 1024) that fits runs the step
    kernel, with its fewest stages and reduction slots, and the next one runs
    the row-tile kernel.  Every element of both against the oracle."""
    assert K_fit // 32 * (64 * M + 16) <= 136 * 1024 < (K_fit + 1024) // 32 * (64 * M + 16)
    for K, step in ((K_fit, True), (K_fit + 1024, False)):
        N = 300
        assert ("step kernel" in mnb.launch_info(M, N, K)["kernel"]) == step, (M, K)
        inp = make_inputs(M, N, K, seed=M + K)
        dev = _gpu.to_device(inp)
        c0 = mnb.counters()[13]
        y16 = _gpu.bits(_gpu.run(dev, "f16"))
        ybf = _gpu.bits(_gpu.run(dev, "bf16"))
        assert mnb.counters()[13] - c0 == (2 if step else 0), (M, K)
        _gpu.compare(inp, y16, ybf)


TC_SHAPES = [(1, 1024), (17, 1024), (130, 2048), (33, 3072), (300, 5120), (19, 8192)]


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", TC_SHAPES)
def test_tensor_core_small_shapes(M, N, K):
    """Ragged N (partial tiles zero-filled by the tensor copies) and every K
    layout the tensor-core kernel takes (1 to 8 stages per tile, odd and even
    slice counts)."""
    if mnb_x_bytes(M, K) > 66 * 1024:
        pytest.skip("activations too large for the tensor-core kernel")
    inp = make_inputs(M, N, K, seed=300 + M * 11 + N + K)
    dev = _gpu.to_device(inp)
    before = mnb.counters()[12]
    y16 = _gpu.bits(_gpu.run(dev, "f16", 1, tensor_cores=True))
    ybf = _gpu.bits(_gpu.run(dev, "bf16", 1, tensor_cores=True))
    assert mnb.counters()[12] - before == 2
    _gpu.compare(inp, y16, ybf)


def mnb_x_bytes(M, K):
    C = K // 32
    return M * (C * 64 + (0 if C & 1 else 64))


def test_all_zero_weight_rows_give_exact_zero():
    """Rows whose codes all equal their block's zero-point contribute exactly
    zero: the bound is 0 there, so the result must be +-0, on both kernels."""
    for M in (1, 2, 8):
        inp = make_inputs(M, 64, 1024, seed=40 + M)
        q = inp.qweight.copy()
        zp = inp.zp.copy()
        q[::2] = 0x77                      # every code 7 in even rows
        zp[::2] = 0x77                     # every zero-point 7 in even rows
        inp.qweight, inp.zp = q, zp
        for tc in (False, True):
            y16 = _gpu.bits(_gpu.run(_gpu.to_device(inp), "f16", 1, tensor_cores=tc))
            assert np.all((y16[:, ::2] & 0x7FFF) == 0)
            _gpu.compare(inp, y16, None)


def test_misaligned_pointers():
    """x, scales and zp need not be 16-byte aligned (qweight must be)."""
    M, N, K = 2, 75, 96 * 3
    inp = make_inputs(M, N, K, seed=9)
    x, q, s, z = _gpu.to_device(inp)
    xb = torch.empty(M * K + 3, dtype=torch.float16, device="cuda")
    sb = torch.empty(s.numel() + 5, dtype=torch.float16, device="cuda")
    zb = torch.empty(z.numel() + 7, dtype=torch.uint8, device="cuda")
    xo = xb[1:1 + M * K].view(M, K); xo.copy_(x)
    so = sb[3:3 + s.numel()].view(s.shape); so.copy_(s)
    zo = zb[5:5 + z.numel()].view(z.shape); zo.copy_(z)
    ref16 = _gpu.bits(_gpu.run((x, q, s, z), "f16", 1))
    got16 = _gpu.bits(_gpu.run((xo, q, so, zo), "f16", 1))
    assert np.array_equal(ref16, got16)
    got_bf = _gpu.bits(_gpu.run((xo, q, so, zo), "bf16", 2))
    _gpu.compare(inp, _gpu.bits(_gpu.run((xo, q, so, zo), "f16", 2)), got_bf)


def test_zero_point_padding_nibble_ignored():
    M, N, K = 1, 40, 96   # 3 blocks per row: the last high zp nibble is padding
    inp = make_inputs(M, N, K, seed=4)
    dev = list(_gpu.to_device(inp))
    a = _gpu.bits(_gpu.run(tuple(dev), "f16"))
    dev[3] = dev[3] ^ torch.tensor([0, 0xF0], dtype=torch.uint8, device="cuda")
    b = _gpu.bits(_gpu.run(tuple(dev), "f16"))
    assert np.array_equal(a, b)


def test_cuda_graph_capture_matches_eager():
    inp = make_inputs(1, 1000, 4096, seed=11)
    x, q, s, z = _gpu.to_device(inp)
    eager = mnb.gemv(x, q, s, z, "bf16")
    torch.cuda.synchronize()
    y = torch.empty_like(eager)
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            mnb.gemv(x, q, s, z, "bf16", y=y)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("M,N,K,tc", [(1, 16, 64, False), (2, 40, 1024, True)])
def test_non_finite_inputs_follow_ieee(M, N, K, tc):
    inp = make_inputs(M, N, K, seed=2)
    xs = inp.x.copy()
    xs[0, 3] = 0x7C00          # +inf
    inp.x = xs
    # row 0: code at k = 3 equals its block's zero-point, so +inf * 0 = NaN
    qw = inp.qweight.copy()
    z0 = int(inp.zp[0, 0]) & 0xF
    qw[0, 1] = (qw[0, 1] & 0x0F) | (z0 << 4)
    inp.qweight = qw
    dev = _gpu.to_device(inp)
    y16 = _gpu.bits(_gpu.run(dev, "f16", 1, tensor_cores=tc))
    ybf = _gpu.bits(_gpu.run(dev, "bf16", 1, tensor_cores=tc))
    ref = _gpu.oracle().gemv(inp.x, inp.qweight, inp.scales, inp.zp, M, N, K)
    o = _gpu.oracle()
    g, r = o.f16_to_f64(y16), o.f16_to_f64(ref["y_f16"])
    assert np.isnan(r).any()
    assert np.array_equal(np.isnan(g), np.isnan(r))
    assert np.array_equal(g[np.isinf(r)], r[np.isinf(r)])
    # the bf16 arm is the narrowed fp16 arm bit for bit, NaNs included
    assert np.array_equal(ybf, o.f16_to_bf16(y16))


@pytest.mark.parametrize("tc", [False, True], ids=["default", "tensor_cores"])
def test_weights_ready_chain_matches_plain_calls(tc):
    """Back-to-back calls with the early-weights promise (programmatic
    dependent launch) give the same bits as plain calls, also when each call's
    activations are the previous call's output."""
    inp = make_inputs(1, 4096, 4096, seed=17)
    x, q, s, z = _gpu.to_device(inp)
    ref = [x]
    for i in range(8):
        ref.append(mnb.gemv(ref[-1], q, s, z, "f16", tensor_cores=tc))
    torch.cuda.synchronize()
    got = [x]
    for i in range(8):
        got.append(mnb.gemv(got[-1], q, s, z, "f16", weights_ready=True, tensor_cores=tc))
    torch.cuda.synchronize()
    for a, b in zip(ref[1:], got[1:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _gpu.compare(inp, _gpu.bits(got[1]), None)


def test_no_device_error_recorded():
    assert mnb.device_error() == 0
