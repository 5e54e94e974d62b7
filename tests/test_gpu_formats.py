"""GPU parity of the other formats of the family -- block sizes 16, 64 and 128
and the symmetric (no zero-point, every zp 8) dequant -- against the CPU
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import _gpu
import int4_block_quantized_mnb_gb300 as mnb
from int4_block_quantized_mnb_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu

FORMATS = [(16, False), (16, True), (32, True), (64, False), (64, True), (128, False), (128, True)]
FORMAT_IDS = [f"b{b}-{'sym' if s else 'zp'}" for b, s in FORMATS]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    mnb.load()


def expects_step(M, K, block, symmetric):
    """Whether a default launch of this format may take the step kernel:
    every block size, with or without zero-points, when K is a multiple of
    1024 and the staged activations, K / 32 * (64 M + 16) bytes, fit in
    136 KiB; else the general kernel (or, for block 32 with zero-points, the
    row-tile kernel)."""
    return K % 1024 == 0 and K // 32 * (64 * M + 16) <= 136 * 1024


def takes_step(M, N, K, block, symmetric):
    """Whether a default launch runs the step kernel, as the library reports
    it; never outside the routing conditions of expects_step (inside them the
    stage ring may still not fit beside the activations, and the launch then
    runs the general kernel)."""
    step = "step kernel" in mnb.launch_info(M, N, K, block=block, symmetric=symmetric)["kernel"]
    assert not step or expects_step(M, K, block, symmetric), (M, N, K, block, symmetric)
    return step


def _run_both(inp, symmetric, split=0):
    dev = _gpu.to_device(inp, symmetric=symmetric)
    y16 = _gpu.bits(_gpu.run(dev, "f16", split, block=inp.block))
    ybf = _gpu.bits(_gpu.run(dev, "bf16", split, block=inp.block))
    return _gpu.compare(inp, y16, ybf, symmetric=symmetric)


@pytest.mark.parametrize("block,symmetric", FORMATS, ids=FORMAT_IDS)
@pytest.mark.parametrize("M", [1, 2, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (33, 512), (130, 1024), (257, 384)])
def test_small_shapes(block, symmetric, M, N, K):
    if K % block:
        pytest.skip("K not a multiple of the block size")
    inp = make_inputs(M, N, K, seed=M * 7 + N + K + block, block=block)
    c0 = mnb.counters()
    _run_both(inp, symmetric)
    c1 = mnb.counters()
    step = takes_step(M, N, K, block, symmetric)
    assert c1[13] - c0[13] == (2 if step else 0) and c1[15] - c0[15] == (0 if step else 2)


@pytest.mark.parametrize("block,symmetric", FORMATS, ids=FORMAT_IDS)
@pytest.mark.parametrize("split", [1, 2, 3, 8])
def test_every_split(block, symmetric, split):
    """Each requested split (warps per row pair) meets the bound."""
    inp = make_inputs(3, 45, 1024, seed=split + block, block=block)
    _run_both(inp, symmetric, split=split)


@pytest.mark.parametrize("M,N,K,block,symmetric", [
    (1, 4096, 4096, 16, False), (1, 4096, 4096, 64, True), (1, 4096, 4096, 128, False),
    (1, 4096, 4096, 32, True), (1, 27648, 5120, 64, False), (1, 27648, 5120, 64, True),
    (1, 151936, 4096, 128, False), (1, 151936, 4096, 16, True), (8, 8192, 8192, 16, True),
    (4, 8192, 8192, 128, True),
])
def test_full_size(M, N, K, block, symmetric):
    """Decode-layer sizes, every output element compared with the oracle, on
    the kernel the format takes there."""
    inp = make_inputs(M, N, K, seed=N + block, block=block)
    c0 = mnb.counters()[13]
    _run_both(inp, symmetric)
    assert mnb.counters()[13] - c0 == (2 if takes_step(M, N, K, block, symmetric) else 0)


# (block, symmetric, N, K): tiles of 16, 32 and 64 rows, ragged N, stages of 3
# to 16 segments (K = 5120 at N = 4864 takes 32-row tiles and 5 segments a
# stage, so the scale and zero-point boxes start inside a chunk), and the
# largest K whose activations stage
STEP_FORMATS = [
    (16, False, 1, 1024), (16, False, 77, 3072), (16, False, 4864, 5120), (16, True, 1000, 1024),
    (16, True, 4864, 5120), (64, False, 77, 2048), (64, False, 4864, 4096), (64, False, 1000, 6144),
    (64, False, 300, 12288), (64, True, 77, 1024), (64, True, 4864, 5120), (128, False, 1, 4096),
    (128, False, 4864, 8192), (128, False, 1000, 12288), (128, True, 77, 1024),
    (128, True, 4864, 5120), (128, True, 300, 3072), (64, False, 33, 53248),
    # zero-point rows that are not whole 16-byte chunks: per-thread copies
    (64, False, 4864, 5120), (64, False, 27648, 5120), (64, False, 77, 1024), (64, False, 300, 3072),
    (128, False, 4864, 5120), (128, False, 77, 1024), (128, False, 1000, 3072),
    (128, False, 130, 6144), (64, False, 33, 54272),
]


@pytest.mark.parametrize("block,symmetric,N,K", STEP_FORMATS)
def test_step_kernel_formats(block, symmetric, N, K):
    """Blocks 16, 64 and 128 at M = 1 on the step kernel: its scale and
    zero-point boxes follow the block size; every element against the
    oracle, both output dtypes."""
    assert expects_step(1, K, block, symmetric)
    info = mnb.launch_info(1, N, K, block=block, symmetric=symmetric)
    assert "step kernel (CUDA-core" in info["kernel"], info
    inp = make_inputs(1, N, K, seed=N + K + block, block=block)
    c0 = mnb.counters()[13]
    _run_both(inp, symmetric)
    assert mnb.counters()[13] - c0 == 2


@pytest.mark.parametrize("block,symmetric", [(16, False), (16, True), (64, False), (64, True),
                                             (128, False), (128, True)])
@pytest.mark.parametrize("M,N,K", [(2, 300, 4096), (3, 77, 8192), (4, 4864, 5120), (8, 1000, 8192)])
def test_step_kernel_formats_small_batch(block, symmetric, M, N, K):
    """The other block sizes at M = 2 to 8 on the step kernel's two-row
    layout, where the format's K allows it; every element of both dtypes."""
    if K % block:
        pytest.skip("K not a multiple of the block size")
    inp = make_inputs(M, N, K, seed=M * 100 + N + block, block=block)
    c0 = mnb.counters()[13]
    _run_both(inp, symmetric)
    step = takes_step(M, N, K, block, symmetric)
    assert mnb.counters()[13] - c0 == (2 if step else 0)
    if step:
        assert "two rows per lane" in mnb.launch_info(M, N, K, block=block,
                                                      symmetric=symmetric)["kernel"]
    if M <= 4 and expects_step(M, K, block, symmetric):
        assert step                                    # the ring fits at these sizes


@pytest.mark.parametrize("block", [64, 128])
def test_zero_points_by_thread_copies(block):
    """Blocks 64 and 128 with zero-points at K not a multiple of 32 * block:
    the zero-point rows are not whole 16-byte chunks, so the producer warp
    copies them per thread; against the symmetric format and K where the
    tensor copy applies, on the same step kernel, every element."""
    for K in (32 * block + 1024, 32 * block):
        inp = make_inputs(1, 130, K, seed=block + K, block=block)
        for symmetric in (False, True):
            assert takes_step(1, 130, K, block, symmetric)
            c0 = mnb.counters()[13]
            _run_both(inp, symmetric)
            assert mnb.counters()[13] - c0 == 2


@pytest.mark.parametrize("block", [16, 64, 128])
def test_exact_zero_rows(block):
    """Codes equal to their zero-point (asymmetric) or to 8 (symmetric) give an
    exact 0 whatever the activations and scales."""
    M, N, K = 2, 40, 512
    inp = make_inputs(M, N, K, seed=block, block=block)
    q = inp.qweight.copy()
    q[::3] = 0x88                                      # rows 0, 3, ...: every code 8
    x, qd, s, _ = _gpu.to_device(inp, symmetric=True)
    qd = torch.from_numpy(q).cuda()
    y = _gpu.bits(mnb.gemv(x, qd, s, None, "f16", block=block))
    assert np.all(y[:, ::3] == 0)
    z = inp.zp.copy()
    z[::3] = 0x88
    zd = torch.from_numpy(z).cuda()
    y2 = _gpu.bits(mnb.gemv(x, qd, s, zd, "f16", block=block))
    assert np.all(y2[:, ::3] == 0)


@pytest.mark.parametrize("block,symmetric", [(16, True), (64, False)])
def test_misaligned_activations(block, symmetric):
    """x only 2-byte aligned: the scalar activation loads give the same bits."""
    M, N, K = 2, 70, 512
    inp = make_inputs(M, N, K, seed=9, block=block)
    x, q, s, z = _gpu.to_device(inp, symmetric=symmetric)
    buf = torch.empty(M * K + 8, dtype=torch.float16, device="cuda")
    xm = buf[1:1 + M * K].view(M, K)
    xm.copy_(x)
    assert xm.data_ptr() % 16 != 0
    a = _gpu.bits(mnb.gemv(x, q, s, z, "f16", block=block))
    b = _gpu.bits(mnb.gemv(xm, q, s, z, "f16", block=block))
    assert np.array_equal(a, b)
    _gpu.compare(inp, b, None, symmetric=symmetric)


def test_weights_ready_chain_matches_plain_calls():
    """Back-to-back general-format calls, each reading the previous output,
    with the early-weights promise give the bits of plain calls."""
    layers = [(64, True), (16, False), (128, True), (32, True)]
    devs = [_gpu.to_device(make_inputs(1, 2048, 2048, seed=60 + i, block=b), symmetric=sym)
            for i, (b, sym) in enumerate(layers)]
    x = devs[0][0]
    ref, got = [x], [x]
    for (b, _), (_, q, s, z) in zip(layers, devs):
        ref.append(mnb.gemv(ref[-1], q, s, z, "f16", block=b))
    torch.cuda.synchronize()
    for (b, _), (_, q, s, z) in zip(layers, devs):
        got.append(mnb.gemv(got[-1], q, s, z, "f16", block=b, weights_ready=True))
    torch.cuda.synchronize()
    for a, c in zip(ref[1:], got[1:]):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
        assert torch.isfinite(a.float()).all()


def test_weights_ready_chain_with_zero_point_copies():
    """A chain of K = N = 5120 layers, each reading the previous output with
    the early-weights promise: blocks 64 and 128 take their zero-points by
    per-thread copies, blocks 16 and 32 by tensor copies; the bits equal plain
    calls."""
    layers = [(64, False), (128, False), (16, False), (32, False), (64, False)]
    devs = [_gpu.to_device(make_inputs(1, 5120, 5120, seed=80 + i, block=b), symmetric=sym)
            for i, (b, sym) in enumerate(layers)]
    for b, sym in layers:
        assert takes_step(1, 5120, 5120, b, sym)
    x = devs[0][0]
    ref, got = [x], [x]
    for (b, _), (_, q, s, z) in zip(layers, devs):
        ref.append(mnb.gemv(ref[-1], q, s, z, "f16", block=b))
    torch.cuda.synchronize()
    for (b, _), (_, q, s, z) in zip(layers, devs):
        got.append(mnb.gemv(got[-1], q, s, z, "f16", block=b, weights_ready=True))
    torch.cuda.synchronize()
    for a, c in zip(ref[1:], got[1:]):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
    assert mnb.device_error() == 0


@pytest.mark.parametrize("tc", [False, True], ids=["default", "tensor_cores"])
@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (1, 27648, 5120), (2, 300, 8192), (4, 1000, 2048),
                                   (8, 8192, 8192), (1, 1, 1024), (3, 129, 3072)])
def test_symmetric_block32_on_the_step_kernel(M, N, K, tc):
    """Block 32 without zero-points runs the TMA step kernel (constant
    zero-points of 8 in its stages instead of copied ones): parity, the bf16
    invariant, and the kernel that ran."""
    if tc and (K % 1024 or M * K > 33792):
        pytest.skip("outside the tensor-core math's shapes")
    inp = make_inputs(M, N, K, seed=M + N + K, block=32)
    dev = _gpu.to_device(inp, symmetric=True)
    c0 = mnb.counters()
    y16 = _gpu.bits(_gpu.run(dev, "f16", 0, tensor_cores=tc))
    ybf = _gpu.bits(_gpu.run(dev, "bf16", 0, tensor_cores=tc))
    c1 = mnb.counters()
    assert c1[13] - c0[13] == 2 and c1[15] == c0[15]
    assert c1[12] - c0[12] == (2 if tc else 0)
    _gpu.compare(inp, y16, ybf, symmetric=True)


def test_symmetric_and_asymmetric_step_launches_interleave():
    """Symmetric and asymmetric block-32 step launches back to back (with early
    weight streaming) give the bits of plain calls: a launch's constant
    zero-points never leak into the next launch's stages."""
    M, N, K = 1, 4096, 4096
    devs = [_gpu.to_device(make_inputs(M, N, K, seed=90 + i), symmetric=bool(i % 2)) for i in range(4)]
    x = devs[0][0]
    ref = [_gpu.bits(mnb.gemv(x, q, s, z, "f16")) for (_, q, s, z) in devs]
    torch.cuda.synchronize()
    got = [mnb.gemv(x, q, s, z, "f16", weights_ready=True) for (_, q, s, z) in devs * 3]
    torch.cuda.synchronize()
    for i, g in enumerate(got):
        assert np.array_equal(_gpu.bits(g), ref[i % 4])


def test_block32_with_zero_points_keeps_its_kernels():
    """The tuned block-32 asymmetric path never takes the general kernel."""
    inp = make_inputs(1, 4096, 4096, seed=3)
    dev = _gpu.to_device(inp)
    c0 = mnb.counters()
    _gpu.run(dev, "f16", 0)
    c1 = mnb.counters()
    assert c1[15] == c0[15] and c1[13] - c0[13] == 1


def test_no_device_error_recorded():
    assert mnb.device_error() == 0
