"""The C-ABI library loads, exports every symbol include/mnb.h declares, and
rejects bad arguments on the host before touching a device (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mnb.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mnb_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from int4_block_quantized_mnb_gb300 import build, _native
    build.build()
    return _native.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mnb_gemv", "mnb_status_string", "mnb_last_error_detail", "mnb_last_cuda_error",
              "mnb_split_k_auto", "mnb_device_error", "mnb_debug_counters",
              "mnb_gemv_launch_info"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from int4_block_quantized_mnb_gb300 import _native
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in mnb.h but not exported"
        assert name in _native.SIGNATURES, f"{name} has no ctypes declaration"


def test_status_numbering_matches_the_header(lib):
    """The values the header gives each status (MNB_ERR_CUDA is 7), read from
    the header text itself, agree with the Python binding's table."""
    from int4_block_quantized_mnb_gb300 import _native
    text = open(HEADER).read()
    pairs = dict((name, int(v)) for name, v in re.findall(r"\b(MNB_(?:OK|ERR_[A-Z]+)) = (\d+)", text))
    assert pairs["MNB_ERR_CUDA"] == 7 and pairs["MNB_ERR_ALIAS"] == 8
    assert {v: k for k, v in pairs.items()} == _native.STATUS


def test_last_cuda_error_is_the_detail_text(lib):
    assert call(lib, x=0) == 1
    assert lib.mnb_last_cuda_error() == lib.mnb_last_error_detail() != b""


def test_launch_info_validates_before_any_device_call(lib):
    from int4_block_quantized_mnb_gb300._native import LaunchInfo
    info = LaunchInfo()
    assert lib.mnb_gemv_launch_info(X, Q, S, Z, Y, 1, 64, 256, 32, 0, 1, 0, None) == 1
    assert lib.mnb_gemv_launch_info(0, Q, S, Z, Y, 1, 64, 256, 32, 0, 1, 0, ctypes.byref(info)) == 1
    assert lib.mnb_gemv_launch_info(X, Q, S, Z, Y, 1, 64, 256, 48, 0, 1, 0, ctypes.byref(info)) == 3
    assert lib.mnb_gemv_launch_info(X, Q, S, Z, X, 1, 64, 256, 32, 0, 1, 0, ctypes.byref(info)) == 8


def test_status_strings(lib):
    for s in range(11):
        assert lib.mnb_status_string(s) != b"unknown status"
    assert lib.mnb_status_string(99) == b"unknown status"
    assert lib.mnb_abi_version() == 2


# Fake but 16-byte-aligned, non-overlapping addresses: validation fails before
# anything is dereferenced or launched.
X, Q, S, Z, Y = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000


def call(lib, x=X, q=Q, s=S, z=Z, y=Y, M=1, N=64, K=256, block=32, out=0, split=1):
    return lib.mnb_gemv(x, q, s, z, y, M, N, K, block, out, split, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=0), 1), (dict(q=0), 1), (dict(s=0), 1), (dict(y=0), 1),
    (dict(block=48), 3), (dict(block=256), 3), (dict(block=8), 3), (dict(block=0), 3),
    (dict(K=64, block=128), 2), (dict(K=96, block=64), 2), (dict(K=160, block=64, z=0), 2),
    (dict(M=0), 2), (dict(M=4194241), 2), (dict(N=0), 2), (dict(N=-3), 2),
    (dict(M=9, block=16), 3), (dict(M=64, split=2), 5), (dict(M=9, K=96, block=64), 2),
    (dict(M=16, out=2), 4), (dict(M=16, q=Q + 8), 6), (dict(M=16, y=X), 8),
    (dict(K=0), 2), (dict(K=48), 2), (dict(K=31), 2),
    (dict(out=2), 4), (dict(out=-1), 4),
    (dict(q=Q + 8), 6), (dict(x=X + 1), 6), (dict(s=S + 1), 6), (dict(y=Y + 1), 6),
    (dict(y=X), 8), (dict(y=Q + 16), 8), (dict(y=S), 8), (dict(y=Z), 8),
    (dict(split=9), 5), (dict(split=-1), 5), (dict(K=64, split=3), 5),
    (dict(M=8, K=16384, split=1), 5),
])
def test_host_validation(lib, kw, status):
    assert call(lib, **kw) == status
    assert lib.mnb_last_error_detail()


def test_unknown_flags_rejected(lib):
    for bad in (8, 16, 0x80000000, 9):
        assert lib.mnb_gemv_flags(X, Q, S, Z, Y, 1, 64, 256, 32, 0, 1, bad, None) == 10
    # valid flags fall through to the ordinary checks (here: a NULL pointer)
    for ok in (1, 2, 3, 4, 7):
        assert lib.mnb_gemv_flags(0, Q, S, Z, Y, 1, 64, 256, 32, 0, 1, ok, None) == 1


def test_split_limits(lib):
    out = ctypes.c_int(0)
    assert lib.mnb_max_split_k(4096, ctypes.byref(out)) == 0 and out.value == 8
    assert lib.mnb_max_split_k(64, ctypes.byref(out)) == 0 and out.value == 2
    assert lib.mnb_min_split_k(8, 16384, ctypes.byref(out)) == 0 and out.value == 2
    assert lib.mnb_min_split_k(1, 12288, ctypes.byref(out)) == 0 and out.value == 1
    assert lib.mnb_min_split_k(1, 16384, ctypes.byref(out)) == 0 and out.value == 2
    assert lib.mnb_min_split_k(9, 4096, ctypes.byref(out)) == 2
    assert lib.mnb_max_split_k(4096, None) == 1


def test_no_fallback_when_library_missing(tmp_path):
    from int4_block_quantized_mnb_gb300 import _native
    with pytest.raises(RuntimeError, match="not found"):
        _native.load(str(tmp_path / "libmnb.so"))


def test_cast_host_validation(lib):
    """mnb_cast_f16_to_bf16 checks its arguments before touching the device."""
    assert lib.mnb_cast_f16_to_bf16(0, 0, 0, None) == 0                 # n = 0: nothing to do
    assert lib.mnb_cast_f16_to_bf16(0, 4096, 8, None) == 1              # NULL
    assert lib.mnb_cast_f16_to_bf16(4096, 0, 8, None) == 1
    assert lib.mnb_cast_f16_to_bf16(4097, 8192, 8, None) == 6           # odd address
    assert lib.mnb_cast_f16_to_bf16(4096, 4100, 8, None) == 8           # partial overlap
