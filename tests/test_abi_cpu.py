"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/mx.h declares, and rejects bad arguments on the host before any
CUDA call (no GPU needed)."""
import pytest

from gemm_decode_register_gb300 import build as b
from gemm_decode_register_gb300 import ops


@pytest.fixture(scope="module")
def lib():
    b.build()
    return ops.load()


def test_exports_every_declared_symbol(lib):
    names = ops.header_symbols()
    assert set(names) >= {"mx_qmv", "mx_moe_qmv", "mx_qmm", "mx_dequant", "mx_set_stream",
                          "mx_device_error", "mx_strerror", "mx_swiglu", "mx_moe_combine"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in (0, -1, -2, -3, -4, -5):
        assert lib.mx_strerror(s)
    assert lib.mx_strerror(-99) == b"unknown status"


A = 1 << 20  # an aligned fake address: validation fails before it is used


@pytest.mark.parametrize("args,want", [
    ((9, A, A, A, A, 1, 8, 32), -2),      # unknown format
    ((0, 0, A, A, A, 1, 8, 32), -1),      # null codes
    ((0, A, A, A, A, 0, 8, 32), -1),      # M = 0
    ((0, A, A, A, A, 1, 0, 32), -1),      # N = 0
    ((0, A, A, A, A, 1, 8, 48), -1),      # K not a multiple of 32
    ((2, A, A, A, A, 1, 8, 40), -1),      # NVFP4 K not a multiple of 16
    ((0, A + 4, A, A, A, 1, 8, 32), -3),  # misaligned codes
    ((0, A, A, A, A + 8, 1, 8, 32), -3),  # misaligned y
    ((0, A, A, A, A, 1, 8, (1 << 20) + 32), -2),  # K too large
])
def test_qmv_rejects(lib, args, want):
    assert lib.mx_qmv(*args) == want


@pytest.mark.parametrize("args,want", [
    ((0, A, A, A, A, A, 1, 4, 5, 8, 32), -1),       # topk > E
    ((0, A, A, A, 0, A, 1, 8, 2, 8, 32), -1),       # null ids
    ((0, A, A, A, A, A, 200, 8, 8, 8, 32), -2),     # T * topk > 1024
    ((0, A, A, A, A + 2, A, 1, 8, 2, 8, 32), -3),   # misaligned ids
    ((1, A, A, A, A, A, 1, 8, 2, 8, 16), -1),       # MXFP8 K = 16
])
def test_moe_rejects(lib, args, want):
    assert lib.mx_moe_qmv(*args) == want


@pytest.mark.parametrize("args,want", [
    ((0, A, A, A, A, 128, 200, 64), -2),   # N not a multiple of 256
    ((0, A, A, A, A, 128, 256, 96), -2),   # K not a multiple of 64
    ((0, A, A, A, 0, 128, 256, 64), -1),   # null Y
])
def test_qmm_rejects(lib, args, want):
    assert lib.mx_qmm(*args) == want
