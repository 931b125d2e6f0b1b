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
    ((2, A, A, A, A, 128, 200, 48), -2),   # NVFP4 K % 32 == 16: code rows not 16 bytes apart for the TMA
    ((0, A, A, A, A, 128, 256, 80), -1),   # K not a multiple of the block
    ((0, A, A, A, 0, 128, 256, 64), -1),   # null Y
])
def test_qmm_rejects(lib, args, want):
    assert lib.mx_qmm(*args) == want


Z = 1 << 30  # a workspace size large enough for every case below


@pytest.mark.parametrize("args,want", [
    ((9, A, A, A, A, A, 8, 4, 2, 256, 64, A, Z), -2),       # unknown format
    ((0, A, A, A, A, A, 8, 4, 5, 256, 64, A, Z), -1),       # topk > E
    ((0, A, A, A, 0, A, 8, 4, 2, 256, 64, A, Z), -1),       # null ids
    ((0, A, A, A, A, A, 8, 4, 2, 256, 64, 0, Z), -1),       # null workspace
    ((2, A, A, A, A, A, 8, 4, 2, 200, 48, A, Z), -2),       # NVFP4 K % 32 == 16
    ((0, A, A, A, A, A, 8, 5000, 2, 256, 64, A, Z), -2),    # E > 4096
    ((0, A, A, A, A, A, 8, 4, 2, 256, 64, A, 1024), -1),    # workspace too small
    ((0, A, A, A, A, A, 8, 4, 2, 256, 64, A + 16, Z), -3),  # workspace not 256-byte aligned
    ((0, A, A, A, A + 2, A, 8, 4, 2, 256, 64, A, Z), -3),   # misaligned ids
])
def test_moe_qmm_rejects(lib, args, want):
    assert lib.mx_moe_qmm(*args) == want


@pytest.mark.parametrize("args,want", [
    ((0, A, A, A, A, A, A, A, A, 8, 4, 2, 256, 128, A, Z), 0),     # valid (not called: see below)
    ((2, A, A, A, A, A, A, A, A, 8, 4, 2, 48, 128, A, Z), -2),     # NVFP4 H % 32 == 16 (the gate-up GEMM's K)
    ((2, A, A, A, A, A, A, A, A, 8, 4, 2, 256, 80, A, Z), -2),     # NVFP4 I % 32 == 16 (the down GEMM's K)
    ((0, A, A, A, A, A, A, 0, A, 8, 4, 2, 256, 128, A, Z), -1),    # null router weights
    ((0, A, A, A, A, A, A, A, A, 8, 4, 2, 256, 128, A, 4096), -1),  # workspace too small
    ((0, A, A, A, A, A, A, A + 2, A, 8, 4, 2, 256, 128, A, Z), -3),  # misaligned router weights
])
def test_moe_ffn_prefill_rejects(lib, args, want):
    if want == 0:
        return  # a valid call would launch kernels
    assert lib.mx_moe_ffn_prefill(*args) == want


def _align256(v):
    return (v + 255) // 256 * 256


@pytest.mark.parametrize("T,E,topk,K,I", [(4096, 128, 8, 2048, 768), (1, 8, 8, 256, 128), (37, 300, 3, 64, 0),
                                         (1000, 1, 1, 512, 256)])
def test_prefill_workspace_sizes(lib, T, E, topk, K, I):
    """Workspace = tile table (16 bytes + 16 per group tile of up to 512
    rows, at most (S + 511 * min(S, E)) / 512 tiles for S = T * topk routed
    rows) + sorted row -> slot (4 S) + for E <= 256 the routing's count
    table (4 bytes per expert and chunk of 128 slots, the chunk count
    rounded up to 128, plus 4 bytes per expert) + gathered activations
    (2 S K) [+ SwiGLU output 2 S I], each part 256-byte aligned."""
    S = T * topk
    tiles = (S + 511 * min(S, E)) // 512
    chunks = (S + 127) // 128
    blk = 4 * E * ((chunks + 127) // 128 * 128 + 1) if E <= 256 else 0
    xs = _align256(_align256(_align256(16 + 16 * tiles) + 4 * S) + blk)
    plain = _align256(xs + 2 * S * K)
    assert lib.mx_moe_qmm_workspace_size(T, E, topk, K) == plain
    if I:
        assert lib.mx_moe_ffn_prefill_workspace_size(T, E, topk, K, I) == _align256(plain + 2 * S * I)
    assert lib.mx_moe_qmm_workspace_size(0, E, topk, K) == 0
    assert lib.mx_moe_qmm_workspace_size(T, E, E + 1, K) == 0


@pytest.mark.parametrize("G", [256, 512])
def test_group_tile_bound(G):
    """The grid bound (S + (G - 1) * min(S, E)) / G on the number of group
    tiles of up to G rows covers every routing: brute force over random and
    adversarial row counts per expert."""
    import numpy as np

    rng = np.random.default_rng(G)
    for _ in range(2000):
        E = int(rng.integers(1, 300))
        S = int(rng.integers(1, 5000))
        kind = rng.integers(0, 3)
        if kind == 0:
            counts = np.bincount(rng.integers(0, E, S), minlength=E)
        elif kind == 1:  # as many experts as possible just above a multiple of G
            counts = np.zeros(E, np.int64)
            left = S
            for e in range(E):
                take = min(left, G + 1)
                counts[e] = take
                left -= take
            counts[0] += left
        else:
            counts = np.zeros(E, np.int64)
            counts[rng.integers(0, E)] = S
        tiles = int(sum((c + G - 1) // G for c in counts))
        assert tiles <= (S + (G - 1) * min(S, E)) // G


@pytest.mark.parametrize("args,want", [
    ((9, A, A, A, 4, 64), -2),       # unknown format
    ((0, 0, A, A, 4, 64), -1),       # null x
    ((0, A, A, 0, 4, 64), -1),       # null scales
    ((0, A, A, A, 0, 64), -1),       # M = 0
    ((0, A, A, A, 4, 48), -1),       # K not a multiple of 32
    ((2, A, A, A, 4, 40), -1),       # NVFP4 K not a multiple of 16
    ((0, A + 2, A, A, 4, 64), -3),   # misaligned x
    ((1, A, A + 8, A, 4, 64), -3),   # misaligned codes
])
def test_quantize_rejects(lib, args, want):
    assert lib.mx_quantize(*args) == want


@pytest.mark.parametrize("kind", [-1, 5, 0x105, 0xF05, 0x1000, 0x2003])
def test_mma_peak_rejects_unknown_kinds(lib, kind):
    """kind: 0..4, optionally plus the MX_PEAK_* flags (0x100-0x800);
    anything else is MX_EINVAL, checked before the device is touched."""
    import ctypes

    ms = ctypes.c_float()
    assert lib.mx_mma_peak(kind, 8, ctypes.byref(ms)) == -1


def test_mma_peak_rejects_bad_arguments(lib):
    import ctypes

    ms = ctypes.c_float()
    assert lib.mx_mma_peak(0x103, 0, ctypes.byref(ms)) == -1
    assert lib.mx_mma_peak(3, 8, None) == -1


def test_no_undeclared_exports(lib):
    """Every mx_* function the library exports is declared in include/mx.h
    (the header is the whole ABI)."""
    import shutil
    import subprocess

    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", b.LIB], capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T mx_" in ln}
    assert exported == set(ops.header_symbols())
