"""mx_qmv_noalloc, the decode GEMV for callers that cannot allocate device
memory (an engine whose allocator owns the whole device pool, or a decode
loop that cannot take the synchronisation of a first-call cudaMalloc): it
must give the same results as mx_qmv, call after call, while its split-K
workspace lives in a fixed array inside the library.  This file is named
to be collected last."""
import ctypes

import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import check_close, dev_bf16, dev_u8, need_gpu

pytestmark = pytest.mark.gpu


def _noalloc(lib, fmt, c, s, x, y, M, N, K):
    import torch

    lib.mx_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return lib.mx_qmv_noalloc(fmt, c.data_ptr(), s.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, K)


# (fmt, M, N, K): the first shape splits K into windows and so passes its
# partial sums and arrival counters through the array (see
# test_first_shape_splits_k); the others run in one window or, K not a
# multiple of 128, on the direct-load kernel
SHAPES = [(0, 4, 2048, 28672), (0, 1, 4096, 8192), (2, 3, 1000, 16384), (1, 2, 512, 96)]


def test_first_shape_splits_k():
    """4 tokens of 28,672 activations are 229,632 bytes once staged as f16
    (rows padded to 28,704): with the weight ring of 4-token passes (116,736
    bytes) they exceed a CTA's shared memory, so the call must split K
    across CTAs and use the array."""
    torch = need_gpu()
    props = torch.cuda.get_device_properties(0)
    smem = getattr(props, "shared_memory_per_block_optin", 232448)
    assert 4 * 28704 * 2 + 116736 > smem


@pytest.mark.parametrize("fmt,M,N,K", SHAPES)
def test_noalloc_matches_qmv_on_two_calls(orc, fmt, M, N, K):
    """The same kernels on the same shape as mx_qmv: the same bits, on two
    calls in a row (the second finds the array as the first left it), and
    the oracle's result within the tolerance."""
    torch = need_gpu()
    from gemm_decode_register_gb300 import ops

    lib = ops.load()
    codes, scales = synth.weights(fmt, N, K, 600 + M, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 700 + M)
    c, s, xd = dev_u8(codes), dev_u8(scales), dev_bf16(x).view(M, K)
    want = ops.qmv(fmt, c, s, xd, N).cpu().numpy()
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(lib, fmt, c, s, xd, y, M, N, K) == 0
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(N).choice(N, 30)]))
    check_close(y.cpu().numpy()[:, rows], orc.qmv_rows(fmt, codes, scales, x, M, N, K, rows),
                f"noalloc fmt{fmt} {M}x{N}x{K}")


def test_noalloc_serves_shapes_beyond_the_array(orc):
    """Eight tokens over a 16384 x 16384 weight would need K windows whose
    partial sums (about 0.4 M floats) exceed the fixed array: that group of
    tokens runs on the direct-load kernel, which needs no workspace, and the
    result agrees with mx_qmv and with the oracle."""
    torch = need_gpu()
    from gemm_decode_register_gb300 import ops

    lib = ops.load()
    fmt, M, N, K = 0, 8, 16384, 16384
    codes, scales = synth.weights(fmt, N, K, 611)
    x = synth.activations(M, K, 612)
    c, s, xd = dev_u8(codes), dev_u8(scales), dev_bf16(x).view(M, K)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, fmt, c, s, xd, y, M, N, K) == 0
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    check_close(got, ops.qmv(fmt, c, s, xd, N).cpu().numpy().astype(np.float64), "noalloc vs qmv")
    rows = np.array([0, 1, 4095, 8191, 12000, N - 1])
    check_close(got[:, rows], orc.qmv_rows(fmt, codes, scales, x, M, N, K, rows), "noalloc vs oracle")
