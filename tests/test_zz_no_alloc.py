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


# (fmt, M, N, K): the first shape splits K into windows (uses the array's
# partial sums and counters), the others run in one window or fall back to
# the direct-load kernel
SHAPES = [(0, 4, 2048, 28672), (0, 1, 4096, 8192), (2, 3, 1000, 16384), (1, 2, 512, 96)]


@pytest.mark.parametrize("fmt,M,N,K", SHAPES)
def test_noalloc_matches_qmv_on_two_calls(fmt, M, N, K):
    torch = need_gpu()
    from gemm_decode_register_gb300 import ops

    lib = ops.load()
    codes, scales = synth.weights(fmt, N, K, 600 + M, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 700 + M)
    c, s, xd = dev_u8(codes), dev_u8(scales), dev_bf16(x).view(M, K)
    want = ops.qmv(fmt, c, s, xd, N).cpu().numpy().astype(np.float64)
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(lib, fmt, c, s, xd, y, M, N, K) == 0
        torch.cuda.synchronize()
        check_close(y.cpu().numpy(), want, f"noalloc fmt{fmt} {M}x{N}x{K}")


def test_noalloc_rejects_workspace_beyond_the_array():
    """Eight tokens over a 16384 x 16384 weight need K windows whose partial
    sums (about 0.5 M floats) exceed the fixed array: a clear
    MX_EUNSUPPORTED, nothing launched, and mx_qmv still serves the shape."""
    torch = need_gpu()
    from gemm_decode_register_gb300 import ops

    lib = ops.load()
    M, N, K = 8, 16384, 16384
    c = torch.zeros(N * K // 2, dtype=torch.uint8, device="cuda")
    s = torch.full((N * K // 32,), 127, dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, 0, c, s, x, y, M, N, K) == -2
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    assert torch.all(ops.qmv(0, c, s, x, N) == 0)
