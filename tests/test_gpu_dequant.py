"""GPU decode is bit-exact with the oracle: every code byte under every
scale byte, for each format (the kernels' decode path, through
mx_dequant)."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import dev_u8, need_gpu, same_bits_f32

pytestmark = pytest.mark.gpu


def _exhaustive(fmt, g=None):
    # row e: all 256 code bytes, every block scaled by byte e
    N = 256
    if fmt == synth.FMT_MXFP8:
        K = 256
        codes = np.tile(np.arange(256, dtype=np.uint8), (N, 1))
    else:
        K = 512
        codes = np.tile(np.arange(256, dtype=np.uint8), (N, 1))
    nblk = K // synth.block_of(fmt)
    scales = np.repeat(np.arange(256, dtype=np.uint8), nblk)
    if fmt == synth.FMT_NVFP4:
        scales = np.concatenate([scales, np.array([g], dtype="<f4").view(np.uint8)])
    return codes, scales, N, K


@pytest.mark.parametrize("fmt,g", [(0, None), (1, None), (2, 1.0), (2, float(np.float32(1) / np.float32(448))),
                                   (2, 3.0), (2, 2.0 ** -20)])
def test_dequant_exhaustive_bit_exact(orc, fmt, g):
    torch = need_gpu()
    from gemm_decode_register_gb300 import ops

    codes, scales, N, K = _exhaustive(fmt, g)
    W = ops.dequant(fmt, dev_u8(codes), dev_u8(scales), N, K)
    torch.cuda.synchronize()
    want = orc.dequant(fmt, codes, scales, N, K)
    assert same_bits_f32(W.cpu().numpy(), want)


@pytest.mark.parametrize("fmt,N,K", [(0, 37, 96), (1, 19, 160), (2, 23, 48), (2, 5, 16)])
def test_dequant_random_ragged(orc, fmt, N, K):
    need_gpu()
    from gemm_decode_register_gb300 import ops

    codes, scales = synth.weights(fmt, N, K, 7, exp_lo=0, exp_hi=255)
    W = ops.dequant(fmt, dev_u8(codes), dev_u8(scales), N, K)
    assert same_bits_f32(W.cpu().numpy(), orc.dequant(fmt, codes, scales, N, K))
