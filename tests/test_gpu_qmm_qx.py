"""Prefill GEMM over block-float activations on the block-scaled tensor cores
(mx_qmm_qx) against the oracle's product of the two decoded block-float
operands (or_qmm_qx), on the same quantised activations; the activations
are quantised by the oracle here and by mx_quantize (bit-exact with it) in
the end-to-end case.  The distance to the bf16-activation product is a
property of quantising the activations, reported by the benchmark, not
gated here."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import bf16_bits_to_f64, bf16_host, check_close, check_special, dev_bf16, dev_u8, need_gpu

pytestmark = pytest.mark.gpu


def run_qx(fmt, codes, scales, xc, xs, M, N, K):
    from gemm_decode_register_gb300 import ops

    Y = ops.qmm_qx(fmt, dev_u8(codes), dev_u8(scales), dev_u8(xc), dev_u8(xs), M, N, K)
    return bf16_bits_to_f64(bf16_host(Y))


SHAPES = [(128, 128, 512), (100, 256, 512), (300, 384, 1024), (1000, 512, 2048), (257, 1280, 1536),
          (64, 128, 256)]


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_qmm_qx_parity(orc, fmt, M, N, K):
    """128 x 128 and 128 x 256 tiles (N % 256 decides), ragged M, several
    k-blocks and scale stages, a last scale stage that is only partly used
    (MXFP8 K = 1536: 12 k-blocks in stages of 4; MXFP4: 6 in stages of 2);
    activations N(0,1) quantised by the oracle."""
    need_gpu()
    if K % (256 if fmt == 2 else 512):
        pytest.skip("K outside this format's k-block and scale-row granularity")
    codes, scales = synth.weights(fmt, N, K, M + N + fmt, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, K + fmt)
    xc, xs = orc.quantize(fmt, x, M, K)
    got = run_qx(fmt, codes, scales, xc, xs, M, N, K)
    want = orc.qmm_qx(fmt, codes, scales, xc, xs, M, N, K)
    check_close(got, want, f"qmm_qx fmt{fmt} {M}x{N}x{K}", bf16_out=True)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_qmm_qx_one_hot_scales(orc, fmt):
    """Scales that single out one block: every weight block scale 2^-20
    except one block per row at 2^0 (NVFP4: E4M3 1/512 and 1.0), so a scale
    byte applied to the wrong row or the wrong K block moves outputs by
    orders of magnitude."""
    need_gpu()
    M, N, K = 128, 256, 1024
    codes, scales = synth.weights(fmt, N, K, 5, exp_lo=118, exp_hi=132)
    nb = K // synth.block_of(fmt)
    sc = scales[: N * nb].reshape(N, nb)
    rng = np.random.default_rng(6)
    if fmt == synth.FMT_NVFP4:
        sc[...] = 0x08  # E4M3 2^-9 * 1: 1/512
        sc[np.arange(N), rng.integers(0, nb, size=N)] = 0x38  # 1.0
    else:
        sc[...] = 107
        sc[np.arange(N), rng.integers(0, nb, size=N)] = 127
    x = synth.activations(M, K, 7)
    xc, xs = orc.quantize(fmt, x, M, K)
    got = run_qx(fmt, codes, scales, xc, xs, M, N, K)
    want = orc.qmm_qx(fmt, codes, scales, xc, xs, M, N, K)
    check_close(got, want, f"qmm_qx one-hot scales fmt{fmt}", bf16_out=True)


def test_qmm_qx_rejects_unsupported_k():
    """K not a multiple of 512 (MX formats) or 256 (NVFP4): MX_EUNSUPPORTED."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    M, N, K = 128, 128, 256
    codes, scales = synth.weights(0, N, K, 1)
    with pytest.raises(ops.MxError) as ei:
        ops.qmm_qx(0, dev_u8(codes), dev_u8(scales), dev_u8(codes), dev_u8(scales), M, N, K)
    assert ei.value.status == -2


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_qmm_qx_after_device_quantiser(orc, fmt):
    """mx_quantize then mx_qmm_qx, all on the device, against the oracle's
    quantiser and product; a token holding a NaN gets NaN block scales and
    a NaN output row."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    M, N, K = 200, 512, 2048
    codes, scales = synth.weights(fmt, N, K, 11, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 12)
    x[3, 100] = 0x7FC0  # NaN
    xc, xs = ops.quantize(fmt, dev_bf16(x).view(M, K))
    Y = ops.qmm_qx(fmt, dev_u8(codes), dev_u8(scales), xc, xs, M, N, K)
    got = bf16_bits_to_f64(bf16_host(Y))
    oc, os_ = orc.quantize(fmt, x, M, K)
    assert np.array_equal(xc.cpu().numpy(), oc) and np.array_equal(xs.cpu().numpy(), os_)
    want = orc.qmm_qx(fmt, codes, scales, oc, os_, M, N, K)
    check_special(got, want, f"quantise + qmm_qx fmt{fmt}", bf16_out=True)
    assert np.all(np.isnan(got[3]))


@pytest.mark.parametrize("kind", ["bf16", "mxfp8", "mxfp4", "nvfp4"])
def test_mma_peak_zero_and_filled_operands(kind):
    """The tensor-pipe microbenchmark runs on zero and on random finite
    operands (MX_PEAK_FILLED) without a device error, at rates within a
    factor of two of each other."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    ops.device_error()  # clear
    z = ops.mma_peak_tflops(kind, iters=512, reps=2)
    f = ops.mma_peak_tflops(kind, iters=512, reps=2, filled=True)
    assert ops.device_error() == 0
    assert z > 0 and f > 0
    assert 0.5 < f / z < 2.0


@pytest.mark.parametrize("flags", [0x200, 0x300, 0x700, 0xB00])
def test_mma_peak_probe_modes(flags):
    """The microbenchmark's probes of a GEMM pipeline (rotating operand
    stages, other warps storing into shared or tensor memory meanwhile) run
    without a device error."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    ops.device_error()  # clear
    assert ops.mma_peak_tflops("mxfp4", iters=512, reps=1, flags=flags) > 0
    assert ops.device_error() == 0
