"""Prefill GEMM (tcgen05) on the GPU against the oracle: small and ragged
shapes for every format, exact one-hot rows, agreement with qmv, and the two
4096-token prefill shapes at full size checked on whole sampled rows."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import (bf16_bits_to_f64, bf16_host, check_close, dev_bf16, dev_u8, need_gpu,
                      same_values)

pytestmark = pytest.mark.gpu


def run_qmm(fmt, codes, scales, X, N):
    from gemm_decode_register_gb300 import ops

    Y = ops.qmm(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(X), N)
    return bf16_bits_to_f64(bf16_host(Y))


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (256, 512, 256), (512, 256, 1024), (100, 256, 128),
                                   (300, 768, 320), (1000, 9728, 192)])
def test_qmm_parity(orc, fmt, M, N, K):
    """Pair tiles of 256 rows, and (1000 x 9728: 76 pairs, one wave) of 512
    rows with a ragged last tile."""
    need_gpu()
    codes, scales = synth.weights(fmt, N, K, M + K, exp_lo=118, exp_hi=132)
    X = synth.activations(M, K, N + K)
    check_close(run_qmm(fmt, codes, scales, X, N), orc.qmv(fmt, codes, scales, X, M, N, K),
                f"qmm fmt{fmt} {M}x{N}x{K}", bf16_out=True)


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(300, 1, 64), (256, 255, 96), (100, 257, 160), (513, 1000, 224),
                                   (64, 300, 32), (1000, 9828, 96)])
def test_qmm_ragged(orc, fmt, M, N, K):
    """N not a multiple of the 256-column pair tile (a masked last tile;
    rows 2 bytes, 8 bytes or 16 bytes apart) and K not a multiple of the
    64-element k-block (the last k-block's codes zero-filled by the TMA, its
    missing scales read as 1.0); 1000 x 9828 takes 512-row pair tiles."""
    need_gpu()
    codes, scales = synth.weights(fmt, N, K, M + N + K, exp_lo=118, exp_hi=132)
    X = synth.activations(M, K, 7 * M + K)
    check_close(run_qmm(fmt, codes, scales, X, N), orc.qmv(fmt, codes, scales, X, M, N, K),
                f"qmm ragged fmt{fmt} {M}x{N}x{K}", bf16_out=True)


def test_qmm_rejects_nvfp4_k_16_mod_32():
    """NVFP4 rows of K = 48 elements are 24 bytes apart: the TMA loads cannot
    take them, MX_EUNSUPPORTED."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    codes, scales = synth.weights(2, 256, 48, 1)
    with pytest.raises(ops.MxError) as ei:
        ops.qmm(2, dev_u8(codes), dev_u8(scales), dev_bf16(synth.activations(8, 48, 2)), 256)
    assert ei.value.status == -2


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_qmm_onehot_rows_exact(orc, fmt):
    """Row m of X is e_{k_m}: Y[m] must be bf16(W[:, k_m]) exactly (every
    decoded weight has at most 6 significant bits, one nonzero product per
    output)."""
    need_gpu()
    M, N, K = 256, 256, 512
    codes, scales = synth.weights(fmt, N, K, 5, exp_lo=110, exp_hi=140)
    ks = np.random.default_rng(1).integers(0, K, size=M)
    X = np.zeros((M, K), dtype=np.uint16)
    X[np.arange(M), ks] = 0x3F80
    Y = run_qmm(fmt, codes, scales, X, N)
    W = orc.dequant(fmt, codes, scales, N, K)
    want = np.array([[orc.bf16(orc.round_bf16(float(v))) for v in W[:, k]] for k in ks])
    assert same_values(Y, want)


def test_qmm_agrees_with_qmv():
    need_gpu()
    from gemm_decode_register_gb300 import ops

    fmt, M, N, K = 0, 256, 512, 2048
    codes, scales = synth.weights(fmt, N, K, 17)
    X = synth.activations(M, K, 18)
    Y = run_qmm(fmt, codes, scales, X, N)
    y = ops.qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(X[:4]), N).cpu().numpy()
    check_close(Y[:4], y.astype(np.float64), "qmm vs qmv", bf16_out=True)


@pytest.mark.parametrize("fmt,N,K,seed", [(0, 28672, 8192, 8), (0, 8192, 28672, 9), (2, 28672, 8192, 10)])
def test_qmm_prefill_full_size(orc, fmt, N, K, seed):
    """M = 4096 prefill shapes, launched as the benchmark launches them;
    three whole output rows against the oracle (NVFP4 too: its tensor scale
    is applied only in the epilogue)."""
    need_gpu()
    M = 4096
    codes, scales = synth.weights(fmt, N, K, seed, exp_lo=118, exp_hi=132)
    X = synth.activations(M, K, 50 + seed)
    Y = run_qmm(fmt, codes, scales, X, N)
    rows = np.array([0, 2049, M - 1])
    ms = np.repeat(rows, N)
    ns = np.tile(np.arange(N), rows.size)
    want = orc.qmm_points(fmt, codes, scales, X, M, N, K, ms, ns).reshape(rows.size, N)
    check_close(Y[rows], want, f"qmm full fmt{fmt} {N}x{K}", bf16_out=True)
    assert np.all(np.isfinite(Y))


def test_qmm_output_alignment_paths():
    """Y 32-byte aligned (the epilogue stores 32 bytes per instruction) and
    Y only 16-byte aligned (16-byte stores): the same bits."""
    need_gpu()
    import torch
    from gemm_decode_register_gb300 import ops

    fmt, M, N, K = 0, 300, 512, 256
    codes, scales = synth.weights(fmt, N, K, 61)
    X = dev_bf16(synth.activations(M, K, 62))
    c, s = dev_u8(codes), dev_u8(scales)
    y_al = ops.qmm(fmt, c, s, X, N)
    big = torch.empty(M * N + 8, dtype=torch.bfloat16, device="cuda")
    y_16 = big[8:].view(M, N)
    assert y_16.data_ptr() % 32 == 16
    ops.qmm(fmt, c, s, X, N, Y=y_16)
    assert torch.equal(y_al.view(torch.int16), y_16.view(torch.int16))
