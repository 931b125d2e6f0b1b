"""qmv on the GPU against the fp64 oracle (tolerance gate), plus bit-exact
checks that need no tolerance: one-hot activations read decoded weights
back exactly, and power-of-two / sign invariances hold bit for bit."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import check_close, dev_bf16, dev_u8, need_gpu, same_values

pytestmark = pytest.mark.gpu


def run_qmv(fmt, codes, scales, x, N):
    from gemm_decode_register_gb300 import ops

    y = ops.qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x), N)
    return y.cpu().numpy()


def test_config0_full(orc):
    """MXFP4, M=1, N=2048, K=2048, E8M0 exponents in [120, 130], seed 0."""
    need_gpu()
    fmt, M, N, K = synth.FMT_MXFP4, 1, 2048, 2048
    codes, scales = synth.weights(fmt, N, K, 0, exp_lo=120, exp_hi=130)
    x = synth.activations(M, K, 1000)
    check_close(run_qmv(fmt, codes, scales, x, N), orc.qmv(fmt, codes, scales, x, M, N, K), "C0")


CASES = []
for fmt in (0, 1, 2):
    for M in (1, 2, 3, 4, 5, 8, 9, 12):
        CASES.append((fmt, M, 67, 320))        # ragged N (tiles of 2*MC rows)
    CASES += [(fmt, 1, 1000, 4096), (fmt, 4, 513, 2048), (fmt, 8, 129, 1056)]
CASES += [(2, 1, 33, 48), (2, 4, 31, 16), (2, 3, 70, 1040)]   # NVFP4 with K % 32 == 16
# streamed shapes whose CTAs deal equal runs of stages to their warps, cutting
# tiles where runs meet (M=1: 13-14 tiles of 4 stages per CTA; M=2: 4-5 tiles)
CASES += [(fmt, 1, 4096, 8192) for fmt in (0, 1, 2)] + [(fmt, 2, 3000, 4096) for fmt in (0, 2)]
# more tokens than one pass of 8 (speculative-decode verify sizes): 2 and 3
# passes over the weights
CASES += [(0, 16, 300, 1024), (1, 13, 67, 320), (2, 24, 130, 512), (0, 6, 1000, 4096)]


# activations staged through shared memory: more than 8 chunks of 8
# elements per thread (3-4 rows share 512 threads as 4 rows of 128 threads;
# K = 10240 is 1280 chunks per row, one K window), so the raw bf16 chunks are
# parked in the staging buffer and converted there in place (NVFP4: whole
# units, its permuted layout)
STAGED_IN_SMEM = [(fmt, M, 150, 10240) for fmt in (0, 1, 2) for M in (3, 4)]


@pytest.mark.parametrize("fmt,M,N,K", STAGED_IN_SMEM)
def test_qmv_staging_in_shared_memory(orc, fmt, M, N, K):
    need_gpu()
    codes, scales = synth.weights(fmt, N, K, 30 + M, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 40 + M)
    check_close(run_qmv(fmt, codes, scales, x, N), orc.qmv(fmt, codes, scales, x, M, N, K),
                f"fmt{fmt} M{M} N{N} K{K} (staging in shared memory)")


# long rows: the tokens' activations span tens of K windows (a 2-D grid of
# tile groups x windows, partial sums through the workspace)
@pytest.mark.parametrize("fmt,M,N,K", [(0, 8, 40, 262144), (2, 3, 70, 131072), (0, 8, 16, 1 << 20), (1, 4, 16, 1 << 20),
                                       (2, 2, 24, 1 << 20), (0, 1, 24, 1 << 20)])
def test_qmv_many_k_windows(orc, fmt, M, N, K):
    need_gpu()
    codes, scales = synth.weights(fmt, N, K, 60 + M, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 70 + M)
    check_close(run_qmv(fmt, codes, scales, x, N), orc.qmv(fmt, codes, scales, x, M, N, K),
                f"fmt{fmt} M{M} N{N} K{K} (many K windows)")


def test_qmv_windows_beyond_the_workspace(orc):
    """8 tokens of rows of 2^20 elements and 3456 weight rows (1.8 GB of
    codes, drawn on the device): the K windows' partial sums of one group
    exceed the stream's 16 MiB workspace and the row is too long for the
    direct-load kernel, so the group runs as two groups of 4; checked on 64
    sampled weight rows."""
    need_gpu()
    import torch
    from gemm_decode_register_gb300 import ops

    fmt, M, N, K = 0, 8, 3456, 1 << 20
    dev = torch.device("cuda")
    c, sc = synth.weights_device(fmt, N, K, 77, dev, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 78)
    y = ops.qmv(fmt, c, sc, dev_bf16(x).view(M, K), N).cpu().numpy()
    rng = np.random.default_rng(79)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(N - 16, N), rng.integers(0, N, 32)]))
    sub_c = c.view(N, K // 2)[torch.from_numpy(rows).cuda()].cpu().numpy().reshape(-1)
    sub_s = sc.view(N, K // 32)[torch.from_numpy(rows).cuda()].cpu().numpy().reshape(-1)
    want = orc.qmv(fmt, sub_c, sub_s, x, M, rows.size, K)
    check_close(y[:, rows], want, "8 x 3456 x 2^20 (groups split for the workspace)")
    del c, sc


@pytest.mark.parametrize("fmt,M,N,K", CASES)
def test_qmv_parity(orc, fmt, M, N, K):
    need_gpu()
    codes, scales = synth.weights(fmt, N, K, 10 + M, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 20 + M)
    check_close(run_qmv(fmt, codes, scales, x, N), orc.qmv(fmt, codes, scales, x, M, N, K),
                f"fmt{fmt} M{M} N{N} K{K}")


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_onehot_reads_decoded_weights_exactly(orc, fmt, M):
    need_gpu()
    N, K = 48, 256
    codes, scales = synth.weights(fmt, N, K, 3, exp_lo=110, exp_hi=140)
    rng = np.random.default_rng(M)
    ks = rng.choice(K, size=M, replace=False)
    x = np.zeros((M, K), dtype=np.uint16)
    x[np.arange(M), ks] = 0x3F80  # 1.0
    y = run_qmv(fmt, codes, scales, x, N)
    W = orc.dequant(fmt, codes, scales, N, K)
    assert same_values(y, W[:, ks].T)


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M", [1, 4])
def test_invariants_bit_exact(fmt, M):
    need_gpu()
    N, K = 96, 1024
    codes, scales = synth.weights(fmt, N, K, 5, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 6)
    y = run_qmv(fmt, codes, scales, x, N)
    if fmt == synth.FMT_NVFP4:
        s2 = scales.copy()
        s2[-4:] = (s2[-4:].view("<f4") * np.float32(2)).view(np.uint8)
    else:
        s2 = (scales.astype(np.int64) + 1).astype(np.uint8)
    assert np.array_equal(run_qmv(fmt, codes, s2, x, N), 2 * y)
    flip = np.uint8(0x80 if fmt == synth.FMT_MXFP8 else 0x88)
    assert np.array_equal(run_qmv(fmt, codes ^ flip, scales, x, N), -y)
    assert np.array_equal(run_qmv(fmt, codes, scales, x ^ np.uint16(0x8000), N), -y)
    assert np.all(run_qmv(fmt, np.zeros_like(codes), scales, x, N) == 0)


@pytest.mark.parametrize("fmt,N,K", [(0, 10240, 8192), (0, 57344, 8192), (0, 8192, 28672),
                                     (1, 57344, 8192), (2, 57344, 8192)])
@pytest.mark.parametrize("M", [1, 4])
def test_full_size_sampled_rows(orc, fmt, N, K, M):
    """The decode-projection and format-sweep shapes at full size, in the
    launch configuration the benchmark times; 64 sampled rows (first,
    last and random) against the oracle."""
    need_gpu()
    seed = {(10240, 8192): 1, (57344, 8192): 2, (8192, 28672): 3}[(N, K)] + 5 * fmt
    codes, scales = synth.weights(fmt, N, K, seed, exp_lo=118, exp_hi=132)
    x = synth.activations(M, K, 100 + seed)
    y = run_qmv(fmt, codes, scales, x, N)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(seed).choice(N, 62)]))
    want = orc.qmv_rows(fmt, codes, scales, x, M, N, K, rows)
    check_close(y[:, rows], want, f"full fmt{fmt} {N}x{K} M{M}")
