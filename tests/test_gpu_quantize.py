"""On-device block-float quantisation (mx_quantize) against the oracle:
codes and scales must match bit for bit (the quantised code is an integer
decided by the same fp32 steps on both sides)."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import dev_bf16, need_gpu

pytestmark = pytest.mark.gpu


def bf16_of(f):
    """bf16 bits (nearest-even) of float32 values, through torch."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(f, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def gpu_quantize(fmt, x_bits, M, K):
    from gemm_decode_register_gb300 import ops

    c, s = ops.quantize(fmt, dev_bf16(x_bits).view(M, K))
    return c.cpu().numpy(), s.cpu().numpy()


def wide_range(M, K, seed):
    rng = np.random.default_rng(seed)
    f = rng.standard_normal((M, K)).astype(np.float32) * np.exp2(rng.integers(-40, 40, size=(M, 1))).astype(np.float32)
    return bf16_of(f)


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("M,K,seed", [(1, 32, 1), (7, 96, 2), (64, 2048, 3), (300, 1024, 4), (33, 4096, 5)])
def test_quantize_matches_oracle(orc, fmt, M, K, seed):
    need_gpu()
    if K % synth.block_of(fmt):
        pytest.skip("K not a multiple of the block")
    x = wide_range(M, K, seed) if seed % 2 else synth.activations(M, K, seed)
    c, s = gpu_quantize(fmt, x, M, K)
    wc, ws = orc.quantize(fmt, x, M, K)
    assert np.array_equal(s, ws), f"scales differ at {np.flatnonzero(s != ws)[:8]}"
    assert np.array_equal(c, wc), f"codes differ at {np.flatnonzero(c != wc)[:8]}"


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_quantize_special_values(orc, fmt):
    """Ties, saturation, signed zeros, bf16 subnormals, huge values, NaN and
    infinities, all-zero blocks: the same codes and scales as the oracle."""
    need_gpu()
    K = 64
    rows = []
    r = np.zeros(K, np.float32)
    r[:10] = [4.0, 0.25, 0.75, 2.5, 3.5, -5.0, -0.0, -0.1, 7.5, -7.0]
    rows.append(r)
    rows.append(np.zeros(K, np.float32))                       # all zero
    r = np.full(K, -0.0, np.float32); r[3] = 1e-40; rows.append(r)  # -0 and a subnormal
    r = np.linspace(-3e38, 3e38, K, dtype=np.float32); rows.append(r)  # near the bf16 maximum
    r = np.ones(K, np.float32); r[5] = np.nan; rows.append(r)
    r = np.ones(K, np.float32); r[40] = np.inf; rows.append(r)
    r = np.ones(K, np.float32) * 2.0 ** -130; r[1] = 2.0 ** -133; rows.append(r)  # all subnormal
    r = np.array([448.0, 500.0, 300.0, -2.0 ** -9] + [1.0] * (K - 4), np.float32); rows.append(r)
    x = bf16_of(np.stack(rows))
    M = x.shape[0]
    c, s = gpu_quantize(fmt, x, M, K)
    wc, ws = orc.quantize(fmt, x, M, K)
    assert np.array_equal(s, ws), f"scales differ at {np.flatnonzero(s != ws)[:8]}: {s[s != ws][:8]} vs {ws[s != ws][:8]}"
    assert np.array_equal(c, wc), f"codes differ at {np.flatnonzero(c != wc)[:8]}: {c[c != wc][:8]} vs {wc[c != wc][:8]}"


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_quantize_full_size_sampled_rows(orc, fmt):
    """4096 x 8192 activations (the prefill X): every code and scale of 8
    sampled rows against the oracle; for NVFP4 the sample includes the row
    that holds the tensor maximum, so the oracle's tensor scale is the
    tensor's."""
    need_gpu()
    M, K = 4096, 8192
    x = synth.activations(M, K, 7)
    c, s = gpu_quantize(fmt, x, M, K)
    blk = synth.block_of(fmt)
    cpr = K if fmt == 1 else K // 2
    rows = [0, 1, 1000, 2047, 3333, M - 1]
    if fmt == 2:
        f = np.abs((x.astype(np.uint32) << 16).view(np.float32))
        rows.append(int(np.argmax(f.max(axis=1))))
    rows = sorted(set(rows))
    wc, ws = orc.quantize(fmt, x[rows], len(rows), K)
    for i, m in enumerate(rows):
        assert np.array_equal(s[m * (K // blk):(m + 1) * (K // blk)], ws[i * (K // blk):(i + 1) * (K // blk)]), m
        assert np.array_equal(c[m * cpr:(m + 1) * cpr], wc[i * cpr:(i + 1) * cpr]), m
    if fmt == 2:
        assert np.array_equal(s[M * K // 16:], ws[len(rows) * K // 16:])  # tensor scale


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_quantized_weights_feed_qmv(orc, fmt):
    """A bf16 weight matrix quantised on the device and used by mx_qmv: the
    codes equal the oracle's, and the GEMV over them passes the tolerance
    gate against the oracle's GEMV over the oracle's codes."""
    need_gpu()
    from gemm_decode_register_gb300 import ops
    from gpu_util import check_close

    N, K, M = 256, 1024, 2
    w = synth.activations(N, K, 8)
    c, s = ops.quantize(fmt, dev_bf16(w).view(N, K))
    wc, ws = orc.quantize(fmt, w, N, K)
    assert np.array_equal(c.cpu().numpy(), wc) and np.array_equal(s.cpu().numpy(), ws)
    x = synth.activations(M, K, 9)
    y = ops.qmv(fmt, c, s, dev_bf16(x).view(M, K), N).cpu().numpy()
    check_close(y, orc.qmv(fmt, wc, ws, x, M, N, K), f"qmv over quantised fmt{fmt}")
