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


def _bf16_up(bits, n):
    """bf16 bit patterns n steps away from zero (positive finite values)."""
    return (bits.astype(np.int64) + n).astype(np.uint16)


def test_quantize_nvfp4_rounding_boundaries(orc):
    """NVFP4 quotients x / (s g) that land exactly on E2M1 rounding midpoints
    (ties to even) and one bf16 step either side of them: the tensor maximum
    G = 2688 * 2^3 makes g = 8, each block's maximum 6 * g * 2^j makes
    s = 2^j, so x = m * s * g is a bf16 value with an exact quotient m.  Also
    a tensor whose maximum is below 2^-117, where 1 / (s g) overflows fp32.
    Codes and scales bit for bit against the oracle."""
    need_gpu()
    K = 64
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    rows = []
    for j in range(-3, 4):
        d = np.float32(8.0 * 2.0 ** j)
        r = np.zeros(K, np.float32)
        for b in range(K // 16):  # every 16-element block: its maximum first, then the midpoints
            blk = np.concatenate([[6.0 * d], mids * d, -mids * d, [0.0]]).astype(np.float32)
            r[16 * b: 16 * b + 16] = blk[:16]
        rows.append(r)
    x = bf16_of(np.stack(rows))
    # neighbours: every midpoint element moved one bf16 step up, and one down
    up = x.copy()
    dn = x.copy()
    for t in range(x.shape[0]):
        for b in range(K // 16):
            sl = slice(16 * b + 1, 16 * b + 15)
            up[t, sl] = _bf16_up(x[t, sl], 1)
            dn[t, sl] = _bf16_up(x[t, sl], -1)
    g_row = np.zeros((1, K), np.uint16)
    g_row[0, 0] = bf16_of(np.array([[2688.0 * 8.0]], np.float32))[0, 0]  # the tensor maximum G
    x = np.concatenate([x, up, dn, g_row])
    M = x.shape[0]
    c, s = gpu_quantize(2, x, M, K)
    wc, ws = orc.quantize(2, x, M, K)
    assert np.array_equal(s, ws), f"scales differ at {np.flatnonzero(s != ws)[:8]}"
    assert np.array_equal(c, wc), f"codes differ at {np.flatnonzero(c != wc)[:8]}"
    # a tiny tensor: s g below 2^-128
    rng = np.random.default_rng(3)
    t = (rng.standard_normal((4, K)) * 2.0 ** -125).astype(np.float32)
    xt = bf16_of(t)
    c, s = gpu_quantize(2, xt, 4, K)
    wc, ws = orc.quantize(2, xt, 4, K)
    assert np.array_equal(s, ws) and np.array_equal(c, wc)
