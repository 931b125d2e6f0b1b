"""The bounded waits of the tensor-core GEMM (the pages' fault handling: talk
slide 10 "70 Fixes to the ROCm Fork", waits that blocked forever after a
fault now give up and report it).  The test hook withholds every activation
load, a flag that nothing else will set, so the MMA issuer's first wait can
only time out: the pairs must write NaN, set MX_DEVERR_TIMEOUT, drain what
they have in flight and leave the context usable, so that the next normal
call is right."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import bf16_bits_to_f64, bf16_host, check_close, dev_bf16, dev_i32, dev_u8, need_gpu

pytestmark = pytest.mark.gpu

TIMEOUT = 0x2
WAIT_NS = 1_000_000  # 1 ms


def _stalled(fn):
    from gemm_decode_register_gb300 import ops

    ops.device_error()  # clear
    ops.debug_qmm_stall(True, WAIT_NS)
    try:
        out = fn()
        err = ops.device_error()
    finally:
        ops.debug_qmm_stall(False, 0)
    return out, err


@pytest.mark.parametrize("fmt,M,N,K", [(0, 300, 512, 512), (2, 600, 19456, 128), (1, 256, 256, 64)])
def test_qmm_timeout_then_recovers(orc, fmt, M, N, K):
    """256-row pair tiles, 512-row pair tiles (76 column tiles: two
    accumulators per pair), and a single k-block."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    codes, scales = synth.weights(fmt, N, K, M + N)
    X = synth.activations(M, K, K)
    c, s, x = dev_u8(codes), dev_u8(scales), dev_bf16(X).view(M, K)
    Y, err = _stalled(lambda: ops.qmm(fmt, c, s, x, N))
    assert err & TIMEOUT
    assert np.all(np.isnan(bf16_bits_to_f64(bf16_host(Y))))
    Y = ops.qmm(fmt, c, s, x, N)
    assert ops.device_error() == 0
    rows = np.array([0, M // 2, M - 1])
    got = bf16_bits_to_f64(bf16_host(Y))[rows]
    want = orc.qmm_points(fmt, codes, scales, X, M, N, K, np.repeat(rows, N), np.tile(np.arange(N), rows.size))
    check_close(got, want.reshape(rows.size, N), f"qmm after timeout fmt{fmt}", bf16_out=True)


def test_grouped_prefill_timeout_then_recovers(orc):
    need_gpu()
    from gemm_decode_register_gb300 import ops

    fmt, T, E, topk, N, K = 0, 64, 4, 2, 256, 256
    codes, scales = synth.weights(fmt, N, K, 71, E=E)
    x = synth.activations(T, K, 72)
    ids = synth.expert_ids(T, E, topk, 73)
    c, s, xd, idd = dev_u8(codes), dev_u8(scales), dev_bf16(x).view(T, K), dev_i32(ids)
    y, err = _stalled(lambda: ops.moe_qmm(fmt, c, s, xd, idd, E, N))
    assert err & TIMEOUT
    assert np.all(np.isnan(bf16_bits_to_f64(bf16_host(y))))
    y = ops.moe_qmm(fmt, c, s, xd, idd, E, N)
    assert ops.device_error() == 0
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    assert rc == 0
    check_close(bf16_bits_to_f64(bf16_host(y)).reshape(T * topk, N), want.reshape(T * topk, N),
                "grouped after timeout", bf16_out=True)
