"""MoE decode GEMV on the GPU against the oracle: the 128-expert top-8
workload (gate+up 1536x2048, down 2048x768, T = 1 and 4), ragged shapes,
the E = 1 reduction to qmv, bad expert ids, and the full MoE FFN
(gate-up, SwiGLU, down, router combine)."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import (bf16_bits_to_f64, bf16_host, bf16_ulp_diff, check_close, dev_bf16, dev_i32, dev_u8,
                      need_gpu, same_values)

pytestmark = pytest.mark.gpu


def run_moe(fmt, codes, scales, x, ids, E, N):
    from gemm_decode_register_gb300 import ops

    y = ops.moe_qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x), dev_i32(ids), E, N)
    return y.cpu().numpy()


@pytest.mark.parametrize("T", [1, 4])
@pytest.mark.parametrize("proj", ["gate_up", "down"])
def test_moe_config(orc, T, proj):
    need_gpu()
    fmt, E, topk = synth.FMT_MXFP4, 128, 8
    N, K = (1536, 2048) if proj == "gate_up" else (2048, 768)
    codes, scales = synth.weights(fmt, N, K, 40 + (proj == "down"), E=E, exp_lo=118, exp_hi=132)
    ids = synth.expert_ids(T, E, topk, 50 + T)
    if proj == "gate_up":
        x = synth.activations(T, K, 60 + T)
        y = run_moe(fmt, codes, scales, x, ids, E, N)
        want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    else:
        x = synth.activations(T * topk, K, 70 + T)
        ids1 = ids.reshape(-1, 1)
        y = run_moe(fmt, codes, scales, x, ids1, E, N)
        want, rc = orc.moe_qmv(fmt, codes, scales, x, ids1, T * topk, E, 1, N, K)
    assert rc == 0
    check_close(y.reshape(-1, N), want.reshape(-1, N), f"moe {proj} T{T}")


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("T,E,topk,N,K", [(3, 5, 2, 37, 96), (9, 4, 3, 70, 64), (2, 7, 7, 19, 160),
                                         (16, 2, 1, 33, 32)])
def test_moe_ragged(orc, fmt, T, E, topk, N, K):
    """Shared experts across tokens, groups above 8 slots, ragged N."""
    need_gpu()
    codes, scales = synth.weights(fmt, N, K, T + E, E=E, exp_lo=118, exp_hi=132)
    x = synth.activations(T, K, 3 * T)
    ids = synth.expert_ids(T, E, topk, 4 * T)
    y = run_moe(fmt, codes, scales, x, ids, E, N)
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    check_close(y.reshape(-1, N), want.reshape(-1, N), f"moe ragged fmt{fmt}")


@pytest.mark.parametrize("fmt", [0, 2])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_moe_single_expert_equals_qmv(orc, fmt, T):
    """E = 1, topk = 1: every token routes to the one expert, so MoE reduces
    to qmv.  The two kernels may split K differently (qmv spreads a tile's K
    over several warps), so they agree within the tolerance gate, and both
    match the oracle."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    N, K = 200, 512
    codes, scales = synth.weights(fmt, N, K, 9)
    x = synth.activations(T, K, 10)
    y_moe = run_moe(fmt, codes, scales, x, np.zeros((T, 1), np.int32), 1, N).reshape(T, N)
    y_qmv = ops.qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x), N).cpu().numpy()
    want = orc.qmv(fmt, codes, scales, x, T, N, K)
    check_close(y_moe, y_qmv.astype(np.float64), "moe vs qmv")
    check_close(y_moe, want, "moe vs oracle")


def test_moe_bad_expert_id(orc):
    need_gpu()
    from gemm_decode_register_gb300 import ops

    ops.device_error()  # clear
    fmt, T, E, topk, N, K = 0, 2, 6, 3, 40, 64
    codes, scales = synth.weights(fmt, N, K, 11, E=E)
    x = synth.activations(T, K, 12)
    ids = synth.expert_ids(T, E, topk, 13)
    ids[1, 2] = E
    ids[0, 1] = -1
    y = run_moe(fmt, codes, scales, x, ids, E, N)
    assert ops.device_error() & 0x1
    assert ops.device_error() == 0  # cleared
    assert np.all(np.isnan(y[1, 2])) and np.all(np.isnan(y[0, 1]))
    good = np.ones((T, topk), bool)
    good[1, 2] = good[0, 1] = False
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    assert rc == -3
    check_close(y[good], want[good], "moe good slots")


@pytest.mark.parametrize("T", [1, 4])
def test_moe_ffn_composite(orc, T):
    """gate+up (N=1536 = 768 gate rows then 768 up rows) -> SwiGLU -> down
    (N=2048, K=768) -> router-weighted combine, against the oracle chain
    (fp64 throughout, h rounded to bf16 as the GPU does)."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    fmt, E, topk, H, I = 0, 128, 8, 2048, 768
    c1, s1 = synth.weights(fmt, 2 * I, H, 80, E=E)
    c2, s2 = synth.weights(fmt, H, I, 81, E=E)
    x = synth.activations(T, H, 82 + T)
    ids = synth.expert_ids(T, E, topk, 83 + T)
    r = synth.router_weights(T, topk, 84 + T)
    import torch

    d_ids = dev_i32(ids)
    gu = ops.moe_qmv(fmt, dev_u8(c1), dev_u8(s1), dev_bf16(x), d_ids, E, 2 * I)
    h = ops.swiglu(gu, I)
    yd = ops.moe_qmv(fmt, dev_u8(c2), dev_u8(s2), h, d_ids.reshape(-1, 1).contiguous(), E, H)
    out = ops.moe_combine(yd, torch.from_numpy(r).cuda()).cpu().numpy()

    gu_o, _ = orc.moe_qmv(fmt, c1, s1, x, ids, T, E, topk, 2 * I, H)
    h_o = orc.swiglu_bf16(gu_o.reshape(T * topk, 2 * I), I)
    yd_o, _ = orc.moe_qmv(fmt, c2, s2, h_o, ids.reshape(-1, 1), T * topk, E, 1, H, I)
    out_o = orc.moe_combine(yd_o.reshape(T * topk, H), r, T, topk, H)
    check_close(out, out_o, f"moe ffn T{T}")
    # SwiGLU alone on the GPU's own gate/up output: bf16 within one ulp
    # wherever the value is not vanishingly small (fp32 exp underflows near
    # 2^-126, where the oracle's fp64 still resolves digits)
    h_chk = orc.swiglu_bf16(gu.cpu().numpy().astype(np.float64).reshape(T * topk, 2 * I), I)
    hb = bf16_host(h)
    big = np.abs(bf16_bits_to_f64(h_chk)) >= 2.0 ** -100
    diff = bf16_ulp_diff(hb, h_chk)[big]
    assert diff.max() <= 1
    assert np.all(np.abs(bf16_bits_to_f64(hb[~big])) < 2.0 ** -99)


def test_combine_exact_one_hot_router():
    need_gpu()
    import torch
    from gemm_decode_register_gb300 import ops

    T, topk, N = 3, 4, 50
    yd = torch.randn(T * topk, N, device="cuda")
    r = torch.zeros(T, topk, device="cuda")
    r[:, 2] = 1.0
    out = ops.moe_combine(yd, r)
    assert same_values(out.cpu().numpy(), yd.reshape(T, topk, N)[:, 2].cpu().numpy())
