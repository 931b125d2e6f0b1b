"""Fused MoE FFN kernels on the GPU: mx_moe_gate_up_swiglu (gate and up
rows of each routed expert with the SwiGLU in the epilogue) and
mx_moe_down_combine (down rows with the router-weighted sum over a token's
slots), against the oracle chain and against the unfused GPU path."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import (bf16_bits_to_f64, bf16_host, bf16_ulp_diff, check_close, dev_bf16, dev_i32, dev_u8,
                      need_gpu)

pytestmark = pytest.mark.gpu


def fused_gate_up(fmt, codes, scales, x, ids, E, I):
    from gemm_decode_register_gb300 import ops

    return ops.moe_gate_up_swiglu(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x), dev_i32(ids), E, I)


def fused_down(fmt, codes, scales, h, ids, r, E, N):
    import torch
    from gemm_decode_register_gb300 import ops

    hd = h if isinstance(h, torch.Tensor) else dev_bf16(h)
    return ops.moe_down_combine(fmt, dev_u8(codes), dev_u8(scales), hd.reshape(-1, hd.shape[-1]).contiguous(),
                                dev_i32(ids), torch.from_numpy(np.ascontiguousarray(r, np.float32)).cuda(), E, N)


def oracle_h(orc, fmt, codes, scales, x, ids, T, E, topk, I, K):
    gu, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, 2 * I, K)
    assert rc == 0
    return orc.swiglu_bf16(gu.reshape(T * topk, 2 * I), I)


def oracle_out(orc, fmt, codes, scales, h_bits, ids, r, T, E, topk, N, K):
    yd, rc = orc.moe_qmv(fmt, codes, scales, h_bits, ids.reshape(-1, 1), T * topk, E, 1, N, K)
    assert rc == 0
    return orc.moe_combine(yd.reshape(T * topk, N), r, T, topk, N)


@pytest.mark.parametrize("T", [1, 4])
def test_gate_up_swiglu_config(orc, T):
    """128 experts, top-8, hidden 2048, intermediate 768: h against the
    oracle (gate/up in fp64, SwiGLU rounded to bf16) within the gate for
    bf16 outputs, and against the unfused GPU path (mx_moe_qmv, then
    mx_swiglu) to within one bf16 ulp."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    fmt, E, topk, H, I = 0, 128, 8, 2048, 768
    codes, scales = synth.weights(fmt, 2 * I, H, 90, E=E)
    x = synth.activations(T, H, 91 + T)
    ids = synth.expert_ids(T, E, topk, 92 + T)
    h = fused_gate_up(fmt, codes, scales, x, ids, E, I)
    hb = bf16_host(h).reshape(T * topk, I)
    want = oracle_h(orc, fmt, codes, scales, x, ids, T, E, topk, I, H)
    check_close(bf16_bits_to_f64(hb), bf16_bits_to_f64(want), f"gate-up swiglu T{T}", bf16_out=True)
    gu = ops.moe_qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x), dev_i32(ids), E, 2 * I)
    h2 = bf16_host(ops.swiglu(gu, I)).reshape(T * topk, I)
    assert bf16_ulp_diff(hb, h2).max() <= 1


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("T,E,topk,I,K", [(3, 5, 2, 37, 256), (9, 4, 3, 64, 128), (2, 7, 7, 19, 384),
                                         (12, 6, 4, 24, 128)])
def test_gate_up_swiglu_ragged(orc, fmt, T, E, topk, I, K):
    """Experts shared across tokens (groups above one slot, groups split at
    eight), intermediate sizes that leave the last gate/up tile partly
    empty, and more than 32 slots (block-wide routing)."""
    need_gpu()
    codes, scales = synth.weights(fmt, 2 * I, K, T + E + I, E=E)
    x = synth.activations(T, K, 5 * T)
    ids = synth.expert_ids(T, E, topk, 6 * T)
    hb = bf16_host(fused_gate_up(fmt, codes, scales, x, ids, E, I)).reshape(T * topk, I)
    want = oracle_h(orc, fmt, codes, scales, x, ids, T, E, topk, I, K)
    check_close(bf16_bits_to_f64(hb), bf16_bits_to_f64(want), f"gate-up fmt{fmt}", bf16_out=True)


@pytest.mark.parametrize("T", [1, 4])
def test_down_combine_config(orc, T):
    """down 2048 x 768 over the routed experts, router-weighted sum: against
    the oracle (fp64 products and sum) and against the unfused GPU path
    (mx_moe_qmv per slot, then mx_moe_combine)."""
    need_gpu()
    import torch
    from gemm_decode_register_gb300 import ops

    fmt, E, topk, H, I = 0, 128, 8, 2048, 768
    codes, scales = synth.weights(fmt, H, I, 93, E=E)
    h = synth.activations(T * topk, I, 94 + T)
    ids = synth.expert_ids(T, E, topk, 95 + T)
    r = synth.router_weights(T, topk, 96 + T)
    out = fused_down(fmt, codes, scales, h, ids, r, E, H).cpu().numpy()
    want = oracle_out(orc, fmt, codes, scales, h, ids, r, T, E, topk, H, I)
    check_close(out, want, f"down combine T{T}")
    yd = ops.moe_qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(h), dev_i32(ids.reshape(-1, 1)), E, H)
    out2 = ops.moe_combine(yd, torch.from_numpy(r).cuda()).cpu().numpy()
    check_close(out, out2.astype(np.float64), f"down combine vs unfused T{T}")


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("T,E,topk,N,K", [(3, 5, 2, 37, 128), (9, 4, 3, 70, 256), (5, 6, 6, 19, 128),
                                         (12, 6, 4, 33, 128)])
def test_down_combine_ragged(orc, fmt, T, E, topk, N, K):
    need_gpu()
    codes, scales = synth.weights(fmt, N, K, T + E + N, E=E)
    h = synth.activations(T * topk, K, 7 * T)
    ids = synth.expert_ids(T, E, topk, 8 * T)
    r = synth.router_weights(T, topk, 9 * T)
    out = fused_down(fmt, codes, scales, h, ids, r, E, N).cpu().numpy()
    want = oracle_out(orc, fmt, codes, scales, h, ids, r, T, E, topk, N, K)
    check_close(out, want, f"down combine fmt{fmt}")


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_down_combine_rows_in_passes(orc, fmt):
    """48 activation rows (12 tokens x top-4) of K = 768: the staging covers
    them in three passes of 16 rows with 32 threads per row, nine chunks per
    thread, so through shared memory."""
    need_gpu()
    T, E, topk, N, K = 12, 6, 4, 72, 768
    codes, scales = synth.weights(fmt, N, K, 51 + fmt, E=E)
    h = synth.activations(T * topk, K, 52)
    ids = synth.expert_ids(T, E, topk, 53)
    r = synth.router_weights(T, topk, 54)
    out = fused_down(fmt, codes, scales, h, ids, r, E, N).cpu().numpy()
    want = oracle_out(orc, fmt, codes, scales, h, ids, r, T, E, topk, N, K)
    check_close(out, want, f"down combine fmt{fmt} (rows in passes)")


def test_down_combine_workspace_path(orc):
    """Row tiles whose partial sums do not fit in a CTA's shared memory next
    to its ring (8 tokens x top-8, 57344 rows: 24 tiles of 16 rows per CTA)
    take the device-workspace combine instead of the CTA-local one; the sum
    is the same slot-order one."""
    need_gpu()
    fmt, E, topk, T, N, K = 0, 8, 8, 8, 57344, 128
    codes, scales = synth.weights(fmt, N, K, 41, E=E)
    h = synth.activations(T * topk, K, 42)
    ids = synth.expert_ids(T, E, topk, 43)
    r = synth.router_weights(T, topk, 44)
    out = fused_down(fmt, codes, scales, h, ids, r, E, N).cpu().numpy()
    # the oracle on 512 sampled rows (tile edges, the last tile, random rows) of every expert
    rng = np.random.default_rng(45)
    rows = np.unique(np.concatenate([np.arange(0, 40), np.arange(N - 40, N), rng.integers(0, N, 432)]))
    rb, sb = K // 2, K // 32
    sub_c = codes.reshape(E, N, rb)[:, rows].reshape(-1)
    sub_s = scales.reshape(E, N, sb)[:, rows].reshape(-1)
    want = oracle_out(orc, fmt, sub_c, sub_s, h, ids, r, T, E, topk, rows.size, K)
    check_close(out[:, rows], want, "down combine through the workspace")


def test_down_combine_deterministic():
    """The partial sums are combined in slot order by whichever warp closes a
    tile: repeated calls give the same bits."""
    need_gpu()
    fmt, E, topk, T, N, K = 0, 16, 4, 4, 512, 256
    codes, scales = synth.weights(fmt, N, K, 31, E=E)
    h = synth.activations(T * topk, K, 32)
    ids = synth.expert_ids(T, E, topk, 33)
    r = synth.router_weights(T, topk, 34)
    a = fused_down(fmt, codes, scales, h, ids, r, E, N).cpu().numpy()
    for _ in range(3):
        b = fused_down(fmt, codes, scales, h, ids, r, E, N).cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("T", [1, 4])
def test_fused_ffn_composite(orc, T):
    """The two fused kernels chained (the MoE FFN in two launches) against
    the oracle chain."""
    need_gpu()
    fmt, E, topk, H, I = 0, 128, 8, 2048, 768
    c1, s1 = synth.weights(fmt, 2 * I, H, 80, E=E)
    c2, s2 = synth.weights(fmt, H, I, 81, E=E)
    x = synth.activations(T, H, 82 + T)
    ids = synth.expert_ids(T, E, topk, 83 + T)
    r = synth.router_weights(T, topk, 84 + T)
    h = fused_gate_up(fmt, c1, s1, x, ids, E, I)
    out = fused_down(fmt, c2, s2, h, ids, r, E, H).cpu().numpy()
    h_o = oracle_h(orc, fmt, c1, s1, x, ids, T, E, topk, I, H)
    out_o = oracle_out(orc, fmt, c2, s2, h_o, ids, r, T, E, topk, H, I)
    check_close(out, out_o, f"fused moe ffn T{T}")


def test_fused_bad_expert_ids(orc):
    """An id outside [0, E): the gate-up kernel writes NaN for that slot's
    h row, the down kernel NaN for that token's outputs; the other slots and
    tokens are unaffected and the device error word records it."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    ops.device_error()  # clear
    fmt, T, E, topk, I, K, N = 0, 3, 6, 2, 40, 128, 64
    c1, s1 = synth.weights(fmt, 2 * I, K, 41, E=E)
    x = synth.activations(T, K, 42)
    ids = synth.expert_ids(T, E, topk, 43)
    ids[1, 0] = E + 3
    hb = bf16_host(fused_gate_up(fmt, c1, s1, x, ids, E, I)).reshape(T * topk, I)
    assert ops.device_error() & 0x1
    assert np.all(np.isnan(bf16_bits_to_f64(hb[1 * topk + 0])))
    good = np.ones(T * topk, bool)
    good[1 * topk + 0] = False
    ids_ok = ids.copy()
    ids_ok[1, 0] = 0
    want = oracle_h(orc, fmt, c1, s1, x, ids_ok, T, E, topk, I, K)
    check_close(bf16_bits_to_f64(hb[good]), bf16_bits_to_f64(want[good]), "gate-up good slots", bf16_out=True)

    c2, s2 = synth.weights(fmt, N, K, 44, E=E)
    h = synth.activations(T * topk, K, 45)
    r = synth.router_weights(T, topk, 46)
    out = fused_down(fmt, c2, s2, h, ids, r, E, N).cpu().numpy()
    assert ops.device_error() & 0x1
    assert np.all(np.isnan(out[1]))
    want = oracle_out(orc, fmt, c2, s2, h, ids_ok, r, T, E, topk, N, K)
    check_close(out[[0, 2]], want[[0, 2]], "down good tokens")
    # every id bad: no work group at all, every output NaN
    bad = np.full((T, topk), -1, np.int32)
    out = fused_down(fmt, c2, s2, h, bad, r, E, N).cpu().numpy()
    assert ops.device_error() & 0x1
    assert np.all(np.isnan(out))


@pytest.mark.parametrize("fmt,K", [(0, 96), (1, 160), (2, 48), (2, 336)])
def test_fused_k_not_multiple_of_128(orc, fmt, K):
    """Rows that are not 128-element aligned: the direct-load MoE kernel
    through the workspace, then the glue (SwiGLU; router combine), against
    the oracle chain."""
    need_gpu()
    T, E, topk, I, N = 3, 6, 2, 40, 72
    c1, s1 = synth.weights(fmt, 2 * I, K, 47 + K, E=E)
    x = synth.activations(T, K, 48)
    ids = synth.expert_ids(T, E, topk, 49)
    hb = bf16_host(fused_gate_up(fmt, c1, s1, x, ids, E, I)).reshape(T * topk, I)
    want = oracle_h(orc, fmt, c1, s1, x, ids, T, E, topk, I, K)
    check_close(bf16_bits_to_f64(hb), bf16_bits_to_f64(want), f"gate-up K{K} fmt{fmt}", bf16_out=True)
    c2, s2 = synth.weights(fmt, N, K, 50 + K, E=E)
    h = synth.activations(T * topk, K, 51)
    r = synth.router_weights(T, topk, 52)
    out = fused_down(fmt, c2, s2, h, ids, r, E, N).cpu().numpy()
    check_close(out, oracle_out(orc, fmt, c2, s2, h, ids, r, T, E, topk, N, K), f"down-combine K{K} fmt{fmt}")



@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("T,K", [(1, 65536), (2, 49152)])
def test_gate_up_swiglu_rows_beyond_the_ring(orc, fmt, T, K):
    """Rows of x too long to stage beside the streaming kernel's weight ring
    (65536 elements of one token, 49152 of two: more than 227 KB together)
    run through the direct-load kernel and the SwiGLU glue; h is the same
    bf16 rounding of the same products."""
    need_gpu()
    E, topk, I = 4, 2, 40
    codes, scales = synth.weights(fmt, 2 * I, K, 61 + fmt, E=E)
    x = synth.activations(T, K, 62 + T)
    ids = synth.expert_ids(T, E, topk, 63 + T)
    hb = bf16_host(fused_gate_up(fmt, codes, scales, x, ids, E, I)).reshape(T * topk, I)
    want = oracle_h(orc, fmt, codes, scales, x, ids, T, E, topk, I, K)
    check_close(bf16_bits_to_f64(hb), bf16_bits_to_f64(want), f"gate-up fmt{fmt} K{K}", bf16_out=True)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_down_combine_rows_beyond_the_ring(orc, fmt):
    """Four rows of h (2 tokens x top-2) of 16384 elements do not fit beside
    the streaming kernel's ring: per-slot products from the direct-load
    kernel, then the slot-order router combine."""
    need_gpu()
    T, E, topk, N, K = 2, 5, 2, 37, 16384
    codes, scales = synth.weights(fmt, N, K, 71 + fmt, E=E)
    h = synth.activations(T * topk, K, 72)
    ids = synth.expert_ids(T, E, topk, 73)
    r = synth.router_weights(T, topk, 74)
    out = fused_down(fmt, codes, scales, h, ids, r, E, N).cpu().numpy()
    want = oracle_out(orc, fmt, codes, scales, h, ids, r, T, E, topk, N, K)
    check_close(out, want, f"down combine fmt{fmt} K{K}")
