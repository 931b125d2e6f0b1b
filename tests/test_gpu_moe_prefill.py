"""Expert-batched MoE prefill on the GPU: mx_moe_qmm (routed rows grouped by
expert, one tensor-core GEMM per group tile of up to 512 rows, outputs in slot order)
and mx_moe_ffn_prefill (gate-up with the SwiGLU in the GEMM epilogue, down,
router-weighted combine), against the oracle."""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import bf16_bits_to_f64, bf16_host, check_close, dev_bf16, dev_i32, dev_u8, need_gpu

pytestmark = pytest.mark.gpu


def run_moe_qmm(fmt, codes, scales, x, ids, E, N, **kw):
    from gemm_decode_register_gb300 import ops

    return ops.moe_qmm(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x), dev_i32(ids), E, N, **kw)


def oracle_ffn(orc, fmt, c1, s1, c2, s2, x, ids, r, T, E, topk, H, I):
    """The FFN as the ABI defines it: h rounded to bf16 (oracle SwiGLU), the
    down outputs rounded to bf16, then the fp64 router-weighted sum."""
    gu, rc = orc.moe_qmv(fmt, c1, s1, x, ids, T, E, topk, 2 * I, H)
    assert rc == 0
    h = orc.swiglu_bf16(gu.reshape(T * topk, 2 * I), I)
    yd, rc = orc.moe_qmv(fmt, c2, s2, h, ids.reshape(-1, 1), T * topk, E, 1, H, I)
    assert rc == 0
    yd_b = np.array([orc.bf16(orc.round_bf16(float(v))) for v in yd.reshape(-1)]).reshape(T * topk, H)
    return orc.moe_combine(yd_b, r, T, topk, H)


CASES = []
for fmt in (0, 1, 2):
    CASES += [
        (fmt, 40, 6, 3, 256, 128),   # ~20 rows per expert: one partial group tile each
        (fmt, 300, 4, 2, 512, 192),  # ~150 rows per expert, two column tiles, 3 k-blocks
        (fmt, 700, 3, 2, 256, 64),   # ~470 rows per expert: one tile using both 256-row halves
        (fmt, 1, 8, 8, 256, 256),    # one token
        (fmt, 90, 5, 2, 200, 96),    # ragged: a partly covered column tile, a last k-block K only partly covers
        (fmt, 60, 3, 2, 1000, 160),  # ragged N (rows 16 bytes apart) and K
        (fmt, 30, 2, 1, 1, 32),      # one output column, one half k-block
    ]


@pytest.mark.parametrize("fmt,T,E,topk,N,K", CASES)
def test_moe_qmm_parity(orc, fmt, T, E, topk, N, K):
    need_gpu()
    codes, scales = synth.weights(fmt, N, K, T + E, E=E)
    x = synth.activations(T, K, 3 * T + 1)
    ids = synth.expert_ids(T, E, topk, 5 * T + 2)
    y = bf16_host(run_moe_qmm(fmt, codes, scales, x, ids, E, N)).reshape(T * topk, N)
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    assert rc == 0
    check_close(bf16_bits_to_f64(y), want.reshape(T * topk, N), f"moe_qmm fmt{fmt} T{T}", bf16_out=True)


def test_moe_qmm_many_experts(orc):
    """More experts than the multi-block routing takes (E = 300): one routing
    block with shared counters, then the separate gather."""
    need_gpu()
    fmt, T, E, topk, N, K = 0, 64, 300, 4, 256, 64
    codes, scales = synth.weights(fmt, N, K, 60, E=E)
    x = synth.activations(T, K, 59)
    ids = synth.expert_ids(T, E, topk, 58)
    ids[:20, 0] = 7  # one expert with more rows than the rest
    ids[:20, 1:] = synth.expert_ids(20, E - 8, topk - 1, 57) + 8
    y = bf16_host(run_moe_qmm(fmt, codes, scales, x, ids, E, N)).reshape(T * topk, N)
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    assert rc == 0
    check_close(bf16_bits_to_f64(y), want.reshape(T * topk, N), "moe_qmm E=300", bf16_out=True)


@pytest.mark.parametrize("E", [256, 32, 7])
def test_moe_qmm_route_chunks(orc, E):
    """3000 routed rows in 24 chunks of 128 slots (the last one partial), one
    expert taking a third of them across every chunk: per-chunk counts,
    their scan over the chunks (4, 32 and 32 threads per expert) and the
    placement with the gather."""
    need_gpu()
    fmt, T, topk, N, K = 0, 1500, 2, 128, 64
    codes, scales = synth.weights(fmt, N, K, 68, E=E)
    x = synth.activations(T, K, 69)
    ids = synth.expert_ids(T, E, topk, 70)
    ids[::3, 0] = E - 1
    ids[::3, 1] = (ids[::3, 1] + 1) % (E - 1)  # distinct from the first slot
    y = bf16_host(run_moe_qmm(fmt, codes, scales, x, ids, E, N)).reshape(T * topk, N)
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    assert rc == 0
    check_close(bf16_bits_to_f64(y), want.reshape(T * topk, N), f"moe_qmm E={E} chunks", bf16_out=True)


def test_moe_qmm_skewed_routing(orc):
    """Every slot on one expert (a 512-row and an 88-row group tile), the others idle; and the
    down-projection call form (topk = 1 over T * topk rows)."""
    need_gpu()
    fmt, T, E, N, K = 0, 600, 5, 256, 128
    codes, scales = synth.weights(fmt, N, K, 61, E=E)
    x = synth.activations(T, K, 62)
    ids = np.full((T, 1), 2, np.int32)
    y = bf16_host(run_moe_qmm(fmt, codes, scales, x, ids, E, N)).reshape(T, N)
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, 1, N, K)
    assert rc == 0
    check_close(bf16_bits_to_f64(y), want.reshape(T, N), "moe_qmm one expert", bf16_out=True)


def test_moe_qmm_e1_equals_qmm():
    """With one expert the grouped GEMM is the dense GEMM: same bits as mx_qmm
    (each output row depends only on its own X row, whatever its position in
    the group)."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    fmt, T, N, K = 0, 700, 512, 256
    codes, scales = synth.weights(fmt, N, K, 63)
    x = synth.activations(T, K, 64)
    ids = np.zeros((T, 1), np.int32)
    y = bf16_host(run_moe_qmm(fmt, codes, scales, x, ids, 1, N)).reshape(T, N)
    y2 = bf16_host(ops.qmm(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x), N))
    assert np.array_equal(y, y2)


def test_moe_qmm_bad_ids(orc):
    """An id outside [0, E): that slot's row is NaN and the device error word
    records it; every other slot is computed as usual."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    ops.device_error()
    fmt, T, E, topk, N, K = 0, 50, 4, 2, 256, 128
    codes, scales = synth.weights(fmt, N, K, 65, E=E)
    x = synth.activations(T, K, 66)
    ids = synth.expert_ids(T, E, topk, 67)
    ids[7, 1] = E
    ids[20, 0] = -1
    y = bf16_host(run_moe_qmm(fmt, codes, scales, x, ids, E, N)).reshape(T * topk, N)
    assert ops.device_error() & 0x1
    bad = [7 * topk + 1, 20 * topk + 0]
    assert np.all(np.isnan(bf16_bits_to_f64(y[bad])))
    ok = np.ones(T * topk, bool)
    ok[bad] = False
    fixed = ids.copy()
    fixed[7, 1] = 0
    fixed[20, 0] = 0
    want, _ = orc.moe_qmv(fmt, codes, scales, x, fixed, T, E, topk, N, K)
    check_close(bf16_bits_to_f64(y[ok]), want.reshape(T * topk, N)[ok], "moe_qmm good slots", bf16_out=True)


def test_moe_qmm_workspace_checks():
    """A workspace below mx_moe_qmm_workspace_size is MX_EINVAL, one that is
    not 256-byte aligned MX_EALIGN; NVFP4 with K % 32 == 16 (code rows the
    TMA cannot take) MX_EUNSUPPORTED."""
    torch = need_gpu()
    from gemm_decode_register_gb300 import ops

    fmt, T, E, topk, N, K = 0, 8, 4, 2, 256, 64
    codes, scales = synth.weights(fmt, N, K, 68, E=E)
    x = synth.activations(T, K, 69)
    ids = synth.expert_ids(T, E, topk, 70)
    need = ops.load().mx_moe_qmm_workspace_size(T, E, topk, K)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.MxError) as ei:
        run_moe_qmm(fmt, codes, scales, x, ids, E, N, workspace=small)
    assert ei.value.status == -1
    big = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.MxError) as ei:
        run_moe_qmm(fmt, codes, scales, x, ids, E, N, workspace=big[16:])
    assert ei.value.status == -3
    c2, s2 = synth.weights(2, 128, 48, 71, E=E)
    with pytest.raises(ops.MxError) as ei:
        run_moe_qmm(2, c2, s2, synth.activations(T, 48, 72), ids, E, 128)
    assert ei.value.status == -2


@pytest.mark.parametrize("N,K,T,topk,seed", [(1536, 2048, 4096, 8, 0), (2048, 768, 32768, 1, 1)])
def test_moe_qmm_full_size_sampled(orc, N, K, T, topk, seed):
    """128 experts at the MoE layer's sizes: gate+up (1536 x 2048) over 4096
    tokens with top-8 routing, and down (2048 x 768) over their 32768 slot
    rows; every output of 12 sampled tokens (rows) against the oracle."""
    need_gpu()
    fmt, E = 0, 128
    codes, scales = synth.weights(fmt, N, K, 72 + seed, E=E)
    x = synth.activations(T, K, 73 + seed)
    ids = synth.expert_ids(T, E, topk, 74 + seed) if topk > 1 else \
        synth.expert_ids(T // 8, E, 8, 74 + seed).reshape(T, 1)
    y = bf16_host(run_moe_qmm(fmt, codes, scales, x, ids, E, N)).reshape(T, topk, N)
    rng = np.random.default_rng(75 + seed)
    ts = np.sort(np.concatenate([[0, T - 1], rng.choice(np.arange(1, T - 1), 10, replace=False)]))
    want, rc = orc.moe_qmv(fmt, codes, scales, x[ts], ids[ts], len(ts), E, topk, N, K)
    assert rc == 0
    check_close(bf16_bits_to_f64(y[ts].reshape(-1, N)), want.reshape(-1, N), f"moe_qmm full {N}x{K}",
                bf16_out=True)


FFN_CASES = [(fmt, 50, 6, 3, 256, 128) for fmt in (0, 1, 2)] + [(0, 300, 5, 4, 512, 256)]
# ragged: H and I not multiples of the tiles (a partly used gate/up column
# tile, last k-blocks that H and I only partly cover)
FFN_CASES += [(fmt, 40, 4, 2, 160, 96) for fmt in (0, 1, 2)] + [(0, 30, 3, 2, 96, 224)]


@pytest.mark.parametrize("fmt,T,E,topk,H,I", FFN_CASES)
def test_ffn_prefill_parity(orc, fmt, T, E, topk, H, I):
    need_gpu()
    import torch
    from gemm_decode_register_gb300 import ops

    c1, s1 = synth.weights(fmt, 2 * I, H, 80 + T, E=E)
    c2, s2 = synth.weights(fmt, H, I, 81 + T, E=E)
    x = synth.activations(T, H, 82 + T)
    ids = synth.expert_ids(T, E, topk, 83 + T)
    r = synth.router_weights(T, topk, 84 + T)
    out = ops.moe_ffn_prefill(fmt, dev_u8(c1), dev_u8(s1), dev_u8(c2), dev_u8(s2), dev_bf16(x), dev_i32(ids),
                              torch.from_numpy(r).cuda(), E, I).cpu().numpy()
    want = oracle_ffn(orc, fmt, c1, s1, c2, s2, x, ids, r, T, E, topk, H, I)
    check_close(out, want, f"ffn prefill fmt{fmt} T{T}")


def test_ffn_prefill_full_size_sampled(orc):
    """128 experts, top-8, hidden 2048, intermediate 768, 4096 tokens: every
    output of 6 sampled tokens against the oracle chain."""
    need_gpu()
    import torch
    from gemm_decode_register_gb300 import ops

    fmt, T, E, topk, H, I = 0, 4096, 128, 8, 2048, 768
    c1, s1 = synth.weights(fmt, 2 * I, H, 86, E=E)
    c2, s2 = synth.weights(fmt, H, I, 87, E=E)
    x = synth.activations(T, H, 88)
    ids = synth.expert_ids(T, E, topk, 89)
    r = synth.router_weights(T, topk, 90)
    out = ops.moe_ffn_prefill(fmt, dev_u8(c1), dev_u8(s1), dev_u8(c2), dev_u8(s2), dev_bf16(x), dev_i32(ids),
                              torch.from_numpy(r).cuda(), E, I).cpu().numpy()
    ts = np.array([0, 1, 777, 2048, 3000, T - 1])
    want = oracle_ffn(orc, fmt, c1, s1, c2, s2, x[ts], ids[ts], r[ts], len(ts), E, topk, H, I)
    check_close(out[ts], want, "ffn prefill full size")


def test_ffn_prefill_bad_id_and_determinism(orc):
    """A bad id makes its token's outputs NaN (and sets the error word); the
    other tokens match the oracle, and a second call gives the same bits."""
    need_gpu()
    import torch
    from gemm_decode_register_gb300 import ops

    ops.device_error()
    fmt, T, E, topk, H, I = 0, 40, 4, 2, 256, 128
    c1, s1 = synth.weights(fmt, 2 * I, H, 91, E=E)
    c2, s2 = synth.weights(fmt, H, I, 92, E=E)
    x = synth.activations(T, H, 93)
    ids = synth.expert_ids(T, E, topk, 94)
    r = synth.router_weights(T, topk, 95)
    ids[5, 1] = 99
    args = (fmt, dev_u8(c1), dev_u8(s1), dev_u8(c2), dev_u8(s2), dev_bf16(x), dev_i32(ids),
            torch.from_numpy(r).cuda(), E, I)
    out = ops.moe_ffn_prefill(*args).cpu().numpy()
    assert ops.device_error() & 0x1
    assert np.all(np.isnan(out[5]))
    good = np.array([t for t in range(T) if t != 5])
    want = oracle_ffn(orc, fmt, c1, s1, c2, s2, x[good], ids[good], r[good], len(good), E, topk, H, I)
    check_close(out[good], want, "ffn prefill good tokens")
    out2 = ops.moe_ffn_prefill(*args).cpu().numpy()
    assert np.array_equal(out.view(np.uint32), out2.view(np.uint32))
    ops.device_error()
