"""The formats' extreme values through the hot kernels (qmv, MoE qmv, the
fused MoE FFN pair, the prefill GEMM and the grouped prefill GEMM), element
by element against the oracle with NaN and infinity positions compared
exactly (gpu_util.check_special):

* NaN block scales (E8M0 0xFF, E4M3 0x7F / 0xFF): every output that reads
  such a block is NaN, as the oracle's NaN weight makes it.
* the smallest E8M0 scales (2^-127 .. 2^-122): decoded weights down in
  fp32's (and bf16's) subnormal range.  NVFP4: E4M3 subnormal and zero
  block scales.
* the largest E8M0 scales (2^125 .. 2^127) with codes that keep every
  decoded weight finite, and small activations so that the products are
  finite too (also through the fold of a token's power of two into the
  block scales, which these activations switch on).
* decoded weights beyond fp32's range (E8M0 254, |code| >= 2) in one block
  per row, with positive activations: the oracle's weights are infinite and
  every product in the block has the row's sign, so the output is that
  infinity; the kernels scale the block's partial sum and reach the same
  infinity.
* MXFP8 elements: NaN codes (0x7F / 0xFF) and the largest finite +-448.
* activations: tokens spanning 2^-30 .. 2^10, a 2^12 outlier among N(0,1)
  values, a token holding +inf or NaN.
"""
import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import (bf16_bits_to_f64, bf16_host, check_special, dev_bf16, dev_i32, dev_u8,
                      need_gpu)

pytestmark = pytest.mark.gpu

F4, F8, NV = synth.FMT_MXFP4, synth.FMT_MXFP8, synth.FMT_NVFP4


# ------------------------------------------------------------------ inputs

def _split(fmt, scales, E, N, K):
    """The block-scale bytes as an [E][N][K/block] view (NVFP4: without the
    tensor scales that follow them)."""
    nb = K // synth.block_of(fmt)
    return scales[: E * N * nb].reshape(E, N, nb)


def _codes3(fmt, codes, E, N, K):
    return codes.reshape(E, N, synth.code_bytes_per_row(fmt, K))


def special_weights(fmt, kind, N, K, seed, E=1):
    """(codes, scales) with the extreme values of `kind` (see the module
    docstring); the rest as the workloads draw them."""
    rng = np.random.default_rng(seed)
    codes, scales = synth.weights(fmt, N, K, seed, E=E, exp_lo=118, exp_hi=132)
    codes = codes.reshape(-1).copy()
    scales = scales.copy()
    sc = _split(fmt, scales, E, N, K)
    cd = _codes3(fmt, codes, E, N, K)
    nb = sc.shape[2]
    if kind == "nan_scale":
        mask = rng.random(sc.shape) < 0.02
        if fmt == NV:
            sc[mask] = rng.choice(np.array([0x7F, 0xFF], np.uint8), size=int(mask.sum()))
        else:
            sc[mask] = 0xFF
    elif kind == "tiny_scale":
        if fmt == NV:
            # E4M3 subnormal scales (2^-9 .. 7 * 2^-9), and some +-0
            sc[...] = rng.integers(1, 8, size=sc.shape, dtype=np.uint8)
            sc[rng.random(sc.shape) < 0.05] = 0x00
            sc[rng.random(sc.shape) < 0.05] = 0x80
        else:
            sc[...] = rng.integers(0, 6, size=sc.shape, dtype=np.uint8)
    elif kind == "huge_scale":
        if fmt == NV:
            # the largest E4M3 block scales and a tensor scale of 2^100
            sc[...] = rng.choice(np.array([0x7E, 0x7D, 0x76, 0xFE], np.uint8), size=sc.shape)
            scales[-4 * E:] = np.full(E, 2.0 ** 100, dtype="<f4").view(np.uint8)
        elif fmt == F8:
            sc[...] = rng.integers(244, 247, size=sc.shape, dtype=np.uint8)  # 448 * 2^119 < 2^128
        else:
            e = rng.integers(252, 255, size=sc.shape, dtype=np.uint8)
            sc[...] = e
            # keep |code| * 2^(e-127) finite: |code| <= 1.5 at 254, <= 3 at 253
            for n_e in range(E):
                for n in range(N):
                    for b in range(nb):
                        lim = {252: 8, 253: 6, 254: 4}[int(e[n_e, n, b])]
                        blk = cd[n_e, n, b * 16:(b + 1) * 16]
                        lo = rng.integers(0, lim, size=blk.shape) | (rng.integers(0, 2, size=blk.shape) << 3)
                        hi = rng.integers(0, lim, size=blk.shape) | (rng.integers(0, 2, size=blk.shape) << 3)
                        cd[n_e, n, b * 16:(b + 1) * 16] = (lo | (hi << 4)).astype(np.uint8)
    elif kind == "overflow":
        # one block per row at E8M0 254 whose codes all have |code| >= 2 and
        # the row's sign: its decoded weights are that signed infinity
        bsel = rng.integers(0, nb, size=(E, N))
        sign = rng.integers(0, 2, size=(E, N))
        for n_e in range(E):
            for n in range(N):
                b = int(bsel[n_e, n])
                sc[n_e, n, b] = 254
                if fmt == F8:
                    # E4M3 exponent field 8..14: values 2 .. 240 (never NaN)
                    v = (rng.integers(8, 15, size=32) << 3) | rng.integers(0, 8, size=32)
                    cd[n_e, n, b * 32:(b + 1) * 32] = (v | (sign[n_e, n] << 7)).astype(np.uint8)
                else:
                    lo = rng.integers(4, 8, size=16) | (sign[n_e, n] << 3)
                    hi = rng.integers(4, 8, size=16) | (sign[n_e, n] << 3)
                    cd[n_e, n, b * 16:(b + 1) * 16] = (lo | (hi << 4)).astype(np.uint8)
    elif kind == "fp8_elements":
        assert fmt == F8
        r = rng.random(cd.shape)
        cd[r < 0.001] = rng.choice(np.array([0x7F, 0xFF], np.uint8), size=int((r < 0.001).sum()))
        big = (r >= 0.001) & (r < 0.15)
        cd[big] = rng.choice(np.array([0x7E, 0xFE], np.uint8), size=int(big.sum()))
    else:
        raise ValueError(kind)
    if E == 1:
        codes = codes.reshape(N, -1)
    return codes, scales


def _bf16(f):
    import torch

    return torch.from_numpy(np.ascontiguousarray(f, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def special_x(kind, M, K, seed):
    """bf16 bit patterns [M][K] of the activation kind."""
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return synth.activations(M, K, seed)
    if kind == "small":
        return _bf16(rng.standard_normal((M, K)) * 2.0 ** -16)
    if kind == "positive":
        return _bf16(np.abs(rng.standard_normal((M, K))) + 2.0 ** -4)
    if kind == "wide":
        e = rng.uniform(-30.0, 10.0, size=(M, K))
        return _bf16(np.where(rng.random((M, K)) < 0.5, -1.0, 1.0) * 2.0 ** e)
    if kind == "outlier":
        f = rng.standard_normal((M, K)).astype(np.float32)
        f[np.arange(M), rng.integers(0, K, size=M)] = np.where(rng.random(M) < 0.5, -1.0, 1.0) * 2.0 ** 12
        return _bf16(f)
    if kind == "nonfinite":
        f = rng.standard_normal((M, K)).astype(np.float32)
        f[0, rng.integers(0, K)] = np.inf
        if M > 1:
            f[1, rng.integers(0, K)] = np.nan
        return _bf16(f)
    raise ValueError(kind)


# which activations each weight kind is paired with
WEIGHT_CASES = [
    (F4, "nan_scale", "normal"), (F8, "nan_scale", "normal"), (NV, "nan_scale", "normal"),
    (F4, "tiny_scale", "normal"), (F8, "tiny_scale", "normal"), (NV, "tiny_scale", "normal"),
    (F4, "huge_scale", "small"), (F8, "huge_scale", "small"), (NV, "huge_scale", "small"),
    (F4, "overflow", "positive"), (F8, "overflow", "positive"),
    (F8, "fp8_elements", "normal"),
]
X_CASES = [(fmt, xk) for fmt in (F4, F8, NV) for xk in ("wide", "outlier", "nonfinite")]


def _weights_for(fmt, wk, N, K, seed, E=1):
    if wk is None:
        codes, scales = synth.weights(fmt, N, K, seed, E=E, exp_lo=118, exp_hi=132)
        return codes, scales
    return special_weights(fmt, wk, N, K, seed, E=E)


ALL_CASES = [(f, w, x) for f, w, x in WEIGHT_CASES] + [(f, None, x) for f, x in X_CASES]
IDS = [f"fmt{f}-{w or 'plain'}-{x}" for f, w, x in ALL_CASES]


# ------------------------------------------------------------------ qmv

@pytest.mark.parametrize("fmt,wk,xk", ALL_CASES, ids=IDS)
@pytest.mark.parametrize("M,N,K", [(1, 192, 512), (4, 100, 512), (3, 70, 96)])
def test_qmv_extremes(orc, fmt, wk, xk, M, N, K):
    """Streaming kernel (K = 512) and direct-load kernel (K = 96)."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    codes, scales = _weights_for(fmt, wk, N, K, 7 * N + K)
    x = special_x(xk, M, K, N + M)
    y = ops.qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x).view(M, K), N).cpu().numpy()
    want = orc.qmv(fmt, codes, scales, x, M, N, K)
    check_special(y, want, f"qmv fmt{fmt} {wk} {xk} {M}x{N}x{K}")


@pytest.mark.parametrize("fmt", [F4, F8, NV])
@pytest.mark.parametrize("xk", ["nonfinite", "outlier", "wide"])
def test_qmv_extremes_staged_in_shared_memory(orc, fmt, xk):
    """Activations with an infinity and a NaN, an outlier or a wide range
    through the staging path that parks raw chunks in shared memory (4 rows
    of K = 10240): the row maxima ignore the non-finite elements there too."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    M, N, K = 4, 96, 10240
    codes, scales = _weights_for(fmt, None, N, K, 5 * N + fmt)
    x = special_x(xk, M, K, 77 + fmt)
    y = ops.qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x).view(M, K), N).cpu().numpy()
    want = orc.qmv(fmt, codes, scales, x, M, N, K)
    check_special(y, want, f"qmv fmt{fmt} {xk} {M}x{N}x{K} (staging in shared memory)")


# ------------------------------------------------------------------ MoE

@pytest.mark.parametrize("fmt,wk,xk", ALL_CASES, ids=IDS)
def test_moe_qmv_extremes(orc, fmt, wk, xk):
    need_gpu()
    from gemm_decode_register_gb300 import ops

    T, E, topk, N, K = 3, 6, 2, 64, 256
    codes, scales = _weights_for(fmt, wk, N, K, 11 + fmt, E=E)
    x = special_x(xk, T, K, 12)
    ids = synth.expert_ids(T, E, topk, 13)
    y = ops.moe_qmv(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x).view(T, K), dev_i32(ids), E, N).cpu().numpy()
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    assert rc == 0
    check_special(y.reshape(T * topk, N), want.reshape(T * topk, N), f"moe fmt{fmt} {wk} {xk}")


# (format, gate-up weights, down weights, activations): the SwiGLU of two
# tiny projections underflows to zero, so tiny scales go into the down stack
FUSED_CASES = ([(f, "nan_scale", "nan_scale", "normal") for f in (F4, F8, NV)]
               + [(f, None, "tiny_scale", "normal") for f in (F4, F8, NV)]
               + [(f, None, None, xk) for f in (F4, F8, NV) for xk in ("wide", "outlier")])


@pytest.mark.parametrize("fmt,wgu,wdn,xk", FUSED_CASES,
                         ids=[f"fmt{f}-{a or 'plain'}-{b or 'plain'}-{x}" for f, a, b, x in FUSED_CASES])
def test_fused_moe_ffn_extremes(orc, fmt, wgu, wdn, xk):
    """Gate-up + SwiGLU and down + combine; h against the oracle chain, out
    against the oracle's down projection and combine of the GPU's h."""
    need_gpu()
    import torch
    from gemm_decode_register_gb300 import ops

    T, E, topk, H, I = 3, 5, 2, 256, 128
    c1, s1 = _weights_for(fmt, wgu, 2 * I, H, 21 + fmt, E=E)
    c2, s2 = _weights_for(fmt, wdn, H, I, 22 + fmt, E=E)
    x = special_x(xk, T, H, 23)
    ids = synth.expert_ids(T, E, topk, 24)
    r = synth.router_weights(T, topk, 25)
    d_ids = dev_i32(ids)
    h = ops.moe_gate_up_swiglu(fmt, dev_u8(c1), dev_u8(s1), dev_bf16(x).view(T, H), d_ids, E, I)
    out = ops.moe_down_combine(fmt, dev_u8(c2), dev_u8(s2), h.view(T * topk, I), d_ids,
                               torch.from_numpy(r).cuda(), E, H).cpu().numpy()
    gu, rc = orc.moe_qmv(fmt, c1, s1, x, ids, T, E, topk, 2 * I, H)
    assert rc == 0
    h_o = orc.swiglu_bf16(gu.reshape(T * topk, 2 * I), I)
    hb = bf16_host(h).reshape(T * topk, I)
    check_special(bf16_bits_to_f64(hb), bf16_bits_to_f64(h_o), f"gate-up fmt{fmt} {wgu} {xk}", bf16_out=True)
    # the down projection of the GPU's own h (a rounding difference in h does
    # not count twice)
    yd, rc = orc.moe_qmv(fmt, c2, s2, hb, ids.reshape(-1, 1), T * topk, E, 1, H, I)
    want = orc.moe_combine(yd.reshape(T * topk, H), r, T, topk, H)
    check_special(out, want, f"down-combine fmt{fmt} {wdn} {xk}")


# ------------------------------------------------------------------ prefill

QMM_CASES = [c for c in ALL_CASES]


@pytest.mark.parametrize("fmt,wk,xk", QMM_CASES, ids=IDS)
@pytest.mark.parametrize("M", [200, 600])
def test_qmm_extremes(orc, fmt, wk, xk, M):
    """The tensor-core GEMM decodes to bf16 in shared memory: NaN scales and
    NaN E4M3 codes must stay NaN, infinities stay infinities, and decoded
    weights below 2^-126 are bf16 subnormals fed to tcgen05.mma."""
    need_gpu()
    from gemm_decode_register_gb300 import ops

    N, K = 256, 512
    codes, scales = _weights_for(fmt, wk, N, K, 31 + fmt)
    X = special_x(xk, M, K, 32)
    Y = ops.qmm(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(X).view(M, K), N)
    got = bf16_bits_to_f64(bf16_host(Y))
    want = orc.qmv(fmt, codes, scales, X, M, N, K)
    check_special(got, want, f"qmm fmt{fmt} {wk} {xk} M{M}", bf16_out=True)


@pytest.mark.parametrize("fmt,wk,xk", [c for c in ALL_CASES if c[2] != "nonfinite"],
                         ids=[i for c, i in zip(ALL_CASES, IDS) if c[2] != "nonfinite"])
def test_moe_qmm_extremes(orc, fmt, wk, xk):
    need_gpu()
    from gemm_decode_register_gb300 import ops

    T, E, topk, N, K = 90, 4, 2, 256, 256
    codes, scales = _weights_for(fmt, wk, N, K, 41 + fmt, E=E)
    x = special_x(xk, T, K, 42)
    ids = synth.expert_ids(T, E, topk, 43)
    y = ops.moe_qmm(fmt, dev_u8(codes), dev_u8(scales), dev_bf16(x).view(T, K), dev_i32(ids), E, N)
    got = bf16_bits_to_f64(bf16_host(y)).reshape(T * topk, N)
    want, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    assert rc == 0
    check_special(got, want.reshape(T * topk, N), f"moe qmm fmt{fmt} {wk} {xk}", bf16_out=True)
