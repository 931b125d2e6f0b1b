"""Pins that tie the CPU oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises
AssertionError when the oracle disagrees with:

* the pages' own decode method (E2M1 nibble placed into fp16 bits, then one
  multiply by 2^14 -- "MLxcel 0.8 release", section "Decoding block-float
  formats in software"; Strix Halo talk, slide 12),
* library routines that implement the same formats (torch's float8_e4m3fn
  and float8_e8m0fnu, numpy's float16 and float64 matmul),
* exact rational arithmetic (Python ``fractions``) on tiny inputs,
* invariants the mathematics fixes (power-of-two scaling, sign symmetry),
* hand-derived worked examples in ``tests/golden/worked_examples.jsonl``.

They are plain functions so that the plant test can run all of them on a
copy of the oracle compiled with a deliberate mistake and check that at
least one of them fails.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

from gemm_decode_register_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
F4, F8, NV = synth.FMT_MXFP4, synth.FMT_MXFP8, synth.FMT_NVFP4


# ----------------------------------------------------------- independent decodes

def e2m1_by_fp16_placement(code: int) -> float:
    """The pages' method: sign -> fp16 bit 15, the two exponent bits -> the
    two lowest fp16 exponent bits (10, 11), the mantissa bit -> the top
    fp16 mantissa bit (9); then multiply by 2^14."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    bits = np.array([(s << 15) | (e << 10) | (m << 9)], dtype=np.uint16)
    return float(bits.view(np.float16)[0]) * 2.0 ** 14


def e4m3_by_torch(b: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def e8m0_by_ldexp(e: np.ndarray) -> np.ndarray:
    e = np.asarray(e, dtype=np.int64)
    out = np.ldexp(1.0, e - 127)
    return np.where(e == 255, np.nan, out)


def nibbles(codes: np.ndarray, K: int) -> np.ndarray:
    """[N][K] nibble codes from [N][K/2] bytes, even k in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1, K // 2)
    out = np.empty((c.shape[0], K), dtype=np.uint8)
    out[:, 0::2] = c & 0xF
    out[:, 1::2] = c >> 4
    return out


def independent_dequant(fmt: int, codes, scales, N: int, K: int) -> np.ndarray:
    """fp32 [N][K] built from library decodes, vectorised, for comparison."""
    blk = synth.block_of(fmt)
    scales = np.asarray(scales, dtype=np.uint8)
    sc = scales[: N * (K // blk)].reshape(N, K // blk)
    sc = np.repeat(sc, blk, axis=1)
    if fmt == F8:
        v = e4m3_by_torch(np.asarray(codes).reshape(N, K))
    else:
        table = np.array([e2m1_by_fp16_placement(c) for c in range(16)])
        v = table[nibbles(codes, K)]
    with np.errstate(over="ignore", invalid="ignore"):
        if fmt == NV:
            s = e4m3_by_torch(sc)
            g = scales[N * (K // 16):N * (K // 16) + 4].view("<f4")[0]
            w = (v * s).astype(np.float32) * np.float32(g)  # fp32 * fp32, one rounding
        else:
            w = (v * e8m0_by_ldexp(sc)).astype(np.float32)
    return w


def bf16_to_f64(x: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        f = (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
        return f.astype(np.float64)


def rne_bf16_exact(v: float) -> int:
    """bf16 bits of v by exact rational rounding (nearest, ties to even),
    independent of any float rounding mode."""
    if math.isnan(v):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    if math.isinf(v):
        return sign | 0x7F80
    a = Fraction(abs(v))
    if a == 0:
        return sign
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1                                  # now 2^e <= a < 2^(e+1)
    q = max(e - 7, -133)
    n = a / Fraction(2) ** q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = Fraction(fl) * Fraction(2) ** q
    if r >= Fraction(2) ** 128:
        return sign | 0x7F80
    f = np.array([float(r)], dtype=np.float32)
    return sign | int(f.view(np.uint32)[0] >> 16)


def same_bits_f32(a: np.ndarray, b: np.ndarray) -> bool:
    a = np.asarray(a, dtype=np.float32).reshape(-1)
    b = np.asarray(b, dtype=np.float32).reshape(-1)
    na, nb = np.isnan(a), np.isnan(b)
    if not np.array_equal(na, nb):
        return False
    return np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32))


# ------------------------------------------------------------------- the pins

def pin_e2m1(orc):
    """All 16 codes equal the pages' fp16 bit-placement decode, sign of zero
    included, and the familiar value set {0, .5, 1, 1.5, 2, 3, 4, 6}."""
    for c in range(16):
        want = e2m1_by_fp16_placement(c)
        got = orc.e2m1(c)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (c, got, want)
    mags = [orc.e2m1(c) for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], mags
    assert all(orc.e2m1(c + 8) == -orc.e2m1(c) for c in range(8))


def pin_e8m0(orc):
    """2^(e-127) for e = 0..254 (2^-127 kept, not flushed), NaN at 0xFF;
    also equal to torch's float8_e8m0fnu."""
    import torch

    want = e8m0_by_ldexp(np.arange(256))
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for e in range(256):
        got = orc.e8m0(e)
        if e == 255:
            assert math.isnan(got) and math.isnan(lib[e])
        else:
            assert got == want[e] == lib[e], (e, got, want[e], lib[e])


def pin_e4m3(orc):
    """All 256 bytes equal torch's float8_e4m3fn; anchors 448 (0x7E),
    2^-9 (0x01), 1.0 (0x38), -0.0 (0x80), NaN at 0x7F / 0xFF."""
    lib = e4m3_by_torch(np.arange(256, dtype=np.uint8))
    for b in range(256):
        got = orc.e4m3(b)
        if math.isnan(lib[b]):
            assert math.isnan(got), b
        else:
            assert got == lib[b] and math.copysign(1, got) == math.copysign(1, lib[b]), (b, got)
    assert orc.e4m3(0x7E) == 448.0 and orc.e4m3(0x01) == 2.0 ** -9 and orc.e4m3(0x38) == 1.0
    assert math.isnan(orc.e4m3(0x7F)) and math.isnan(orc.e4m3(0xFF))
    assert math.copysign(1, orc.e4m3(0x80)) == -1
    vals = sorted(orc.e4m3(int(b)) for b in synth.NVFP4_SCALE_CODES)
    assert len(vals) == 33 and vals[0] == 0.25 and vals[-1] == 4.0
    assert all(0.25 <= v <= 4.0 for v in vals)


def pin_bf16(orc):
    """bf16 decode equals numpy's fp32 view; bf16 rounding equals exact
    rational nearest-even on ties, subnormals and overflow."""
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    ref = bf16_to_f64(bits)
    for b, r in zip(bits, ref):
        got = orc.bf16(int(b))
        assert (math.isnan(got) and math.isnan(r)) or got == r, (b, got, r)
    cases = [1.0, -1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -30,
             2.0 ** -130 * 1.5, 2.0 ** -133, 2.0 ** -134, 2.0 ** -134 * 1.5, 3.0e38, 3.5e38,
             -0.0, 0.0, float("inf"), -float("inf"), 65504.0, 1e-40, -2.5e-39]
    cases += list(rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 39, size=2000))
    for v in cases:
        assert orc.round_bf16(float(v)) == rne_bf16_exact(float(v)), v


def pin_dequant(orc):
    """Whole-matrix dequantisation equals the independent library decode bit
    for bit, for every format, on random data and on edge scales
    (E8M0 0xFF -> NaN, 254 -> overflow to inf, 0 -> 2^-127 kept)."""
    for fmt, N, K, seed in ((F4, 6, 64, 1), (F8, 5, 96, 2), (NV, 7, 48, 3)):
        codes, scales = synth.weights(fmt, N, K, seed, exp_lo=0, exp_hi=255)
        got = orc.dequant(fmt, codes, scales, N, K)
        want = independent_dequant(fmt, codes, scales, N, K)
        assert same_bits_f32(got, want), fmt
    # edge scales, MXFP4 and MXFP8
    for fmt in (F4, F8):
        N, K = 3, 64
        codes, scales = synth.weights(fmt, N, K, 5)
        scales = scales.copy()
        scales[0], scales[1], scales[2] = 0xFF, 254, 0
        got = orc.dequant(fmt, codes, scales, N, K)
        assert np.all(np.isnan(got[0, :32]))
        assert same_bits_f32(got, independent_dequant(fmt, codes, scales, N, K))


def _rand_case(fmt, M, N, K, seed, lo=120, hi=130):
    codes, scales = synth.weights(fmt, N, K, seed, exp_lo=lo, exp_hi=hi)
    x = synth.activations(M, K, seed + 1000)
    return codes, scales, x


def pin_qmv_bruteforce(orc):
    """Tiny K: the fp64 result is within the recursive-summation bound of
    the exact rational sum of exact products, built from the independent
    decode; for these sizes that bound is below one part in 2^46."""
    for fmt, K in ((F4, 32), (F4, 64), (F8, 32), (NV, 16), (NV, 48)):
        for seed in range(4):
            M, N = 2, 5
            codes, scales, x = _rand_case(fmt, M, N, K, 100 + seed)
            W = independent_dequant(fmt, codes, scales, N, K)
            xs = bf16_to_f64(x)
            y = orc.qmv(fmt, codes, scales, x, M, N, K)
            for m in range(M):
                for n in range(N):
                    terms = [Fraction(float(xs[m, k])) * Fraction(float(W[n, k])) for k in range(K)]
                    exact = sum(terms, Fraction(0))
                    bound = Fraction(K) * Fraction(1, 2 ** 53) * sum(abs(t) for t in terms)
                    assert abs(Fraction(y[m, n]) - exact) <= bound, (fmt, K, m, n)


def pin_qmv_matmul(orc):
    """Moderate sizes: equals numpy float64 matmul of the independent
    dequantisation to 1e-12 relative (row norm)."""
    for fmt, M, N, K in ((F4, 3, 40, 256), (F8, 2, 33, 192), (NV, 4, 17, 320)):
        codes, scales, x = _rand_case(fmt, M, N, K, 7 + fmt)
        W = independent_dequant(fmt, codes, scales, N, K).astype(np.float64)
        want = bf16_to_f64(x) @ W.T
        got = orc.qmv(fmt, codes, scales, x, M, N, K)
        err = np.abs(got - want).max(axis=1) / np.linalg.norm(want, axis=1)
        assert np.all(err < 1e-12), (fmt, err)


def pin_invariants(orc):
    """Exact fp64 invariants: every E8M0 +1 doubles y; NVFP4 tensor scale x2
    doubles y; flipping every code sign or every activation sign negates y;
    all-zero codes give 0."""
    M, N, K = 2, 6, 128
    for fmt in (F4, F8, NV):
        codes, scales, x = _rand_case(fmt, M, N, K, 21 + fmt)
        y = orc.qmv(fmt, codes, scales, x, M, N, K)
        if fmt == NV:
            s2 = scales.copy()
            tail = s2[-4:].view("<f4") * np.float32(2)
            s2[-4:] = tail.view(np.uint8)
        else:
            s2 = (scales.astype(np.int64) + 1).astype(np.uint8)
        assert np.array_equal(orc.qmv(fmt, codes, s2, x, M, N, K), 2 * y), fmt
        flip = np.uint8(0x80 if fmt == F8 else 0x88)
        assert np.array_equal(orc.qmv(fmt, codes ^ flip, scales, x, M, N, K), -y), fmt
        assert np.array_equal(orc.qmv(fmt, codes, scales, x ^ np.uint16(0x8000), M, N, K), -y)
        z = orc.qmv(fmt, np.zeros_like(codes), scales, x, M, N, K)
        assert np.all(z == 0.0)


def pin_worked_examples(orc):
    """Hand-derived examples (tests/golden/worked_examples.jsonl)."""
    with open(os.path.join(HERE, "golden", "worked_examples.jsonl")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ex = json.loads(line)
            fmt = synth.FMT_NAMES[ex["fmt"]]
            K = ex["K"]
            N = 1
            rb = synth.code_bytes_per_row(fmt, K)
            nblk = K // synth.block_of(fmt)
            codes = np.array(ex["code_bytes"] if "code_bytes" in ex else [ex["code_byte"]] * rb,
                             dtype=np.uint8)
            scales = np.array(ex["scale_bytes"] if "scale_bytes" in ex
                              else [ex["scale_byte"]] * nblk, dtype=np.uint8)
            if fmt == NV:
                scales = np.concatenate([scales, np.array([ex["g"]], dtype="<f4").view(np.uint8)])
            xb = ex["x_bf16"]
            x = np.array(xb if isinstance(xb, list) else [xb] * K, dtype=np.uint16).reshape(1, K)
            y = orc.qmv(fmt, codes.reshape(N, rb), scales, x, 1, N, K)
            assert y[0, 0] == ex["expect"], (ex["name"], y[0, 0], ex["expect"])


def pin_moe(orc):
    """MoE reduces to qmv: with E = 1 every slot equals qmv; in general slot
    (t, j) equals qmv on expert ids[t][j]'s slice (numpy matmul of the
    independent dequantisation); an id outside [0, E) is reported."""
    fmt, T, E, topk, N, K = F4, 3, 5, 2, 12, 64
    codes, scales = synth.weights(fmt, N, K, 31, E=E)
    x = synth.activations(T, K, 32)
    ids = synth.expert_ids(T, E, topk, 33)
    y, rc = orc.moe_qmv(fmt, codes, scales, x, ids, T, E, topk, N, K)
    assert rc == 0
    cb = N * K // 2
    sb = N * K // 32
    for t in range(T):
        for j in range(topk):
            e = int(ids[t, j])
            W = independent_dequant(fmt, codes[e * cb:(e + 1) * cb], scales[e * sb:(e + 1) * sb],
                                    N, K).astype(np.float64)
            want = W @ bf16_to_f64(x[t])
            assert np.allclose(y[t, j], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
    # NVFP4: per-expert tensor scales after the whole block-scale stack
    fmt = NV
    codes, scales = synth.weights(fmt, N, 32, 34, E=E)
    scales = scales.copy()
    g = np.array([0.5, 1.0, 2.0, 4.0, 0.25], dtype="<f4")
    scales[-4 * E:] = g.view(np.uint8)
    ids1 = np.arange(E, dtype=np.int32).reshape(E, 1)
    x1 = np.repeat(synth.activations(1, 32, 35), E, axis=0)
    y, rc = orc.moe_qmv(fmt, codes, scales, x1, ids1, E, E, 1, N, 32)
    assert rc == 0
    for e in range(E):
        cb, sb = N * 16, N * 2
        one = np.concatenate([scales[e * sb:(e + 1) * sb], np.array([1.0], "<f4").view(np.uint8)])
        ref = orc.qmv(fmt, codes[e * cb:(e + 1) * cb].reshape(N, 16), one, x1[:1], 1, N, 32)[0]
        assert np.array_equal(y[e, 0], ref * float(g[e])), e
    bad = ids.copy()
    bad[1, 0] = E
    _, rc = orc.moe_qmv(F4, *synth.weights(F4, N, K, 31, E=E), x, bad, T, E, topk, N, K)
    assert rc == -3


def pin_points(orc):
    """qmm_points and qmv_rows pick exactly the matching qmv entries."""
    fmt, M, N, K = F4, 5, 9, 96
    codes, scales, x = _rand_case(fmt, M, N, K, 41)
    y = orc.qmv(fmt, codes, scales, x, M, N, K)
    rows = np.array([8, 0, 3])
    assert np.array_equal(orc.qmv_rows(fmt, codes, scales, x, M, N, K, rows), y[:, rows])
    ms, ns = np.array([0, 4, 2, 2]), np.array([1, 1, 8, 0])
    assert np.array_equal(orc.qmm_points(fmt, codes, scales, x, M, N, K, ms, ns), y[ms, ns])


def pin_rows_threads(orc):
    """qmv_rows_mt (the row list cut into ranges over host threads) returns
    the single-threaded qmv_rows result bit for bit, for thread counts that
    do and do not divide the row count, more threads than rows, and rows in
    any order."""
    for fmt in (F4, F8, NV):
        M, N, K = 3, 37, 128
        codes, scales, x = _rand_case(fmt, M, N, K, 43 + fmt)
        rows = np.random.default_rng(fmt).permutation(N)[:29]
        want = orc.qmv_rows(fmt, codes, scales, x, M, N, K, rows)
        for nt in (1, 2, 3, 7, 29, 64):
            got = orc.qmv_rows_mt(fmt, codes, scales, x, M, N, K, rows, nt)
            assert np.array_equal(got.view(np.uint64), want.view(np.uint64)), (fmt, nt)


def pin_swiglu_combine(orc):
    """SwiGLU: bf16 of torch's float64 silu(gate) * up by exact rational
    rounding; combine: numpy einsum in float64."""
    import torch

    rng = np.random.default_rng(51)
    Q, I = 4, 24
    gu = rng.standard_normal((Q, 2 * I)) * 3.0
    h = orc.swiglu_bf16(gu, I)
    g = torch.from_numpy(gu[:, :I])
    s = (torch.nn.functional.silu(g).numpy() * gu[:, I:])
    want = np.array([[rne_bf16_exact(float(v)) for v in row] for row in s], dtype=np.uint16)
    assert np.array_equal(h, want)
    T, topk, N = 3, 4, 10
    yd = rng.standard_normal((T * topk, N))
    r = synth.router_weights(T, topk, 52)
    out = orc.moe_combine(yd, r, T, topk, N)
    want = np.einsum("tj,tjn->tn", r.astype(np.float64), yd.reshape(T, topk, N))
    assert np.allclose(out, want, rtol=1e-14, atol=1e-14)
    assert np.allclose(r.sum(axis=1), 1.0, atol=1e-6)


# ------------------------------------------------------------- quantisation

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def f32_to_bf16_exact(v: np.ndarray) -> np.ndarray:
    """bf16 bits of fp32 values that bf16 holds exactly (asserted)."""
    f = np.asarray(v, dtype=np.float32).reshape(-1)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not representable in bf16"
    return (bits >> 16).astype(np.uint16)


def canonical_zero(fmt: int, codes: np.ndarray) -> np.ndarray:
    """Codes with -0 replaced by +0 (the quantiser stores every zero as +0)."""
    c = np.asarray(codes, dtype=np.uint8).copy()
    if fmt == F8:
        c[c == 0x80] = 0
        return c
    lo, hi = c & 0xF, c >> 4
    lo[lo == 8] = 0
    hi[hi == 8] = 0
    return (lo | (hi << 4)).astype(np.uint8)


def pin_quantize_roundtrip(orc):
    """Codes and scales built so that every block's largest magnitude sits in
    the element format's top binade (MX) or is 6 times the block scale with a
    power-of-two tensor scale (NVFP4): decoding them (independent decode) and
    quantising the bf16 result must give the same codes and scales back."""
    rng = np.random.default_rng(11)
    M, K = 6, 128
    for fmt in (F4, F8):
        codes, scales = synth.weights(fmt, M, K, 12, exp_lo=110, exp_hi=140)
        if fmt == F8:
            c = codes.reshape(M, K).copy()
            c[(c & 0x7F) == 0x7F] = 0x7E  # no NaN elements
            top = rng.integers(0x78, 0x7F, size=(M, K // 32)) | (rng.integers(0, 2, size=(M, K // 32)) << 7)
            c[:, rng.integers(0, 32) + 32 * np.arange(K // 32)] = top.astype(np.uint8)
            codes = c.reshape(-1)
        else:
            nib = nibbles(codes, K).copy()
            top = rng.integers(4, 8, size=(M, K // 32)) | (rng.integers(0, 2, size=(M, K // 32)) << 3)
            nib[:, rng.integers(0, 32) + 32 * np.arange(K // 32)] = top
            codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8).reshape(-1)
        W = independent_dequant(fmt, codes, scales, M, K)
        c2, s2 = orc.quantize(fmt, f32_to_bf16_exact(W), M, K)
        assert np.array_equal(s2, np.asarray(scales).reshape(-1)), f"fmt {fmt}: scales"
        assert np.array_equal(c2, canonical_zero(fmt, codes)), f"fmt {fmt}: codes"
    # NVFP4: tensor scale 2^-3, block scales any positive E4M3 >= 2^-6, one
    # block at 448; every block holds a +-6
    nb = M * K // 16
    sc = rng.integers(0x08, 0x7F, size=nb).astype(np.uint8)
    sc[rng.integers(0, nb)] = 0x7E
    nib = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    nib.reshape(-1, 16)[np.arange(nb), rng.integers(0, 16, size=nb)] = 7 | (rng.integers(0, 2, size=nb) << 3)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8).reshape(-1)
    scales = np.concatenate([sc, np.array([0.125], dtype="<f4").view(np.uint8)])
    W = independent_dequant(NV, codes, scales, M, K)
    c2, s2 = orc.quantize(NV, f32_to_bf16_exact(W), M, K)
    assert np.array_equal(s2, scales), "nvfp4: scales"
    assert np.array_equal(c2, canonical_zero(NV, codes)), "nvfp4: codes"


def _nearest_even(mags: np.ndarray, a: float) -> int:
    """Index of the nearest magnitude to a (ties to the even index), a beyond
    the largest saturating to it."""
    d = np.abs(mags - a)
    best = np.flatnonzero(d == d.min())
    return int(best[0] if len(best) == 1 else [i for i in best if i % 2 == 0][0])


def pin_quantize_nearest(orc):
    """Random activations over a wide range of magnitudes: the MX scale is
    floor(log2(amax)) - emax + 127 (from frexp), the NVFP4 tensor and block
    scales follow their fp32 formulas (numpy float32 steps, torch E4M3
    rounding), and every code is the nearest-even (saturating) element."""
    rng = np.random.default_rng(13)
    M, K = 8, 96
    xf = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-30, 30, size=(M, 1)))).astype(np.float32)
    x = (xf.view(np.uint32) >> 16).astype(np.uint16)  # truncation: any bf16 values will do
    xv = bf16_to_f64(x).reshape(M, K)
    e4m3_mags = e4m3_by_torch(np.arange(0x7F, dtype=np.uint8))
    for fmt in (F4, F8):
        emax = 8 if fmt == F8 else 2
        mags = e4m3_mags if fmt == F8 else E2M1_MAG
        codes, scales = orc.quantize(fmt, x, M, K)
        cv = e4m3_by_torch(codes).reshape(M, K) if fmt == F8 else \
            np.array([e2m1_by_fp16_placement(c) for c in range(16)])[nibbles(codes, K)]
        for m in range(M):
            for b in range(K // 32):
                blk = xv[m, 32 * b:32 * b + 32]
                amax = np.abs(blk).max()
                e = math.frexp(amax)[1] - 1 - emax if amax > 0 else -127
                e = min(max(e, -127), 127)
                assert scales[m * (K // 32) + b] == e + 127, f"fmt {fmt}: scale of block {m},{b}"
                for k in range(32):
                    v = math.ldexp(blk[k], -e)
                    want = mags[_nearest_even(mags, abs(v))]
                    got = cv[m, 32 * b + k]
                    assert abs(got) == want and (want == 0 or np.sign(got) == np.sign(v)), \
                        f"fmt {fmt}: element {m},{32 * b + k}"
    codes, scales = orc.quantize(NV, x, M, K)
    G = np.float32(np.abs(xv).max())
    g = G / np.float32(2688.0)
    assert scales[M * K // 16:].view("<f4")[0] == g, "nvfp4 tensor scale"
    import torch

    cv = np.array([e2m1_by_fp16_placement(c) for c in range(16)])[nibbles(codes, K)]
    for m in range(M):
        for b in range(K // 16):
            blk = xv[m, 16 * b:16 * b + 16].astype(np.float32)
            t = np.float32(np.abs(blk).max()) / (np.float32(6.0) * g)
            s = int(torch.tensor([float(t)], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])
            assert scales[m * (K // 16) + b] == s, f"nvfp4 block scale {m},{b}"
            den = np.float32(e4m3_by_torch(np.array([s], np.uint8))[0]) * g
            for k in range(16):
                if den == 0:  # block scale rounded to zero: all codes zero
                    assert cv[m, 16 * b + k] == 0, f"nvfp4 element {m},{b},{k}"
                    continue
                v = float(blk[k] / den)
                want = E2M1_MAG[_nearest_even(E2M1_MAG, abs(v))]
                got = cv[m, 16 * b + k]
                assert abs(got) == want and (want == 0 or np.sign(got) == np.sign(v)), f"nvfp4 element {m},{b},{k}"


def pin_quantize_specials(orc):
    """Hand-derived cases (definitions above or_quantize): a block whose
    largest |x| is 4 has scale 2^0 (E8M0 127) in MXFP4; then 0.25 -> 0 and
    0.75 -> 1 and 2.5 -> 2 and 5 -> 4 (ties to the even code), 7.5 in a
    block of max 7.5 saturates to 6, -0 and -0.1 are stored as +0, a NaN or
    an infinity makes the block's scale NaN with zero codes, and an all-zero
    block has scale byte 0 (MX) or 0 (NVFP4)."""
    def bits(vals):
        return (np.asarray(vals, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)

    K = 32
    row = np.zeros(K, np.float32)
    row[:8] = [4.0, 0.25, 0.75, 2.5, 5.0 / 1.0, -5.0, -0.0, -0.1]
    row[4] = 3.5   # tie between 3 and 4 -> 4 (code 6, even)
    codes, scales = orc.quantize(F4, bits(row), 1, K)
    assert scales[0] == 127
    want = [6, 0, 2, 4, 6, 14, 0, 0]  # 4, 0, 1, 2, 4, -4, +0, +0
    assert list(nibbles(codes, K)[0, :8]) == want
    row2 = np.zeros(K, np.float32)
    row2[0], row2[1] = 7.5, -7.0
    codes, scales = orc.quantize(F4, bits(row2), 1, K)
    assert scales[0] == 127 and list(nibbles(codes, K)[0, :2]) == [7, 15]  # saturate to +-6
    for bad in (np.nan, np.inf, -np.inf):
        r3 = np.ones(K, np.float32)
        r3[5] = bad
        for fmt, nanscale in ((F4, 0xFF), (F8, 0xFF)):
            codes, scales = orc.quantize(fmt, bits(r3), 1, K)
            assert scales[0] == nanscale and not codes.any()
        codes, scales = orc.quantize(NV, bits(r3), 1, K)
        assert scales[0] == 0x7F and scales[1] != 0x7F and not codes[:8].any()
    z = np.zeros(K, np.float32)
    for fmt in (F4, F8, NV):
        codes, scales = orc.quantize(fmt, bits(z), 1, K)
        assert not codes.any() and not scales[: K // synth.block_of(fmt)].any()
    codes, scales = orc.quantize(NV, bits(z), 1, K)
    assert scales[2:].view("<f4")[0] == 1.0  # no finite non-zero value: tensor scale 1
    # MXFP8: block max 448 -> floor(log2 448) = 8 -> scale 2^0; 500 -> saturates to 448
    r4 = np.zeros(K, np.float32)
    r4[0], r4[1], r4[2] = 448.0, 300.0, -2.0 ** -9
    codes, scales = orc.quantize(F8, bits(r4), 1, K)
    assert scales[0] == 127 and list(codes[:3]) == [0x7E, 0x79, 0x81]  # 448, 288 (300 -> 288), -2^-9
    r4[0] = 500.0
    codes, scales = orc.quantize(F8, bits(r4), 1, K)
    assert scales[0] == 127 and codes[0] == 0x7E


def pin_qmm_qx(orc):
    """The product over quantised activations equals the float64 matmul of
    the two independently decoded tensors, and swapping the roles of the
    operands (activations as weights and back) transposes it bit for bit."""
    M, N, K = 5, 7, 96
    for fmt in (F4, F8, NV):
        wc, ws = synth.weights(fmt, N, K, 21)
        x = synth.activations(M, K, 22)
        xc, xs = orc.quantize(fmt, x, M, K)
        y = orc.qmm_qx(fmt, wc, ws, xc, xs, M, N, K)
        Xd = independent_dequant(fmt, xc, xs, M, K).astype(np.float64)
        Wd = independent_dequant(fmt, wc, ws, N, K).astype(np.float64)
        assert np.allclose(y, Xd @ Wd.T, rtol=1e-12, atol=1e-30), f"fmt {fmt}"
        yt = orc.qmm_qx(fmt, xc, xs, wc, ws, N, M, K)
        assert np.array_equal(y.view(np.uint64), yt.T.copy().view(np.uint64)), f"fmt {fmt}: roles"
    # tiny K, exact rationals: K = 32 products of decoded values summed exactly
    fmt, M, N, K = F4, 2, 3, 32
    wc, ws = synth.weights(fmt, N, K, 23)
    xc, xs = orc.quantize(fmt, synth.activations(M, K, 24), M, K)
    y = orc.qmm_qx(fmt, wc, ws, xc, xs, M, N, K)
    Xd = independent_dequant(fmt, xc, xs, M, K)
    Wd = independent_dequant(fmt, wc, ws, N, K)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(Xd[m, k])) * Fraction(float(Wd[n, k])) for k in range(K))
            assert abs(Fraction(y[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


ALL_PINS = [pin_e2m1, pin_e8m0, pin_e4m3, pin_bf16, pin_dequant, pin_qmv_bruteforce,
            pin_qmv_matmul, pin_invariants, pin_worked_examples, pin_moe, pin_points, pin_rows_threads,
            pin_swiglu_combine, pin_quantize_roundtrip, pin_quantize_nearest, pin_quantize_specials,
            pin_qmm_qx]
