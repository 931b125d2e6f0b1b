"""Helpers for the GPU parity tests: device upload and the tolerance gate.

Tolerance (the method's floating-point bar): per output tensor and per
token row, relative L2 error <= 2e-3, and per row the largest absolute
error divided by that row's L2 norm <= 1e-2, against the fp64 oracle.
"""
from __future__ import annotations

import numpy as np
import pytest

REL_L2 = 2e-3
MAX_ROWNORM = 1e-2
# A bf16 output is rounded to 8 significant bits: that alone moves each
# element by up to 2^-9 of itself, so for bf16 outputs the per-row relative
# L2 allows that rounding on top of the 2e-3 budget (the per-tensor relL2 and
# the max-error bound stay as they are).
BF16_ROUNDING = 2.0 ** -9


def need_gpu():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_decode_register_gb300 import build as b
    b.build()
    return torch


def dev_u8(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8).reshape(-1)).cuda()


def dev_bf16(bits):
    import torch

    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()


def dev_i32(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def bf16_host(t):
    """bf16 torch tensor -> uint16 bit patterns (numpy)."""
    import torch

    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(bits):
    with np.errstate(invalid="ignore"):
        return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_close(got, want, what="", bf16_out=False):
    """Tolerance gate on [rows][cols] arrays (got fp32/bf16-as-float, want fp64)."""
    got = np.asarray(got, dtype=np.float64).reshape(want.shape[0], -1)
    want = np.asarray(want, dtype=np.float64).reshape(want.shape[0], -1)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = got - want
    tot = np.linalg.norm(err) / np.linalg.norm(want)
    rn = np.linalg.norm(want, axis=1)
    rel_rows = np.linalg.norm(err, axis=1) / rn
    mx = np.abs(err).max(axis=1) / rn
    assert tot <= REL_L2, f"{what}: relL2 {tot:.3e}"
    row_lim = REL_L2 + (BF16_ROUNDING if bf16_out else 0.0)
    assert rel_rows.max() <= row_lim, f"{what}: worst row relL2 {rel_rows.max():.3e}"
    assert mx.max() <= MAX_ROWNORM, f"{what}: max |err| / row norm {mx.max():.3e}"
    return tot, rel_rows.max(), mx.max()


def check_special(got, want, what="", bf16_out=False):
    """The tolerance gate for outputs that may hold NaN or +-inf: NaN
    positions must agree exactly with the oracle's, every infinite oracle
    value must be matched by the same infinity (and the GPU may give an
    infinity nowhere else), and the finite entries pass the usual gate, with
    each row's norm taken over its finite entries."""
    got = np.asarray(got, dtype=np.float64).reshape(want.shape[0], -1)
    want = np.asarray(want, dtype=np.float64).reshape(want.shape[0], -1)
    gn, wn = np.isnan(got), np.isnan(want)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ in {int((gn != wn).sum())} entries"
    gi, wi = np.isinf(got), np.isinf(want)
    assert np.array_equal(gi, wi), f"{what}: infinity positions differ in {int((gi != wi).sum())} entries"
    assert np.array_equal(got[wi], want[wi]), f"{what}: infinities of the wrong sign"
    fin = np.isfinite(want)
    with np.errstate(invalid="ignore"):
        err = np.where(fin, got - want, 0.0)
    ref = np.where(fin, want, 0.0)
    tot_n = np.linalg.norm(ref)
    if tot_n == 0.0:
        assert not np.any(err), f"{what}: nonzero output where the oracle is zero"
        return 0.0, 0.0, 0.0
    tot = np.linalg.norm(err) / tot_n
    rn = np.linalg.norm(ref, axis=1)
    live = rn > 0
    rel_rows = np.linalg.norm(err[live], axis=1) / rn[live]
    mx = np.abs(err[live]).max(axis=1) / rn[live]
    assert not np.any(err[~live]), f"{what}: nonzero output in a row the oracle has at zero"
    assert tot <= REL_L2, f"{what}: relL2 {tot:.3e}"
    row_lim = REL_L2 + (BF16_ROUNDING if bf16_out else 0.0)
    assert rel_rows.max() <= row_lim, f"{what}: worst row relL2 {rel_rows.max():.3e}"
    assert mx.max() <= MAX_ROWNORM, f"{what}: max |err| / row norm {mx.max():.3e}"
    return tot, rel_rows.max(), mx.max()


def bf16_ulp_diff(a, b):
    """Distance in units in the last place between bf16 bit patterns: the
    patterns are mapped to integers that increase with the value (negative
    numbers below -0, -0 and +0 one apart), so the difference counts the
    representable numbers between the two, across zero and signs too."""
    def key(bits):
        v = np.asarray(bits, dtype=np.uint16).astype(np.int64)
        mag = v & 0x7FFF
        return np.where(v & 0x8000, -mag - 1, mag)

    return np.abs(key(a) - key(b))


def same_values(got, want):
    """Value equality with NaN == NaN (and +0 == -0)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    ng, nw = np.isnan(got), np.isnan(want)
    return np.array_equal(ng, nw) and np.array_equal(got[~ng], want[~nw])


def same_bits_f32(got, want):
    got = np.asarray(got, dtype=np.float32).reshape(-1)
    want = np.asarray(want, dtype=np.float32).reshape(-1)
    ng, nw = np.isnan(got), np.isnan(want)
    if not np.array_equal(ng, nw):
        return False
    return np.array_equal(got[~ng].view(np.uint32), want[~nw].view(np.uint32))
