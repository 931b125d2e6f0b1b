"""Seeded synthetic inputs for the block-float matmul (weights, activations,
routing).  Shared by the tests, the benchmark and the oracle checks.

This module only draws random bit patterns with the distributions the
workloads call for; it holds none of the decode or matmul arithmetic.
Every array is a numpy array of raw bytes / bit patterns:

* codes  -- uint8.  MXFP4 / NVFP4: [N][K/2], element k in byte k/2, even k
            in the low nibble.  MXFP8: [N][K], one E4M3 byte per element.
* scales -- uint8.  MXFP4 / MXFP8: E8M0 exponents [N][K/32].  NVFP4: E4M3
            bytes [N][K/16] followed by the fp32 per-tensor scale (4 bytes,
            little-endian); an expert stack [E][N][K/16] is followed by E
            such fp32 values, one per expert.
* x      -- uint16 bf16 bit patterns [M][K], round-to-nearest-even from
            fp32 N(0, 1) samples.
"""
from __future__ import annotations

import numpy as np

FMT_MXFP4, FMT_MXFP8, FMT_NVFP4 = 0, 1, 2
FMT_NAMES = {"mxfp4": FMT_MXFP4, "mxfp8": FMT_MXFP8, "nvfp4": FMT_NVFP4}

# E4M3 bit patterns that are NaN in the "FN" variant (S.1111.111).
E4M3_NAN_BYTES = (0x7F, 0xFF)

# The 33 E4M3 bit patterns whose value lies in [0.25, 4]: exponent field
# 5..8 with any mantissa (0.25 .. 3.75), plus exponent field 9 with mantissa
# 0 (4.0).  The bit pattern is (exponent << 3) | mantissa.
NVFP4_SCALE_CODES = np.array([(e << 3) | m for e in range(5, 9) for m in range(8)] + [9 << 3],
                             dtype=np.uint8)

# fp32(1/448): one correctly rounded fp32 division.
NVFP4_TENSOR_SCALE = np.float32(1.0) / np.float32(448.0)


def block_of(fmt: int) -> int:
    return 16 if fmt == FMT_NVFP4 else 32


def code_bytes_per_row(fmt: int, K: int) -> int:
    return K if fmt == FMT_MXFP8 else K // 2


def scale_bytes(fmt: int, N: int, K: int, E: int = 1) -> int:
    n = E * N * (K // block_of(fmt))
    return n + (4 * E if fmt == FMT_NVFP4 else 0)


def weight_bytes(fmt: int, N: int, K: int, E: int = 1) -> int:
    """Bytes a kernel must stream to read the whole weight once."""
    return E * N * code_bytes_per_row(fmt, K) + scale_bytes(fmt, N, K, E)


def weights(fmt: int, N: int, K: int, seed: int, *, E: int = 1, exp_lo: int = 118,
            exp_hi: int = 132, tensor_scale: np.float32 | None = None):
    """(codes, scales) for E stacked [N][K] weights.

    Codes are uniform over all 16 E2M1 codes (a uniform byte holds two
    independent uniform nibbles) or, for MXFP8, uniform over the 254 finite
    E4M3 bytes.  E8M0 exponents are uniform integers in [exp_lo, exp_hi].
    NVFP4 block scales are uniform over NVFP4_SCALE_CODES and the
    per-tensor scale defaults to fp32(1/448).
    """
    if K % block_of(fmt):
        raise ValueError("K must be a multiple of the block size")
    rng = np.random.default_rng(seed)
    rb = code_bytes_per_row(fmt, K)
    if fmt == FMT_MXFP8:
        finite = np.array([b for b in range(256) if b not in E4M3_NAN_BYTES], dtype=np.uint8)
        codes = finite[rng.integers(0, finite.size, size=(E, N, rb))]
    else:
        codes = rng.integers(0, 256, size=(E, N, rb), dtype=np.uint8)
    nblk = K // block_of(fmt)
    if fmt == FMT_NVFP4:
        sc = NVFP4_SCALE_CODES[rng.integers(0, NVFP4_SCALE_CODES.size, size=(E, N, nblk))]
        g = NVFP4_TENSOR_SCALE if tensor_scale is None else np.float32(tensor_scale)
        tail = np.full(E, g, dtype="<f4").view(np.uint8)
        scales = np.concatenate([sc.reshape(-1), tail])
    else:
        scales = rng.integers(exp_lo, exp_hi + 1, size=(E, N, nblk), dtype=np.uint8).reshape(-1)
    codes = codes.reshape(-1) if E > 1 else codes.reshape(N, rb)
    return codes, scales


def weights_device(fmt: int, N: int, K: int, seed: int, device, *, exp_lo: int = 118, exp_hi: int = 132):
    """(codes, scales) as uint8 torch tensors on `device`, drawn with the
    same distributions as weights() by a seeded generator on that device
    (for workloads too large to draw on the host: tens of GB of weights).
    The values differ from weights() for the same seed."""
    import torch

    if K % block_of(fmt):
        raise ValueError("K must be a multiple of the block size")
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    u8 = dict(dtype=torch.uint8, device=device, generator=g)
    nc = N * code_bytes_per_row(fmt, K)
    if fmt == FMT_MXFP8:
        # 254 finite E4M3 bytes: 0..126 and 128..254 (0x7F and 0xFF are NaN)
        v = torch.randint(0, 254, (nc,), **u8)
        codes = v + (v >= 127).to(torch.uint8)
    else:
        codes = torch.randint(0, 256, (nc,), **u8)
    nblk = N * (K // block_of(fmt))
    if fmt == FMT_NVFP4:
        table = torch.from_numpy(NVFP4_SCALE_CODES).to(device)
        idx = torch.randint(0, NVFP4_SCALE_CODES.size, (nblk,), dtype=torch.int64, device=device, generator=g)
        tail = torch.from_numpy(np.array([NVFP4_TENSOR_SCALE], dtype="<f4").view(np.uint8)).to(device)
        scales = torch.cat([table[idx], tail])
    else:
        scales = torch.randint(exp_lo, exp_hi + 1, (nblk,), **u8)
    return codes, scales


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """bf16 bit patterns of N(0, 1) samples, [M][K] uint16."""
    import torch

    rng = np.random.default_rng(seed)
    f = rng.standard_normal((M, K), dtype=np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def expert_ids(T: int, E: int, topk: int, seed: int) -> np.ndarray:
    """[T][topk] int32: topk distinct experts per token, uniform."""
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, size=topk, replace=False) for _ in range(T)]).astype(np.int32)


def router_weights(T: int, topk: int, seed: int) -> np.ndarray:
    """[T][topk] fp32: softmax over topk N(0, 1) logits per token (the
    renormalised weights of the selected experts)."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, topk))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
