"""CPU oracle for the block-float decode-in-kernel matmul.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the package smoke
check and the benchmark's CPU-baseline / reference leg, never by the
product path.  The arithmetic lives in ``mx_oracle.c`` (plain C, fp64
accumulation, single-threaded); this module only compiles it with gcc and
marshals numpy arrays through ctypes.

What each function computes (formats per "MLxcel 0.8 release", section
"Decoding block-float formats in software", and the Strix Halo talk,
slide 12; E8M0 / E4M3 / NVFP4 details per OCP MX v1.0 and NVFP4, since the
pages name those formats without defining them):

* ``dequant``  -- W[n][k] = fp32(code * block scale) (NVFP4: then x fp32 g)
* ``qmv``      -- y[m][n] = sum_k x[m][k] * W[n][k] in fp64
* ``qmv_rows`` -- the same on a chosen subset of weight rows
* ``qmv_rows_mt`` -- qmv_rows cut into row ranges over several host threads
* ``qmm_points`` -- the same on chosen (m, n) output points
* ``moe_qmv``  -- y[t][j][n] = sum_k x[t][k] * W_{ids[t][j]}[n][k]
* ``swiglu_bf16`` -- h = bf16_rne(silu(gate) * up) from fp64 inputs
* ``moe_combine`` -- out[t][n] = sum_j r[t][j] * y[t*topk+j][n]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

FMT_MXFP4, FMT_MXFP8, FMT_NVFP4 = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[tuple, ctypes.CDLL] = {}

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-Wall", "-Wextra",
          "-shared", "-fPIC", "-pthread"]


def build(defines: tuple[str, ...] = (), out_dir: str | None = None) -> str:
    """Compile the oracle with gcc; returns the shared-object path.

    ``defines`` are extra ``-D`` macros: the test suite uses them to plant
    known mistakes in a separate copy and check that the pins catch them.
    """
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    tag = "_".join(d.lower() for d in defines)
    so = os.path.join(out_dir, f"liboracle{('_' + tag) if tag else ''}.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(_SRC):
        tmp = so + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, *[f"-D{d}" for d in defines], _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, so)
    return so


def _load(defines: tuple[str, ...] = ()) -> ctypes.CDLL:
    with _LOCK:
        if defines not in _LIBS:
            lib = ctypes.CDLL(build(defines))
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.or_e2m1.restype = ctypes.c_double
            lib.or_e2m1.argtypes = [ctypes.c_uint]
            lib.or_e8m0.restype = ctypes.c_double
            lib.or_e8m0.argtypes = [ctypes.c_uint]
            lib.or_e4m3.restype = ctypes.c_double
            lib.or_e4m3.argtypes = [ctypes.c_uint]
            lib.or_bf16.restype = ctypes.c_double
            lib.or_bf16.argtypes = [ctypes.c_uint16]
            lib.or_round_bf16.restype = ctypes.c_uint16
            lib.or_round_bf16.argtypes = [ctypes.c_double]
            lib.or_dequant.restype = I
            lib.or_dequant.argtypes = [I, P, P, P, I64, I64]
            lib.or_qmv.restype = I
            lib.or_qmv.argtypes = [I, P, P, P, P, I64, I64, I64]
            lib.or_qmv_rows.restype = I
            lib.or_qmv_rows.argtypes = [I, P, P, P, P, I64, I64, I64, P, I64]
            lib.or_qmv_rows_mt.restype = I
            lib.or_qmv_rows_mt.argtypes = [I, P, P, P, P, I64, I64, I64, P, I64, I]
            lib.or_qmm_points.restype = I
            lib.or_qmm_points.argtypes = [I, P, P, P, I64, I64, I64, P, P, I64, P]
            lib.or_moe_qmv.restype = I
            lib.or_moe_qmv.argtypes = [I, P, P, P, P, P, I64, I64, I64, I64, I64]
            lib.or_swiglu_bf16.restype = I
            lib.or_swiglu_bf16.argtypes = [P, P, I64, I64]
            lib.or_moe_combine.restype = I
            lib.or_moe_combine.argtypes = [P, P, P, I64, I64, I64]
            lib.or_quantize.restype = I
            lib.or_quantize.argtypes = [I, P, P, P, I64, I64]
            lib.or_qmm_qx.restype = I
            lib.or_qmm_qx.argtypes = [I, P, P, P, P, P, I64, I64, I64]
            _LIBS[defines] = lib
        return _LIBS[defines]


class Oracle:
    """Thin numpy front end over one compiled copy of the oracle."""

    def __init__(self, defines: tuple[str, ...] = ()):
        self.lib = _load(tuple(defines))

    # -- scalar decodes
    def e2m1(self, code: int) -> float:
        return self.lib.or_e2m1(code)

    def e8m0(self, e: int) -> float:
        return self.lib.or_e8m0(e)

    def e4m3(self, b: int) -> float:
        return self.lib.or_e4m3(b)

    def bf16(self, bits: int) -> float:
        return self.lib.or_bf16(bits)

    def round_bf16(self, v: float) -> int:
        return int(self.lib.or_round_bf16(v))

    # -- arrays
    @staticmethod
    def _u8(a):
        a = np.ascontiguousarray(a, dtype=np.uint8)
        return a, a.ctypes.data

    @staticmethod
    def _bf16bits(x):
        x = np.ascontiguousarray(x)
        if x.dtype != np.uint16:
            raise TypeError("activations are passed as bf16 bit patterns (uint16)")
        return x, x.ctypes.data

    def dequant(self, fmt, codes, scales, N, K) -> np.ndarray:
        codes, pc = self._u8(codes)
        scales, ps = self._u8(scales)
        W = np.empty((N, K), dtype=np.float32)
        rc = self.lib.or_dequant(fmt, pc, ps, W.ctypes.data, N, K)
        if rc:
            raise ValueError(f"or_dequant rc={rc}")
        return W

    def qmv(self, fmt, codes, scales, x, M, N, K) -> np.ndarray:
        codes, pc = self._u8(codes)
        scales, ps = self._u8(scales)
        x, px = self._bf16bits(x)
        y = np.empty((M, N), dtype=np.float64)
        rc = self.lib.or_qmv(fmt, pc, ps, px, y.ctypes.data, M, N, K)
        if rc:
            raise ValueError(f"or_qmv rc={rc}")
        return y

    def qmv_rows(self, fmt, codes, scales, x, M, N, K, rows) -> np.ndarray:
        codes, pc = self._u8(codes)
        scales, ps = self._u8(scales)
        x, px = self._bf16bits(x)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        y = np.empty((M, rows.size), dtype=np.float64)
        rc = self.lib.or_qmv_rows(fmt, pc, ps, px, y.ctypes.data, M, N, K, rows.ctypes.data,
                                  rows.size)
        if rc:
            raise ValueError(f"or_qmv_rows rc={rc}")
        return y

    def qmv_rows_mt(self, fmt, codes, scales, x, M, N, K, rows, nthreads) -> np.ndarray:
        """qmv_rows with the row list cut into nthreads contiguous ranges, one
        host thread each (bit for bit the single-threaded result)."""
        codes, pc = self._u8(codes)
        scales, ps = self._u8(scales)
        x, px = self._bf16bits(x)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        y = np.empty((M, rows.size), dtype=np.float64)
        rc = self.lib.or_qmv_rows_mt(fmt, pc, ps, px, y.ctypes.data, M, N, K, rows.ctypes.data,
                                     rows.size, int(nthreads))
        if rc:
            raise ValueError(f"or_qmv_rows_mt rc={rc}")
        return y

    def qmm_points(self, fmt, codes, scales, x, M, N, K, ms, ns) -> np.ndarray:
        codes, pc = self._u8(codes)
        scales, ps = self._u8(scales)
        x, px = self._bf16bits(x)
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        y = np.empty(ms.size, dtype=np.float64)
        rc = self.lib.or_qmm_points(fmt, pc, ps, px, M, N, K, ms.ctypes.data, ns.ctypes.data,
                                    ms.size, y.ctypes.data)
        if rc:
            raise ValueError(f"or_qmm_points rc={rc}")
        return y

    def moe_qmv(self, fmt, ecodes, escales, x, ids, T, E, topk, N, K):
        """Returns (y [T][topk][N] fp64, rc); rc == -3 flags an id outside [0, E)."""
        ecodes, pc = self._u8(ecodes)
        escales, ps = self._u8(escales)
        x, px = self._bf16bits(x)
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        y = np.full((T, topk, N), np.nan, dtype=np.float64)
        rc = self.lib.or_moe_qmv(fmt, pc, ps, px, ids.ctypes.data, y.ctypes.data, T, E, topk,
                                 N, K)
        if rc not in (0, -3):
            raise ValueError(f"or_moe_qmv rc={rc}")
        return y, rc

    def swiglu_bf16(self, gu: np.ndarray, I: int) -> np.ndarray:
        gu = np.ascontiguousarray(gu, dtype=np.float64)
        Q = gu.size // (2 * I)
        h = np.empty((Q, I), dtype=np.uint16)
        self.lib.or_swiglu_bf16(gu.ctypes.data, h.ctypes.data, Q, I)
        return h

    def moe_combine(self, yd: np.ndarray, r: np.ndarray, T: int, topk: int, N: int):
        yd = np.ascontiguousarray(yd, dtype=np.float64)
        r = np.ascontiguousarray(r, dtype=np.float32)
        out = np.empty((T, N), dtype=np.float64)
        self.lib.or_moe_combine(yd.ctypes.data, r.ctypes.data, out.ctypes.data, T, topk, N)
        return out


    def quantize(self, fmt, x, M, K):
        """bf16 bits [M][K] -> (codes, scales) in the layouts the decode reads
        (NVFP4: the fp32 tensor scale appended to the scales)."""
        x, px = self._bf16bits(x)
        nc = M * K if fmt == 1 else M * K // 2
        ns = M * K // (16 if fmt == 2 else 32) + (4 if fmt == 2 else 0)
        codes = np.zeros(nc, dtype=np.uint8)
        scales = np.zeros(ns, dtype=np.uint8)
        rc = self.lib.or_quantize(fmt, px, codes.ctypes.data, scales.ctypes.data, M, K)
        if rc:
            raise ValueError(f"or_quantize rc={rc}")
        return codes, scales


    def qmm_qx(self, fmt, codes, scales, xcodes, xscales, M, N, K) -> np.ndarray:
        """y [M][N] fp64 = decoded activations (block-float, same format) x
        decoded weights^T."""
        codes, pc = self._u8(codes)
        scales, ps = self._u8(scales)
        xcodes, pxc = self._u8(xcodes)
        xscales, pxs = self._u8(xscales)
        y = np.empty((M, N), dtype=np.float64)
        rc = self.lib.or_qmm_qx(fmt, pc, ps, pxc, pxs, y.ctypes.data, M, N, K)
        if rc:
            raise ValueError(f"or_qmm_qx rc={rc}")
        return y


_DEFAULT: Oracle | None = None


def get() -> Oracle:
    """The unmodified oracle (built on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
