"""Python binding of the C ABI in include/mx.h (argument marshalling only).

Each function takes torch CUDA tensors, passes their device pointers and
the current torch stream to libmxgemm.so, and raises MxError on a non-zero
status.  Every step of the computation runs in the library's kernels; there
is no fallback path: if the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from .synth import FMT_MXFP4, FMT_MXFP8, FMT_NVFP4, block_of  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmxgemm.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "mx.h")

_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


class MxError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmxgemm.so (built by ``gemm_decode_register_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} is missing "
                               "(run __graft_entry__.build() or python -m "
                               "gemm_decode_register_gb300.build)")
        lib = ctypes.CDLL(p)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "mx_qmv": [I, P, P, P, P, I, I, I],
            "mx_qmv_noalloc": [I, P, P, P, P, I, I, I],
            "mx_moe_qmv": [I, P, P, P, P, P, I, I, I, I, I],
            "mx_moe_gate_up_swiglu": [I, P, P, P, P, P, I, I, I, I, I],
            "mx_moe_down_combine": [I, P, P, P, P, P, P, I, I, I, I, I],
            "mx_qmm": [I, P, P, P, P, I, I, I],
            "mx_set_stream": [P],
            "mx_dequant": [I, P, P, P, I, I],
            "mx_swiglu": [P, P, I, I],
            "mx_moe_combine": [P, P, P, I, I, I],
            "mx_device_error": [],
            "mx_debug_qmm_stall": [I, ctypes.c_ulonglong],
            "mx_qmm_qx": [I, P, P, P, P, P, I, I, I],
            "mx_mma_peak": [I, I, P],
            "mx_moe_qmm": [I, P, P, P, P, P, I, I, I, I, I, P, Z],
            "mx_quantize": [I, P, P, P, I, I],
            "mx_moe_ffn_prefill": [I, P, P, P, P, P, P, P, P, I, I, I, I, I, P, Z],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = I
        for name, args in {"mx_moe_qmm_workspace_size": [I, I, I, I],
                           "mx_moe_ffn_prefill_workspace_size": [I, I, I, I, I]}.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = Z
        lib.mx_strerror.argtypes = [I]
        lib.mx_strerror.restype = ctypes.c_char_p
        _lib = lib
        return lib


def header_symbols() -> list[str]:
    """Names of the functions include/mx.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"^\s*(?:const\s+char\s*\*|int|size_t)\s*(mx_\w+)\s*\(", text, flags=re.M)


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MxError(fn, status, load().mx_strerror(status).decode())


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream() -> None:
    load().mx_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def qmv(fmt: int, codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, N: int,
        y: torch.Tensor | None = None) -> torch.Tensor:
    """y[M][N] fp32 = x (bf16 [M][K]) . W^T, W block-float [N][K]."""
    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _stream()
    _check("mx_qmv", load().mx_qmv(fmt, _ptr(codes), _ptr(scales), _ptr(x), _ptr(y), M, N, K))
    return y


def qmv_noalloc(fmt: int, codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, N: int,
                y: torch.Tensor | None = None) -> torch.Tensor:
    """mx_qmv_noalloc: the same product, with no device allocation."""
    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _stream()
    _check("mx_qmv_noalloc", load().mx_qmv_noalloc(fmt, _ptr(codes), _ptr(scales), _ptr(x), _ptr(y), M, N, K))
    return y


def moe_qmv(fmt: int, codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor,
            expert_ids: torch.Tensor, E: int, N: int, y: torch.Tensor | None = None) -> torch.Tensor:
    """y[T][topk][N] fp32 over the routed experts of each token."""
    T, K = x.shape
    topk = expert_ids.shape[1]
    if y is None:
        y = torch.empty((T, topk, N), dtype=torch.float32, device=x.device)
    _stream()
    _check("mx_moe_qmv", load().mx_moe_qmv(fmt, _ptr(codes), _ptr(scales), _ptr(x),
                                           _ptr(expert_ids), _ptr(y), T, E, topk, N, K))
    return y


def moe_gate_up_swiglu(fmt: int, codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor,
                       expert_ids: torch.Tensor, E: int, I: int, h: torch.Tensor | None = None) -> torch.Tensor:
    """h[T][topk][I] bf16 = SwiGLU of the routed experts' gate and up rows."""
    T, K = x.shape
    topk = expert_ids.shape[1]
    if h is None:
        h = torch.empty((T, topk, I), dtype=torch.bfloat16, device=x.device)
    _stream()
    _check("mx_moe_gate_up_swiglu", load().mx_moe_gate_up_swiglu(fmt, _ptr(codes), _ptr(scales), _ptr(x),
                                                                 _ptr(expert_ids), _ptr(h), T, E, topk, I, K))
    return h


def moe_down_combine(fmt: int, codes: torch.Tensor, scales: torch.Tensor, h: torch.Tensor,
                     expert_ids: torch.Tensor, router_weights: torch.Tensor, E: int, N: int,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """out[T][N] fp32 = router-weighted sum of the routed experts' down rows."""
    T, topk = expert_ids.shape
    K = h.shape[-1]
    if out is None:
        out = torch.empty((T, N), dtype=torch.float32, device=h.device)
    _stream()
    _check("mx_moe_down_combine", load().mx_moe_down_combine(fmt, _ptr(codes), _ptr(scales), _ptr(h),
                                                             _ptr(expert_ids), _ptr(router_weights), _ptr(out),
                                                             T, E, topk, N, K))
    return out


def qmm(fmt: int, codes: torch.Tensor, scales: torch.Tensor, X: torch.Tensor, N: int,
        Y: torch.Tensor | None = None) -> torch.Tensor:
    """Y[M][N] bf16 = X (bf16 [M][K]) . W^T with fp32 accumulation."""
    M, K = X.shape
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _stream()
    _check("mx_qmm", load().mx_qmm(fmt, _ptr(codes), _ptr(scales), _ptr(X), _ptr(Y), M, N, K))
    return Y


def qmm_qx(fmt: int, codes: torch.Tensor, scales: torch.Tensor, xcodes: torch.Tensor, xscales: torch.Tensor,
           M: int, N: int, K: int, Y: torch.Tensor | None = None) -> torch.Tensor:
    """Y[M][N] bf16 = Xq . W^T on the block-scaled tensor cores, Xq given as
    block-float codes and scales in the weights' format."""
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=codes.device)
    _stream()
    _check("mx_qmm_qx", load().mx_qmm_qx(fmt, _ptr(codes), _ptr(scales), _ptr(xcodes), _ptr(xscales), _ptr(Y),
                                         M, N, K))
    return Y


MMA_KINDS = {"bf16": (0, 16), "e4m3": (1, 32), "mxfp8": (2, 32), "mxfp4": (3, 64), "nvfp4": (4, 64)}


PEAK_FILLED, PEAK_ROTATE, PEAK_SMEM_STORES, PEAK_TMEM_STORES = 0x100, 0x200, 0x400, 0x800


def mma_peak_tflops(kind: str, iters: int = 8192, reps: int = 5, filled: bool = False, flags: int = 0) -> float:
    """Best of `reps` mx_mma_peak runs, as dense TFLOP/s of the whole GPU
    (filled: random finite operands instead of zeros; flags: the other
    MX_PEAK_* bits)."""
    code, k = MMA_KINDS[kind]
    code |= flags
    if filled:
        code |= PEAK_FILLED
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    best = 0.0
    ms = ctypes.c_float()
    for _ in range(reps):
        _stream()
        _check("mx_mma_peak", load().mx_mma_peak(code, iters, ctypes.byref(ms)))
        best = max(best, 2.0 * 128 * 256 * k * 4 * iters * sms / (ms.value * 1e-3) / 1e12)
    return best


def _workspace(nbytes: int, ws: torch.Tensor | None, device) -> torch.Tensor:
    if nbytes == 0:
        raise ValueError("sizes outside the library's limits")
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws


def moe_qmm(fmt: int, codes: torch.Tensor, scales: torch.Tensor, x: torch.Tensor, expert_ids: torch.Tensor,
            E: int, N: int, y: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y[t][j] bf16 = W_{expert_ids[t][j]} x[t] for many tokens (grouped tensor-core GEMM)."""
    T, K = x.shape
    topk = expert_ids.shape[1]
    if y is None:
        y = torch.empty((T, topk, N), dtype=torch.bfloat16, device=x.device)
    lib = load()
    ws = _workspace(lib.mx_moe_qmm_workspace_size(T, E, topk, K), workspace, x.device)
    _stream()
    _check("mx_moe_qmm", lib.mx_moe_qmm(fmt, _ptr(codes), _ptr(scales), _ptr(x), _ptr(expert_ids), _ptr(y),
                                        T, E, topk, N, K, _ptr(ws), ws.numel()))
    return y


def moe_ffn_prefill_workspace(T: int, E: int, topk: int, H: int, I: int, device="cuda") -> torch.Tensor:
    return _workspace(load().mx_moe_ffn_prefill_workspace_size(T, E, topk, H, I), None, device)


def moe_ffn_prefill(fmt: int, gu_codes: torch.Tensor, gu_scales: torch.Tensor, dn_codes: torch.Tensor,
                    dn_scales: torch.Tensor, x: torch.Tensor, expert_ids: torch.Tensor,
                    router_weights: torch.Tensor, E: int, I: int, out: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None) -> torch.Tensor:
    """out[t] fp32 = sum_j r[t][j] down_e(SwiGLU(gate_up_e x[t])) over many tokens."""
    T, H = x.shape
    topk = expert_ids.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    lib = load()
    ws = _workspace(lib.mx_moe_ffn_prefill_workspace_size(T, E, topk, H, I), workspace, x.device)
    _stream()
    _check("mx_moe_ffn_prefill", lib.mx_moe_ffn_prefill(fmt, _ptr(gu_codes), _ptr(gu_scales), _ptr(dn_codes),
                                                        _ptr(dn_scales), _ptr(x), _ptr(expert_ids),
                                                        _ptr(router_weights), _ptr(out), T, E, topk, H, I,
                                                        _ptr(ws), ws.numel()))
    return out


def quantize(fmt: int, x: torch.Tensor, codes: torch.Tensor | None = None,
             scales: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """bf16 x [M][K] -> (codes, scales) uint8 in the decode's layouts (NVFP4:
    the fp32 tensor scale appended to the scales)."""
    M, K = x.shape
    blk = block_of(fmt)
    if codes is None:
        codes = torch.empty(M * K if fmt == FMT_MXFP8 else M * K // 2, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(M * K // blk + (4 if fmt == FMT_NVFP4 else 0), dtype=torch.uint8, device=x.device)
    _stream()
    _check("mx_quantize", load().mx_quantize(fmt, _ptr(x), _ptr(codes), _ptr(scales), M, K))
    return codes, scales


def dequant(fmt: int, codes: torch.Tensor, scales: torch.Tensor, N: int, K: int,
            W: torch.Tensor | None = None) -> torch.Tensor:
    if W is None:
        W = torch.empty((N, K), dtype=torch.float32, device=codes.device)
    _stream()
    _check("mx_dequant", load().mx_dequant(fmt, _ptr(codes), _ptr(scales), _ptr(W), N, K))
    return W


def swiglu(gu: torch.Tensor, I: int, h: torch.Tensor | None = None) -> torch.Tensor:
    Q = gu.numel() // (2 * I)
    if h is None:
        h = torch.empty((Q, I), dtype=torch.bfloat16, device=gu.device)
    _stream()
    _check("mx_swiglu", load().mx_swiglu(_ptr(gu), _ptr(h), Q, I))
    return h


def moe_combine(yd: torch.Tensor, r: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    T, topk = r.shape
    N = yd.numel() // (T * topk)
    if out is None:
        out = torch.empty((T, N), dtype=torch.float32, device=yd.device)
    _stream()
    _check("mx_moe_combine", load().mx_moe_combine(_ptr(yd), _ptr(r), _ptr(out), T, topk, N))
    return out


def debug_qmm_stall(stall: bool, wait_ns: int = 0) -> None:
    """Test hook: make later tensor-core GEMM launches withhold their
    activation loads so that their bounded waits time out (see mx.h)."""
    _check("mx_debug_qmm_stall", load().mx_debug_qmm_stall(1 if stall else 0, wait_ns))


def device_error() -> int:
    """Synchronise the current stream; return and clear the device error word."""
    _stream()
    s = load().mx_device_error()
    if s < 0:
        _check("mx_device_error", s)
    return s


def raw_call(name: str, *args) -> int:
    """Call an ABI function with raw integer/pointer arguments (tests)."""
    return getattr(load(), name)(*args)
