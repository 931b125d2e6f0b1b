"""gemm_decode_register_gb300: block-float (MXFP4 / MXFP8 / NVFP4) matmul with
the weights decoded inside hand-written sm_103a CUDA kernels.

The compute path is the C-ABI library built from ``csrc/`` (see
``include/mx.h``); ``ops`` is its thin Python binding.  The CUDA library is
loaded on first use and every call fails loudly if it is missing: there is
no CPU fallback.
"""
from .synth import FMT_MXFP4, FMT_MXFP8, FMT_NVFP4, FMT_NAMES  # noqa: F401

__all__ = ["FMT_MXFP4", "FMT_MXFP8", "FMT_NVFP4", "FMT_NAMES"]
