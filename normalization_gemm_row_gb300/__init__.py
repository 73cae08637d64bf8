"""Fused pre-norm linear layer for NVIDIA GB300 (sm_103a).

A LayerNorm or RMSNorm row reduction whose normalized rows feed a tcgen05
matrix product directly, with a bias / SiLU epilogue, as hand-written CUDA
kernels behind a C ABI (include/ngr.h).  This package holds the build step,
the ctypes binding (argument marshalling only) and the seeded input
generator used by tests and benchmarks.
"""
from ._build import build, LIB_PATH  # noqa: F401
from .binding import (  # noqa: F401
    NgrError, ffn_linear_silu_linear, fused_layernorm_linear,
    fused_linear_silu, fused_rmsnorm_linear, row_stats)
