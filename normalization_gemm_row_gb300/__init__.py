"""Fused pre-norm linear layer for NVIDIA GB300 (sm_103a).

A LayerNorm or RMSNorm row reduction whose normalized rows feed a tcgen05
matrix product directly, with a bias / activation epilogue (and the
two-layer chains and SwiGLU built on it), as hand-written CUDA kernels
behind a C ABI (include/ngr.h).  This package holds the build step,
the ctypes binding (argument marshalling only) and the seeded input
generator used by tests and benchmarks.
"""
from ._build import build, LIB_PATH  # noqa: F401
from .binding import (  # noqa: F401
    ACT_GELU, ACT_NONE, ACT_RELU, ACT_SILU, NORM_LAYER, NORM_NONE, NORM_RMS,
    NgrError, ffn_linear_silu_linear, fold_prepare, fused_layernorm_linear,
    fused_linear_residual_norm, fused_linear_silu, fused_mlp, fused_mlp_swiglu,
    fused_norm_linear_act,
    fused_norm_linear_folded, fused_norm_swiglu, fused_rmsnorm_linear,
    row_stats)
