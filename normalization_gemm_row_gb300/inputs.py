"""Seeded synthetic inputs for the fused pre-norm linear layer.

This module draws random tensors and nothing else: it holds none of the
layer's arithmetic, so both the CUDA path and the fp64 oracle can be fed from
it without sharing any of the method.  Every tensor is drawn on the CPU from
one ``torch.Generator`` per case, in fp32, then cast to the case's 16-bit
type.

The workload shapes and value distributions are the ones the pages quote for
this path ("LayerNorm 融合算子如何让大模型推理再快 15%？深度拆解 ATB 的实现",
§2.1: x [8, 128, 8192] into an 8192x8192 linear; "昇腾CANN的MatMul融合玩法，
让大模型推理快3倍", §二 strategies 1-3: [512, 14336] against [49152, 14336]
weights, and the FFN 14336 -> 49152 -> 14336), at the sizes of the five
workloads below.  No dataset or trained weight is involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

F16, BF16 = torch.float16, torch.bfloat16

# Rows of W drawn per randn call: bounds the fp32 temporary and fixes the
# draw order (changing it changes the tensors).
_CHUNK_ROWS = 2048


@dataclass(frozen=True)
class Workload:
    """One named workload: the op, its sizes and its input distribution."""
    name: str
    op: str                   # layernorm_linear | rmsnorm_linear | linear_silu | ffn |
                              # norm_linear | mlp | swiglu | mlp_swiglu |
                              # linear_residual_norm
    M: int
    K: int
    N: int                    # output features (F, the hidden width, for ffn)
    dtype: torch.dtype
    bias: bool
    eps: float
    seed: int
    x_mean: float = 0.0       # mean offset added to x
    outlier_frac: float = 0.0  # fraction of rows scaled by outlier_scale
    outlier_scale: float = 1.0
    m_choices: tuple = field(default_factory=tuple)  # decode: allowed M
    norm: str = "none"        # norm_linear / mlp / swiglu / mlp_swiglu: none | layer | rms
    act: str = "none"         # norm_linear / mlp: none | silu | relu | gelu

    @property
    def flops(self) -> float:
        """2*M*N*K per product: the FFN and the MLP chain have two, SwiGLU
        two (gate, up) and its MLP form three."""
        g = 2.0 * self.M * self.N * self.K
        return g * {"ffn": 2, "mlp": 2, "swiglu": 2, "mlp_swiglu": 3}.get(self.op, 1)

    def with_m(self, M: int) -> "Workload":
        d = dict(self.__dict__)
        d["M"] = M
        return Workload(**d)


WORKLOADS = [
    Workload("ln_linear_bias_f16_m64_k256_n512", "layernorm_linear",
             64, 256, 512, F16, True, 1e-5, 1234),
    Workload("ln_linear_bias_f16_m1024_k8192_n8192", "layernorm_linear",
             1024, 8192, 8192, F16, True, 1e-5, 1235),
    Workload("rms_linear_f16_m512_k14336_n49152_outliers", "rmsnorm_linear",
             512, 14336, 49152, F16, False, 1e-6, 1236,
             outlier_frac=0.01, outlier_scale=50.0),
    Workload("ffn_linear_silu_linear_f16_m512_k14336_f49152", "ffn",
             512, 14336, 49152, F16, False, 0.0, 1237),
    Workload("decode_ln_linear_bias_bf16_k8192_n28672", "layernorm_linear",
             16, 8192, 28672, BF16, True, 1e-5, 1238, x_mean=3.0,
             m_choices=(1, 4, 16)),
    # LayerNorm -> MatMul -> BiasAdd -> ReLU -> MatMul -> BiasAdd at width 8192
    # (the LayerNorm page's fusion chain), batch as the 8 x 128 token case.
    Workload("chain_ln_linear_bias_relu_linear_bias_f16_m1024_k8192_f8192", "mlp",
             1024, 8192, 8192, F16, True, 1e-5, 1239, norm="layer", act="relu"),
    # RMSNorm -> gate/up -> SiLU-gated product -> down at the Llama2-70B MLP
    # widths (hidden 8192, intermediate 28672).
    Workload("mlp_swiglu_rms_bf16_m512_k8192_f28672", "mlp_swiglu",
             512, 8192, 28672, BF16, False, 1e-5, 1240, norm="rms"),
    # The attention output projection with its residual and the RMSNorm that
    # follows it (Llama2-70B widths).
    Workload("linear_residual_rmsnorm_bf16_m512_k8192_n8192", "linear_residual_norm",
             512, 8192, 8192, BF16, False, 1e-5, 1241, norm="rms"),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _normal(gen, shape, std=1.0, mean=0.0):
    return torch.randn(shape, generator=gen, dtype=torch.float32) * std + mean


def _weight(gen, rows: int, cols: int, std: float, dtype) -> torch.Tensor:
    out = torch.empty((rows, cols), dtype=dtype)
    for r0 in range(0, rows, _CHUNK_ROWS):
        r1 = min(rows, r0 + _CHUNK_ROWS)
        out[r0:r1] = (torch.randn((r1 - r0, cols), generator=gen,
                                  dtype=torch.float32) * std).to(dtype)
    return out


def make(w: Workload, seed: int | None = None) -> dict:
    """Draw the inputs of workload ``w`` (CPU tensors).

    Keys: x [M, K]; gamma, beta [K] (norm ops); W [N, K]; bias [N] or None;
    for ffn: W1 [F, K], W2 [K, F].  Also 'outlier_rows' (long tensor).
    Distributions: x ~ N(x_mean, 1) with a seeded ``outlier_frac`` of rows
    scaled by ``outlier_scale``; gamma ~ 1 + 0.1 N(0,1); beta, bias ~
    0.1 N(0,1); W ~ N(0, 1/K) (W2 ~ N(0, 1/F)).
    """
    g = torch.Generator("cpu")
    g.manual_seed(w.seed if seed is None else seed)
    M, K, N, dt = w.M, w.K, w.N, w.dtype
    x = _normal(g, (M, K), 1.0, w.x_mean)
    n_out = int(round(w.outlier_frac * M))
    outliers = torch.randperm(M, generator=g)[:n_out].sort().values
    if n_out:
        x[outliers] *= w.outlier_scale
    d = {"x": x.to(dt), "outlier_rows": outliers, "gamma": None,
         "beta": None, "bias": None}
    if w.op == "ffn":
        d["W1"] = _weight(g, N, K, K ** -0.5, dt)
        d["W2"] = _weight(g, K, N, N ** -0.5, dt)
        return d
    if w.op == "linear_residual_norm":
        # x; W [N, K]; bias [N]; residual [M, N] ~ N(0, 1); the norm's gamma
        # (and beta) of length N.
        d["W"] = _weight(g, N, K, K ** -0.5, dt)
        if w.bias:
            d["bias"] = (0.1 * _normal(g, (N,))).to(dt)
        d["residual"] = _normal(g, (M, N)).to(dt)
        d["gamma"] = (1.0 + 0.1 * _normal(g, (N,))).to(dt)
        if w.norm == "layer":
            d["beta"] = (0.1 * _normal(g, (N,))).to(dt)
        return d
    if w.op in ("norm_linear", "mlp", "swiglu", "mlp_swiglu"):
        # x; gamma (and beta for layer) by the norm; then the weights:
        # norm_linear W [N, K] (+ bias [N]); mlp W1 [F, K], b1 [F], W2 [K, F],
        # b2 [K]; swiglu Wg, Wu [F, K]; mlp_swiglu also Wd [K, F].
        if w.norm in ("layer", "rms"):
            d["gamma"] = (1.0 + 0.1 * _normal(g, (K,))).to(dt)
        if w.norm == "layer":
            d["beta"] = (0.1 * _normal(g, (K,))).to(dt)
        if w.op == "norm_linear":
            d["W"] = _weight(g, N, K, K ** -0.5, dt)
            if w.bias:
                d["bias"] = (0.1 * _normal(g, (N,))).to(dt)
        elif w.op == "mlp":
            d["W1"] = _weight(g, N, K, K ** -0.5, dt)
            d["W2"] = _weight(g, K, N, N ** -0.5, dt)
            d["b1"] = (0.1 * _normal(g, (N,))).to(dt) if w.bias else None
            d["b2"] = (0.1 * _normal(g, (K,))).to(dt) if w.bias else None
        else:
            d["Wg"] = _weight(g, N, K, K ** -0.5, dt)
            d["Wu"] = _weight(g, N, K, K ** -0.5, dt)
            if w.op == "mlp_swiglu":
                d["Wd"] = _weight(g, K, N, N ** -0.5, dt)
        return d
    if w.op in ("layernorm_linear", "rmsnorm_linear"):
        d["gamma"] = (1.0 + 0.1 * _normal(g, (K,))).to(dt)
    if w.op == "layernorm_linear":
        d["beta"] = (0.1 * _normal(g, (K,))).to(dt)
    d["W"] = _weight(g, N, K, K ** -0.5, dt)
    if w.bias:
        d["bias"] = (0.1 * _normal(g, (N,))).to(dt)
    return d


def case(op: str, M: int, K: int, N: int, dtype=F16, bias: bool = True,
         eps: float = 1e-5, seed: int = 7, x_mean: float = 0.0,
         outlier_frac: float = 0.0, outlier_scale: float = 1.0,
         norm: str = "none", act: str = "none") -> dict:
    """Inputs for an ad-hoc shape (edge-case sweeps) with the same recipe."""
    w = Workload(f"{op}_{M}x{K}x{N}", op, M, K, N, dtype, bias, eps, seed,
                 x_mean=x_mean, outlier_frac=outlier_frac,
                 outlier_scale=outlier_scale, norm=norm, act=act)
    return make(w)


def sample_rows(M: int, count: int, seed: int, always=()) -> torch.Tensor:
    """A seeded sorted sample of ``count`` distinct rows of M, plus the rows
    in ``always`` (e.g. the outlier rows)."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    pick = torch.randperm(M, generator=g)[:min(count, M)]
    rows = torch.cat([pick, torch.as_tensor(list(always), dtype=torch.long)])
    return torch.unique(rows).sort().values


# Edge rows: the degenerate inputs of the normalization (a constant row has
# zero variance; an all-zero row has zero mean square; rows far from zero
# mean stress cancellation in the variance; rows near the top of the fp16
# range stress overflow).  Each kind maps to how the row is drawn.
EDGE_KINDS = ("constant", "zero", "mean1e3", "near_fp16_max")


def with_edge_rows(d: dict, kinds, rows, seed: int = 99, constant: float = 2.5) -> dict:
    """Return a copy of the inputs ``d`` whose x rows ``rows[i]`` are
    replaced by an edge row of kind ``kinds[i]``:
      constant       every element ``constant``;
      zero           every element 0;
      mean1e3        1000 + N(0, 1) (rounded to x's 16-bit type);
      near_fp16_max  2e4 N(0, 1), clipped to +-6e4 (the fp16 maximum is 65504).
    Values are drawn in fp32 from a seeded generator and cast once."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    x = d["x"].clone()
    K = x.shape[1]
    for kind, r in zip(kinds, rows):
        if kind == "constant":
            v = torch.full((K,), float(constant))
        elif kind == "zero":
            v = torch.zeros(K)
        elif kind == "mean1e3":
            v = _normal(g, (K,), 1.0, 1000.0)
        elif kind == "near_fp16_max":
            v = (2e4 * _normal(g, (K,))).clamp(-6e4, 6e4)
        else:
            raise ValueError(kind)
        x[r] = v.to(x.dtype)
    out = dict(d)
    out["x"] = x
    return out
