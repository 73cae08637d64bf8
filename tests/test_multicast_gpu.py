"""GPU parity of the multicast cluster kernel (clusters of two CTA pairs that
share each weight box; 512 x 464 super-tiles of sub-tiles 224 + 240),
forced through ngr_set_tile_config(2, 0, 0), against the fp64 oracle.

Shapes cover: a second pair wholly or partly past M (M = 300, 600), several
super-tiles in M (M = 1112), a last super-tile whose second sub-tile is
wholly past N (N = 1000: 72 columns), one whose second sub-tile is partly
past N (N = 700: 236 columns), exactly whole super-tiles (N = 928), a
ragged last k block (K = 1000) and several k blocks per stage ring turn.
Bar: |y - y_ref| <= 1e-2 + 1e-2 |y_ref|, every element.
"""
import numpy as np
import pytest
import torch

import oracle
import normalization_gemm_row_gb300 as ngr
from normalization_gemm_row_gb300 import binding as B
from normalization_gemm_row_gb300 import inputs

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    ngr.build()
    oracle.build()
    torch.cuda.init()
    yield
    B.set_tile_config(-1, 0, 0)


@pytest.fixture
def multicast():
    B.set_tile_config(2, 0, 0)
    yield
    B.set_tile_config(-1, 0, 0)


def check(got, ref, what):
    got = got.double().cpu().numpy()
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} / {bad.size} out of tolerance, max err "
                           f"{err.max():.4e} at {np.unravel_index(err.argmax(), err.shape)}")


SHAPES = [(600, 1000, 1000), (300, 512, 928), (1112, 4096, 700), (600, 2048, 1856)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("op", ["layernorm_linear", "rmsnorm_linear"])
def test_multicast_against_oracle(multicast, op, dtype, M, K, N):
    code = B.OP_LAYERNORM_LINEAR if op == "layernorm_linear" else B.OP_RMSNORM_LINEAR
    assert B.tile_plan(code, M, K, N)["pair"] == 2
    d = inputs.case(op, M, K, N, dtype, op == "layernorm_linear", 1e-5, seed=M + K + N,
                    x_mean=2.0 if op == "layernorm_linear" else 0.0,
                    outlier_frac=0.02 if op == "rmsnorm_linear" else 0.0, outlier_scale=50.0)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
         for k, v in d.items()}
    ws = torch.empty(B.ngr_workspace_bytes(code, M, K, N), dtype=torch.uint8, device="cuda")
    if op == "layernorm_linear":
        y = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5,
                                       workspace=ws)
        ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5)
    else:
        y = ngr.fused_rmsnorm_linear(g["x"], g["gamma"], g["W"], g["bias"], 1e-5, workspace=ws)
        ref = oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], d["bias"], 1e-5)
    s = torch.cuda.current_stream().cuda_stream
    assert B.ngr_workspace_error(ws.data_ptr(), s) == 0, "a bounded wait ran out"
    check(y, ref, f"multicast {op} {dtype} {M}x{K}x{N}")


def test_multicast_repeat_is_deterministic(multicast):
    d = inputs.case("layernorm_linear", 1024, 2048, 1856, torch.float16, True, 1e-5, seed=5)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
         for k, v in d.items()}
    y1 = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5)
    y2 = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


# ------------------------------------------------------ products with no norm
# The multicast kernel without a norm: the transform warps only relay each
# landed stage to the MMA issuer; epilogues with bias, activations and a
# residual, and a chain whose second product takes the first one's output.
PLAIN_SHAPES = [(600, 1000, 1000), (300, 512, 928), (1112, 4096, 700)]


@pytest.mark.parametrize("M,K,N", PLAIN_SHAPES)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_multicast_plain_products(multicast, dtype, M, K, N):
    assert B.tile_plan(B.OP_LINEAR_SILU, M, K, N)["pair"] == 2
    d = inputs.case("linear_silu", M, K, N, dtype, True, 0.0, seed=M + K + N + 3)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
         for k, v in d.items()}
    y = ngr.fused_linear_silu(g["x"], g["W"], g["bias"])
    check(y, oracle.linear_silu(d["x"], d["W"], d["bias"]), f"multicast linear+SiLU {dtype} {M}x{K}x{N}")
    for act, bact in ((oracle.ACT_GELU, B.ACT_GELU), (oracle.ACT_NONE, B.ACT_NONE)):
        y = ngr.fused_norm_linear_act(g["x"], g["W"], norm=B.NORM_NONE, act=bact, bias=g["bias"])
        ref = oracle.norm_linear(oracle.NORM_NONE, act, d["x"], None, None, d["W"], d["bias"], 0.0)
        check(y, ref, f"multicast plain act={act} {dtype} {M}x{K}x{N}")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_multicast_plain_residual_and_chain(multicast, dtype):
    M, K, N = 600, 1000, 1000
    d = inputs.case("norm_linear", M, K, N, dtype, True, 1e-5, seed=77, norm="none")
    gen = torch.Generator().manual_seed(78)
    res = (torch.randn((M, N), generator=gen) + 1.0).to(dtype)
    gamma = (1.0 + 0.1 * torch.randn((N,), generator=gen)).to(dtype)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
         for k, v in d.items()}
    h, y = ngr.fused_linear_residual_norm(g["x"], g["W"], gamma.cuda(), norm=B.NORM_RMS,
                                          bias=g["bias"], residual=res.cuda(), eps=1e-5)
    href, yref = oracle.linear_residual_norm(oracle.NORM_RMS, d["x"], d["W"], d["bias"], res,
                                             gamma, None, 1e-5)
    check(h, href, f"multicast post-norm h {dtype}")
    check(y, yref, f"multicast post-norm y {dtype}")
    f = inputs.case("ffn", M, K, N, dtype, False, 0.0, seed=79)
    gf = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
          for k, v in f.items()}
    yf = ngr.ffn_linear_silu_linear(gf["x"], gf["W1"], gf["W2"])
    check(yf, oracle.ffn(f["x"], f["W1"], f["W2"]), f"multicast FFN {dtype}")


# Several tiles per cluster (or pair) over a short K: the transform warps
# finish their stages long before the first tile's products, then help drain
# the last tile; they must wait for each tile's accumulator in turn.  Every
# element against the oracle, and two calls agree bit for bit.
@pytest.mark.parametrize("config", [(2, 0, 0), (1, 224, 2), (1, 224, 1)],
                         ids=["multicast", "pair-2sub", "pair-1sub"])
@pytest.mark.parametrize("norm", ["layer", "none"])
def test_helpers_wait_every_tile(config, norm):
    M, K, N = 2048, 128, 8192
    B.set_tile_config(*config)
    try:
        if norm == "layer":
            d = inputs.case("layernorm_linear", M, K, N, torch.float16, True, 1e-5, seed=11)
        else:
            d = inputs.case("linear_silu", M, K, N, torch.float16, True, 0.0, seed=12)
        g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
             for k, v in d.items()}
        run = (lambda: ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5)) \
            if norm == "layer" else (lambda: ngr.fused_linear_silu(g["x"], g["W"], g["bias"]))
        y1 = run()
        y2 = run()
        torch.cuda.synchronize()
    finally:
        B.set_tile_config(-1, 0, 0)
    assert torch.equal(y1, y2)
    ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5) \
        if norm == "layer" else oracle.linear_silu(d["x"], d["W"], d["bias"])
    check(y1, ref, f"helpers {config} {norm}")


# ------------------------------------------------- folded weights (inference)
# The folded form (gamma folded into W once; statistics and the folded bias
# in the epilogue) on the multicast kernel: its transform warps only relay
# each landed stage, and the epilogue applies y = rstd acc - rstd mu c + b'.
# Held to the direct layer's oracle (LayerNorm rows at mean 3, where the
# fold's two epilogue terms cancel most).
@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("norm", [oracle.NORM_LAYER, oracle.NORM_RMS], ids=["ln", "rms"])
def test_multicast_folded_against_oracle(multicast, norm, dtype, M, K, N):
    op = "layernorm_linear" if norm == oracle.NORM_LAYER else "rmsnorm_linear"
    d = inputs.case(op, M, K, N, dtype, True, 1e-5, seed=M * 3 + N,
                    x_mean=3.0 if norm == oracle.NORM_LAYER else 0.0,
                    outlier_frac=0.02 if norm == oracle.NORM_RMS else 0.0, outlier_scale=50.0)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
         for k, v in d.items()}
    Wf, cb = B.fold_prepare(norm, g["gamma"], g["beta"] if norm == oracle.NORM_LAYER else None,
                            g["W"], g["bias"])
    y1 = B.fused_norm_linear_folded(norm, g["x"], Wf, cb, 1e-5)
    y2 = B.fused_norm_linear_folded(norm, g["x"], Wf, cb, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    if norm == oracle.NORM_LAYER:
        ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5)
    else:
        ref = oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], d["bias"], 1e-5)
    check(y1, ref, f"multicast folded {op} {dtype} {M}x{K}x{N}")


# ------------------------------------------------- K split on the multicast kernel
# When the super-tiles fill at most half of the clusters, the multicast
# kernel splits K in two: each half writes FP32 partials of its 32 x 32
# chunks, and the last of a chunk's two units sums them in range order and
# finishes it.  Shapes: a second pair partly past M (300 rows), a last
# super-tile partly past N (1000 and 928 columns), several m super-tiles
# (1112 rows), and a full 8192-column output (18 super-tiles).  Every element
# against the oracle, and two calls agree bit for bit.
MC_SPLIT_SHAPES = [(600, 4096, 1000), (300, 8192, 928), (1112, 4096, 700), (512, 4096, 8192)]


@pytest.mark.parametrize("M,K,N", MC_SPLIT_SHAPES)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("op", ["layernorm_linear", "rmsnorm_linear", "linear_silu"])
def test_multicast_k_split_against_oracle(multicast, op, dtype, M, K, N):
    code = {"layernorm_linear": B.OP_LAYERNORM_LINEAR, "rmsnorm_linear": B.OP_RMSNORM_LINEAR,
            "linear_silu": B.OP_LINEAR_SILU}[op]
    plan = B.tile_plan(code, M, K, N)
    if N == 8192 and plan["splits"] == 1:
        # 18 super-tiles split in two need 36 resident clusters of four
        pytest.skip(f"fewer than 36 resident clusters of four on this device: {plan}")
    assert plan["pair"] == 2 and plan["splits"] == 2, plan
    d = inputs.case(op, M, K, N, dtype, op != "rmsnorm_linear", 1e-5 if op != "linear_silu" else 0.0,
                    seed=M + K + N + 61, x_mean=2.0 if op == "layernorm_linear" else 0.0,
                    outlier_frac=0.02 if op == "rmsnorm_linear" else 0.0, outlier_scale=50.0)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
         for k, v in d.items()}
    ws = torch.empty(B.ngr_workspace_bytes(code, M, K, N), dtype=torch.uint8, device="cuda")
    if op == "layernorm_linear":
        run = lambda: ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5,
                                                 workspace=ws)
        ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5)
    elif op == "rmsnorm_linear":
        run = lambda: ngr.fused_rmsnorm_linear(g["x"], g["gamma"], g["W"], g["bias"], 1e-5, workspace=ws)
        ref = oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], d["bias"], 1e-5)
    else:
        run = lambda: ngr.fused_linear_silu(g["x"], g["W"], g["bias"], workspace=ws)
        ref = oracle.linear_silu(d["x"], d["W"], d["bias"])
    y1 = run()
    y2 = run()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream().cuda_stream
    assert B.ngr_workspace_error(ws.data_ptr(), s) == 0, "a bounded wait ran out"
    assert torch.equal(y1, y2)
    check(y1, ref, f"multicast K split {op} {dtype} {M}x{K}x{N}")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_multicast_k_split_residual_and_fold(multicast, dtype):
    M, K, N = 300, 4096, 1000
    assert B.tile_plan(B.OP_LINEAR_RESIDUAL_NORM, M, K, N)["splits"] == 2
    d = inputs.case("norm_linear", M, K, N, dtype, True, 1e-5, seed=71, norm="none")
    gen = torch.Generator().manual_seed(72)
    res = (torch.randn((M, N), generator=gen) + 1.0).to(dtype)
    gamma = (1.0 + 0.1 * torch.randn((N,), generator=gen)).to(dtype)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
         for k, v in d.items()}
    h, y = ngr.fused_linear_residual_norm(g["x"], g["W"], gamma.cuda(), norm=B.NORM_RMS,
                                          bias=g["bias"], residual=res.cuda(), eps=1e-5)
    href, yref = oracle.linear_residual_norm(oracle.NORM_RMS, d["x"], d["W"], d["bias"], res,
                                             gamma, None, 1e-5)
    check(h, href, f"multicast K split post-norm h {dtype}")
    check(y, yref, f"multicast K split post-norm y {dtype}")
    e = inputs.case("layernorm_linear", M, K, N, dtype, True, 1e-5, seed=73, x_mean=3.0)
    ge = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
          for k, v in e.items()}
    Wf, cb = B.fold_prepare(oracle.NORM_LAYER, ge["gamma"], ge["beta"], ge["W"], ge["bias"])
    yf = B.fused_norm_linear_folded(oracle.NORM_LAYER, ge["x"], Wf, cb, 1e-5)
    check(yf, oracle.layernorm_linear(e["x"], e["gamma"], e["beta"], e["W"], e["bias"], 1e-5),
          f"multicast K split folded {dtype}")
