"""GPU parity of every tile-kernel variant the planner can choose, each
forced through ngr_set_tile_config, against the fp64 oracle on the same
seeded inputs: the single-CTA kernel (128-row tiles), the CTA-pair kernel
(256-row tiles, one N sub-tile, two accumulators) and its two-sub-tile form
(256 x 2 BN tiles sharing each x stage, one accumulator).

The shapes span several tiles in M, N and K with ragged tails everywhere:
M = 600 is two full 256-row pair tiles plus 88 rows; K = 1000 ends in a
40-column k block; N = 1000 leaves a last two-sub-tile tile whose second
sub-tile lies wholly past N (skipped) and whose first holds 104 columns, so
that the second CTA's half of it is wholly past N as well.

Bar: |y - y_ref| <= 1e-2 + 1e-2 |y_ref| (fp16/bf16 output, FP32 statistics
and accumulation), every element.
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

# (pair, bn, nsub) as ngr_set_tile_config takes them.
CONFIGS = [(0, 128, 1), (0, 192, 1), (0, 224, 1), (0, 256, 1),
           (1, 128, 1), (1, 192, 1), (1, 224, 1), (1, 256, 1),
           (1, 192, 2), (1, 224, 2), (1, 256, 2)]
IDS = [f"{'pair' if p else 'single'}-bn{bn}x{ns}" for p, bn, ns in CONFIGS]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ngr.build()
    oracle.build()
    torch.cuda.init()
    yield
    B.set_tile_config(-1, 0, 0)


@pytest.fixture(params=CONFIGS, ids=IDS)
def tile_config(request):
    pair, bn, nsub = request.param
    B.set_tile_config(pair, bn, nsub)
    yield request.param
    B.set_tile_config(-1, 0, 0)


def to_dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
            for k, v in d.items()}


def check(got, ref, what):
    got = got.double().cpu().numpy()
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} / {bad.size} out of tolerance, max err "
                           f"{err.max():.4e} at {np.unravel_index(err.argmax(), err.shape)}")


M, K, N = 600, 1000, 1000


def test_layernorm_f16_bias(tile_config):
    d = inputs.case("layernorm_linear", M, K, N, torch.float16, True, 1e-5, seed=11, x_mean=2.0)
    g = to_dev(d)
    y = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5)
    torch.cuda.synchronize()
    check(y, oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5),
          f"LN {tile_config}")


def test_rmsnorm_bf16(tile_config):
    d = inputs.case("rmsnorm_linear", M, K, N + 480, torch.bfloat16, False, 1e-6, seed=12)
    g = to_dev(d)
    y = ngr.fused_rmsnorm_linear(g["x"], g["gamma"], g["W"], None, 1e-6)
    torch.cuda.synchronize()
    check(y, oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], None, 1e-6), f"RMS {tile_config}")


def test_linear_silu_f16(tile_config):
    d = inputs.case("linear_silu", M, K, N, torch.float16, True, 0.0, seed=13)
    g = to_dev(d)
    y = ngr.fused_linear_silu(g["x"], g["W"], g["bias"])
    torch.cuda.synchronize()
    check(y, oracle.linear_silu(d["x"], d["W"], d["bias"]), f"SiLU {tile_config}")


def test_folded_layernorm_bf16(tile_config):
    d = inputs.case("layernorm_linear", M, K, N, torch.bfloat16, True, 1e-5, seed=14, x_mean=3.0)
    g = to_dev(d)
    Wf, cb = B.fold_prepare(oracle.NORM_LAYER, g["gamma"], g["beta"], g["W"], g["bias"])
    y = B.fused_norm_linear_folded(oracle.NORM_LAYER, g["x"], Wf, cb, 1e-5)
    torch.cuda.synchronize()
    check(y, oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5),
          f"folded LN {tile_config}")


def test_ffn_f16(tile_config):
    d = inputs.case("ffn", 300, 512, 1000, torch.float16, False, 0.0, seed=15)
    g = to_dev(d)
    y = ngr.ffn_linear_silu_linear(g["x"], g["W1"], g["W2"])
    torch.cuda.synchronize()
    check(y, oracle.ffn(d["x"], d["W1"], d["W2"]), f"FFN {tile_config}")


# --------------------------------------------------------------- K splits
SPLIT_CONFIGS = [(1, 224, 1), (1, 256, 1), (1, 224, 2), (1, 192, 2), (1, 256, 2)]


@pytest.fixture(params=SPLIT_CONFIGS, ids=[f"pair-bn{bn}x{ns}" for _, bn, ns in SPLIT_CONFIGS])
def split_config(request):
    pair, bn, nsub = request.param
    B.set_tile_config(pair, bn, nsub)
    yield request.param
    B.set_tile_config(-1, 0, 0)


SM, SK, SN = 300, 16384, 1000  # few output tiles, 256 k blocks: the planner splits K in two


def test_split_k_is_planned(split_config):
    plan = B.tile_plan(B.OP_LAYERNORM_LINEAR, SM, SK, SN)
    assert plan["pair"] == 1 and plan["splits"] == 2, plan
    assert plan["bn"] == split_config[1] and plan["nsub"] == split_config[2], plan


def test_split_k_layernorm_and_silu(split_config):
    d = inputs.case("layernorm_linear", SM, SK, SN, torch.bfloat16, True, 1e-5, seed=21,
                    x_mean=2.0)
    g = to_dev(d)
    y = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5)
    torch.cuda.synchronize()
    check(y, oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5),
          f"split LN {split_config}")
    d = inputs.case("linear_silu", SM, SK, SN, torch.float16, True, 0.0, seed=22)
    g = to_dev(d)
    y = ngr.fused_linear_silu(g["x"], g["W"], g["bias"])
    torch.cuda.synchronize()
    check(y, oracle.linear_silu(d["x"], d["W"], d["bias"]), f"split SiLU {split_config}")


def test_split_k_folded_and_post_norm(split_config):
    d = inputs.case("rmsnorm_linear", SM, SK, SN, torch.float16, True, 1e-5, seed=23)
    g = to_dev(d)
    Wf, cb = B.fold_prepare(oracle.NORM_RMS, g["gamma"], None, g["W"], g["bias"])
    y = B.fused_norm_linear_folded(oracle.NORM_RMS, g["x"], Wf, cb, 1e-5)
    torch.cuda.synchronize()
    check(y, oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], d["bias"], 1e-5),
          f"split folded RMS {split_config}")
    gen = torch.Generator().manual_seed(24)
    res = torch.randn((SM, SN), generator=gen).to(torch.float16)
    gam = (1.0 + 0.1 * torch.randn((SN,), generator=gen)).to(torch.float16)
    h, y = ngr.fused_linear_residual_norm(g["x"], g["W"], gam.cuda(), norm=B.NORM_RMS,
                                          bias=g["bias"], residual=res.cuda(), eps=1e-5)
    torch.cuda.synchronize()
    href, yref = oracle.linear_residual_norm(oracle.NORM_RMS, d["x"], d["W"], d["bias"], res, gam,
                                             None, 1e-5)
    check(h, href, f"split post-norm h {split_config}")
    check(y, yref, f"split post-norm y {split_config}")


def test_split_k_is_deterministic():
    d = inputs.case("layernorm_linear", SM, SK, SN, torch.bfloat16, True, 1e-5, seed=25)
    g = to_dev(d)
    ys = [ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5)
          for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])


def test_split_k_default_plan_llama_down_projection():
    """512 x 28672 -> 8192 (448 k blocks, few output tiles): the default plan
    splits K in two, on the multicast kernel (18 super-tiles for 36 clusters)
    or on the CTA-pair kernel (38 wide tiles for 76 pairs) where fewer
    clusters are resident; 512 x 8192 -> 8192 without a norm (128 k blocks)
    does not, its halves would be too short to repay the split.  Sampled
    rows against the oracle."""
    assert B.tile_plan(B.OP_LINEAR_SILU, 512, 8192, 8192)["splits"] == 1
    plan = B.tile_plan(B.OP_LINEAR_SILU, 512, 28672, 8192)
    assert plan["splits"] == 2, plan
    d = inputs.case("linear_silu", 512, 28672, 8192, torch.bfloat16, True, 0.0, seed=26)
    g = to_dev(d)
    y = ngr.fused_linear_silu(g["x"], g["W"], g["bias"])
    torch.cuda.synchronize()
    rows = inputs.sample_rows(512, 12, seed=3, always=(0, 255, 256, 511)).tolist()
    got = y[torch.as_tensor(rows, device="cuda")]
    check(got, oracle.linear_silu(d["x"], d["W"], d["bias"], rows), "split default 512x28672")


# ------------------------------------------- K split on the single-CTA kernel
# Batches of 33-128 rows against a W with few 128-row tiles: the default plan
# splits K on the single-CTA kernel (up to 4 ranges of at least 16 k
# blocks), each range writing FP32 partials and the last of a chunk's ranges
# summing them in range order.  Shapes: 128 and 64 rows at 8192 -> 8192 (a
# 4-way split of 224-column tiles), 96 rows at 4096 -> 4096, a ragged N (a
# last tile of 104 columns) with a 2-way split, a ragged last k block, and
# 33 rows (just above the decode kernel).  Every element against the oracle,
# and two calls agree bit for bit.
SPLIT1_CASES = [("layernorm_linear", 128, 8192, 8192, torch.float16),
                ("rmsnorm_linear", 64, 8192, 8192, torch.bfloat16),
                ("linear_silu", 96, 4096, 4096, torch.float16),
                ("layernorm_linear", 100, 2048, 1000, torch.bfloat16),
                ("rmsnorm_linear", 128, 4000, 520, torch.float16),
                ("linear_silu", 33, 4096, 520, torch.bfloat16)]


@pytest.mark.parametrize("op,M,K,N,dtype", SPLIT1_CASES,
                         ids=[f"{c[0]}-{c[1]}x{c[2]}x{c[3]}-{'bf16' if c[4] == torch.bfloat16 else 'f16'}"
                              for c in SPLIT1_CASES])
def test_single_cta_k_split_against_oracle(op, M, K, N, dtype):
    code = {"layernorm_linear": B.OP_LAYERNORM_LINEAR, "rmsnorm_linear": B.OP_RMSNORM_LINEAR,
            "linear_silu": B.OP_LINEAR_SILU}[op]
    plan = B.tile_plan(code, M, K, N)
    assert plan["pair"] == 0 and plan["splits"] > 1, plan
    d = inputs.case(op, M, K, N, dtype, True, 1e-5 if op != "linear_silu" else 0.0, seed=M + K + N + 41,
                    x_mean=2.0 if op == "layernorm_linear" else 0.0)
    g = to_dev(d)
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
    check(y1, ref, f"single-CTA split {op} {M}x{K}x{N}")


@pytest.mark.parametrize("norm", [oracle.NORM_LAYER, oracle.NORM_RMS], ids=["ln", "rms"])
def test_single_cta_k_split_folded_and_chain(norm):
    M, K, N = 100, 4096, 1000
    op = "layernorm_linear" if norm == oracle.NORM_LAYER else "rmsnorm_linear"
    d = inputs.case(op, M, K, N, torch.float16, True, 1e-5, seed=43 + norm,
                    x_mean=3.0 if norm == oracle.NORM_LAYER else 0.0)
    g = to_dev(d)
    Wf, cb = B.fold_prepare(norm, g["gamma"], g["beta"] if norm == oracle.NORM_LAYER else None,
                            g["W"], g["bias"])
    y = B.fused_norm_linear_folded(norm, g["x"], Wf, cb, 1e-5)
    ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5) \
        if norm == oracle.NORM_LAYER else oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], d["bias"], 1e-5)
    check(y, ref, f"single-CTA split folded {op}")
    # the FFN's second product (1000 -> 4096 columns of K = 1000... here
    # F = 4096 input columns): its K splits too
    f = inputs.case("ffn", M, 1000, 4096, torch.float16, False, 0.0, seed=44 + norm)
    assert B.tile_plan(B.OP_FFN, M, 1000, 4096)["splits"] > 1
    gf = to_dev(f)
    yf = ngr.ffn_linear_silu_linear(gf["x"], gf["W1"], gf["W2"])
    check(yf, oracle.ffn(f["x"], f["W1"], f["W2"]), "single-CTA split FFN")


# The K split at 100 rows through the other entry points whose product may
# split: the MLP chain's and the SwiGLU MLP's second products, the post-GEMM
# norm's product and a plain product (their split counters cleared by a
# memset where the planned product splits, not by the statistics kernel).
@pytest.mark.parametrize("which", ["mlp", "mlp_swiglu", "post_norm", "plain"])
def test_single_cta_k_split_other_entry_points(which):
    M = 100
    if which == "mlp":
        K, F = 512, 4096
        assert B.tile_plan(B.OP_MLP, M, K, F)["splits"] > 1
        d = inputs.case("mlp", M, K, F, torch.float16, True, 1e-5, seed=51, x_mean=0.5,
                        norm="layer", act="relu")
        g = to_dev(d)
        y = ngr.fused_mlp(g["x"], g["W1"], g["W2"], norm=B.NORM_LAYER, act=B.ACT_RELU,
                          gamma=g["gamma"], beta=g["beta"], b1=g["b1"], b2=g["b2"], eps=1e-5)
        ref = oracle.mlp(oracle.NORM_LAYER, oracle.ACT_RELU, d["x"], d["gamma"], d["beta"], d["W1"],
                         d["b1"], d["W2"], d["b2"], 1e-5)
        check(y, ref, "split MLP chain")
    elif which == "mlp_swiglu":
        K, F = 512, 4096
        assert B.tile_plan(B.OP_MLP_SWIGLU, M, K, F)["splits"] > 1
        d = inputs.case("mlp_swiglu", M, K, F, torch.bfloat16, False, 1e-5, seed=52, norm="rms")
        g = to_dev(d)
        y = ngr.fused_mlp_swiglu(g["x"], g["Wg"], g["Wu"], g["Wd"], norm=B.NORM_RMS,
                                 gamma=g["gamma"], beta=None, eps=1e-5)
        ref = oracle.mlp_swiglu(oracle.NORM_RMS, d["x"], d["gamma"], None, d["Wg"], d["Wu"],
                                d["Wd"], 1e-5)
        check(y, ref, "split SwiGLU MLP")
    elif which == "post_norm":
        K, N = 4096, 520
        assert B.tile_plan(B.OP_LINEAR_RESIDUAL_NORM, M, K, N)["splits"] > 1
        d = inputs.case("norm_linear", M, K, N, torch.float16, True, 1e-5, seed=53, norm="none")
        gen = torch.Generator().manual_seed(54)
        res = (torch.randn((M, N), generator=gen) + 1.0).half()
        gamma = (1.0 + 0.1 * torch.randn((N,), generator=gen)).half()
        g = to_dev(d)
        h, y = ngr.fused_linear_residual_norm(g["x"], g["W"], gamma.cuda(), norm=B.NORM_RMS,
                                              bias=g["bias"], residual=res.cuda(), eps=1e-5)
        href, yref = oracle.linear_residual_norm(oracle.NORM_RMS, d["x"], d["W"], d["bias"], res,
                                                 gamma, None, 1e-5)
        check(h, href, "split post-norm h")
        check(y, yref, "split post-norm y")
    else:
        K, N = 4096, 520
        assert B.tile_plan(B.OP_NORM_LINEAR, M, K, N)["splits"] > 1
        d = inputs.case("norm_linear", M, K, N, torch.bfloat16, True, 1e-5, seed=55, norm="none",
                        act="gelu")
        g = to_dev(d)
        y1 = ngr.fused_norm_linear_act(g["x"], g["W"], norm=B.NORM_NONE, act=B.ACT_GELU, bias=g["bias"])
        y2 = ngr.fused_norm_linear_act(g["x"], g["W"], norm=B.NORM_NONE, act=B.ACT_GELU, bias=g["bias"])
        torch.cuda.synchronize()
        assert torch.equal(y1, y2)
        ref = oracle.norm_linear(oracle.NORM_NONE, oracle.ACT_GELU, d["x"], None, None, d["W"],
                                 d["bias"], 0.0)
        check(y1, ref, "split plain product")
