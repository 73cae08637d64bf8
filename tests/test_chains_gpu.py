"""GPU parity of the general layer (any norm, any activation), the two-layer
fusion chain, SwiGLU and the SwiGLU MLP, called through the C ABI, against
the fp64 oracle on the same seeded inputs.

Sources: the LayerNorm page's fusion chain (LayerNorm -> MatMul -> BiasAdd
-> ReLU -> MatMul -> BiasAdd), the MatMul page's fused GEMM table (ReLU /
GELU / SiLU), the ATB page's Llama2 fusion opportunities (one RMSNorm
feeding the Q/K/V projections; SwiGLU, a SiLU-gated linear transform).

Bar: |y - y_ref| <= 1e-2 + 1e-2 |y_ref| (fp16/bf16 outputs, FP32 statistics
and accumulation).  The chains round their hidden activations to the
16-bit type once on the GPU; the oracle keeps them in fp64, and the bar
covers that rounding (it is about sqrt(F) |h| |W2| u, as for x's rounding
in the single layer).

SwiGLU's h = SiLU(g) u multiplies two products, each within the
single-product bar e = 1e-2 (+ 1e-2 of itself); by the product rule its
error is at most |dh/dg| e_g + |dh/du| e_u with |dh/dg| = |u| |SiLU'(g)|
<= 1.1 |u| and |dh/du| = |SiLU(g)|, so h is held to
    e (1 + 1.1 |u| + |SiLU(g)|) + 1e-2 |h|,
with g and u taken from the (pinned) oracle's single-layer products.
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
NORMS = {"none": (oracle.NORM_NONE, B.NORM_NONE), "layer": (oracle.NORM_LAYER, B.NORM_LAYER),
         "rms": (oracle.NORM_RMS, B.NORM_RMS)}
ACTS = {"none": (oracle.ACT_NONE, B.ACT_NONE), "silu": (oracle.ACT_SILU, B.ACT_SILU),
        "relu": (oracle.ACT_RELU, B.ACT_RELU), "gelu": (oracle.ACT_GELU, B.ACT_GELU)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ngr.build()
    oracle.build()
    torch.cuda.init()
    yield
    B.set_tile_config(-1, 0, 0)


def dev(t):
    return None if t is None else t.cuda()


def check(got, ref, what, atol=None):
    got = got.double().cpu().numpy()
    assert got.shape == ref.shape, what
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > (ATOL if atol is None else atol) + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} / {bad.size} out of tolerance, max err "
                           f"{err.max():.4e} at {np.unravel_index(err.argmax(), err.shape)}")


# ------------------------------------------------------------ general layer
@pytest.mark.parametrize("M", [5, 300], ids=["decode", "tile"])
@pytest.mark.parametrize("act", list(ACTS))
@pytest.mark.parametrize("norm", list(NORMS))
def test_norm_linear_act(norm, act, M):
    K, N = 1000, 520
    for dtype in (torch.float16, torch.bfloat16):
        d = inputs.case("norm_linear", M, K, N, dtype, True, 1e-5, seed=M + len(norm) + len(act),
                        x_mean=1.0, norm=norm, act=act)
        y = ngr.fused_norm_linear_act(dev(d["x"]), dev(d["W"]), norm=NORMS[norm][1],
                                      act=ACTS[act][1], gamma=dev(d["gamma"]),
                                      beta=dev(d["beta"]), bias=dev(d["bias"]), eps=1e-5)
        torch.cuda.synchronize()
        ref = oracle.norm_linear(NORMS[norm][0], ACTS[act][0], d["x"], d["gamma"], d["beta"],
                                 d["W"], d["bias"], 1e-5)
        check(y, ref, f"norm_linear {norm} {act} M={M} {dtype}")


# ----------------------------------------------------------- two-layer chain
@pytest.mark.parametrize("M", [3, 300], ids=["decode", "tile"])
@pytest.mark.parametrize("norm,act,bias", [("layer", "relu", True), ("layer", "gelu", True),
                                           ("rms", "silu", False), ("none", "relu", True),
                                           ("none", "silu", False)])
def test_mlp_chain(norm, act, bias, M):
    K, F = 512, 1000
    d = inputs.case("mlp", M, K, F, torch.float16, bias, 1e-5, seed=M * 3 + len(act),
                    x_mean=0.5, norm=norm, act=act)
    y = ngr.fused_mlp(dev(d["x"]), dev(d["W1"]), dev(d["W2"]), norm=NORMS[norm][1],
                      act=ACTS[act][1], gamma=dev(d["gamma"]), beta=dev(d["beta"]),
                      b1=dev(d["b1"]), b2=dev(d["b2"]), eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.mlp(NORMS[norm][0], ACTS[act][0], d["x"], d["gamma"], d["beta"], d["W1"],
                     d["b1"], d["W2"], d["b2"], 1e-5)
    check(y, ref, f"mlp {norm} {act} bias={bias} M={M}")


def test_mlp_chain_with_h_buffer_matches_workspace_h():
    d = inputs.case("mlp", 200, 256, 520, torch.bfloat16, True, 1e-5, seed=5, norm="layer",
                    act="gelu")
    args = (dev(d["x"]), dev(d["W1"]), dev(d["W2"]))
    kw = dict(norm=B.NORM_LAYER, act=B.ACT_GELU, gamma=dev(d["gamma"]), beta=dev(d["beta"]),
              b1=dev(d["b1"]), b2=dev(d["b2"]))
    h = torch.empty((200, 520), dtype=torch.bfloat16, device="cuda")
    y1 = ngr.fused_mlp(*args, h=h, **kw)
    y2 = ngr.fused_mlp(*args, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    # h is the rounded hidden activation: check it against the single layer
    href = oracle.norm_linear(oracle.NORM_LAYER, oracle.ACT_GELU, d["x"], d["gamma"], d["beta"],
                              d["W1"], d["b1"], 1e-5)
    check(h, href, "mlp hidden activations")


# ------------------------------------------------------------------- SwiGLU
GATED_BN = [192, 224, 256]


def swiglu_atol(norm_id, d, eps):
    """Per-element absolute bar for h (product rule; see the module doc)."""
    g = oracle.norm_linear(norm_id, oracle.ACT_NONE, d["x"], d["gamma"], d["beta"], d["Wg"],
                           None, eps)
    u = oracle.norm_linear(norm_id, oracle.ACT_NONE, d["x"], d["gamma"], d["beta"], d["Wu"],
                           None, eps)
    return ATOL * (1.0 + 1.1 * np.abs(u) + np.abs(g / (1.0 + np.exp(-g))))


def report_plain_bar(h, ref, what):
    """How h fares against the single-product bar 1e-2 + 1e-2 |h| that the
    product-rule bar widens: the number of elements above it and the largest
    ratio of error to that bar.  Printed (pytest -s shows it) and bounded:
    the widening may not hide an error of more than twice the plain bar."""
    err = np.abs(h.double().cpu().numpy() - ref)
    ratio = err / (ATOL + RTOL * np.abs(ref))
    over = int((ratio > 1.0).sum())
    print(f"{what}: {over} of {ratio.size} elements above the plain bar "
          f"({100.0 * over / ratio.size:.4f} %), largest error / plain bar {ratio.max():.2f}")
    assert ratio.max() <= 2.0, (what, float(ratio.max()))
    return over, float(ratio.max())


@pytest.mark.parametrize("bn", GATED_BN)
@pytest.mark.parametrize("norm", list(NORMS))
def test_swiglu_tile_widths(norm, bn):
    """M spans two 256-row pair tiles and a tail; F = 1000 leaves a ragged
    last tile for every width; K = 1000 ends in a 40-column k block."""
    B.set_tile_config(1, bn, 2)
    try:
        M, K, F = 600, 1000, 1000
        for dtype in (torch.float16, torch.bfloat16):
            d = inputs.case("swiglu", M, K, F, dtype, False, 1e-5, seed=bn + len(norm),
                            x_mean=1.0, norm=norm)
            h = ngr.fused_norm_swiglu(dev(d["x"]), dev(d["Wg"]), dev(d["Wu"]),
                                      norm=NORMS[norm][1], gamma=dev(d["gamma"]),
                                      beta=dev(d["beta"]), eps=1e-5)
            torch.cuda.synchronize()
            ref = oracle.swiglu(NORMS[norm][0], d["x"], d["gamma"], d["beta"], d["Wg"], d["Wu"],
                                1e-5)
            check(h, ref, f"swiglu {norm} bn={bn} {dtype}",
                  atol=swiglu_atol(NORMS[norm][0], d, 1e-5))
            report_plain_bar(h, ref, f"swiglu {norm} bn={bn} {dtype}")
    finally:
        B.set_tile_config(-1, 0, 0)


@pytest.mark.parametrize("M", [1, 7, 32, 130])
def test_swiglu_small_batches(M):
    d = inputs.case("swiglu", M, 512, 776, torch.bfloat16, False, 1e-5, seed=M, norm="rms")
    h = ngr.fused_norm_swiglu(dev(d["x"]), dev(d["Wg"]), dev(d["Wu"]), norm=B.NORM_RMS,
                              gamma=dev(d["gamma"]), eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.swiglu(oracle.NORM_RMS, d["x"], d["gamma"], None, d["Wg"], d["Wu"], 1e-5)
    check(h, ref, f"swiglu M={M}", atol=swiglu_atol(oracle.NORM_RMS, d, 1e-5))
    report_plain_bar(h, ref, f"swiglu M={M}")


@pytest.mark.parametrize("M", [4, 300], ids=["decode", "tile"])
@pytest.mark.parametrize("norm", ["rms", "layer"])
def test_mlp_swiglu(norm, M):
    K, F = 512, 1000
    d = inputs.case("mlp_swiglu", M, K, F, torch.float16, False, 1e-5, seed=M + 17, norm=norm)
    y = ngr.fused_mlp_swiglu(dev(d["x"]), dev(d["Wg"]), dev(d["Wu"]), dev(d["Wd"]),
                             norm=NORMS[norm][1], gamma=dev(d["gamma"]), beta=dev(d["beta"]),
                             eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.mlp_swiglu(NORMS[norm][0], d["x"], d["gamma"], d["beta"], d["Wg"], d["Wu"],
                            d["Wd"], 1e-5)
    check(y, ref, f"mlp_swiglu {norm} M={M}")


# ------------------------------------------------ one norm feeding Q, K, V
def test_rmsnorm_qkv_concatenated():
    """RMSNorm feeding the Q, K and V projections in one call: the weights
    concatenated along N; each slice of y matches its own projection."""
    M, K = 300, 1024
    Nq, Nk, Nv = 1024, 256, 256
    d = inputs.case("rmsnorm_linear", M, K, Nq + Nk + Nv, torch.bfloat16, False, 1e-5, seed=99)
    W = d["W"]
    y = ngr.fused_rmsnorm_linear(dev(d["x"]), dev(d["gamma"]), dev(W), None, 1e-5)
    torch.cuda.synchronize()
    offs = [0, Nq, Nq + Nk, Nq + Nk + Nv]
    for i, name in enumerate("qkv"):
        ref = oracle.rmsnorm_linear(d["x"], d["gamma"], W[offs[i]:offs[i + 1]].contiguous(),
                                    None, 1e-5)
        check(y[:, offs[i]:offs[i + 1]], ref, f"qkv {name}")


# ------------------------------------------------------- full-size workloads
def _full(idx_name, count=64):
    w = inputs.BY_NAME[idx_name]
    d = inputs.make(w)
    rows = inputs.sample_rows(w.M, count, seed=7).tolist()
    return w, d, rows


def test_chain_full_size_sampled_rows():
    w, d, rows = _full("chain_ln_linear_bias_relu_linear_bias_f16_m1024_k8192_f8192")
    y = ngr.fused_mlp(dev(d["x"]), dev(d["W1"]), dev(d["W2"]), norm=B.NORM_LAYER,
                      act=B.ACT_RELU, gamma=dev(d["gamma"]), beta=dev(d["beta"]),
                      b1=dev(d["b1"]), b2=dev(d["b2"]), eps=w.eps)
    torch.cuda.synchronize()
    got = y[torch.as_tensor(rows, device="cuda")]
    ref = oracle.mlp(oracle.NORM_LAYER, oracle.ACT_RELU, d["x"], d["gamma"], d["beta"],
                     d["W1"], d["b1"], d["W2"], d["b2"], w.eps, rows)
    check(got, ref, w.name)


def test_mlp_swiglu_full_size_sampled_rows():
    w, d, rows = _full("mlp_swiglu_rms_bf16_m512_k8192_f28672")
    y = ngr.fused_mlp_swiglu(dev(d["x"]), dev(d["Wg"]), dev(d["Wu"]), dev(d["Wd"]),
                             norm=B.NORM_RMS, gamma=dev(d["gamma"]), eps=w.eps)
    torch.cuda.synchronize()
    got = y[torch.as_tensor(rows, device="cuda")]
    ref = oracle.mlp_swiglu(oracle.NORM_RMS, d["x"], d["gamma"], None, d["Wg"], d["Wu"],
                            d["Wd"], w.eps, rows)
    check(got, ref, w.name)


# ------------------------------------------------- norm after the product
@pytest.mark.parametrize("M", [3, 300], ids=["decode", "tile"])
@pytest.mark.parametrize("norm", ["rms", "layer"])
@pytest.mark.parametrize("with_res,with_bias", [(True, False), (False, True), (True, True)])
def test_linear_residual_norm(norm, with_res, with_bias, M):
    K, N = 512, 520
    for dtype in (torch.float16, torch.bfloat16):
        d = inputs.case("norm_linear", M, K, N, dtype, with_bias, 1e-5, seed=M + N + with_res,
                        norm="none")
        g = torch.Generator().manual_seed(M + 1)
        res = (torch.randn((M, N), generator=g) + 1.0).to(dtype) if with_res else None
        gamma = (1.0 + 0.1 * torch.randn((N,), generator=g)).to(dtype)
        beta = (0.1 * torch.randn((N,), generator=g)).to(dtype) if norm == "layer" else None
        h, y = ngr.fused_linear_residual_norm(dev(d["x"]), dev(d["W"]), dev(gamma),
                                              norm=NORMS[norm][1], beta=dev(beta),
                                              bias=dev(d["bias"]), residual=dev(res), eps=1e-5)
        torch.cuda.synchronize()
        href, yref = oracle.linear_residual_norm(NORMS[norm][0], d["x"], d["W"], d["bias"], res,
                                                 gamma, beta, 1e-5)
        check(h, href, f"post-norm h {norm} res={with_res} bias={with_bias} M={M} {dtype}")
        check(y, yref, f"post-norm y {norm} res={with_res} bias={with_bias} M={M} {dtype}")


def test_linear_residual_norm_llama_output_projection():
    """The Llama-70B attention output projection (8192 x 8192) with the
    residual and the following RMSNorm, 512 tokens, sampled rows."""
    M, K, N = 512, 8192, 8192
    d = inputs.case("norm_linear", M, K, N, torch.bfloat16, False, 1e-5, seed=4242)
    g = torch.Generator().manual_seed(4243)
    res = torch.randn((M, N), generator=g).to(torch.bfloat16)
    gamma = (1.0 + 0.1 * torch.randn((N,), generator=g)).to(torch.bfloat16)
    h, y = ngr.fused_linear_residual_norm(dev(d["x"]), dev(d["W"]), dev(gamma), norm=B.NORM_RMS,
                                          residual=dev(res), eps=1e-5)
    torch.cuda.synchronize()
    rows = inputs.sample_rows(M, 64, seed=2).tolist()
    idx = torch.as_tensor(rows, device="cuda")
    href, yref = oracle.linear_residual_norm(oracle.NORM_RMS, d["x"], d["W"], None, res, gamma,
                                             None, 1e-5, rows)
    check(h[idx], href, "llama o-proj h")
    check(y[idx], yref, "llama o-proj y")


@pytest.mark.parametrize("M,N", [(512, 4096), (2048, 8192)], ids=["one-wave", "multi-wave"])
@pytest.mark.parametrize("norm", ["rms", "layer"])
def test_linear_residual_norm_row_mean(norm, M, N):
    """The norm after the product with rows whose mean is well above their
    spread (the residual is centred at 8), on a grid of one wave of tiles and
    on one of several, against the oracle; fp16, whose spacing there (2^-7)
    keeps the rounding of the stored h -- which the norm reads, as the
    unfused norm would -- far inside the bar.  Two calls agree bit for bit."""
    K = 256
    dt = torch.float16
    d = inputs.case("norm_linear", M, K, N, dt, True, 1e-5, seed=M + N, norm="none")
    g = torch.Generator().manual_seed(N)
    res = (torch.randn((M, N), generator=g) + 8.0).to(dt)
    gamma = (1.0 + 0.1 * torch.randn((N,), generator=g)).to(dt)
    beta = (0.1 * torch.randn((N,), generator=g)).to(dt) if norm == "layer" else None
    args = (dev(d["x"]), dev(d["W"]), dev(gamma))
    kw = dict(norm=NORMS[norm][1], beta=dev(beta), bias=dev(d["bias"]), residual=dev(res), eps=1e-5)
    h, y = ngr.fused_linear_residual_norm(*args, **kw)
    h2, y2 = ngr.fused_linear_residual_norm(*args, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(h, h2)
    rows = inputs.sample_rows(M, 64, seed=3).tolist()
    idx = torch.as_tensor(rows, device="cuda")
    href, yref = oracle.linear_residual_norm(NORMS[norm][0], d["x"], d["W"], d["bias"], res,
                                             gamma, beta, 1e-5, rows)
    check(h[idx], href, f"post-norm h {norm} {M}x{K}x{N}")
    check(y[idx], yref, f"post-norm y {norm} {M}x{K}x{N}")
