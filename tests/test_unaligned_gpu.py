"""GPU parity of the single-layer entry points on shapes whose K or N is not
a multiple of 8, and on operands whose pointers are only 2-byte aligned,
against the fp64 oracle ("昇腾CANN的MatMul融合玩法，让大模型推理快3倍", §五
optimization 1: a 513 x 14337 activation against a [49152, 14337] weight).

The library pads the rows with zeros in its workspace; the statistics must
count only the K real columns (a LayerNorm whose padding leaked into the
variance would fail here), and y must hold exactly N columns.
Bar: |y - y_ref| <= 1e-2 + 1e-2 |y_ref|.
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


def dev(t):
    return None if t is None else t.cuda()


def check(got, ref, what):
    got = got.double().cpu().numpy()
    assert got.shape == ref.shape, what
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} / {bad.size} out of tolerance, max err "
                           f"{err.max():.4e} at {np.unravel_index(err.argmax(), err.shape)}")


SHAPES = [(513, 1001, 520), (300, 256, 517), (129, 1003, 131), (1, 777, 515), (17, 64, 9),
          (600, 57, 1000), (5, 13, 3)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("op", ["layernorm_linear", "rmsnorm_linear", "linear_silu"])
def test_unaligned_shapes(op, M, K, N):
    for dtype in (torch.float16, torch.bfloat16):
        d = inputs.case(op, M, K, N, dtype, True, 1e-5, seed=M + K + N,
                        x_mean=3.0 if op == "layernorm_linear" else 0.0)
        g = {k: dev(v) for k, v in d.items() if k != "outlier_rows"}
        if op == "layernorm_linear":
            y = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5)
            ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5)
        elif op == "rmsnorm_linear":
            y = ngr.fused_rmsnorm_linear(g["x"], g["gamma"], g["W"], g["bias"], 1e-5)
            ref = oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], d["bias"], 1e-5)
        else:
            y = ngr.fused_linear_silu(g["x"], g["W"], g["bias"])
            ref = oracle.linear_silu(d["x"], d["W"], d["bias"])
        torch.cuda.synchronize()
        check(y, ref, f"{op} {M}x{K}x{N} {dtype}")


@pytest.mark.parametrize("norm,act", [(B.NORM_LAYER, B.ACT_GELU), (B.NORM_RMS, B.ACT_RELU),
                                      (B.NORM_NONE, B.ACT_NONE)])
def test_unaligned_general_layer(norm, act):
    M, K, N = 200, 999, 261
    names = {B.NORM_NONE: "none", B.NORM_LAYER: "layer", B.NORM_RMS: "rms"}
    d = inputs.case("norm_linear", M, K, N, torch.bfloat16, True, 1e-5, seed=norm * 7 + act,
                    x_mean=1.0, norm=names[norm])
    y = ngr.fused_norm_linear_act(dev(d["x"]), dev(d["W"]), norm=norm, act=act,
                                  gamma=dev(d["gamma"]), beta=dev(d["beta"]),
                                  bias=dev(d["bias"]), eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.norm_linear(norm, act, d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5)
    check(y, ref, f"general layer norm={norm} act={act}")


def test_two_byte_aligned_operands():
    """x, W, gamma, beta, bias and y each start one element into a larger
    buffer (2-byte aligned only), with K and N not multiples of 8."""
    M, K, N = 70, 301, 203
    d = inputs.case("layernorm_linear", M, K, N, torch.float16, True, 1e-5, seed=3, x_mean=2.0)

    def shifted(t):
        buf = torch.zeros(t.numel() + 1, dtype=t.dtype, device="cuda")
        buf[1:] = t.reshape(-1).cuda()
        return buf[1:].view(t.shape)

    x, W, gm, bt, bias = (shifted(d[k]) for k in ("x", "W", "gamma", "beta", "bias"))
    ybuf = torch.zeros(M * N + 1, dtype=torch.float16, device="cuda")
    y = ybuf[1:].view(M, N)
    assert x.data_ptr() % 16 != 0 and y.data_ptr() % 16 != 0
    out = ngr.fused_layernorm_linear(x, gm, bt, W, bias, 1e-5, out=y)
    torch.cuda.synchronize()
    assert out.data_ptr() == y.data_ptr() and ybuf[0].item() == 0.0
    ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5)
    check(y, ref, "2-byte aligned operands")


def test_pages_example_shape_sampled_rows():
    """The pages' shape: x [513, 14337] against W [49152, 14337] (SiLU),
    sampled rows against the oracle."""
    M, K, N = 513, 14337, 49152
    d = inputs.case("linear_silu", M, K, N, torch.float16, False, 0.0, seed=513)
    y = ngr.fused_linear_silu(dev(d["x"]), dev(d["W"]), None)
    torch.cuda.synchronize()
    rows = inputs.sample_rows(M, 6, seed=1, always=(0, M - 1)).tolist()
    got = y[torch.as_tensor(rows, device="cuda")]
    ref = oracle.linear_silu(d["x"], d["W"], None, rows)
    check(got, ref, "513 x 14337 -> 49152")


# ----------------------------------------- the chains, SwiGLU, fold, post-norm
# Each of these pads its operands (and the hidden width F) the same way; the
# padded hidden units must contribute nothing, the statistics must count the
# real columns only, and h and y must hold exactly their real columns.
CHAIN_SHAPES = [(5, 250, 517), (300, 1001, 264), (129, 64, 131), (17, 13, 9), (600, 200, 1003)]


@pytest.mark.parametrize("M,K,F", CHAIN_SHAPES)
@pytest.mark.parametrize("norm,act,bias", [("layer", "relu", True), ("rms", "silu", False),
                                           ("none", "gelu", True)])
def test_unaligned_mlp_chain(norm, act, bias, M, K, F):
    ids = {"none": (B.NORM_NONE, oracle.NORM_NONE), "layer": (B.NORM_LAYER, oracle.NORM_LAYER),
           "rms": (B.NORM_RMS, oracle.NORM_RMS)}
    acts = {"relu": (B.ACT_RELU, oracle.ACT_RELU), "silu": (B.ACT_SILU, oracle.ACT_SILU),
            "gelu": (B.ACT_GELU, oracle.ACT_GELU)}
    for dtype in (torch.float16, torch.bfloat16):
        d = inputs.case("mlp", M, K, F, dtype, bias, 1e-5, seed=M + K + F + len(act),
                        x_mean=2.0 if norm == "layer" else 0.0, norm=norm, act=act)
        h = torch.empty((M, F), dtype=dtype, device="cuda")
        y = ngr.fused_mlp(dev(d["x"]), dev(d["W1"]), dev(d["W2"]), norm=ids[norm][0],
                          act=acts[act][0], gamma=dev(d["gamma"]), beta=dev(d["beta"]),
                          b1=dev(d["b1"]), b2=dev(d["b2"]), eps=1e-5, h=h)
        y2 = ngr.fused_mlp(dev(d["x"]), dev(d["W1"]), dev(d["W2"]), norm=ids[norm][0],
                           act=acts[act][0], gamma=dev(d["gamma"]), beta=dev(d["beta"]),
                           b1=dev(d["b1"]), b2=dev(d["b2"]), eps=1e-5)   # H in the workspace
        torch.cuda.synchronize()
        ref = oracle.mlp(ids[norm][1], acts[act][1], d["x"], d["gamma"], d["beta"], d["W1"],
                         d["b1"], d["W2"], d["b2"], 1e-5)
        href = oracle.norm_linear(ids[norm][1], acts[act][1], d["x"], d["gamma"], d["beta"],
                                  d["W1"], d["b1"], 1e-5)
        what = f"mlp {norm} {act} {M}x{K}x{F} {dtype}"
        check(y, ref, what)
        check(h, href, what + " h")
        assert torch.equal(y, y2), what + ": h in the workspace differs"


@pytest.mark.parametrize("M,K,F", [(3, 1001, 517), (260, 250, 1003)])
def test_unaligned_ffn(M, K, F):
    d = inputs.case("ffn", M, K, F, torch.float16, False, 0.0, seed=M + F)
    y = ngr.ffn_linear_silu_linear(dev(d["x"]), dev(d["W1"]), dev(d["W2"]))
    torch.cuda.synchronize()
    check(y, oracle.ffn(d["x"], d["W1"], d["W2"]), f"ffn {M}x{K}x{F}")


def _swiglu_atol(nid, d, eps):
    g = oracle.norm_linear(nid, oracle.ACT_NONE, d["x"], d["gamma"], d["beta"], d["Wg"], None, eps)
    u = oracle.norm_linear(nid, oracle.ACT_NONE, d["x"], d["gamma"], d["beta"], d["Wu"], None, eps)
    return ATOL * (1.0 + 1.1 * np.abs(u) + np.abs(g / (1.0 + np.exp(-g))))


@pytest.mark.parametrize("M,K,F", [(7, 250, 517), (300, 1001, 131), (600, 13, 264)])
@pytest.mark.parametrize("norm", ["rms", "layer"])
def test_unaligned_swiglu_and_mlp(norm, M, K, F):
    bn, on = (B.NORM_RMS, oracle.NORM_RMS) if norm == "rms" else (B.NORM_LAYER, oracle.NORM_LAYER)
    d = inputs.case("mlp_swiglu", M, K, F, torch.bfloat16, False, 1e-5, seed=M * 3 + K,
                    x_mean=1.0, norm=norm)
    g = {k: dev(v) for k, v in d.items() if k != "outlier_rows"}
    h = ngr.fused_norm_swiglu(g["x"], g["Wg"], g["Wu"], norm=bn, gamma=g["gamma"],
                              beta=g["beta"], eps=1e-5)
    h2 = torch.empty_like(h)
    y = ngr.fused_mlp_swiglu(g["x"], g["Wg"], g["Wu"], g["Wd"], norm=bn, gamma=g["gamma"],
                             beta=g["beta"], eps=1e-5, h=h2)
    torch.cuda.synchronize()
    href = oracle.swiglu(on, d["x"], d["gamma"], d["beta"], d["Wg"], d["Wu"], 1e-5)
    got = h.double().cpu().numpy()
    err = np.abs(got - href)
    assert (err <= _swiglu_atol(on, d, 1e-5) + RTOL * np.abs(href)).all(), f"swiglu {norm}"
    assert torch.equal(h, h2)
    yref = oracle.mlp_swiglu(on, d["x"], d["gamma"], d["beta"], d["Wg"], d["Wu"], d["Wd"], 1e-5)
    check(y, yref, f"mlp_swiglu {norm} {M}x{K}x{F}")


@pytest.mark.parametrize("M,K,N", [(1, 1001, 517), (40, 250, 131), (300, 13, 1003)])
@pytest.mark.parametrize("norm", [oracle.NORM_LAYER, oracle.NORM_RMS], ids=["ln", "rms"])
def test_unaligned_fold(norm, M, K, N):
    op = "layernorm_linear" if norm == oracle.NORM_LAYER else "rmsnorm_linear"
    for dtype in (torch.float16, torch.bfloat16):
        d = inputs.case(op, M, K, N, dtype, True, 1e-5, seed=M + K + N + norm)
        g = {k: dev(v) for k, v in d.items() if k != "outlier_rows"}
        Wf, cb = B.fold_prepare(norm, g["gamma"], g["beta"], g["W"], g["bias"])
        assert Wf.shape == (N, (K + 7) // 8 * 8) and cb.shape == (2, (N + 7) // 8 * 8)
        y = B.fused_norm_linear_folded(norm, g["x"], Wf, cb, 1e-5)
        torch.cuda.synchronize()
        assert not Wf[:, K:].any() and not cb[:, N:].any(), "padding of the folded weight"
        ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], 1e-5) \
            if norm == oracle.NORM_LAYER else \
            oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], d["bias"], 1e-5)
        check(y, ref, f"folded {op} {M}x{K}x{N} {dtype}")


@pytest.mark.parametrize("M,K,N", [(3, 250, 517), (300, 1001, 131), (129, 13, 1003)])
@pytest.mark.parametrize("norm", ["rms", "layer"])
def test_unaligned_post_norm(norm, M, K, N):
    bn, on = (B.NORM_RMS, oracle.NORM_RMS) if norm == "rms" else (B.NORM_LAYER, oracle.NORM_LAYER)
    for dtype in (torch.float16, torch.bfloat16):
        d = inputs.case("norm_linear", M, K, N, dtype, True, 1e-5, seed=M + N, norm="none")
        gen = torch.Generator().manual_seed(M + K)
        res = (torch.randn((M, N), generator=gen) + 1.0).to(dtype)
        gamma = (1.0 + 0.1 * torch.randn((N,), generator=gen)).to(dtype)
        beta = (0.1 * torch.randn((N,), generator=gen)).to(dtype) if norm == "layer" else None
        h, y = ngr.fused_linear_residual_norm(dev(d["x"]), dev(d["W"]), dev(gamma), norm=bn,
                                              beta=dev(beta), bias=dev(d["bias"]),
                                              residual=dev(res), eps=1e-5)
        torch.cuda.synchronize()
        href, yref = oracle.linear_residual_norm(on, d["x"], d["W"], d["bias"], res, gamma, beta,
                                                 1e-5)
        check(h, href, f"post-norm h {norm} {M}x{K}x{N} {dtype}")
        check(y, yref, f"post-norm y {norm} {M}x{K}x{N} {dtype}")
