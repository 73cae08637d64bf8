"""Pins of the fp64 oracle against things other than itself.

Each ``pin_*`` function takes a loaded oracle library handle and raises
``AssertionError`` when the oracle disagrees with what the pages and the
mathematics fix:

- closed-form cases derived by hand (``golden/closed_form_cases.json``);
- invariants of the normalized rows (mean 0, variance sigma^2/(sigma^2+eps),
  mean square ms/(ms+eps));
- RMSNorm's invariance to scaling x (exact at eps = 0);
- special cases that reduce to a library routine: torch's float64
  ``layer_norm``, ``rms_norm``, ``linear`` and ``silu``, numpy's binary16
  decoding;
- brute force on tiny inputs (unfused Python loops, a different evaluation
  order: normalized matrix materialized, then the product);
- row selection: a sampled row equals the same row of a full evaluation;
- the inference-mode fold agrees with the direct form in fp64;
- the activations, the two-layer chain and SwiGLU against torch's float64
  ``relu``, ``gelu`` (exact erf form), ``silu``, ``layer_norm``, ``rms_norm``
  and ``linear``, SwiGLU also against brute force on tiny inputs.

The same functions run against oracle builds with planted mistakes
(``test_oracle_pins.py``) to show that each plausible mistake fails a pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")
DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _t(v, dt):
    return None if v is None else torch.tensor(v, dtype=torch.float64).to(dt)


def _close(got, want, rtol=1e-12, atol=1e-12, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    assert not bad.any(), (f"{what}: max err {err.max():.3e} "
                           f"(worst at {np.unravel_index(err.argmax(), err.shape)})")


def _rand(shape, seed, dt, scale=1.0, mean=0.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float64) * scale
            + mean).to(dt)


def _exact(t):
    """Exact float64 values of a 16-bit tensor via torch's own conversion."""
    return t.to(torch.float64)


# ---------------------------------------------------------------------------
def pin_decode(lib):
    """Every fp16 bit pattern decodes as numpy's binary16 does; every bf16
    pattern as torch's bfloat16 does (library routines)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    t16 = torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16)
    got = oracle.decode(t16, lib)
    want = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin]), "binary16 decode"
    assert np.array_equal(np.isnan(got), np.isnan(want)), "binary16 NaN"
    tb = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    gotb = oracle.decode(tb, lib)
    wantb = tb.to(torch.float64).numpy()
    finb = np.isfinite(wantb)
    assert np.array_equal(gotb[finb], wantb[finb]), "bfloat16 decode"


def pin_closed_forms(lib):
    with open(os.path.join(GOLDEN, "closed_form_cases.json")) as f:
        cases = json.load(f)["cases"]
    env = {"sqrt": math.sqrt, "exp": math.exp}
    for c in cases:
        dt = DT[c["dtype"]]
        x = _t(c["x"], dt)
        want = [[eval(e, {"__builtins__": {}}, env) for e in row]
                for row in c["expected"]]
        if c["op"] == "ffn":
            got = oracle.ffn(x, _t(c["W1"], dt), _t(c["W2"], dt), lib=lib)
        elif c["op"] == "layernorm_linear":
            got = oracle.layernorm_linear(x, _t(c["gamma"], dt),
                                          _t(c["beta"], dt), _t(c["W"], dt),
                                          _t(c["bias"], dt), c["eps"], lib=lib)
        elif c["op"] == "rmsnorm_linear":
            got = oracle.rmsnorm_linear(x, _t(c["gamma"], dt), _t(c["W"], dt),
                                        _t(c["bias"], dt), c["eps"], lib=lib)
        else:
            got = oracle.linear_silu(x, _t(c["W"], dt), _t(c["bias"], dt),
                                     lib=lib)
        _close(got, want, rtol=1e-13, atol=1e-13, what=c["name"])


def pin_layernorm_invariants(lib):
    """gamma=1, beta=0: each normalized row has mean 0 and biased variance
    sigma^2/(sigma^2+eps), sigma^2 from numpy's var (a library routine)."""
    K = 96
    for dt in (torch.float16, torch.bfloat16):
        x = _rand((7, K), 11, dt, 2.0, 3.0)
        one = torch.ones(K, dtype=dt)
        zero = torch.zeros(K, dtype=dt)
        for eps in (0.0, 0.5):
            a = oracle.normalize(oracle.NORM_LAYER, x, one, zero, eps, lib=lib)
            xs = _exact(x).numpy()
            var = xs.var(axis=1)
            _close(a.mean(axis=1), np.zeros(7), atol=1e-12, what="LN mean")
            _close(a.var(axis=1), var / (var + eps), rtol=1e-12,
                   what=f"LN variance eps={eps}")


def pin_rms_invariants(lib):
    """gamma=1: mean(a^2) = ms/(ms+eps); and at eps=0 RMSNorm(c x) equals
    RMSNorm(x) for exact power-of-two scalings c."""
    K = 80
    x = _rand((5, K), 12, torch.float16, 1.5)
    one = torch.ones(K, dtype=torch.float16)
    for eps in (0.0, 2.0):
        a = oracle.normalize(oracle.NORM_RMS, x, one, None, eps, lib=lib)
        ms = (_exact(x).numpy() ** 2).mean(axis=1)
        _close((a ** 2).mean(axis=1), ms / (ms + eps), rtol=1e-12,
               what=f"RMS mean square eps={eps}")
    a0 = oracle.normalize(oracle.NORM_RMS, x, one, None, 0.0, lib=lib)
    for c in (64.0, 0.125):
        xc = (_exact(x) * c).to(torch.float16)
        assert torch.equal(xc.to(torch.float64), _exact(x) * c)
        ac = oracle.normalize(oracle.NORM_RMS, xc, one, None, 0.0, lib=lib)
        _close(ac, a0, rtol=1e-13, atol=1e-13, what=f"RMS scale {c}")


def pin_identity_reduces_to_norm(lib):
    """gamma, beta arbitrary, W = I, no bias: y equals torch's float64
    layer_norm / rms_norm (library routines)."""
    K = 64
    for dt in (torch.float16, torch.bfloat16):
        x = _rand((6, K), 13, dt, 1.0, 0.5)
        g = _rand((K,), 14, dt, 0.1, 1.0)
        b = _rand((K,), 15, dt, 0.1)
        eye = torch.eye(K, dtype=dt)
        y = oracle.layernorm_linear(x, g, b, eye, None, 1e-5, lib=lib)
        ref = F.layer_norm(_exact(x), (K,), _exact(g), _exact(b), 1e-5)
        _close(y, ref.numpy(), rtol=1e-12, atol=1e-12, what="LN vs torch")
        y = oracle.rmsnorm_linear(x, g, eye, None, 1e-6, lib=lib)
        ref = F.rms_norm(_exact(x), (K,), _exact(g), 1e-6)
        _close(y, ref.numpy(), rtol=1e-12, atol=1e-12, what="RMS vs torch")


def pin_full_path_vs_torch(lib):
    """The whole layer against torch float64 layer_norm/rms_norm -> linear
    (+bias) -> silu on a non-square, non-identity case."""
    M, K, N = 9, 40, 24
    for dt in (torch.float16, torch.bfloat16):
        x = _rand((M, K), 16, dt, 1.0, 3.0)
        g = _rand((K,), 17, dt, 0.1, 1.0)
        b = _rand((K,), 18, dt, 0.1)
        W = _rand((N, K), 19, dt, K ** -0.5)
        bias = _rand((N,), 20, dt, 0.1)
        X, G, B, Wd, Bi = map(_exact, (x, g, b, W, bias))
        for act in (oracle.ACT_NONE, oracle.ACT_SILU):
            y = oracle.norm_linear(oracle.NORM_LAYER, act, x, g, b, W, bias,
                                   1e-5, lib=lib)
            ref = F.linear(F.layer_norm(X, (K,), G, B, 1e-5), Wd, Bi)
            ref = F.silu(ref) if act == oracle.ACT_SILU else ref
            _close(y, ref.numpy(), rtol=1e-11, atol=1e-12,
                   what=f"LN layer act={act}")
        y = oracle.rmsnorm_linear(x, g, W, None, 1e-6, lib=lib)
        ref = F.linear(F.rms_norm(X, (K,), G, 1e-6), Wd)
        _close(y, ref.numpy(), rtol=1e-11, atol=1e-12, what="RMS layer")
        y = oracle.linear_silu(x, W, bias, lib=lib)
        ref = F.silu(F.linear(X, Wd, Bi))
        _close(y, ref.numpy(), rtol=1e-11, atol=1e-12, what="linear silu")


def pin_ffn_vs_torch(lib):
    M, K, Fh = 5, 24, 40
    x = _rand((M, K), 21, torch.float16)
    W1 = _rand((Fh, K), 22, torch.float16, K ** -0.5)
    W2 = _rand((K, Fh), 23, torch.float16, Fh ** -0.5)
    y = oracle.ffn(x, W1, W2, lib=lib)
    ref = F.linear(F.silu(F.linear(_exact(x), _exact(W1))), _exact(W2))
    _close(y, ref.numpy(), rtol=1e-11, atol=1e-12, what="ffn vs torch")


def pin_brute_force(lib):
    """Unfused brute force in pure Python on tiny inputs: statistics by
    explicit sums, the normalized matrix materialized, then a triple loop."""
    M, K, N = 3, 6, 4
    x = _rand((M, K), 24, torch.float16, 1.0, 2.0)
    g = _rand((K,), 25, torch.float16, 0.1, 1.0)
    b = _rand((K,), 26, torch.float16, 0.1)
    W = _rand((N, K), 27, torch.float16, 0.5)
    bias = _rand((N,), 28, torch.float16, 0.1)
    X = _exact(x).tolist()
    G, B, Wl, Bi = (_exact(t).tolist() for t in (g, b, W, bias))
    eps = 1e-3
    for norm in ("layer", "rms"):
        A = []
        for i in range(M):
            if norm == "layer":
                mean = math.fsum(X[i]) / K
                var = math.fsum((v - mean) ** 2 for v in X[i]) / K
                A.append([(X[i][k] - mean) / math.sqrt(var + eps) * G[k] + B[k]
                          for k in range(K)])
            else:
                ms = math.fsum(v * v for v in X[i]) / K
                A.append([X[i][k] / math.sqrt(ms + eps) * G[k]
                          for k in range(K)])
        Z = [[math.fsum(A[i][k] * Wl[n][k] for k in range(K)) + Bi[n]
              for n in range(N)] for i in range(M)]
        S = [[z / (1.0 + math.exp(-z)) for z in row] for row in Z]
        nid = oracle.NORM_LAYER if norm == "layer" else oracle.NORM_RMS
        bb = b if norm == "layer" else None
        y = oracle.norm_linear(nid, oracle.ACT_NONE, x, g, bb, W, bias, eps,
                               lib=lib)
        _close(y, Z, rtol=1e-12, atol=1e-12, what=f"brute {norm}")
        y = oracle.norm_linear(nid, oracle.ACT_SILU, x, g, bb, W, bias, eps,
                               lib=lib)
        _close(y, S, rtol=1e-12, atol=1e-12, what=f"brute {norm} silu")


def pin_row_selection(lib):
    """A sampled row evaluates exactly as the same row of the full set."""
    M, K, N = 12, 32, 16
    x = _rand((M, K), 29, torch.bfloat16, 1.0, 1.0)
    g = _rand((K,), 30, torch.bfloat16, 0.1, 1.0)
    b = _rand((K,), 31, torch.bfloat16, 0.1)
    W = _rand((N, K), 32, torch.bfloat16, 0.2)
    bias = _rand((N,), 33, torch.bfloat16, 0.1)
    full = oracle.layernorm_linear(x, g, b, W, bias, 1e-5, lib=lib)
    rows = [0, 5, 11, 7]
    part = oracle.layernorm_linear(x, g, b, W, bias, 1e-5, rows=rows, lib=lib)
    assert np.array_equal(part, full[rows]), "row selection (layer)"
    W1 = _rand((20, K), 34, torch.bfloat16, 0.2)
    W2 = _rand((K, 20), 35, torch.bfloat16, 0.2)
    fullf = oracle.ffn(x, W1, W2, lib=lib)
    partf = oracle.ffn(x, W1, W2, rows=rows, lib=lib)
    assert np.array_equal(partf, fullf[rows]), "row selection (ffn)"
    mu, r = oracle.row_stats(oracle.NORM_LAYER, x, 1e-5, lib=lib)
    mus, rs = oracle.row_stats(oracle.NORM_LAYER, x, 1e-5, rows=rows, lib=lib)
    assert np.array_equal(mus, mu[rows]) and np.array_equal(rs, r[rows])


def pin_fold_identity(lib):
    """rstd (x . W'^T) - rstd mu c + b' equals the direct form to 1e-10."""
    M, K, N = 6, 48, 20
    for norm in (oracle.NORM_LAYER, oracle.NORM_RMS):
        x = _rand((M, K), 36, torch.float16, 1.0, 3.0)
        g = _rand((K,), 37, torch.float16, 0.1, 1.0)
        b = _rand((K,), 38, torch.float16, 0.1)
        W = _rand((N, K), 39, torch.float16, K ** -0.5)
        bias = _rand((N,), 40, torch.float16, 0.1)
        bb = b if norm == oracle.NORM_LAYER else None
        Wf, c, bp = oracle.fold_prepare(norm, g, bb, W, bias, lib=lib)
        for act in (oracle.ACT_NONE, oracle.ACT_SILU):
            yf = oracle.folded_linear(norm, act, x, Wf, c, bp, 1e-5, lib=lib)
            yd = oracle.norm_linear(norm, act, x, g, bb, W, bias, 1e-5,
                                    lib=lib)
            _close(yf, yd, rtol=1e-10, atol=1e-10, what=f"fold norm={norm}")


def pin_stats_vs_numpy(lib):
    """(mu, rstd) against numpy mean/var (library routines), including a
    row with a large mean offset."""
    K = 200
    x = _rand((4, K), 41, torch.bfloat16, 1.0, 3.0)
    xs = _exact(x).numpy()
    mu, r = oracle.row_stats(oracle.NORM_LAYER, x, 1e-5, lib=lib)
    _close(mu, xs.mean(axis=1), rtol=1e-13, what="mu")
    _close(r, 1.0 / np.sqrt(xs.var(axis=1) + 1e-5), rtol=1e-12, what="rstd")
    mu, r = oracle.row_stats(oracle.NORM_RMS, x, 1e-6, lib=lib)
    _close(mu, np.zeros(4), what="rms mu")
    _close(r, 1.0 / np.sqrt((xs ** 2).mean(axis=1) + 1e-6), rtol=1e-12,
           what="rms rstd")


def pin_activations_vs_library(lib):
    """Identity layer (no norm, W = I, no bias): y = act(x) exactly as
    torch's float64 relu / gelu (erf form) / silu, on values that include 0,
    +-1, +-2 and the tails."""
    vals = [0.0, 1.0, -1.0, 2.0, -2.0, 0.5, -0.5, 3.0, -3.0, 8.0, -8.0, 0.125, -6.0, 4.0, -4.0, 1.5]
    K = len(vals)
    x = torch.tensor([vals], dtype=torch.float64).to(torch.float16)
    eye = torch.eye(K, dtype=torch.float16)
    X = _exact(x)
    for act, ref in ((oracle.ACT_RELU, F.relu(X)),
                     (oracle.ACT_GELU, F.gelu(X, approximate="none")),
                     (oracle.ACT_SILU, F.silu(X)),
                     (oracle.ACT_NONE, X)):
        y = oracle.norm_linear(oracle.NORM_NONE, act, x, None, None, eye, None,
                               0.0, lib=lib)
        _close(y, ref.numpy(), rtol=1e-14, atol=1e-15, what=f"act {act}")
    # GELU(1) = Phi(1) and GELU(-1) = -(1 - Phi(1)), Phi from scipy's ndtr
    from scipy.special import ndtr
    y = oracle.norm_linear(oracle.NORM_NONE, oracle.ACT_GELU, x, None, None,
                           eye, None, 0.0, lib=lib)
    _close([y[0][1], y[0][2]], [ndtr(1.0), -ndtr(-1.0)], rtol=1e-14,
           what="GELU(+-1) vs normal CDF")


def pin_mlp_vs_torch(lib):
    """The two-layer chain norm -> linear(+b1) -> act -> linear(+b2) against
    torch float64, for every norm and activation, biases present and not."""
    M, K, Fh, N = 5, 32, 24, 20
    for dt in (torch.float16, torch.bfloat16):
        x = _rand((M, K), 50, dt, 1.0, 2.0)
        g = _rand((K,), 51, dt, 0.1, 1.0)
        b = _rand((K,), 52, dt, 0.1)
        W1 = _rand((Fh, K), 53, dt, K ** -0.5)
        b1 = _rand((Fh,), 54, dt, 0.2)
        W2 = _rand((N, Fh), 55, dt, Fh ** -0.5)
        b2 = _rand((N,), 56, dt, 0.2)
        X, G, B, A1, C1, A2, C2 = map(_exact, (x, g, b, W1, b1, W2, b2))
        acts = {oracle.ACT_NONE: lambda t: t, oracle.ACT_SILU: F.silu,
                oracle.ACT_RELU: F.relu,
                oracle.ACT_GELU: lambda t: F.gelu(t, approximate="none")}
        norms = {oracle.NORM_NONE: lambda t: t,
                 oracle.NORM_LAYER: lambda t: F.layer_norm(t, (K,), G, B, 1e-5),
                 oracle.NORM_RMS: lambda t: F.rms_norm(t, (K,), G, 1e-5)}
        for nid, nf in norms.items():
            for aid, af in acts.items():
                for with_bias in (True, False):
                    bb1, bb2 = (b1, b2) if with_bias else (None, None)
                    y = oracle.mlp(nid, aid, x, g if nid else None,
                                   b if nid == oracle.NORM_LAYER else None,
                                   W1, bb1, W2, bb2, 1e-5, lib=lib)
                    h = af(F.linear(nf(X), A1, C1 if with_bias else None))
                    ref = F.linear(h, A2, C2 if with_bias else None)
                    _close(y, ref.numpy(), rtol=1e-11, atol=1e-12,
                           what=f"mlp norm={nid} act={aid} bias={with_bias}")


def pin_swiglu_vs_torch(lib):
    """SwiGLU h = SiLU(a . Wg^T) * (a . Wu^T) and the Llama MLP h . Wd^T
    against torch float64 for every norm."""
    M, K, Fh, N = 4, 40, 24, 16
    x = _rand((M, K), 60, torch.bfloat16, 1.0, 1.0)
    g = _rand((K,), 61, torch.bfloat16, 0.1, 1.0)
    b = _rand((K,), 62, torch.bfloat16, 0.1)
    Wg = _rand((Fh, K), 63, torch.bfloat16, K ** -0.5)
    Wu = _rand((Fh, K), 64, torch.bfloat16, K ** -0.5)
    Wd = _rand((N, Fh), 65, torch.bfloat16, Fh ** -0.5)
    X, G, B, AG, AU, AD = map(_exact, (x, g, b, Wg, Wu, Wd))
    norms = {oracle.NORM_NONE: lambda t: t,
             oracle.NORM_LAYER: lambda t: F.layer_norm(t, (K,), G, B, 1e-5),
             oracle.NORM_RMS: lambda t: F.rms_norm(t, (K,), G, 1e-5)}
    for nid, nf in norms.items():
        gg = g if nid else None
        bb = b if nid == oracle.NORM_LAYER else None
        a = nf(X)
        href = F.silu(F.linear(a, AG)) * F.linear(a, AU)
        h = oracle.swiglu(nid, x, gg, bb, Wg, Wu, 1e-5, lib=lib)
        _close(h, href.numpy(), rtol=1e-11, atol=1e-12, what=f"swiglu norm={nid}")
        y = oracle.mlp_swiglu(nid, x, gg, bb, Wg, Wu, Wd, 1e-5, lib=lib)
        _close(y, F.linear(href, AD).numpy(), rtol=1e-11, atol=1e-12,
               what=f"mlp_swiglu norm={nid}")


def pin_swiglu_brute_force(lib):
    """SwiGLU in pure Python loops on tiny inputs, RMSNorm first; with the
    gate and up weights equal the result is SiLU(z) * z; with the up weight
    zero it is exactly zero; rows can be sampled."""
    M, K, Fh = 3, 8, 5
    x = _rand((M, K), 66, torch.float16, 1.0, 0.5)
    g = _rand((K,), 67, torch.float16, 0.1, 1.0)
    Wg = _rand((Fh, K), 68, torch.float16, 0.4)
    Wu = _rand((Fh, K), 69, torch.float16, 0.4)
    X, G, AG, AU = (_exact(t).tolist() for t in (x, g, Wg, Wu))
    eps = 1e-3
    H = []
    for i in range(M):
        r = 1.0 / math.sqrt(math.fsum(v * v for v in X[i]) / K + eps)
        a = [X[i][k] * r * G[k] for k in range(K)]
        row = []
        for j in range(Fh):
            zg = math.fsum(a[k] * AG[j][k] for k in range(K))
            zu = math.fsum(a[k] * AU[j][k] for k in range(K))
            row.append(zg / (1.0 + math.exp(-zg)) * zu)
        H.append(row)
    h = oracle.swiglu(oracle.NORM_RMS, x, g, None, Wg, Wu, eps, lib=lib)
    _close(h, H, rtol=1e-12, atol=1e-12, what="swiglu brute force")
    hs = oracle.swiglu(oracle.NORM_RMS, x, g, None, Wg, Wu, eps, rows=[2, 0], lib=lib)
    assert np.array_equal(hs, h[[2, 0]]), "swiglu row selection"
    hz = oracle.swiglu(oracle.NORM_RMS, x, g, None, Wg, torch.zeros_like(Wu), eps, lib=lib)
    assert np.all(hz == 0.0), "swiglu with a zero up projection"
    hgg = oracle.swiglu(oracle.NORM_RMS, x, g, None, Wg, Wg, eps, lib=lib)
    z = oracle.norm_linear(oracle.NORM_RMS, oracle.ACT_NONE, x, g, None, Wg, None, eps, lib=lib)
    _close(hgg, z * z / (1.0 + np.exp(-z)), rtol=1e-12, atol=1e-14, what="swiglu Wu = Wg")


def pin_post_norm_vs_torch(lib):
    """h = x . W^T + bias + residual and y = LayerNorm / RMSNorm of h over N
    against torch float64; without a residual too; and brute force in pure
    Python on a tiny case (statistics by explicit sums over the N outputs)."""
    M, K, N = 6, 40, 24
    for dt in (torch.float16, torch.bfloat16):
        x = _rand((M, K), 70, dt)
        W = _rand((N, K), 71, dt, K ** -0.5)
        bias = _rand((N,), 72, dt, 0.1)
        res = _rand((M, N), 73, dt, 1.0, 2.0)
        g = _rand((N,), 74, dt, 0.1, 1.0)
        b = _rand((N,), 75, dt, 0.1)
        X, A, C, R, G, Bt = map(_exact, (x, W, bias, res, g, b))
        for with_res in (True, False):
            rr = res if with_res else None
            href = F.linear(X, A, C) + (R if with_res else 0.0)
            h, y = oracle.linear_residual_norm(oracle.NORM_RMS, x, W, bias, rr, g, None, 1e-6,
                                               lib=lib)
            _close(h, href.numpy(), rtol=1e-12, atol=1e-12, what="post-norm h")
            _close(y, F.rms_norm(href, (N,), G, 1e-6).numpy(), rtol=1e-11, atol=1e-12,
                   what=f"post RMSNorm res={with_res}")
            h, y = oracle.linear_residual_norm(oracle.NORM_LAYER, x, W, bias, rr, g, b, 1e-5,
                                               lib=lib)
            _close(y, F.layer_norm(href, (N,), G, Bt, 1e-5).numpy(), rtol=1e-11, atol=1e-12,
                   what=f"post LayerNorm res={with_res}")
    # brute force
    M, K, N = 2, 5, 4
    x = _rand((M, K), 76, torch.float16)
    W = _rand((N, K), 77, torch.float16, 0.5)
    res = _rand((M, N), 78, torch.float16)
    g = _rand((N,), 79, torch.float16, 0.1, 1.0)
    Xl, Wl, Rl, Gl = (_exact(t).tolist() for t in (x, W, res, g))
    Y = []
    for i in range(M):
        hrow = [math.fsum(Xl[i][k] * Wl[n][k] for k in range(K)) + Rl[i][n] for n in range(N)]
        r = 1.0 / math.sqrt(math.fsum(v * v for v in hrow) / N + 1e-3)
        Y.append([hrow[n] * r * Gl[n] for n in range(N)])
    _, y = oracle.linear_residual_norm(oracle.NORM_RMS, x, W, None, res, g, None, 1e-3, lib=lib)
    _close(y, Y, rtol=1e-12, atol=1e-12, what="post-norm brute force")


ALL_PINS = [pin_decode, pin_closed_forms, pin_layernorm_invariants,
            pin_rms_invariants, pin_identity_reduces_to_norm,
            pin_full_path_vs_torch, pin_ffn_vs_torch, pin_brute_force,
            pin_row_selection, pin_fold_identity, pin_stats_vs_numpy,
            pin_activations_vs_library, pin_mlp_vs_torch, pin_swiglu_vs_torch,
            pin_swiglu_brute_force, pin_post_norm_vs_torch]
