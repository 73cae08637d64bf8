"""The fp64 oracle against its pins, and proof that the pins bite: each
plausible mistake planted into a copy of the oracle (compiled here, on the
CPU) fails at least one pin."""
import json
import os

import pytest

import oracle
import oracle_pins
from normalization_gemm_row_gb300 import inputs

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


# (description, text in oracle.c, replacement): each one is a mistake a
# careful reader could make while writing the oracle from the pages.
MUTANTS = [
    ("unbiased variance", "v /= (double)K;", "v /= (double)(K - 1);"),
    ("eps outside the square root", "*rstd_out = 1.0 / sqrt(v + eps);",
     "*rstd_out = 1.0 / (sqrt(v) + eps);"),
    ("beta dropped", "a[k] = (x[k] - mu) * rstd * gamma[k] + beta[k];",
     "a[k] = (x[k] - mu) * rstd * gamma[k];"),
    ("mean sign flipped", "a[k] = (x[k] - mu) * rstd * gamma[k] + beta[k];",
     "a[k] = (x[k] + mu) * rstd * gamma[k] + beta[k];"),
    ("gamma dropped from RMSNorm", "a[k] = x[k] * rstd * gamma[k];",
     "a[k] = x[k] * rstd;"),
    ("RMS divides by K-1", "*rstd_out = 1.0 / sqrt(s / (double)K + eps);",
     "*rstd_out = 1.0 / sqrt(s / (double)(K - 1) + eps);"),
    ("bias subtracted", "if (bias) z += bias[n];", "if (bias) z -= bias[n];"),
    ("bias dropped", "if (bias) z += bias[n];", "if (bias) z += 0.0;"),
    ("SiLU sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("activation before bias", "if (bias) z += bias[n];\n        y[n] = activation(act, z);",
     "y[n] = activation(act, z);\n        if (bias) y[n] += bias[n];"),
    ("GELU without the 1/sqrt(2)", "return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
     "return 0.5 * z * (1.0 + erf(z));"),
    ("GELU as z * sigmoid(1.702 z)", "return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
     "return z / (1.0 + exp(-1.702 * z));"),
    ("ReLU leaks", "case NGO_ACT_RELU: return z > 0.0 ? z : 0.0;",
     "case NGO_ACT_RELU: return z > 0.0 ? z : 0.01 * z;"),
    ("SwiGLU gate and up swapped", "h[j] = silu(zg) * zu;", "h[j] = zg * silu(zu);"),
    ("SwiGLU gate not activated", "h[j] = silu(zg) * zu;", "h[j] = zg * zu;"),
    ("chain drops the second bias", "linear_row(h, W2, T, c2, NGO_ACT_NONE, F, N, y + i * N);",
     "linear_row(h, W2, T, NULL, NGO_ACT_NONE, F, N, y + i * N);"),
    ("chain activation after the second layer",
     "linear_row(a, W1, T, c1, act, K, F, h);\n        linear_row(h, W2, T, c2, NGO_ACT_NONE, F, N, y + i * N);",
     "linear_row(a, W1, T, c1, NGO_ACT_NONE, K, F, h);\n        linear_row(h, W2, T, c2, act, F, N, y + i * N);"),
    ("chain skips the norm", "normalize_row(norm, xr, K, mu, rstd, g, b, a);\n        linear_row(a, W1, T, c1, act, K, F, h);",
     "normalize_row(NGO_NORM_NONE, xr, K, mu, rstd, g, b, a);\n        linear_row(a, W1, T, c1, act, K, F, h);"),
    ("binary16 exponent off by one", "v = ldexp((double)(f | 0x400), e - 25);",
     "v = ldexp((double)(f | 0x400), e - 24);"),
    ("FFN without SiLU", "linear_row(xr, W1, T, NULL, NGO_ACT_SILU, K, F, h);",
     "linear_row(xr, W1, T, NULL, NGO_ACT_NONE, K, F, h);"),
    ("sample index used as row", "        row_stats(norm, xr, K, eps, &mu, &rstd);\n        normalize_row(norm, xr, K, mu, rstd, g, b, a);\n        linear_row(a, W, T, bi, act, K, N, y + i * N);",
     "        for (int64_t k = 0; k < K; ++k) xr[k] = T[x[i * K + k]];\n        row_stats(norm, xr, K, eps, &mu, &rstd);\n        normalize_row(norm, xr, K, mu, rstd, g, b, a);\n        linear_row(a, W, T, bi, act, K, N, y + i * N);"),
    ("post-norm drops the residual", "for (int64_t n = 0; n < N; ++n) hr[n] += T[residual[r * N + n]];",
     "for (int64_t n = 0; n < N; ++n) hr[n] += 0.0 * T[residual[r * N + n]];"),
    ("post-norm statistics over N - 1 columns", "row_stats(norm, hr, N, eps, &mu, &rstd);",
     "row_stats(norm, hr, N - 1, eps, &mu, &rstd);"),
    ("post-norm residual after the norm",
     "        if (residual)\n            for (int64_t n = 0; n < N; ++n) hr[n] += T[residual[r * N + n]];\n        double mu, rstd;\n        row_stats(norm, hr, N, eps, &mu, &rstd);",
     "        double mu, rstd;\n        row_stats(norm, hr, N, eps, &mu, &rstd);"),
    ("fold drops the mean term", "double z = rstd * s - rstd * mu * c[n] + bprime[n];",
     "double z = rstd * s + bprime[n];"),
]


@pytest.mark.parametrize("desc,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, desc, find, repl):
    src = open(ORACLE_SRC).read()
    assert src.count(find) == 1, f"mutation site for '{desc}' not unique"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(find, repl))
    so = oracle.compile_oracle(str(mutant), str(tmp_path / "libmutant.so"))
    mlib = oracle.load(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mlib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake: {desc}"


def test_workload_shapes_match_pages():
    """The generator's workloads have the shapes the pages print."""
    with open(os.path.join(oracle_pins.GOLDEN, "page_shapes.json")) as f:
        items = {it["name"]: it for it in json.load(f)["items"]}
    w = inputs.BY_NAME["ln_linear_bias_f16_m1024_k8192_n8192"]
    s = items["layernorm_linear_shape"]
    assert (w.M, w.K) == (s["x"][0] * s["x"][1], s["x"][2])
    assert (w.N, w.K) == tuple(s["W"])
    r = items["rmsnorm_matmul_shape"]
    w = inputs.BY_NAME["rms_linear_f16_m512_k14336_n49152_outliers"]
    assert (w.M, w.K) == tuple(r["x"]) and (w.N, w.K) == tuple(r["W"])
    f = items["ffn_shape"]
    w = inputs.BY_NAME["ffn_linear_silu_linear_f16_m512_k14336_f49152"]
    assert (w.M, w.K) == tuple(f["x"]) and (w.N, w.K) == tuple(f["W1"])
    assert (w.K, w.N) == tuple(f["W2"])
    b = items["layernorm_output_fp32_bytes"]
    n = b["shape"][0] * b["shape"][1] * b["shape"][2] * b["bytes_per_element"]
    assert n == b["mib"] * 2 ** 20


def test_generator_is_seeded_and_shaped():
    w = inputs.BY_NAME["ln_linear_bias_f16_m64_k256_n512"]
    a, b = inputs.make(w), inputs.make(w)
    for k in ("x", "gamma", "beta", "W", "bias"):
        assert a[k].dtype == w.dtype and __import__("torch").equal(a[k], b[k])
    assert tuple(a["x"].shape) == (64, 256) and tuple(a["W"].shape) == (512, 256)
    d = inputs.case("rmsnorm_linear", 200, 64, 16, outlier_frac=0.01,
                    outlier_scale=50.0, bias=False)
    assert d["beta"] is None and d["bias"] is None
    assert len(d["outlier_rows"]) == 2
