"""GPU parity: the CUDA library, called through its C ABI, against the fp64
oracle on the same seeded inputs, element by element.

Bar (from the layer's stated tolerance): |y - y_ref| <= 1e-2 + 1e-2 |y_ref|
for fp16/bf16 outputs with FP32 statistics and accumulation.  Small cases
compare every element; the full-size workloads compare a seeded sample of
rows against all N columns (the outlier rows of the RMSNorm workload always
included), in the launch configuration the benchmark times.
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


def to_dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
            for k, v in d.items()}


def assert_parity(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, what
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (
        f"{what}: {bad.sum()} / {bad.size} elements out of tolerance, "
        f"max err {err.max():.4e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def run_op(op, g, eps):
    if op == "layernorm_linear":
        return ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], eps)
    if op == "rmsnorm_linear":
        return ngr.fused_rmsnorm_linear(g["x"], g["gamma"], g["W"], g["bias"], eps)
    if op == "linear_silu":
        return ngr.fused_linear_silu(g["x"], g["W"], g["bias"])
    if op == "ffn":
        return ngr.ffn_linear_silu_linear(g["x"], g["W1"], g["W2"])
    raise ValueError(op)


def ref_op(op, d, eps, rows=None):
    if op == "layernorm_linear":
        return oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d["bias"], eps, rows)
    if op == "rmsnorm_linear":
        return oracle.rmsnorm_linear(d["x"], d["gamma"], d["W"], d["bias"], eps, rows)
    if op == "linear_silu":
        return oracle.linear_silu(d["x"], d["W"], d["bias"], rows)
    if op == "ffn":
        return oracle.ffn(d["x"], d["W1"], d["W2"], rows)
    raise ValueError(op)


# ---------------------------------------------------------------- small cases
def test_smallest_workload_all_rows():
    w = inputs.WORKLOADS[0]
    d = inputs.make(w)
    y = run_op(w.op, to_dev(d), w.eps)
    torch.cuda.synchronize()
    assert_parity(y.double().cpu().numpy(), ref_op(w.op, d, w.eps), w.name)


SHAPES = [(M, K, N) for M in (1, 3, 17, 127, 129, 300)
          for K in (64, 256, 1000) for N in (8, 136, 520)]


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_layernorm_shapes_f16(M, K, N):
    d = inputs.case("layernorm_linear", M, K, N, torch.float16, True, 1e-5,
                    seed=M * 131 + K * 7 + N)
    y = run_op("layernorm_linear", to_dev(d), 1e-5)
    torch.cuda.synchronize()
    assert_parity(y.double().cpu().numpy(), ref_op("layernorm_linear", d, 1e-5),
                  f"LN {M}x{K}x{N}")


OPS = ["layernorm_linear", "rmsnorm_linear", "linear_silu"]
MIXED = [(1, 1000, 520), (16, 256, 136), (32, 512, 264), (33, 64, 8),
         (200, 1000, 136), (300, 256, 520), (64, 4096, 1024)]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("M,K,N", MIXED)
def test_ops_dtypes_bias(op, dtype, M, K, N):
    for bias in (True, False):
        d = inputs.case(op, M, K, N, dtype, bias, 1e-5, seed=M + K + N + bias,
                        x_mean=1.5 if op == "layernorm_linear" else 0.0)
        y = run_op(op, to_dev(d), 1e-5)
        torch.cuda.synchronize()
        assert_parity(y.double().cpu().numpy(), ref_op(op, d, 1e-5),
                      f"{op} {dtype} {M}x{K}x{N} bias={bias}")


@pytest.mark.parametrize("M", [31, 32, 33, 127, 128, 129, 255, 256, 257, 513])
def test_path_boundaries(M):
    """Batch sizes on both sides of each kernel switch (decode up to 32 rows,
    single-CTA tiles up to 128, 256-row CTA-pair tiles above), with K = 576
    (nine 64-column stages) and N = 904 (a last output tile of 8 columns)."""
    K, N = 576, 904
    for op in ("layernorm_linear", "linear_silu"):
        d = inputs.case(op, M, K, N, torch.float16, True, 1e-5, seed=M + 7,
                        x_mean=2.0 if op == "layernorm_linear" else 0.0)
        y = run_op(op, to_dev(d), 1e-5)
        torch.cuda.synchronize()
        assert_parity(y.double().cpu().numpy(), ref_op(op, d, 1e-5), f"{op} M={M}")


@pytest.mark.parametrize("pair", [1, 2], ids=["cta-pair", "multicast"])
def test_many_tiles_per_pair(pair):
    """4096 x 256 -> 2048: more output tiles than resident CTA pairs (or
    clusters), so each runs several tiles through its accumulators; every
    element, on the CTA-pair kernel and on the multicast cluster kernel."""
    M, K, N = 4096, 256, 2048
    d = inputs.case("rmsnorm_linear", M, K, N, torch.bfloat16, True, 1e-5, seed=4096)
    B.set_tile_config(pair, 0, 0)
    try:
        plan = B.tile_plan(B.OP_RMSNORM_LINEAR, M, K, N)
        assert plan["pair"] == pair, plan
        y = run_op("rmsnorm_linear", to_dev(d), 1e-5)
        torch.cuda.synchronize()
    finally:
        B.set_tile_config(-1, 0, 0)
    assert_parity(y.double().cpu().numpy(), ref_op("rmsnorm_linear", d, 1e-5), "4096x256x2048")


@pytest.mark.parametrize("M", [1, 5, 40, 130])
def test_ffn_small(M):
    K, F = 256, 520
    d = inputs.case("ffn", M, K, F, torch.float16, False, 0.0, seed=M)
    y = run_op("ffn", to_dev(d), 0.0)
    torch.cuda.synchronize()
    assert_parity(y.double().cpu().numpy(), ref_op("ffn", d, 0.0), f"ffn M={M}")


def test_empty_batch_is_noop():
    x = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    W = torch.randn(64, 64, device="cuda").half()
    g = torch.ones(64, device="cuda").half()
    y = ngr.fused_layernorm_linear(x, g, g, W, None, 1e-5)
    assert y.shape == (0, 64)


def test_deterministic_repeat():
    d = to_dev(inputs.case("layernorm_linear", 300, 1000, 520, torch.bfloat16, True, seed=3))
    y1 = run_op("layernorm_linear", d, 1e-5)
    y2 = run_op("layernorm_linear", d, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    d = to_dev(inputs.case("layernorm_linear", 16, 8192, 4096, torch.bfloat16, True, seed=4))
    y1 = run_op("layernorm_linear", d, 1e-5)
    y2 = run_op("layernorm_linear", d, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


# Decode grids with several weight tiles per CTA and k groups of unequal
# length: 4 k groups with a short last one (K = 8000: 32 + 32 + 32 + 29
# blocks), 2 groups (K = 4000), 1 group with more tiles than SMs
# (K = 2048, N = 40000); the partials of each tile are summed in k-group
# order, so two calls agree bit for bit.
DECODE_GRID_SHAPES = [(16, 8000, 6000), (1, 8192, 6000), (5, 4000, 20000), (9, 2048, 40000)]


@pytest.mark.parametrize("M,K,N", DECODE_GRID_SHAPES)
@pytest.mark.parametrize("op,dtype", [("layernorm_linear", torch.float16),
                                      ("rmsnorm_linear", torch.bfloat16),
                                      ("linear_silu", torch.bfloat16)], ids=["ln-f16", "rms-bf16", "silu-bf16"])
def test_decode_grids(op, dtype, M, K, N):
    d = inputs.case(op, M, K, N, dtype, True, 1e-5, seed=M + K + N,
                    x_mean=1.0 if op == "layernorm_linear" else 0.0)
    g = to_dev(d)
    y1 = run_op(op, g, 1e-5)
    y2 = run_op(op, g, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "the partial sums are added in a fixed order"
    assert_parity(y1.double().cpu().numpy(), ref_op(op, d, 1e-5), f"{op} {M}x{K}x{N}")


@pytest.mark.parametrize("M", [16, 300])
def test_garbage_workspace(M):
    """A workspace full of garbage (here 0xFF bytes) must not matter: every
    call initialises what it reads from it."""
    d = inputs.case("layernorm_linear", M, 8192, 1024, torch.float16, True, seed=5)
    g = to_dev(d)
    nb = B.ngr_workspace_bytes(B.OP_LAYERNORM_LINEAR, M, 8192, 1024)
    ws = torch.full((nb,), 255, dtype=torch.uint8, device="cuda")
    y = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5,
                                   workspace=ws)
    s = torch.cuda.current_stream().cuda_stream
    assert B.ngr_workspace_error(ws.data_ptr(), s) == 0
    assert_parity(y.double().cpu().numpy(), ref_op("layernorm_linear", d, 1e-5), f"garbage ws M={M}")


def test_side_stream_and_kernel_timing():
    """Calls on a non-default torch stream, with per-kernel timing on."""
    d = inputs.case("layernorm_linear", 300, 1024, 520, torch.float16, True, seed=9)
    g = to_dev(d)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        B.kernel_timing_start(3)
        for _ in range(2):
            y = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g["bias"], 1e-5)
        times = B.kernel_timing_stop()
    side.synchronize()
    assert len(times) == 2 and all(len(t) == 2 for t in times)   # statistics + GEMM
    assert all(0 < t < 100 for row in times for t in row)
    assert B.kernel_timing_stop() == []                          # nothing armed any more
    assert_parity(y.double().cpu().numpy(), ref_op("layernorm_linear", d, 1e-5), "side stream")


def test_row_stats_against_oracle():
    for norm in (oracle.NORM_LAYER, oracle.NORM_RMS):
        for dt in (torch.float16, torch.bfloat16):
            d = inputs.case("layernorm_linear", 37, 8192, 8, dt, True, seed=11, x_mean=3.0)
            st = B.row_stats(d["x"].cuda(), norm, 1e-5).cpu().double().numpy()
            mu, rstd = oracle.row_stats(norm, d["x"], 1e-5)
            assert np.allclose(st[:, 0], mu, rtol=1e-5, atol=1e-5)
            assert np.allclose(st[:, 1], rstd, rtol=1e-4, atol=0)


def test_bounded_wait_reports_timeout():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert B.ngr_debug_bounded_wait(ws.data_ptr(), 2000, s) == 0
    assert B.ngr_workspace_error(ws.data_ptr(), s) == -8
    assert B.ngr_workspace_error(ws.data_ptr(), s) == 0   # cleared by the read
    # the context is still usable afterwards
    d = inputs.make(inputs.WORKLOADS[0])
    y = run_op("layernorm_linear", to_dev(d), 1e-5)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()


# ------------------------------------------------------------- full-size workloads
SAMPLE_ROWS = 64


def full_case(w, M=None):
    if M is not None:
        w = w.with_m(M)
    d = inputs.make(w)
    rows = inputs.sample_rows(w.M, SAMPLE_ROWS, seed=w.seed + 1,
                              always=d["outlier_rows"].tolist())
    return w, d, rows.numpy()


@pytest.mark.parametrize("idx", [1, 2])
def test_full_size_workload_sampled_rows(idx):
    w, d, rows = full_case(inputs.WORKLOADS[idx])
    g = to_dev(d)
    y = run_op(w.op, g, w.eps)
    torch.cuda.synchronize()
    got = y[torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
    del g, y
    assert_parity(got, ref_op(w.op, d, w.eps, rows), w.name)


def test_full_size_ffn_sampled_rows():
    """The largest workload: all N columns of a seeded sample of 64 rows."""
    w = inputs.WORKLOADS[3]
    d = inputs.make(w)
    rows = inputs.sample_rows(w.M, SAMPLE_ROWS, seed=w.seed + 1).numpy()
    g = to_dev(d)
    y = run_op("ffn", g, 0.0)
    torch.cuda.synchronize()
    got = y[torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
    del g, y
    assert_parity(got, ref_op("ffn", d, 0.0, rows), w.name)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_full_size_decode_all_rows(M):
    w, d, _ = full_case(inputs.WORKLOADS[4], M)
    y = run_op(w.op, to_dev(d), w.eps)
    torch.cuda.synchronize()
    assert_parity(y.double().cpu().numpy(), ref_op(w.op, d, w.eps), f"{w.name} M={M}")


# ------------------------------------------------------- inference-mode fold (a7)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("norm", [oracle.NORM_LAYER, oracle.NORM_RMS], ids=["ln", "rms"])
def test_fold_prepare_against_oracle(norm, dtype):
    d = inputs.case("layernorm_linear", 4, 1000, 136, dtype, True, 1e-5, seed=21)
    g = to_dev(d)
    beta = g["beta"] if norm == oracle.NORM_LAYER else None
    Wf, cb = B.fold_prepare(norm, g["gamma"], beta, g["W"], g["bias"])
    torch.cuda.synchronize()
    Wf_ref, c_ref, b_ref = oracle.fold_prepare(norm, d["gamma"], d["beta"] if beta is not None else None,
                                               d["W"], d["bias"])
    # W' is gamma * W rounded once to the 16-bit type: within half a unit in
    # the last place of the exact product (relative 2^-11 / 2^-8), or half the
    # subnormal spacing (2^-25 for fp16) where the product underflows.
    u = 2.0 ** -11 if dtype == torch.float16 else 2.0 ** -8
    tiny = 2.0 ** -25 if dtype == torch.float16 else 2.0 ** -134
    got = Wf.double().cpu().numpy()
    err = np.abs(got - Wf_ref)
    assert (err <= u * np.abs(Wf_ref) + tiny).all(), float((err - u * np.abs(Wf_ref)).max())
    cbh = cb.double().cpu().numpy()
    # c comes from the rounded W' (so it differs from the exact sum by the
    # accumulated roundings); b' from the unrounded product.
    assert np.allclose(cbh[0], c_ref, rtol=1e-2, atol=1e-2)
    assert np.allclose(cbh[1], b_ref, rtol=1e-4, atol=1e-4)


FOLD_SHAPES = [(1, 1000, 136), (16, 4096, 520), (32, 512, 264), (33, 1000, 136),
               (300, 1000, 520), (129, 256, 8)]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("norm", [oracle.NORM_LAYER, oracle.NORM_RMS], ids=["ln", "rms"])
@pytest.mark.parametrize("M,K,N", FOLD_SHAPES)
def test_folded_layer_against_direct_oracle(norm, dtype, M, K, N):
    op = "layernorm_linear" if norm == oracle.NORM_LAYER else "rmsnorm_linear"
    d = inputs.case(op, M, K, N, dtype, True, 1e-5, seed=M * 7 + N,
                    x_mean=3.0 if norm == oracle.NORM_LAYER else 0.0)
    g = to_dev(d)
    Wf, cb = B.fold_prepare(norm, g["gamma"], g["beta"], g["W"], g["bias"])
    y = B.fused_norm_linear_folded(norm, g["x"], Wf, cb, 1e-5)
    torch.cuda.synchronize()
    assert_parity(y.double().cpu().numpy(), ref_op(op, d, 1e-5), f"folded {op} {M}x{K}x{N}")


@pytest.mark.parametrize("idx,M", [(1, None), (2, None), (4, 16), (4, 1)])
def test_folded_full_size(idx, M):
    w, d, rows = full_case(inputs.WORKLOADS[idx], M)
    g = to_dev(d)
    norm = oracle.NORM_RMS if w.op == "rmsnorm_linear" else oracle.NORM_LAYER
    Wf, cb = B.fold_prepare(norm, g["gamma"], g["beta"] if norm == oracle.NORM_LAYER else None,
                            g["W"], g["bias"])
    y = B.fused_norm_linear_folded(norm, g["x"], Wf, cb, w.eps)
    torch.cuda.synchronize()
    got = y[torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
    del g, y, Wf
    assert_parity(got, ref_op(w.op, d, w.eps, rows), f"folded {w.name} M={w.M}")
