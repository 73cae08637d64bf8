"""The workspace-free LayerNorm + linear entry point, for callers that
cannot allocate device memory and therefore cannot hand the library a
workspace.  Called through the C ABI on two calls in a row (the second call
reuses the library's fixed scratch array after the first), its output must
be identical to the regular entry point's wherever both run the same tile
kernel without a K split, and must match the fp64 oracle within the tolerance
of every other parity test.  This file is collected last on purpose, so a run
that stops at the first failure has run everything else.
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


def _close(got, ref, what):
    got = got.double().cpu().numpy()
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), f"{what}: max err {err.max():.3e}"


def _same_kernel_as_workspace_path(M, K, N):
    """True when the workspace entry point runs the tile kernel variant the
    no-allocation path runs (no decode kernel, no K split)."""
    if M <= 32:
        return False
    return B.tile_plan(B.OP_LAYERNORM_LINEAR, M, K, N)["splits"] == 1


@pytest.mark.parametrize("M,K,N,dtype,bias", [
    (300, 1024, 520, torch.float16, True),
    (300, 1000, 520, torch.float16, True),     # K % 64 != 0: ragged last k block
    (300, 1000, 520, torch.bfloat16, True),
    (300, 1000, 520, torch.bfloat16, False),   # no bias
    (1024, 8192, 1024, torch.float16, True),
    (129, 512, 136, torch.float16, False),
    (16, 4096, 1024, torch.bfloat16, True),    # decode-sized M: the workspace path differs
])
def test_noalloc_matches_workspace_entry_point_and_oracle(M, K, N, dtype, bias):
    ngr.build()
    d = inputs.case("layernorm_linear", M, K, N, dtype, bias, 1e-5, seed=M + N + K, x_mean=1.0)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) and k != "outlier_rows" else v)
         for k, v in d.items()}
    code = B.NGR_BF16 if dtype == torch.bfloat16 else B.NGR_F16
    s = torch.cuda.current_stream().cuda_stream
    ref_ws = ngr.fused_layernorm_linear(g["x"], g["gamma"], g["beta"], g["W"], g.get("bias"), 1e-5)
    ref = oracle.layernorm_linear(d["x"], d["gamma"], d["beta"], d["W"], d.get("bias"), 1e-5)
    same = _same_kernel_as_workspace_path(M, K, N)
    bias_ptr = g["bias"].data_ptr() if g.get("bias") is not None else None
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=dtype, device="cuda")
        rc = B.ngr_fused_layernorm_linear_noalloc(
            g["x"].data_ptr(), g["gamma"].data_ptr(), g["beta"].data_ptr(), g["W"].data_ptr(),
            bias_ptr, 1e-5, M, K, N, code, y.data_ptr(), s)
        assert rc == 0, B.status_string(rc)
        assert B.ngr_noalloc_error(s) == 0
        torch.cuda.synchronize()
        what = f"no-alloc call {call} M={M} K={K} N={N} {dtype} bias={bias}"
        if same:
            assert torch.equal(y, ref_ws), what + ": differs from the workspace entry point"
        _close(y, ref, what)


def test_noalloc_rejects_sizes_beyond_its_limit():
    ngr.build()
    # Size checks come before any pointer is looked at: nothing runs here.
    rc = B.ngr_fused_layernorm_linear_noalloc(16, 16, 16, 16, None, 1e-5, 16384 + 1, 64, 64,
                                              0, 16, None)
    assert rc == -2
    rc = B.ngr_fused_layernorm_linear_noalloc(16, 16, 16, 16, None, 1e-5, 64, 16384 + 8, 64,
                                              0, 16, None)
    assert rc == -2
