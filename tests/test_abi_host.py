"""The C-ABI library on the host: it loads, exports every symbol the header
declares, and rejects bad arguments before touching a GPU (no compute call
is made here)."""
import ctypes
import os
import re

import pytest

import normalization_gemm_row_gb300 as pkg
from normalization_gemm_row_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ngr.h")


@pytest.fixture(scope="module")
def lib():
    pkg.build()
    return B.lib()


def header_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ngr_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    syms = header_symbols()
    assert len(syms) >= 10
    for s in syms:
        assert hasattr(lib, s), f"{s} declared in ngr.h but not exported"
    # The binding marshals every declared entry point, and nothing else.
    assert sorted(B.SIGNATURES) == syms


def test_version_and_status_strings(lib):
    assert B.ngr_version() >= 100
    for code, name in B.STATUS.items():
        assert B.ngr_status_string(code).startswith(name)
    assert "unknown" in B.ngr_status_string(12345)


def test_workspace_bytes_layout(lib):
    wb = B.ngr_workspace_bytes
    assert wb(B.OP_LAYERNORM_LINEAR, 0, 8, 8) == 256 + 2 * 256  # header, fp32 gamma, beta
    assert wb(B.OP_LINEAR_SILU, 0, 8, 8) == 256
    big = wb(B.OP_LAYERNORM_LINEAR, 1024, 8192, 8192)
    # header + stats (8 B/row) + fp32 gamma and beta
    assert big == 256 + 1024 * 8 + 2 * 8192 * 4
    assert wb(B.OP_RMSNORM_LINEAR, 1024, 8192, 8192) == big
    assert wb(B.OP_LINEAR_SILU, 1024, 8192, 8192) == 256
    # decode sizes carry split-K partials and counters
    dec = wb(B.OP_LAYERNORM_LINEAR, 16, 8192, 28672)
    tiles = 28672 // 128
    assert dec >= 256 + 256 + 2 * 8192 * 4 + tiles * 4 * 16 * 128 * 4 + tiles * 16
    assert wb(B.OP_LAYERNORM_LINEAR, 17, 64, 64) > wb(B.OP_LAYERNORM_LINEAR, 16, 64, 64)
    # the FFN's H only when it lives in the workspace
    h0 = wb(B.OP_FFN, 512, 14336, 49152, 0)
    h1 = wb(B.OP_FFN, 512, 14336, 49152, 1)
    assert h1 - h0 == 512 * 49152 * 2
    # invalid sizes or ops give 0
    assert wb(B.OP_FFN, -1, 8, 8) == 0 and wb(9, 1, 8, 8) == 0 and wb(0, 1, 0, 8) == 0
    assert wb(-1, 1, 8, 8) == 0


def test_workspace_bytes_padded_shapes(lib):
    wb = B.ngr_workspace_bytes
    a256 = lambda v: (v + 255) // 256 * 256
    M, K, N = 513, 14337, 520
    K8 = 14344
    base = wb(B.OP_LINEAR_SILU, M, K8, N)
    pads = (a256(M * K8 * 2) + a256(N * K8 * 2) + 2 * a256(K8 * 2) + a256(N * 2)
            + a256(M * N * 2))
    assert wb(B.OP_LINEAR_SILU, M, K, N) == base + pads
    # N not a multiple of 8: the output is padded too
    assert wb(B.OP_LAYERNORM_LINEAR, 64, 256, 517) > wb(B.OP_LAYERNORM_LINEAR, 64, 256, 520)
    # the chains pad too: the aligned problem's workspace, then the copies
    # (x, gamma, beta, W1 [F8, K8], b1, W2 [K8, F8], b2, y, and H when the
    # caller keeps it)
    M, K, F = 64, 256, 517
    F8 = 520
    inner = wb(B.OP_FFN, M, K, F8, 0)
    copies = (a256(M * K * 2) + 2 * a256(K * 2) + a256(F8 * K * 2) + a256(F8 * 2)
              + a256(K * F8 * 2) + a256(K * 2) + a256(M * K * 2) + a256(M * F8 * 2))
    assert wb(B.OP_FFN, M, K, F, 0) == inner + copies
    # H in the workspace: the aligned problem holds it, the copies do not
    assert wb(B.OP_FFN, M, K, F, 1) == wb(B.OP_FFN, M, K, F8, 1) + copies - a256(M * F8 * 2)
    for op in (B.OP_MLP, B.OP_SWIGLU, B.OP_MLP_SWIGLU, B.OP_LINEAR_RESIDUAL_NORM):
        assert wb(op, M, 250, 520) > wb(op, M, 256, 520)


def test_unaligned_shapes_need_two_byte_pointers(lib):
    """Any K and N are accepted, but an odd address cannot hold a 16-bit
    element: rejected before anything runs."""
    big = 1 << 24
    odd = A16 + 1
    assert B.ngr_fused_norm_swiglu(0, odd, None, None, A16, A16, 0.0, 4, 60, 64, 0, A16,
                                   A16 * 16, big, None) == -3
    assert B.ngr_fused_mlp(0, 1, A16, None, None, odd, None, A16, None, 0.0, 4, 60, 64, 0,
                           None, A16, A16 * 16, big, None) == -3
    assert B.ngr_fused_norm_linear_folded(1, odd, A16, A16, 1e-5, 4, 60, 64, 0, A16,
                                          A16 * 16, big, None) == -3
    # the prepared fold operands are read with 16-byte accesses
    assert B.ngr_fused_norm_linear_folded(1, A16, A16 + 2, A16, 1e-5, 4, 60, 64, 0, A16,
                                          A16 * 16, big, None) == -3
    assert B.ngr_fold_prepare(1, A16, A16, A16, None, 60, 64, 0, A16 + 2, A16, None) == -3


def test_split_k_reserve(lib):
    """Room for a two-way K split only where the output has few 256 x 448
    tiles: the 1024 x 8192 output (76 tiles) gets none, 512 x 8192 (38)
    does; it is the largest two-way plan over the pair tile widths."""
    wb = B.ngr_workspace_bytes
    a256 = lambda v: (v + 255) // 256 * 256
    assert wb(B.OP_LINEAR_SILU, 1024, 8192, 8192) == 256
    got = wb(B.OP_LINEAR_SILU, 512, 8192, 8192)
    mt = 2
    cnt = max(mt * -(-8192 // tw) * 2 * 4 * (tw // 32) * 4 for tw in (128, 192, 224, 256, 384, 448, 512))
    part = max(mt * -(-8192 // tw) * 2 * 128 * tw * 2 * 4 for tw in (128, 192, 224, 256, 384, 448, 512))
    # ... and the multicast kernel's two-way split of 512 x 464 super-tiles:
    # [super-tiles][4 CTAs][4][15 chunks] counters, 32 x 32 partials each
    sup = 1 * -(-8192 // 464)
    cnt = max(cnt, sup * 4 * 4 * 15 * 4)
    part = max(part, sup * 4 * 4 * 15 * 1024 * 2 * 4)
    assert got == 256 + a256(cnt) + a256(part)
    # none at decode sizes
    assert wb(B.OP_LINEAR_SILU, 16, 8192, 8192) == wb(B.OP_LINEAR_SILU, 16, 8192, 8192, 0)
    # at M <= 128 the single-CTA kernel may split K up to 4 ways: partials of
    # 128-row tiles over the tile widths, when the output has fewer than 256
    # tiles of 128 columns and K has at least 32 k blocks
    cnt1 = max(-(-8192 // tw) * 4 * (tw // 32) * 4 for tw in (128, 192, 224, 256))
    part1 = max(-(-8192 // tw) * 128 * tw * 4 * 4 for tw in (128, 192, 224, 256))
    assert wb(B.OP_LINEAR_SILU, 128, 8192, 8192) == 256 + a256(cnt1) + a256(part1)
    assert wb(B.OP_LINEAR_SILU, 64, 8192, 8192) == 256 + a256(cnt1) + a256(part1)
    assert wb(B.OP_LINEAR_SILU, 128, 1024, 8192) == 256          # K too short to split
    assert wb(B.OP_LINEAR_SILU, 128, 8192, 32768) == 256         # enough tiles
    # the chains reserve for their second product (K output columns)
    assert wb(B.OP_FFN, 512, 4096, 11008) > 256 and wb(B.OP_FFN, 512, 14336, 11008) == 256


def test_tile_plan_rejects(lib):
    plan = (ctypes.c_int * 6)()
    p = ctypes.cast(plan, ctypes.c_void_p)
    assert B.ngr_tile_plan(9, 512, 64, 64, p) == -9
    assert B.ngr_tile_plan(B.OP_SWIGLU, 512, 64, 64, p) == -9
    assert B.ngr_tile_plan(B.OP_LINEAR_SILU, 16, 64, 64, p) == -9     # decode kernel
    assert B.ngr_tile_plan(B.OP_LINEAR_SILU, 512, 64, 64, None) == -1


def test_post_norm_workspace_and_rejections(lib):
    wb = B.ngr_workspace_bytes
    w0 = wb(B.OP_LINEAR_RESIDUAL_NORM, 1024, 8192, 8192, 0)
    assert w0 == 256 + 1024 * 8
    assert wb(B.OP_LINEAR_RESIDUAL_NORM, 1024, 8192, 8192, 1) - w0 == 1024 * 8192 * 2
    assert wb(B.OP_LINEAR_RESIDUAL_NORM, 8, 8192, 8192) > 256 + 8 * 8 + 256   # split-K regions
    f = B.ngr_fused_linear_residual_norm
    big, ws = 1 << 24, A16 * 16
    assert f(0, A16, A16, None, None, A16, None, 1e-5, 4, 64, 64, 0, None, A16, ws, big, None) == -9
    assert f(2, A16, A16, None, None, 0, None, 1e-5, 4, 64, 64, 0, None, A16, ws, big, None) == -1
    assert f(1, A16, A16, None, None, A16, 0, 1e-5, 4, 64, 64, 0, None, A16, ws, big, None) == -1
    assert f(2, A16, A16, None, A16 + 8, A16, None, 1e-5, 4, 64, 64, 0, None, A16, ws, big,
             None) == -3                                               # misaligned residual
    assert f(2, A16, A16, None, A16 + 1, A16, None, 1e-5, 4, 64, 60, 0, None, A16, ws, big,
             None) == -3                               # N % 8 is padded; an odd pointer is not
    assert f(2, A16, A16, None, None, A16, None, 1e-5, 4, 64, 64, 0, None, A16, ws, 300,
             None) == -5
    assert f(2, A16, A16, None, None, A16, None, 1e-5, 0, 64, 64, 0, None, A16, ws, big,
             None) == 0


def test_workspace_bytes_new_ops(lib):
    wb = B.ngr_workspace_bytes
    # the general layer is sized like the LayerNorm layer
    assert wb(B.OP_NORM_LINEAR, 1024, 8192, 8192) == wb(B.OP_LAYERNORM_LINEAR, 1024, 8192, 8192)
    assert wb(B.OP_NORM_LINEAR, 16, 8192, 28672) == wb(B.OP_LAYERNORM_LINEAR, 16, 8192, 28672)
    # the chain adds norm regions to the FFN's, and H only when asked
    m0 = wb(B.OP_MLP, 512, 4096, 11008, 0)
    assert m0 == wb(B.OP_FFN, 512, 4096, 11008, 0) + 2 * 4096 * 4 + 512 * 8
    assert wb(B.OP_MLP, 512, 4096, 11008, 1) - m0 == 512 * 11008 * 2
    # SwiGLU runs on the tile kernel at every M: no split-K regions, no H
    assert wb(B.OP_SWIGLU, 4, 4096, 11008) == 256 + 256 + 2 * 4096 * 4
    assert wb(B.OP_SWIGLU, 4, 4096, 11008, 1) == wb(B.OP_SWIGLU, 4, 4096, 11008)
    # ... but its MLP form keeps the down projection's split-K regions at decode sizes
    assert wb(B.OP_MLP_SWIGLU, 4, 4096, 11008) > wb(B.OP_SWIGLU, 4, 4096, 11008)
    # (its down product, 512 x 4096, has few output tiles: room for a K split)
    assert wb(B.OP_MLP_SWIGLU, 512, 4096, 11008) > wb(B.OP_SWIGLU, 512, 4096, 11008)
    assert (wb(B.OP_MLP_SWIGLU, 512, 4096, 11008, 1) - wb(B.OP_MLP_SWIGLU, 512, 4096, 11008)
            == 512 * 11008 * 2)


def test_new_entry_points_reject(lib):
    big = 1 << 24
    ws = A16 * 16
    # norm / act out of range
    assert B.ngr_fused_norm_linear_act(3, 0, A16, A16, A16, A16, None, 1e-5, 4, 64, 64, 0,
                                       A16, ws, big, None) == -9
    assert B.ngr_fused_norm_linear_act(0, 4, A16, None, None, A16, None, 0.0, 4, 64, 64, 0,
                                       A16, ws, big, None) == -9
    # gamma required with a norm, beta with LayerNorm
    assert B.ngr_fused_norm_linear_act(2, 0, A16, 0, None, A16, None, 1e-5, 4, 64, 64, 0,
                                       A16, ws, big, None) == -1
    assert B.ngr_fused_mlp(1, 2, A16, A16, 0, A16, None, A16, None, 1e-5, 4, 64, 64, 0,
                           None, A16, ws, big, None) == -1
    assert B.ngr_fused_mlp(0, 5, A16, None, None, A16, None, A16, None, 0.0, 4, 64, 64, 0,
                           None, A16, ws, big, None) == -9
    assert B.ngr_fused_mlp(0, 1, A16, None, None, A16, A16 + 4, A16, None, 0.0, 4, 64, 64, 0,
                           None, A16, ws, big, None) == -3           # misaligned b1
    assert B.ngr_fused_norm_swiglu(2, A16, A16, None, A16, 0, 1e-5, 4, 64, 64, 0, A16, ws,
                                   big, None) == -1                  # no up weight
    assert B.ngr_fused_norm_swiglu(0, A16, None, None, A16 + 1, A16, 0.0, 4, 64, 60, 0, A16,
                                   ws, big, None) == -3              # F % 8 padded, odd pointer
    assert B.ngr_fused_norm_swiglu(0, A16, None, None, A16, A16, 0.0, 4, 64, 64, 0, A16, ws,
                                   100, None) == -5                  # workspace too small
    assert B.ngr_fused_mlp_swiglu(2, A16, A16, None, A16, A16, 0, 1e-5, 4, 64, 64, 0, None,
                                  A16, ws, big, None) == -1          # no down weight
    assert B.ngr_fused_mlp_swiglu(2, A16, A16, None, A16, A16, A16, 1e-5, 0, 64, 64, 0, None,
                                  A16, ws, big, None) == 0           # empty batch


A16 = 0x10000  # a fake, 16-byte aligned address: never dereferenced here


@pytest.mark.parametrize("kw,expect", [
    (dict(x=0), -1),                                # NULL x
    (dict(gamma=0), -1),                            # NULL gamma
    (dict(beta=0), -1),                             # NULL beta (LayerNorm)
    (dict(K=12, ws_bytes=600), -5),                 # K % 8: padded copies need workspace
    (dict(N=20, ws_bytes=600), -5),                 # N % 8: likewise
    (dict(K=12, x=A16 + 1), -3),                    # padded path: x not even 2-byte aligned
    (dict(N=20, y=A16 + 1), -3),                    # padded path: y not 2-byte aligned
    (dict(K=12, N=24, y=A16 + 2), -3),              # N % 8 == 0: y stored directly, 16-byte
    (dict(x=A16 + 2), -3),                          # aligned shapes: misaligned x
    (dict(bias=A16 + 8), -3),                       # misaligned bias
    (dict(ws=A16 + 16), -3),                        # workspace not 256-B aligned
    (dict(dtype=3), -4),                            # bad dtype
    (dict(M=-1), -2),                               # negative M
    (dict(K=0), -2),
    (dict(ws_bytes=100), -5),                       # workspace too small
    (dict(ws=0), -5),                               # no workspace
    (dict(M=0), 0),                                 # empty batch is a no-op
])
def test_layernorm_linear_rejects_before_launch(lib, kw, expect):
    a = dict(x=A16, gamma=A16, beta=A16, W=A16, bias=None, eps=1e-5, M=4,
             K=64, N=64, dtype=0, y=A16, ws=A16 * 16, ws_bytes=1 << 20,
             stream=None)
    a.update(kw)
    rc = B.ngr_fused_layernorm_linear(a["x"], a["gamma"], a["beta"], a["W"],
                                      a["bias"], a["eps"], a["M"], a["K"],
                                      a["N"], a["dtype"], a["y"], a["ws"],
                                      a["ws_bytes"], a["stream"])
    assert rc == expect, B.ngr_status_string(rc)


def test_other_entry_points_reject(lib):
    assert B.ngr_fused_rmsnorm_linear(A16, 0, A16, None, 1e-6, 4, 64, 64, 0,
                                      A16, A16 * 16, 1 << 20, None) == -1
    assert B.ngr_fused_linear_silu(A16 + 1, A16, None, 4, 60, 64, 1, A16, A16 * 16,
                                   1 << 20, None) == -3
    assert B.ngr_ffn_linear_silu_linear(A16, A16, 0, 4, 64, 64, 0, None, A16,
                                        A16 * 16, 1 << 20, None) == -1
    # H in the workspace needs room for it
    need = B.ngr_workspace_bytes(B.OP_FFN, 64, 64, 64, 1)
    assert B.ngr_ffn_linear_silu_linear(A16, A16, A16, 64, 64, 64, 0, None,
                                        A16, A16 * 16, need - 256, None) == -5
    assert B.ngr_row_stats(3, A16, 1e-5, 4, 64, 0, A16, None) == -9
    assert B.ngr_row_stats(1, A16, 1e-5, 4, 64, 0, 0, None) == -1
    assert B.ngr_workspace_error(None, None) == -5
    assert B.ngr_debug_bounded_wait(None, 10, None) == -5


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not found"):
        B.lib()


def test_set_tile_config_arguments(lib):
    ok = [(-1, 0, 0), (0, 128, 0), (1, 224, 2), (1, 0, 2), (-1, 256, 1), (2, 0, 0)]
    bad = [(3, 0, 0), (-2, 0, 0), (1, 100, 0), (1, 128, 2), (0, 0, 2), (-1, 0, 3),
           (-1, 0, -1)]
    try:
        for a in ok:
            assert B.ngr_set_tile_config(*a) == 0, a
        for a in bad:
            assert B.ngr_set_tile_config(*a) == -9, a
    finally:
        assert B.ngr_set_tile_config(-1, 0, 0) == 0
