"""ctypes binding of the CUDA library (the C ABI declared in include/ngr.h).

Two layers, both argument marshalling only -- every step of the layer runs in
the library's kernels:

- ``ngr_*`` functions with the C names and C arguments (device pointers as
  integers, sizes, dtype code, stream handle), returning the status code;
- tensor-level helpers with the op names (``fused_layernorm_linear`` ...)
  that take CUDA torch tensors, allocate the output and workspace with torch
  when not given, pass pointers and the current stream, and raise
  ``NgrError`` on a non-zero status.

There is no fallback: if the shared library is missing or fails to load,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB_PATH

NGR_F16, NGR_BF16 = 0, 1
OP_LAYERNORM_LINEAR, OP_RMSNORM_LINEAR, OP_LINEAR_SILU, OP_FFN = 0, 1, 2, 3
OP_NORM_LINEAR, OP_MLP, OP_SWIGLU, OP_MLP_SWIGLU, OP_LINEAR_RESIDUAL_NORM = 4, 5, 6, 7, 8
NORM_NONE, NORM_LAYER, NORM_RMS = 0, 1, 2
ACT_NONE, ACT_SILU, ACT_RELU, ACT_GELU = 0, 1, 2, 3
STATUS = {0: "NGR_OK", -1: "NGR_ERR_NULL", -2: "NGR_ERR_SHAPE",
          -3: "NGR_ERR_ALIGN", -4: "NGR_ERR_DTYPE", -5: "NGR_ERR_WORKSPACE",
          -6: "NGR_ERR_ARCH", -7: "NGR_ERR_CUDA", -8: "NGR_ERR_TIMEOUT",
          -9: "NGR_ERR_ARG"}

# Every symbol include/ngr.h declares, with (restype, argtypes).
_P, _I64, _I, _F, _SZ, _U32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                               ctypes.c_float, ctypes.c_size_t, ctypes.c_uint32)
SIGNATURES = {
    "ngr_workspace_bytes": (_SZ, [_I, _I64, _I64, _I64, _I]),
    "ngr_fused_layernorm_linear": (_I, [_P, _P, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P, _SZ, _P]),
    "ngr_fused_layernorm_linear_noalloc": (_I, [_P, _P, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P]),
    "ngr_fused_rmsnorm_linear": (_I, [_P, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P, _SZ, _P]),
    "ngr_fused_linear_silu": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _P, _P, _SZ, _P]),
    "ngr_ffn_linear_silu_linear": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _P, _P, _P, _SZ, _P]),
    "ngr_fused_norm_linear_act": (_I, [_I, _I, _P, _P, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P, _SZ, _P]),
    "ngr_fused_mlp": (_I, [_I, _I, _P, _P, _P, _P, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P, _P, _SZ, _P]),
    "ngr_fused_norm_swiglu": (_I, [_I, _P, _P, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P, _SZ, _P]),
    "ngr_fused_mlp_swiglu": (_I, [_I, _P, _P, _P, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P, _P, _SZ, _P]),
    "ngr_fused_linear_residual_norm": (_I, [_I, _P, _P, _P, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P, _P, _SZ, _P]),
    "ngr_row_stats": (_I, [_I, _P, _F, _I64, _I64, _I, _P, _P]),
    "ngr_fold_prepare": (_I, [_I, _P, _P, _P, _P, _I64, _I64, _I, _P, _P, _P]),
    "ngr_fused_norm_linear_folded": (_I, [_I, _P, _P, _P, _F, _I64, _I64, _I64, _I, _P, _P, _SZ, _P]),
    "ngr_workspace_error": (_I, [_P, _P]),
    "ngr_noalloc_error": (_I, [_P]),
    "ngr_debug_bounded_wait": (_I, [_P, _U32, _P]),
    "ngr_status_string": (ctypes.c_char_p, [_I]),
    "ngr_version": (_I, []),
    "ngr_last_error": (ctypes.c_char_p, []),
    "ngr_set_tile_config": (_I, [_I, _I, _I]),
    "ngr_tile_plan": (_I, [_I, _I64, _I64, _I64, _P]),
    "ngr_kernel_timing_start": (_I, [_I]),
    "ngr_kernel_timing_stop": (_I, [_P, _I]),
}


class NgrError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what} failed: {status_string(status)}"
        if status == -7:
            try:
                msg += f" [{ngr_last_error()}]"
            except Exception:
                pass
        super().__init__(msg)


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"CUDA library not found at {LIB_PATH}; build it with "
                        "normalization_gemm_row_gb300.build()")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    f = getattr(handle, name)
                    f.restype, f.argtypes = res, args
                _lib = handle
    return _lib


# ---- C-named entry points ------------------------------------------------------
def ngr_workspace_bytes(op, M, K, N, ffn_h_in_workspace=0) -> int:
    return int(lib().ngr_workspace_bytes(op, M, K, N, ffn_h_in_workspace))


def ngr_fused_layernorm_linear(x, gamma, beta, W, bias, eps, M, K, N, dtype, y,
                               ws, ws_bytes, stream) -> int:
    return lib().ngr_fused_layernorm_linear(x, gamma, beta, W, bias, eps, M, K,
                                            N, dtype, y, ws, ws_bytes, stream)


def ngr_fused_layernorm_linear_noalloc(x, gamma, beta, W, bias, eps, M, K, N,
                                       dtype, y, stream) -> int:
    return lib().ngr_fused_layernorm_linear_noalloc(x, gamma, beta, W, bias, eps,
                                                    M, K, N, dtype, y, stream)


def ngr_fused_rmsnorm_linear(x, gamma, W, bias, eps, M, K, N, dtype, y, ws,
                             ws_bytes, stream) -> int:
    return lib().ngr_fused_rmsnorm_linear(x, gamma, W, bias, eps, M, K, N,
                                          dtype, y, ws, ws_bytes, stream)


def ngr_fused_linear_silu(x, W, bias, M, K, N, dtype, y, ws, ws_bytes,
                          stream) -> int:
    return lib().ngr_fused_linear_silu(x, W, bias, M, K, N, dtype, y, ws,
                                       ws_bytes, stream)


def ngr_ffn_linear_silu_linear(x, W1, W2, M, K, F, dtype, h, y, ws, ws_bytes,
                               stream) -> int:
    return lib().ngr_ffn_linear_silu_linear(x, W1, W2, M, K, F, dtype, h, y,
                                            ws, ws_bytes, stream)


def ngr_fused_norm_linear_act(norm, act, x, gamma, beta, W, bias, eps, M, K, N, dtype, y,
                              ws, ws_bytes, stream) -> int:
    return lib().ngr_fused_norm_linear_act(norm, act, x, gamma, beta, W, bias, eps, M, K, N,
                                           dtype, y, ws, ws_bytes, stream)


def ngr_fused_mlp(norm, act, x, gamma, beta, W1, b1, W2, b2, eps, M, K, F, dtype, h, y,
                  ws, ws_bytes, stream) -> int:
    return lib().ngr_fused_mlp(norm, act, x, gamma, beta, W1, b1, W2, b2, eps, M, K, F,
                               dtype, h, y, ws, ws_bytes, stream)


def ngr_fused_norm_swiglu(norm, x, gamma, beta, Wg, Wu, eps, M, K, F, dtype, h, ws,
                          ws_bytes, stream) -> int:
    return lib().ngr_fused_norm_swiglu(norm, x, gamma, beta, Wg, Wu, eps, M, K, F, dtype, h,
                                       ws, ws_bytes, stream)


def ngr_fused_mlp_swiglu(norm, x, gamma, beta, Wg, Wu, Wd, eps, M, K, F, dtype, h, y, ws,
                         ws_bytes, stream) -> int:
    return lib().ngr_fused_mlp_swiglu(norm, x, gamma, beta, Wg, Wu, Wd, eps, M, K, F, dtype,
                                      h, y, ws, ws_bytes, stream)


def ngr_fused_linear_residual_norm(norm, x, W, bias, residual, gamma, beta, eps, M, K, N,
                                   dtype, h, y, ws, ws_bytes, stream) -> int:
    return lib().ngr_fused_linear_residual_norm(norm, x, W, bias, residual, gamma, beta, eps,
                                                M, K, N, dtype, h, y, ws, ws_bytes, stream)


def ngr_fold_prepare(norm, gamma, beta, W, bias, K, N, dtype, Wf, cb, stream) -> int:
    return lib().ngr_fold_prepare(norm, gamma, beta, W, bias, K, N, dtype, Wf, cb, stream)


def ngr_fused_norm_linear_folded(norm, x, Wf, cb, eps, M, K, N, dtype, y, ws,
                                 ws_bytes, stream) -> int:
    return lib().ngr_fused_norm_linear_folded(norm, x, Wf, cb, eps, M, K, N, dtype,
                                              y, ws, ws_bytes, stream)


def ngr_row_stats(norm, x, eps, M, K, dtype, stats, stream) -> int:
    return lib().ngr_row_stats(norm, x, eps, M, K, dtype, stats, stream)


def ngr_workspace_error(ws, stream) -> int:
    return lib().ngr_workspace_error(ws, stream)


def ngr_noalloc_error(stream) -> int:
    return lib().ngr_noalloc_error(stream)


def ngr_debug_bounded_wait(ws, timeout_us, stream) -> int:
    return lib().ngr_debug_bounded_wait(ws, timeout_us, stream)


def ngr_status_string(status: int) -> str:
    return lib().ngr_status_string(status).decode()


def ngr_version() -> int:
    return int(lib().ngr_version())


def ngr_last_error() -> str:
    return lib().ngr_last_error().decode()


def ngr_set_tile_config(pair, bn, nsub) -> int:
    return lib().ngr_set_tile_config(pair, bn, nsub)


def ngr_tile_plan(op, M, K, N, plan) -> int:
    return lib().ngr_tile_plan(op, M, K, N, plan)


def tile_plan(op: int, M: int, K: int, N: int) -> dict:
    """The tile-kernel variant a call would launch on the current device."""
    arr = (ctypes.c_int * 6)()
    _raise(ngr_tile_plan(op, M, K, N, ctypes.cast(arr, ctypes.c_void_p)), "ngr_tile_plan")
    return dict(zip(("pair", "bn", "nsub", "splits", "grid", "stages"), list(arr)))


def set_tile_config(pair: int = -1, bn: int = 0, nsub: int = 0):
    """Restrict the tile-kernel choice (-1/0/0 restores the planner's)."""
    _raise(ngr_set_tile_config(pair, bn, nsub), "ngr_set_tile_config")


MAX_KERNELS_PER_CALL = 4


def ngr_kernel_timing_start(n_calls) -> int:
    return lib().ngr_kernel_timing_start(n_calls)


def ngr_kernel_timing_stop(ms, capacity) -> int:
    return lib().ngr_kernel_timing_stop(ms, capacity)


def kernel_timing_start(n_calls: int):
    """Time each kernel of this thread's next ``n_calls`` library calls."""
    _raise(ngr_kernel_timing_start(n_calls), "ngr_kernel_timing_start")


def kernel_timing_stop():
    """Per-call lists of kernel times (ms) of the calls timed since
    ``kernel_timing_start``."""
    k = MAX_KERNELS_PER_CALL
    cap = 65536 * k
    buf = (ctypes.c_float * cap)()
    n = ngr_kernel_timing_stop(buf, cap)
    if n < 0:
        raise NgrError(n, "ngr_kernel_timing_stop")
    return [[buf[c * k + j] for j in range(k) if buf[c * k + j] >= 0] for c in range(n)]


def status_string(status: int) -> str:
    try:
        return ngr_status_string(status)
    except Exception:
        return STATUS.get(status, f"status {status}")


# ---- tensor-level helpers ----------------------------------------------------------
def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return NGR_F16
    if t.dtype == torch.bfloat16:
        return NGR_BF16
    raise TypeError(f"tensors must be float16 or bfloat16, got {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(*ts, dtype):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if t.dtype != dtype:
            raise TypeError("all tensors must share one dtype")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _workspace(nbytes, device, workspace):
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace smaller than the {nbytes} bytes needed")
    return workspace


def _raise(rc, what):
    if rc != 0:
        raise NgrError(rc, what)


def fused_layernorm_linear(x, gamma, beta, W, bias=None, eps=1e-5, out=None,
                           workspace=None, stream=None):
    """y = LayerNorm(x) . W^T (+ bias); x [..., K], W [N, K]."""
    K = x.shape[-1]
    N = W.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, gamma, beta, W, bias, out, dtype=x.dtype)
    y = out if out is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_LAYERNORM_LINEAR, M, K, N)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_fused_layernorm_linear(_ptr(x2), _ptr(gamma), _ptr(beta), _ptr(W),
                                    _ptr(bias), float(eps), M, K, N,
                                    _dtype_code(x), _ptr(y), _ptr(ws),
                                    ws.numel() * ws.element_size(),
                                    _stream(stream))
    _raise(rc, "fused_layernorm_linear")
    return y.reshape(*x.shape[:-1], N)


def fused_rmsnorm_linear(x, gamma, W, bias=None, eps=1e-6, out=None,
                         workspace=None, stream=None):
    """y = RMSNorm(x) . W^T (+ bias)."""
    K = x.shape[-1]
    N = W.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, gamma, W, bias, out, dtype=x.dtype)
    y = out if out is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_RMSNORM_LINEAR, M, K, N)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_fused_rmsnorm_linear(_ptr(x2), _ptr(gamma), _ptr(W), _ptr(bias),
                                  float(eps), M, K, N, _dtype_code(x), _ptr(y),
                                  _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream))
    _raise(rc, "fused_rmsnorm_linear")
    return y.reshape(*x.shape[:-1], N)


def fused_linear_silu(x, W, bias=None, out=None, workspace=None, stream=None):
    """y = SiLU(x . W^T + bias)."""
    K = x.shape[-1]
    N = W.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, W, bias, out, dtype=x.dtype)
    y = out if out is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_LINEAR_SILU, M, K, N)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_fused_linear_silu(_ptr(x2), _ptr(W), _ptr(bias), M, K, N,
                               _dtype_code(x), _ptr(y), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream))
    _raise(rc, "fused_linear_silu")
    return y.reshape(*x.shape[:-1], N)


def ffn_linear_silu_linear(x, W1, W2, out=None, h=None, workspace=None,
                           stream=None):
    """y = SiLU(x . W1^T) . W2^T; W1 [F, K], W2 [K, F].  H goes to ``h``
    when given, else into the workspace."""
    K = x.shape[-1]
    F = W1.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, W1, W2, out, h, dtype=x.dtype)
    y = out if out is not None else torch.empty((M, K), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_FFN, M, K, F, 1 if h is None else 0)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_ffn_linear_silu_linear(_ptr(x2), _ptr(W1), _ptr(W2), M, K, F,
                                    _dtype_code(x), _ptr(h), _ptr(y), _ptr(ws),
                                    ws.numel() * ws.element_size(),
                                    _stream(stream))
    _raise(rc, "ffn_linear_silu_linear")
    return y.reshape(*x.shape[:-1], K)


def fused_norm_linear_act(x, W, norm: int = NORM_NONE, act: int = ACT_NONE, gamma=None,
                          beta=None, bias=None, eps=1e-5, out=None, workspace=None,
                          stream=None):
    """y = act(norm(x) . W^T + bias) for any norm (NORM_*) and activation
    (ACT_*)."""
    K = x.shape[-1]
    N = W.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, W, gamma, beta, bias, out, dtype=x.dtype)
    y = out if out is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_NORM_LINEAR, M, K, N)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_fused_norm_linear_act(norm, act, _ptr(x2), _ptr(gamma), _ptr(beta), _ptr(W),
                                   _ptr(bias), eps, M, K, N, _dtype_code(x), _ptr(y),
                                   _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _raise(rc, "fused_norm_linear_act")
    return y.reshape(*x.shape[:-1], N)


def fused_mlp(x, W1, W2, norm: int = NORM_NONE, act: int = ACT_SILU, gamma=None, beta=None,
              b1=None, b2=None, eps=1e-5, out=None, h=None, workspace=None, stream=None):
    """y = act(norm(x) . W1^T + b1) . W2^T + b2; W1 [F, K], W2 [K, F]."""
    K = x.shape[-1]
    F = W1.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, W1, W2, gamma, beta, b1, b2, out, h, dtype=x.dtype)
    y = out if out is not None else torch.empty((M, K), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_MLP, M, K, F, 1 if h is None else 0)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_fused_mlp(norm, act, _ptr(x2), _ptr(gamma), _ptr(beta), _ptr(W1), _ptr(b1),
                       _ptr(W2), _ptr(b2), eps, M, K, F, _dtype_code(x), _ptr(h), _ptr(y),
                       _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _raise(rc, "fused_mlp")
    return y.reshape(*x.shape[:-1], K)


def fused_norm_swiglu(x, Wg, Wu, norm: int = NORM_NONE, gamma=None, beta=None, eps=1e-5,
                      out=None, workspace=None, stream=None):
    """h = SiLU(norm(x) . Wg^T) * (norm(x) . Wu^T); Wg, Wu [F, K]."""
    K = x.shape[-1]
    F = Wg.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, Wg, Wu, gamma, beta, out, dtype=x.dtype)
    h = out if out is not None else torch.empty((M, F), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_SWIGLU, M, K, F)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_fused_norm_swiglu(norm, _ptr(x2), _ptr(gamma), _ptr(beta), _ptr(Wg), _ptr(Wu),
                               eps, M, K, F, _dtype_code(x), _ptr(h), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream))
    _raise(rc, "fused_norm_swiglu")
    return h.reshape(*x.shape[:-1], F)


def fused_mlp_swiglu(x, Wg, Wu, Wd, norm: int = NORM_NONE, gamma=None, beta=None, eps=1e-5,
                     out=None, h=None, workspace=None, stream=None):
    """y = (SiLU(norm(x) . Wg^T) * (norm(x) . Wu^T)) . Wd^T; Wd [K, F]."""
    K = x.shape[-1]
    F = Wg.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, Wg, Wu, Wd, gamma, beta, out, h, dtype=x.dtype)
    y = out if out is not None else torch.empty((M, K), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_MLP_SWIGLU, M, K, F, 1 if h is None else 0)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_fused_mlp_swiglu(norm, _ptr(x2), _ptr(gamma), _ptr(beta), _ptr(Wg), _ptr(Wu),
                              _ptr(Wd), eps, M, K, F, _dtype_code(x), _ptr(h), _ptr(y),
                              _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _raise(rc, "fused_mlp_swiglu")
    return y.reshape(*x.shape[:-1], K)


def fused_linear_residual_norm(x, W, gamma, norm: int = NORM_RMS, beta=None, bias=None,
                               residual=None, eps=1e-5, out=None, h=None, workspace=None,
                               stream=None):
    """(h, y): h = x . W^T + bias + residual, y = norm(h) over its N columns
    (gamma, beta of length N).  h goes to ``h`` when given."""
    K = x.shape[-1]
    N = W.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    r2 = residual.reshape(-1, N) if residual is not None else None
    _check(x2, W, gamma, beta, bias, r2, out, h, dtype=x.dtype)
    y = out if out is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    hh = h if h is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    nb = ngr_workspace_bytes(OP_LINEAR_RESIDUAL_NORM, M, K, N, 0)
    ws = _workspace(nb, x.device, workspace)
    rc = ngr_fused_linear_residual_norm(norm, _ptr(x2), _ptr(W), _ptr(bias), _ptr(r2),
                                        _ptr(gamma), _ptr(beta), eps, M, K, N, _dtype_code(x),
                                        _ptr(hh), _ptr(y), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream))
    _raise(rc, "fused_linear_residual_norm")
    return hh.reshape(*x.shape[:-1], N), y.reshape(*x.shape[:-1], N)


def fold_prepare(norm: int, gamma, beta, W, bias=None, stream=None):
    """Inference-mode fold of gamma (and beta, bias) into the weight:
    returns (Wf [N, K8] in W's dtype, cb float32 [2, N8] = (c, b')), with
    K8, N8 = K, N rounded up to multiples of 8 (zero padding)."""
    N, K = W.shape
    _check(gamma, beta, W, bias, dtype=W.dtype)
    K8, N8 = (K + 7) // 8 * 8, (N + 7) // 8 * 8
    Wf = torch.empty((N, K8), dtype=W.dtype, device=W.device)
    cb = torch.empty((2, N8), dtype=torch.float32, device=W.device)
    rc = ngr_fold_prepare(norm, _ptr(gamma), _ptr(beta), _ptr(W), _ptr(bias), K, N,
                          _dtype_code(W), _ptr(Wf), _ptr(cb), _stream(stream))
    _raise(rc, "fold_prepare")
    return Wf, cb


def fused_norm_linear_folded(norm: int, x, Wf, cb, eps, out=None, workspace=None,
                             stream=None):
    """y = norm(x) . W^T (+ bias) computed from the folded weight."""
    K = x.shape[-1]
    N = Wf.shape[0]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, Wf, out, dtype=x.dtype)
    if Wf.shape[1] != (K + 7) // 8 * 8:
        raise ValueError("Wf must be [N, K8] as fold_prepare returns it")
    if cb.dtype != torch.float32 or not cb.is_cuda or not cb.is_contiguous():
        raise TypeError("cb must be a contiguous float32 CUDA tensor [2, N8]")
    y = out if out is not None else torch.empty((M, N), dtype=x.dtype, device=x.device)
    op = OP_LAYERNORM_LINEAR if norm == 1 else OP_RMSNORM_LINEAR
    ws = _workspace(ngr_workspace_bytes(op, M, K, N), x.device, workspace)
    rc = ngr_fused_norm_linear_folded(norm, _ptr(x2), _ptr(Wf), _ptr(cb), float(eps), M, K, N,
                                      _dtype_code(x), _ptr(y), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream))
    _raise(rc, "fused_norm_linear_folded")
    return y.reshape(*x.shape[:-1], N)


def row_stats(x, norm: int, eps: float, stream=None) -> torch.Tensor:
    """(mu, rstd) per row as a float32 [M, 2] tensor (norm 1 = LayerNorm,
    2 = RMSNorm)."""
    K = x.shape[-1]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    _check(x2, dtype=x.dtype)
    st = torch.empty((M, 2), dtype=torch.float32, device=x.device)
    rc = ngr_row_stats(norm, _ptr(x2), float(eps), M, K, _dtype_code(x),
                       _ptr(st), _stream(stream))
    _raise(rc, "row_stats")
    return st
