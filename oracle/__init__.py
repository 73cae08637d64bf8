"""fp64 CPU oracle for the fused pre-norm linear layer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never loads it, and it imports nothing from the product
package: inputs arrive as CPU torch tensors (fp16 or bf16), results leave as
float64 numpy arrays.

The arithmetic lives in ``oracle.c`` (plain loops in double precision, one
row at a time); see that file's header for the definitions, their sources on
the pages and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libngr_oracle.so")

NORM_NONE, NORM_LAYER, NORM_RMS = 0, 1, 2
ACT_NONE, ACT_SILU, ACT_RELU, ACT_GELU = 0, 1, 2, 3
_DT = {torch.float16: 0, torch.bfloat16: 1}

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` into a shared library at ``out`` with gcc (OpenMP when
    the compiler has it).  Returns ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", out, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return out


def build() -> str:
    """Compile the oracle if its library is missing or older than its source."""
    with _lock:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            compile_oracle()
    return _LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P, I64, D, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
    lib.ngo_decode.argtypes = [P, I64, I, P]
    lib.ngo_row_stats.argtypes = [I, P, I64, I64, I, D, P, I64, P, P]
    lib.ngo_normalize.argtypes = [I, P, P, P, D, I64, I64, I, P, I64, P]
    lib.ngo_norm_linear.argtypes = [I, I, P, P, P, P, P, D, I64, I64, I64, I, P, I64, P]
    lib.ngo_ffn.argtypes = [P, P, P, I64, I64, I64, I, P, I64, P]
    lib.ngo_fold_prepare.argtypes = [I, P, P, P, P, I64, I64, I, P, P, P]
    lib.ngo_folded_linear.argtypes = [I, I, P, P, P, P, D, I64, I64, I64, I, P, I64, P]
    lib.ngo_mlp.argtypes = [I, I, P, P, P, P, P, P, P, D, I64, I64, I64, I64, I, P, I64, P]
    lib.ngo_swiglu.argtypes = [I, P, P, P, P, P, D, I64, I64, I64, I, P, I64, P]
    lib.ngo_mlp_swiglu.argtypes = [I, P, P, P, P, P, P, D, I64, I64, I64, I64, I, P, I64, P]
    lib.ngo_linear_residual_norm.argtypes = [I, P, P, P, P, P, P, D, I64, I64, I64, I, P, I64, P, P]
    lib.ngo_num_threads.argtypes = []
    for f in (lib.ngo_linear_residual_norm, lib.ngo_decode, lib.ngo_row_stats, lib.ngo_normalize,
              lib.ngo_norm_linear, lib.ngo_ffn, lib.ngo_fold_prepare,
              lib.ngo_folded_linear, lib.ngo_mlp, lib.ngo_swiglu,
              lib.ngo_mlp_swiglu, lib.ngo_num_threads):
        f.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed).  A ``path``
    loads that library instead, uncached (used to test planted mistakes)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


# ---- marshalling ---------------------------------------------------------------

def _bits(t: torch.Tensor | None):
    """CPU fp16/bf16 tensor -> contiguous int16 numpy view of its bits."""
    if t is None:
        return None
    if t.dtype not in _DT:
        raise TypeError(f"oracle inputs are fp16 or bf16, got {t.dtype}")
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, int(r.size)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


def decode(t: torch.Tensor, lib=None) -> np.ndarray:
    """Exact float64 values of a fp16/bf16 tensor, decoded by the oracle."""
    lib = lib or load()
    b = _bits(t).reshape(-1)
    out = np.empty(b.size, dtype=np.float64)
    _check(lib.ngo_decode(_ptr(b), b.size, _DT[t.dtype], _ptr(out)), "decode")
    return out.reshape(tuple(t.shape))


def row_stats(norm: int, x: torch.Tensor, eps: float, rows=None, lib=None):
    """(mu, rstd) in float64 for the listed rows of x [M, K]."""
    lib = lib or load()
    M, K = x.shape
    r, nr = _rows(rows, M)
    mu = np.empty(nr, dtype=np.float64)
    rstd = np.empty(nr, dtype=np.float64)
    xb = _bits(x)
    _check(lib.ngo_row_stats(norm, _ptr(xb), M, K, _DT[x.dtype], eps, _ptr(r),
                             nr, _ptr(mu), _ptr(rstd)), "row_stats")
    return mu, rstd


def normalize(norm: int, x, gamma, beta, eps: float, rows=None, lib=None):
    """The normalized, affine-transformed rows a [nrows, K] in float64."""
    lib = lib or load()
    M, K = x.shape
    r, nr = _rows(rows, M)
    a = np.empty((nr, K), dtype=np.float64)
    xb, gb, bb = _bits(x), _bits(gamma), _bits(beta)
    _check(lib.ngo_normalize(norm, _ptr(xb), _ptr(gb), _ptr(bb), eps, M, K,
                             _DT[x.dtype], _ptr(r), nr, _ptr(a)), "normalize")
    return a


def norm_linear(norm: int, act: int, x, gamma, beta, W, bias, eps: float,
                rows=None, lib=None) -> np.ndarray:
    """y [nrows, N] = act(norm(x[rows]) . W^T + bias) in float64."""
    lib = lib or load()
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("W must be [N, K]")
    r, nr = _rows(rows, M)
    y = np.empty((nr, N), dtype=np.float64)
    xb, gb, bb, wb, cb = (_bits(x), _bits(gamma), _bits(beta), _bits(W),
                          _bits(bias))
    _check(lib.ngo_norm_linear(norm, act, _ptr(xb), _ptr(gb), _ptr(bb),
                               _ptr(wb), _ptr(cb), eps, M, K, N, _DT[x.dtype],
                               _ptr(r), nr, _ptr(y)), "norm_linear")
    return y


def layernorm_linear(x, gamma, beta, W, bias, eps, rows=None, lib=None):
    return norm_linear(NORM_LAYER, ACT_NONE, x, gamma, beta, W, bias, eps,
                       rows, lib)


def rmsnorm_linear(x, gamma, W, bias, eps, rows=None, lib=None):
    return norm_linear(NORM_RMS, ACT_NONE, x, gamma, None, W, bias, eps, rows,
                       lib)


def linear_silu(x, W, bias, rows=None, lib=None):
    return norm_linear(NORM_NONE, ACT_SILU, x, None, None, W, bias, 0.0, rows,
                       lib)


def ffn(x, W1, W2, rows=None, lib=None) -> np.ndarray:
    """y [nrows, K] = SiLU(x[rows] . W1^T) . W2^T in float64 (H unrounded)."""
    lib = lib or load()
    M, K = x.shape
    F = W1.shape[0]
    if W1.shape[1] != K or tuple(W2.shape) != (K, F):
        raise ValueError("W1 must be [F, K] and W2 [K, F]")
    r, nr = _rows(rows, M)
    y = np.empty((nr, K), dtype=np.float64)
    xb, w1, w2 = _bits(x), _bits(W1), _bits(W2)
    _check(lib.ngo_ffn(_ptr(xb), _ptr(w1), _ptr(w2), M, K, F, _DT[x.dtype],
                       _ptr(r), nr, _ptr(y)), "ffn")
    return y


def mlp(norm: int, act: int, x, gamma, beta, W1, b1, W2, b2, eps: float,
        rows=None, lib=None) -> np.ndarray:
    """y [nrows, N] = act(norm(x[rows]) . W1^T + b1) . W2^T + b2 in float64
    (the hidden activations unrounded).  W1 is [F, K], W2 [N, F]."""
    lib = lib or load()
    M, K = x.shape
    F = W1.shape[0]
    N = W2.shape[0]
    if W1.shape[1] != K or W2.shape[1] != F:
        raise ValueError("W1 must be [F, K] and W2 [N, F]")
    r, nr = _rows(rows, M)
    y = np.empty((nr, N), dtype=np.float64)
    bits = [_bits(t) for t in (x, gamma, beta, W1, b1, W2, b2)]
    _check(lib.ngo_mlp(norm, act, *[_ptr(b) for b in bits], eps, M, K, F, N,
                       _DT[x.dtype], _ptr(r), nr, _ptr(y)), "mlp")
    return y


def swiglu(norm: int, x, gamma, beta, Wg, Wu, eps: float, rows=None,
           lib=None) -> np.ndarray:
    """h [nrows, F] = SiLU(a . Wg^T) * (a . Wu^T), a = norm(x[rows]), float64."""
    lib = lib or load()
    M, K = x.shape
    F = Wg.shape[0]
    if tuple(Wg.shape) != (F, K) or tuple(Wu.shape) != (F, K):
        raise ValueError("Wg and Wu must be [F, K]")
    r, nr = _rows(rows, M)
    h = np.empty((nr, F), dtype=np.float64)
    bits = [_bits(t) for t in (x, gamma, beta, Wg, Wu)]
    _check(lib.ngo_swiglu(norm, *[_ptr(b) for b in bits], eps, M, K, F,
                          _DT[x.dtype], _ptr(r), nr, _ptr(h)), "swiglu")
    return h


def mlp_swiglu(norm: int, x, gamma, beta, Wg, Wu, Wd, eps: float, rows=None,
               lib=None) -> np.ndarray:
    """y [nrows, N] = swiglu(...) . Wd^T in float64 (h unrounded); Wd [N, F]."""
    lib = lib or load()
    M, K = x.shape
    F = Wg.shape[0]
    N = Wd.shape[0]
    if tuple(Wg.shape) != (F, K) or tuple(Wu.shape) != (F, K) or Wd.shape[1] != F:
        raise ValueError("Wg, Wu must be [F, K] and Wd [N, F]")
    r, nr = _rows(rows, M)
    y = np.empty((nr, N), dtype=np.float64)
    bits = [_bits(t) for t in (x, gamma, beta, Wg, Wu, Wd)]
    _check(lib.ngo_mlp_swiglu(norm, *[_ptr(b) for b in bits], eps, M, K, F, N,
                              _DT[x.dtype], _ptr(r), nr, _ptr(y)), "mlp_swiglu")
    return y


def linear_residual_norm(norm: int, x, W, bias, residual, gamma, beta, eps: float,
                         rows=None, lib=None):
    """(h, y) [nrows, N] in float64: h = x . W^T + bias + residual, y = norm(h)
    over its N columns (gamma, beta of length N)."""
    lib = lib or load()
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("W must be [N, K]")
    r, nr = _rows(rows, M)
    h = np.empty((nr, N), dtype=np.float64)
    y = np.empty((nr, N), dtype=np.float64)
    bits = [_bits(t) for t in (x, W, bias, residual, gamma, beta)]
    _check(lib.ngo_linear_residual_norm(norm, *[_ptr(b) for b in bits], eps, M, K, N,
                                        _DT[x.dtype], _ptr(r), nr, _ptr(h), _ptr(y)),
           "linear_residual_norm")
    return h, y


def fold_prepare(norm: int, gamma, beta, W, bias, lib=None):
    """(W' [N, K], c [N], b' [N]) of the inference-mode fold, in float64."""
    lib = lib or load()
    N, K = W.shape
    Wf = np.empty((N, K), dtype=np.float64)
    c = np.empty(N, dtype=np.float64)
    bp = np.empty(N, dtype=np.float64)
    gb, bb, wb, cb = _bits(gamma), _bits(beta), _bits(W), _bits(bias)
    _check(lib.ngo_fold_prepare(norm, _ptr(gb), _ptr(bb), _ptr(wb), _ptr(cb),
                                K, N, _DT[W.dtype], _ptr(Wf), _ptr(c),
                                _ptr(bp)), "fold_prepare")
    return Wf, c, bp


def folded_linear(norm: int, act: int, x, Wf, c, bp, eps: float, rows=None,
                  lib=None) -> np.ndarray:
    """y = act(rstd (x . W'^T) - rstd mu c + b') in float64."""
    lib = lib or load()
    M, K = x.shape
    N = Wf.shape[0]
    r, nr = _rows(rows, M)
    y = np.empty((nr, N), dtype=np.float64)
    xb = _bits(x)
    Wf = np.ascontiguousarray(Wf, dtype=np.float64)
    c = np.ascontiguousarray(c, dtype=np.float64)
    bp = np.ascontiguousarray(bp, dtype=np.float64)
    _check(lib.ngo_folded_linear(norm, act, _ptr(xb), _ptr(Wf), _ptr(c),
                                 _ptr(bp), eps, M, K, N, _DT[x.dtype], _ptr(r),
                                 nr, _ptr(y)), "folded_linear")
    return y


def num_threads(lib=None) -> int:
    return int((lib or load()).ngo_num_threads())
