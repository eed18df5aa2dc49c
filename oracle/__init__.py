"""CPU oracle for the SmoothQuant W8A8 INT8 linear block (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package; the product
library never does, and the two share no code.

The arithmetic lives in ``sq_oracle.c`` (plain C, scalar loops, fp32 where the
quantiser decides an integer code, exact int64 sums, double epilogue).  This
module compiles it with gcc on first use and wraps it with ctypes over numpy
arrays.  Every function names the passage it follows in its docstring; the C
file states the readings taken where the pages are silent.

Parity status per function (what pins each one, see ``tests/test_oracle.py``):
  channel_absmax   brute force in Python on small inputs
  smooth_factor    closed forms (alpha 0 / 0.5 / 1, powers of two), zero rule
  smooth           exact invariant X W^T == (X/s)(W*s)^T for power-of-two s
  quantize_rows    hand-worked round-half-even example (golden file),
                   error bound |v - q*scale| <= scale/2, max code = 127
  act_absmax /     hand-worked saturating example (golden file); a one-row
  quantize_static  calibration set reproduces the dynamic codes
  gemm_i32         brute force in an outer-product order, closed forms
                   (all 127, cancelling signs, one-hot rows), overflow check
  epilogue         textbook normal-CDF values for GELU, zero-input cases
  layernorm        closed forms (constant row -> beta, alternating +-a -> +-1),
                   scale and shift invariance, zero mean / unit variance
  attention        closed forms (zero queries -> the mean of the values; two
                   keys -> logistic weights), near-one-hot limit, token
                   permutation equivariance, head and sequence independence
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sq_oracle.c")
_LIB = os.path.join(_HERE, "libsq_oracle.so")
_lock = threading.Lock()
_lib = None

EPI_NONE, EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESIDUAL = 0, 1, 2, 3
_OK, _ERR_ARG, _ERR_OVERFLOW = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``sq_oracle.c`` into ``libsq_oracle.so`` beside it (gcc, no
    fast-math, no fused multiply-add contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_channel_absmax.argtypes = [p, i64, i64, p]
            lib.oracle_smooth_factor.argtypes = [p, p, i64, dbl, p]
            lib.oracle_smooth.argtypes = [p, p, i64, i64, i32, p]
            lib.oracle_quantize_rows.argtypes = [p, p, i64, i64, i32, p, p]
            lib.oracle_gemm_i32.argtypes = [p, p, i64, i64, i64, p]
            lib.oracle_epilogue.argtypes = [p, p, p, p, p, i64, i64, i32, p]
            lib.oracle_linear_block.argtypes = [p, p, p, p, p, p, i64, i64, i64, i32,
                                                p, p, p, p]
            lib.oracle_num_threads.argtypes = []
            lib.oracle_act_absmax.argtypes = [p, p, i64, i64, p]
            lib.oracle_quantize_static.argtypes = [p, p, i64, i64, ctypes.c_float, p]
            lib.oracle_layernorm.argtypes = [p, p, p, dbl, i64, i64, p]
            lib.oracle_attention.argtypes = [p, i64, i64, i64, i64, dbl, p]
            for f in (lib.oracle_channel_absmax, lib.oracle_smooth_factor,
                      lib.oracle_smooth, lib.oracle_quantize_rows,
                      lib.oracle_gemm_i32, lib.oracle_epilogue,
                      lib.oracle_linear_block, lib.oracle_num_threads,
                      lib.oracle_act_absmax, lib.oracle_quantize_static,
                      lib.oracle_layernorm, lib.oracle_attention):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc == _ERR_OVERFLOW:
        raise OverflowError(f"oracle {what}: integer sum outside the int32 range")
    if rc != _OK:
        raise ValueError(f"oracle {what}: invalid argument (status {rc})")


def channel_absmax(A):
    """max over rows of |A[:, j]| (fp32).  Smoothing-factor statistics
    (SmoothQuant, cited in the reference list)."""
    A = _c(A, np.float32)
    rows, cols = A.shape
    out = np.empty(cols, np.float32)
    _check(_load().oracle_channel_absmax(_ptr(A), rows, cols, _ptr(out)), "channel_absmax")
    return out


def smooth_factor(x_amax, w_amax, alpha):
    """s_j = max|X_j|^alpha / max|W_j|^(1-alpha), double then fp32; a zero
    max gives 1.  Alpha per model: Table 15."""
    x_amax = _c(x_amax, np.float32)
    w_amax = _c(w_amax, np.float32)
    assert x_amax.shape == w_amax.shape
    s = np.empty_like(x_amax)
    _check(_load().oracle_smooth_factor(_ptr(x_amax), _ptr(w_amax), x_amax.size,
                                        float(alpha), _ptr(s)), "smooth_factor")
    return s


def smooth(A, s, direction):
    """direction 'act': X / s;  direction 'weight': W * s (fp32)."""
    A = _c(A, np.float32)
    s = _c(s, np.float32)
    rows, K = A.shape
    out = np.empty_like(A)
    d = {"act": 0, "weight": 1}[direction]
    _check(_load().oracle_smooth(_ptr(A), _ptr(s), rows, K, d, _ptr(out)), "smooth")
    return out


def quantize_rows(A, s, direction):
    """Per-row symmetric int8 of the smoothed matrix: returns (q int8, scale fp32).
    'act' = dynamic per-token activation quantisation (Table 10,
    Smooth-Dynamic); 'weight' = per-output-channel weight quantisation."""
    A = _c(A, np.float32)
    s = _c(s, np.float32)
    rows, K = A.shape
    assert s.shape == (K,)
    q = np.empty((rows, K), np.int8)
    scale = np.empty(rows, np.float32)
    d = {"act": 0, "weight": 1}[direction]
    _check(_load().oracle_quantize_rows(_ptr(A), _ptr(s), rows, K, d, _ptr(q),
                                        _ptr(scale)), "quantize_rows")
    return q, scale


def act_absmax(X, s, amax=0.0):
    """Per-tensor running max of |X / s| (Smooth-Static calibration, Table 10)."""
    X = _c(X, np.float32)
    s = _c(s, np.float32)
    rows, K = X.shape
    out = np.array([amax], np.float32)
    _check(_load().oracle_act_absmax(_ptr(X), _ptr(s), rows, K, _ptr(out)), "act_absmax")
    return out[0]


def static_scale(amax):
    """fl32(amax / 127), or 1 for a zero maximum."""
    amax = np.float32(amax)
    return np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(127.0))


def quantize_static(X, s, scale):
    """Smooth-Static codes with one offline per-tensor scale (saturating)."""
    X = _c(X, np.float32)
    s = _c(s, np.float32)
    rows, K = X.shape
    q = np.empty((rows, K), np.int8)
    _check(_load().oracle_quantize_static(_ptr(X), _ptr(s), rows, K, float(np.float32(scale)),
                                          _ptr(q)), "quantize_static")
    return q


def layernorm(H, gamma, beta, eps=1e-12):
    """Row LayerNorm in double, rounded once to fp32 (Table 3's LayerNorm; the
    input the next linear quantises)."""
    H = _c(H, np.float32)
    gamma = _c(gamma, np.float32)
    beta = _c(beta, np.float32)
    rows, K = H.shape
    assert gamma.shape == (K,) and beta.shape == (K,)
    y = np.empty_like(H)
    _check(_load().oracle_layernorm(_ptr(H), _ptr(gamma), _ptr(beta), float(eps), rows, K,
                                    _ptr(y)), "layernorm")
    return y


def attention(QKV, B, S, H, D, scale=None):
    """Encoder self-attention (Table 3's attention beside the linear block):
    QKV [B*S, 3*H*D] (the fused QKV projection's output: Q | K | V blocks,
    head h at columns h*D of each) -> O [B*S, H*D], softmax(scale Q K^T) V per
    sequence and head, scale = 1/sqrt(D) by default, no mask, double, rounded
    once to fp32."""
    QKV = _c(QKV, np.float32)
    assert QKV.shape == (B * S, 3 * H * D)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.empty((B * S, H * D), np.float32)
    _check(_load().oracle_attention(_ptr(QKV), B, S, H, D, float(scale), _ptr(O)), "attention")
    return O


def gemm_i32(xq, wq):
    """acc = xq @ wq^T, exact integer (int64 checked into int32)."""
    xq = _c(xq, np.int8)
    wq = _c(wq, np.int8)
    M, K = xq.shape
    N, K2 = wq.shape
    assert K == K2
    acc = np.empty((M, N), np.int32)
    _check(_load().oracle_gemm_i32(_ptr(xq), _ptr(wq), M, N, K, _ptr(acc)), "gemm_i32")
    return acc


def epilogue(acc, sx, sw, bias=None, residual=None, mode=EPI_NONE):
    """Dequantise and apply the linear block's post-ops (Table 3 caption) in
    double, rounded once to fp32."""
    acc = _c(acc, np.int32)
    M, N = acc.shape
    sx = _c(sx, np.float32)
    sw = _c(sw, np.float32)
    bias = None if bias is None else _c(bias, np.float32)
    residual = None if residual is None else _c(residual, np.float32)
    y = np.empty((M, N), np.float32)
    _check(_load().oracle_epilogue(_ptr(acc), _ptr(sx), _ptr(sw), _ptr(bias),
                                   _ptr(residual), M, N, int(mode), _ptr(y)), "epilogue")
    return y


def linear_block(X, s, wq, sw, bias=None, residual=None, mode=EPI_NONE):
    """Quantise activations, integer GEMM, epilogue: returns (xq, sx, acc, y)."""
    X = _c(X, np.float32)
    s = _c(s, np.float32)
    wq = _c(wq, np.int8)
    sw = _c(sw, np.float32)
    M, K = X.shape
    N = wq.shape[0]
    bias = None if bias is None else _c(bias, np.float32)
    residual = None if residual is None else _c(residual, np.float32)
    xq = np.empty((M, K), np.int8)
    sx = np.empty(M, np.float32)
    acc = np.empty((M, N), np.int32)
    y = np.empty((M, N), np.float32)
    _check(_load().oracle_linear_block(_ptr(X), _ptr(s), _ptr(wq), _ptr(sw), _ptr(bias),
                                       _ptr(residual), M, N, K, int(mode), _ptr(xq),
                                       _ptr(sx), _ptr(acc), _ptr(y)), "linear_block")
    return xq, sx, acc, y


def num_threads() -> int:
    """Threads an OpenMP region of the oracle uses (OMP_NUM_THREADS etc.)."""
    return int(_load().oracle_num_threads())
