"""ctypes binding of libsq_gb300.so: the C-ABI entry points under the same
names, taking torch CUDA tensors.  Argument marshalling only -- every step
runs in the library's CUDA kernels, on the caller's current torch stream.

There is no fallback: if the library is missing or fails to load, the first
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsq_gb300.so")

SQ_OK, SQ_ERR_INVALID_ARG, SQ_ERR_ALIGNMENT, SQ_ERR_UNSUPPORTED, SQ_ERR_CUDA, SQ_ERR_TIMEOUT = range(6)
EPI_NONE, EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESIDUAL, EPI_RAW_I32 = range(5)

EXPORTS = ("sq_status_string", "sq_version", "sq_operand_bytes", "sq_packed_weight_bytes",
           "sq_channel_absmax",
           "sq_smooth_factor", "sq_pack_weight", "sq_quantize_act", "sq_act_absmax",
           "sq_static_scale", "sq_quantize_act_static", "sq_layernorm_quant", "sq_linear_i8",
           "sq_linear_codes_workspace_bytes", "sq_linear_i8_codes",
           "sq_linear_i8_requant", "sq_division_table", "sq_linear_i8_rowmax",
           "sq_quantize_act_rowmax", "sq_quantize_act_table", "sq_attention",
           "sq_linear_workspace_bytes", "sq_linear_i8_ws", "sq_linear_i8_requant_ws", "sq_linear_i8_static_ws", "sq_static_workspace_reset",
           "sq_static_workspace", "sq_linear_i8_mma_sync", "sq_linear_block_host_scratch_bytes",
           "sq_linear_block_host",
           "sq_check_division", "sq_device_status", "sq_get_device_status")

class LinearLayerC(ctypes.Structure):
    """sq_linear_layer (include/sq.h): one layer of sq_linear_block_host."""
    _fields_ = [("K", ctypes.c_int64), ("N", ctypes.c_int64), ("mode", ctypes.c_int),
                ("static_scale", ctypes.c_float), ("s", ctypes.c_void_p),
                ("s_table", ctypes.c_void_p), ("Wop", ctypes.c_void_p),
                ("w_scale", ctypes.c_void_p), ("w_row_l1", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("residual", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


class SQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (once).  Raises OSError if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise OSError(f"{p} is missing: build it with "
                              "`python -m smoothquant_w8a8_int8_gb300.build`")
            lib = ctypes.CDLL(p)
            vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            sig = {
                "sq_status_string": ([i32], ctypes.c_char_p),
                "sq_version": ([], i32),
                "sq_operand_bytes": ([i64, i64], ctypes.c_size_t),
                "sq_packed_weight_bytes": ([i64, i64], ctypes.c_size_t),
                "sq_channel_absmax": ([vp, i64, i64, vp, vp], i32),
                "sq_smooth_factor": ([vp, vp, i64, f32, vp, vp], i32),
                "sq_pack_weight": ([vp, vp, i64, i64, vp, vp, vp, vp, vp], i32),
                "sq_quantize_act": ([vp, vp, i64, i64, vp, vp, vp, vp, vp], i32),
                "sq_act_absmax": ([vp, vp, i64, i64, vp, vp], i32),
                "sq_static_scale": ([vp, vp, vp], i32),
                "sq_quantize_act_static": ([vp, vp, i64, i64, f32, vp, vp, vp, vp, vp], i32),
                "sq_layernorm_quant": ([vp, vp, vp, f32, vp, i64, i64, f32, vp, vp, vp, vp, vp,
                                        vp], i32),
                "sq_linear_i8": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, vp],
                                 i32),
                "sq_linear_i8_requant": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp,
                                          f32, vp, vp, vp, vp], i32),
                "sq_division_table": ([vp, i64, vp, vp], i32),
                "sq_linear_i8_rowmax": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp,
                                         vp, vp, vp], i32),
                "sq_quantize_act_rowmax": ([vp, vp, vp, i64, i64, vp, vp, vp, vp, vp], i32),
                "sq_quantize_act_table": ([vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, vp], i32),
                "sq_attention": ([vp, i64, i64, i64, i64, f32, vp, vp], i32),
                "sq_linear_workspace_bytes": ([i64, i64, i64, vp], i32),
                "sq_linear_codes_workspace_bytes": ([i64, i64, vp], i32),
                "sq_linear_i8_codes": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp,
                                        vp, ctypes.c_size_t, vp], i32),
                "sq_linear_i8_ws": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, vp,
                                     ctypes.c_size_t, vp], i32),
                "sq_linear_i8_requant_ws": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32,
                                             vp, f32, vp, vp, vp, vp, ctypes.c_size_t, vp], i32),
                "sq_linear_i8_static_ws": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp,
                                            vp], i32),
                "sq_static_workspace_reset": ([vp], i32),
                "sq_static_workspace": ([ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)], i32),
                "sq_linear_i8_mma_sync": ([vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, vp], i32),
                "sq_linear_block_host_scratch_bytes": ([i64, i64, i64,
                                                        ctypes.POINTER(ctypes.c_size_t)], i32),
                "sq_linear_block_host": ([ctypes.POINTER(LinearLayerC), i64, i64, vp, vp, vp,
                                          ctypes.c_size_t, vp, vp, vp], i32),
                "sq_check_division": ([ctypes.c_uint32] * 4 + [i32, vp, vp], i32),
                "sq_device_status": ([vp], i32),
                "sq_get_device_status": ([vp], i32),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().sq_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != SQ_OK:
        raise SQError(rc, what)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def operand_bytes(rows: int, K: int) -> int:
    return int(load().sq_operand_bytes(rows, K))


def packed_weight_bytes(N: int, K: int) -> int:
    return int(load().sq_packed_weight_bytes(N, K))


def empty_operand(rows: int, K: int, device="cuda") -> torch.Tensor:
    """A GEMM-operand buffer (int8 codes held as exact bf16 values)."""
    return torch.empty(rows, K, dtype=torch.bfloat16, device=device)


def channel_absmax(A: torch.Tensor, amax: Optional[torch.Tensor] = None, stream=None):
    """amax[j] = max(amax[j], max_i |A[i, j]|); a fresh zero statistic if None."""
    _need(A, torch.float32, "A")
    rows, cols = A.shape
    if amax is None:
        amax = torch.zeros(cols, dtype=torch.float32, device=A.device)
    _need(amax, torch.float32, "amax", (cols,))
    _check(load().sq_channel_absmax(_p(A), rows, cols, _p(amax), _stream(stream)),
           "sq_channel_absmax")
    return amax


def smooth_factor(x_amax: torch.Tensor, w_amax: torch.Tensor, alpha: float, stream=None):
    _need(x_amax, torch.float32, "x_amax")
    _need(w_amax, torch.float32, "w_amax", x_amax.shape)
    s = torch.empty_like(x_amax)
    _check(load().sq_smooth_factor(_p(x_amax), _p(w_amax), x_amax.numel(), float(alpha), _p(s),
                                   _stream(stream)), "sq_smooth_factor")
    return s


def pack_weight(W: torch.Tensor, s: torch.Tensor, want_q: bool = True, want_op: bool = True,
                want_l1: bool = False, stream=None):
    """Returns (Wq int8 or None, w_scale fp32, Wop operand or None), plus the
    per-row code L1 norms (int32) as a fourth item when want_l1."""
    _need(W, torch.float32, "W")
    N, K = W.shape
    _need(s, torch.float32, "s", (K,))
    Wq = torch.empty(N, K, dtype=torch.int8, device=W.device) if want_q else None
    Wop = empty_operand(N, K, W.device) if want_op else None
    sw = torch.empty(N, dtype=torch.float32, device=W.device)
    l1 = torch.empty(N, dtype=torch.int32, device=W.device) if want_l1 else None
    _check(load().sq_pack_weight(_p(W), _p(s), N, K, _p(Wq), _p(sw), _p(Wop), _p(l1),
                                 _stream(stream)), "sq_pack_weight")
    return (Wq, sw, Wop, l1) if want_l1 else (Wq, sw, Wop)


def quantize_act(X: torch.Tensor, s: torch.Tensor, want_q: bool = True, want_op: bool = True,
                 want_l1: bool = False, out=None, stream=None):
    """Returns (Xq int8 or None, x_scale fp32, Xop operand or None), plus the
    per-token code L1 norms (int32) as a fourth item when want_l1.  `out` may
    give preallocated (Xq, x_scale, Xop[, x_l1]) buffers."""
    _need(X, torch.float32, "X")
    M, K = X.shape
    _need(s, torch.float32, "s", (K,))
    if out is not None:
        Xq, sx, Xop = out[:3]
        l1 = out[3] if len(out) > 3 else None
    else:
        Xq = torch.empty(M, K, dtype=torch.int8, device=X.device) if want_q else None
        Xop = empty_operand(M, K, X.device) if want_op else None
        sx = torch.empty(M, dtype=torch.float32, device=X.device)
        l1 = torch.empty(M, dtype=torch.int32, device=X.device) if want_l1 else None
    _check(load().sq_quantize_act(_p(X), _p(s), M, K, _p(Xq), _p(sx), _p(Xop), _p(l1),
                                  _stream(stream)), "sq_quantize_act")
    if want_l1 or (out is not None and len(out) > 3):
        return Xq, sx, Xop, l1
    return Xq, sx, Xop


def act_absmax(X: torch.Tensor, s: torch.Tensor, amax: Optional[torch.Tensor] = None,
               stream=None):
    """Smooth-Static calibration: amax = max(amax, max |X / s|) (one float)."""
    _need(X, torch.float32, "X")
    M, K = X.shape
    _need(s, torch.float32, "s", (K,))
    if amax is None:
        amax = torch.zeros(1, dtype=torch.float32, device=X.device)
    _check(load().sq_act_absmax(_p(X), _p(s), M, K, _p(amax), _stream(stream)), "sq_act_absmax")
    return amax


def static_scale(amax: torch.Tensor, stream=None) -> float:
    """The per-tensor static scale the library computes from the calibration
    statistic `amax` (one float on the device, from act_absmax), read back
    once (offline)."""
    _need(amax, torch.float32, "amax", (1,))
    out = torch.empty(1, dtype=torch.float32, device=amax.device)
    _check(load().sq_static_scale(_p(amax), _p(out), _stream(stream)), "sq_static_scale")
    return float(out.item())


def quantize_act_static(X: torch.Tensor, s: torch.Tensor, scale: float, want_q: bool = True,
                        want_op: bool = True, want_l1: bool = False, out=None, stream=None):
    """Smooth-Static quantisation with a fixed per-tensor scale; returns
    (Xq or None, x_scale [M] filled with scale, Xop or None), plus the
    per-token code L1 norms as a fourth item when want_l1 (or a 4-tuple
    `out`)."""
    _need(X, torch.float32, "X")
    M, K = X.shape
    _need(s, torch.float32, "s", (K,))
    l1 = None
    if out is not None:
        Xq, sx, Xop = out[:3]
        l1 = out[3] if len(out) > 3 else None
    else:
        Xq = torch.empty(M, K, dtype=torch.int8, device=X.device) if want_q else None
        Xop = empty_operand(M, K, X.device) if want_op else None
        sx = torch.empty(M, dtype=torch.float32, device=X.device)
        l1 = torch.empty(M, dtype=torch.int32, device=X.device) if want_l1 else None
    _check(load().sq_quantize_act_static(_p(X), _p(s), M, K, float(scale), _p(Xq), _p(sx),
                                         _p(Xop), _p(l1), _stream(stream)),
           "sq_quantize_act_static")
    if want_l1 or (out is not None and len(out) > 3):
        return Xq, sx, Xop, l1
    return Xq, sx, Xop


def layernorm_quant(H: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float,
                    s: torch.Tensor, static_scale: float = 0.0, want_y: bool = False,
                    want_q: bool = True, want_op: bool = True, want_l1: bool = False, out=None,
                    stream=None):
    """LayerNorm of H with the next linear's quantiser fused in (dynamic when
    static_scale is 0); returns (Xq or None, x_scale, Xop or None, Y or None,
    l1 or None).  `out` may give those five (Xq, Xop, Y, l1 may be None)."""
    _need(H, torch.float32, "H")
    M, K = H.shape
    for t, n in ((gamma, "gamma"), (beta, "beta"), (s, "s")):
        _need(t, torch.float32, n, (K,))
    if out is not None:
        Xq, sx, Xop, Y, l1 = out
    else:
        Xq = torch.empty(M, K, dtype=torch.int8, device=H.device) if want_q else None
        Xop = empty_operand(M, K, H.device) if want_op else None
        sx = torch.empty(M, dtype=torch.float32, device=H.device)
        Y = torch.empty(M, K, dtype=torch.float32, device=H.device) if want_y else None
        l1 = torch.empty(M, dtype=torch.int32, device=H.device) if want_l1 else None
    _check(load().sq_layernorm_quant(_p(H), _p(gamma), _p(beta), float(eps), _p(s), M, K,
                                     float(static_scale), _p(Y), _p(Xq), _p(sx), _p(Xop),
                                     _p(l1), _stream(stream)), "sq_layernorm_quant")
    return Xq, sx, Xop, Y, l1


def _out(Xa, Wa, mode, out):
    M, K = Xa.shape
    N = Wa.shape[0]
    if Wa.shape[1] != K:
        raise ValueError("operand K mismatch")
    if out is None:
        dt = torch.int32 if mode == EPI_RAW_I32 else torch.float32
        out = torch.empty(M, N, dtype=dt, device=Xa.device)
    return M, N, K, out


def linear_i8(Xop, x_scale, Wop, w_scale, bias=None, residual=None, mode=EPI_BIAS, out=None,
              x_l1=None, w_l1=None, stream=None):
    """tcgen05 INT8 GEMM + epilogue on GEMM-operand buffers.  x_l1 / w_l1:
    optional per-row code L1 norms from quantize_act / pack_weight."""
    _need(Xop, torch.bfloat16, "Xop")
    _need(Wop, torch.bfloat16, "Wop")
    M, N, K, out = _out(Xop, Wop, mode, out)
    _check(load().sq_linear_i8(_p(Xop), _p(x_scale), _p(x_l1), _p(Wop), _p(w_scale), _p(w_l1),
                               _p(bias), _p(residual), M, N, K, int(mode), _p(out),
                               _stream(stream)), "sq_linear_i8")
    return out


def codes_workspace_bytes(M: int, K: int) -> int:
    """Bytes of the workspace linear_i8_codes widens an M x K code matrix into."""
    n = ctypes.c_size_t(0)
    _check(load().sq_linear_codes_workspace_bytes(M, K, ctypes.byref(n)),
           "sq_linear_codes_workspace_bytes")
    return int(n.value)


def linear_i8_codes(Xq, x_scale, Wop, w_scale, bias=None, residual=None, mode=EPI_BIAS,
                    out=None, x_l1=None, w_l1=None, workspace=None, stream=None):
    """linear_i8 on int8 activation codes Xq [M, K]: the codes are widened
    exactly into the bf16 operand in `workspace` (uint8, at least
    codes_workspace_bytes(M, K); allocated here if None), then the tcgen05
    GEMM runs on it."""
    _need(Xq, torch.int8, "Xq")
    _need(Wop, torch.bfloat16, "Wop")
    M, N, K, out = _out(Xq, Wop, mode, out)
    if workspace is None:
        workspace = torch.empty(max(codes_workspace_bytes(M, K), 16), dtype=torch.uint8,
                                device=Xq.device)
    wp, wn = _workspace(workspace)
    _check(load().sq_linear_i8_codes(_p(Xq), _p(x_scale), _p(x_l1), _p(Wop), _p(w_scale),
                                     _p(w_l1), _p(bias), _p(residual), M, N, K, int(mode),
                                     _p(out), wp, wn, _stream(stream)), "sq_linear_i8_codes")
    return out


def linear_i8_requant(Xop, x_scale, Wop, w_scale, bias, residual, mode, s_next, scale: float,
                      want_q: bool = False, want_op: bool = True, want_x_scale: bool = True,
                      out=None, x_l1=None, w_l1=None, stream=None):
    """tcgen05 INT8 GEMM whose epilogue emits the next linear's Smooth-Static
    codes (smoothing factor s_next [N], per-tensor scale) instead of fp32 Y.
    Returns (Yq or None, Yop or None, x_scale_next or None); `out` may give
    those three (each may be None)."""
    _need(Xop, torch.bfloat16, "Xop")
    _need(Wop, torch.bfloat16, "Wop")
    M, K = Xop.shape
    N = Wop.shape[0]
    if Wop.shape[1] != K:
        raise ValueError("operand K mismatch")
    _need(s_next, torch.float32, "s_next", (N,))
    if out is not None:
        Yq, Yop, xs = out
    else:
        Yq = torch.empty(M, N, dtype=torch.int8, device=Xop.device) if want_q else None
        Yop = empty_operand(M, N, Xop.device) if want_op else None
        xs = torch.empty(M, dtype=torch.float32, device=Xop.device) if want_x_scale else None
    _check(load().sq_linear_i8_requant(_p(Xop), _p(x_scale), _p(x_l1), _p(Wop), _p(w_scale),
                                       _p(w_l1), _p(bias), _p(residual), M, N, K, int(mode),
                                       _p(s_next), float(scale), _p(Yq), _p(Yop), _p(xs),
                                       _stream(stream)), "sq_linear_i8_requant")
    return Yq, Yop, xs


def division_table(s: torch.Tensor, stream=None) -> torch.Tensor:
    """(-s, RN(1/s)) per column ([K, 2] fp32) for linear_i8_rowmax."""
    _need(s, torch.float32, "s")
    K = s.numel()
    table = torch.empty(K, 2, dtype=torch.float32, device=s.device)
    _check(load().sq_division_table(_p(s), K, _p(table), _stream(stream)), "sq_division_table")
    return table


def linear_i8_rowmax(Xop, x_scale, Wop, w_scale, bias, residual, mode, next_table,
                     row_amax=None, out=None, x_l1=None, w_l1=None, stream=None):
    """linear_i8 whose epilogue also merges each row's max |Y / s_next| into
    row_amax (zero-filled here when None).  Returns (Y, row_amax)."""
    _need(Xop, torch.bfloat16, "Xop")
    _need(Wop, torch.bfloat16, "Wop")
    M, N, K, out = _out(Xop, Wop, mode, out)
    _need(next_table, torch.float32, "next_table", (N, 2))
    if row_amax is None:
        row_amax = torch.zeros(M, dtype=torch.float32, device=Xop.device)
    _need(row_amax, torch.float32, "row_amax", (M,))
    _check(load().sq_linear_i8_rowmax(_p(Xop), _p(x_scale), _p(x_l1), _p(Wop), _p(w_scale),
                                      _p(w_l1), _p(bias), _p(residual), M, N, K, int(mode),
                                      _p(out), _p(next_table), _p(row_amax), _stream(stream)),
           "sq_linear_i8_rowmax")
    return out, row_amax


def quantize_act_rowmax(X, s, row_amax, want_q: bool = True, want_op: bool = True,
                        want_l1: bool = False, out=None, stream=None):
    """quantize_act with the per-token maxima given (from linear_i8_rowmax);
    returns (Xq or None, x_scale, Xop or None) (+ l1 when want_l1 or a 4-tuple out)."""
    _need(X, torch.float32, "X")
    M, K = X.shape
    _need(s, torch.float32, "s", (K,))
    _need(row_amax, torch.float32, "row_amax", (M,))
    l1 = None
    if out is not None:
        Xq, sx, Xop = out[:3]
        l1 = out[3] if len(out) > 3 else None
    else:
        Xq = torch.empty(M, K, dtype=torch.int8, device=X.device) if want_q else None
        Xop = empty_operand(M, K, X.device) if want_op else None
        sx = torch.empty(M, dtype=torch.float32, device=X.device)
        l1 = torch.empty(M, dtype=torch.int32, device=X.device) if want_l1 else None
    _check(load().sq_quantize_act_rowmax(_p(X), _p(s), _p(row_amax), M, K, _p(Xq), _p(sx),
                                         _p(Xop), _p(l1), _stream(stream)),
           "sq_quantize_act_rowmax")
    if want_l1 or (out is not None and len(out) > 3):
        return Xq, sx, Xop, l1
    return Xq, sx, Xop


def quantize_act_table(X, s, table, row_amax=None, want_q: bool = True, want_op: bool = True,
                       want_l1: bool = False, out=None, stream=None):
    """quantize_act (row_amax None) or quantize_act_rowmax (row_amax given)
    with s's division table (division_table(s)); same returns."""
    _need(X, torch.float32, "X")
    M, K = X.shape
    _need(s, torch.float32, "s", (K,))
    _need(table, torch.float32, "table", (K, 2))
    if row_amax is not None:
        _need(row_amax, torch.float32, "row_amax", (M,))
    l1 = None
    if out is not None:
        Xq, sx, Xop = out[:3]
        l1 = out[3] if len(out) > 3 else None
    else:
        Xq = torch.empty(M, K, dtype=torch.int8, device=X.device) if want_q else None
        Xop = empty_operand(M, K, X.device) if want_op else None
        sx = torch.empty(M, dtype=torch.float32, device=X.device)
        l1 = torch.empty(M, dtype=torch.int32, device=X.device) if want_l1 else None
    _check(load().sq_quantize_act_table(_p(X), _p(s), _p(table), _p(row_amax), M, K, _p(Xq),
                                        _p(sx), _p(Xop), _p(l1), _stream(stream)),
           "sq_quantize_act_table")
    if want_l1 or (out is not None and len(out) > 3):
        return Xq, sx, Xop, l1
    return Xq, sx, Xop


def attention(QKV: torch.Tensor, B: int, S: int, H: int, D: int = 64, scale=None, out=None,
              stream=None) -> torch.Tensor:
    """Encoder self-attention on the fused QKV output [B*S, 3*H*D] -> O [B*S, H*D]."""
    _need(QKV, torch.float32, "QKV", (B * S, 3 * H * D))
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty(B * S, H * D, dtype=torch.float32, device=QKV.device)
    _need(out, torch.float32, "O", (B * S, H * D))
    _check(load().sq_attention(_p(QKV), B, S, H, D, float(scale), _p(out), _stream(stream)),
           "sq_attention")
    return out


def linear_workspace_bytes(M: int, N: int, K: int) -> int:
    """Bytes of the split-K workspace of an M x N x K linear (0: none needed)."""
    n = ctypes.c_size_t(0)
    _check(load().sq_linear_workspace_bytes(M, N, K, ctypes.byref(n)), "sq_linear_workspace_bytes")
    return int(n.value)


def empty_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled split-K workspace (uint8).  Completed launches leave its
    counters at zero, so it is reused as it is."""
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def _workspace(ws):
    if ws is None:
        return None, 0
    _need(ws, torch.uint8, "workspace")
    return _p(ws), ws.numel()


def linear_i8_ws(Xop, x_scale, Wop, w_scale, bias=None, residual=None, mode=EPI_BIAS, out=None,
                 x_l1=None, w_l1=None, workspace=None, stream=None):
    """linear_i8 with the split-K schedule on `workspace` (see
    linear_workspace_bytes / empty_workspace); bit for bit the same output."""
    _need(Xop, torch.bfloat16, "Xop")
    _need(Wop, torch.bfloat16, "Wop")
    M, N, K, out = _out(Xop, Wop, mode, out)
    wp, wn = _workspace(workspace)
    _check(load().sq_linear_i8_ws(_p(Xop), _p(x_scale), _p(x_l1), _p(Wop), _p(w_scale), _p(w_l1),
                                  _p(bias), _p(residual), M, N, K, int(mode), _p(out), wp, wn,
                                  _stream(stream)), "sq_linear_i8_ws")
    return out


STATIC_WORKSPACE_BYTES = 40 * 1024 * 1024  # SQ_STATIC_WORKSPACE_BYTES of sq.h


def linear_i8_static_ws(Xop, x_scale, Wop, w_scale, bias=None, residual=None, mode=EPI_BIAS,
                        out=None, x_l1=None, w_l1=None, stream=None):
    """linear_i8_ws on the library's static scratch (no workspace argument, no
    allocation); calls that may overlap must be serialised by the caller."""
    _need(Xop, torch.bfloat16, "Xop")
    _need(Wop, torch.bfloat16, "Wop")
    M, N, K, out = _out(Xop, Wop, mode, out)
    _check(load().sq_linear_i8_static_ws(_p(Xop), _p(x_scale), _p(x_l1), _p(Wop), _p(w_scale),
                                         _p(w_l1), _p(bias), _p(residual), M, N, K, int(mode),
                                         _p(out), _stream(stream)), "sq_linear_i8_static_ws")
    return out


def static_workspace_reset(stream=None) -> None:
    """Zero-fill the static scratch's split-K counters on the current device."""
    _check(load().sq_static_workspace_reset(_stream(stream)), "sq_static_workspace_reset")


def static_workspace():
    """(device address, bytes) of the static scratch on the current device."""
    p, n = ctypes.c_void_p(), ctypes.c_size_t()
    _check(load().sq_static_workspace(ctypes.byref(p), ctypes.byref(n)), "sq_static_workspace")
    return int(p.value), int(n.value)


def linear_i8_requant_ws(Xop, x_scale, Wop, w_scale, bias, residual, mode, s_next,
                         scale: float, want_q: bool = False, want_op: bool = True,
                         want_x_scale: bool = True, out=None, x_l1=None, w_l1=None,
                         workspace=None, stream=None):
    """linear_i8_requant with the split-K schedule on `workspace`."""
    _need(Xop, torch.bfloat16, "Xop")
    _need(Wop, torch.bfloat16, "Wop")
    M, K = Xop.shape
    N = Wop.shape[0]
    if Wop.shape[1] != K:
        raise ValueError("operand K mismatch")
    _need(s_next, torch.float32, "s_next", (N,))
    if out is not None:
        Yq, Yop, xs = out
    else:
        Yq = torch.empty(M, N, dtype=torch.int8, device=Xop.device) if want_q else None
        Yop = empty_operand(M, N, Xop.device) if want_op else None
        xs = torch.empty(M, dtype=torch.float32, device=Xop.device) if want_x_scale else None
    wp, wn = _workspace(workspace)
    _check(load().sq_linear_i8_requant_ws(_p(Xop), _p(x_scale), _p(x_l1), _p(Wop), _p(w_scale),
                                          _p(w_l1), _p(bias), _p(residual), M, N, K, int(mode),
                                          _p(s_next), float(scale), _p(Yq), _p(Yop), _p(xs), wp,
                                          wn, _stream(stream)), "sq_linear_i8_requant_ws")
    return Yq, Yop, xs


def linear_block_host_scratch_bytes(M: int, max_K: int, max_N: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().sq_linear_block_host_scratch_bytes(M, max_K, max_N, ctypes.byref(n)),
           "sq_linear_block_host_scratch_bytes")
    return n.value


def linear_block_host(layers, M: int, X_host, Y_host, scratch: torch.Tensor, streams) -> None:
    """sq_linear_block_host: `layers` a sequence of LinearLayerC, X_host / Y_host
    pinned host tensors (one per layer), `scratch` a device uint8 tensor of at
    least linear_block_host_scratch_bytes bytes, `streams` the (h2d, compute,
    d2h) torch streams.  Returns once everything is enqueued."""
    n = len(layers)
    arr = (LinearLayerC * n)(*layers)
    xs = (ctypes.c_void_p * n)(*[x.data_ptr() for x in X_host])
    ys = (ctypes.c_void_p * n)(*[y.data_ptr() for y in Y_host])
    h2d, comp, d2h = (st.cuda_stream for st in streams)
    _check(load().sq_linear_block_host(arr, n, M, ctypes.cast(xs, ctypes.c_void_p),
                                       ctypes.cast(ys, ctypes.c_void_p), _p(scratch),
                                       scratch.numel(), h2d, comp, d2h),
           "sq_linear_block_host")


def linear_i8_mma_sync(Xq, x_scale, Wq, w_scale, bias=None, residual=None, mode=EPI_BIAS,
                       out=None, stream=None):
    """Legacy mma.sync INT8 GEMM + epilogue on int8 codes."""
    _need(Xq, torch.int8, "Xq")
    _need(Wq, torch.int8, "Wq")
    M, N, K, out = _out(Xq, Wq, mode, out)
    _check(load().sq_linear_i8_mma_sync(_p(Xq), _p(x_scale), _p(Wq), _p(w_scale), _p(bias),
                                        _p(residual), M, N, K, int(mode), _p(out),
                                        _stream(stream)), "sq_linear_i8_mma_sync")
    return out


def check_division(b_first: int, b_count: int, a_first: int, a_count: int,
                   corrected: bool = True, out: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
    """Run the requantising epilogue's division against IEEE division on the
    significand pairs (see sq_check_division); returns the int64[2] device
    tensor (mismatch count, 1 + (af << 32 | bf) of one mismatch or 0)."""
    if out is None:
        out = torch.zeros(2, dtype=torch.int64, device="cuda")
    _check(load().sq_check_division(b_first, b_count, a_first, a_count, int(bool(corrected)),
                                    _p(out), _stream(stream)), "sq_check_division")
    return out


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status."""
    return int(load().sq_device_status(_stream(stream)))


def get_device_status(stream=None) -> int:
    """The same as device_status."""
    return int(load().sq_get_device_status(_stream(stream)))
