"""Host-side checks of the C-ABI library (no GPU needed): it builds, loads,
exports every function include/sq.h declares, and rejects bad arguments with
the documented status before touching the GPU."""
import ctypes
import os
import re

import pytest

from smoothquant_w8a8_int8_gb300 import build as sqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = sqbuild.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "sq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sq_pack_weight", "sq_quantize_act", "sq_linear_i8", "sq_channel_absmax",
              "sq_smooth_factor", "sq_device_status", "sq_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in sq.h but not exported"


def test_binding_covers_every_declared_symbol():
    from smoothquant_w8a8_int8_gb300 import binding
    assert sorted(binding.EXPORTS) == declared_functions()


def test_status_strings_and_sizes(lib):
    lib.sq_status_string.restype = ctypes.c_char_p
    lib.sq_status_string.argtypes = [ctypes.c_int]
    assert lib.sq_status_string(0) == b"SQ_OK"
    for code in range(1, 6):
        assert lib.sq_status_string(code).startswith(b"SQ_ERR_")
    assert b"unknown" in lib.sq_status_string(99)
    lib.sq_operand_bytes.restype = ctypes.c_size_t
    lib.sq_operand_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    assert lib.sq_operand_bytes(8192, 1024) == 8192 * 1024 * 2
    assert lib.sq_operand_bytes(-1, 16) == 0
    lib.sq_packed_weight_bytes.restype = ctypes.c_size_t
    lib.sq_packed_weight_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    assert lib.sq_packed_weight_bytes(4096, 1024) == 4096 * 1024 * 2
    assert lib.sq_version() >> 16 == 1


def _fake(addr):
    # a non-null, 16-byte aligned address that is never dereferenced: every
    # call below fails its host-side argument check before any CUDA call
    return ctypes.c_void_p(addr)


def test_argument_checks_fail_before_any_launch(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.sq_quantize_act.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp, vp]
    lib.sq_pack_weight.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp, vp]
    lib.sq_linear_i8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, vp]
    lib.sq_linear_i8_mma_sync.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, vp]
    lib.sq_smooth_factor.argtypes = [vp, vp, i64, ctypes.c_float, vp, vp]
    lib.sq_channel_absmax.argtypes = [vp, i64, i64, vp, vp]
    a = _fake(0x10000)
    INVALID, ALIGN, UNSUP = 1, 2, 3
    # quantiser
    assert lib.sq_quantize_act(None, a, 4, 32, a, a, None, None, None) == INVALID
    assert lib.sq_quantize_act(a, a, 4, 32, None, a, None, None, None) == INVALID   # no output
    assert lib.sq_quantize_act(a, a, 4, 32, a, None, None, None, None) == INVALID   # no scale
    assert lib.sq_quantize_act(a, a, -1, 32, a, a, None, None, None) == INVALID
    assert lib.sq_quantize_act(a, a, 4, 0, a, a, None, None, None) == INVALID
    assert lib.sq_quantize_act(a, a, 4, 24, a, a, None, None, None) == ALIGN       # K % 16
    assert lib.sq_quantize_act(_fake(0x10004), a, 4, 32, a, a, None, None, None) == ALIGN
    assert lib.sq_quantize_act(a, a, 0, 32, a, a, None, None, None) == 0           # empty: no launch
    assert lib.sq_quantize_act(None, None, 0, 32, None, None, None, None, None) == 0
    assert lib.sq_quantize_act(None, None, 0, 24, None, None, None, None, None) == ALIGN
    assert lib.sq_pack_weight(a, a, 4, 40, a, a, None, None, None) == ALIGN
    assert lib.sq_pack_weight(a, a, 0, 32, None, a, a, None, None) == 0
    # GEMM (the tcgen05 entry point also takes the two optional row-L1 arrays)
    def tc(X, sx, W, sw, b, r, M, N, K, mode, Y, st):
        return lib.sq_linear_i8(X, sx, None, W, sw, None, b, r, M, N, K, mode, Y, st)
    bad_l1 = lib.sq_linear_i8(a, a, _fake(0x10002), a, a, None, a, None, 8, 8, 32, 1, a, None)
    assert bad_l1 == ALIGN
    for fn in (tc, lib.sq_linear_i8_mma_sync):
        assert fn(None, a, a, a, a, None, 8, 8, 32, 1, a, None) == INVALID
        assert fn(a, a, a, a, None, None, 8, 8, 32, 1, a, None) == INVALID   # bias missing
        assert fn(a, a, a, a, a, None, 8, 8, 32, 3, a, None) == INVALID      # residual missing
        assert fn(a, a, a, a, a, a, 8, 8, 32, 5, a, None) == INVALID         # bad mode
        assert fn(a, a, a, a, a, a, 8, 8, 32, -1, a, None) == INVALID
        assert fn(a, a, a, a, a, None, 8, 8, 40, 1, a, None) == ALIGN
        assert fn(a, a, a, a, a, None, 8, 8, 133152, 1, a, None) == UNSUP  # |acc| could overflow
        assert fn(a, a, a, a, a, None, 8, 8, 32, 1, _fake(0x10008), None) == ALIGN
        assert fn(a, a, a, a, a, None, 0, 8, 32, 1, a, None) == 0          # empty
        assert fn(a, a, a, a, a, None, 8, 0, 32, 1, a, None) == 0
        assert fn(None, None, None, None, None, None, 0, 0, 32, 3, None, None) == 0
    # Smooth-Static
    lib.sq_act_absmax.argtypes = [vp, vp, i64, i64, vp, vp]
    lib.sq_quantize_act_static.argtypes = [vp, vp, i64, i64, ctypes.c_float, vp, vp, vp, vp, vp]
    assert lib.sq_act_absmax(None, a, 4, 32, a, None) == INVALID
    assert lib.sq_act_absmax(a, a, 4, 24, a, None) == ALIGN
    assert lib.sq_act_absmax(None, None, 0, 32, None, None) == 0
    lib.sq_static_scale.argtypes = [vp, vp, vp]
    assert lib.sq_static_scale(None, a, None) == INVALID
    assert lib.sq_static_scale(a, None, None) == INVALID
    assert lib.sq_static_scale(_fake(0x10002), a, None) == ALIGN
    assert lib.sq_quantize_act_static(a, a, 4, 32, 0.0, a, a, None, None, None) == INVALID
    assert lib.sq_quantize_act_static(a, a, 4, 32, -1.0, a, a, None, None, None) == INVALID
    assert lib.sq_quantize_act_static(a, a, 4, 32, float("inf"), a, a, None, None, None) == INVALID
    assert lib.sq_quantize_act_static(a, a, 4, 32, float("nan"), a, a, None, None, None) == INVALID
    assert lib.sq_quantize_act_static(a, a, 4, 32, 1.0, None, a, None, None, None) == INVALID
    assert lib.sq_quantize_act_static(a, a, 0, 32, 1.0, None, None, None, None, None) == 0
    # smoothing factor
    assert lib.sq_smooth_factor(a, a, 8, 1.5, a, None) == INVALID
    assert lib.sq_smooth_factor(a, a, 8, -0.1, a, None) == INVALID
    assert lib.sq_smooth_factor(a, None, 8, 0.5, a, None) == INVALID
    assert lib.sq_channel_absmax(a, 4, 0, a, None) == INVALID
    assert lib.sq_channel_absmax(a, 0, 4, a, None) == 0
    assert lib.sq_channel_absmax(None, 0, 4, None, None) == 0
    # producer-fused requantisation
    f = lib.sq_linear_i8_requant
    f.argtypes = [vp] * 8 + [i64, i64, i64, ctypes.c_int, vp, ctypes.c_float, vp, vp, vp, vp]
    assert f(a, a, None, a, a, None, a, None, 8, 8, 32, 4, a, 1.0, a, a, None, None) == INVALID
    assert f(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, 0.0, a, a, None, None) == INVALID
    assert f(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, float("inf"), a, a, None,
             None) == INVALID
    assert f(a, a, None, a, a, None, a, None, 8, 8, 32, 1, None, 1.0, a, a, None, None) == INVALID
    assert f(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, 1.0, None, None, None,
             None) == INVALID                                                # no code output
    assert f(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, 1.0, None, _fake(0x10001), None,
             None) == ALIGN                                                  # odd bf16 address
    assert f(a, a, None, a, a, None, a, None, 0, 8, 32, 1, None, 1.0, None, None, None,
             None) == 0                                                      # empty
    # division self-check: ranges within the 2^23 fraction fields, output aligned
    u32 = ctypes.c_uint32
    lib.sq_check_division.argtypes = [u32, u32, u32, u32, ctypes.c_int, vp, vp]
    F = 1 << 23
    assert lib.sq_check_division(F - 1, 2, 0, 1, 1, a, None) == INVALID
    assert lib.sq_check_division(0, 1, F, 1, 1, a, None) == INVALID
    assert lib.sq_check_division(0, 1, 0, 1, 1, None, None) == INVALID
    assert lib.sq_check_division(0, 1, 0, 1, 1, _fake(0x10004), None) == ALIGN
    assert lib.sq_check_division(0, 0, 0, 1, 1, None, None) == 0        # empty
    # fused LayerNorm + quantiser
    f = lib.sq_layernorm_quant
    f.argtypes = [vp, vp, vp, ctypes.c_float, vp, i64, i64, ctypes.c_float] + [vp] * 6
    assert f(a, a, a, -1.0, a, 4, 32, 0.0, None, a, a, None, None, None) == INVALID   # eps
    assert f(a, a, a, 1e-5, a, 4, 32, -1.0, None, a, a, None, None, None) == INVALID  # scale
    assert f(a, None, a, 1e-5, a, 4, 32, 0.0, None, a, a, None, None, None) == INVALID  # gamma
    assert f(a, a, a, 1e-5, a, 4, 24, 0.0, None, a, a, None, None, None) == ALIGN     # K % 16
    assert f(a, a, a, 1e-5, a, 4, 8208, 0.0, None, a, a, None, None, None) == UNSUP   # K > 8192
    assert f(None, None, None, 1e-5, None, 0, 32, 0.0, None, None, None, None, None, None) == 0


def test_workspace_entry_points_check_arguments_first(lib):
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    INVALID, ALIGN, UNSUP = 1, 2, 3
    a = _fake(0x10000)
    wb = lib.sq_linear_workspace_bytes
    wb.argtypes = [i64, i64, i64, vp]
    n = ctypes.c_size_t(123)
    assert wb(8, 8, 32, None) == INVALID
    assert wb(-1, 8, 32, ctypes.byref(n)) == INVALID
    assert wb(8, 8, 0, ctypes.byref(n)) == INVALID
    assert wb(8, 8, 133152, ctypes.byref(n)) == UNSUP
    assert wb(0, 8, 32, ctypes.byref(n)) == 0 and n.value == 0     # empty: no workspace
    ws = lib.sq_linear_i8_ws
    ws.argtypes = [vp] * 8 + [i64, i64, i64, i32, vp, vp, sz, vp]
    assert ws(None, a, None, a, a, None, a, None, 8, 8, 32, 1, a, a, 1 << 20, None) == INVALID
    assert ws(a, a, None, a, a, None, a, None, 8, 8, 40, 1, a, a, 1 << 20, None) == ALIGN
    assert ws(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, _fake(0x10008), 1 << 20,
              None) == ALIGN                                           # workspace alignment
    assert ws(a, a, None, a, a, None, a, None, 0, 8, 32, 1, a, None, 0, None) == 0
    rq = lib.sq_linear_i8_requant_ws
    rq.argtypes = [vp] * 8 + [i64, i64, i64, i32, vp, ctypes.c_float, vp, vp, vp, vp, sz, vp]
    assert rq(a, a, None, a, a, None, a, None, 8, 8, 32, 4, a, 1.0, a, a, None, a, 1 << 20,
              None) == INVALID                                         # raw int32 mode
    assert rq(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, 1.0, a, a, None, _fake(0x10004),
              1 << 20, None) == ALIGN
    cb = lib.sq_linear_codes_workspace_bytes
    cb.argtypes = [i64, i64, vp]
    assert cb(8, 32, None) == INVALID
    assert cb(-1, 32, ctypes.byref(n)) == INVALID
    assert cb(8, 40, ctypes.byref(n)) == ALIGN
    assert cb(8, 133152, ctypes.byref(n)) == UNSUP
    assert cb(3, 32, ctypes.byref(n)) == 0 and n.value == 256       # 2*3*32 rounded up
    assert cb(1024, 1024, ctypes.byref(n)) == 0 and n.value == 2 << 20
    cd = lib.sq_linear_i8_codes
    cd.argtypes = [vp] * 8 + [i64, i64, i64, i32, vp, vp, sz, vp]
    assert cd(None, a, None, a, a, None, a, None, 8, 8, 32, 1, a, a, 1 << 20, None) == INVALID
    assert cd(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, None, 1 << 20, None) == INVALID
    assert cd(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, a, 256, None) == INVALID  # small
    assert cd(_fake(0x10004), a, None, a, a, None, a, None, 8, 8, 32, 1, a, a, 1 << 20,
              None) == ALIGN
    assert cd(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, _fake(0x10008), 1 << 20,
              None) == ALIGN
    assert cd(a, a, None, a, a, None, None, None, 8, 8, 32, 1, a, a, 1 << 20,
              None) == INVALID                                         # bias mode, no bias
    assert cd(a, a, None, a, a, None, a, None, 8, 8, 40, 1, a, a, 1 << 20, None) == ALIGN
    assert cd(None, None, None, None, None, None, None, None, 0, 8, 32, 1, None, None, 0,
              None) == 0
    st = lib.sq_linear_i8_static_ws
    st.argtypes = [vp] * 8 + [i64, i64, i64, i32, vp, vp]
    assert st(a, a, None, a, a, None, a, None, 8, 8, 133152, 1, a, None) == UNSUP
    assert st(a, a, None, a, a, None, a, None, -1, 8, 32, 1, a, None) == INVALID
    assert st(None, None, None, None, None, None, None, None, 0, 8, 32, 1, None, None) == 0
    assert st(None, None, None, None, None, None, None, None, 0, 8, 24, 1, None, None) == ALIGN
    # the static-scratch entry point checks its arguments exactly as the
    # caller-workspace one does: the same status for every call below
    f4 = _fake(0x10004)
    cases = [(None, a, None, a, a, None, a, None, 8, 8, 32, 1, a),       # X missing
             (a, a, None, a, a, None, None, None, 8, 8, 32, 1, a),       # bias missing
             (a, a, None, a, a, None, a, None, 8, 8, 32, 3, a),          # residual missing
             (a, a, None, a, a, None, a, a, 8, 8, 32, 7, a),             # bad mode
             (a, a, None, a, a, None, a, None, 8, 8, 40, 1, a),          # K % 16
             (a, a, f4, a, a, None, a, None, 8, 8, 32, 1, a),            # x_l1 alignment ok (4)
             (a, a, _fake(0x10002), a, a, None, a, None, 8, 8, 32, 1, a),  # x_l1 misaligned
             (a, a, None, a, a, None, a, None, 8, 8, 133152, 1, a),      # K too large
             (a, a, None, a, a, None, a, None, 8, 8, 32, 1, _fake(0x10008)),  # Y misaligned
             (a, a, None, a, a, None, a, None, -3, 8, 32, 1, a)]
    for c in cases:
        assert st(*c, None) == ws(*c, None, 0, None), c
    # producer-fused dynamic quantisation
    dt = lib.sq_division_table
    dt.argtypes = [vp, i64, vp, vp]
    assert dt(None, 8, a, None) == INVALID
    assert dt(a, -1, a, None) == INVALID
    assert dt(a, 8, _fake(0x10008), None) == ALIGN
    assert dt(None, 0, None, None) == 0
    rm = lib.sq_linear_i8_rowmax
    rm.argtypes = [vp] * 8 + [i64, i64, i64, i32, vp, vp, vp, vp]
    assert rm(a, a, None, a, a, None, a, None, 8, 8, 32, 4, a, a, a, None) == INVALID  # raw
    assert rm(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, None, a, None) == INVALID
    assert rm(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, a, None, None) == INVALID
    assert rm(a, a, None, a, a, None, a, None, 8, 8, 32, 1, a, _fake(0x10008), a,
              None) == ALIGN
    assert rm(a, a, None, a, a, None, a, None, 8, 8, 40, 1, a, a, a, None) == ALIGN
    assert rm(None, None, None, None, None, None, None, None, 0, 8, 32, 1, None, None, None,
              None) == 0
    qr = lib.sq_quantize_act_rowmax
    qr.argtypes = [vp, vp, vp, i64, i64, vp, vp, vp, vp, vp]
    assert qr(a, a, None, 4, 32, a, a, None, None, None) == INVALID     # no maxima
    assert qr(a, a, a, 4, 32, None, a, None, None, None) == INVALID     # no output
    assert qr(a, a, _fake(0x10002), 4, 32, a, a, None, None, None) == ALIGN
    assert qr(None, None, None, 0, 32, None, None, None, None, None) == 0
    qt = lib.sq_quantize_act_table
    qt.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, vp]
    assert qt(a, a, None, None, 4, 32, a, a, None, None, None) == INVALID   # no table
    assert qt(a, None, a, None, 4, 32, a, a, None, None, None) == INVALID   # no s
    assert qt(a, a, a, None, 4, 32, None, a, None, None, None) == INVALID   # no output
    assert qt(a, a, _fake(0x10008), None, 4, 32, a, a, None, None, None) == ALIGN
    assert qt(a, a, a, _fake(0x10002), 4, 32, a, a, None, None, None) == ALIGN  # maxima
    assert qt(a, a, a, None, 4, 40, a, a, None, None, None) == ALIGN        # K % 16
    assert qt(None, None, None, None, 0, 32, None, None, None, None, None) == 0
    # the host-buffer pipeline: argument checks before anything is enqueued
    from smoothquant_w8a8_int8_gb300.binding import LinearLayerC
    hb = lib.sq_linear_block_host_scratch_bytes
    hb.argtypes = [i64, i64, i64, ctypes.POINTER(ctypes.c_size_t)]
    nb = ctypes.c_size_t(0)
    assert hb(8, 32, 16, None) == INVALID
    assert hb(8, 0, 16, ctypes.byref(nb)) == INVALID
    assert hb(8, 32, 16, ctypes.byref(nb)) == 0
    assert nb.value == 2 * 1024 + 2 * 512 + 512 + 256   # 256-byte parts: x, y slots, operand, scales
    hp = lib.sq_linear_block_host
    hp.argtypes = [ctypes.POINTER(LinearLayerC), i64, i64, vp, vp, vp, ctypes.c_size_t, vp, vp, vp]
    lay = LinearLayerC(32, 16, 1, 0.0, 0x10000, None, 0x10000, 0x10000, None, 0x10000, None)
    arr = (LinearLayerC * 1)(lay)
    hx = (ctypes.c_void_p * 1)(0x20000)
    hy = (ctypes.c_void_p * 1)(0x30000)
    big = 1 << 20
    assert hp(arr, 1, 8, hx, hy, None, big, None, None, None) == INVALID            # no scratch
    assert hp(arr, 1, 8, hx, hy, _fake(0x10010), big, None, None, None) == ALIGN   # scratch
    assert hp(arr, 1, 8, hx, hy, a, 100, None, None, None) == INVALID             # too small
    assert hp(None, 1, 8, hx, hy, a, big, None, None, None) == INVALID
    assert hp(arr, 1, 8, None, hy, a, big, None, None, None) == INVALID
    assert hp(arr, -1, 8, hx, hy, a, big, None, None, None) == INVALID
    assert hp(None, 0, 8, None, None, None, 0, None, None, None) == 0             # empty
    bad = [LinearLayerC(40, 16, 1, 0.0, 0x10000, None, 0x10000, 0x10000, None, 0x10000, None),
           LinearLayerC(32, 16, 7, 0.0, 0x10000, None, 0x10000, 0x10000, None, 0x10000, None),
           LinearLayerC(32, 16, 1, 0.0, None, None, 0x10000, 0x10000, None, 0x10000, None),
           LinearLayerC(32, 16, 1, 0.0, 0x10004, None, 0x10000, 0x10000, None, 0x10000, None),
           LinearLayerC(32, 16, 1, -1.0, 0x10000, None, 0x10000, 0x10000, None, 0x10000, None),
           LinearLayerC(32, 16, 1, 0.0, 0x10000, None, 0x10000, 0x10000, None, None, None)]
    want = [ALIGN, INVALID, INVALID, ALIGN, INVALID, INVALID]   # K % 16, mode, s, s, scale, bias
    for L, w in zip(bad, want):
        assert hp((LinearLayerC * 1)(L), 1, 8, hx, hy, a, big, None, None, None) == w, (L.K, w)
    at = lib.sq_attention
    at.argtypes = [vp, i64, i64, i64, i64, ctypes.c_float, vp, vp]
    assert at(a, 2, 128, 4, 64, 0.125, None, None) == INVALID
    assert at(a, -1, 128, 4, 64, 0.125, a, None) == INVALID
    assert at(a, 2, 128, 4, 64, float("nan"), a, None) == INVALID
    assert at(a, 2, 128, 4, 32, 0.125, a, None) == UNSUP          # head dimension
    assert at(a, 2, 100, 4, 64, 0.125, a, None) == UNSUP          # S % 64
    assert at(a, 2, 512, 4, 64, 0.125, a, None) == UNSUP          # S > 448
    assert at(a, 1 << 25, 64, 4, 64, 0.125, a, None) == UNSUP     # B*S = 2^31
    assert at(a, 2, 128, 65537, 64, 0.125, a, None) == UNSUP      # H
    assert at(_fake(0x10008), 2, 128, 4, 64, 0.125, a, None) == ALIGN
    assert at(None, 0, 128, 4, 64, 0.125, None, None) == 0
    sw = lib.sq_static_workspace
    sw.argtypes = [vp, vp]
    assert sw(None, ctypes.byref(n)) == INVALID
    assert sw(ctypes.byref(ctypes.c_void_p()), None) == INVALID
