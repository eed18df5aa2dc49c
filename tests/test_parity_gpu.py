"""GPU parity: every kernel through the C-ABI against the CPU oracle on the
same seeded inputs.  Codes, scale bit patterns and int32 accumulators must
match exactly; fp32 outputs within max|err| <= 1e-5 max|ref| + 1e-6."""
import os

import numpy as np
import pytest
import torch

import oracle
from paritylib import (assert_bits_equal, assert_close_fp32, assert_codes_equal, op_as_int,
                       oracle_smoothing, to_dev)
from smoothquant_w8a8_int8_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

PATHS = ["tc", "mma_sync"]


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


def gpu_pack(sq, W, s):
    Wq, sw, Wop = sq.pack_weight(to_dev(W), to_dev(s))
    return Wq, sw, Wop


def gpu_linear(sq, path, Xq, Xop, sx, Wq, Wop, sw, bias=None, residual=None,
               mode=wl.EPI_BIAS):
    if path == "tc":
        return sq.linear_i8(Xop, sx, Wop, sw, bias, residual, mode)
    return sq.linear_i8_mma_sync(Xq, sx, Wq, sw, bias, residual, mode)


# ------------------------------------------------------------------ quantiser

# The last rows span many staged chunks per SM with a ragged final chunk (the
# activation quantiser streams each SM's row range through a ring of stages).
QUANT_SHAPES = [(1, 16), (7, 48), (37, 1024), (130, 768), (64, 4096), (300, 3072), (3, 8192),
                (5, 8208), (2, 16384), (6847, 1024), (1900, 4096), (4000, 768), (777, 3072)]


@pytest.mark.parametrize("M,K", QUANT_SHAPES)
def test_quantize_act_parity(sq, M, K):
    c = wl.make_case(M, K, 8, wl.EPI_BIAS, seed=M * 31 + K)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle_smoothing(X, W, 0.5)
    q_ref, sx_ref = oracle.quantize_rows(X, s, "act")
    Xq, sx, Xop, l1 = sq.quantize_act(to_dev(X), to_dev(s), want_l1=True)
    torch.cuda.synchronize()
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    assert_codes_equal(op_as_int(Xop), q_ref, "Xop")
    np.testing.assert_array_equal(l1.cpu().numpy(), np.abs(q_ref.astype(np.int64)).sum(axis=1))
    # each output alone
    _, sx2, Xop2 = sq.quantize_act(to_dev(X), to_dev(s), want_q=False)
    Xq3, sx3, _ = sq.quantize_act(to_dev(X), to_dev(s), want_op=False)
    assert_codes_equal(op_as_int(Xop2), q_ref, "Xop only")
    assert_codes_equal(Xq3.cpu().numpy(), q_ref, "Xq only")
    assert_bits_equal(sx2.cpu().numpy(), sx_ref, "x_scale (op only)")


def test_quantize_degenerate_rows(sq):
    K = 64
    X = np.zeros((6, K), np.float32)
    X[1, 3] = -2.5                      # one-hot row
    X[2, :] = 1.0                       # constant row -> all 127
    X[3, ::2], X[3, 1::2] = 3.0, -3.0   # alternating signs
    X[4, :] = np.float32(1e-30)         # tiny values
    X[5, 0], X[5, 1] = 127.0, -63.5     # ties: -63.5 -> -64
    s = np.ones(K, np.float32)
    q_ref, sx_ref = oracle.quantize_rows(X, s, "act")
    Xq, sx, Xop = sq.quantize_act(to_dev(X), to_dev(s))
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    assert sx.cpu().numpy()[0] == 1.0 and not Xq.cpu().numpy()[0].any()


def test_quantize_ties_and_near_ties(sq):
    """Codes whose quotient is a half-integer or within a few ulp of one:
    the cases where round-half-to-even decides and a rounding slip shows."""
    K = 256
    ties = np.concatenate([np.arange(-127, 127) + 0.5, [127.0, 0.0]]).astype(np.float32)
    rows = [ties,                                   # scale 1: exact ties
            ties * np.float32(2.0 ** -7),           # scale 2^-7: exact ties
            ties * np.float32(1 + 2.0 ** -20),      # just above the ties
            ties * np.float32(1 - 2.0 ** -20)]      # just below
    rng = np.random.default_rng(5)
    sc = np.float32(0.7531)
    k = rng.integers(-126, 126, K).astype(np.float32)
    r = ((k + np.float32(0.5)) * sc).astype(np.float32)
    r[0] = np.float32(127) * sc                     # amax -> scale close to sc
    rows.append(r)
    for ulps in (-2, -1, 1, 2):                     # quotients within ulps of a tie
        rows.append(np.nextafter(r, np.float32(np.inf) if ulps > 0 else np.float32(-np.inf))
                    if abs(ulps) == 1 else
                    np.nextafter(np.nextafter(r, np.float32(np.sign(ulps) * np.inf)),
                                 np.float32(np.sign(ulps) * np.inf)))
    X = np.stack(rows).astype(np.float32)
    s = np.ones(K, np.float32)
    q_ref, sx_ref = oracle.quantize_rows(X, s, "act")
    Xq, sx, Xop = sq.quantize_act(to_dev(X), to_dev(s))
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    assert_codes_equal(op_as_int(Xop), q_ref, "Xop")
    np.testing.assert_array_equal(q_ref[0, :254], np.round(ties[:254]).astype(np.int8))


def test_quantize_row_max_near_ties(sq):
    """Rows whose smoothed values x/s are all within a few ulp of each other,
    so that only exact division finds the row maximum; rows of tiny and of
    very large values (where reciprocal estimates lose their error bound)."""
    rng = np.random.default_rng(9)
    K = 1024
    s = (rng.uniform(0.05, 20.0, K)).astype(np.float32)
    rows = []
    for target in (1.0, 3.7, 1e-3, 250.0):
        x = (np.float32(target) * s).astype(np.float32)           # x/s = target +- 1 ulp
        x *= rng.choice(np.array([-1, 1], np.float32), K)
        rows.append(x)
    rows.append((rng.standard_normal(K) * 1e-36).astype(np.float32))  # tiny / subnormal
    rows.append((rng.standard_normal(K) * 1e35).astype(np.float32))   # large
    big = np.zeros(K, np.float32)
    big[7] = np.float32(1.5e37 * float(s[7]))                       # quotient near 1.5e37
    rows.append(big)
    X = np.stack(rows).astype(np.float32)
    q_ref, sx_ref = oracle.quantize_rows(X, s, "act")
    Xq, sx, Xop = sq.quantize_act(to_dev(X), to_dev(s))
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_codes_equal(op_as_int(Xop), q_ref, "Xop")


# 1024 and 4096: the register kernel on rows of 1024 * 2^k; 3072: the register
# kernel on rows it fills unevenly; 768: the ring kernel (the rows repeated to
# 2520, at least 16 per SM of a GB300, where the dispatch takes the ring)
@pytest.mark.parametrize("K", [768, 1024, 3072, 4096])
def test_quantize_extreme_magnitudes(sq, K):
    """Rows whose largest |x/s| sits at extreme magnitudes (2^-61 .. 2^101,
    each a hair below, at and above a power of two), smoothing factors far
    outside the usual range (1e-7, 3e7), and static scales from 2^-71 to
    2^98: codes, scales and L1 norms bit for bit (dynamic and static)."""
    rng = np.random.default_rng(K)
    s = rng.uniform(0.05, 20.0, K).astype(np.float32)
    base = rng.standard_normal(K).astype(np.float32)
    base /= np.abs(base).max()
    rows = []
    for m in (2.0 ** -60, 2.0 ** -59, 2.0 ** -61, 2.0 ** 100, 2.0 ** 99, 2.0 ** 101):
        for f in (np.float32(1 - 2.0 ** -20), np.float32(1), np.float32(1 + 2.0 ** -20)):
            rows.append((base * np.float32(m) * f * s).astype(np.float32))
    X = np.stack(rows).astype(np.float32)
    if K == 768:
        X = np.tile(X, (140, 1))
    for s_case in (s, np.where(np.arange(K) == 5, np.float32(1e-7), s).astype(np.float32),
                   np.where(np.arange(K) == 9, np.float32(3e7), s).astype(np.float32)):
        q_ref, sx_ref = oracle.quantize_rows(X, s_case, "act")
        Xq, sx, Xop, l1 = sq.quantize_act(to_dev(X), to_dev(s_case), want_l1=True)
        assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
        assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
        assert_codes_equal(op_as_int(Xop), q_ref, "Xop")
        np.testing.assert_array_equal(l1.cpu().numpy(),
                                      np.abs(q_ref.astype(np.int64)).sum(axis=1))
        for scale in (np.float32(2.0 ** -71), np.float32(2.0 ** -69), np.float32(3.0),
                      np.float32(2.0 ** 98)):
            q_ref = oracle.quantize_static(X, s_case, scale)
            Xq, _, Xop = sq.quantize_act_static(to_dev(X), to_dev(s_case), float(scale))
            assert_codes_equal(Xq.cpu().numpy(), q_ref, f"static Xq, scale {scale}")
            assert_codes_equal(op_as_int(Xop), q_ref, f"static Xop, scale {scale}")


# The register kernel builds its tables of s while the kernel before it on the
# stream may still run, then checks s after the wait: here that kernel is the
# library's smoothing-factor kernel rewriting the same buffer each time.
@pytest.mark.parametrize("M,K", [(2400, 1024), (700, 4096)])
def test_quantize_after_smoothing_factor_rewrite(sq, M, K):
    rng = np.random.default_rng(M + K)
    X = (rng.standard_normal((M, K)) * 2).astype(np.float32)
    X[:, 7] *= 40.0
    ax = np.abs(X).max(axis=0).astype(np.float32)
    aw = np.abs(rng.standard_normal(K) * 0.05).astype(np.float32) + np.float32(1e-3)
    lib, st = sq.load(), torch.cuda.current_stream().cuda_stream
    X_d, ax_d, aw_d = to_dev(X), to_dev(ax), to_dev(aw)
    s_buf = to_dev(np.ones(K, np.float32))
    Xq = torch.empty(M, K, dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    Xop = sq.empty_operand(M, K)
    torch.cuda.synchronize()
    outs = []
    for alpha in (0.5, 0.8, 0.25, 0.5, 0.65, 0.9):
        rc = lib.sq_smooth_factor(ax_d.data_ptr(), aw_d.data_ptr(), K, alpha, s_buf.data_ptr(),
                                  st)
        assert rc == 0
        sq.quantize_act(X_d, s_buf, out=(Xq, sx, Xop))
        outs.append((s_buf.clone(), Xq.clone(), sx.clone(), Xop.clone()))
    torch.cuda.synchronize()
    for s_used, q, scale, op in outs:
        q_ref, sx_ref = oracle.quantize_rows(X, s_used.cpu().numpy(), "act")
        assert_bits_equal(scale.cpu().numpy(), sx_ref, "x_scale")
        assert_codes_equal(q.cpu().numpy(), q_ref, "Xq")
        assert_codes_equal(op_as_int(op), q_ref, "Xop")


@pytest.mark.parametrize("N,K", [(1, 16), (5, 48), (1024, 1024), (3072, 1024), (768, 3072),
                                 (9, 8208)])
def test_pack_weight_parity(sq, N, K):
    c = wl.make_case(16, K, N, wl.EPI_BIAS, seed=N + K)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle_smoothing(X, W, 0.5)
    q_ref, sw_ref = oracle.quantize_rows(W, s, "weight")
    Wq, sw, Wop, l1 = sq.pack_weight(to_dev(W), to_dev(s), want_l1=True)
    torch.cuda.synchronize()
    assert_codes_equal(Wq.cpu().numpy(), q_ref, "Wq")
    assert_bits_equal(sw.cpu().numpy(), sw_ref, "w_scale")
    assert_codes_equal(op_as_int(Wop), q_ref, "Wop")
    np.testing.assert_array_equal(l1.cpu().numpy(), np.abs(q_ref.astype(np.int64)).sum(axis=1))


# ------------------------------------------------------------ smoothing factor

@pytest.mark.parametrize("rows,cols", [(1, 16), (33, 100), (8192, 1024), (3, 4096)])
def test_channel_absmax_parity(sq, rows, cols):
    rng = np.random.default_rng(rows + cols)
    A = rng.standard_normal((rows, cols)).astype(np.float32)
    B = (rng.standard_normal((rows, cols)) * 3).astype(np.float32)
    amax = sq.channel_absmax(to_dev(A))
    np.testing.assert_array_equal(amax.cpu().numpy(), oracle.channel_absmax(A))
    sq.channel_absmax(to_dev(B), amax)           # running max over two batches
    want = np.maximum(oracle.channel_absmax(A), oracle.channel_absmax(B))
    np.testing.assert_array_equal(amax.cpu().numpy(), want)


@pytest.mark.parametrize("alpha", [0.5, 0.6, 0.75, 0.0, 1.0])
def test_smooth_factor_parity(sq, alpha):
    rng = np.random.default_rng(11)
    ax = np.abs(rng.standard_normal(4096) * 5).astype(np.float32)
    aw = np.abs(rng.standard_normal(4096) * 0.05).astype(np.float32)
    ax[:3] = 0.0
    aw[10:12] = 0.0
    s = sq.smooth_factor(to_dev(ax), to_dev(aw), alpha).cpu().numpy()
    ref = oracle.smooth_factor(ax, aw, np.float32(alpha))
    # double pow on both sides, one rounding to fp32: equal up to 1 ulp
    ulp = np.abs(s.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1
    if alpha in (0.5, 0.0, 1.0):
        assert ulp.max() == 0


# ----------------------------------------------------------------- GEMM

GEMM_SHAPES = [(1, 1, 16), (5, 7, 48), (129, 130, 1040), (200, 300, 2064), (128, 256, 1024),
               (256, 1024, 4096), (300, 260, 3072), (64, 96, 5008)]


def _quantised_case(sq, M, K, N, mode, seed):
    c = wl.make_case(M, K, N, mode, seed=seed)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle_smoothing(X, W, 0.5)
    wq, sw = oracle.quantize_rows(W, s, "weight")
    xq, sx = oracle.quantize_rows(X, s, "act")
    dev = dict(Xq=to_dev(xq), sx=to_dev(sx), Wq=to_dev(wq), sw=to_dev(sw),
               Xop=to_dev(xq.astype(np.float32), torch.bfloat16),
               Wop=to_dev(wq.astype(np.float32), torch.bfloat16))
    return c, xq, sx, wq, sw, dev


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_raw_int32_exact(sq, path, M, N, K):
    _, xq, _, wq, _, d = _quantised_case(sq, M, K, N, wl.EPI_NONE, seed=M + N + K)
    acc = gpu_linear(sq, path, d["Xq"], d["Xop"], None, d["Wq"], d["Wop"], None,
                     mode=sq.EPI_RAW_I32)
    assert_codes_equal(acc.cpu().numpy(), oracle.gemm_i32(xq, wq), "acc")


# Shapes with more tiles (128 x 256) than a GB300 has SMs and a partial last
# wave of at most half the SMs: the tcgen05 GEMM cuts that wave's tiles into
# 128-column halves.
#   (2560, 2304): 180 tiles, 28 in the last wave -> halves
#   (2560, 2816): 220 tiles, 68 in the last wave -> halves
#   (2560, 3328): 260 tiles, 108 in the last wave -> no split (control)
# K = 1088 takes two exact fp32 chunks (no L1 bound passed); 4096 with
# residual exercises the multi-chunk epilogue with the residual prefetch.
SPLIT_SHAPES = [(2560, 2304, 1088, wl.EPI_NONE), (2560, 2816, 256, wl.EPI_BIAS_GELU),
                (2560, 3328, 512, wl.EPI_BIAS), (2560, 2304, 4096, wl.EPI_BIAS_RESIDUAL)]


@pytest.mark.parametrize("M,N,K,mode", SPLIT_SHAPES)
def test_gemm_tail_wave_slices(sq, M, N, K, mode):
    c, xq, sx, wq, sw, d = _quantised_case(sq, M, K, N, wl.EPI_BIAS_RESIDUAL, seed=M + N + K)
    acc_ref = oracle.gemm_i32(xq, wq)
    acc = sq.linear_i8(d["Xop"], None, d["Wop"], None, None, None, sq.EPI_RAW_I32)
    assert_codes_equal(acc.cpu().numpy(), acc_ref, "acc")
    if mode != wl.EPI_NONE:
        b, r = c.bias.numpy(), c.residual.numpy()
        ref = oracle.epilogue(acc_ref, sx, sw, b, r, mode)
        y = sq.linear_i8(d["Xop"], d["sx"], d["Wop"], d["sw"], to_dev(b),
                         to_dev(r) if mode == wl.EPI_BIAS_RESIDUAL else None, mode)
        assert_close_fp32(y.cpu().numpy(), ref, f"mode {mode}")


# CTA-pair shapes (M >= 256) with a partial last wave of 256 x 256 tiles.  On
# 152 SMs (76 clusters):
#   (2048, 2560): 80 tiles, 4 in the last wave -> 256 x 128 halves, whose 128
#     columns the two epilogue warps of a lane quarter split 64 / 64
#   (2304, 3584): 126 tiles, 50 in the last wave -> whole tiles (control)
# K = 1088 without row L1 norms takes two exact passes (the chunked epilogue,
# whose int32 partial each warp keeps in its own columns from item to item).
PAIR_TAIL_SHAPES = [(2048, 2560, 256, wl.EPI_BIAS), (2304, 3584, 256, wl.EPI_BIAS_RESIDUAL),
                    (2304, 3584, 1088, wl.EPI_BIAS_GELU), (2048, 2560, 1088, wl.EPI_BIAS_RESIDUAL)]


@pytest.mark.parametrize("M,N,K,mode", PAIR_TAIL_SHAPES)
def test_pair_tail_halves(sq, M, N, K, mode):
    c, xq, sx, wq, sw, d = _quantised_case(sq, M, K, N, wl.EPI_BIAS_RESIDUAL, seed=M + 3 * N + K)
    acc_ref = oracle.gemm_i32(xq, wq)
    acc = sq.linear_i8(d["Xop"], None, d["Wop"], None, None, None, sq.EPI_RAW_I32)
    assert_codes_equal(acc.cpu().numpy(), acc_ref, "acc")
    b, r = c.bias.numpy(), c.residual.numpy()
    ref = oracle.epilogue(acc_ref, sx, sw, b, r, mode)
    y = sq.linear_i8(d["Xop"], d["sx"], d["Wop"], d["sw"], to_dev(b),
                     to_dev(r) if mode == wl.EPI_BIAS_RESIDUAL else None, mode)
    assert_close_fp32(y.cpu().numpy(), ref, f"mode {mode}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("K", [1024, 1040, 2048, 4096, 8192])
def test_gemm_adversarial_exactness(sq, path, K):
    """Worst-case sums: all +127 (K * 16129, above 2^24 once K > 1024),
    alternating signs that cancel, and random +-127."""
    M, N = 160, 136
    rng = np.random.default_rng(K)
    xq = np.full((M, K), 127, np.int8)
    wq = np.full((N, K), 127, np.int8)
    xq[1::3, 1::2] = -127
    wq[2::5, :] = -127
    xq[100:] = rng.choice(np.array([-127, 127], np.int8), (M - 100, K))
    wq[100:] = rng.choice(np.array([-127, 127], np.int8), (N - 100, K))
    xq[50, :] = 0
    acc = gpu_linear(sq, path, to_dev(xq), to_dev(xq.astype(np.float32), torch.bfloat16), None,
                     to_dev(wq), to_dev(wq.astype(np.float32), torch.bfloat16), None,
                     mode=sq.EPI_RAW_I32)
    ref = oracle.gemm_i32(xq, wq)
    assert ref[0, 0] == K * 16129
    assert_codes_equal(acc.cpu().numpy(), ref, "acc")
    if path == "tc":
        # with the row L1 norms passed: these rows exceed the single-pass bound
        xl1 = to_dev(np.abs(xq.astype(np.int64)).sum(1).astype(np.int32))
        wl1 = to_dev(np.abs(wq.astype(np.int64)).sum(1).astype(np.int32))
        acc = sq.linear_i8(to_dev(xq.astype(np.float32), torch.bfloat16), None,
                           to_dev(wq.astype(np.float32), torch.bfloat16), None,
                           mode=sq.EPI_RAW_I32, x_l1=xl1, w_l1=wl1)
        assert_codes_equal(acc.cpu().numpy(), ref, "acc (row L1 given)")


@pytest.mark.parametrize("limit_ok", [True, False])
@pytest.mark.parametrize("K", [2048, 4096])
def test_gemm_single_pass_bound(sq, limit_ok, K):
    """At the single-pass limit (127 * L1 < 2^24) the whole K is summed in one
    fp32 pass; one more unit of L1 forces chunks.  Both must be exact: the
    boundary rows make the sum 127 * 132104 = 16,777,208 = 2^24 - 8."""
    M, N = 130, 144
    L1 = 132104 if limit_ok else 132105
    xq = np.zeros((M, K), np.int8)
    full, rest = divmod(L1, 127)
    xq[:, :full] = 127
    xq[:, full] = rest
    xq[1::2] = -xq[1::2]
    rng = np.random.default_rng(K + L1)
    xq[64:] = np.clip(rng.integers(-3, 4, (M - 64, K)), -127, 127).astype(np.int8)
    xq[64:, :4] = 127                                   # keep every row's max code 127
    wq = np.full((N, K), 127, np.int8)
    wq[N // 2:] = rng.choice(np.array([-127, 127], np.int8), (N - N // 2, K))
    xl1 = np.abs(xq.astype(np.int64)).sum(1).astype(np.int32)
    assert xl1.max() == L1
    ref = oracle.gemm_i32(xq, wq)
    acc = sq.linear_i8(to_dev(xq.astype(np.float32), torch.bfloat16), None,
                       to_dev(wq.astype(np.float32), torch.bfloat16), None, mode=sq.EPI_RAW_I32,
                       x_l1=to_dev(xl1))
    assert_codes_equal(acc.cpu().numpy(), ref, "acc")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("mode", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU,
                                  wl.EPI_BIAS_RESIDUAL])
@pytest.mark.parametrize("M,N,K", [(77, 136, 1024), (256, 512, 3072)])
def test_epilogue_modes(sq, path, mode, M, N, K):
    c, xq, sx, wq, sw, d = _quantised_case(sq, M, K, N, wl.EPI_BIAS_RESIDUAL, seed=mode + M)
    acc = oracle.gemm_i32(xq, wq)
    b, r = c.bias.numpy(), c.residual.numpy()
    ref = oracle.epilogue(acc, sx, sw, b, r, mode)
    y = gpu_linear(sq, path, d["Xq"], d["Xop"], d["sx"], d["Wq"], d["Wop"], d["sw"],
                   to_dev(b), to_dev(r), mode)
    assert_close_fp32(y.cpu().numpy(), ref, f"mode {mode}")


@pytest.mark.parametrize("path", PATHS)
def test_gelu_sweep(sq, path):
    """GELU(erf) over pre-activations spanning [-10, 10], against the oracle's
    double-precision erf."""
    M, N, K = 128, 256, 16
    xq = np.zeros((M, K), np.int8)
    wq = np.zeros((N, K), np.int8)
    xq[:, 0] = np.arange(M) - 64                    # -64 .. 63
    wq[:, 0] = (np.arange(N) % 127) - 63            # -63 .. 63
    sx = np.ones(M, np.float32)
    sw = np.full(N, 1.0 / 400.0, np.float32)        # d in about [-10, 10]
    b = np.linspace(-0.5, 0.5, N).astype(np.float32)
    ref = oracle.epilogue(oracle.gemm_i32(xq, wq), sx, sw, b, mode=oracle.EPI_BIAS_GELU)
    y = gpu_linear(sq, path, to_dev(xq), to_dev(xq.astype(np.float32), torch.bfloat16),
                   to_dev(sx), to_dev(wq), to_dev(wq.astype(np.float32), torch.bfloat16),
                   to_dev(sw), to_dev(b), None, wl.EPI_BIAS_GELU)
    assert_close_fp32(y.cpu().numpy(), ref, "gelu sweep")


@pytest.mark.parametrize("path", PATHS)
def test_residual_in_place(sq, path):
    c, xq, sx, wq, sw, d = _quantised_case(sq, 96, 1024, 160, wl.EPI_BIAS_RESIDUAL, seed=3)
    ref = oracle.epilogue(oracle.gemm_i32(xq, wq), sx, sw, c.bias.numpy(), c.residual.numpy(),
                          wl.EPI_BIAS_RESIDUAL)
    r = to_dev(c.residual.numpy())
    fn = sq.linear_i8 if path == "tc" else sq.linear_i8_mma_sync
    a, w = (d["Xop"], d["Wop"]) if path == "tc" else (d["Xq"], d["Wq"])
    fn(a, d["sx"], w, d["sw"], to_dev(c.bias.numpy()), r, wl.EPI_BIAS_RESIDUAL, out=r)
    assert_close_fp32(r.cpu().numpy(), ref, "in-place residual")


def test_zero_input_gives_bias_and_residual(sq):
    M, N, K = 40, 72, 256
    X = np.zeros((M, K), np.float32)
    W = np.random.default_rng(0).standard_normal((N, K)).astype(np.float32)
    s = np.ones(K, np.float32)
    b = np.linspace(-1, 1, N).astype(np.float32)
    r = np.random.default_rng(1).standard_normal((M, N)).astype(np.float32)
    _, sx, Xop = sq.quantize_act(to_dev(X), to_dev(s), want_q=False)
    _, sw, Wop = sq.pack_weight(to_dev(W), to_dev(s), want_q=False)
    y = sq.linear_i8(Xop, sx, Wop, sw, to_dev(b), None, wl.EPI_BIAS)
    np.testing.assert_array_equal(y.cpu().numpy(), np.broadcast_to(b, (M, N)))
    y = sq.linear_i8(Xop, sx, Wop, sw, to_dev(b), to_dev(r), wl.EPI_BIAS_RESIDUAL)
    np.testing.assert_array_equal(y.cpu().numpy(), (r + b).astype(np.float32))


def test_empty_calls(sq):
    s = torch.ones(32, device="cuda")
    X = torch.empty(0, 32, device="cuda")
    Xq, sx, Xop = sq.quantize_act(X, s)
    assert Xq.shape == (0, 32) and sx.shape == (0,)
    W = torch.randn(8, 32, device="cuda")
    _, sw, Wop = sq.pack_weight(W, s)
    y = sq.linear_i8(Xop, sx, Wop, sw, torch.zeros(8, device="cuda"), None, wl.EPI_BIAS)
    assert y.shape == (0, 8)
    assert sq.device_status() == 0


# ------------------------------------------------ full pipeline on workloads

def _pipeline_gpu(sq, case, s, path):
    """The hot path as the benchmark runs it: pack once, then quantise the
    activations to the GEMM operand and run the fused GEMM."""
    X, W = case.X.cuda(), case.W.cuda()
    sd = to_dev(s)
    b = case.bias.cuda() if case.bias is not None else None
    r = case.residual.cuda() if case.residual is not None else None
    if path == "tc":
        _, sw, Wop, wl1 = sq.pack_weight(W, sd, want_q=False, want_l1=True)
        _, sx, Xop, xl1 = sq.quantize_act(X, sd, want_q=False, want_l1=True)
        y = sq.linear_i8(Xop, sx, Wop, sw, b, r, case.mode, x_l1=xl1, w_l1=wl1)
        return sx, y
    Wq, sw, _ = sq.pack_weight(W, sd, want_op=False)
    Xq, sx, _ = sq.quantize_act(X, sd, want_op=False)
    y = gpu_linear(sq, path, Xq, None, sx, Wq, None, sw, b, r, case.mode)
    return sx, y


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", ["bert_large_qkv_slice_m256", "bert_large_ffn_up_m256",
                                  "bert_large_ffn_down_m256"])
def test_small_workloads_full(sq, path, name):
    w = wl.WORKLOADS[name]
    case = wl.workload_case(w, 0, 0)
    X, W = case.X.numpy(), case.W.numpy()
    s = oracle_smoothing(X, W, w.alpha)
    wq, sw = oracle.quantize_rows(W, s, "weight")
    xq, sx_ref, acc, y_ref = oracle.linear_block(
        X, s, wq, sw, None if case.bias is None else case.bias.numpy(),
        None if case.residual is None else case.residual.numpy(), case.mode)
    sx, y = _pipeline_gpu(sq, case, s, path)
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    assert_close_fp32(y.cpu().numpy(), y_ref, name)


@pytest.mark.parametrize("path", ["tc"])
@pytest.mark.parametrize("name,index", [("bert_large_encoder_b32_s256", i) for i in range(4)] +
                         [("xlmr_base_b64_s512", i) for i in range(4)])
def test_large_workloads_sampled(sq, path, name, index):
    """Full-size M on the GPU, checked on a seeded sample of rows (rows are
    independent through quantisation, GEMM and epilogue)."""
    w = wl.WORKLOADS[name]
    case = wl.workload_case(w, 0, index)
    X, W = case.X.numpy(), case.W.numpy()
    # the smoothing factor from the oracle, computed on the full calibration X
    s = oracle_smoothing(X, W, w.alpha)
    wq, sw = oracle.quantize_rows(W, s, "weight")
    rng = np.random.default_rng(index)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, w.M - 1],
                                     rng.choice(w.M, 59, replace=False)]))
    b = None if case.bias is None else case.bias.numpy()
    r = None if case.residual is None else case.residual.numpy()[rows]
    _, sx_ref, _, y_ref = oracle.linear_block(X[rows], s, wq, sw, b, r, case.mode)
    sx, y = _pipeline_gpu(sq, case, s, path)
    assert_bits_equal(sx.cpu().numpy()[rows], sx_ref, "x_scale sample")
    assert_close_fp32(y[torch.from_numpy(rows).cuda()].cpu().numpy(), y_ref, f"{name}[{index}]")
    # all rows: the scales are the per-row maxima / 127 of the smoothed input
    sx_all = sx.cpu().numpy()
    v = X / s
    np.testing.assert_allclose(sx_all, np.abs(v).max(axis=1) / 127.0, rtol=2.5e-7)


def test_host_pipeline_matches_direct_calls(sq):
    """The host-buffer pipeline (sq_linear_block_host: copies overlapped with
    kernels on three streams) returns exactly what the direct device calls
    return, for Smooth-Dynamic (with and without s's division table) and
    Smooth-Static layers."""
    from smoothquant_w8a8_int8_gb300.pipeline import HostLinearPipeline, LinearLayer
    M = 300
    shapes = [(256, 384, wl.EPI_BIAS), (384, 256, wl.EPI_BIAS_GELU), (256, 256, wl.EPI_BIAS_RESIDUAL),
              (1040, 272, wl.EPI_BIAS_RESIDUAL), (272, 128, wl.EPI_NONE)]
    layers, xh, yh, ref = [], [], [], []
    for i, (K, N, mode) in enumerate(shapes):
        c = wl.make_case(M, K, N, mode, seed=700 + i)
        X, W = c.X.cuda(), c.W.cuda()
        s = sq.smooth_factor(sq.channel_absmax(X), sq.channel_absmax(W), 0.5)
        _, sw, Wop, wl1 = sq.pack_weight(W, s, want_q=False, want_l1=True)
        b = c.bias.cuda() if c.bias is not None else None
        r = c.residual.cuda() if c.residual is not None else None
        # layer 2 Smooth-Static (a quarter of its calibrated scale: some codes
        # saturate), odd layers with s's division table (sq_quantize_act_table)
        static = float(sq.static_scale(sq.act_absmax(X, s))) * 0.25 if i == 2 else None
        if static is None:
            _, sx, Xop = sq.quantize_act(X, s, want_q=False)
        else:
            _, sx, Xop = sq.quantize_act_static(X, s, static, want_q=False)
        ref.append(sq.linear_i8(Xop, sx, Wop, sw, b, r, mode, w_l1=wl1).cpu())
        layers.append(LinearLayer(s, Wop, sw, mode, b, r, wl1, static_scale=static,
                                  s_table=sq.division_table(s) if i % 2 else None))
        xh.append(c.X.pin_memory())
        yh.append(torch.empty(M, N, dtype=torch.float32).pin_memory())
    pipe = HostLinearPipeline(M, max(k for k, _, _ in shapes), max(n for _, n, _ in shapes))
    for _ in range(2):
        for y in yh:
            y.zero_()
        pipe.run(layers, xh, yh)
        torch.cuda.synchronize()
        for y, r in zip(yh, ref):
            assert torch.equal(y, r)
    # the three streams may be one: the same outputs, in order
    cur = torch.cuda.current_stream()
    table = []
    for L, x, y in zip(layers, xh, yh):
        y.zero_()
        table.append(sq.LinearLayerC(
            x.shape[1], y.shape[1], int(L.mode),
            0.0 if L.static_scale is None else float(L.static_scale), L.s.data_ptr(),
            None if L.s_table is None or L.static_scale is not None else L.s_table.data_ptr(),
            L.Wop.data_ptr(), L.w_scale.data_ptr(), L.w_l1.data_ptr(),
            None if L.bias is None else L.bias.data_ptr(),
            None if L.residual is None else L.residual.data_ptr()))
    sq.linear_block_host(table, M, xh, yh, pipe.scratch, (cur, cur, cur))
    torch.cuda.synchronize()
    for y, r in zip(yh, ref):
        assert torch.equal(y, r)
    assert sq.device_status() == sq.SQ_OK


# ------------------------------------------------------------- Smooth-Static

@pytest.mark.parametrize("M,K", [(5, 48), (300, 1024), (64, 4096), (3, 8208), (5000, 1024)])
def test_static_calibration_and_quantize_parity(sq, M, K):
    c = wl.make_case(M, K, 8, wl.EPI_BIAS, seed=K + 3 * M)
    # a separate calibration batch from the same distribution (same outlier channels)
    calib = wl.make_activation(2 * M + 7, K, seed=K + 3 * M + 1, outlier_frac=0.01,
                               outlier_scale=20.0, channel_seed=K + 3 * M).numpy()
    X = c.X.numpy()
    s = oracle_smoothing(X, c.W.numpy(), 0.5)
    amax_ref = oracle.act_absmax(calib[: M + 3], s)
    amax_ref = oracle.act_absmax(calib[M + 3:], s, amax_ref)
    amax = sq.act_absmax(to_dev(calib[: M + 3]), to_dev(s))
    sq.act_absmax(to_dev(calib[M + 3:]), to_dev(s), amax)
    assert np.float32(amax.item()).view(np.uint32) == np.float32(amax_ref).view(np.uint32)
    for scale in (oracle.static_scale(amax_ref), oracle.static_scale(amax_ref) * np.float32(0.25)):
        q_ref = oracle.quantize_static(X, s, scale)
        Xq, sx, Xop, l1 = sq.quantize_act_static(to_dev(X), to_dev(s), float(scale),
                                                 want_l1=True)
        assert_codes_equal(Xq.cpu().numpy(), q_ref, "static Xq")
        assert_codes_equal(op_as_int(Xop), q_ref, "static Xop")
        assert np.all(sx.cpu().numpy() == np.float32(scale))
        np.testing.assert_array_equal(l1.cpu().numpy(),
                                      np.abs(q_ref.astype(np.int64)).sum(axis=1))
        _, _, Xop2 = sq.quantize_act_static(to_dev(X), to_dev(s), float(scale), want_q=False)
        assert_codes_equal(op_as_int(Xop2), q_ref, "static Xop only")
    # the quarter scale saturates: the clamp is exercised
    assert np.abs(q_ref).max() == 127 and (np.abs(q_ref) == 127).sum() > M


def test_static_saturation_and_ties(sq, golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "quantize_static_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([c.strip() for c in line.split("|")])
    scale, vals, codes = rows[0]
    K = 16
    x = np.zeros((2, K), np.float32)
    v = np.array([float(t) for t in vals.split()], np.float32)
    x[0, :v.size] = v
    x[1, :v.size] = -v
    s = np.ones(K, np.float32)
    Xq, _, _ = sq.quantize_act_static(to_dev(x), to_dev(s), float(scale))
    want = np.array([int(t) for t in codes.split()], np.int8)
    np.testing.assert_array_equal(Xq.cpu().numpy()[0, :v.size], want)
    np.testing.assert_array_equal(Xq.cpu().numpy()[1, :v.size], -want)


# Smooth-Static scales on both sides of the register kernel's range
# [2^-60, 2^60] (outside it the IEEE-division kernel codes), rows in registers
# (1024, 4096) and unevenly filled (3072), codes across the whole range with
# saturation far beyond it (products at and above 2^22 take the IEEE division)
@pytest.mark.parametrize("K", [1024, 3072, 4096])
def test_static_scale_range_and_saturation(sq, K):
    rng = np.random.default_rng(K + 3)
    s = rng.uniform(0.1, 10.0, K).astype(np.float32)
    s[7] = np.float32(1e-7)                            # no reciprocal: IEEE divisions
    for scale in (np.float32(2.0 ** -61), np.float32(2.0 ** -60), np.float32(0.37),
                  np.float32(2.0 ** 60), np.float32(2.0 ** 61)):
        u = rng.uniform(-200.0, 200.0, (64, K)).astype(np.float32)
        u[3] *= np.float32(2.0 ** 30)                  # far beyond saturation
        u[5, :16] = (np.arange(16) - 7.5).astype(np.float32)  # exact half-integers
        X = (u.astype(np.float64) * s * np.float64(scale)).astype(np.float32)
        q_ref = oracle.quantize_static(X, s, scale)
        Xq, sx, Xop = sq.quantize_act_static(to_dev(X), to_dev(s), float(scale))
        assert_codes_equal(Xq.cpu().numpy(), q_ref, f"static Xq, scale {scale}")
        assert_codes_equal(op_as_int(Xop), q_ref, f"static Xop, scale {scale}")
        assert np.all(sx.cpu().numpy() == scale)


def test_static_linear_block(sq):
    """Static codes through the tcgen05 GEMM + epilogue against the oracle."""
    M, K, N = 256, 1024, 512
    c = wl.make_case(M, K, N, wl.EPI_BIAS_GELU, seed=17)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle_smoothing(X, W, 0.5)
    scale = oracle.static_scale(oracle.act_absmax(X, s))
    wq, sw = oracle.quantize_rows(W, s, "weight")
    xq = oracle.quantize_static(X, s, scale)
    ref = oracle.epilogue(oracle.gemm_i32(xq, wq), np.full(M, scale, np.float32), sw,
                          c.bias.numpy(), mode=wl.EPI_BIAS_GELU)
    _, sw_d, Wop = sq.pack_weight(to_dev(W), to_dev(s), want_q=False)
    _, sx_d, Xop = sq.quantize_act_static(to_dev(X), to_dev(s), float(scale), want_q=False)
    y = sq.linear_i8(Xop, sx_d, Wop, sw_d, to_dev(c.bias.numpy()), None, wl.EPI_BIAS_GELU)
    assert_close_fp32(y.cpu().numpy(), ref, "static linear block")


# ------------------------------------------------ producer-fused requantisation

@pytest.mark.parametrize("mode", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU,
                                  wl.EPI_BIAS_RESIDUAL])
@pytest.mark.parametrize("M,N,K", [(77, 136, 1024), (256, 1024, 1024), (300, 4096, 1024),
                                   (2560, 2304, 512), (130, 200, 2064),
                                   (2560, 2304, 2064)])  # pair kernel: halves + 3 exact passes
def test_requant_epilogue_matches_static_quantiser(sq, mode, M, N, K):
    """The requantising epilogue's codes equal the oracle's Smooth-Static
    quantiser applied to the fp32 output the plain epilogue stores (the same
    y, bit for bit), for a calibrated scale and for a quarter of it
    (saturating codes); x_scale_next is the scale everywhere."""
    c, xq, sx, wq, sw, d = _quantised_case(sq, M, K, N, wl.EPI_BIAS_RESIDUAL, seed=3 * M + N + mode)
    b = to_dev(c.bias.numpy())
    r = to_dev(c.residual.numpy()) if mode == wl.EPI_BIAS_RESIDUAL else None
    y = sq.linear_i8(d["Xop"], d["sx"], d["Wop"], d["sw"], b, r, mode).cpu().numpy()
    rng = np.random.default_rng(M + N)
    s_next = rng.uniform(0.2, 6.0, N).astype(np.float32)
    calib = oracle.static_scale(oracle.act_absmax(y, s_next))
    for scale in (calib, calib * np.float32(0.25)):
        Yq, Yop, xs = sq.linear_i8_requant(d["Xop"], d["sx"], d["Wop"], d["sw"], b, r, mode,
                                           to_dev(s_next), float(scale), want_q=True)
        ref = oracle.quantize_static(y, s_next, scale)
        assert_codes_equal(Yq.cpu().numpy(), ref, "Yq")
        assert_codes_equal(op_as_int(Yop), ref, "Yop")
        assert np.all(xs.cpu().numpy() == np.float32(scale))
    assert np.abs(ref).max() == 127  # the quarter scale saturates
    # smoothing factors outside [2^-20, 2^20] and a scale below 2^-70 take the
    # exact path (IEEE divisions)
    s_odd = s_next.copy()
    s_odd[min(3, N - 1)] = np.float32(1e-7)
    s_odd[min(5, N - 1)] = np.float32(3e7)
    for s_case, scale in ((s_odd, calib), (s_next, np.float32(2.0 ** -71))):
        _, Yop, _ = sq.linear_i8_requant(d["Xop"], d["sx"], d["Wop"], d["sw"], b, r, mode,
                                         to_dev(s_case), float(scale), want_x_scale=False)
        assert_codes_equal(op_as_int(Yop), oracle.quantize_static(y, s_case, scale), "Yop")


def test_requant_feeds_next_linear(sq):
    """FFN-up with the requantising epilogue feeding FFN-down: the down
    projection's output equals the unfused chain's (the same codes go in)."""
    M, K1, N1, N2 = 512, 1024, 4096, 1024
    c1 = wl.make_case(M, K1, N1, wl.EPI_BIAS_GELU, seed=11)
    W2 = wl.make_weight(N2, N1, 12)
    b2 = wl.make_bias(N2, 12)
    r2 = wl.make_residual(M, N2, 12)
    Xd, Wd = c1.X.cuda(), c1.W.cuda()
    s1 = sq.smooth_factor(sq.channel_absmax(Xd), sq.channel_absmax(Wd), 0.5)
    _, sw1, Wop1 = sq.pack_weight(Wd, s1, want_q=False)
    _, sx1, Xop1 = sq.quantize_act(Xd, s1, want_q=False)
    y1 = sq.linear_i8(Xop1, sx1, Wop1, sw1, c1.bias.cuda(), None, wl.EPI_BIAS_GELU)
    s2 = sq.smooth_factor(sq.channel_absmax(y1), sq.channel_absmax(W2.cuda()), 0.5)
    _, sw2, Wop2 = sq.pack_weight(W2.cuda(), s2, want_q=False)
    scale = float(oracle.static_scale(oracle.act_absmax(y1.cpu().numpy(), s2.cpu().numpy())))
    # unfused: fp32 y1, then the static quantiser
    _, sx2, Xop2 = sq.quantize_act_static(y1, s2, scale, want_q=False)
    y2 = sq.linear_i8(Xop2, sx2, Wop2, sw2, b2.cuda(), r2.cuda(), wl.EPI_BIAS_RESIDUAL)
    # fused: FFN-up emits FFN-down's operand
    _, Xop2f, sx2f = sq.linear_i8_requant(Xop1, sx1, Wop1, sw1, c1.bias.cuda(), None,
                                          wl.EPI_BIAS_GELU, s2, scale)
    y2f = sq.linear_i8(Xop2f, sx2f, Wop2, sw2, b2.cuda(), r2.cuda(), wl.EPI_BIAS_RESIDUAL)
    assert torch.equal(Xop2f, Xop2) and torch.equal(sx2f, sx2)
    assert torch.equal(y2f, y2)


# ------------------------------------------------ LayerNorm + quantiser

@pytest.mark.parametrize("M,K", [(7, 48), (300, 1024), (64, 4096), (5, 768), (130, 8192)])
def test_layernorm_quant_parity(sq, M, K):
    """The fused LayerNorm's fp32 output matches the oracle's LayerNorm within
    the fp32 tolerance, and its codes, scales and L1 norms equal the oracle's
    quantisers applied to that output bit for bit (dynamic and static)."""
    rng = np.random.default_rng(M * 7 + K)
    H = (rng.standard_normal((M, K)) * 3.0 + 0.5).astype(np.float32)
    H[:, rng.integers(0, K, max(1, K // 100))] *= np.float32(20.0)  # outlier channels
    gamma = (1.0 + 0.05 * rng.standard_normal(K)).astype(np.float32)
    beta = (0.05 * rng.standard_normal(K)).astype(np.float32)
    s = rng.uniform(0.3, 4.0, K).astype(np.float32)
    eps = 1e-12
    y_ref = oracle.layernorm(H, gamma, beta, eps)
    Xq, sx, Xop, Y, l1 = sq.layernorm_quant(to_dev(H), to_dev(gamma), to_dev(beta), eps,
                                            to_dev(s), want_y=True, want_l1=True)
    y = Y.cpu().numpy()
    assert_close_fp32(y, y_ref, "LayerNorm output")
    q_ref, sx_ref = oracle.quantize_rows(y, s, "act")
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_codes_equal(op_as_int(Xop), q_ref, "Xop")
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    np.testing.assert_array_equal(l1.cpu().numpy(), np.abs(q_ref.astype(np.int64)).sum(axis=1))
    # without the fp32 output: the same codes
    _, sx2, Xop2, _, _ = sq.layernorm_quant(to_dev(H), to_dev(gamma), to_dev(beta), eps,
                                            to_dev(s), want_q=False)
    assert_codes_equal(op_as_int(Xop2), q_ref, "Xop (no Y)")
    # static scale (a quarter of the calibrated one saturates)
    scale = oracle.static_scale(oracle.act_absmax(y, s)) * np.float32(0.25)
    Xq3, sx3, _, _, _ = sq.layernorm_quant(to_dev(H), to_dev(gamma), to_dev(beta), eps,
                                           to_dev(s), static_scale=float(scale), want_op=False)
    assert_codes_equal(Xq3.cpu().numpy(), oracle.quantize_static(y, s, scale), "static Xq")
    assert np.all(sx3.cpu().numpy() == np.float32(scale))


@pytest.mark.parametrize("K", [1024, 3072])
def test_layernorm_quant_extreme_factors_and_scales(sq, K):
    """Smoothing factors without a reciprocal in the division tables (|s|
    outside [2^-20, 2^20]: IEEE divisions for those columns), beta alone in a
    row of zeros (constant rows), and static scales on both sides of the fast
    path's range [2^-60, 2^60]: codes and scales bit for bit against the
    oracle's quantisers applied to the LayerNorm's own output."""
    rng = np.random.default_rng(K + 17)
    M = 70
    H = (rng.standard_normal((M, K)) * 2.0).astype(np.float32)
    H[4] = 0.0
    gamma = (1.0 + 0.05 * rng.standard_normal(K)).astype(np.float32)
    beta = (0.05 * rng.standard_normal(K)).astype(np.float32)
    s = rng.uniform(0.3, 4.0, K).astype(np.float32)
    s[[2, 9]] = np.float32(1e-7), np.float32(3e7)
    eps = 1e-12
    Xq, sx, Xop, Y, l1 = sq.layernorm_quant(to_dev(H), to_dev(gamma), to_dev(beta), eps,
                                            to_dev(s), want_y=True, want_l1=True)
    y = Y.cpu().numpy()
    q_ref, sx_ref = oracle.quantize_rows(y, s, "act")
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_codes_equal(op_as_int(Xop), q_ref, "Xop")
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    np.testing.assert_array_equal(l1.cpu().numpy(), np.abs(q_ref.astype(np.int64)).sum(axis=1))
    s2 = rng.uniform(0.3, 4.0, K).astype(np.float32)
    for scale in (np.float32(2.0 ** -61), np.float32(2.0 ** -60), np.float32(0.01),
                  np.float32(2.0 ** 60), np.float32(2.0 ** 61)):
        H2 = (rng.standard_normal((M, K)) * 2.0).astype(np.float32)
        g2 = (gamma * np.float32(scale) * 40.0).astype(np.float32)  # codes across the range
        Xq2, sx2, _, Y2, _ = sq.layernorm_quant(to_dev(H2), to_dev(g2), to_dev(beta), eps,
                                                to_dev(s2), static_scale=float(scale),
                                                want_y=True, want_op=False)
        q2 = oracle.quantize_static(Y2.cpu().numpy(), s2, scale)
        assert_codes_equal(Xq2.cpu().numpy(), q2, f"static Xq, scale {scale}")
        assert np.all(sx2.cpu().numpy() == scale)


def test_layernorm_quant_constant_rows(sq):
    """Rows with no spread normalise to beta exactly (zero deviation)."""
    K = 256
    H = np.full((3, K), 2.5, np.float32)
    H[1] = -7.0
    gamma = np.ones(K, np.float32)
    beta = np.linspace(-1, 1, K).astype(np.float32)
    s = np.ones(K, np.float32)
    _, _, _, Y, _ = sq.layernorm_quant(to_dev(H), to_dev(gamma), to_dev(beta), 1e-5, to_dev(s),
                                       want_y=True)
    np.testing.assert_array_equal(Y.cpu().numpy(), np.tile(beta, (3, 1)))
