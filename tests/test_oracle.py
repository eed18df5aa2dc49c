"""Pins for the CPU oracle: each check is fixed by something other than the
oracle itself (hand-worked values, textbook values, closed forms, exact
invariants, brute force in a different order), chosen so that a dropped term,
a wrong sign or index, or a transposed operand fails at least one of them."""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from smoothquant_w8a8_int8_gb300 import workloads


def f32_bits(x):
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def parse_golden(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


# --------------------------------------------------------------- quantiser

def test_quantize_hand_example(golden_dir):
    for name, s, vals, bits, codes in parse_golden(
            os.path.join(golden_dir, "quantize_rne_example.txt")):
        row = np.array([[float(v) for v in vals.split()]], np.float32)
        K = row.shape[1]
        svec = np.full(K, float(s), np.float32)
        want_q = np.array([int(c) for c in codes.split()], np.int8)
        for direction in ("act", "weight"):
            # the weight side multiplies by s: feed it W = row * s^-2 so that
            # W * s equals row / s, the activation side's smoothed row
            A = row if direction == "act" else row / (svec * svec)
            q, sc = oracle.quantize_rows(A, svec, direction)
            assert f32_bits(sc[0]) == int(bits, 16), (name, direction, sc[0])
            np.testing.assert_array_equal(q[0], want_q, err_msg=f"{name} {direction}")


def test_quantize_error_bound_and_full_range():
    c = workloads.make_case(37, 96, 8, workloads.EPI_BIAS, seed=5)
    X = c.X.numpy()
    s = (np.abs(np.random.default_rng(1).standard_normal(96)) + 0.25).astype(np.float32)
    q, sx = oracle.quantize_rows(X, s, "act")
    v = oracle.smooth(X, s, "act").astype(np.float64)
    err = np.abs(v - q.astype(np.float64) * sx[:, None].astype(np.float64))
    # half a step plus the fp32 rounding of v / scale
    assert np.all(err <= sx[:, None] * (0.5 + 1e-5))
    assert np.all(np.abs(q).max(axis=1) == 127)
    # the scale is amax / 127 to within one fp32 rounding
    amax = np.abs(v).max(axis=1)
    np.testing.assert_allclose(sx, amax / 127.0, rtol=1.2e-7)


def test_quantize_smoothing_direction_power_of_two():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((9, 32)).astype(np.float32)
    s = (2.0 ** rng.integers(-3, 4, 32)).astype(np.float32)
    q1, s1 = oracle.quantize_rows(X, s, "act")
    q2, s2 = oracle.quantize_rows(X / s, np.ones(32, np.float32), "act")   # exact
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1.view(np.uint32), s2.view(np.uint32))
    W = rng.standard_normal((5, 32)).astype(np.float32)
    q3, s3 = oracle.quantize_rows(W, s, "weight")
    q4, s4 = oracle.quantize_rows(W * s, np.ones(32, np.float32), "weight")
    np.testing.assert_array_equal(q3, q4)
    np.testing.assert_array_equal(s3.view(np.uint32), s4.view(np.uint32))


def test_quantize_zero_and_one_hot_rows():
    X = np.zeros((3, 16), np.float32)
    X[1, 5] = -3.0
    X[2, 0] = 1e-30
    q, sx = oracle.quantize_rows(X, np.ones(16, np.float32), "act")
    assert sx[0] == 1.0 and not q[0].any()
    assert q[1, 5] == -127 and np.count_nonzero(q[1]) == 1
    assert f32_bits(sx[1]) == f32_bits(np.float32(3.0) / np.float32(127.0))
    assert q[2, 0] == 127 and np.count_nonzero(q[2]) == 1


# --------------------------------------------------------------- smoothing

def test_smooth_factor_closed_forms():
    ax = np.array([2.0 ** 10, 4.0, 9.0, 0.0, 5.0], np.float32)
    aw = np.array([2.0 ** 5, 16.0, 1.0, 3.0, 0.0], np.float32)
    s = oracle.smooth_factor(ax, aw, 0.5)
    assert s[0] == np.float32(2.0 ** 5 / 2.0 ** 2.5)
    assert s[1] == 0.5 and s[2] == 3.0
    assert s[3] == 1.0 and s[4] == 1.0      # zero rule
    s6 = oracle.smooth_factor(ax[:1], aw[:1], 0.6)
    assert s6[0] == 16.0                    # 2^6 / 2^2
    np.testing.assert_array_equal(oracle.smooth_factor(ax[:3], aw[:3], 1.0), ax[:3])
    np.testing.assert_allclose(oracle.smooth_factor(ax[:3], aw[:3], 0.0), 1.0 / aw[:3],
                               rtol=1e-7)


def test_channel_absmax_brute_force():
    rng = np.random.default_rng(3)
    A = rng.standard_normal((7, 5)).astype(np.float32)
    want = [max(abs(float(A[i, j])) for i in range(7)) for j in range(5)]
    np.testing.assert_array_equal(oracle.channel_absmax(A), np.array(want, np.float32))


def test_smoothing_invariant_exact_power_of_two():
    """X W^T is unchanged by diag(s)^-1 on X and diag(s) on W."""
    rng = np.random.default_rng(4)
    X = rng.standard_normal((6, 40)).astype(np.float32)
    W = rng.standard_normal((4, 40)).astype(np.float32)
    s = (2.0 ** rng.integers(-4, 5, 40)).astype(np.float32)
    Xs, Ws = oracle.smooth(X, s, "act"), oracle.smooth(W, s, "weight")

    def dot(A, B):  # same summation order for both calls
        return (A.astype(np.float64)[:, None, :] * B.astype(np.float64)[None, :, :]).sum(-1)

    np.testing.assert_array_equal(dot(Xs, Ws), dot(X, W))
    assert not np.array_equal(Xs, X)


def test_smoothing_invariant_general_s():
    c = workloads.make_case(64, 128, 32, workloads.EPI_BIAS, seed=6)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle.smooth_factor(oracle.channel_absmax(X), oracle.channel_absmax(W), 0.5)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    got = oracle.smooth(X, s, "act").astype(np.float64) @ oracle.smooth(W, s, "weight").astype(np.float64).T
    assert np.max(np.abs(got - ref)) <= 1e-6 * np.max(np.abs(ref))
    # smoothing equalises the channel maxima: max|X_j/s_j| == max|W_j*s_j|
    ax = oracle.channel_absmax(oracle.smooth(X, s, "act"))
    aw = oracle.channel_absmax(oracle.smooth(W, s, "weight"))
    np.testing.assert_allclose(ax, aw, rtol=1e-6)


# --------------------------------------------------------------- integer GEMM

def test_gemm_brute_force_outer_product_order():
    vals = np.array([-127, -1, 0, 1, 127], np.int8)
    rng = np.random.default_rng(7)
    for M, N, K in [(1, 1, 1), (2, 3, 4), (5, 2, 6), (6, 6, 3), (3, 5, 6)]:
        xq = vals[rng.integers(0, 5, (M, K))]
        wq = vals[rng.integers(0, 5, (N, K))]
        acc = [[0] * N for _ in range(M)]
        for k in range(K):            # rank-1 updates, k outermost
            for m in range(M):
                for n in range(N):
                    acc[m][n] += int(xq[m, k]) * int(wq[n, k])
        np.testing.assert_array_equal(oracle.gemm_i32(xq, wq), np.array(acc, np.int32))


def test_gemm_closed_forms():
    for K in (1024, 4096):
        ones = np.full((2, K), 127, np.int8)
        assert np.all(oracle.gemm_i32(ones, ones) == K * 127 * 127)
        neg = ones.copy()
        neg[:, 1::2] = -127
        assert np.all(oracle.gemm_i32(ones, neg) == 0)
    assert oracle.gemm_i32(np.full((1, 1024), 127, np.int8),
                           np.full((1, 1024), 127, np.int8))[0, 0] == 16516096
    x = np.zeros((3, 8), np.int8)
    x[0, 1] = 1
    x[1, 5] = -1
    x[2, 7] = 2
    w = np.arange(-20, 20, dtype=np.int8).reshape(5, 8)
    acc = oracle.gemm_i32(x, w)
    np.testing.assert_array_equal(acc[0], w[:, 1])
    np.testing.assert_array_equal(acc[1], -w[:, 5].astype(np.int32))
    np.testing.assert_array_equal(acc[2], 2 * w[:, 7].astype(np.int32))


def test_gemm_overflow_detected():
    K = 133145  # 133145 * 127^2 > 2^31 - 1 > 133144 * 127^2
    a = np.full((1, K), 127, np.int8)
    with pytest.raises(OverflowError):
        oracle.gemm_i32(a, a)
    a[0, 0] = 0
    assert oracle.gemm_i32(a, a)[0, 0] == (K - 1) * 16129


# --------------------------------------------------------------- epilogue

def test_epilogue_gelu_textbook(golden_dir):
    rows = parse_golden(os.path.join(golden_dir, "gelu_normal_cdf.txt"))
    ts = [float(r[0]) for r in rows]
    phis = [float(r[1]) for r in rows]
    # d = acc * sx * sw = t exactly with acc = t * 4, sx = 0.5, sw = 0.5
    acc = np.array([[int(t * 4) for t in ts]], np.int32)
    y = oracle.epilogue(acc, [0.5], np.full(len(ts), 0.5), bias=np.zeros(len(ts)),
                        mode=oracle.EPI_BIAS_GELU)
    for t, phi, got in zip(ts, phis, y[0]):
        assert abs(float(got) - t * phi) <= 1e-7 * max(1.0, abs(t * phi)) + 1e-9, (t, got)


def test_epilogue_zero_input_and_modes():
    M, N = 3, 4
    acc = np.zeros((M, N), np.int32)
    sx = np.array([0.5, 2.0, 3.0], np.float32)
    sw = np.array([1.0, 0.25, 4.0, 8.0], np.float32)
    b = np.array([0.1, -0.2, 0.3, 0.0], np.float32)
    r = np.arange(12, dtype=np.float32).reshape(M, N)
    np.testing.assert_array_equal(oracle.epilogue(acc, sx, sw, b, mode=oracle.EPI_BIAS),
                                  np.broadcast_to(b, (M, N)))
    np.testing.assert_array_equal(oracle.epilogue(acc, sx, sw, b, r, oracle.EPI_BIAS_RESIDUAL),
                                  (r.astype(np.float64) + b).astype(np.float32))
    assert not oracle.epilogue(acc, sx, sw, b, mode=oracle.EPI_BIAS_GELU)[:, 3].any()
    # per-token (rows) x per-channel (columns), asymmetric so a transpose fails
    acc = np.arange(1, 13, dtype=np.int32).reshape(M, N)
    y = oracle.epilogue(acc, sx, sw, mode=oracle.EPI_NONE)
    for m in range(M):
        for n in range(N):
            assert y[m, n] == np.float32(acc[m, n] * float(sx[m]) * float(sw[n]))


def test_epilogue_single_rounding():
    acc = np.array([[3, -7]], np.int32)
    sx = np.array([0.1], np.float32)
    sw = np.array([0.3, 0.7], np.float32)
    b = np.array([0.05, 1e-3], np.float32)
    y = oracle.epilogue(acc, sx, sw, b, mode=oracle.EPI_BIAS)
    for n in range(2):
        exact = (Fraction(int(acc[0, n])) * Fraction(float(sx[0])) * Fraction(float(sw[n]))
                 + Fraction(float(b[n])))
        assert y[0, n] == np.float32(float(exact))


def test_linear_block_matches_steps():
    c = workloads.make_case(19, 64, 24, workloads.EPI_BIAS_RESIDUAL, seed=8)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle.smooth_factor(oracle.channel_absmax(X), oracle.channel_absmax(W), 0.5)
    wq, sw = oracle.quantize_rows(W, s, "weight")
    xq, sx, acc, y = oracle.linear_block(X, s, wq, sw, c.bias.numpy(), c.residual.numpy(),
                                         oracle.EPI_BIAS_RESIDUAL)
    xq2, sx2 = oracle.quantize_rows(X, s, "act")
    np.testing.assert_array_equal(xq, xq2)
    np.testing.assert_array_equal(acc, oracle.gemm_i32(xq, wq))
    # the quantised block approximates the fp64 linear layer
    ref = X.astype(np.float64) @ W.astype(np.float64).T + c.bias.numpy() + c.residual.numpy()
    assert np.max(np.abs(y - ref)) < 0.05 * np.max(np.abs(ref))


# --------------------------------------------------------------- Smooth-Static

def test_static_hand_example(golden_dir):
    for scale, vals, codes in parse_golden(os.path.join(golden_dir, "quantize_static_example.txt")):
        X = np.array([[float(v) for v in vals.split()]], np.float32)
        q = oracle.quantize_static(X, np.ones(X.shape[1], np.float32), np.float32(float(scale)))
        np.testing.assert_array_equal(q[0], np.array([int(c) for c in codes.split()], np.int8))


def test_static_calibration_on_one_row_equals_dynamic():
    """Calibrating the static scale on a single row gives that row's dynamic
    scale and therefore the dynamic codes."""
    c = workloads.make_case(6, 64, 8, workloads.EPI_BIAS, seed=21)
    X = c.X.numpy()
    s = (np.abs(np.random.default_rng(3).standard_normal(64)) + 0.5).astype(np.float32)
    qd, sd = oracle.quantize_rows(X, s, "act")
    for i in range(X.shape[0]):
        amax = oracle.act_absmax(X[i:i + 1], s)
        sc = oracle.static_scale(amax)
        assert sc.view(np.uint32) == sd[i].view(np.uint32)
        np.testing.assert_array_equal(oracle.quantize_static(X[i:i + 1], s, sc)[0], qd[i])


def test_static_absmax_running_and_brute_force():
    rng = np.random.default_rng(4)
    A = rng.standard_normal((5, 16)).astype(np.float32)
    B = (rng.standard_normal((3, 16)) * 4).astype(np.float32)
    s = (rng.uniform(0.5, 2.0, 16)).astype(np.float32)
    want = max(abs(float(np.float32(A[i, j]) / np.float32(s[j]))) for i in range(5) for j in range(16))
    a = oracle.act_absmax(A, s)
    assert a == np.float32(want)
    want2 = max(want, max(abs(float(np.float32(B[i, j]) / np.float32(s[j])))
                          for i in range(3) for j in range(16)))
    assert oracle.act_absmax(B, s, a) == np.float32(want2)
    assert oracle.static_scale(0.0) == 1.0


# ---------------------------------------------------------------- LayerNorm

def test_layernorm_closed_forms():
    K = 64
    g = np.ones(K, np.float32)
    b = np.linspace(-1, 1, K).astype(np.float32)
    # a constant row has zero deviation from its mean: the output is beta
    y = oracle.layernorm(np.full((1, K), 3.25, np.float32), g, b, eps=1e-5)
    np.testing.assert_array_equal(y[0], b)
    # +-a alternating: mean 0, variance a^2, so with eps = 0 the output is +-1
    a = np.float32(2.5)
    h = np.tile(np.array([a, -a], np.float32), K // 2)[None]
    y = oracle.layernorm(h, g, np.zeros(K, np.float32), eps=0.0)
    np.testing.assert_array_equal(y[0], np.tile(np.array([1, -1], np.float32), K // 2))
    # gamma and beta act per channel
    y2 = oracle.layernorm(h, np.full(K, 2.0, np.float32), np.full(K, 0.5, np.float32), eps=0.0)
    np.testing.assert_array_equal(y2[0], 2.0 * y[0] + 0.5)


def test_layernorm_invariances():
    rng = np.random.default_rng(3)
    K = 256
    h = rng.standard_normal((8, K)).astype(np.float32)
    g, b = np.ones(K, np.float32), np.zeros(K, np.float32)
    y = oracle.layernorm(h, g, b, eps=0.0)
    # zero mean and unit (biased) variance per row
    np.testing.assert_allclose(y.astype(np.float64).mean(axis=1), 0.0, atol=1e-6)
    np.testing.assert_allclose(y.astype(np.float64).var(axis=1), 1.0, rtol=1e-6)
    # invariant under scaling by a power of two and under a shift
    y4 = oracle.layernorm(h * np.float32(4.0), g, b, eps=0.0)
    np.testing.assert_array_equal(y4, y)
    ys = oracle.layernorm(h + np.float32(0.75), g, b, eps=0.0)
    np.testing.assert_allclose(ys, y, atol=2e-6)


# ------------------------------------------------------------- attention

def _qkv(rng, B, S, H, D, scale=1.0):
    return (rng.standard_normal((B * S, 3 * H * D)) * scale).astype(np.float32)


def _blocks(QKV, B, S, H, D):
    """(Q, K, V) as [B, H, S, D] views of the fused projection's output."""
    x = QKV.reshape(B, S, 3, H, D).astype(np.float64)
    return x[:, :, 0].transpose(0, 2, 1, 3), x[:, :, 1].transpose(0, 2, 1, 3), \
        x[:, :, 2].transpose(0, 2, 1, 3)


def test_attention_zero_queries_average_the_values():
    """All scores equal: the softmax is uniform and every output row is the
    mean of the sequence's value rows."""
    B, S, H, D = 2, 5, 3, 4
    QKV = _qkv(np.random.default_rng(1), B, S, H, D)
    QKV[:, : H * D] = 0.0
    O = oracle.attention(QKV, B, S, H, D).reshape(B, S, H, D)
    _, _, V = _blocks(QKV, B, S, H, D)
    mean = V.mean(axis=2)                                  # [B, H, D]
    for i in range(S):
        np.testing.assert_allclose(O[:, i], mean.astype(np.float32), rtol=0, atol=2e-7)


def test_attention_two_keys_logistic_weights():
    """Two tokens: p_i1 = 1 / (1 + exp(-(z_i1 - z_i2))), the logistic function
    of the scaled score difference (a wrong scale, sign or normalisation fails)."""
    B, S, H, D = 1, 2, 1, 4
    QKV = _qkv(np.random.default_rng(2), B, S, H, D)
    Q, K, V = _blocks(QKV, B, S, H, D)
    O = oracle.attention(QKV, B, S, H, D)
    scale = 1.0 / np.sqrt(D)                               # 0.5
    for i in range(S):
        dz = scale * (Q[0, 0, i] @ K[0, 0, 0] - Q[0, 0, i] @ K[0, 0, 1])
        p1 = 1.0 / (1.0 + np.exp(-dz))
        ref = p1 * V[0, 0, 0] + (1.0 - p1) * V[0, 0, 1]
        np.testing.assert_allclose(O[i], ref, rtol=2e-7, atol=1e-7)


def test_attention_near_one_hot():
    """Orthogonal keys and queries aligned with one key each, at a large
    scale: each query picks its key's value row (to within e^-40)."""
    B, S, H, D = 1, 4, 1, 4
    QKV = np.zeros((B * S, 3 * H * D), np.float32)
    pick = [2, 0, 3, 1]
    for j in range(S):
        QKV[j, H * D + j] = 1.0                            # key j = e_j
    for i in range(S):
        QKV[i, pick[i]] = 80.0                             # query i = 80 e_pick(i)
    QKV[:, 2 * H * D:] = np.random.default_rng(3).standard_normal((S, D)).astype(np.float32)
    O = oracle.attention(QKV, B, S, H, D)                  # scores 40 apart
    for i in range(S):
        np.testing.assert_allclose(O[i], QKV[pick[i], 2 * H * D:], rtol=0, atol=1e-12)


def test_attention_token_permutation_equivariance():
    B, S, H, D = 1, 7, 2, 8
    rng = np.random.default_rng(4)
    QKV = _qkv(rng, B, S, H, D)
    perm = rng.permutation(S)
    O = oracle.attention(QKV, B, S, H, D)
    Op = oracle.attention(QKV[perm], B, S, H, D)
    np.testing.assert_allclose(Op, O[perm], rtol=1e-6, atol=1e-7)


def test_attention_heads_and_sequences_are_independent():
    B, S, H, D = 2, 6, 3, 4
    rng = np.random.default_rng(5)
    QKV = _qkv(rng, B, S, H, D)
    O = oracle.attention(QKV, B, S, H, D).reshape(B, S, H, D)
    other = QKV.reshape(B, S, 3, H, D).copy()
    other[:, :, :, 1] += 1.0                               # every input of head 1
    other[1] *= 3.0                                        # every input of sequence 1
    O2 = oracle.attention(other.reshape(B * S, -1), B, S, H, D).reshape(B, S, H, D)
    assert np.array_equal(O2[0, :, 0], O[0, :, 0]) and np.array_equal(O2[0, :, 2], O[0, :, 2])
    assert not np.array_equal(O2[0, :, 1], O[0, :, 1])
    assert not np.array_equal(O2[1], O[1])
