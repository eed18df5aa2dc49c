"""Producer-fused Smooth-Dynamic quantisation (the FFN up-projection's
epilogue hands the FFN down-projection its per-token statistic).

sq_linear_i8_rowmax must write exactly the Y that sq_linear_i8 writes and, per
row, max_n |fl(Y / s_next)| bit for bit (checked against the oracle's
smoothing of that Y); sq_quantize_act_rowmax, given those maxima, must write
the codes, scale bits and row L1 norms of the oracle's dynamic quantiser on the
same Y.  "Efficient INT8 Inference of Small NLP Models on Server CPUs with
PyTorch Native Stack", Table 10 (Smooth-Dynamic) and the INT8 subgraph fusion
of the Figure 1 caption.
"""
import numpy as np
import pytest
import torch

import oracle
from paritylib import assert_bits_equal, assert_codes_equal, op_as_int, oracle_smoothing, to_dev
from smoothquant_w8a8_int8_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


def _case(M, K, N, mode, seed):
    c = wl.make_case(M, K, N, wl.EPI_BIAS_RESIDUAL, seed=seed)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle_smoothing(X, W, 0.5)
    wq, sw = oracle.quantize_rows(W, s, "weight")
    xq, sx = oracle.quantize_rows(X, s, "act")
    d = dict(Xop=to_dev(xq.astype(np.float32), torch.bfloat16), sx=to_dev(sx),
             Wop=to_dev(wq.astype(np.float32), torch.bfloat16), sw=to_dev(sw),
             b=to_dev(c.bias.numpy()),
             r=to_dev(c.residual.numpy()) if mode == wl.EPI_BIAS_RESIDUAL else None)
    return d


def _row_max_ref(Y, s):
    """max_n |fl(Y[m, n] / s[n])| per row, from the oracle's smoothing."""
    return np.abs(oracle.smooth(Y, s, "act")).max(axis=1).astype(np.float32)


# (M, N, K): pair kernel (M >= 256), the one-CTA kernel (M < 256), partial
# last slices (N % 32 != 0; the maxima alone where N % 16 != 0), the FFN
# up-projection's shape at M = 1024
SHAPES = [(512, 1024, 1024), (77, 136, 1024), (300, 200, 512), (200, 400, 1024),
          (1024, 4096, 1024)]


@pytest.mark.parametrize("mode", [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU,
                                  wl.EPI_BIAS_RESIDUAL])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_rowmax_epilogue_and_given_max_quantiser(sq, M, N, K, mode):
    d = _case(M, K, N, mode, seed=5 * M + N + mode)
    y_plain = sq.linear_i8(d["Xop"], d["sx"], d["Wop"], d["sw"], d["b"], d["r"], mode)
    rng = np.random.default_rng(M + N + K)
    s_next = rng.uniform(0.2, 6.0, N).astype(np.float32)
    table = sq.division_table(to_dev(s_next))
    y_rm, amax = sq.linear_i8_rowmax(d["Xop"], d["sx"], d["Wop"], d["sw"], d["b"], d["r"], mode,
                                     table)
    assert torch.equal(y_rm, y_plain)
    Y = y_plain.cpu().numpy()
    assert_bits_equal(amax.cpu().numpy(), _row_max_ref(Y, s_next), "row maxima")
    if N % 16:
        return  # not a valid K for the next linear: the maxima alone
    # the given-maximum quantiser on the same Y equals the oracle's dynamic quantiser
    q_ref, sx_ref = oracle.quantize_rows(Y, s_next, "act")
    Xq, sx, Xop, l1 = sq.quantize_act_rowmax(y_plain, to_dev(s_next), amax, want_l1=True)
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_codes_equal(op_as_int(Xop), q_ref, "Xop")
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    np.testing.assert_array_equal(l1.cpu().numpy(), np.abs(q_ref.astype(np.int64)).sum(axis=1))


def test_rowmax_accumulates_and_extreme_columns(sq):
    """Smoothing factors outside [2^-20, 2^20] (IEEE divisions for those
    columns), rows of zeros, and a running maximum carried in from before."""
    M, N, K = 384, 520, 1024
    d = _case(M, K, N, wl.EPI_BIAS, seed=91)
    d["Xop"][7].zero_()                                   # row 7: y = bias only
    rng = np.random.default_rng(3)
    s_next = rng.uniform(0.5, 2.0, N).astype(np.float32)
    s_next[[3, 100, 515]] = np.float32(1e-7), np.float32(3e7), np.float32(2.0 ** -21)
    y_plain = sq.linear_i8(d["Xop"], d["sx"], d["Wop"], d["sw"], d["b"], None, wl.EPI_BIAS)
    Y = y_plain.cpu().numpy()
    ref = _row_max_ref(Y, s_next)
    start = np.zeros(M, np.float32)
    start[::5] = ref[::5] * np.float32(2.0)               # larger maxima already recorded
    amax = to_dev(start)
    y_rm, _ = sq.linear_i8_rowmax(d["Xop"], d["sx"], d["Wop"], d["sw"], d["b"], None,
                                  wl.EPI_BIAS, sq.division_table(to_dev(s_next)), row_amax=amax)
    assert torch.equal(y_rm, y_plain)
    assert_bits_equal(amax.cpu().numpy(), np.maximum(ref, start), "running maxima")


def test_given_max_quantiser_zero_rows_and_too_small_maxima(sq):
    K = 1024
    X = np.random.default_rng(4).standard_normal((6, K)).astype(np.float32)
    X[2] = 0.0
    s = np.ones(K, np.float32)
    ref_amax = np.abs(X).max(axis=1).astype(np.float32)
    q_ref, sx_ref = oracle.quantize_rows(X, s, "act")
    Xq, sx, _ = sq.quantize_act_rowmax(to_dev(X), to_dev(s), to_dev(ref_amax))
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    # a maximum below the true one: the codes saturate, they never wrap
    Xq2, _, Xop2 = sq.quantize_act_rowmax(to_dev(X), to_dev(s), to_dev(ref_amax * 0.25))
    q2 = Xq2.cpu().numpy()
    assert np.abs(q2.astype(np.int32)).max() == 127
    assert np.all(np.sign(q2[X != 0]) == np.sign(X[X != 0]) * (q2[X != 0] != 0))
    assert_codes_equal(op_as_int(Xop2), q2, "Xop")


def test_division_table(sq):
    s = np.array([1.0, -3.0, 0.1, 2.0 ** -20, 2.0 ** 20, 2.0 ** -21, 3e7, 7.0], np.float32)
    t = sq.division_table(to_dev(s)).cpu().numpy()
    np.testing.assert_array_equal(t[:, 0], -s)
    inside = np.abs(s) <= 2.0 ** 20
    inside &= np.abs(s) >= 2.0 ** -20
    np.testing.assert_array_equal(t[inside, 1], (np.float32(1.0) / s[inside]).astype(np.float32))
    assert np.all(np.isnan(t[~inside, 1]))
