"""The Smooth-Dynamic quantiser given s's division table
(sq_quantize_act_table): codes, scale bit patterns and row L1 norms must be
those of the oracle's dynamic quantiser, on every kernel the dispatch picks
(rows in registers reading the table; the staged-ring and two-read kernels,
which take s), with and without the per-token maxima given.
"Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
Native Stack", Table 10 (Smooth-Dynamic).
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


def _check(sq, X, s, row_amax=None):
    q_ref, sx_ref = oracle.quantize_rows(X, s, "act")
    s_d = to_dev(s)
    table = sq.division_table(s_d)
    amax = None if row_amax is None else to_dev(row_amax)
    Xq, sx, Xop, l1 = sq.quantize_act_table(to_dev(X), s_d, table, row_amax=amax, want_l1=True)
    assert_codes_equal(Xq.cpu().numpy(), q_ref, "Xq")
    assert_codes_equal(op_as_int(Xop), q_ref, "Xop")
    assert_bits_equal(sx.cpu().numpy(), sx_ref, "x_scale")
    np.testing.assert_array_equal(l1.cpu().numpy(), np.abs(q_ref.astype(np.int64)).sum(axis=1))
    # each output alone
    _, sx2, Xop2 = sq.quantize_act_table(to_dev(X), s_d, table, row_amax=amax, want_q=False)
    Xq3, _, _ = sq.quantize_act_table(to_dev(X), s_d, table, row_amax=amax, want_op=False)
    assert_codes_equal(op_as_int(Xop2), q_ref, "Xop only")
    assert_codes_equal(Xq3.cpu().numpy(), q_ref, "Xq only")
    assert_bits_equal(sx2.cpu().numpy(), sx_ref, "x_scale (op only)")


# registers with the table: 1024 / 4096 / 8192 (rows of 1024 * 2^k) and 3072
# (above 2048), a ragged last row group (37 rows); 768 with 2520 rows: the ring
# kernel (s); 768 with 37 rows: registers; 16384: the two-read kernel (s)
SHAPES = [(37, 1024), (2048, 1024), (301, 4096), (9, 8192), (130, 3072), (2520, 768),
          (37, 768), (3, 16384), (1, 16)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_quantize_act_table_parity(sq, M, K):
    c = wl.make_case(M, K, 8, wl.EPI_BIAS, seed=M * 13 + K)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle_smoothing(X, W, 0.5)
    _check(sq, X, s)


@pytest.mark.parametrize("M,K", [(37, 1024), (301, 4096), (130, 3072), (2520, 768)])
def test_quantize_act_table_given_maxima(sq, M, K):
    c = wl.make_case(M, K, 8, wl.EPI_BIAS, seed=M + 7 * K)
    X, W = c.X.numpy(), c.W.numpy()
    s = oracle_smoothing(X, W, 0.5)
    amax = np.abs(oracle.smooth(X, s, "act")).max(axis=1).astype(np.float32)
    _check(sq, X, s, amax)


@pytest.mark.parametrize("K", [1024, 4096])
def test_quantize_act_table_extremes(sq, K):
    """Row maxima at extreme magnitudes and smoothing factors outside
    [2^-20, 2^20] (NaN reciprocals in the table: IEEE divisions there)."""
    rng = np.random.default_rng(K + 1)
    s = rng.uniform(0.05, 20.0, K).astype(np.float32)
    base = rng.standard_normal(K).astype(np.float32)
    base /= np.abs(base).max()
    rows = [(base * np.float32(m) * s).astype(np.float32)
            for m in (2.0 ** -61, 2.0 ** -60, 1.0, 2.0 ** 100, 2.0 ** 101)]
    X = np.stack(rows + [np.zeros(K, np.float32)]).astype(np.float32)
    for s_case in (s, np.where(np.arange(K) == 5, np.float32(1e-7), s).astype(np.float32),
                   np.where(np.arange(K) == 9, np.float32(3e7), s).astype(np.float32)):
        _check(sq, X, s_case)


# (rows, K): the register kernel (1024, 3072) and the staged-ring kernel (768
# with 2520 rows) in their given-maximum form
@pytest.mark.parametrize("M,K", [(40, 1024), (40, 3072), (2520, 768)])
def test_given_maxima_with_extreme_smoothing_factors(sq, M, K):
    """Columns whose smoothing factor lies outside [2^-20, 2^20] have no
    reciprocal in the division table (NaN): their codes come from IEEE
    divisions also when the row maxima are given and in range."""
    rng = np.random.default_rng(M * K)
    s = rng.uniform(0.5, 2.0, K).astype(np.float32)
    s[[3, 11]] = np.float32(1e-7), np.float32(3e7)
    X = rng.standard_normal((M, K)).astype(np.float32)
    X[:, 3] *= np.float32(1e-7)          # |x / s| of order 1 in the tiny-s column
    X[:, 11] *= np.float32(3e7)          # and in the huge-s column
    X[::7, 11] = 0.0
    amax = np.abs(oracle.smooth(X, s, "act")).max(axis=1).astype(np.float32)
    q_ref, sx_ref = oracle.quantize_rows(X, s, "act")
    s_d, a_d = to_dev(s), to_dev(amax)
    for label, (Xq, sx, Xop) in (
            ("rowmax", sq.quantize_act_rowmax(to_dev(X), s_d, a_d)),
            ("table", sq.quantize_act_table(to_dev(X), s_d, sq.division_table(s_d),
                                            row_amax=a_d))):
        assert_bits_equal(sx.cpu().numpy(), sx_ref, f"x_scale ({label})")
        assert_codes_equal(Xq.cpu().numpy(), q_ref, f"Xq ({label})")
        assert_codes_equal(op_as_int(Xop), q_ref, f"Xop ({label})")
