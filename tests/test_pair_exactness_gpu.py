"""Exact int32 sums of the CTA-pair tcgen05 kernel (launches of >= 256 rows)
in both of its accumulation schedules, against the oracle's int64-checked
triple loop, bit for bit.

The kernel multiplies int8 codes as exact bf16 numbers and sums them in fp32,
which is exact while every partial sum stays below 2^24.  Without row L1
norms it sums K in passes of <= 1024 and adds the passes in int32; with them
it sums all of K in one fp32 pass whenever 127 * (row L1) < 2^24 holds for
every row of either operand (L1 <= 132104).  These tests sit on both sides of
that bound (L1 = 132104: every sum reaches 2^24 - 8; L1 = 132105: chunked),
for the x-side norms alone, the w-side alone and both, on adversarial +-127
codes, at K = 2048, 4096 and 8192, and at the full BERT-large M = 8192 (rows
sampled; the remaining rows are checked against a closed form).

"Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
Native Stack", Table 5 (the GEMM shapes) and the INT8 recipe of per-token x
per-channel scales: the GEMM is int8 x int8 -> int32, exact.
"""
import numpy as np
import pytest
import torch

import oracle
from paritylib import assert_codes_equal, to_dev

pytestmark = pytest.mark.gpu

BOUND = 132104  # largest row L1 with 127 * L1 < 2^24


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


def _bound_rows(rows, K, L1, rng):
    """Codes whose row L1 norm is exactly L1 (a run of +-127, then the
    remainder), alternating row signs, the first rows exactly at L1 and the
    rest random small codes with a few 127s."""
    q = np.zeros((rows, K), np.int8)
    full, rest = divmod(L1, 127)
    q[:, :full] = 127
    q[:, full] = rest
    q[1::2] = -q[1::2]
    q[3::4, : full // 2] = -q[3::4, : full // 2]        # sign changes inside the run
    tail = rows // 2
    q[tail:] = rng.integers(-3, 4, (rows - tail, K)).astype(np.int8)
    q[tail:, :4] = 127
    q[tail::7] = q[0]                                    # more rows at the bound
    return q


def _pm127(rows, K, rng):
    q = np.full((rows, K), 127, np.int8)
    q[rows // 2:] = rng.choice(np.array([-127, 127], np.int8), (rows - rows // 2, K))
    q[1:rows // 2:3] = -127
    return q


def _as_op(q):
    return to_dev(q.astype(np.float32), torch.bfloat16)


def _l1(q):
    return to_dev(np.abs(q.astype(np.int64)).sum(1).astype(np.int32))


@pytest.mark.parametrize("K", [2048, 4096, 8192])
@pytest.mark.parametrize("L1", [BOUND, BOUND + 1])
@pytest.mark.parametrize("side", ["x", "w", "both"])
def test_pair_kernel_l1_bound(sq, K, L1, side):
    """M = 512 (two pair tiles along M), N = 768 (three along N; the bounded
    operand alone decides the pass count)."""
    M, N = 512, 768
    rng = np.random.default_rng(K + L1 + len(side))
    if side == "x":
        xq, wq = _bound_rows(M, K, L1, rng), _pm127(N, K, rng)
    elif side == "w":
        xq, wq = _pm127(M, K, rng), _bound_rows(N, K, L1, rng)
    else:
        xq, wq = _bound_rows(M, K, L1, rng), _bound_rows(N, K, L1, rng)
    x_l1 = _l1(xq) if side in ("x", "both") else None
    w_l1 = _l1(wq) if side in ("w", "both") else None
    ref = oracle.gemm_i32(xq, wq)
    if L1 == BOUND and side != "both":
        # the sums sit at the largest value one exact fp32 pass may reach
        assert np.abs(ref).max() == 127 * BOUND == 2 ** 24 - 8
    acc = sq.linear_i8(_as_op(xq), None, _as_op(wq), None, mode=sq.EPI_RAW_I32, x_l1=x_l1,
                       w_l1=w_l1)
    assert_codes_equal(acc.cpu().numpy(), ref, f"acc (side {side}, L1 {L1}, K {K})")


@pytest.mark.parametrize("N,K", [(1024, 4096), (3072, 2048)])
@pytest.mark.parametrize("L1", [BOUND, BOUND + 1])
def test_pair_kernel_l1_bound_full_m(sq, N, K, L1):
    """M = 8192 with the weight-side norms passed, as the benchmark calls the
    FFN down-projection: N = 1024 is the down-projection's shape, N = 3072
    runs the halved tiles of a short last wave.  Every weight row is at the
    bound; the activations are all +-127 with a known row pattern, so every
    output has a closed form; 96 seeded rows are also checked against the
    oracle's triple loop."""
    M = 8192
    rng = np.random.default_rng(N + K + L1)
    wq = _bound_rows(N, K, L1, rng)
    sgn = np.where(rng.random(M) < 0.5, -1, 1).astype(np.int8)   # row m of X = sgn[m] * 127
    xq = np.repeat((127 * sgn)[:, None], K, axis=1).astype(np.int8)
    acc = sq.linear_i8(_as_op(xq), None, _as_op(wq), None, mode=sq.EPI_RAW_I32, w_l1=_l1(wq))
    got = acc.cpu().numpy()
    rows = np.unique(np.concatenate([[0, 1, 255, 256, M - 1], rng.choice(M, 91, replace=False)]))
    assert_codes_equal(got[rows], oracle.gemm_i32(xq[rows], wq), "acc (sampled rows)")
    # every row: acc[m, n] = sgn[m] * 127 * sum_k wq[n, k]
    wsum = wq.astype(np.int64).sum(1)
    want = (sgn.astype(np.int64)[:, None] * 127 * wsum[None, :]).astype(np.int32)
    assert_codes_equal(got, want, "acc (closed form, all rows)")
