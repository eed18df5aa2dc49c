"""Split-K schedule of the tcgen05 GEMM (caller workspace): the outputs equal
the whole-tile schedule's bit for bit, the int32 sums equal the oracle's on
sampled rows, and a workspace is reusable across calls and shapes."""
import numpy as np
import pytest
import torch

import oracle
from paritylib import assert_close_fp32, assert_codes_equal, to_dev
from smoothquant_w8a8_int8_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


def _codes(rng, rows, K, lo=-127, hi=127):
    return rng.integers(lo, hi + 1, (rows, K)).astype(np.int8)


def _case(M, N, K, seed, lo=-127, hi=127):
    rng = np.random.default_rng(seed)
    xq, wq = _codes(rng, M, K, lo, hi), _codes(rng, N, K, lo, hi)
    sx = rng.uniform(1e-3, 2e-2, M).astype(np.float32)
    sw = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    bias = rng.normal(0, 1, N).astype(np.float32)
    res = rng.normal(0, 1, (M, N)).astype(np.float32)
    return xq, wq, sx, sw, bias, res


def _op(q):
    return to_dev(q.astype(np.float32), torch.bfloat16)


# On 152 SMs (tiles of 128 x 256).  K is split when the tiles are fewer than
# the SMs and K >= 2048: each tile into min(4, SMs // tiles) pieces.
#   (128, 1024, 4096): 4 tiles x 4 pieces of 16 K blocks
#   (256, 1024, 4096): 8 tiles x 4 pieces (the small FFN-down)
#   (1000, 1000, 2080): ragged M, N, K (33 K blocks): chunk border inside pieces
#   (640, 512, 8192): 10 tiles x 4 pieces of 32 blocks, two exact passes each
#   (2560, 1024, 4096): 80 tiles, 1 piece: not split (no workspace needed)
#   (8192, 1024, 1024): more tiles than SMs: not split
SK_SHAPES = [(128, 1024, 4096), (256, 1024, 4096), (1000, 1000, 2080), (640, 512, 8192),
             (2560, 1024, 4096), (8192, 1024, 1024)]
MODES = [wl.EPI_NONE, wl.EPI_BIAS, wl.EPI_BIAS_GELU, wl.EPI_BIAS_RESIDUAL]


@pytest.mark.parametrize("M,N,K", SK_SHAPES)
def test_split_k_matches_whole_tiles_and_oracle(sq, M, N, K):
    xq, wq, sx, sw, bias, res = _case(M, N, K, seed=M + 7 * N + K)
    Xop, Wop = _op(xq), _op(wq)
    sx_d, sw_d, b_d, r_d = to_dev(sx), to_dev(sw), to_dev(bias), to_dev(res)
    nbytes = sq.linear_workspace_bytes(M, N, K)
    ws = sq.empty_workspace(nbytes)
    acc = sq.linear_i8_ws(Xop, None, Wop, None, mode=sq.EPI_RAW_I32, workspace=ws)
    acc_plain = sq.linear_i8(Xop, None, Wop, None, mode=sq.EPI_RAW_I32)
    assert torch.equal(acc, acc_plain)
    rows = np.unique(np.random.default_rng(M).integers(0, M, 96))
    acc_ref = oracle.gemm_i32(xq[rows], wq)
    assert_codes_equal(acc.cpu().numpy()[rows], acc_ref, "acc (sampled rows)")
    for mode in MODES:
        r = r_d if mode == wl.EPI_BIAS_RESIDUAL else None
        b = None if mode == wl.EPI_NONE else b_d
        y = sq.linear_i8_ws(Xop, sx_d, Wop, sw_d, b, r, mode, workspace=ws)
        y2 = sq.linear_i8_ws(Xop, sx_d, Wop, sw_d, b, r, mode, workspace=ws)  # reused as left
        y_plain = sq.linear_i8(Xop, sx_d, Wop, sw_d, b, r, mode)
        assert torch.equal(y, y_plain), f"mode {mode}"
        assert torch.equal(y2, y_plain), f"mode {mode} (second call)"
        ref = oracle.epilogue(acc_ref, sx[rows], sw, bias, res[rows], mode)
        assert_close_fp32(y.cpu().numpy()[rows], ref, f"mode {mode} vs oracle")


def test_split_k_workspace_reused_across_shapes(sq):
    """One workspace sized for the largest launch serves a sequence of shapes."""
    shapes = [(640, 512, 8192), (256, 1024, 4096), (1000, 1000, 2080), (128, 3072, 2048)]
    ws = sq.empty_workspace(max(sq.linear_workspace_bytes(*s) for s in shapes))
    for i, (M, N, K) in enumerate(shapes * 2):
        xq, wq, *_ = _case(M, N, K, seed=100 + i)
        Xop, Wop = _op(xq), _op(wq)
        a = sq.linear_i8_ws(Xop, None, Wop, None, mode=sq.EPI_RAW_I32, workspace=ws)
        assert torch.equal(a, sq.linear_i8(Xop, None, Wop, None, mode=sq.EPI_RAW_I32))


def test_split_k_single_pass_pieces(sq):
    """Small codes with their row L1 norms given: the whole K is one exact fp32
    pass, so each piece (32 K blocks) is summed in fp32 before the int32 fixup."""
    M, N, K = 256, 1024, 8192
    xq, wq, *_ = _case(M, N, K, seed=5, lo=-2, hi=2)
    xl1 = np.abs(xq.astype(np.int64)).sum(1).astype(np.int32)
    assert 127 * int(xl1.max()) < 2 ** 24
    Xop, Wop = _op(xq), _op(wq)
    ws = sq.empty_workspace(sq.linear_workspace_bytes(M, N, K))
    a = sq.linear_i8_ws(Xop, None, Wop, None, mode=sq.EPI_RAW_I32, x_l1=to_dev(xl1), workspace=ws)
    assert torch.equal(a, sq.linear_i8(Xop, None, Wop, None, mode=sq.EPI_RAW_I32))
    assert_codes_equal(a.cpu().numpy(), oracle.gemm_i32(xq, wq), "acc")


@pytest.mark.parametrize("K", [2064, 8192])
def test_split_k_adversarial_exactness(sq, K):
    """All +-127 codes (sums up to K * 16129, far above 2^24) split into many pieces."""
    M, N = 384, 512
    rng = np.random.default_rng(K)
    xq = np.full((M, K), 127, np.int8)
    wq = rng.choice(np.array([-127, 127], np.int8), (N, K))
    wq[0] = 127
    xq[1::3, 1::2] = -127
    ws = sq.empty_workspace(sq.linear_workspace_bytes(M, N, K))
    a = sq.linear_i8_ws(_op(xq), None, _op(wq), None, mode=sq.EPI_RAW_I32, workspace=ws)
    ref = oracle.gemm_i32(xq, wq)
    assert ref[0, 0] == K * 16129
    assert_codes_equal(a.cpu().numpy(), ref, "acc")


@pytest.mark.parametrize("mode", [wl.EPI_BIAS_GELU, wl.EPI_BIAS_RESIDUAL])
def test_split_k_requant(sq, mode):
    """The requantising epilogue on the split-K schedule: codes and scales
    equal the whole-tile schedule's (256 x 4096 x 4096: 32 tiles x 4 pieces)."""
    M, N, K = 256, 4096, 4096
    xq, wq, sx, sw, bias, res = _case(M, N, K, seed=mode)
    s_next = np.random.default_rng(1).uniform(0.2, 6.0, N).astype(np.float32)
    args = (_op(xq), to_dev(sx), _op(wq), to_dev(sw), to_dev(bias),
            to_dev(res) if mode == wl.EPI_BIAS_RESIDUAL else None, mode, to_dev(s_next), 0.05)
    ws = sq.empty_workspace(sq.linear_workspace_bytes(M, N, K))
    q1, o1, x1 = sq.linear_i8_requant_ws(*args, want_q=True, workspace=ws)
    q0, o0, x0 = sq.linear_i8_requant(*args, want_q=True)
    assert torch.equal(q1, q0) and torch.equal(o1, o0) and torch.equal(x1, x0)
    assert int((q0 != 0).sum()) > 0


def test_split_k_workspace_checks(sq):
    M, N, K = 256, 1024, 4096
    need = sq.linear_workspace_bytes(M, N, K)
    assert need > 0
    assert sq.linear_workspace_bytes(0, N, K) == 0
    assert sq.linear_workspace_bytes(8192, 1024, 1024) == 0  # more tiles than SMs
    assert sq.linear_workspace_bytes(256, 1024, 1024) == 0   # K below the split threshold
    xq, wq, *_ = _case(M, N, K, seed=9)
    Xop, Wop = _op(xq), _op(wq)
    small = sq.empty_workspace(need - 16)
    with pytest.raises(sq.SQError) as e:
        sq.linear_i8_ws(Xop, None, Wop, None, mode=sq.EPI_RAW_I32, workspace=small)
    assert e.value.status == sq.SQ_ERR_INVALID_ARG
    big = sq.empty_workspace(need + 64)
    with pytest.raises(sq.SQError) as e:
        sq.linear_i8_ws(Xop, None, Wop, None, mode=sq.EPI_RAW_I32, workspace=big[8:])
    assert e.value.status == sq.SQ_ERR_ALIGNMENT
    # no workspace: the whole-tile schedule
    a = sq.linear_i8_ws(Xop, None, Wop, None, mode=sq.EPI_RAW_I32, workspace=None)
    assert torch.equal(a, sq.linear_i8(Xop, None, Wop, None, mode=sq.EPI_RAW_I32))
    assert sq.device_status() == sq.SQ_OK
