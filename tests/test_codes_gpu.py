"""sq_linear_i8_codes: the linear on int8 activation codes (the per-token x
per-channel INT8 recipe's own input) against sq_linear_i8 on the quantiser's
GEMM operand and against the oracle.

The codes are widened exactly into the bf16 operand (every |q| <= 127 is a
bf16 integer), so every output must equal sq_linear_i8's bit for bit, the raw
int32 sums must equal the oracle's int64-checked triple loop, and the widened
workspace must equal the operand sq_quantize_act writes.  "Efficient INT8
Inference of Small NLP Models on Server CPUs with PyTorch Native Stack", the
INT8 recipe of per-token x per-channel scales and Table 5 (the GEMM shapes).
"""
import numpy as np
import pytest
import torch

import oracle
from paritylib import assert_codes_equal, oracle_smoothing, to_dev
from smoothquant_w8a8_int8_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


# one-CTA kernel (M < 256), pair kernel whole tiles and halves, a multi-pass K
SHAPES = [(77, 136, 1024, wl.EPI_NONE), (300, 200, 512, wl.EPI_BIAS),
          (512, 1024, 1024, wl.EPI_BIAS_GELU), (256, 1024, 4096, wl.EPI_BIAS_RESIDUAL),
          (2048, 768, 1088, wl.EPI_BIAS_RESIDUAL)]


@pytest.mark.parametrize("M,N,K,mode", SHAPES)
def test_codes_input_equals_operand_input(sq, M, N, K, mode):
    c = wl.make_case(M, K, N, wl.EPI_BIAS_RESIDUAL, seed=7 * M + N + K + mode)
    X, W = c.X.numpy(), c.W.numpy()
    s = to_dev(oracle_smoothing(X, W, 0.5))
    Wq, sw, Wop, wl1 = sq.pack_weight(to_dev(W), s, want_l1=True)
    Xq, sx, Xop, xl1 = sq.quantize_act(to_dev(X), s, want_l1=True)
    b = to_dev(c.bias.numpy())
    r = to_dev(c.residual.numpy()) if mode == wl.EPI_BIAS_RESIDUAL else None
    ws = torch.empty(sq.codes_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    y_op = sq.linear_i8(Xop, sx, Wop, sw, b, r, mode, x_l1=xl1, w_l1=wl1)
    y_q = sq.linear_i8_codes(Xq, sx, Wop, sw, b, r, mode, x_l1=xl1, w_l1=wl1, workspace=ws)
    assert torch.equal(y_q, y_op)
    # the widened operand is the quantiser's, bit for bit
    assert torch.equal(ws[: M * K * 2].view(torch.bfloat16).view(M, K), Xop)
    # raw sums against the oracle
    acc = sq.linear_i8_codes(Xq, None, Wop, None, None, None, sq.EPI_RAW_I32)
    assert_codes_equal(acc.cpu().numpy(),
                       oracle.gemm_i32(Xq.cpu().numpy(), Wq.cpu().numpy()), "acc")
    assert sq.device_status() == 0


def test_codes_extremes(sq):
    """Every code value -127..127 (and -128, which the quantiser never writes
    but the widening must still carry exactly) through the widening."""
    M, K = 16, 256
    vals = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    Xq = np.tile(vals, (M, 1)).astype(np.int8)
    Xq[1::2] = Xq[1::2, ::-1]
    W = np.zeros((8, K), np.int8)
    W[0] = 1
    W[1, 5] = 127
    W[2] = -1
    Wop = to_dev(W.astype(np.float32), torch.bfloat16)
    acc = sq.linear_i8_codes(to_dev(Xq), None, Wop, None, None, None, sq.EPI_RAW_I32)
    assert_codes_equal(acc.cpu().numpy(), oracle.gemm_i32(Xq, W), "acc")
