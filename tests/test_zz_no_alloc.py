"""sq_linear_i8_static_ws (scratch in the library's static device memory, no
workspace argument) against sq_linear_i8_ws on a caller workspace: identical
outputs on two calls in a row, for split-K shapes and an unsplit one."""
import numpy as np
import pytest
import torch

from paritylib import to_dev
from smoothquant_w8a8_int8_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


@pytest.mark.parametrize("M,N,K", [(256, 1024, 4096), (640, 512, 8192), (1000, 1000, 2080),
                                   (8192, 1024, 1024)])
@pytest.mark.parametrize("mode", [4, wl.EPI_BIAS_RESIDUAL])  # 4: raw int32 sums
def test_static_scratch_matches_caller_workspace(sq, M, N, K, mode):
    rng = np.random.default_rng(M + N + K + mode)
    Xop = to_dev(rng.integers(-127, 128, (M, K)).astype(np.float32), torch.bfloat16)
    Wop = to_dev(rng.integers(-127, 128, (N, K)).astype(np.float32), torch.bfloat16)
    raw = mode == sq.EPI_RAW_I32
    sx = None if raw else to_dev(rng.uniform(1e-3, 1e-2, M).astype(np.float32))
    sw = None if raw else to_dev(rng.uniform(1e-4, 1e-3, N).astype(np.float32))
    bias = None if raw else to_dev(rng.normal(0, 1, N).astype(np.float32))
    res = None if raw else to_dev(rng.normal(0, 1, (M, N)).astype(np.float32))
    need = sq.linear_workspace_bytes(M, N, K)
    assert need <= sq.STATIC_WORKSPACE_BYTES
    ws = sq.empty_workspace(need)
    for call in range(2):
        y_ws = sq.linear_i8_ws(Xop, sx, Wop, sw, bias, res, mode, workspace=ws)
        y_st = sq.linear_i8_static_ws(Xop, sx, Wop, sw, bias, res, mode)
        assert torch.equal(y_st, y_ws), f"call {call}"
    assert sq.device_status() == sq.SQ_OK
