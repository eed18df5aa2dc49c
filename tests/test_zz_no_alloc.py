"""sq_linear_i8_static_ws: the GEMM with its split-K scratch in the library's
own static device memory, for callers that cannot allocate device memory
(a runtime with no allocator of its own, or code that must not touch the
memory pool of the framework it runs in).  Checked against sq_linear_i8_ws on
a caller workspace: identical outputs on two calls in a row, for split-K
shapes and an unsplit one; a warm call allocates nothing; stale counters that
a timed-out launch leaves are cleared by sq_device_status, after which the
outputs are identical again."""
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


def test_static_call_allocates_nothing(sq):
    """A warm static-scratch call leaves torch's allocator statistics and the
    device's free memory exactly as they were (the output is preallocated)."""
    M, N, K = 256, 1024, 4096
    rng = np.random.default_rng(7)
    Xop = to_dev(rng.integers(-127, 128, (M, K)).astype(np.float32), torch.bfloat16)
    Wop = to_dev(rng.integers(-127, 128, (N, K)).astype(np.float32), torch.bfloat16)
    out = torch.empty(M, N, dtype=torch.int32, device="cuda")
    sq.linear_i8_static_ws(Xop, None, Wop, None, None, None, sq.EPI_RAW_I32, out=out)
    torch.cuda.synchronize()
    stats0 = torch.cuda.memory_stats()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        sq.linear_i8_static_ws(Xop, None, Wop, None, None, None, sq.EPI_RAW_I32, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0
    for key in ("allocation.all.allocated", "reserved_bytes.all.current",
                "allocated_bytes.all.current", "segment.all.allocated"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key
    assert sq.device_status() == sq.SQ_OK


class _DeviceBytes:
    """A view of `n` bytes of device memory at `ptr` for torch.as_tensor."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3}


def test_static_scratch_recovers_after_a_timeout(sq):
    """Stale split-K counters in the static scratch (as a launch that gave up
    would leave them: every piece counted, no partial written) make the next
    split launch's bounded wait run out; sq_device_status reports
    SQ_ERR_TIMEOUT and clears the counters, after which static calls are bit
    for bit the caller-workspace path's again."""
    M, N, K = 256, 1024, 4096                       # 8 tiles x 4 pieces: split K
    assert sq.linear_workspace_bytes(M, N, K) > 0
    rng = np.random.default_rng(11)
    Xop = to_dev(rng.integers(-127, 128, (M, K)).astype(np.float32), torch.bfloat16)
    Wop = to_dev(rng.integers(-127, 128, (N, K)).astype(np.float32), torch.bfloat16)
    want = sq.linear_i8_ws(Xop, None, Wop, None, None, None, sq.EPI_RAW_I32,
                           workspace=sq.empty_workspace(sq.linear_workspace_bytes(M, N, K)))
    sq.linear_i8_static_ws(Xop, None, Wop, None, None, None, sq.EPI_RAW_I32)  # set-up
    assert sq.device_status() == sq.SQ_OK
    ptr, nbytes = sq.static_workspace()
    assert nbytes == sq.STATIC_WORKSPACE_BYTES
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    counters = torch.as_tensor(_DeviceBytes(ptr, sms * 64), device="cuda").view(torch.int32)
    assert int(counters.abs().sum()) == 0           # completed launches leave them at zero
    pairs = counters.view(-1, 2)
    pairs[:, 0] = 1000                              # "arrived": every piece thinks it is last
    pairs[:, 1] = 0                                 # "written": nothing ever arrives
    torch.cuda.synchronize()
    sq.linear_i8_static_ws(Xop, None, Wop, None, None, None, sq.EPI_RAW_I32)
    assert sq.device_status() == sq.SQ_ERR_TIMEOUT
    assert int(counters.abs().sum()) == 0           # cleared by the status report
    for call in range(2):
        got = sq.linear_i8_static_ws(Xop, None, Wop, None, None, None, sq.EPI_RAW_I32)
        assert torch.equal(got, want), f"call {call} after the reset"
    assert sq.device_status() == sq.SQ_OK
