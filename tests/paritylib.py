"""Helpers for the GPU-vs-oracle parity tests: run one linear case through
the oracle (CPU) and through the C-ABI (GPU) on the same seeded inputs and
compare.  Integer results and scale bit patterns must match exactly; fp32
outputs must satisfy max|Y - Y_ref| <= 1e-5 * max|Y_ref| + 1e-6."""
import numpy as np
import torch

import oracle

RTOL_MAX = 1e-5
ATOL = 1e-6


def assert_close_fp32(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, what
    if ref.size == 0:
        return
    err = np.max(np.abs(got - ref))
    bound = RTOL_MAX * np.max(np.abs(ref)) + ATOL
    assert err <= bound, f"{what}: max err {err:.3e} > bound {bound:.3e}"


def assert_bits_equal(got, ref, what=""):
    got = np.ascontiguousarray(got, np.float32).view(np.uint32)
    ref = np.ascontiguousarray(ref, np.float32).view(np.uint32)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{what}: {bad.size} scale bit mismatches, first at {bad[:5]}"


def assert_codes_equal(got, ref, what=""):
    got = np.asarray(got)
    ref = np.asarray(ref)
    assert got.shape == ref.shape, what
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{what}: {len(bad)} code mismatches, first at {bad[:5].tolist()}"


def oracle_smoothing(X, W, alpha):
    """The oracle's smoothing factor for inputs X (tokens x K), W (N x K)."""
    return oracle.smooth_factor(oracle.channel_absmax(X), oracle.channel_absmax(W),
                                np.float32(alpha))


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def op_as_int(op):
    """GEMM-operand buffer (bf16 holding integer codes) -> int8 numpy."""
    f = op.float().cpu().numpy()
    assert np.all(f == np.round(f)) and np.all(np.abs(f) <= 127)
    return f.astype(np.int8)
