"""The requantising GEMM epilogue divides by the next layer's smoothing factor
with a per-column reciprocal and one fused correction instead of an IEEE
division, and its codes are compared bit-exactly with the oracle's (which
divides).  Scaling x or s by a power of two scales every step exactly, so it is
enough to check significand pairs; these tests run the kernel's own division
routine (sq_check_division) against IEEE division where an error is most
likely -- every divisor against the largest and smallest dividend significands,
every dividend against the largest and smallest divisor significands -- and on
random blocks.  With SQ_EXHAUSTIVE_DIVISION=1 the last test sweeps all 2^46
pairs (about a minute).
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

FRAC = 1 << 23


@pytest.fixture(scope="module")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


def _run(sq, blocks, corrected=True):
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    for b0, bn, a0, an in blocks:
        sq.check_division(b0, bn, a0, an, corrected=corrected, out=out)
    torch.cuda.synchronize()
    assert sq.device_status() == 0
    n, where = (int(v) for v in out.cpu())
    return n, where


def _describe(where):
    if where == 0:
        return "none"
    w = where - 1
    return f"a_frac={w >> 32:#x} b_frac={w & 0xffffffff:#x}"


def test_every_divisor_extreme_dividends(sq):
    n, where = _run(sq, [(0, FRAC, FRAC - 256, 256), (0, FRAC, 0, 256)])
    assert n == 0, f"{n} mismatches, e.g. {_describe(where)}"


def test_every_dividend_extreme_divisors(sq):
    n, where = _run(sq, [(FRAC - 64, 64, 0, FRAC), (0, 64, 0, FRAC)])
    assert n == 0, f"{n} mismatches, e.g. {_describe(where)}"


def test_random_blocks(sq):
    rng = np.random.default_rng(20261202)
    blocks = [(int(rng.integers(0, FRAC - 4096)), 4096, int(rng.integers(0, FRAC - 65536)),
               65536) for _ in range(16)]
    n, where = _run(sq, blocks)
    assert n == 0, f"{n} mismatches, e.g. {_describe(where)}"


def test_check_can_fail(sq):
    """The checker is not vacuous: the uncorrected product x * RN(1/s) differs
    from the quotient, e.g. at b = 2 - 2^-23, a = 2 - 2^-22 (more than an ulp
    off), where the corrected quotient is exact; bad ranges are rejected."""
    from smoothquant_w8a8_int8_gb300.binding import SQError
    n, where = _run(sq, [(FRAC - 1, 1, FRAC - 2, 1)], corrected=False)
    assert n == 1 and where == 1 + (((FRAC - 2) << 32) | (FRAC - 1))
    n, _ = _run(sq, [(0, 4096, 0, 4096)], corrected=False)
    assert n > 0
    n, where = _run(sq, [(FRAC - 1, 1, FRAC - 2, 1)])
    assert n == 0, _describe(where)
    with pytest.raises(SQError):
        sq.check_division(FRAC - 1, 2, 0, 1)
    with pytest.raises(SQError):
        sq.check_division(0, 1, FRAC, 1)


@pytest.mark.skipif(os.environ.get("SQ_EXHAUSTIVE_DIVISION") != "1",
                    reason="full 2^46 sweep only with SQ_EXHAUSTIVE_DIVISION=1")
def test_all_significand_pairs(sq):
    step = 1 << 17
    n, where = _run(sq, [(b0, step, 0, FRAC) for b0 in range(0, FRAC, step)])
    assert n == 0, f"{n} mismatches, e.g. {_describe(where)}"
