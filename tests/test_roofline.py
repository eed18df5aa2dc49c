"""The roofline / metric arithmetic reproduces the numbers printed in "Efficient
INT8 Inference of Small NLP Models on Server CPUs with PyTorch Native Stack",
Tables 4, 5 and 7 (fixture: tests/golden/table5_table7.txt)."""
import os

import pytest

from smoothquant_w8a8_int8_gb300 import roofline as R


def _rows(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "table5_table7.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append([c.strip() for c in line.split("|")])
    return out


def test_table5_arithmetic_intensity(golden_dir):
    for r in _rows(golden_dir):
        if len(r) != 7:
            continue
        M, K, N = map(int, r[0].split())
        for dt, want in (("fp32", r[2]), ("bf16", r[3]), ("int8", r[4])):
            assert round(R.arithmetic_intensity(M, K, N, dt), 2) == pytest.approx(float(want), abs=1e-9)


def test_table7_estimates_and_weighted_average(golden_dir):
    rows = _rows(golden_dir)
    shapes = []
    for r in rows:
        if len(r) != 7:
            continue
        M, K, N = map(int, r[0].split())
        est = R.estimated_tops(float(r[5]), R.arithmetic_intensity(M, K, N))
        assert round(est, 2) == pytest.approx(float(r[6]), abs=0.011)
        shapes.append((M, K, N, int(r[1]), float(r[6])))
    want = [float(r[1]) for r in rows if r[0] == "weighted_int8_tops"][0]
    assert round(R.weighted_tops(shapes), 2) == pytest.approx(want, abs=1e-9)


def test_table4_balance_point(golden_dir):
    r = [r for r in _rows(golden_dir) if r[0] == "gnr_balance"][0]
    assert round(R.balance_point(float(r[1]), float(r[2])), 2) == pytest.approx(float(r[3]), abs=1e-9)


def test_linear_and_quantizer_bytes():
    assert R.linear_bytes(2, 16, 3, R.EPI_NONE) == 2 * 16 + 16 * 3 + 4 * 6 + 8 + 12
    assert R.linear_bytes(2, 16, 3, R.EPI_BIAS) == R.linear_bytes(2, 16, 3, R.EPI_NONE) + 12
    assert R.linear_bytes(2, 16, 3, R.EPI_BIAS_RESIDUAL) == R.linear_bytes(2, 16, 3, R.EPI_BIAS) + 24
    assert R.quantize_bytes(8192, 1024) == 5 * 8192 * 1024 + 4 * 8192 + 4 * 1024
