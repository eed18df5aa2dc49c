"""The seeded synthetic input recipe (no method arithmetic): outlier-channel
counts and scaling, channels fixed by their seed alone, reproducibility, the
GELU-input range, per-GEMM seeds and the workloads' operation counts."""
import math

import pytest
import torch

from smoothquant_w8a8_int8_gb300 import workloads as wl


@pytest.mark.parametrize("K,frac,count", [(1024, 0.01, 10), (4096, 0.01, 41), (768, 0.005, 4),
                                          (3072, 0.005, 15)])
def test_outlier_channel_counts(K, frac, count):
    ch = wl.outlier_channels(K, frac, torch.Generator().manual_seed(1))
    assert ch.numel() == count == math.floor(frac * K + 0.5)
    assert len(set(ch.tolist())) == count and 0 <= int(ch.min()) and int(ch.max()) < K


def _outlier_columns(X, scale):
    std = X.std(dim=0)
    return set(torch.nonzero(std > scale / 3).flatten().tolist()), std


@pytest.mark.parametrize("K,frac,scale", [(1024, 0.01, 20.0), (768, 0.005, 30.0)])
def test_outlier_columns_are_scaled(K, frac, scale):
    X = wl.make_activation(4096, K, seed=3, outlier_frac=frac, outlier_scale=scale)
    cols, std = _outlier_columns(X, scale)
    expected = set(wl.outlier_channels(K, frac, torch.Generator().manual_seed(3)).tolist())
    assert cols == expected
    inl = torch.tensor([j for j in range(K) if j not in cols])
    assert 0.9 < float(std[inl].min()) and float(std[inl].max()) < 1.1
    out = torch.tensor(sorted(cols))
    assert 0.9 * scale < float(std[out].min()) and float(std[out].max()) < 1.1 * scale


def test_channel_seed_fixes_the_outlier_channels():
    a = wl.make_activation(2048, 1024, seed=11, outlier_frac=0.01, outlier_scale=20.0,
                           channel_seed=99)
    b = wl.make_activation(1024, 1024, seed=12, outlier_frac=0.01, outlier_scale=20.0,
                           channel_seed=99)
    assert _outlier_columns(a, 20.0)[0] == _outlier_columns(b, 20.0)[0]
    assert not torch.equal(a[:1024], b)  # other values, same channels


def test_reproducible_and_row_prefix_stable():
    a = wl.make_case(256, 1024, 64, wl.EPI_BIAS_RESIDUAL, seed=5)
    b = wl.make_case(256, 1024, 64, wl.EPI_BIAS_RESIDUAL, seed=5)
    for x, y in ((a.X, b.X), (a.W, b.W), (a.bias, b.bias), (a.residual, b.residual)):
        assert torch.equal(x, y)
    short = wl.make_activation(64, 1024, seed=5, outlier_frac=0.01, outlier_scale=20.0)
    assert torch.equal(short, a.X[:64])
    c = wl.make_case(256, 1024, 64, wl.EPI_BIAS_RESIDUAL, seed=6)
    assert not torch.equal(a.X, c.X)


def test_weights_bias_residual_distributions():
    c = wl.make_case(1024, 1024, 1024, wl.EPI_BIAS_RESIDUAL, seed=7)
    assert abs(float(c.W.std()) - 0.02) < 0.001
    assert abs(float(c.bias.std()) - 0.02) < 0.003
    assert abs(float(c.residual.std()) - 1.0) < 0.01
    assert wl.make_case(8, 64, 8, wl.EPI_NONE, seed=7).bias is None
    assert wl.make_case(8, 64, 8, wl.EPI_BIAS, seed=7).residual is None


def test_gelu_input_range():
    X = wl.make_activation(2048, 4096, seed=9, outlier_frac=0.01, outlier_scale=20.0,
                           gelu_input=True)
    cols, _ = _outlier_columns(X, 20.0)
    inl = [j for j in range(4096) if j not in cols]
    gelu_min = -0.1700  # min over t of t * Phi(t), at t = -0.7518
    assert float(X[:, inl].min()) >= gelu_min
    assert float(X[:, sorted(cols)].min()) >= 20.0 * gelu_min


def test_workload_seeds_and_operation_counts():
    for w in wl.WORKLOADS.values():
        seeds = [wl.gemm_seed(w, l, i) for l in range(w.layers) for i in range(len(w.linears))]
        assert len(set(seeds)) == len(seeds)
    bert = wl.WORKLOADS["bert_large_encoder_b32_s256"]
    per_layer = 1024 * 3072 + 1024 * 1024 + 1024 * 4096 + 4096 * 1024
    assert bert.ops() == 2 * 8192 * 24 * per_layer == 4947802324992
    assert wl.WORKLOADS["bert_large_ffn_down_m256"].ops() == 2 * 256 * 4096 * 1024
