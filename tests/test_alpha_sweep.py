"""Migration-strength sweep: its selection logic, the behaviour the pages'
method relies on (an interior alpha beats both no smoothing of the
activations and moving all of their range into the weights, on activations
with outlier channels), evaluated with the CPU oracle; and on the GPU, the
kernels' error curve against the oracle's."""
import numpy as np
import pytest

import oracle
from smoothquant_w8a8_int8_gb300 import alpha_sweep
from smoothquant_w8a8_int8_gb300 import workloads as wl


def oracle_error(X, W, alpha):
    """Relative output error of the oracle's INT8 linear block at alpha."""
    s = oracle.smooth_factor(oracle.channel_absmax(X), oracle.channel_absmax(W),
                             np.float32(alpha))
    wq, sw = oracle.quantize_rows(W, s, "weight")
    _, _, _, y = oracle.linear_block(X, s, wq, sw)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    return float(np.linalg.norm(y - ref) / np.linalg.norm(ref))


def test_sweep_selection():
    res = alpha_sweep.sweep(lambda a: (a - 0.6) ** 2 + 1.0, [0.0, 0.3, 0.6, 0.9])
    assert res["best_alpha"] == 0.6 and res["best_rel_err"] == 1.0
    assert [p["alpha"] for p in res["curve"]] == [0.0, 0.3, 0.6, 0.9]
    res = alpha_sweep.sweep(lambda a: 1.0, [0.2, 0.4])
    assert res["best_alpha"] == 0.2  # first on ties
    with pytest.raises(ValueError):
        alpha_sweep.sweep(lambda a: 0.0, [1.5])
    with pytest.raises(ValueError):
        alpha_sweep.sweep(lambda a: 0.0, [])


def test_interior_alpha_wins_on_outlier_activations():
    c = wl.make_case(96, 256, 64, wl.EPI_NONE, seed=7, outlier_frac=0.02, outlier_scale=30.0)
    X, W = c.X.numpy(), c.W.numpy()
    res = alpha_sweep.sweep(lambda a: oracle_error(X, W, a), [0.0, 0.25, 0.5, 0.75, 1.0])
    errs = {p["alpha"]: p["rel_err"] for p in res["curve"]}
    assert 0.0 < res["best_alpha"] < 1.0
    assert errs[res["best_alpha"]] < 0.5 * errs[0.0]
    assert errs[res["best_alpha"]] < errs[1.0]


@pytest.mark.gpu
@pytest.mark.parametrize("quant", ["dynamic", "static"])
def test_gpu_error_matches_oracle(quant):
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    binding.load()
    c = wl.make_case(200, 512, 136, wl.EPI_NONE, seed=5)
    X, W = c.X.numpy(), c.W.numpy()
    for a in (0.0, 0.5, 0.8):
        got = alpha_sweep.gpu_error(c.X.cuda(), c.W.cuda(), a, quant)
        if quant == "dynamic":
            want = oracle_error(X, W, a)
        else:
            s = oracle.smooth_factor(oracle.channel_absmax(X), oracle.channel_absmax(W),
                                     np.float32(a))
            wq, sw = oracle.quantize_rows(W, s, "weight")
            scale = oracle.static_scale(oracle.act_absmax(X, s))
            xq = oracle.quantize_static(X, s, scale)
            y = oracle.epilogue(oracle.gemm_i32(xq, wq), np.full(200, scale, np.float32), sw)
            ref = X.astype(np.float64) @ W.astype(np.float64).T
            want = float(np.linalg.norm(y - ref) / np.linalg.norm(ref))
        # same codes; the fp32 epilogue differs from the oracle's double one by
        # far less than the quantisation error itself
        assert abs(got - want) <= 1e-4 * want + 1e-7, (a, got, want)
