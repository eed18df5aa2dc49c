"""Migration-strength (alpha) calibration sweep on synthetic data.

"Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
Native Stack", Table 15, picks SmoothQuant's migration strength alpha per model
and method (0.6 to 0.8) by task accuracy on datasets, which are not available
here.  This sweep uses the plainest synthetic proxy for that choice: for each
alpha on a grid, the relative Frobenius error of the INT8 linear block's output
against the exact product, on a calibration batch,

    err(alpha) = || Y_int8(alpha) - X W^T ||_F / || X W^T ||_F,

where Y_int8 runs the library's own kernels (smoothing factor, weight pack,
activation quantisation -- dynamic per token or static per tensor -- and the
tcgen05 GEMM with the plain dequantising epilogue), and the exact product is
taken in float64.  The alpha with the smallest error is reported.

`sweep()` is generic over the evaluation function; `gpu_error()` is the GPU
evaluation.  Run as a module for a JSON report on a workload's linears.
"""
from __future__ import annotations

import argparse
import json
import time
from typing import Callable, Dict, List, Sequence

import torch

DEFAULT_ALPHAS = tuple(round(0.1 * i, 1) for i in range(11))


def sweep(evaluate: Callable[[float], float], alphas: Sequence[float] = DEFAULT_ALPHAS) -> Dict:
    """evaluate(alpha) -> error for every alpha of the grid; returns the curve
    and the alpha with the smallest error (the first one on ties)."""
    alphas = [float(a) for a in alphas]
    if not alphas or any(not 0.0 <= a <= 1.0 for a in alphas):
        raise ValueError("alphas must lie in [0, 1]")
    curve = [{"alpha": a, "rel_err": float(evaluate(a))} for a in alphas]
    best = min(curve, key=lambda p: p["rel_err"])
    return {"curve": curve, "best_alpha": best["alpha"], "best_rel_err": best["rel_err"]}


def rel_error(y: torch.Tensor, ref: torch.Tensor) -> float:
    """|| y - ref ||_F / || ref ||_F in float64."""
    d = y.double() - ref.double()
    return float(torch.linalg.vector_norm(d) / torch.linalg.vector_norm(ref.double()))


def gpu_error(X: torch.Tensor, W: torch.Tensor, alpha: float, quant: str = "dynamic",
              X_calib: torch.Tensor = None, ref: torch.Tensor = None) -> float:
    """Relative output error of the INT8 linear block at migration strength
    alpha, with the library's kernels.  X [M, K] and W [N, K] fp32 on the GPU;
    the smoothing statistics (and the static scale) come from X_calib
    (default: X itself)."""
    from . import binding as sq
    Xc = X if X_calib is None else X_calib
    s = sq.smooth_factor(sq.channel_absmax(Xc), sq.channel_absmax(W), alpha)
    _, sw, Wop = sq.pack_weight(W, s, want_q=False)
    if quant == "static":
        scale = sq.static_scale(sq.act_absmax(Xc, s))
        _, sx, Xop = sq.quantize_act_static(X, s, scale, want_q=False)
    elif quant == "dynamic":
        _, sx, Xop = sq.quantize_act(X, s, want_q=False)
    else:
        raise ValueError("quant must be 'dynamic' or 'static'")
    y = sq.linear_i8(Xop, sx, Wop, sw, None, None, sq.EPI_NONE)
    if ref is None:
        ref = X.double() @ W.double().T
    return rel_error(y, ref)


def main():
    from . import workloads as wl
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="bert_large_encoder_b32_s256", choices=list(wl.WORKLOADS))
    ap.add_argument("--rows", type=int, default=2048, help="calibration tokens per linear")
    ap.add_argument("--quant", choices=["dynamic", "static"], default="dynamic")
    ap.add_argument("--alphas", default=",".join(str(a) for a in DEFAULT_ALPHAS))
    args = ap.parse_args()
    w = wl.WORKLOADS[args.workload]
    alphas = [float(a) for a in args.alphas.split(",")]
    dev = torch.device("cuda")
    report: List[Dict] = []
    t0 = time.perf_counter()
    for idx, lin in enumerate(w.linears):
        c = wl.workload_case(w, 0, idx, rows=args.rows, device=dev)
        # the static scale is calibrated on a separate batch of the same distribution
        calib = (wl.make_activation(512, lin.K, wl.gemm_seed(w, 0, idx) + 555, w.outlier_frac,
                                    w.outlier_scale, lin.gelu_input, device=dev,
                                    channel_seed=wl.gemm_seed(w, 0, idx))
                 if args.quant == "static" else None)
        ref = c.X.double() @ c.W.double().T
        res = sweep(lambda a: gpu_error(c.X, c.W, a, args.quant, calib, ref), alphas)
        res.update(linear=lin.name, K=lin.K, N=lin.N)
        report.append(res)
    torch.cuda.synchronize()
    print(json.dumps({"workload": w.name, "rows": args.rows, "quantisation": args.quant,
                      "seconds": round(time.perf_counter() - t0, 2), "linears": report}))


if __name__ == "__main__":
    main()
