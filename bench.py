#!/usr/bin/env python3
"""Benchmark of the SmoothQuant W8A8 INT8 linear block on one GB300.

One step = one forward pass of a workload's linear blocks: for every linear
layer, smoothing + dynamic per-token quantisation of its activations
(sq_quantize_act) and the INT8 GEMM with its fused dequantising epilogue
(sq_linear_i8).  Weights are packed once (offline, as the method prescribes)
before the timed region.  Default workload: BERT-large, 24 layers x
{QKV, attention out-proj, FFN up + GELU, FFN down + residual} at batch 32 x
sequence 256 (M = 8192).  Inputs are seeded synthetic data resident in HBM;
every GEMM reads its own activations (5.4 GB per step, far above the 129 MB
L2), so no step re-reads another's data from L2.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle
instead, on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from smoothquant_w8a8_int8_gb300 import replicas  # noqa: E402
from smoothquant_w8a8_int8_gb300 import roofline as R  # noqa: E402
from smoothquant_w8a8_int8_gb300 import workloads as wl  # noqa: E402

METRIC = "INT8 linear-block TOPS on BERT GEMM shapes; % of GB300 INT8 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def kernel_traffic():
    """Per-launch DRAM traffic of the GEMM kernel from the committed ncu
    capture, if that capture was taken of the kernel source as it is now."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "gemm_tc_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        h = hashlib.sha256()
        for src in d["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != d["source_sha256_16"]:
            return None, "kernel changed since the capture"
        return float(d["mean_traffic_bytes_per_launch"]), d["capture"]
    except (OSError, KeyError, ValueError):
        return None, "no capture"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            out = {}
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                if v is not None:
                    out[k] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"sq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # let nvidia-smi come up before the timed region starts
        time.sleep(0.5)

    def stop(self, window=None):
        """Summary of the samples whose timestamps fall in `window` (a pair
        of host datetimes around the timed region), else of all samples."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            lines = f.readlines()
        try:
            os.remove(self.path)
        except OSError:
            pass
        return clock_summary(lines, window)


CLOCK_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def clock_summary(lines, window=None):
    """Summary of nvidia-smi samples (lines of the ClockSampler query, CSV with
    no header and no units): median SM clock, highest maximum clock, and the
    throttle reasons seen active, over the samples whose timestamps fall in
    `window` (a pair of host datetimes around the timed region, widened by one
    sampling period), else over all samples.  Malformed lines are skipped."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            rows.append((ts, float(parts[2]), float(parts[3]),
                         [n for n, v in zip(CLOCK_REASONS, parts[6:10]) if v.lower() == "active"]))
        except ValueError:
            continue
    picked = []
    if window is not None:
        lo = window[0] - datetime.timedelta(milliseconds=60)
        hi = window[1] + datetime.timedelta(milliseconds=60)
        picked = [r for r in rows if lo <= r[0] <= hi]
    in_region = bool(picked)
    if not picked:
        picked = rows
    if not picked:
        return None
    reasons = sorted({n for r in picked for n in r[3]})
    return {"sm_mhz": statistics.median(r[1] for r in picked),
            "sm_max_mhz": max(r[2] for r in picked), "samples": len(picked),
            "in_timed_region": in_region, "reasons": reasons}


# ------------------------------------------------------------------- our arm

class Layer:
    __slots__ = ("lin", "X", "s", "Wop", "Wq", "sw", "wl1", "bias", "residual", "Y", "Xhost",
                 "Yhost", "static_scale", "feeds", "fed_by", "ln", "table", "row_amax",
                 "qtab")


LN_EPS = 1e-12


def step_bytes(layers, M):
    """Bytes one step's kernels touch: activations, packed weights, outputs."""
    return sum(M * L.lin.K * 4 + L.lin.N * L.lin.K * 2 + 2 * M * L.lin.N * 4 for L in layers)


def setup_workload(w: wl.Workload, gemm: str, rank: int, want_host: bool,
                   quant: str = "dynamic", ffn_chain: str = "off", ln: bool = False,
                   division_table: bool = True):
    from smoothquant_w8a8_int8_gb300 import binding as sq
    dev = torch.device("cuda")
    layers = []
    maxMK = max(w.M * lin.K for lin in w.linears)
    Xop_buf = torch.empty(maxMK, dtype=torch.bfloat16, device=dev)
    Xq_buf = torch.empty(maxMK, dtype=torch.int8, device=dev)
    sx_buf = torch.empty(w.M, dtype=torch.float32, device=dev)
    l1_buf = torch.empty(w.M, dtype=torch.int32, device=dev)
    chained = ffn_chain != "off"
    if chained:
        # codes of a chained FFN-down input (written by FFN-up's requantising
        # epilogue, or by the static quantiser from FFN-up's fp32 output)
        maxN = max(lin.N for lin in w.linears)
        bufs_chain = (torch.empty(w.M * maxN, dtype=torch.bfloat16, device=dev),
                      torch.empty(w.M, dtype=torch.float32, device=dev),
                      torch.zeros(w.M, dtype=torch.float32, device=dev))
    for layer, idx in [(l, i) for l in range(w.layers) for i in range(len(w.linears))]:
        lin = w.linears[idx]
        seed = replicas.rank_seed(wl.gemm_seed(w, layer, idx), rank)
        up = layers[-1] if (chained and lin.gelu_input and layers) else None
        if up is not None:
            # FFN-down fed by this layer's FFN-up: its smoothing factor and
            # Smooth-Static scale are calibrated offline on FFN-up's output for a
            # separate 512-token batch
            c = wl.make_case(w.M, lin.K, lin.N, lin.mode, seed, w.outlier_frac,
                             w.outlier_scale, lin.gelu_input, w.alpha, device=dev)
            calib_x = wl.make_activation(512, up.lin.K, seed + 555, w.outlier_frac,
                                         w.outlier_scale, False, device=dev,
                                         channel_seed=replicas.rank_seed(
                                             wl.gemm_seed(w, layer, idx - 1), rank))
            _, sxc, Xopc = sq.quantize_act(calib_x, up.s, want_q=False)
            y_cal = sq.linear_i8(Xopc, sxc, up.Wop, up.sw, up.bias, None, up.lin.mode)
            s = sq.smooth_factor(sq.channel_absmax(y_cal), sq.channel_absmax(c.W), w.alpha)
            L = Layer()
            L.lin = lin
            L.X = None
            L.s = s
            Wq, sw, Wop, wl1 = sq.pack_weight(c.W, s, want_q=(gemm == "mma_sync"),
                                              want_op=(gemm == "tc"), want_l1=True)
            L.Wq, L.sw, L.Wop, L.wl1 = Wq, sw, Wop, wl1
            L.bias, L.residual = c.bias, c.residual
            L.static_scale = (sq.static_scale(sq.act_absmax(y_cal, s))
                              if ffn_chain in ("unfused", "fused") else None)
            # the dynamic chain's division table of FFN-down's smoothing factor
            L.table = sq.division_table(s) if ffn_chain == "dynamic-fused" else None
            # the Smooth-Dynamic quantiser's own copy of it (offline, like Wop)
            L.qtab = (sq.division_table(s)
                      if division_table and ffn_chain in ("dynamic-unfused", "dynamic-fused")
                      else None)
            L.row_amax = None
            L.Y = torch.empty(w.M, lin.N, dtype=torch.float32, device=dev)
            L.Xhost = L.Yhost = None
            L.feeds = None
            L.ln = None
            L.fed_by = up
            up.feeds = L
            del c.W, c.X
            layers.append(L)
            continue
        c = wl.make_case(w.M, lin.K, lin.N, lin.mode, seed, w.outlier_frac, w.outlier_scale,
                         lin.gelu_input, w.alpha, device=dev)
        L = Layer()
        L.lin = lin
        L.X = c.X
        L.ln = None
        stats_src = c.X
        if ln and idx in (0, 2):
            # the QKV and FFN-up inputs come from the encoder's LayerNorms: X is
            # the pre-normalisation hidden state, gamma ~ 1 + N(0, 0.05),
            # beta ~ N(0, 0.05); the smoothing statistics are the LayerNorm's
            g = torch.Generator(device=dev)
            g.manual_seed(seed + 4242)
            gamma = 1.0 + 0.05 * torch.randn(lin.K, generator=g, device=dev)
            beta = 0.05 * torch.randn(lin.K, generator=g, device=dev)
            L.ln = (gamma.contiguous(), beta.contiguous())
            ones = torch.ones(lin.K, dtype=torch.float32, device=dev)
            _, _, _, stats_src, _ = sq.layernorm_quant(c.X, L.ln[0], L.ln[1], LN_EPS, ones,
                                                       want_q=False, want_y=True)
        # smoothing factor from this batch's own statistics (calibration = the input)
        s = sq.smooth_factor(sq.channel_absmax(stats_src), sq.channel_absmax(c.W), w.alpha)
        L.s = s
        Wq, sw, Wop, wl1 = sq.pack_weight(c.W, s, want_q=(gemm == "mma_sync"),
                                          want_op=(gemm == "tc"), want_l1=True)
        L.Wq, L.sw, L.Wop, L.wl1 = Wq, sw, Wop, wl1
        L.bias, L.residual = c.bias, c.residual
        L.static_scale = None
        if quant == "static":
            # Smooth-Static: the per-tensor scale is calibrated offline on a
            # separate batch drawn from the same distribution
            calib = wl.make_activation(512, lin.K, seed + 555, w.outlier_frac, w.outlier_scale,
                                       lin.gelu_input, device=dev, channel_seed=seed)
            if L.ln is not None:
                ones = torch.ones(lin.K, dtype=torch.float32, device=dev)
                _, _, _, calib, _ = sq.layernorm_quant(calib, L.ln[0], L.ln[1], LN_EPS, ones,
                                                       want_q=False, want_y=True)
            L.static_scale = sq.static_scale(sq.act_absmax(calib, s))
        L.Y = torch.empty(w.M, lin.N, dtype=torch.float32, device=dev)
        L.table = L.row_amax = None
        # the Smooth-Dynamic quantiser's division table of s (offline, like Wop)
        L.qtab = (sq.division_table(s) if division_table and quant == "dynamic" and L.ln is None
                  else None)
        L.Xhost = L.Yhost = None
        L.feeds = L.fed_by = None
        if want_host:
            L.Xhost = torch.empty(c.X.shape, dtype=torch.float32, pin_memory=True)
            L.Xhost.copy_(c.X)
            L.Yhost = torch.empty(L.Y.shape, dtype=torch.float32, pin_memory=True)
        del c.W
        layers.append(L)
    torch.cuda.synchronize()
    bufs = (Xq_buf, sx_buf, Xop_buf, l1_buf)
    return layers, bufs + (bufs_chain if chained else (None, None, None))


def quantise(sq, L, X, sx_buf, Xop):
    """The activation quantiser of one linear: fused with its LayerNorm when
    the input comes from one, Smooth-Static or Smooth-Dynamic."""
    static = 0.0 if L.static_scale is None else L.static_scale
    if L.ln is not None:
        sq.layernorm_quant(X, L.ln[0], L.ln[1], LN_EPS, L.s, static,
                           out=(None, sx_buf, Xop, None, None))
    elif L.static_scale is not None:
        sq.quantize_act_static(X, L.s, L.static_scale, out=(None, sx_buf, Xop))
    elif L.qtab is not None:
        sq.quantize_act_table(X, L.s, L.qtab, out=(None, sx_buf, Xop))
    else:
        sq.quantize_act(X, L.s, out=(None, sx_buf, Xop))


def linear(sq, ws, *a, **k):
    """The tcgen05 linear: split-K schedule on workspace `ws`, or whole tiles."""
    if ws is None:
        return sq.linear_i8(*a, **k)
    return sq.linear_i8_ws(*a, workspace=ws, **k)


def linear_requant(sq, ws, *a, **k):
    if ws is None:
        return sq.linear_i8_requant(*a, **k)
    return sq.linear_i8_requant_ws(*a, workspace=ws, **k)


def run_layer(sq, gemm, L, bufs, M, X=None, ev=None, ffn_chain="off", ws=None):
    """One linear of the step.  Returns whether an activation quantiser ran."""
    Xq_buf, sx_buf, Xop_buf, l1_buf, Xop_chain, sx_chain, amax_chain = bufs
    K, N = L.lin.K, L.lin.N
    X = L.X if X is None else X
    if ffn_chain != "off" and (L.feeds is not None or L.fed_by is not None):
        # the chained FFN pair (tcgen05 path)
        if L.fed_by is not None:
            if ev is not None:
                ev[0].record()
            chain_op = Xop_chain[: M * K].view(M, K)
            if ffn_chain == "unfused":
                sq.quantize_act_static(L.fed_by.Y, L.s, L.static_scale,
                                       out=(None, sx_chain, chain_op))
            elif ffn_chain == "dynamic-unfused" and L.qtab is not None:
                sq.quantize_act_table(L.fed_by.Y, L.s, L.qtab, out=(None, sx_chain, chain_op))
            elif ffn_chain == "dynamic-unfused":
                sq.quantize_act(L.fed_by.Y, L.s, out=(None, sx_chain, chain_op))
            elif ffn_chain == "dynamic-fused" and L.qtab is not None:
                sq.quantize_act_table(L.fed_by.Y, L.s, L.qtab, row_amax=amax_chain,
                                      out=(None, sx_chain, chain_op))
            elif ffn_chain == "dynamic-fused":
                sq.quantize_act_rowmax(L.fed_by.Y, L.s, amax_chain, out=(None, sx_chain, chain_op))
            if ev is not None:
                ev[1].record()
            linear(sq, ws, Xop_chain[: M * K].view(M, K), sx_chain, L.Wop, L.sw, L.bias,
                   L.residual, L.lin.mode, out=L.Y, w_l1=L.wl1)
            if ev is not None:
                ev[2].record()
            return ffn_chain != "fused"
        Xop = Xop_buf[: M * K].view(M, K)
        if ev is not None:
            ev[0].record()
        quantise(sq, L, X, sx_buf, Xop)
        if ev is not None:
            ev[1].record()
        if ffn_chain == "fused":
            nxt = L.feeds
            linear_requant(sq, ws, Xop, sx_buf, L.Wop, L.sw, L.bias, L.residual, L.lin.mode,
                           nxt.s, nxt.static_scale,
                           out=(None, Xop_chain[: M * N].view(M, N), sx_chain), w_l1=L.wl1)
        elif ffn_chain == "dynamic-fused":
            # the epilogue also merges FFN-down's per-token statistic
            amax_chain.zero_()
            sq.linear_i8_rowmax(Xop, sx_buf, L.Wop, L.sw, L.bias, L.residual, L.lin.mode,
                                L.feeds.table, row_amax=amax_chain, out=L.Y, w_l1=L.wl1)
        else:
            linear(sq, ws, Xop, sx_buf, L.Wop, L.sw, L.bias, L.residual, L.lin.mode, out=L.Y,
                   w_l1=L.wl1)
        if ev is not None:
            ev[2].record()
        return True
    if gemm == "tc":
        Xop = Xop_buf[: M * K].view(M, K)
        if ev is not None:
            ev[0].record()
        quantise(sq, L, X, sx_buf, Xop)
        if ev is not None:
            ev[1].record()
        # the packed weights' row L1 norms let the GEMM prove single-pass exactness
        linear(sq, ws, Xop, sx_buf, L.Wop, L.sw, L.bias, L.residual, L.lin.mode, out=L.Y,
               w_l1=L.wl1)
        if ev is not None:
            ev[2].record()
    else:
        Xq = Xq_buf[: M * K].view(M, K)
        if ev is not None:
            ev[0].record()
        sq.quantize_act(X, L.s, out=(Xq, sx_buf, None))
        if ev is not None:
            ev[1].record()
        sq.linear_i8_mma_sync(Xq, sx_buf, L.Wq, L.sw, L.bias, L.residual, L.lin.mode, out=L.Y)
        if ev is not None:
            ev[2].record()
    return True


def copy_ceiling(h2d_pairs, d2h_pairs, reps: int = 2) -> float:
    """Milliseconds per step of the e2e leg's copies alone: every host-to-
    device and device-to-host copy of one step, the two directions on two
    streams at once (the link's duplex rate on this machine, in this run)."""
    cur = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(cur)
    s_in.wait_stream(cur)
    s_out.wait_stream(cur)
    for _ in range(reps):
        with torch.cuda.stream(s_in):
            for dst, src in h2d_pairs:
                dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(s_out):
            for dst, src in d2h_pairs:
                dst.copy_(src, non_blocking=True)
    cur.wait_stream(s_in)
    cur.wait_stream(s_out)
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def codes_operand_leg(args, layers, bufs, M, ops_per_step, world):
    """The same step with the activation codes in their int8 format: the
    quantiser writes Xq (1 B per element) and sq_linear_i8_codes widens them
    into the bf16 operand before the GEMM (the default step has the quantiser
    write the bf16 operand itself).  Timed like `value`: K steps, no events
    between kernels, warm-up first."""
    from smoothquant_w8a8_int8_gb300 import binding as sq
    Xq_buf, sx_buf, Xop_buf = bufs[0], bufs[1], bufs[2]
    ws = Xop_buf.view(torch.uint8)  # the widened operand, where the default step keeps it

    def step():
        for L in layers:
            K = L.lin.K
            Xq = Xq_buf[: M * K].view(M, K)
            if L.qtab is not None:
                sq.quantize_act_table(L.X, L.s, L.qtab, out=(Xq, sx_buf, None))
            else:
                sq.quantize_act(L.X, L.s, out=(Xq, sx_buf, None))
            sq.linear_i8_codes(Xq, sx_buf, L.Wop, L.sw, L.bias, L.residual, L.lin.mode,
                               out=L.Y, w_l1=L.wl1, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    replicas.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        step()
    t1.record()
    torch.cuda.synchronize()
    rc = sq.device_status()
    if rc != 0:
        raise RuntimeError(f"device status after the int8-operand run: {sq.status_string(rc)}")
    ms = replicas.max_over_ranks(t0.elapsed_time(t1), device="cuda") / args.steps
    return {"value": round(replicas.whole_job_tops(ops_per_step, world, ms), 3), "unit": "TOPS",
            "ms_per_step": round(ms, 4),
            "path": "sq_quantize_act(_table) writing int8 codes, then sq_linear_i8_codes (an exact "
                    "widening pass into the bf16 operand, then the same tcgen05 GEMM)"}


def e2e_leg(args, layers, M, ops_per_step, world):
    """The block end to end through the public host-buffer API
    (HostLinearPipeline): K steps timed with CUDA events, every output
    compared with the device path's, and the same bytes copied with no
    kernels as the link ceiling of this run."""
    from smoothquant_w8a8_int8_gb300.pipeline import HostLinearPipeline, LinearLayer
    pipe = HostLinearPipeline(M, max(L.lin.K for L in layers), max(L.lin.N for L in layers))
    specs = [LinearLayer(L.s, L.Wop, L.sw, L.lin.mode, L.bias, L.residual, L.wl1,
                         L.static_scale, L.qtab) for L in layers]
    xh = [L.Xhost for L in layers]
    yh = [L.Yhost for L in layers]
    h2d = sum(L.Xhost.numel() * 4 for L in layers)
    d2h = sum(L.Yhost.numel() * 4 for L in layers)
    pipe.run(specs, xh, yh)
    torch.cuda.synchronize()
    replicas.barrier()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(args.e2e_steps):
        pipe.run(specs, xh, yh)
    e1.record(cur)
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e_ms = replicas.max_over_ranks(e_ms, device="cuda")
    # every output that came back equals the device path's output
    ok = all(torch.equal(L.Yhost.cuda(non_blocking=True), L.Y) for L in layers)
    # the same copies alone (both directions at once, on the pipeline's own
    # device slots, after the buffers' first use): the link's rate in this run
    pairs_in = [(pipe.x_slots[i % 2][: x.numel()].view(x.shape), x) for i, x in enumerate(xh)]
    pairs_out = [(y, pipe.y_slots[i % 2][: y.numel()].view(y.shape)) for i, y in enumerate(yh)]
    copy_ceiling(pairs_in, pairs_out, reps=1)
    copy_ms = copy_ceiling(pairs_in, pairs_out, reps=3)
    return {"value": round(replicas.whole_job_tops(ops_per_step, world, e_ms), 3),
            "unit": "TOPS", "ms_per_step": round(e_ms, 3), "steps": args.e2e_steps,
            "timing": "CUDA events on the calling stream around K pipeline runs",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "link_gbs": round((h2d + d2h) / (e_ms * 1e-3) / 1e9, 1),
            "copies_only_ms_per_step": round(copy_ms, 3),
            "copies_only_gbs": round((h2d + d2h) / (copy_ms * 1e-3) / 1e9, 1),
            "outputs_match_device": bool(ok),
            "outputs_checked": "every element of every layer's Y",
            "path": "sq_linear_block_host (C ABI): pinned host X -> device, the layer's "
                    "quantiser + sq_linear_i8, Y -> pinned host, copies overlapped with kernels "
                    "on three streams (called through "
                    "smoothquant_w8a8_int8_gb300.pipeline.HostLinearPipeline)"}


def bench_ours(args, w: wl.Workload, rank: int, world: int, headline: bool = True):
    from smoothquant_w8a8_int8_gb300 import binding as sq
    sq.load()
    peaks, peak_src = load_peaks()
    chained = args.ffn_chain != "off"
    if chained and args.gemm != "tc":
        raise SystemExit("--ffn-chain needs the tcgen05 GEMM (--gemm tc)")
    if args.ln and args.gemm != "tc":
        raise SystemExit("--ln needs the tcgen05 GEMM (--gemm tc)")
    layers, bufs = setup_workload(w, args.gemm, rank,
                                  want_host=(args.e2e_steps > 0 and not chained and not args.ln
                                             and headline),
                                  quant=args.quant, ffn_chain=args.ffn_chain, ln=args.ln,
                                  division_table=args.division_table == "on")
    M = w.M
    n_gemm = len(layers)
    quantised = [True] * n_gemm  # which linears run an activation quantiser kernel
    # one split-K workspace, sized for the largest linear, allocated once
    ws = None
    if args.gemm == "tc" and args.schedule == "split-k":
        ws_bytes = max(sq.linear_workspace_bytes(M, lin.N, lin.K) for lin in w.linears)
        ws = sq.empty_workspace(ws_bytes) if ws_bytes > 0 else None

    def step(ev_list=None):
        for i, L in enumerate(layers):
            quantised[i] = run_layer(sq, args.gemm, L, bufs, M,
                                     ev=None if ev_list is None else ev_list[i],
                                     ffn_chain=args.ffn_chain, ws=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rc = sq.device_status()
    if rc != 0:
        raise RuntimeError(f"device status after warm-up: {sq.status_string(rc)}")

    # per-launch events of the kernel pass (below)
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_gemm)]
           for _ in range(args.steps)]
    # a step whose data fits in L2 would run from L2 when repeated: then every
    # timed step is preceded by a write of a buffer twice the L2 size, outside
    # its events, and the step times are summed
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = None
    if step_bytes(layers, M) < 2 * l2:
        flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device="cuda")
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device()) if headline else None
    replicas.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    host_t0 = datetime.datetime.now()
    t0.record()
    for k in range(args.steps):
        if flush is not None:
            flush.fill_(float(k))
            step_ev[k][0].record()
        step()
        if flush is not None:
            step_ev[k][1].record()
    t1.record()
    torch.cuda.synchronize()
    host_t1 = datetime.datetime.now()
    replicas.barrier()
    clock_info = clocks.stop((host_t0, host_t1)) if clocks is not None else None
    elapsed_ms = t0.elapsed_time(t1)
    if flush is not None:
        elapsed_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    rc = sq.device_status()
    if rc != 0:
        raise RuntimeError(f"device status after timed run: {sq.status_string(rc)}")
    elapsed_ms = replicas.max_over_ranks(elapsed_ms, device="cuda")

    # kernel pass: the same K steps again, with CUDA events around every launch
    # on the launching stream.  An event between two kernels leaves the GPU idle
    # at that boundary (and stops the next launch from overlapping the previous
    # kernel's tail), so this pass yields the per-kernel durations -- the
    # rooflines and kernel_ms_per_step -- and not `value`.
    for k in range(args.steps):
        if flush is not None:
            flush.fill_(float(k))
        step(evs[k])
    torch.cuda.synchronize()
    rc = sq.device_status()
    if rc != 0:
        raise RuntimeError(f"device status after kernel pass: {sq.status_string(rc)}")

    # launch-bound shapes: per-step time over many back-to-back steps, replayed
    # from a CUDA graph (no host launch cost, no L2 flush: the step's data
    # stays in L2)
    back_to_back = None
    if w.M <= 256 and args.back_to_back > 0:
        per_graph = 50
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                step()
        graph.replay()
        torch.cuda.synchronize()
        reps = max(1, args.back_to_back // per_graph)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record()
        for _ in range(reps):
            graph.replay()
        b1.record()
        torch.cuda.synchronize()
        rc = sq.device_status()
        if rc != 0:
            raise RuntimeError(f"device status after back-to-back run: {sq.status_string(rc)}")
        n_b2b = reps * per_graph
        us_b2b = b0.elapsed_time(b1) * 1e3 / n_b2b
        back_to_back = {"steps": n_b2b, "us_per_step": round(us_b2b, 3),
                        "tops": round(w.ops() / (us_b2b * 1e-6) / 1e12, 3),
                        "note": "quantiser + GEMM per step: CUDA-graph replays of 50 captured "
                                "steps, back to back, no L2 flush (warm L2)"}
        del graph

    ops_per_step = w.ops()
    ms_per_step = elapsed_ms / args.steps
    tops = replicas.whole_job_tops(ops_per_step, world, ms_per_step)

    # per-kernel durations from the live events
    q_ms = g_ms = 0.0
    for k in range(args.steps):
        for i in range(n_gemm):
            e = evs[k][i]
            q_ms += e[0].elapsed_time(e[1])
            g_ms += e[1].elapsed_time(e[2])
    n_launch = args.steps * n_gemm
    gemm_ops = args.steps * ops_per_step
    gemm_tops = gemm_ops / (g_ms * 1e-3) / 1e12
    # every GEMM launch of the kernel pass is timed on its own (events on both
    # sides, an idle GPU at each boundary), tens of microseconds long: the
    # burst figure is the peak that applies (the sustained one is for kernels
    # timed inside a seconds-long run)
    peak_tensor = peaks["bf16_tflops"]
    q_bytes = args.steps * sum(R.quantize_bytes(M, L.lin.K)
                               for L, qd in zip(layers, quantised) if qd)
    n_quant = args.steps * sum(quantised)
    q_gbs = q_bytes / (q_ms * 1e-3) / 1e9
    g_bytes = args.steps * sum(R.linear_bytes(M, L.lin.K, L.lin.N, L.lin.mode) for L in layers)

    # e2e through the public API with host buffers: activations in pinned
    # host memory, copied in, the linear block, Y copied out, inside the timed
    # region (three streams overlap copies with the kernels), timed with CUDA
    # events on the calling stream
    e2e = None
    if args.e2e_steps > 0 and not chained and not args.ln and headline:
        e2e = e2e_leg(args, layers, M, ops_per_step, world)
    codes = None
    if headline and args.gemm == "tc" and args.quant == "dynamic" and not chained and not args.ln:
        codes = codes_operand_leg(args, layers, bufs, M, ops_per_step, world)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and headline:
        cpu = cpu_baseline(w, target_s=args.cpu_seconds)

    traffic, traffic_src = kernel_traffic() if args.gemm == "tc" else (None, "not captured")
    gemm_kernel = ("tcgen05.mma kind::f16 (int8 codes as exact bf16, fp32 TMEM chunks of "
                   "K<=1024 summed in int32); launches of >= 256 rows on CTA pairs "
                   "(cta_group::2, 256x256 tiles), smaller ones on single CTAs"
                   if args.gemm == "tc" else "mma.sync m16n8k32 s8 (legacy warp MMA)")
    result = {
        "metric": METRIC, "value": round(tops, 3), "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded N(0,1) activations with outlier channels, N(0,0.02) weights)",
        "config": {"workload": w.name, "description": w.description, "M": M,
                   "layers": w.layers, "gemms_per_step": n_gemm,
                   "ops_per_step": ops_per_step, "gemm_kernel": gemm_kernel,
                   "gemm_schedule": ("split K: linears with fewer tiles than SMs and "
                                     "K >= 2048 cut each tile's K range over up to 4 SMs "
                                     "(sq_linear_i8_ws workspace)"
                                     if ws is not None else
                                     "whole tiles (halves when the last wave is short)"),
                   "launch": "programmatic dependent launch (set-up overlaps the previous "
                             "kernel; all memory access after griddepcontrol.wait)",
                   "l2": ("inputs larger than L2: every GEMM reads its own activations "
                          f"({sum(M * L.lin.K * 4 for L in layers) / 1e9:.1f} GB per step)"
                          if flush is None else
                          f"L2 flushed before every step (a {2 * l2 / 1e6:.0f} MB buffer "
                          f"written outside the step's events; the step touches "
                          f"{step_bytes(layers, M) / 1e6:.0f} MB)"),
                   "weights": "packed once before the timed region",
                   "kernel_timing": ("value: K steps with no event between kernels; roofline and "
                                     "kernel_ms_per_step: a second pass of the same K steps with "
                                     "CUDA events around every launch"),
                   "quantisation": ("Smooth-Static (per-tensor scale calibrated offline on a "
                                    "separate 512-token batch of the same distribution)"
                                    if args.quant == "static"
                                    else "Smooth-Dynamic (per-token scales at run time"
                                    + ("; s's division table made offline with the packed "
                                       "weights, sq_quantize_act_table)"
                                       if args.division_table == "on" else ")")),
                   "parallelism": f"replicas x{world} (rows shard, no collective)",
                   "ffn_chain": {"off": "not chained: every linear has its own input",
                                 "unfused": "FFN-down consumes FFN-up's output: fp32 Y, then "
                                            "the Smooth-Static quantiser",
                                 "fused": "FFN-down consumes FFN-up's output: FFN-up's "
                                          "epilogue emits FFN-down's Smooth-Static codes "
                                          "(sq_linear_i8_requant)",
                                 "dynamic-unfused": "FFN-down consumes FFN-up's output: fp32 Y, "
                                                    "then the Smooth-Dynamic quantiser "
                                                    "(sq_quantize_act)",
                                 "dynamic-fused": "FFN-down consumes FFN-up's output: FFN-up's "
                                                  "epilogue also merges FFN-down's per-token "
                                                  "maxima (sq_linear_i8_rowmax), then the "
                                                  "given-maximum quantiser "
                                                  "(sq_quantize_act_rowmax)"}[args.ffn_chain],
                   "layernorm": ("the QKV and FFN-up inputs pass through LayerNorm fused with "
                                 "their quantiser (sq_layernorm_quant)" if args.ln else "none")},
        "roofline": {"bound": "tensor", "kernel": "gemm+epilogue",
                     "achieved": round(gemm_tops, 2), "peak": peak_tensor,
                     "unit": "TFLOP/s", "frac": round(gemm_tops / peak_tensor, 4),
                     "traffic": traffic,
                     "traffic_source": traffic_src,
                     "peak_source": f"bf16 dense burst, {peak_src} (each launch is timed on "
                                    f"its own; sustained {peaks['bf16_tflops_sustained']} "
                                    f"gives frac "
                                    f"{gemm_tops / peaks['bf16_tflops_sustained']:.4f})",
                     "avg_launch_us": round(g_ms * 1e3 / n_launch, 2),
                     "algorithmic_bytes_per_step": g_bytes // args.steps},
        "quantiser_roofline": {"bound": "hbm", "achieved": round(q_gbs, 1),
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": round(q_gbs / peaks["hbm_gbs"], 4),
                               "peak_source": peak_src,
                               "avg_launch_us": round(q_ms * 1e3 / max(1, n_quant), 2),
                               "algorithmic_bytes_per_step": q_bytes // args.steps},
        "kernel_ms_per_step": {"quantize": round(q_ms / args.steps, 4),
                               "gemm": round(g_ms / args.steps, 4)},
        "gpu_launches": n_gemm * args.steps + n_quant,
        "back_to_back": back_to_back,
        "int8_operand": codes,
        "clocks": clock_info,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    return result


# ------------------------------------------------------------ oracle timing

def _oracle_sample(w: wl.Workload, rows: int):
    """Inputs of one layer's linears with `rows` tokens, plus packed weights
    and the smoothing factor (computed by the oracle, untimed)."""
    import oracle
    items = []
    for idx, lin in enumerate(w.linears):
        c = wl.workload_case(w, 0, idx, rows=rows)
        X, W = c.X.numpy(), c.W.numpy()
        s = oracle.smooth_factor(oracle.channel_absmax(X), oracle.channel_absmax(W), w.alpha)
        wq, sw = oracle.quantize_rows(W, s, "weight")
        items.append((X, s, wq, sw, None if c.bias is None else c.bias.numpy(),
                      None if c.residual is None else c.residual.numpy(), lin.mode))
    return items


def _oracle_step(items):
    import oracle
    for X, s, wq, sw, b, r, mode in items:
        oracle.linear_block(X, s, wq, sw, b, r, mode)


def _sample_ops(w, rows):
    return sum(2 * rows * lin.K * lin.N for lin in w.linears)


def _calibrate_rows(w: wl.Workload, target_s: float):
    rows = 16
    items = _oracle_sample(w, rows)
    t = time.perf_counter()
    _oracle_step(items)
    dt = max(time.perf_counter() - t, 1e-4)
    return int(max(16, min(w.M, rows * target_s / dt)))


def cpu_baseline(w: wl.Workload, target_s: float = 15.0):
    """The oracle as it stands, on the host cores, on a bounded row sample of
    one layer of the workload (quantise + integer GEMM + epilogue)."""
    import oracle
    rows = _calibrate_rows(w, target_s)
    items = _oracle_sample(w, rows)
    # A full layer can take less than the target on many cores: repeat the
    # pass until the target time has elapsed.
    passes = 0
    t = time.perf_counter()
    while True:
        _oracle_step(items)
        passes += 1
        dt = time.perf_counter() - t
        if dt >= target_s or dt * (passes + 1) / passes > 2.5 * target_s:
            break
    ops = _sample_ops(w, rows) * passes
    return {"value": round(ops / dt / 1e12, 6), "unit": "TOPS", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"layer 0 of {w.name}: {len(w.linears)} linears x {rows} of {w.M} rows, "
                      f"{passes} pass(es) ({ops / 1e9:.1f} GOP), quantise + int64 GEMM + "
                      f"double epilogue"}


def bench_reference(args, w: wl.Workload):
    """The CPU oracle timed as the reference arm (each step a bounded sample)."""
    import oracle
    rows = _calibrate_rows(w, args.reference_step_seconds)
    items = _oracle_sample(w, rows)
    for _ in range(args.warmup):
        _oracle_step(items)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(items)
    dt = (time.perf_counter() - t) / args.steps
    ops = _sample_ops(w, rows)
    value = ops / dt / 1e12
    cores = oracle.num_threads()
    sample = (f"layer 0 of {w.name}: {len(w.linears)} linears x {rows} of {w.M} rows "
              f"({ops / 1e9:.2f} GOP per step)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int64 (exact integer sums), fp32 quantiser",
            "data": "synthetic", "config": {"workload": w.name, "M": w.M, "layers": w.layers},
            "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def bench_attention(args, B=32, S=256, H=16, D=64, reps=20):
    """The encoder's self-attention at the BERT-large layer shape on the fused
    QKV output (sq_attention): per-call time with L2 flushed before each call
    (the 101 MB input fits in L2), and its rooflines."""
    from smoothquant_w8a8_int8_gb300 import binding as sq
    peaks, peak_src = load_peaks()
    g = torch.Generator(device="cuda")
    g.manual_seed(1240)
    QKV = (torch.randn(B * S, 3 * H * D, generator=g, device="cuda") * 0.6).contiguous()
    O = torch.empty(B * S, H * D, dtype=torch.float32, device="cuda")
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device="cuda")
    for _ in range(max(3, getattr(args, "warmup", 3))):
        sq.attention(QKV, B, S, H, D, out=O)
    torch.cuda.synchronize()
    times = []
    for r in range(reps):
        flush.fill_(float(r))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        sq.attention(QKV, B, S, H, D, out=O)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    rc = sq.device_status()
    if rc != 0:
        raise RuntimeError(f"device status after attention: {sq.status_string(rc)}")
    ms = statistics.median(times)
    flops = 4 * B * H * S * S * D                 # Q K^T and P V, 2 flops per multiply-add
    issued = 3 * flops                            # three tf32 products per split contraction
    nbytes = B * S * 3 * H * D * 4 + B * S * H * D * 4
    tf32_peak = peaks["bf16_tflops"] * (1.1 / 2.25)
    del flush
    return {"shape": {"batch": B, "seq": S, "heads": H, "head_dim": D},
            "us_per_call": round(ms * 1e3, 2), "calls": reps,
            "l2": "flushed before every call (a 2x L2 buffer written outside the events)",
            "tflops_exact_math": round(flops / (ms * 1e-3) / 1e12, 2),
            "roofline": {"bound": "tensor", "achieved": round(issued / (ms * 1e-3) / 1e12, 2),
                         "peak": round(tf32_peak, 1), "unit": "TFLOP/s (tf32 issued)",
                         "frac": round(issued / (ms * 1e-3) / 1e12 / tf32_peak, 4),
                         "peak_source": f"bf16 dense burst ({peak_src}) x 1.1/2.25, the "
                                        "nominal tf32/bf16 ratio"},
            "hbm": {"achieved_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                    "peak_gbs": peaks["hbm_gbs"],
                    "frac": round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                    "bytes": nbytes}}


def other_configs(args, headline: wl.Workload, rank: int, world: int):
    """Every other workload, measured the same way (its own setup, warm-up,
    timed steps and kernel pass) after the headline one: a compact summary
    each.  The batch-1 single linears (M = 256) are launch-bound: they also
    report the per-step time of many back-to-back steps."""
    out = {}
    sub = argparse.Namespace(**vars(args))
    sub.e2e_steps = 0
    for name in wl.WORKLOAD_ORDER:
        if name == headline.name:
            continue
        r = bench_ours(sub, wl.WORKLOADS[name], rank, world, headline=False)
        out[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "roofline",
                                       "quantiser_roofline", "kernel_ms_per_step",
                                       "back_to_back")}
        out[name]["l2"] = r["config"]["l2"]
        out[name]["gemm_schedule"] = r["config"]["gemm_schedule"]
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bert_large_encoder_b32_s256",
                    choices=list(wl.WORKLOADS))
    ap.add_argument("--gemm", choices=["tc", "mma_sync"], default="tc")
    ap.add_argument("--quant", choices=["dynamic", "static"], default="dynamic",
                    help="activation quantisation: per-token dynamic (Smooth-Dynamic, the "
                         "default) or per-tensor static (Smooth-Static)")
    ap.add_argument("--ffn-chain",
                    choices=["off", "unfused", "fused", "dynamic-unfused", "dynamic-fused"],
                    default="off",
                    help="chain each layer's FFN-down to its FFN-up: Smooth-Static input "
                         "through fp32 Y and the static quantiser (unfused) or the requantising "
                         "epilogue (fused); Smooth-Dynamic input through fp32 Y and the dynamic "
                         "quantiser (dynamic-unfused) or the row-maximum epilogue and the "
                         "given-maximum quantiser (dynamic-fused)")
    ap.add_argument("--schedule", choices=["split-k", "whole"], default="split-k",
                    help="tcgen05 GEMM: split K over several SMs where the tiles are fewer "
                         "than the SMs and K >= 2048 (workspace), or whole tiles only")
    ap.add_argument("--division-table", choices=["on", "off"], default="on",
                    help="Smooth-Dynamic quantisers read s's division table, made offline "
                         "with the packed weights (sq_quantize_act_table), or form the "
                         "reciprocals of s in every block (sq_quantize_act)")
    ap.add_argument("--ln", action="store_true",
                    help="the QKV and FFN-up inputs are pre-LayerNorm hidden states: their "
                         "quantiser is the fused LayerNorm + quantiser")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-step-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--back-to-back", type=int, default=1000,
                    help="steps launched back to back for the per-call time of the M = 256 "
                         "workloads")
    ap.add_argument("--only-attention", action="store_true",
                    help="measure only sq_attention at the BERT-large layer shape")
    ap.add_argument("--no-configs", action="store_true",
                    help="measure only the chosen workload (no sub-results for the others)")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (small cases for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank, world, local = replicas.rank_world()
    w = wl.WORKLOADS[args.workload]
    if args.layers is not None:
        w = dataclasses.replace(w, layers=max(1, min(args.layers, w.layers)))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(bench_reference(args, w)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    if args.only_attention:
        from smoothquant_w8a8_int8_gb300 import binding as sq
        sq.load()
        if rank == 0:
            print(json.dumps({"attention": bench_attention(args, reps=args.steps)}), flush=True)
        return
    res = bench_ours(args, w, rank, world)
    if not args.no_configs and args.layers is None:
        res["configs"] = other_configs(args, w, rank, world)
        res["attention"] = bench_attention(args)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
