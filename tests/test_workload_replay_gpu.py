"""Every linear of the five workloads, replayed exactly as the benchmark
runs it (inputs drawn on the device from the same seeds, smoothing factor and
packing on the GPU, sq_quantize_act to the bf16 operand, sq_linear_i8 with the
packed weights' row L1 norms -- through sq_linear_i8_ws on a workspace where
the shape splits K, as the benchmark's default schedule does), against the
oracle:

  * smoothing factor, weight codes and weight-scale bits: all channels/rows;
  * activation codes and per-token scale bits: ALL M rows;
  * raw int32 sums: a seeded sample of rows, bit for bit;
  * fp32 outputs of the linear's epilogue: the same rows, within
    max|err| <= 1e-5 max|ref| + 1e-6.

Workloads: the three single BERT-large linears at batch 1 x seq 256 (QKV
slice, FFN up + GELU, FFN down + residual; every row is checked), the
BERT-large encoder sweep (batch 32 x seq 256, M = 8192, 24
layers x {QKV, out-proj, FFN up + GELU, FFN down + residual}) and the
768-hidden encoder shapes at M = 32768 ("Efficient INT8 Inference of Small NLP
Models on Server CPUs with PyTorch Native Stack", Tables 5 and 8).
"""
import numpy as np
import pytest
import torch

import oracle
from paritylib import assert_close_fp32, assert_codes_equal
from smoothquant_w8a8_int8_gb300 import replicas
from smoothquant_w8a8_int8_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SAMPLE_ROWS = 48


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


def _codes_of_op(op):
    """bf16 operand holding integer codes -> int8 (on the device)."""
    f = op.float()
    assert bool(torch.all(f == torch.round(f))) and float(f.abs().max()) <= 127
    return f.to(torch.int8)


def _mismatches(got_dev, ref_np):
    ref = torch.from_numpy(np.ascontiguousarray(ref_np)).to(got_dev.device)
    return int((got_dev != ref).sum())


def _replay(sq, w, layer, idx):
    lin = w.linears[idx]
    dev = torch.device("cuda")
    seed = replicas.rank_seed(wl.gemm_seed(w, layer, idx), 0)
    c = wl.make_case(w.M, lin.K, lin.N, lin.mode, seed, w.outlier_frac, w.outlier_scale,
                     lin.gelu_input, w.alpha, device=dev)
    # the benchmark's calls
    s = sq.smooth_factor(sq.channel_absmax(c.X), sq.channel_absmax(c.W), w.alpha)
    _, sw, Wop, wl1 = sq.pack_weight(c.W, s, want_q=False, want_l1=True)
    sx = torch.empty(w.M, dtype=torch.float32, device=dev)
    Xop = torch.empty(w.M, lin.K, dtype=torch.bfloat16, device=dev)
    sq.quantize_act(c.X, s, out=(None, sx, Xop))
    Y = torch.empty(w.M, lin.N, dtype=torch.float32, device=dev)
    need = sq.linear_workspace_bytes(w.M, lin.N, lin.K)
    if need > 0:
        ws = sq.empty_workspace(need)
        sq.linear_i8_ws(Xop, sx, Wop, sw, c.bias, c.residual, lin.mode, out=Y, w_l1=wl1,
                        workspace=ws)
        acc = sq.linear_i8_ws(Xop, None, Wop, None, None, None, sq.EPI_RAW_I32, w_l1=wl1,
                              workspace=ws)
    else:
        sq.linear_i8(Xop, sx, Wop, sw, c.bias, c.residual, lin.mode, out=Y, w_l1=wl1)
        acc = sq.linear_i8(Xop, None, Wop, None, None, None, sq.EPI_RAW_I32, w_l1=wl1)
    assert sq.device_status() == sq.SQ_OK

    X, W = c.X.cpu().numpy(), c.W.cpu().numpy()
    s_ref = oracle.smooth_factor(oracle.channel_absmax(X), oracle.channel_absmax(W), w.alpha)
    what = f"{w.name} layer {layer} {lin.name}"
    # alpha = 0.5: the smoothing factor is bit-exact (one double sqrt / pow)
    assert_codes_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32), f"{what}: s")
    wq, sw_ref = oracle.quantize_rows(W, s_ref, "weight")
    assert _mismatches(_codes_of_op(Wop), wq) == 0, f"{what}: weight codes"
    assert _mismatches(sw.view(torch.int32), sw_ref.view(np.int32)) == 0, f"{what}: w_scale"
    xq, sx_ref = oracle.quantize_rows(X, s_ref, "act")
    assert _mismatches(_codes_of_op(Xop), xq) == 0, f"{what}: activation codes (all rows)"
    assert _mismatches(sx.view(torch.int32), sx_ref.view(np.int32)) == 0, \
        f"{what}: x_scale bits (all rows)"
    # the single-pass exactness argument applies to these weights (K > 1024)
    if lin.K > 1024:
        assert int(wl1.max()) <= 132104
    rng = np.random.default_rng(1000 * layer + idx)
    rows = np.arange(w.M) if w.M <= 256 else np.unique(
        np.concatenate([[0, w.M - 1], rng.choice(w.M, SAMPLE_ROWS - 2, replace=False)]))
    acc_ref = oracle.gemm_i32(xq[rows], wq)
    ridx = torch.from_numpy(rows).to(dev)
    assert_codes_equal(acc[ridx].cpu().numpy(), acc_ref, f"{what}: int32 sums (sampled rows)")
    b = None if c.bias is None else c.bias.cpu().numpy()
    r = None if c.residual is None else c.residual[ridx].cpu().numpy()
    y_ref = oracle.epilogue(acc_ref, sx_ref[rows], sw_ref, b, r, lin.mode)
    assert_close_fp32(Y[ridx].cpu().numpy(), y_ref, f"{what}: Y (sampled rows)")


@pytest.mark.parametrize("name", ["bert_large_qkv_slice_m256", "bert_large_ffn_up_m256",
                                  "bert_large_ffn_down_m256"])
def test_single_linear_replay(sq, name):
    _replay(sq, wl.WORKLOADS[name], 0, 0)


@pytest.mark.parametrize("layer", range(24))
def test_bert_large_encoder_replay(sq, layer):
    w = wl.WORKLOADS["bert_large_encoder_b32_s256"]
    for idx in range(len(w.linears)):
        _replay(sq, w, layer, idx)


@pytest.mark.parametrize("idx", range(4))
def test_xlmr_base_replay(sq, idx):
    _replay(sq, wl.WORKLOADS["xlmr_base_b64_s512"], 0, idx)
