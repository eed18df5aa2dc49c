"""The library's launches (programmatic dependent launch, CTA-pair clusters,
split-K on a caller workspace) captured in a CUDA graph: replays on new input
data equal eager calls bit for bit.  Each entry point is called once eagerly
first, so that the one-time per-device set-up (function attributes, cluster
occupancy, tensor-map encoder) happens outside the capture.  The step runs the
quantiser from s's division table, both GEMM schedules and the attention
kernel."""
import pytest
import torch

from smoothquant_w8a8_int8_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


def test_step_captured_in_graph(sq):
    M, K, N = 1024, 1024, 3072          # pair kernel
    Ms, Ks, Ns = 256, 4096, 1024        # split-K on the workspace
    dev = torch.device("cuda")
    c = wl.make_case(M, K, N, wl.EPI_BIAS_GELU, seed=21, device=dev)
    cs = wl.make_case(Ms, Ks, Ns, wl.EPI_BIAS_RESIDUAL, seed=22, device=dev)
    s = sq.smooth_factor(sq.channel_absmax(c.X), sq.channel_absmax(c.W), 0.5)
    ss = sq.smooth_factor(sq.channel_absmax(cs.X), sq.channel_absmax(cs.W), 0.5)
    _, sw, Wop = sq.pack_weight(c.W, s, want_q=False)
    _, sws, Wops = sq.pack_weight(cs.W, ss, want_q=False)
    ws = sq.empty_workspace(sq.linear_workspace_bytes(Ms, Ns, Ks))
    X = c.X.clone()
    Xs = cs.X.clone()
    sx = torch.empty(M, device=dev)
    Xop = sq.empty_operand(M, K)
    sxs = torch.empty(Ms, device=dev)
    Xops = sq.empty_operand(Ms, Ks)
    Y = torch.empty(M, N, device=dev)
    Ys = torch.empty(Ms, Ns, device=dev)
    table = sq.division_table(s)
    QKV = torch.randn(2 * 128, 3 * 4 * 64, device=dev)
    O = torch.empty(2 * 128, 4 * 64, device=dev)

    def step():
        sq.quantize_act_table(X, s, table, out=(None, sx, Xop))
        sq.linear_i8(Xop, sx, Wop, sw, c.bias, None, wl.EPI_BIAS_GELU, out=Y)
        sq.quantize_act(Xs, ss, out=(None, sxs, Xops))
        sq.linear_i8_ws(Xops, sxs, Wops, sws, cs.bias, cs.residual, wl.EPI_BIAS_RESIDUAL, out=Ys,
                        workspace=ws)
        sq.attention(QKV, 2, 128, 4, 64, out=O)

    step()  # eager, outside capture: one-time set-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (31, 32):
        gen = torch.Generator(device=dev).manual_seed(seed)
        X.copy_(torch.randn(M, K, generator=gen, device=dev))
        Xs.copy_(torch.randn(Ms, Ks, generator=gen, device=dev))
        QKV.copy_(torch.randn(QKV.shape, generator=gen, device=dev))
        g.replay()
        torch.cuda.synchronize()
        Yg, Ysg, Og = Y.clone(), Ys.clone(), O.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(Yg, Y), f"pair GEMM, seed {seed}"
        assert torch.equal(Ysg, Ys), f"split-K GEMM, seed {seed}"
        assert torch.equal(Og, O), f"attention, seed {seed}"
    assert sq.device_status() == sq.SQ_OK
