"""Running a sequence of SmoothQuant linear layers on activations that live in
host memory.

`HostLinearPipeline` streams each layer's activations X (fp32, pinned host
memory) to the GPU, runs the linear block there (sq_quantize_act, or
sq_quantize_act_table when the layer carries s's division table, then
sq_linear_i8 with its fused epilogue) and streams Y back, with the three kinds
of work on three CUDA streams and two device slots for X and for Y, so that
the host-to-device copy of layer i+1 and the device-to-host copy of layer i-1
overlap the kernels of layer i.  Packed weights, scales, bias and residual
stay resident on the device.  Every step of the block runs in the C-ABI
library's kernels; this module only orders copies and launches.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

from . import binding as sq


@dataclasses.dataclass
class LinearLayer:
    """One packed linear layer (device tensors) and its host activations."""
    s: torch.Tensor                     # smoothing factor [K] fp32
    Wop: torch.Tensor                   # packed weight operand [N, K] (bf16 codes)
    w_scale: torch.Tensor               # [N] fp32
    mode: int                           # epilogue mode
    bias: Optional[torch.Tensor] = None
    residual: Optional[torch.Tensor] = None   # [M, N] fp32, device
    w_l1: Optional[torch.Tensor] = None       # [N] int32 row L1 norms of the codes
    static_scale: Optional[float] = None      # Smooth-Static per-tensor scale, else dynamic
    s_table: Optional[torch.Tensor] = None    # [K, 2] division table of s (dynamic only)


class HostLinearPipeline:
    def __init__(self, M: int, max_K: int, max_N: int, device="cuda", slots: int = 2):
        dev = torch.device(device)
        self.M = M
        self.dev = dev
        self.nslots = slots
        self.x_slots = [torch.empty(M * max_K, dtype=torch.float32, device=dev)
                        for _ in range(slots)]
        self.y_slots = [torch.empty(M * max_N, dtype=torch.float32, device=dev)
                        for _ in range(slots)]
        self.xop = torch.empty(M * max_K, dtype=torch.bfloat16, device=dev)
        self.sx = torch.empty(M, dtype=torch.float32, device=dev)
        self.h2d = torch.cuda.Stream(device=dev)
        self.comp = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)

    def run(self, layers: Sequence[LinearLayer], X_host: Sequence[torch.Tensor],
            Y_host: Sequence[torch.Tensor]) -> None:
        """Y_host[i] = linear_block(layers[i], X_host[i]) for every i.  Host
        tensors must be pinned and contiguous.  Returns once every copy has
        been enqueued; call torch.cuda.synchronize() (or wait on the
        device-to-host stream) before reading Y_host."""
        M = self.M
        n = len(layers)
        x_ready = [torch.cuda.Event() for _ in range(n)]
        y_ready = [torch.cuda.Event() for _ in range(n)]
        x_free = [None] * self.nslots
        y_free = [None] * self.nslots
        cur = torch.cuda.current_stream(self.dev)
        for st in (self.h2d, self.comp, self.d2h):
            st.wait_stream(cur)
        for i, (L, Xh, Yh) in enumerate(zip(layers, X_host, Y_host)):
            K = Xh.shape[1]
            N = Yh.shape[1]
            slot = i % self.nslots
            dX = self.x_slots[slot][: M * K].view(M, K)
            dY = self.y_slots[slot][: M * N].view(M, N)
            # host -> device
            with torch.cuda.stream(self.h2d):
                if x_free[slot] is not None:
                    self.h2d.wait_event(x_free[slot])
                dX.copy_(Xh, non_blocking=True)
                x_ready[i].record(self.h2d)
            # the linear block
            with torch.cuda.stream(self.comp):
                self.comp.wait_event(x_ready[i])
                if y_free[slot] is not None:
                    self.comp.wait_event(y_free[slot])
                xop = self.xop[: M * K].view(M, K)
                if L.static_scale is not None:
                    sq.quantize_act_static(dX, L.s, L.static_scale, out=(None, self.sx, xop),
                                           stream=self.comp)
                elif L.s_table is not None:
                    sq.quantize_act_table(dX, L.s, L.s_table, out=(None, self.sx, xop),
                                          stream=self.comp)
                else:
                    sq.quantize_act(dX, L.s, out=(None, self.sx, xop), stream=self.comp)
                ev = torch.cuda.Event()
                ev.record(self.comp)
                x_free[slot] = ev
                sq.linear_i8(xop, self.sx, L.Wop, L.w_scale, L.bias, L.residual, L.mode, out=dY,
                             w_l1=L.w_l1, stream=self.comp)
                y_ready[i].record(self.comp)
            # device -> host
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(y_ready[i])
                Yh.copy_(dY, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(self.d2h)
                y_free[slot] = ev
        cur.wait_stream(self.d2h)
