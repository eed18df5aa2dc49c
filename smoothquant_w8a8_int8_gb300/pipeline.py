"""Running a sequence of SmoothQuant linear layers on activations that live in
host memory.

`HostLinearPipeline` marshals the layers for the C-ABI call
sq_linear_block_host, which streams each layer's activations X (fp32, pinned
host memory) to the GPU, runs the linear block there (the layer's quantiser,
then sq_linear_i8 with its fused epilogue) and streams Y back, with the three
kinds of work on three CUDA streams and two device slots for X and for Y in
one scratch buffer, so that the host-to-device copy of layer i+1 and the
device-to-host copy of layer i-1 overlap the kernels of layer i.  Packed
weights, scales, bias and residual stay resident on the device.  The copies,
the events that order them and every kernel are the library's; this module
only builds the layer table and owns the scratch and the streams.
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


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


class HostLinearPipeline:
    def __init__(self, M: int, max_K: int, max_N: int, device="cuda"):
        dev = torch.device(device)
        self.M = M
        self.dev = dev
        nbytes = sq.linear_block_host_scratch_bytes(M, max_K, max_N)
        self.scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        # the device slots inside the scratch (layout of sq_linear_block_host_scratch_bytes)
        r256 = lambda n: (n + 255) // 256 * 256
        xs, ys = r256(M * max_K * 4), r256(M * max_N * 4)
        self.x_slots = [self.scratch[k * xs: k * xs + M * max_K * 4].view(torch.float32)
                        for k in range(2)]
        self.y_slots = [self.scratch[2 * xs + k * ys: 2 * xs + k * ys + M * max_N * 4]
                        .view(torch.float32) for k in range(2)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.comp = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)

    def run(self, layers: Sequence[LinearLayer], X_host: Sequence[torch.Tensor],
            Y_host: Sequence[torch.Tensor]) -> None:
        """Y_host[i] = linear_block(layers[i], X_host[i]) for every i.  Host
        tensors must be pinned and contiguous.  Returns once every copy has
        been enqueued; call torch.cuda.synchronize() (or wait on the
        device-to-host stream) before reading Y_host."""
        table = []
        for L, Xh, Yh in zip(layers, X_host, Y_host):
            static = L.static_scale is not None
            table.append(sq.LinearLayerC(
                Xh.shape[1], Yh.shape[1], int(L.mode), float(L.static_scale) if static else 0.0,
                _ptr(L.s), None if static else _ptr(L.s_table), _ptr(L.Wop), _ptr(L.w_scale),
                _ptr(L.w_l1), _ptr(L.bias), _ptr(L.residual)))
        cur = torch.cuda.current_stream(self.dev)
        for st in (self.h2d, self.comp, self.d2h):
            st.wait_stream(cur)
        sq.linear_block_host(table, self.M, X_host, Y_host, self.scratch,
                             (self.h2d, self.comp, self.d2h))
        cur.wait_stream(self.d2h)
