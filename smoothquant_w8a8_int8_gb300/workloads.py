"""Seeded synthetic inputs for the SmoothQuant W8A8 linear block.

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic (no smoothing, quantisation, GEMM or epilogue).  Both the
CUDA path's tests/benchmark and the CPU oracle's tests take their inputs from
here.

The shapes are the BERT-family encoder linears that "Efficient INT8 Inference
of Small NLP Models on Server CPUs with PyTorch Native Stack" analyses
(Table 5: the three BERT-large GEMM shapes at batch 1, sequence 256; Table 8:
BERT-large, DistilBERT, XLM-RoBERTa).  No dataset or checkpoint is used:

  X ~ N(0, 1) tokens x in-features, with a fraction of input channels scaled
      up as activation outliers (the outlier structure SmoothQuant targets);
  W ~ N(0, 0.02) out-features x in-features (nn.Linear layout);
  bias ~ N(0, 0.02);  residual ~ N(0, 1).

The FFN down-projection's input is drawn as GELU(Z), Z ~ N(0, 1) (the
distribution an FFN up-projection emits), with the same outlier scaling.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

# Epilogue modes, by name (numbering matches the C-ABI enum).
EPI_NONE, EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESIDUAL = 0, 1, 2, 3
EPI_NAMES = {EPI_NONE: "none", EPI_BIAS: "bias", EPI_BIAS_GELU: "bias_gelu",
             EPI_BIAS_RESIDUAL: "bias_residual"}


@dataclasses.dataclass(frozen=True)
class Linear:
    """One linear layer of the block: Y[M,N] = epi(X[M,K] W[N,K]^T)."""
    name: str
    K: int
    N: int
    mode: int
    gelu_input: bool = False  # X drawn as GELU(Z) (FFN down-projection input)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    layers: int
    linears: tuple
    outlier_frac: float
    outlier_scale: float
    seed: int
    alpha: float = 0.5
    description: str = ""

    def gemms(self):
        """(layer, Linear) for every GEMM of one forward pass."""
        return [(l, lin) for l in range(self.layers) for lin in self.linears]

    def ops(self) -> int:
        """Integer multiply-add operations x 2 of one forward pass."""
        return sum(2 * self.M * lin.N * lin.K for _, lin in self.gemms())


_BERT_LARGE = (
    Linear("qkv", 1024, 3072, EPI_BIAS),
    Linear("attn_out", 1024, 1024, EPI_BIAS),
    Linear("ffn_up", 1024, 4096, EPI_BIAS_GELU),
    Linear("ffn_down", 4096, 1024, EPI_BIAS_RESIDUAL, gelu_input=True),
)
_BASE_768 = (
    Linear("qkv", 768, 2304, EPI_BIAS),
    Linear("attn_out", 768, 768, EPI_BIAS),
    Linear("ffn_up", 768, 3072, EPI_BIAS_GELU),
    Linear("ffn_down", 3072, 768, EPI_BIAS_RESIDUAL, gelu_input=True),
)

WORKLOADS = {
    "bert_large_qkv_slice_m256": Workload(
        "bert_large_qkv_slice_m256", 256, 1,
        (Linear("linear", 1024, 1024, EPI_BIAS),), 0.01, 20.0, 1234,
        description="single linear 256x1024 -> 1024, bias (BERT-large, batch 1, seq 256)"),
    "bert_large_ffn_up_m256": Workload(
        "bert_large_ffn_up_m256", 256, 1,
        (Linear("ffn_up", 1024, 4096, EPI_BIAS_GELU),), 0.01, 20.0, 1235,
        description="FFN up-projection 256x1024 -> 4096, bias + GELU(erf)"),
    "bert_large_ffn_down_m256": Workload(
        "bert_large_ffn_down_m256", 256, 1,
        (Linear("ffn_down", 4096, 1024, EPI_BIAS_RESIDUAL, gelu_input=True),), 0.01, 20.0,
        1236, description="FFN down-projection 256x4096 -> 1024, bias + residual"),
    "bert_large_encoder_b32_s256": Workload(
        "bert_large_encoder_b32_s256", 8192, 24, _BERT_LARGE, 0.01, 20.0, 1237,
        description="BERT-large, 24 layers x {QKV, out-proj, FFN up, FFN down}, "
                    "batch 32 x seq 256 (M=8192)"),
    "xlmr_base_b64_s512": Workload(
        "xlmr_base_b64_s512", 32768, 1, _BASE_768, 0.005, 30.0, 1238,
        description="hidden 768 / FFN 3072 encoder linears at batch 64 x seq 512 (M=32768)"),
}
WORKLOAD_ORDER = list(WORKLOADS)


def outlier_channels(K: int, frac: float, gen: torch.Generator) -> torch.Tensor:
    """round(frac*K) distinct channels chosen by a seeded permutation."""
    n = int(math.floor(frac * K + 0.5))
    perm = torch.randperm(K, generator=gen, device=gen.device)
    return perm[:n]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gemm_seed(w: Workload, layer: int, index: int) -> int:
    return w.seed * 1000 + layer * 16 + index


def make_activation(M: int, K: int, seed: int, outlier_frac: float, outlier_scale: float,
                    gelu_input: bool = False, device="cpu",
                    channel_seed: Optional[int] = None) -> torch.Tensor:
    """X [M, K] fp32: N(0,1) (or GELU(Z)), outlier channels multiplied.  The
    outlier channels come from `channel_seed` (default: `seed`) alone, so a
    calibration batch drawn with another seed but the same channel seed has
    the same outlier channels."""
    ch = outlier_channels(K, outlier_frac, _gen(seed if channel_seed is None else channel_seed,
                                                 device))
    g = _gen(seed, device)
    X = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    if gelu_input:
        X = 0.5 * X * (1.0 + torch.erf(X * (1.0 / math.sqrt(2.0))))
    if ch.numel():
        X[:, ch] *= outlier_scale
    return X.contiguous()


def make_weight(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed + 7919, device)
    return (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * 0.02).contiguous()


def make_bias(N: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed + 104729, device)
    return (torch.randn(N, generator=g, device=device, dtype=torch.float32) * 0.02).contiguous()


def make_residual(M: int, N: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed + 1299709, device)
    return torch.randn(M, N, generator=g, device=device, dtype=torch.float32).contiguous()


@dataclasses.dataclass
class LinearCase:
    X: torch.Tensor
    W: torch.Tensor
    bias: Optional[torch.Tensor]
    residual: Optional[torch.Tensor]
    mode: int
    alpha: float

    @property
    def shape(self):
        return self.X.shape[0], self.X.shape[1], self.W.shape[0]


def make_case(M: int, K: int, N: int, mode: int, seed: int, outlier_frac: float = 0.01,
              outlier_scale: float = 20.0, gelu_input: bool = False, alpha: float = 0.5,
              device="cpu") -> LinearCase:
    """One linear layer's inputs, drawn from the recipe above."""
    X = make_activation(M, K, seed, outlier_frac, outlier_scale, gelu_input, device)
    W = make_weight(N, K, seed, device)
    bias = make_bias(N, seed, device) if mode != EPI_NONE else None
    residual = make_residual(M, N, seed, device) if mode == EPI_BIAS_RESIDUAL else None
    return LinearCase(X, W, bias, residual, mode, alpha)


def workload_case(w: Workload, layer: int, index: int, rows: Optional[int] = None,
                  device="cpu") -> LinearCase:
    """Inputs of GEMM `index` of layer `layer` of a workload.  `rows` draws a
    shorter M (same recipe) for bounded samples."""
    lin = w.linears[index]
    M = w.M if rows is None else rows
    return make_case(M, lin.K, lin.N, lin.mode, gemm_seed(w, layer, index),
                     w.outlier_frac, w.outlier_scale, lin.gelu_input, w.alpha, device)


def all_cases(w: Workload, device="cpu") -> List[LinearCase]:
    return [workload_case(w, l, i, device=device)
            for l in range(w.layers) for i in range(len(w.linears))]
