"""Algorithmic work and roofline arithmetic for the linear block.

The byte model is the one behind "Efficient INT8 Inference of Small NLP Models
on Server CPUs with PyTorch Native Stack", Table 5: a GEMM of shape M x K x N
does 2MKN operations and moves each operand once and the output once, with
INT8 operands (1 byte), an int32 output (4 bytes), BF16 operands (2 bytes)
with an fp32 output, or FP32 throughout.  Table 7 estimates a memory-bound
GEMM's throughput as effective bandwidth x arithmetic intensity and averages
over a forward pass as total operations / total time.

For this library's kernels the epilogue operands are added to the INT8 model:
per-token and per-channel scales (4M + 4N), bias (4N), the fp32 output (4MN,
the same count as the int32 output) and, in residual mode, the fp32 residual
(4MN).  The quantiser reads fp32 X and s and writes int8 codes and fp32
per-token scales.
"""
from __future__ import annotations

from typing import Iterable, Tuple

EPI_NONE, EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESIDUAL = 0, 1, 2, 3


def gemm_ops(M: int, K: int, N: int) -> int:
    return 2 * M * K * N


def gemm_bytes(M: int, K: int, N: int, dtype: str = "int8") -> int:
    """Table 5 byte model: operands once, output once."""
    if dtype == "int8":
        return M * K + K * N + 4 * M * N
    if dtype == "bf16":
        return 2 * M * K + 2 * K * N + 4 * M * N
    if dtype == "fp32":
        return 4 * (M * K + K * N + M * N)
    raise ValueError(dtype)


def arithmetic_intensity(M: int, K: int, N: int, dtype: str = "int8") -> float:
    return gemm_ops(M, K, N) / gemm_bytes(M, K, N, dtype)


def linear_bytes(M: int, K: int, N: int, mode: int) -> int:
    """Algorithmic bytes of one fused GEMM + epilogue launch: int8 operands,
    per-token/per-channel fp32 scales, bias, fp32 output, fp32 residual."""
    b = M * K + K * N + 4 * M * N + 4 * M + 4 * N
    if mode != EPI_NONE:
        b += 4 * N
    if mode == EPI_BIAS_RESIDUAL:
        b += 4 * M * N
    return b


def quantize_bytes(M: int, K: int) -> int:
    """Algorithmic bytes of one activation-quantiser launch: fp32 X and s in,
    int8 codes and fp32 per-token scales out."""
    return 4 * M * K + M * K + 4 * M + 4 * K


def estimated_tops(bandwidth_gbs: float, ai: float) -> float:
    """Table 7's memory-bound estimate: bandwidth (GB/s) x AI (ops/B), in TOPS."""
    return bandwidth_gbs * ai / 1000.0


def weighted_tops(shapes: Iterable[Tuple[int, int, int, int, float]]) -> float:
    """Total ops / total time over a forward pass.  Each entry is
    (M, K, N, occurrences, TOPS of that shape)."""
    ops = 0.0
    secs = 0.0
    for M, K, N, occ, tops in shapes:
        o = gemm_ops(M, K, N) * occ
        ops += o
        secs += o / (tops * 1e12)
    return ops / secs / 1e12


def balance_point(peak_tops: float, bandwidth_gbs: float) -> float:
    """Ops per byte at which compute and memory time are equal (Table 4)."""
    return peak_tops * 1e12 / (bandwidth_gbs * 1e9)


def roofline_time_s(ops: float, nbytes: float, peak_tops: float, bandwidth_gbs: float) -> float:
    """The slower of peak compute and bytes at bandwidth."""
    return max(ops / (peak_tops * 1e12), nbytes / (bandwidth_gbs * 1e9))
