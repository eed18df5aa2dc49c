"""Encoder self-attention on the tensor cores (split tf32) against the oracle's
double-precision softmax(Q K^T / sqrt(d)) V, within the fp32 tolerance
max|O - O_ref| <= 1e-5 max|O_ref| + 1e-6 per output tensor.

"Efficient INT8 Inference of Small NLP Models on Server CPUs with PyTorch
Native Stack", Table 3 (attention beside the linear block of BERT-large); the
input layout is the fused QKV projection's output [B*S, 3*H*D].
"""
import numpy as np
import pytest
import torch

import oracle
from paritylib import assert_close_fp32, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def sq():
    from smoothquant_w8a8_int8_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return binding


def _qkv(B, S, H, seed, spread=0.6):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B * S, 3 * H * 64)) * spread).astype(np.float32)


# (B, S, H): several query tiles, a partial last tile (S = 192), the shortest
# and longest sequences, odd head counts
@pytest.mark.parametrize("B,S,H", [(2, 256, 4), (1, 64, 2), (3, 128, 3), (2, 192, 2), (1, 448, 1)])
def test_attention_parity(sq, B, S, H):
    QKV = _qkv(B, S, H, seed=B * 1000 + S + H)
    ref = oracle.attention(QKV, B, S, H, 64)
    got = sq.attention(to_dev(QKV), B, S, H).cpu().numpy()
    assert_close_fp32(got, ref, f"attention B={B} S={S} H={H}")


# More (sequence, head, query tile) units than a GB300 has SMs, so that each
# persistent CTA takes several in turn: an odd number of 64-key chunks with a
# partial last query tile (S = 192), and the longest sequence (S = 448)
@pytest.mark.parametrize("B,S,H", [(4, 192, 40), (2, 448, 24)])
def test_attention_several_units_per_cta(sq, B, S, H):
    QKV = _qkv(B, S, H, seed=B + S + H)
    ref = oracle.attention(QKV, B, S, H, 64)
    got = sq.attention(to_dev(QKV), B, S, H).cpu().numpy()
    assert sq.device_status() == sq.SQ_OK
    assert_close_fp32(got, ref, f"attention B={B} S={S} H={H}")


@pytest.mark.parametrize("spread", [0.05, 2.0, 4.0])
def test_attention_logit_scales(sq, spread):
    """Nearly uniform weights (small logits) and peaked ones (large logits,
    most exp() terms far below the row maximum)."""
    B, S, H = 2, 256, 2
    QKV = _qkv(B, S, H, seed=int(spread * 100), spread=spread)
    ref = oracle.attention(QKV, B, S, H, 64)
    got = sq.attention(to_dev(QKV), B, S, H).cpu().numpy()
    assert_close_fp32(got, ref, f"spread {spread}")


def test_attention_zero_queries_give_mean_of_values(sq):
    B, S, H = 1, 128, 2
    QKV = _qkv(B, S, H, seed=3)
    QKV[:, : H * 64] = 0.0                      # all queries zero: uniform weights
    got = sq.attention(to_dev(QKV), B, S, H).cpu().numpy()
    V = QKV[:, 2 * H * 64:]
    want = np.broadcast_to(V.astype(np.float64).mean(axis=0), (S, H * 64))
    assert_close_fp32(got, want, "mean of V")


def test_attention_bert_large_sampled(sq):
    """The BERT-large layer shape (batch 32, sequence 256, 16 heads) on the GPU,
    three sequences checked against the oracle."""
    B, S, H = 32, 256, 16
    QKV = _qkv(B, S, H, seed=77)
    got = sq.attention(to_dev(QKV), B, S, H).cpu().numpy()
    assert sq.device_status() == sq.SQ_OK
    for b in (0, 17, 31):
        rows = slice(b * S, (b + 1) * S)
        ref = oracle.attention(QKV[rows], 1, S, H, 64)
        assert_close_fp32(got[rows], ref, f"sequence {b}")
