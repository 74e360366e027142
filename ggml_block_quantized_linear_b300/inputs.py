"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds random-number recipes only (no quantization, no matmul).
The weights stand in for the Gemma 4 checkpoints that the mistral.rs README
benchmarks (section "Benchmarks"); those models are not available here.

* weights: fp32 ~ N(0, 0.02); an independent Bernoulli(0.001) mask multiplies
  0.1 % of the entries by 20 (outliers); then rounded to bf16 (RNE) unless the
  fp32 source is asked for.
* activations: bf16 ~ N(0, 1).

Every draw uses ``torch.Generator`` seeded explicitly; ``device`` selects the
generator's device (a CUDA generator gives a different, still deterministic,
stream than the CPU one).
"""
from __future__ import annotations

import hashlib

import torch

WEIGHT_STD = 0.02
OUTLIER_P = 0.001
OUTLIER_SCALE = 20.0

# Decode / prefill shapes (N x K) of an 8B-class decoder: q/o projection,
# k/v projection, gate/up projection, down projection.
DECODE_SHAPES = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]
DECODE_MS = [1, 4, 16]
PREFILL_SHAPES = [(4096, 4096), (14336, 4096), (4096, 14336)]
PREFILL_MS = [512, 2048]
# mid-size batches (continuous batching between decode and prefill)
MID_MS = [32, 128]
# output head / token embedding of the 8B-shape decoder: vocabulary x hidden
VOCAB = 128256

# Synthetic 8B-shape decoder: 32 layers, hidden 4096, 32 q heads / 8 kv heads
# of 128, MLP 14336.  (name, N, K) per linear, in forward order.
MODEL_LAYERS = 32
MODEL_LINEARS = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096),
                 ("o", 4096, 4096), ("gate", 14336, 4096), ("up", 14336, 4096),
                 ("down", 4096, 14336)]


def seed_for(config: int, shape_index: int = 0, m_index: int = 0) -> int:
    return 1000 * config + 10 * shape_index + m_index


def model_weight_seed(layer: int, linear_index: int) -> int:
    """Seed of linear ``linear_index`` (MODEL_LINEARS order) of model layer ``layer``."""
    return 50000 + 10 * layer + linear_index


def model_activation_seed(layer: int, linear_index: int) -> int:
    return 60000 + 10 * layer + linear_index


def weights(n: int, k: int, seed: int, device="cpu", fp32: bool = False) -> torch.Tensor:
    """W[n x k]: N(0, 0.02) with 0.1 % outliers x20; bf16 unless ``fp32``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
    w.mul_(WEIGHT_STD)
    mask = torch.rand((n, k), generator=g, device=device, dtype=torch.float32) < OUTLIER_P
    w = torch.where(mask, w * OUTLIER_SCALE, w)
    if fp32:
        return w.contiguous()
    return w.to(torch.bfloat16).contiguous()


def activations(m: int, k: int, seed: int, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed + 7919)
    return torch.randn((m, k), generator=g, device=device, dtype=torch.float32).to(
        torch.bfloat16).contiguous()


def digest(t: torch.Tensor) -> str:
    """SHA-256 (first 16 hex digits) of a tensor's bytes, for the bench record."""
    b = t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes()
    return hashlib.sha256(b).hexdigest()[:16]


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
