"""Seeded synthetic inputs of Maple-Preview's shapes.

This module only draws random numbers: it holds none of the ternary method's
arithmetic.  Both the CUDA path and the CPU oracle receive the tensors it makes.

Recipe (the pages measure on no dataset at kernel level, so everything is synthetic):
  * expert weights: fp32 N(0, 0.02) cast to bf16 with round-to-nearest-even,
    gate/up [E, I, H], down [E, H, I];
  * router weights: bf16 [E, H], same distribution;
  * activations: bf16 N(0, 1) [T, H];
  * router bias: N(0, 0.5) per expert (mildly skewed decode batches), or a Zipf
    ranking -gamma * s * ln(rank) over a seeded permutation of the experts
    (prefill with loads from ~0 to several hundred tokens).
Every tensor is drawn from its own torch.Generator seeded from (seed, tag), on the
device it is requested on; the same call on the same device type gives the same
values.
"""
from __future__ import annotations

import numpy as np
import torch

_TAGS = {"gate": 1, "up": 2, "down": 3, "router": 4, "tokens": 5, "bias": 6, "perm": 7,
         "laplace": 8, "misc": 9}


def _gen(seed: int, tag: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1000003 + _TAGS[tag] * 7919) % (2**63 - 1))
    return g


def bf16_normal(shape, std: float, seed: int, tag: str = "misc", device="cpu") -> torch.Tensor:
    """fp32 N(0, std) drawn with a seeded generator, then cast to bf16 (RNE)."""
    g = _gen(seed, tag, device)
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(
        torch.bfloat16)


def expert_weights(E: int, H: int, I: int, seed: int, device="cpu", std: float = 0.02):
    """bf16 gate [E,I,H], up [E,I,H], down [E,H,I] for one MoE layer."""
    return {
        "gate": bf16_normal((E, I, H), std, seed, "gate", device),
        "up": bf16_normal((E, I, H), std, seed, "up", device),
        "down": bf16_normal((E, H, I), std, seed, "down", device),
    }


def router_weights(E: int, H: int, seed: int, device="cpu", std: float = 0.02) -> torch.Tensor:
    return bf16_normal((E, H), std, seed, "router", device)


def tokens(T: int, H: int, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    return bf16_normal((T, H), std, seed, "tokens", device)


def bias_normal(E: int, seed: int, std: float = 0.5) -> torch.Tensor:
    """fp32 per-expert router bias ~ N(0, std) (drawn on the CPU)."""
    g = _gen(seed, "bias", "cpu")
    return torch.randn(E, generator=g, dtype=torch.float32) * std


def bias_zipf(E: int, seed: int, s: float = 1.1, gamma: float = 1.0) -> torch.Tensor:
    """fp32 bias_e = -gamma * s * ln(rank_e), ranks 1..E over a seeded permutation."""
    g = _gen(seed, "perm", "cpu")
    perm = torch.randperm(E, generator=g)
    rank = torch.empty(E, dtype=torch.float64)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64)
    return (-gamma * s * torch.log(rank)).to(torch.float32)


def laplace_bf16(shape, scale: float, seed: int) -> torch.Tensor:
    """bf16 rows with a Laplace(0, scale) distribution (heavier tails than Gaussian)."""
    g = _gen(seed, "laplace", "cpu")
    u = torch.rand(*shape, generator=g, dtype=torch.float64) - 0.5
    v = -scale * torch.sign(u) * torch.log1p(-2.0 * u.abs())
    return v.to(torch.float32).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_float(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact fp32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)

