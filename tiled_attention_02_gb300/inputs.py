"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws random tensors, so
that the CUDA path and the fp64 oracle see exactly the same bytes.

Recipe: one CPU ``torch.Generator`` seeded with ``seed``; each tensor is drawn
as float32 ``randn`` (i.i.d. N(0, 1)) in a fixed order -- q, k, v, then dO
when asked for -- and rounded to bfloat16.  A block of chained layers draws
q, k, v (and dO) for layer 0, then layer 1, and so on, from one generator.
The oracle widens the bfloat16 values to float exactly.

Shapes too large to draw on the host use the same recipe on a seeded CUDA
generator (``make_qkv_device``): other values than the CPU draw, and the
oracle receives copies of the device bytes it needs.
"""
from __future__ import annotations

import torch


def _draw(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_qkv(B: int, Hq: int, Hkv: int, N: int, D: int, *, seed: int = 0,
             with_do: bool = False, gen: torch.Generator | None = None) -> dict:
    """q [B,Hq,N,D], k and v [B,Hkv,N,D] (and dO like q) as bf16 CPU tensors."""
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    out = {"q": _draw(gen, (B, Hq, N, D)),
           "k": _draw(gen, (B, Hkv, N, D)),
           "v": _draw(gen, (B, Hkv, N, D))}
    if with_do:
        out["do"] = _draw(gen, (B, Hq, N, D))
    return out


def make_qkv_device(B: int, Hq: int, Hkv: int, N: int, D: int, *, seed: int = 0,
                    with_do: bool = False, device: str = "cuda") -> dict:
    """As make_qkv, drawn on the device: q [B,Hq,N,D], k and v [B,Hkv,N,D]
    (and dO like q) as bf16 tensors on ``device``."""
    gen = torch.Generator(device=device).manual_seed(seed)

    def draw(shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32,
                           device=device).to(torch.bfloat16)
    out = {"q": draw((B, Hq, N, D)), "k": draw((B, Hkv, N, D)), "v": draw((B, Hkv, N, D))}
    if with_do:
        out["do"] = draw((B, Hq, N, D))
    return out


def make_decode(B: int, Hq: int, Hkv: int, N: int, D: int, *, seed: int = 0) -> dict:
    """One query row per (batch, query head) and an N-row key/value cache:
    q [B,Hq,D], k and v [B,Hkv,N,D] as bf16 CPU tensors."""
    gen = torch.Generator().manual_seed(seed)
    return {"q": _draw(gen, (B, Hq, D)),
            "k": _draw(gen, (B, Hkv, N, D)),
            "v": _draw(gen, (B, Hkv, N, D))}


def make_chain(B: int, Hq: int, Hkv: int, N: int, D: int, *, layers: int = 4,
               seed: int = 0, with_do: bool = False) -> list[dict]:
    """Per-layer q, k, v for a block of chained layers, one generator."""
    gen = torch.Generator().manual_seed(seed)
    return [make_qkv(B, Hq, Hkv, N, D, gen=gen, with_do=with_do) for _ in range(layers)]


def make_bias(B: int, Hq: int, N: int, *, seed: int = 1, std: float = 1.0) -> torch.Tensor:
    """A float32 [B,Hq,N,N] additive logit bias ~ N(0, std^2), for tests of the
    bias input on its own (the chained block produces its own biases)."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(B, Hq, N, N, generator=gen, dtype=torch.float32) * std


def to_oracle(t: torch.Tensor):
    """Exact widening of a bf16/fp32 CPU tensor to a float32 numpy array."""
    return t.detach().to("cpu").float().numpy()
