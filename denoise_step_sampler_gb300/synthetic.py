"""Seeded synthetic inputs (logits, embeddings, temperatures).

These stand in for decoder logits, which need a trained model: Gaussian
logits with one boosted "true" token per position, so that entropies range
from near uniform to near one-hot as the boost grows.  The module holds none
of the sampler's arithmetic; it only draws inputs with torch's seeded
generators, on whatever device it is asked for, so the GPU path and the CPU
oracle read the very same tensors (the oracle gets a host copy).

Workloads (sizes as in the library's benchmark):
* fp32 logits z = 2 * N(0,1) plus U[0, boost_hi) on one uniform token per
  position (e.g. 1 x 256 positions, V = 50257, boost_hi = 12);
* bf16 logits, same recipe, boost_hi = 16, V = 262144;
* multi-step loops: at step s of request r, z = 2 * N(0,1) with the true
  token of (r, i) -- fixed across steps -- boosted by 2 + 0.5 s;
* E ~ N(0, 0.02^2) in bf16, [V, d];
* temperatures U[0.6, 1.2] per request.
"""

from __future__ import annotations

import torch

_MIX = 0x9E3779B97F4A7C15


def _seed(*parts: int) -> int:
    """Fold integers into a 63-bit generator seed (a plain polynomial fold,
    only used to give each (seed, request, step) its own torch generator)."""
    h = 0x243F6A8885A308D3
    for p in parts:
        h = (h * 6364136223846793005 + (int(p) & 0xFFFFFFFFFFFFFFFF) + 1442695040888963407) % (1 << 64)
        h ^= h >> 29
    return h & 0x7FFFFFFFFFFFFFFF


def generator(device, *parts: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def boosted_logits(n_pos: int, V: int, *, seed: int, dtype=torch.bfloat16,
                   device="cpu", boost_hi: float = 16.0, ld: int | None = None,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """[n_pos, ld] logits (columns >= V are padding, left as zero).

    z = 2 * N(0,1) in fp32, plus U[0, boost_hi) on one uniform token per row,
    then rounded to ``dtype``.  Generated in slabs of rows to bound temporary
    memory.
    """
    ld = V if ld is None else ld
    if out is None:
        out = torch.zeros((n_pos, ld), dtype=dtype, device=device)
    g = generator(device, seed, 1)
    slab = max(1, (1 << 26) // max(V, 1))
    for r0 in range(0, n_pos, slab):
        r1 = min(n_pos, r0 + slab)
        z = torch.randn((r1 - r0, V), generator=g, device=device, dtype=torch.float32)
        z.mul_(2.0)
        tok = torch.randint(0, V, (r1 - r0, 1), generator=g, device=device)
        boost = torch.rand((r1 - r0, 1), generator=g, device=device) * boost_hi
        z.scatter_add_(1, tok, boost)
        out[r0:r1, :V] = z.to(dtype)
    return out


def true_tokens(n_pos: int, V: int, *, seed: int, request: int, device="cpu") -> torch.Tensor:
    g = generator(device, seed, 2, request)
    return torch.randint(0, V, (n_pos,), generator=g, device=device)


def loop_logits(C: int, V: int, *, seed: int, request: int, step: int,
                dtype=torch.bfloat16, device="cpu", out: torch.Tensor | None = None,
                boost_base: float = 2.0, boost_slope: float = 0.5) -> torch.Tensor:
    """[C, V] logits of request ``request`` at loop step ``step``: fresh
    2 * N(0,1) noise from (seed, request, step) and the request's fixed true
    tokens boosted by boost_base + boost_slope * step, so confidence rises."""
    if out is None:
        out = torch.empty((C, V), dtype=dtype, device=device)
    g = generator(device, seed, 3, request, step)
    z = torch.randn((C, V), generator=g, device=device, dtype=torch.float32)
    z.mul_(2.0)
    tok = true_tokens(C, V, seed=seed, request=request, device=device).view(C, 1)
    z.scatter_add_(1, tok, torch.full((C, 1), boost_base + boost_slope * step, device=device))
    out.copy_(z.to(dtype))
    return out


def embedding(V: int, d: int, *, seed: int, device="cpu", std: float = 0.02) -> torch.Tensor:
    """E ~ N(0, std^2), [V, d] bf16, generated in row slabs."""
    out = torch.empty((V, d), dtype=torch.bfloat16, device=device)
    g = generator(device, seed, 4)
    slab = max(1, (1 << 26) // max(d, 1))
    for r0 in range(0, V, slab):
        r1 = min(V, r0 + slab)
        out[r0:r1] = (torch.randn((r1 - r0, d), generator=g, device=device) * std).to(torch.bfloat16)
    return out


def temperatures(B: int, *, seed: int, lo: float = 0.6, hi: float = 1.2, device="cpu") -> torch.Tensor:
    g = generator(device, seed, 5)
    return (lo + (hi - lo) * torch.rand((B,), generator=g, device=device)).to(torch.float32)
