"""Seeded synthetic inputs for the draft-attention workloads.

Shared by the tests, the smoke check and the benchmark; this module holds none
of the method's arithmetic (no key selection, ring mapping or attention) --
only random values and random layouts drawn from seeded torch generators.

Workload shapes follow the pages' draft heads ("Windowed-MTP", §6: 2 GQA KV
heads, head_dim 256 for the Qwen drafts, 128 for Nemotron; bf16 KV; n_sink 64,
W 4032; gamma 6 at d = 7; contexts up to 1M).  Values are N(0, 1) drawn in
fp32 and rounded to bf16.
"""
from __future__ import annotations

import math

import torch


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, device, chunk_elems: int = 1 << 28) -> torch.Tensor:
    """N(0, 1) values rounded to bf16, generated in chunks to bound fp32 temps."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = generator(seed, device)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(s + chunk_elems, flat.numel())
        flat[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def scale_random_rows_(pool: torch.Tensor, frac: float, factor: float, seed: int) -> torch.Tensor:
    """Multiply a seeded Bernoulli(frac) subset of (slot, head) rows by `factor`
    in place (the 1 % x4 outlier keys of the million-token workload; a power
    of two keeps the scaled bf16 values exact)."""
    n_slots, H, _ = pool.shape
    g = generator(seed, pool.device)
    mask = torch.rand((n_slots, H), generator=g, device=pool.device) < frac
    pool[mask] = (pool[mask].float() * factor).to(pool.dtype)
    return mask


def permutation(n: int, seed: int, device) -> torch.Tensor:
    return torch.randperm(n, generator=generator(seed, device), device=device).to(torch.int32)


def uniform_lengths(B: int, lo: int, hi: int, seed: int) -> list[int]:
    g = generator(seed, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


def log_uniform_lengths(B: int, lo: int, hi: int, seed: int) -> list[int]:
    g = generator(seed, "cpu")
    u = torch.rand(B, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


def ring_bases(B: int, ring_size: int, n_regions: int, seed: int) -> list[int]:
    """Seeded placement of B rings of `ring_size` slots among `n_regions`
    equal regions of a pool (n_regions >= B)."""
    g = generator(seed, "cpu")
    regions = torch.randperm(n_regions, generator=g)[:B]
    return [int(r) * ring_size for r in regions]


def e4m3_codes(shape, seed: int, device, lo: int = 0x20, hi: int = 0x68) -> torch.Tensor:
    """Random E4M3 codes (uint8): a random sign and a magnitude code drawn
    uniformly from [lo, hi) -- values log-uniform over (hi - lo) / 8 octaves,
    2^-3 .. 2^6 by default; never a NaN code while hi <= 0x7F."""
    g = generator(seed, device)
    mag = torch.randint(lo, hi, shape, generator=g, device=device, dtype=torch.int32)
    sign = torch.randint(0, 2, shape, generator=g, device=device, dtype=torch.int32) * 0x80
    return (mag | sign).to(torch.uint8)
