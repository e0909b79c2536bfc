"""Seeded inputs for the cache write (new K/V rows and their slots).

Generators only: this module draws values and slot numbers and holds none of
the quantisation arithmetic; the oracle and the CUDA path both consume what
it returns.

Shape of a write: N new tokens of Hkv heads x D, fp16 or bf16, laid out as a
paged allocator hands them out -- consecutive tokens fill a page, pages are
physical blocks in a random order.  Values are N(0, std) with a few large
outliers (so some codes saturate); ``edge=True`` mixes in exact midpoints
of the target format's codes (E4M3, or E5M2 with ``edge_format``; times the
scale), signed zeros, values far below the smallest
subnormal, infinities and NaN.  Some tokens are padding (slot -1) and some
name a block beyond the pool.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass
class CacheWriteProblem:
    k: torch.Tensor            # [N][Hkv][D] fp16 or bf16 (CPU)
    v: torch.Tensor
    slots: torch.Tensor        # int64 [N]
    page_size: int
    num_blocks: int
    k_scale: float
    v_scale: float
    poison: int                # byte the caches are filled with before the write

    @property
    def shape(self):
        return tuple(self.k.shape)

    def empty_caches(self, extra_heads: int = 0):
        """Fresh poisoned caches [blocks][page][Hkv + extra][D] (CPU uint8)."""
        N, Hkv, D = self.k.shape
        shape = (self.num_blocks, self.page_size, Hkv + extra_heads, D)
        return (torch.full(shape, self.poison, dtype=torch.uint8),
                torch.full(shape, self.poison, dtype=torch.uint8))


def _edge_values(n: int, scale: float, g: torch.Generator, fmt: str = "e4m3") -> torch.Tensor:
    # magnitudes of the format's finite codes and the midpoints between
    # neighbours, built from the bit layout (E4M3: 1 sign, 4 exponent, 3
    # mantissa, no infinity; E5M2: 1 sign, 5 exponent, 2 mantissa, exponent
    # 31 for infinities and NaNs)
    mags = []
    if fmt == "e4m3":
        for e in range(16):
            for m in range(8):
                if e == 15 and m == 7:
                    continue
                mags.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
        top = [448.0, 460.0]
    else:
        for e in range(31):
            for m in range(4):
                mags.append(m * 2.0 ** -16 if e == 0 else (1 + m / 4) * 2.0 ** (e - 15))
        top = [57344.0, 61440.0]
    mids = [(a + b) / 2 for a, b in zip(mags[:-1], mags[1:])]
    specials = [0.0, -0.0, 1e-12, -1e-12] + top + [1e9, float("inf"), float("-inf"), float("nan")]
    pool = torch.tensor(mags + mids + specials, dtype=torch.float64) * scale
    idx = torch.randint(0, pool.numel(), (n,), generator=g)
    sign = torch.where(torch.rand(n, generator=g) < 0.5, -1.0, 1.0).to(torch.float64)
    return pool[idx] * sign


def make_cache_write(N: int, Hkv: int, D: int, page_size: int, num_blocks: int, *,
                     dtype=torch.float16, seed: int = 0, std: float = 1.0,
                     k_scale: float = 0.0078125, v_scale: float = 0.015625,
                     pad_fraction: float = 0.05, bad_slots: int = 2, edge: bool = False,
                     poison: int = 0x5A, edge_format: str = "e4m3") -> CacheWriteProblem:
    g = torch.Generator().manual_seed(seed)
    pages = (N + page_size - 1) // page_size
    assert pages <= num_blocks, "pool too small for the tokens"
    k = torch.randn(N, Hkv, D, generator=g, dtype=torch.float64) * std
    v = torch.randn(N, Hkv, D, generator=g, dtype=torch.float64) * std
    # a few outliers per tensor, large enough to saturate at these scales
    for t, sc in ((k, k_scale), (v, v_scale)):
        if t.numel() == 0:
            continue
        n_out = max(1, t.numel() // 4096)
        pos = torch.randint(0, t.numel(), (n_out,), generator=g)
        t.view(-1)[pos] = 600.0 * sc * torch.where(torch.rand(n_out, generator=g) < 0.5, -1.0, 1.0).to(torch.float64)
    if edge:
        for t, sc in ((k, k_scale), (v, v_scale)):
            n_e = t.numel() // 3
            if n_e == 0:
                continue
            pos = torch.randperm(t.numel(), generator=g)[:n_e]
            t.view(-1)[pos] = _edge_values(n_e, sc, g, edge_format)
    k = k.to(dtype)
    v = v.to(dtype)
    perm = torch.randperm(num_blocks, generator=g)[:pages].to(torch.int64)
    n = torch.arange(N, dtype=torch.int64)
    slots = perm[n // page_size] * page_size + n % page_size
    if N > 0 and pad_fraction > 0:
        pad = torch.rand(N, generator=g) < pad_fraction
        slots[pad] = -1
    for j in range(min(bad_slots, N)):
        slots[(j * 7919) % N] = (num_blocks + j) * page_size + j % page_size
    return CacheWriteProblem(k=k, v=v, slots=slots, page_size=page_size, num_blocks=num_blocks,
                             k_scale=k_scale, v_scale=v_scale, poison=poison)
