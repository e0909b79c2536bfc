"""Seeded token-ID selections (the sparse path's selection ABI).

Generators only.  For a sparse problem's requests (``make_sparse``; its
``meta["block_table"]`` maps logical to physical microblocks), every query
row r of request b picks token positions among the tokens it may see,
[0, L - q + 1 + r): runs of neighbouring tokens around random centres (as a
top-k over token scores tends to give), some duplicates, unused slots (-1)
and, optionally, positions past the context.  Rows pick independently, so
rows of one request share some microblocks and not others.
"""

from __future__ import annotations

import torch


def make_selection(B: int, q: int, L: int, topk: int, *, seed: int = 0, run: int = 6,
                   unused_fraction: float = 0.1, dup_fraction: float = 0.05,
                   past_end: int = 0) -> torch.Tensor:
    """int32 [B][q][topk] token positions (-1 = unused slot)."""
    g = torch.Generator().manual_seed(seed)
    sel = torch.full((B, q, topk), -1, dtype=torch.int64)
    for b in range(B):
        for r in range(q):
            n_r = L - q + 1 + r
            if n_r <= 0:
                continue
            picks = []
            while len(picks) < topk:
                c = int(torch.randint(0, n_r, (1,), generator=g))
                length = int(torch.randint(1, run + 1, (1,), generator=g))
                picks.extend(t for t in range(c, min(c + length, n_r)))
            row = torch.tensor(picks[:topk], dtype=torch.int64)
            n_dup = int(dup_fraction * topk)
            if n_dup:
                i = torch.randint(0, topk, (n_dup,), generator=g)
                j = torch.randint(0, topk, (n_dup,), generator=g)
                row[i] = row[j]
            n_un = int(unused_fraction * topk)
            if n_un:
                row[torch.randperm(topk, generator=g)[:n_un]] = -1
            sel[b, r] = row
    for j in range(past_end):
        b, r, k = j % B, (j // B) % q, (7 * j) % topk
        sel[b, r, k] = 4 * ((L + 3) // 4) + 4 * j  # at or past the last microblock
    return sel.to(torch.int32)
