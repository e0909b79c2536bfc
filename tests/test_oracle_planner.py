"""Pins of the oracle's grouped planner (token-ID selections -> microblock
entries with per-row masks, null-padded to a multiple of 8), CPU only.

Pinned by a case worked by hand (tests/golden/grouped_planner_case.json), by
invariants on seeded selections (every valid selection is visible in exactly
one entry, no bit without a selection, microblocks strictly increasing,
physical ids from the block table, null padding at the end to a multiple of
8, positions past the table counted as ignored), and end to end: the sparse
attention over the planner's entries equals, row by row, a softmax computed
directly over the row's selected tokens from the cache bytes.
"""

import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

from synth import make_selection, make_sparse

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "grouped_planner_case.json")


def test_hand_worked_case(orc):
    g = json.load(open(GOLDEN))
    tbl, msk, n, ign = orc.select_to_entries(np.array(g["sel"]), np.array(g["block_table"]), g["max_blocks"],
                                             g["null_block"])
    assert tbl.tolist() == g["entry_tbl"] and msk.tolist() == g["entry_mask"]
    assert n.tolist() == g["n_entries"] and ign == 0


def _check_invariants(sel, bt, max_blocks, null, tbl, msk, n, msk_hi=None):
    """msk_hi (rows 8..15) joins msk as the upper 32 bits of one 64-bit mask."""
    B, q, _ = sel.shape
    msk = msk.astype(np.uint64)
    if msk_hi is not None:
        msk = msk | (msk_hi.astype(np.uint64) << np.uint64(32))
    for b in range(B):
        ne = int(n[b])
        assert ne % 8 == 0
        real = [e for e in range(ne) if msk[b, e] != 0]
        assert real == list(range(len(real)))  # padding only at the end
        assert all(tbl[b, e] == null for e in range(len(real), ne))
        phys = {int(tbl[b, e]): e for e in real}
        logical = []
        for e in real:  # invert the (injective) block table
            hits = np.nonzero(bt[b, :max_blocks] == tbl[b, e])[0]
            assert len(hits) == 1
            logical.append(int(hits[0]))
        assert logical == sorted(set(logical)) and len(logical) == len(real)
        want = {}
        for r in range(q):
            for t in sel[b, r].tolist():
                if 0 <= t < 4 * max_blocks:
                    want[t // 4] = want.get(t // 4, 0) | (1 << (4 * r + t % 4))
        got = {logical[i]: int(msk[b, e]) for i, e in enumerate(real)}
        assert got == want
        assert len(phys) == len(real)


@pytest.mark.parametrize("q,topk,L", [(1, 64, 300), (4, 48, 1000), (8, 200, 4000), (12, 64, 2000),
                                     (16, 32, 1000)])
def test_invariants(orc, q, topk, L):
    p = make_sparse(name="pl", B=3, q=q, Hq=2 * q if q <= 4 else q, Hkv=1, D=64, L=L, topk_blocks=4, seed=q)
    bt = p.meta["block_table"].numpy()
    sel = make_selection(3, q, L, topk, seed=7 + q, past_end=3).numpy()
    mb = bt.shape[1]
    tbl, msk, n, ign, msk_hi = orc.select_to_entries(sel, bt, mb, 0, with_hi=True)
    assert ign == 3
    assert (q > 8) == bool(msk_hi.any())
    _check_invariants(sel, bt, mb, 0, tbl, msk, n, msk_hi)


def test_empty_selection_gives_no_entries(orc):
    sel = np.full((2, 3, 5), -1)
    tbl, msk, n, ign = orc.select_to_entries(sel, np.arange(20).reshape(2, 10), 10, 0)
    assert n.tolist() == [0, 0] and ign == 0


def test_attention_over_entries_is_softmax_over_selected_tokens(orc):
    q, L, topk = 4, 600, 40
    p = make_sparse(name="pl", B=2, q=q, Hq=4, Hkv=2, D=64, L=L, topk_blocks=4, seed=5)
    bt = p.meta["block_table"].numpy()
    sel = make_selection(2, q, L, topk, seed=9).numpy()
    tbl, msk, n, _ = orc.select_to_entries(sel, bt, bt.shape[1], 0)
    p2 = dataclasses.replace(p, entry_tbl=torch.from_numpy(tbl), entry_mask=torch.from_numpy(msk.view(np.int32)),
                             n_entries=torch.from_numpy(n))
    got = orc.attention(p2)
    tab = orc.e4m3_table()
    G = p.Hq // p.Hkv
    for b in range(2):
        for r in range(q):
            toks = sorted({int(t) for t in sel[b, r] if t >= 0})
            for h in range(p.Hq):
                g = h // G
                qv = p.q_fp16[b, r, h].double().numpy()
                K = np.stack([tab[p.k_cache[bt[b, t // 4], t % 4, g].numpy().astype(np.int64)] for t in toks])
                V = np.stack([tab[p.v_cache[bt[b, t // 4], t % 4, g].numpy().astype(np.int64)] for t in toks])
                z = p.softmax_scale * p.k_scale * (K @ qv)
                w = np.exp(z - z.max())
                w /= w.sum()
                ref = p.v_scale * (w @ V)
                assert np.allclose(got[b, r, h], ref, rtol=1e-12, atol=1e-14), (b, r, h)
