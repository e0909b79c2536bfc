"""Invariance pins for the oracle.

* relocating pages (another physical permutation, same logical content) leaves
  the result bitwise unchanged;
* the FP64 split-KV partition + combine equals the unsplit result (1e-13);
* sparse: entry order and extra mask-0 padding entries do not matter; a
  sparse table whose masks select every causal token of every microblock
  equals the dense causal result;
* GQA grouping: query head h reads KV head h // (Hq/Hkv) and no other.
"""

import numpy as np
import pytest
import torch

from synth import make_dense, make_sparse
from synth.workloads import _u32_bits, masks_u32


def _relocate(p, seed):
    g = torch.Generator().manual_seed(seed)
    nb = p.k_cache.shape[0]
    perm = torch.randperm(nb - 1, generator=g) + 1
    newk = p.k_cache.clone()
    newv = p.v_cache.clone()
    newk[perm] = p.k_cache[1:]
    newv[perm] = p.v_cache[1:]
    bt = p.block_table.clone()
    used = bt.long() - 1
    bt = perm[used].to(torch.int32)
    return newk, newv, bt


def test_page_permutation_bitwise(orc):
    p = make_dense(B=2, q=3, Hq=4, Hkv=2, D=32, page_size=5, lens=[47, 31], seed=21, extra_pages=3)
    a = orc.attention(p)
    k2, v2, bt2 = _relocate(p, 99)
    p.k_cache, p.v_cache, p.block_table = k2, v2, bt2
    b = orc.attention(p)
    assert np.array_equal(a, b)


def test_split_count_invariance(orc):
    p = make_dense(B=1, q=4, Hq=3, Hkv=1, D=64, page_size=16, lens=[1000], seed=22)
    a = orc.attention(p)
    for S in (1, 2, 3, 7, 64, 1500):
        b = orc.attention_split(p, S)
        np.testing.assert_allclose(b, a, rtol=1e-13, atol=1e-16)


def test_sparse_order_and_padding(orc):
    p = make_sparse(B=2, q=4, Hq=4, Hkv=2, D=16, L=400, topk_blocks=12, seed=23)
    a = orc.attention(p)
    # shuffle the real entries
    g = torch.Generator().manual_seed(5)
    for b in range(p.B):
        n = int(p.n_entries[b])
        perm = torch.randperm(n, generator=g)
        p.entry_tbl[b, :n] = p.entry_tbl[b, :n][perm]
        p.entry_mask[b, :n] = p.entry_mask[b, :n][perm]
    b_ = orc.attention(p)
    np.testing.assert_allclose(b_, a, rtol=1e-13, atol=1e-15)
    # append 8 more null padding entries
    B, E = p.entry_tbl.shape
    et = torch.zeros((B, E + 8), dtype=torch.int32)
    em = torch.zeros((B, E + 8), dtype=torch.int32)
    et[:, :E] = p.entry_tbl
    em[:, :E] = p.entry_mask
    p.entry_tbl, p.entry_mask = et, em
    p.n_entries = p.n_entries + 8
    c = orc.attention(p)
    assert np.array_equal(c, b_)


@pytest.mark.parametrize("q", [3, 12, 16])
def test_sparse_all_visible_equals_dense(orc, q):
    """Rows 8..15 (q > 8) take their bits from the second mask word."""
    L = 61
    d = make_dense(B=1, q=q, Hq=2, Hkv=1, D=16, page_size=4, lens=[L], seed=24)
    # same physical pool viewed as microblocks, every causal token visible
    nmb = (L + 3) // 4
    masks = []
    for m in range(nmb):
        bits = 0
        for r in range(q):
            n_r = L - q + 1 + r
            for t in range(4):
                if 4 * m + t < n_r:
                    bits |= 1 << (4 * r + t)
        masks.append(bits)
    s = make_sparse(B=1, q=q, Hq=2, Hkv=1, D=16, L=max(8, q), topk_blocks=1, seed=0)
    s.k_cache, s.v_cache, s.q_fp16 = d.k_cache, d.v_cache, d.q_fp16
    s.softmax_scale, s.k_scale, s.v_scale = d.softmax_scale, d.k_scale, d.v_scale
    s.entry_tbl = d.block_table[:, :nmb].clone()
    s.entry_mask = _u32_bits(torch.tensor([[m & 0xFFFFFFFF for m in masks]], dtype=torch.int64))
    s.entry_mask_hi = _u32_bits(torch.tensor([[m >> 32 for m in masks]], dtype=torch.int64)) if q > 8 else None
    s.q = q
    s.n_entries = torch.tensor([nmb], dtype=torch.int32)
    assert np.array_equal(orc.attention(s), orc.attention(d))
    assert int(masks_u32(s).max()) < 2**32


def test_gqa_grouping(orc):
    p = make_dense(B=1, q=2, Hq=6, Hkv=3, D=16, page_size=8, lens=[50], seed=25)
    a = orc.attention(p)
    # perturb KV head 2 only: heads 0..3 (groups 0, 1) must not change
    p.k_cache[..., 2, :] = p.k_cache[..., 2, :].flip(-1)
    p.v_cache[..., 2, :] = p.v_cache[..., 2, :].flip(-1)
    b = orc.attention(p)
    assert np.array_equal(a[:, :, :4], b[:, :, :4])
    assert not np.array_equal(a[:, :, 4:], b[:, :, 4:])
    # identical queries in one group give identical outputs
    p.q_fp16[0, :, 1] = p.q_fp16[0, :, 0]
    c = orc.attention(p)
    assert np.array_equal(c[0, :, 0], c[0, :, 1])
