"""Pins of the oracle's base-2 LSE output and its cross-rank merge (CPU).

The context-parallel merge is pinned by an identity that does not use the
merge's own formula: the context of a problem is cut into page ranges (one
per simulated rank), each shard's attention and LSE come from the oracle on
the shard alone, and merging them must give the oracle's attention and LSE
over the whole context.  The LSE is also pinned to closed forms (a single
visible token, equal logits), and the merge to the identity for one rank
and for an added empty rank.  Planted mistakes (natural-base weights for
base-2 LSEs, the sum left out of the LSE) must each fail a pin.
"""

import dataclasses
import math

import numpy as np
import pytest
import torch

from synth import make_dense


def _problem(seed=3, lens=(700, 1300), q=3, page=32):
    return make_dense(name="m", B=len(lens), q=q, Hq=4, Hkv=2, D=64, page_size=page, lens=lens, seed=seed)


def _shard(p, R, rank):
    """Shard `rank` of R: the pages [rank*pp, (rank+1)*pp) of every request,
    with the row lengths measured from the shard's first token."""
    pages = math.ceil(int(p.row_len.max()) / p.page_size)
    pp = math.ceil(pages / R)
    lo = rank * pp
    bt = p.block_table[:, lo:lo + pp]
    if bt.shape[1] < pp:  # past the table: columns no row reaches
        bt = torch.cat([bt, torch.zeros(bt.shape[0], pp - bt.shape[1], dtype=bt.dtype)], 1)
    rl = (p.row_len - lo * p.page_size).clamp(min=0, max=pp * p.page_size).to(torch.int32)
    return dataclasses.replace(p, block_table=bt.contiguous(), row_len=rl.contiguous(),
                               max_kv_len=pp * p.page_size)


def check_shards_merge_to_whole(orc, plant=0, R=3):
    p = _problem()
    full, lse_full = orc.attention_lse(p, plant=plant)
    parts = [orc.attention_lse(_shard(p, R, r), plant=plant) for r in range(R)]
    merged, lse = orc.merge([o for o, _ in parts], [l for _, l in parts], plant=plant)
    ok = np.allclose(merged, full, rtol=1e-11, atol=1e-13)
    ok &= np.allclose(lse, lse_full, rtol=0, atol=1e-10)
    # the merged output is also the plain attention (pinned on its own)
    ok &= np.allclose(merged, orc.attention(p), rtol=1e-11, atol=1e-13)
    return bool(ok)


def check_lse_closed_forms(orc, plant=0):
    # one visible token: lse = its base-2 logit
    p = _problem(lens=(1,), q=1)
    _, lse = orc.attention_lse(p, plant=plant)
    w = orc.row_weights(p, 0, 0, 0)
    ok = w.shape[0] == 1
    q = p.q_fp16[0, 0, 0].double().numpy()
    kb = p.k_cache[int(p.block_table[0, 0]), 0, 0].numpy()
    kd = orc.e4m3_table()[kb.astype(np.int64)]
    z = p.softmax_scale * p.k_scale * float(np.dot(q, kd))
    ok &= abs(lse[0, 0, 0] - z / math.log(2)) <= 1e-12 * max(1, abs(z))
    # equal logits (all keys equal): lse = z / ln 2 + log2(n)
    p = _problem(lens=(96,), q=1)
    kc = p.k_cache.clone()
    kc[:] = kc[int(p.block_table[0, 0]), 0]  # every slot holds the same key row
    _, lse = orc.attention_lse(p, plant=plant, k_cache=kc)
    q = p.q_fp16[0, 0, 0].double().numpy()
    kd = orc.e4m3_table()[kc[0, 0, 0].numpy().astype(np.int64)]
    z = p.softmax_scale * p.k_scale * float(np.dot(q, kd))
    ok &= abs(lse[0, 0, 0] - (z / math.log(2) + math.log2(96))) <= 1e-12 * max(1, abs(z))
    return bool(ok)


def check_merge_identities(orc, plant=0):
    rng = np.random.default_rng(1)
    o = rng.standard_normal((1, 5, 8))
    l = rng.standard_normal((1, 5)) * 3
    m, lm = orc.merge(o, l, plant=plant)
    ok = np.allclose(m, o[0], rtol=1e-15, atol=0) and np.allclose(lm, l[0], rtol=0, atol=1e-15)
    o2 = np.concatenate([o, np.zeros((1, 5, 8))])
    l2 = np.concatenate([l, np.full((1, 5), -np.inf)])
    m2, lm2 = orc.merge(o2, l2, plant=plant)
    ok &= np.allclose(m2, o[0], rtol=1e-15, atol=0) and np.allclose(lm2, l[0], rtol=0, atol=1e-15)
    # two ranks of equal LSE: the mean, and lse + 1
    m3, lm3 = orc.merge(np.stack([o[0], -o[0] + 2]), np.stack([l[0], l[0]]), plant=plant)
    ok &= np.allclose(m3, np.ones_like(o[0]), rtol=0, atol=1e-14) and np.allclose(lm3, l[0] + 1, atol=1e-14)
    # nobody sees the vector: 0 and -inf
    m4, lm4 = orc.merge(np.zeros((2, 1, 8)), np.full((2, 1), -np.inf), plant=plant)
    ok &= bool(np.all(m4 == 0) and np.all(np.isneginf(lm4)))
    return bool(ok)


PINS = [check_shards_merge_to_whole, check_lse_closed_forms, check_merge_identities]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_merge_pin(orc, pin):
    assert pin(orc)


@pytest.mark.parametrize("R", [2, 4, 7])
def test_shards_merge_for_rank_counts(orc, R):
    assert check_shards_merge_to_whole(orc, R=R)


def test_dead_rows_have_minus_infinity_lse(orc):
    p = _problem()
    rl = p.row_len.clone()
    rl[0, 1] = 0
    out, lse = orc.attention_lse(p, row_len=rl)
    assert np.all(np.isneginf(lse[0, 1])) and np.all(out[0, 1] == 0)


@pytest.mark.parametrize("plant", [12, 13])
def test_planted_merge_mistake_is_caught(orc, plant):
    orc.load(plant)
    failures = sum(not pin(orc, plant) for pin in PINS)
    assert failures >= 1, f"planted mistake {plant} passed every pin"
