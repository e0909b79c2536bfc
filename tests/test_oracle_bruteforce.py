"""Brute-force pin: the oracle against an independent 50-digit evaluation.

Tiny problems (a handful of tokens, D <= 4) are evaluated here from scratch:
bytes are decoded by torch's float8_e4m3fn conversion and queries by numpy's
float16, the visible set is rebuilt from the block table / masks in Python,
and softmax attention is computed with mpmath at 50 significant digits.

Tolerance: 1e-13 relative to the element, plus 16 double-precision units
(2^-53) of the element's condition v_scale * sum_j w_j |V_j[d]| (computed in
the same 50-digit evaluation).  The oracle sums in double, so an element that
cancels far below its terms is accurate to a few units of the terms, not of
itself: a purely relative tolerance would fail it, a fixed absolute one would
be blind to the scale.
"""

import itertools

import numpy as np
import pytest
import torch

from synth import make_dense, make_sparse
from synth.workloads import masks_u32

mp = pytest.importorskip("mpmath")
mp.mp.dps = 50


def _dec_cache(t):
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _exact_dense(p):
    K = _dec_cache(p.k_cache)
    V = _dec_cache(p.v_cache)
    Q = p.q_fp16.numpy().astype(np.float64)
    G = p.Hq // p.Hkv
    out = np.zeros((p.B, p.q, p.Hq, p.D))
    cond = np.zeros_like(out)
    for b, r, h in itertools.product(range(p.B), range(p.q), range(p.Hq)):
        n = int(p.row_len[b, r])
        toks = [(int(p.block_table[b, j // p.page_size]), j % p.page_size) for j in range(n)]
        out[b, r, h], cond[b, r, h] = _attend(Q[b, r, h], K, V, toks, h // G, p)
    return out, cond


def _exact_sparse(p):
    K = _dec_cache(p.k_cache)
    V = _dec_cache(p.v_cache)
    Q = p.q_fp16.numpy().astype(np.float64)
    G = p.Hq // p.Hkv
    m = masks_u32(p)
    out = np.zeros((p.B, p.q, p.Hq, p.D))
    cond = np.zeros_like(out)
    for b, r, h in itertools.product(range(p.B), range(p.q), range(p.Hq)):
        toks = []
        for e in range(int(p.n_entries[b])):
            for t in range(4):
                if (int(m[b, e]) >> (4 * r + t)) & 1:
                    toks.append((int(p.entry_tbl[b, e]), t))
        out[b, r, h], cond[b, r, h] = _attend(Q[b, r, h], K, V, toks, h // G, p)
    return out, cond


def _attend(qv, K, V, toks, g, p):
    D = p.D
    if not toks:
        return np.zeros(D), np.zeros(D)
    c = mp.mpf(p.softmax_scale) * mp.mpf(p.k_scale)
    z = []
    for blk, slot in toks:
        z.append(c * mp.fsum(mp.mpf(qv[d]) * mp.mpf(K[blk, slot, g, d]) for d in range(D)))
    M = max(z)
    e = [mp.exp(x - M) for x in z]
    S = mp.fsum(e)
    res, cnd = [], []
    for d in range(D):
        acc = mp.fsum(e[j] * mp.mpf(V[toks[j][0], toks[j][1], g, d]) for j in range(len(toks)))
        ab = mp.fsum(e[j] * abs(mp.mpf(V[toks[j][0], toks[j][1], g, d])) for j in range(len(toks)))
        res.append(float(mp.mpf(p.v_scale) * acc / S))
        cnd.append(float(abs(mp.mpf(p.v_scale)) * ab / S))
    return np.array(res), np.array(cnd)


def _check(got, ref_cond):
    ref, cond = ref_cond
    bound = 1e-13 * np.abs(ref) + 16 * 2.0 ** -53 * cond
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"worst {float((err / np.where(bound > 0, bound, 1)).max()):.3f} of the bound"


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_dense_tiny_exact(orc, seed):
    p = make_dense(B=2, q=3, Hq=4, Hkv=2, D=4, page_size=3, lens=[7, 5], seed=seed,
                   row_len=[[5, 6, 7], [0, 4, 5]], k_scale=None)
    got = orc.attention(p)
    _check(got, _exact_dense(p))
    assert np.all(got[1, 0] == 0.0)


@pytest.mark.parametrize("seed", [4, 5])
def test_dense_tiny_direct_scales(orc, seed):
    p = make_dense(B=1, q=2, Hq=3, Hkv=1, D=3, page_size=2, lens=[8], seed=seed,
                   value_mode="direct", k_scale=0.37, v_scale=1.9, softmax_scale=0.7)
    _check(orc.attention(p), _exact_dense(p))


@pytest.mark.parametrize("seed", [6, 7])
def test_sparse_tiny_exact(orc, seed):
    p = make_sparse(B=2, q=3, Hq=4, Hkv=2, D=2, L=23, topk_blocks=3, seed=seed)
    got = orc.attention(p)
    _check(got, _exact_sparse(p))
    assert np.isfinite(got).all()
