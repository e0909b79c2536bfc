"""Pins of the oracle's bf16 cache format (the unquantised K/V cache of A/B
runs, two little-endian bytes per element).

The bf16 decode itself is pinned against torch for all 65536 codes in
test_oracle_encode.py.  Here: the oracle's attention over a bf16 cache equals
an evaluation written separately in numpy (torch's bfloat16 decode of the
same bytes, float64 softmax), on dense and sparse problems; the single-token
closed form; and poisoned unseen slots (bf16 NaN) never reach the result.
"""

import numpy as np
import torch

from synth import make_dense, make_sparse
from synth.workloads import masks_u64


def _rows(cache, blk, slot, g):
    return cache[blk, slot, g].view(torch.bfloat16).double().numpy()


def _dense_ref(p):
    out = np.zeros((p.B, p.q, p.Hq, p.D))
    G = p.Hq // p.Hkv
    for b in range(p.B):
        for r in range(p.q):
            n = int(p.row_len[b, r])
            if n == 0:
                continue
            for h in range(p.Hq):
                g = h // G
                K = np.array([_rows(p.k_cache, int(p.block_table[b, j // p.page_size]), j % p.page_size, g)
                              for j in range(n)])
                V = np.array([_rows(p.v_cache, int(p.block_table[b, j // p.page_size]), j % p.page_size, g)
                              for j in range(n)])
                z = p.softmax_scale * p.k_scale * (K @ p.q_fp16[b, r, h].double().numpy())
                w = np.exp(z - z.max())
                out[b, r, h] = p.v_scale * (w @ V) / w.sum()
    return out


def test_dense_bf16_matches_numpy(orc):
    p = make_dense(B=2, q=3, Hq=4, Hkv=2, D=64, page_size=16, lens=[100, 37], seed=61, kv_format="bf16")
    assert p.k_cache.shape[-1] == 2 * p.D and p.k_scale == 1.0 == p.v_scale
    np.testing.assert_allclose(orc.attention(p), _dense_ref(p), rtol=1e-12, atol=1e-14)


def test_sparse_bf16_matches_numpy(orc):
    p = make_sparse(B=1, q=4, Hq=4, Hkv=1, D=32, L=300, topk_blocks=10, seed=62, kv_format="bf16")
    m = masks_u64(p)
    want = np.zeros((p.B, p.q, p.Hq, p.D))
    for r in range(p.q):
        K, V = [], []
        for e in range(int(p.n_entries[0])):
            for t in range(4):
                if (int(m[0, e]) >> (4 * r + t)) & 1:
                    blk = int(p.entry_tbl[0, e])
                    K.append(_rows(p.k_cache, blk, t, 0))
                    V.append(_rows(p.v_cache, blk, t, 0))
        K, V = np.array(K), np.array(V)
        for h in range(p.Hq):
            z = p.softmax_scale * (K @ p.q_fp16[0, r, h].double().numpy())
            w = np.exp(z - z.max())
            want[0, r, h] = (w @ V) / w.sum()
    np.testing.assert_allclose(orc.attention(p), want, rtol=1e-12, atol=1e-14)


def test_single_token_bf16_exact(orc):
    p = make_dense(B=1, q=2, Hq=2, Hkv=1, D=8, page_size=4, lens=[6], seed=63, row_len=[[1, 0]],
                   value_mode="direct", k_scale=0.5, v_scale=1.5, kv_format="bf16")
    out = orc.attention(p)
    blk = int(p.block_table[0, 0])
    want = p.v_scale * _rows(p.v_cache, blk, 0, 0)
    assert np.array_equal(out[0, 0, 0], want)
    assert np.all(out[0, 1] == 0.0)


def test_bf16_poison_is_nan_and_excluded(orc):
    p = make_dense(B=1, q=2, Hq=2, Hkv=1, D=16, page_size=8, lens=[13], seed=64, kv_format="bf16")
    # block 0 and the tail slots of the last page hold the bf16 NaN pattern
    assert torch.isnan(p.k_cache[0].view(torch.bfloat16)).all()
    last = int(p.block_table[0, 1])
    assert torch.isnan(p.v_cache[last, 5:].view(torch.bfloat16)).all()
    assert np.isfinite(orc.attention(p)).all()
