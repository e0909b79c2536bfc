"""Closed-form pins for the oracle.

* one visible token: the weight is exactly 1, so out = v_scale * dec(v);
* identical keys: uniform weights, so out = v_scale * mean(dec(V)) (an exact
  rational, compared here with Fractions);
* two tokens: w_1 = 1 / (1 + exp(z_2 - z_1)), the logistic function;
* dead rows (live length 0, or a sparse row with no visible bit) are +0.0;
* v_scale is a pure output factor; k_scale and softmax_scale enter only as a
  product.
"""

import math
from fractions import Fraction

import numpy as np
import torch

from synth import make_dense, make_sparse


def _dec(byte):
    return float(torch.tensor([byte], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64))


def test_single_token_exact(orc):
    p = make_dense(B=1, q=2, Hq=2, Hkv=1, D=8, page_size=4, lens=[6], seed=11,
                   row_len=[[1, 0]], value_mode="direct", k_scale=0.5, v_scale=1.9)
    out = orc.attention(p)
    blk = int(p.block_table[0, 0])
    vbytes = p.v_cache[blk, 0, 0].tolist()
    # the problem holds v_scale as the FP32 value the interface carries
    assert p.v_scale == float(np.float32(1.9))
    want = np.array([p.v_scale * _dec(b) for b in vbytes])
    assert np.array_equal(out[0, 0, 0], want)
    assert np.array_equal(out[0, 0, 1], want)
    assert np.all(out[0, 1] == 0.0) and not np.signbit(out[0, 1]).any()


def test_constant_keys_give_mean(orc):
    p = make_dense(B=1, q=1, Hq=1, Hkv=1, D=16, page_size=5, lens=[13], seed=12)
    # every token gets the same key bytes
    k0 = p.k_cache[int(p.block_table[0, 0]), 0, 0].clone()
    for j in range(13):
        p.k_cache[int(p.block_table[0, j // 5]), j % 5, 0] = k0
    out = orc.attention(p)[0, 0, 0]
    vs = Fraction(p.v_scale)
    for d in range(16):
        vals = [Fraction(_dec(int(p.v_cache[int(p.block_table[0, j // 5]), j % 5, 0, d]))) for j in range(13)]
        exact = vs * sum(vals) / 13
        # a 13-term double sum: error bounded by a few ulps of sum |terms|
        scale = vs * sum(abs(v) for v in vals) / 13
        assert abs(Fraction(out[d]) - exact) <= scale * Fraction(1, 2**48)


def test_two_tokens_logistic(orc):
    p = make_dense(B=1, q=1, Hq=1, Hkv=1, D=4, page_size=2, lens=[2], seed=13, softmax_scale=0.3)
    w = orc.row_weights(p, 0, 0, 0)
    qv = p.q_fp16[0, 0, 0].double().numpy()
    kz = []
    for j in range(2):
        kb = p.k_cache[int(p.block_table[0, 0]), j, 0]
        kd = kb.view(torch.float8_e4m3fn).double().numpy()
        kz.append(p.softmax_scale * p.k_scale * float(qv @ kd))  # the FP32 scales the problem holds
    w1 = 1.0 / (1.0 + math.exp(kz[1] - kz[0]))
    assert len(w) == 2
    assert abs(w[0] - w1) < 1e-15 and abs(w[1] - (1 - w1)) < 1e-15


def test_weights_sum_to_one(orc):
    p = make_dense(B=1, q=4, Hq=2, Hkv=1, D=32, page_size=7, lens=[300], seed=14)
    for r in range(4):
        w = orc.row_weights(p, 0, r, 1)
        assert len(w) == int(p.row_len[0, r])
        assert abs(w.sum() - 1.0) < 1e-12 and (w > 0).all()


def test_dead_sparse_row(orc):
    p = make_sparse(B=1, q=3, Hq=3, Hkv=1, D=8, L=40, topk_blocks=2, seed=15)
    p.entry_mask[:] = torch.where(p.entry_mask != 0, p.entry_mask & 0x0FF, p.entry_mask)  # row 2 sees nothing
    out = orc.attention(p)
    assert np.all(out[0, 2] == 0.0)
    assert np.abs(out[0, 0]).sum() > 0


def test_scale_roles(orc):
    p = make_dense(B=1, q=2, Hq=2, Hkv=1, D=16, page_size=8, lens=[40], seed=16,
                   value_mode="direct", k_scale=0.37, v_scale=1.9, softmax_scale=0.25)
    a = orc.attention(p)
    p2 = make_dense(B=1, q=2, Hq=2, Hkv=1, D=16, page_size=8, lens=[40], seed=16,
                    value_mode="direct", k_scale=0.25, v_scale=3.8, softmax_scale=0.37)
    b = orc.attention(p2)
    np.testing.assert_allclose(b, 2.0 * a, rtol=1e-15, atol=0)
    # k_scale changes the weights (not a pure output factor)
    p3 = make_dense(B=1, q=2, Hq=2, Hkv=1, D=16, page_size=8, lens=[40], seed=16,
                    value_mode="direct", k_scale=0.74, v_scale=1.9, softmax_scale=0.25)
    assert np.abs(orc.attention(p3) - a).max() > 1e-3


def test_abs_condition(orc):
    p = make_dense(B=1, q=3, Hq=2, Hkv=1, D=32, page_size=8, lens=[90], seed=17)
    out = orc.attention(p)
    ab = orc.attention_abs(p)
    assert np.all(ab >= np.abs(out) * (1 - 1e-12))
    # with every V byte non-negative the two coincide exactly
    p.v_cache &= 0x7F
    p.v_cache[p.v_cache == 0x7F] = 0x7E
    assert np.array_equal(orc.attention_abs(p), orc.attention(p))


def _kv_rows(p, b, g, n):
    rows_k, rows_v = [], []
    for j in range(n):
        blk = int(p.block_table[b, j // p.page_size])
        rows_k.append(p.k_cache[blk, j % p.page_size, g].view(torch.float8_e4m3fn).double().numpy())
        rows_v.append(p.v_cache[blk, j % p.page_size, g].view(torch.float8_e4m3fn).double().numpy())
    return rows_k, rows_v


def test_logit_cond_two_tokens(orc):
    """Two tokens: v_1 - out = w_2 (v_1 - v_2) and v_2 - out = w_1 (v_2 - v_1),
    so the condition is w_1 w_2 (a_1 + a_2) |v_1 - v_2| with a_j the scaled
    sum of |q_d k_jd|."""
    p = make_dense(B=1, q=1, Hq=1, Hkv=1, D=8, page_size=2, lens=[2], seed=18, softmax_scale=0.3)
    cnd = orc.attention_logit_cond(p)[0, 0, 0]
    ks, vs = _kv_rows(p, 0, 0, 2)
    qv = p.q_fp16[0, 0, 0].double().numpy()
    sc = p.softmax_scale * p.k_scale
    z = [sc * float(qv @ k) for k in ks]
    w1 = 1.0 / (1.0 + math.exp(z[1] - z[0]))
    w2 = 1.0 - w1
    a = [sc * float(np.abs(qv * k).sum()) for k in ks]
    want = w1 * w2 * (a[0] + a[1]) * np.abs(p.v_scale * (vs[0] - vs[1]))
    np.testing.assert_allclose(cnd, want, rtol=1e-12, atol=0)
    assert (cnd > 0).any()


def test_logit_cond_zero_cases(orc):
    # one visible token: out = v_1 exactly, whatever its logit
    p = make_dense(B=1, q=2, Hq=2, Hkv=1, D=8, page_size=4, lens=[6], seed=19, row_len=[[1, 0]])
    c = orc.attention_logit_cond(p)
    assert np.all(c == 0.0)
    # identical V rows: every v_j equals the output
    p = make_dense(B=1, q=1, Hq=1, Hkv=1, D=16, page_size=5, lens=[13], seed=20)
    v0 = p.v_cache[int(p.block_table[0, 0]), 0, 0].clone()
    for j in range(13):
        p.v_cache[int(p.block_table[0, j // 5]), j % 5, 0] = v0
    # zero up to the FP64 rounding of out = sum_j w_j v_0 (weights summing to 1)
    ks, _ = _kv_rows(p, 0, 0, 13)
    qv = p.q_fp16[0, 0, 0].double().numpy()
    amax = p.softmax_scale * p.k_scale * max(float(np.abs(qv * k).sum()) for k in ks)
    assert np.all(orc.attention_logit_cond(p) <= 1e-14 * amax * orc.attention_abs(p))


def test_logit_cond_bounds_logit_perturbation(orc):
    """Scaling k_scale by (1 + eps) perturbs every logit by eps z_j, |eps z_j| <=
    eps a_j: the output change stays within eps times the condition, and comes
    close to it somewhere (the bound is attained up to sign patterns)."""
    import copy
    p = make_dense(B=2, q=2, Hq=4, Hkv=2, D=32, page_size=8, lens=[150, 77], seed=21,
                   value_mode="direct", k_scale=0.75, v_scale=1.25, softmax_scale=0.5)
    base = orc.attention(p)
    cnd = orc.attention_logit_cond(p)
    ab = orc.attention_abs(p)
    ratios = []
    for f in (1 + 2.0 ** -20, 1 - 2.0 ** -20):
        p2 = copy.copy(p)
        p2.k_scale = p.k_scale * f
        eps = abs(p2.k_scale / p.k_scale - 1.0)
        d = np.abs(orc.attention(p2) - base)
        assert np.all(d <= eps * cnd * (1 + 1e-3) + 1e-13 * ab)
        live = cnd > 0
        ratios.append(float((d[live] / (eps * cnd[live])).max()))
    assert max(ratios) > 0.3, ratios
