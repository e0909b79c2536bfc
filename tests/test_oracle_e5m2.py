"""Pins of the oracle's E5M2 cache format (CPU only).

The E5M2 decode table is pinned to the format definition's closed forms and
to torch's float8_e5m2 (all 256 codes, NaN positions included).  The
format switch inside the attention is pinned against the E4M3 path: an
E5M2 problem whose values all lie where both formats are exact, transcoded
byte by byte to E4M3 (through torch), must give the same attention.  A
planted wrong exponent bias must fail a pin.
"""

import dataclasses

import numpy as np
import pytest
import torch

from synth import make_dense, make_sparse


def check_table(orc, plant=0):
    t = orc.e5m2_table(plant)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    ok = np.array_equal(np.isnan(t), np.isnan(ref)) and np.array_equal(t[~np.isnan(t)], ref[~np.isnan(ref)])
    # closed forms: 1.0, largest finite, infinity, smallest subnormal, -2
    ok &= t[0x3C] == 1.0 and t[0x7B] == 57344.0 and np.isposinf(t[0x7C]) and t[0x01] == 2.0 ** -16
    ok &= t[0xC0] == -2.0 and np.isnan(t[0x7D]) and t[0x80] == 0.0 and np.signbit(t[0x80])
    return bool(ok)


def _transcode(cache_e5m2):
    """E5M2 bytes -> E4M3 bytes of the same values (exact in range)."""
    v = cache_e5m2.view(torch.float8_e5m2).float()
    back = v.to(torch.float8_e4m3fn).float()
    assert torch.equal(back, v) or bool(torch.isnan(v).any()), "value outside the common range"
    return v.to(torch.float8_e4m3fn).view(torch.uint8)


def _common_range(p):
    # clamp the E5M2 codes to the range both formats represent exactly:
    # |x| in [2^-9, 448] or 0 (2-bit mantissas fit in 3)
    def fix(c):
        v = c.view(torch.float8_e5m2).float()
        a = v.abs()
        v = torch.where(a > 448, torch.sign(v) * 448, v)
        v = torch.where((a > 0) & (a < 2.0 ** -9), torch.zeros_like(v), v)
        return v.to(torch.float8_e5m2).view(torch.uint8)
    return dataclasses.replace(p, k_cache=fix(p.k_cache), v_cache=fix(p.v_cache))


def check_attention_against_e4m3(orc, plant=0):
    p = make_dense(name="e5", B=2, q=3, Hq=4, Hkv=2, D=64, page_size=16, lens=(300, 500), seed=4,
                   kv_format="e5m2", poison=0)
    p = _common_range(p)
    q4 = dataclasses.replace(p, kv_format="e4m3", k_cache=_transcode(p.k_cache), v_cache=_transcode(p.v_cache))
    return bool(np.array_equal(orc.attention(p, plant=plant), orc.attention(q4, plant=plant)))


PINS = [check_table, check_attention_against_e4m3]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_e5m2_pin(orc, pin):
    assert pin(orc)


def test_sparse_e5m2_against_e4m3(orc):
    p = _common_range(make_sparse(name="e5s", B=2, q=4, Hq=4, Hkv=2, D=64, L=700, topk_blocks=30, seed=6,
                                  kv_format="e5m2", poison=0))
    q4 = dataclasses.replace(p, kv_format="e4m3", k_cache=_transcode(p.k_cache), v_cache=_transcode(p.v_cache))
    assert np.array_equal(orc.attention(p), orc.attention(q4))


def test_planted_bias_is_caught(orc):
    orc.load(14)
    assert sum(not pin(orc, 14) for pin in PINS) >= 1
