"""Pins of the oracle's E5M2 encoder and E5M2 cache write (CPU only).

As for E4M3, the encoder is pinned to the format's decode table (every
finite code survives a round trip), the exact midpoints between adjacent
codes (ties to the even code) and the nearest code on either side of each
midpoint, saturation of the finite range (57344; infinities too), NaN and
signed zero, and torch's float8_e5m2 conversion inside the range.  The E5M2
cache write is pinned by the half-quantum bound of decode(write(x)) against
x / scale and by its slot placement.
"""

import numpy as np
import pytest
import torch

FINITE = [c for c in range(256) if (c & 0x7F) <= 0x7B]


def _enc(orc, x):
    return orc.e5m2_encode(np.asarray(x, dtype=np.float32))


def test_round_trip(orc):
    tab = orc.e5m2_table()
    vals = np.array([tab[c] for c in FINITE], dtype=np.float32)  # at most 3 significant bits: exact
    assert np.array_equal(_enc(orc, vals), np.array(FINITE, dtype=np.uint8))


def test_midpoints_ties_to_even(orc):
    tab = orc.e5m2_table()
    for sign in (1.0, -1.0):
        s = 0x80 if sign < 0 else 0
        for c in range(0, 0x7B):
            lo, hi = tab[c], tab[c + 1]
            mid = np.float32((lo + hi) / 2)
            assert float(mid) == (lo + hi) / 2
            even = c if c % 2 == 0 else c + 1
            above = np.nextafter(mid, np.float32(np.inf), dtype=np.float32)
            below = np.nextafter(mid, np.float32(0), dtype=np.float32)
            got = _enc(orc, [sign * mid, sign * above, sign * below])
            assert list(got) == [s | even, s | (c + 1), s | c], (c, sign)


def test_saturation(orc):
    big = [57344.0, np.nextafter(np.float32(57344), np.float32(np.inf)), 61439.0, 61440.0, 65536.0,
           1e9, 3.0e38, np.inf]
    assert np.all(_enc(orc, big) == 0x7B)
    assert np.all(_enc(orc, [-x for x in big]) == 0xFB)


def test_nan_and_zero(orc):
    tab = orc.e5m2_table()
    assert np.isnan(tab[int(_enc(orc, [np.nan])[0])])
    tiny = 2.0 ** -18  # below half the smallest subnormal (2^-16)
    assert list(_enc(orc, [0.0, -0.0, tiny, -tiny])) == [0x00, 0x80, 0x00, 0x80]


def test_matches_torch_in_range(orc):
    g = torch.Generator().manual_seed(8)
    mag = torch.exp2(torch.empty(20000).uniform_(-17.0, np.log2(57344.0), generator=g))
    x = (mag * torch.where(torch.rand(20000, generator=g) < 0.5, -1.0, 1.0)).to(torch.float32)
    ref = x.to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(_enc(orc, x.numpy()), ref)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_e5m2_cache_write(orc, dtype):
    g = torch.Generator().manual_seed(9)
    N, Hkv, D, page, blocks = 11, 2, 32, 4, 8
    k = (torch.randn(N, Hkv, D, generator=g) * 300).to(dtype)
    v = (torch.randn(N, Hkv, D, generator=g) * 300).to(dtype)
    slots = torch.randperm(blocks * page, generator=g)[:N].to(torch.int64)
    slots[2] = -1
    kc = torch.full((blocks, page, Hkv, D), 0x55, dtype=torch.uint8)
    vc = kc.clone()
    ks, vs = 0.75, 2.5
    bad = orc.cache_write(k, v, slots, kc, vc, ks, vs, page, kv_format="e5m2")
    assert bad == 0
    tab = orc.e5m2_table()
    for n in range(N):
        s = int(slots[n])
        if s < 0:
            continue
        for cache, x, sc in ((kc, k, ks), (vc, v, vs)):
            y = x[n].double().numpy() / sc
            got = tab[cache[s // page, s % page].numpy().astype(np.int64)]
            # half a quantum: 2^(e-3) for |y| in [2^e, 2^(e+1)), subnormals 2^-17
            e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -14)))
            assert np.all(np.abs(got - np.clip(y, -57344, 57344)) <= 2.0 ** (e - 3) * (1 + 1e-12))
    written = {int(s) for s in slots if s >= 0}
    for s in range(blocks * page):
        if s not in written:
            assert bool((kc[s // page, s % page] == 0x55).all()) and bool((vc[s // page, s % page] == 0x55).all())
