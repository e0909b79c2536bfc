"""Pins of the oracle's E4M3 encoder and cache write (CPU only).

The encoder is pinned to things other than itself: the format's decode table
(every code must survive a round trip), the exact midpoints between adjacent
codes (ties to even) and the nearest code on either side of each midpoint,
saturation of the finite range, signed zero, and torch's float8_e4m3fn
conversion for values inside the range.  The cache write is pinned by slot
placement computed here from the slot number, untouched slots, the skipped
count, strided inputs and caches, and the half-quantum error bound of
decode(write(x)) against x / scale.  Planted mistakes in the oracle (ties
away from zero, overflow to NaN, an offset off by one) must each fail a pin.
"""

import numpy as np
import pytest
import torch

NAN_CODES = (0x7F, 0xFF)


def _table(orc, plant=0):
    return orc.e4m3_table(plant)


def _encode(orc, x, plant=0):
    return orc.e4m3_encode(np.asarray(x, dtype=np.float32), plant)


# ------------------------------------------------------------------ encoder pins

def check_round_trip(orc, plant=0):
    tab = _table(orc, 0)  # the decode table is pinned on its own
    codes = [c for c in range(256) if c not in NAN_CODES]
    vals = np.array([tab[c] for c in codes], dtype=np.float64)
    # every finite value is exact in float32 (at most 4 significant bits)
    got = _encode(orc, vals.astype(np.float32), plant)
    return np.array_equal(got, np.array(codes, dtype=np.uint8))


def check_midpoints(orc, plant=0):
    tab = _table(orc, 0)
    ok = True
    for sign in (1.0, -1.0):
        for c in range(0, 0x7E):  # adjacent finite magnitudes c, c+1
            lo, hi = tab[c], tab[c + 1]
            mid = np.float32((lo + hi) / 2)
            assert float(mid) == (lo + hi) / 2  # exact: at most 5 significant bits
            even = c if c % 2 == 0 else c + 1
            s = 0x80 if sign < 0 else 0
            above = np.nextafter(mid, np.float32(np.inf), dtype=np.float32)
            below = np.nextafter(mid, np.float32(0), dtype=np.float32)
            got = _encode(orc, [sign * mid, sign * above, sign * below], plant)
            ok &= int(got[0]) == (s | even)
            ok &= int(got[1]) == (s | (c + 1))
            ok &= int(got[2]) == (s | c)
    return ok


def check_saturation(orc, plant=0):
    big = [448.0, np.nextafter(np.float32(448), np.float32(np.inf)), 460.0, 464.0, 479.0, 480.0,
           1e6, 3.0e38, np.inf]
    pos = _encode(orc, big, plant)
    neg = _encode(orc, [-x for x in big], plant)
    return bool(np.all(pos == 0x7E) and np.all(neg == 0xFE))


def check_nan_and_zero(orc, plant=0):
    tab = _table(orc, 0)
    n = int(_encode(orc, [np.nan], plant)[0])
    z = _encode(orc, [0.0, -0.0, 1e-9, -1e-9, 2.0 ** -10, -(2.0 ** -10)], plant)
    return np.isnan(tab[n]) and list(z) == [0x00, 0x80, 0x00, 0x80, 0x00, 0x80]


def check_torch(orc, plant=0):
    g = torch.Generator().manual_seed(7)
    mag = torch.exp2(torch.empty(20000).uniform_(-12.0, np.log2(448.0), generator=g))
    x = (mag * torch.where(torch.rand(20000, generator=g) < 0.5, -1.0, 1.0)).to(torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.array_equal(_encode(orc, x.numpy(), plant), ref)


ENCODER_PINS = [check_round_trip, check_midpoints, check_saturation, check_nan_and_zero, check_torch]


@pytest.mark.parametrize("pin", ENCODER_PINS, ids=lambda f: f.__name__)
def test_encoder_pin(orc, pin):
    assert pin(orc)


# ------------------------------------------------------------------ cache write pins

def _problem(dtype=torch.float16, seed=3, N=13, Hkv=2, D=32, page=4, blocks=8, strided=False):
    g = torch.Generator().manual_seed(seed)
    k = (torch.randn(N, Hkv, D, generator=g) * 3).to(dtype)
    v = (torch.randn(N, Hkv, D, generator=g) * 3).to(dtype)
    if strided:  # non-contiguous token / head strides, d contiguous
        k = torch.cat([k, torch.zeros(N, Hkv, 16, dtype=dtype)], dim=2)[:, :, :D]
        v = torch.cat([v, torch.zeros(N, 1, D, dtype=dtype)], dim=1)[:, :Hkv, :]
    slots = torch.randperm(blocks * page, generator=g)[:N].to(torch.int64)
    slots[1] = -1                 # padding token
    slots[4] = blocks * page + 5  # block outside the cache
    if strided:  # caches inside a wider head layout
        kc_full = torch.full((blocks, page, Hkv + 1, D), 0x5A, dtype=torch.uint8)
        vc_full = torch.full((blocks, page, Hkv, D + 16), 0x5A, dtype=torch.uint8)
        kc, vc = kc_full[:, :, 1:, :], vc_full[:, :, :, :D]
    else:
        kc = torch.full((blocks, page, Hkv, D), 0x5A, dtype=torch.uint8)
        vc = torch.full((blocks, page, Hkv, D), 0x5A, dtype=torch.uint8)
    return k, v, slots, kc, vc, page


def check_cache_write(orc, plant=0, dtype=torch.float16, strided=False, k_scale=0.37, v_scale=2.5):
    k, v, slots, kc, vc, page = _problem(dtype=dtype, strided=strided)
    bad = orc.cache_write(k, v, slots, kc, vc, k_scale, v_scale, page, plant=plant)
    ok = bad == 1
    kq = k.float().numpy() / np.float32(k_scale)  # IEEE float32 division
    vq = v.float().numpy() / np.float32(v_scale)
    written = set()
    for n, s in enumerate(slots.tolist()):
        if s < 0 or s >= kc.shape[0] * page:
            continue
        b, o = divmod(s, page)
        written.add((b, o))
        ok &= np.array_equal(kc[b, o].numpy(), _encode(orc, kq[n]))
        ok &= np.array_equal(vc[b, o].numpy(), _encode(orc, vq[n]))
    for b in range(kc.shape[0]):
        for o in range(page):
            if (b, o) not in written:
                ok &= bool((kc[b, o] == 0x5A).all() and (vc[b, o] == 0x5A).all())
    return bool(ok)


def check_half_quantum(orc, plant=0):
    k, v, slots, kc, vc, page = _problem(seed=11)
    orc.cache_write(k, v, slots, kc, vc, 0.5, 0.75, page, plant=plant)
    tab = _table(orc, 0)
    ok = True
    for n, s in enumerate(slots.tolist()):
        if s < 0 or s >= kc.shape[0] * page:
            continue
        b, o = divmod(s, page)
        for src, cache, sc in ((k, kc, 0.5), (v, vc, 0.75)):
            x = src[n].double().numpy() / sc
            dec = tab[cache[b, o].numpy().astype(np.int64)]
            # quantum of the binade of |x| (subnormal quantum below 2^-6)
            e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -6)))
            q = np.exp2(e - 3)
            ok &= bool(np.all(np.abs(dec - np.clip(x, -448, 448)) <= q / 2 + 1e-12))
    return ok


CACHE_PINS = [check_cache_write, check_half_quantum]


@pytest.mark.parametrize("pin", CACHE_PINS, ids=lambda f: f.__name__)
def test_cache_write_pin(orc, pin):
    assert pin(orc)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("strided", [False, True])
def test_cache_write_layouts(orc, dtype, strided):
    assert check_cache_write(orc, dtype=dtype, strided=strided)


def test_power_of_two_scale_is_exact_scaling(orc):
    # x / 2^k is exact, so the stored code equals the encoder on x * 2^-k
    k, v, slots, kc, vc, page = _problem(seed=5)
    orc.cache_write(k, v, slots, kc, vc, 4.0, 0.125, page)
    n = 0 if slots[0] >= 0 else 2
    b, o = divmod(int(slots[n]), page)
    assert np.array_equal(kc[b, o].numpy(), _encode(orc, k[n].float().numpy() * 0.25))
    assert np.array_equal(vc[b, o].numpy(), _encode(orc, v[n].float().numpy() * 8.0))


def test_bf16_decode_matches_torch(orc):
    bits = torch.arange(0, 65536, 97, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double().numpy()
    got = np.array([orc.bf16_value(int(b) & 0xFFFF) for b in bits.tolist()])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])


# ------------------------------------------------------------------ planted mistakes

@pytest.mark.parametrize("plant", [9, 10, 11])
def test_planted_encoder_or_writer_mistake_is_caught(orc, plant):
    orc.load(plant)
    failures = sum(not pin(orc, plant) for pin in ENCODER_PINS + CACHE_PINS)
    assert failures >= 1, f"planted mistake {plant} passed every pin"
