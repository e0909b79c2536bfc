"""Pins for the oracle's decoders (E4M3 cache bytes, fp16 queries).

The E4M3 table is checked against (a) the named codes of the format
definition (tests/golden/e4m3_special_values.json), (b) torch's
float8_e4m3fn -> float64 conversion for all 256 codes, and (c) structural
properties of the format (ordering, sign symmetry, NaN count).  The fp16
decoder is checked against numpy's float16 for all 65536 codes.
"""

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _same(a, b):
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def test_e4m3_named_codes(orc):
    fx = json.load(open(os.path.join(GOLDEN, "e4m3_special_values.json")))
    tab = orc.e4m3_table()
    for code, val in fx["values"].items():
        want = float("nan") if val == "nan" else float(val)
        assert _same(tab[int(code, 16)], want), (code, tab[int(code, 16)], want)


def test_e4m3_all_codes_match_torch(orc):
    tab = orc.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for i in range(256):
        assert _same(tab[i], ref[i]), (hex(i), tab[i], ref[i])


def test_e4m3_structure(orc):
    tab = orc.e4m3_table()
    pos = tab[:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes must increase strictly"
    for i in range(0x80):
        a, b = tab[i], tab[i | 0x80]
        if math.isnan(a):
            assert math.isnan(b)
        else:
            assert _same(b, -a)
    assert int(np.isnan(tab).sum()) == 2
    assert np.nanmax(tab) == 448.0 and np.nanmin(tab) == -448.0
    # smallest positive step is the subnormal quantum 2^-9
    assert tab[1] == 2.0 ** -9
    # every finite value times 2^8 is exactly representable in fp16
    fin = tab[~np.isnan(tab)] / 256.0
    assert np.all(fin.astype(np.float16).astype(np.float64) == fin)


def test_fp16_all_codes_match_numpy(orc):
    lib = orc.load()
    codes = np.arange(65536, dtype=np.uint32)
    ref = codes.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([lib.orc_f16(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
