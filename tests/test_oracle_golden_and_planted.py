"""Pins from the pages' printed facts, and a check that the pins have teeth.

* QSA mask rule (tests/golden/qsa_mask_rule.json): under the bit layout
  "bit 4r+t = row r sees token t", the null-block fix's test (some mask bit
  at a position congruent to t modulo 4 is set) must coincide with "token t
  is seen by some row", and the oracle's visible sets must follow the
  fixture row by row.
* FP16 output-rounding floor: rounding the FP64 output to fp16 costs a
  relative L2 of about 2.03e-4 ("DFlash2 E4M3 attention with FP32 state",
  results: the FP64 reference gives an FP16 rounding floor of 0.000203267).
  This checks that the oracle's outputs have the magnitude spread of real
  attention outputs; it is a sanity pin, the pages' data are not ours.
* Planted mistakes: every deliberately broken oracle variant (wrong subnormal
  decode, dropped k_scale, wrong GQA grouping, off-by-one causal limit,
  dropped v_scale, transposed mask bits, K read for V, unnormalised weights)
  must fail at least one of the pins above and in the sibling test files.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from synth import make_dense, make_problem, make_sparse
from synth.workloads import _u32_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _one_entry_problem(mask: int):
    p = make_sparse(B=1, q=8, Hq=1, Hkv=1, D=4, L=64, topk_blocks=1, seed=31)
    blk = 5
    p.k_cache[blk] = 0  # all-zero keys: uniform weights
    for t in range(4):
        p.v_cache[blk, t, 0, :] = 0
        # E4M3 code of 2^t: exponent field 7+t, mantissa 0
        p.v_cache[blk, t, 0, 0] = (7 + t) << 3
    p.entry_tbl = torch.tensor([[blk] + [0] * 7], dtype=torch.int32)
    p.entry_mask = _u32_bits(torch.tensor([[mask] + [0] * 7], dtype=torch.int64))
    p.n_entries = torch.tensor([8], dtype=torch.int32)
    p.softmax_scale, p.k_scale, p.v_scale = 1.0, 1.0, 1.0
    return p


def _row_sets(orc, mask):
    p = _one_entry_problem(mask)
    out = orc.attention(p)
    sets = []
    for r in range(8):
        n = len(orc.row_weights(p, 0, r, 0))
        subset = int(round(out[0, r, 0, 0] * n)) if n else 0
        sets.append({t for t in range(4) if (subset >> t) & 1})
    return sets


def test_qsa_mask_rule(orc):
    fx = json.load(open(os.path.join(GOLDEN, "qsa_mask_rule.json")))
    for case in fx["cases"]:
        mask = int(case["mask"], 16)
        rule = [(mask & (0x11111111 << t)) != 0 for t in range(4)]
        assert rule == case["attended"], case
        sets = _row_sets(orc, mask)
        seen = [any(t in s for s in sets) for t in range(4)]
        assert seen == case["attended"], (case, sets)
    for case in fx["rows_seeing_token"]:
        sets = _row_sets(orc, int(case["mask"], 16))
        rows = [r for r in range(8) if case["token"] in sets[r]]
        assert rows == case["rows"], (case, sets)


def test_fp16_rounding_floor(orc):
    p = make_problem("c2")
    ref = orc.attention(p)
    r16 = ref.astype(np.float16).astype(np.float64)
    rel = np.linalg.norm(r16 - ref) / np.linalg.norm(ref)
    assert 1.8e-4 < rel < 2.3e-4, rel


# ---------------------------------------------------------------- planted

class _Planted:
    def __init__(self, plant):
        self.plant = plant

    def load(self):
        return oracle.load(self.plant)

    def e4m3_table(self):
        return oracle.e4m3_table(self.plant)

    def attention(self, p, **kw):
        return oracle.attention(p, plant=self.plant, **kw)

    def attention_split(self, p, s, **kw):
        return oracle.attention_split(p, s, plant=self.plant, **kw)

    def row_weights(self, p, b, r, h, **kw):
        return oracle.row_weights(p, b, r, h, plant=self.plant, **kw)


def _pins():
    from tests import test_oracle_bruteforce as bf
    from tests import test_oracle_closed_forms as cf
    from tests import test_oracle_decode as dc
    from tests import test_oracle_invariants as iv

    pins = [
        dc.test_e4m3_all_codes_match_torch,
        cf.test_single_token_exact,
        cf.test_scale_roles,
        cf.test_weights_sum_to_one,
        iv.test_gqa_grouping,
        lambda o: iv.test_sparse_all_visible_equals_dense(o, 3),
        lambda o: iv.test_sparse_all_visible_equals_dense(o, 12),
        test_qsa_mask_rule,
        lambda o: bf.test_dense_tiny_exact(o, 1),
        lambda o: bf.test_sparse_tiny_exact(o, 6),
    ]
    return pins


@pytest.mark.parametrize("plant", [1, 2, 3, 4, 5, 6, 7, 8])
def test_planted_mistake_is_caught(plant):
    pytest.importorskip("mpmath")
    o = _Planted(plant)
    failures = 0
    for pin in _pins():
        try:
            pin(o)
        except AssertionError:
            failures += 1
    assert failures >= 1, f"planted mistake {plant} passed every pin"


def test_unplanted_passes_all_pins(orc):
    pytest.importorskip("mpmath")
    for pin in _pins():
        pin(orc)
