"""GPU parity for the E5M2 cache format and for non-finite bytes in seen tokens.

E5M2 workloads (dense verify on the tensor-core path, D 256 and 128; the
QSA sparse path; decode on the generic path; the generic path forced on the
verify shape) are compared with the oracle as every other workload is
(tests/_check: rel L2 <= 5e-4, <= 4 fp16 ulps).  A NaN code in a K or V byte
of a token that some row sees must make exactly the oracle's elements NaN
(all of a seeing row's output for a K byte, column d for a V byte) on both
split kernels -- and no other element: the rows that do not see the token
stay finite even though the kernels multiply their exactly-zero weight into
the token's V row.  Cases: a token every row sees, the last draft-tail token
of the verify workload (seen by the last row only), a sparse token selected
by one query row only, and E5M2 infinities of both signs.  Padding NaNs
never reach the output (tested elsewhere).
"""

import numpy as np
import pytest
import torch

import oracle
from synth import make_dense, make_problem, make_sparse
from tests._check import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_e4m3_paged_gb300 import build_lib

    build_lib.build()
    oracle.build()


def _run(p, **kw):
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem

    dp = DeviceProblem(p, **kw)
    out = dp.run()
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), dp


@pytest.mark.parametrize("case", ["c2_tc", "c2_generic", "c3_64k", "sparse", "decode"])
def test_e5m2_matches_oracle(case):
    kw = {}
    if case.startswith("c2"):
        p = make_problem("c2", kv_format="e5m2")
        kw["kernel"] = 1 if case == "c2_generic" else 2
    elif case == "c3_64k":
        p = make_problem("c3_64k", kv_format="e5m2")
    elif case == "sparse":
        p = make_sparse(name="e5s", B=2, q=4, Hq=24, Hkv=2, D=128, L=32768, topk_blocks=256, seed=8,
                        kv_format="e5m2")
    else:
        p = make_dense(name="e5d", B=16, q=1, Hq=32, Hkv=8, D=128, page_size=16,
                       lens=[512 * (i + 1) for i in range(16)], seed=9, kv_format="e5m2")
    got, dp = _run(p, **kw)
    assert dp.status() == 0
    compare(got, oracle.attention(p), what=f"e5m2 {case}")


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("plane", ["k", "v"])
def test_nan_byte_in_a_seen_token(kernel, plane):
    p = make_problem("c2")
    cache = (p.k_cache if plane == "k" else p.v_cache).clone()
    # token 5 of the request (every row sees it), KV head 0, column 3
    blk = int(p.block_table[0, 5 // p.page_size])
    cache[blk, 5 % p.page_size, 0, 3] = 0x7F
    over = {"k_cache": cache} if plane == "k" else {"v_cache": cache}
    ref = oracle.attention(p, **over)
    got, _ = _run(p, kernel=kernel, **over)
    assert np.isnan(ref).any()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    compare(got[fin], ref[fin], what=f"finite elements, NaN in {plane}")


def _poke(p, plane, blk, slot, head, col, code):
    cache = (p.k_cache if plane == "k" else p.v_cache).clone()
    cache[blk, slot, head, col] = code
    return {"k_cache": cache} if plane == "k" else {"v_cache": cache}


def _check_nonfinite_pattern(got, ref, what):
    bad_ref = ~np.isfinite(ref)
    assert bad_ref.any(), what
    assert np.array_equal(np.isnan(got), np.isnan(ref)), f"{what}: NaN pattern differs"
    assert np.array_equal(np.isposinf(got), np.isposinf(ref)), f"{what}: +inf pattern differs"
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: -inf pattern differs"
    compare(got[~bad_ref], ref[~bad_ref], what=f"{what}: finite elements")


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("plane", ["k", "v"])
def test_nan_byte_in_last_draft_token(kernel, plane):
    """Token L-1 of the 8-row verify workload is seen by row 7 only."""
    p = make_problem("c2")
    t = p.max_kv_len - 1
    over = _poke(p, plane, int(p.block_table[0, t // p.page_size]), t % p.page_size, 0, 200, 0x7F)
    ref = oracle.attention(p, **over)
    got, dp = _run(p, kernel=kernel, **over)
    assert dp.status() == 0
    # only row 7 (all heads for K, column 200 for V) is non-finite
    assert np.isnan(ref[0, 7]).any() and not np.isnan(ref[0, :7]).any()
    _check_nonfinite_pattern(got, ref, f"draft-tail NaN in {plane}, kernel {kernel}")


def _single_row_token(p, b=0):
    """(entry, token, row) of a sparse token that exactly one query row sees."""
    masks = p.entry_mask[b].numpy().astype(np.int64) & 0xFFFFFFFF
    for e in range(int(p.n_entries[b])):
        mk = int(masks[e])
        if mk == 0:
            continue
        for tk in range(4):
            rows = [r for r in range(p.q) if (mk >> (4 * r + tk)) & 1]
            if len(rows) == 1:
                return e, tk, rows[0]
    raise AssertionError("no single-row token in the selection")


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("plane", ["k", "v"])
def test_nan_byte_in_sparse_token_one_row_sees(kernel, plane):
    p = make_sparse(name="nan1", B=2, q=4, Hq=24, Hkv=2, D=128, L=32768, topk_blocks=256, seed=21)
    e, tk, r = _single_row_token(p)
    blk = int(p.entry_tbl[0, e])
    over = _poke(p, plane, blk, tk, 1, 77, 0xFF)
    ref = oracle.attention(p, **over)
    got, dp = _run(p, kernel=kernel, **over)
    assert dp.status() == 0
    others = [x for x in range(p.q) if x != r]
    assert np.isnan(ref[0, r]).any() and not np.isnan(ref[0, others]).any() and not np.isnan(ref[1]).any()
    _check_nonfinite_pattern(got, ref, f"sparse single-row NaN in {plane}, kernel {kernel}")


@pytest.mark.parametrize("kernel", [1, 2])
def test_e5m2_infinities_in_v(kernel):
    """E5M2 +inf and -inf V codes in two columns of the last draft token and
    both signs in one column of an earlier token: +inf, -inf and NaN (inf - inf)
    exactly where the oracle has them."""
    p = make_problem("c2", kv_format="e5m2")
    t1 = p.max_kv_len - 1          # row 7 only
    t2 = p.max_kv_len - 3          # rows 5..7
    v = p.v_cache.clone()
    b1, s1 = int(p.block_table[0, t1 // p.page_size]), t1 % p.page_size
    b2, s2 = int(p.block_table[0, t2 // p.page_size]), t2 % p.page_size
    v[b1, s1, 0, 10] = 0x7C        # +inf
    v[b1, s1, 0, 11] = 0xFC        # -inf
    v[b2, s2, 0, 12] = 0x7C        # +inf ...
    v[b1, s1, 0, 12] = 0xFC        # ... and -inf in the same column: NaN for row 7
    ref = oracle.attention(p, v_cache=v)
    got, dp = _run(p, kernel=kernel, v_cache=v)
    assert dp.status() == 0
    assert np.isposinf(ref).any() and np.isneginf(ref).any() and np.isnan(ref).any()
    _check_nonfinite_pattern(got, ref, f"e5m2 infinities, kernel {kernel}")
