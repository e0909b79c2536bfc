"""GPU parity for the bf16 K/V cache (the unquantised cache of A/B runs
against the FP8 path), served by the CUDA-core split kernel.

Dense verify (D 256), decode (D 128) and QSA sparse workloads against the
oracle (tests/_check: rel L2 <= 5e-4, <= 4 fp16 ulps), with the poison of
unseen slots as bf16 NaN and as the largest finite bf16; and a bf16 NaN in
the V row of the last draft token, which must reach exactly the oracle's
NaN elements (column d of the one row that sees the token).
"""

import numpy as np
import pytest
import torch

import oracle
from synth import make_dense, make_sparse
from synth.workloads import POISON_MAX, POISON_NAN
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
    assert dp.plan.kernel == 1  # bf16: the CUDA-core kernel
    out = dp.run()
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), dp


@pytest.mark.parametrize("case", ["verify", "decode", "sparse"])
@pytest.mark.parametrize("poison", [POISON_NAN, POISON_MAX])
def test_bf16_matches_oracle(case, poison):
    if case == "verify":
        p = make_dense(name="bf_v", B=1, q=8, Hq=6, Hkv=1, D=256, page_size=1728, lens=[20000], seed=71,
                       poison=poison, kv_format="bf16")
    elif case == "decode":
        p = make_dense(name="bf_d", B=8, q=1, Hq=32, Hkv=8, D=128, page_size=16,
                       lens=[700 * (i + 1) for i in range(8)], seed=72, poison=poison, kv_format="bf16")
    else:
        p = make_sparse(name="bf_s", B=2, q=4, Hq=24, Hkv=2, D=128, L=16384, topk_blocks=256, seed=73,
                        poison=poison, kv_format="bf16")
    got, dp = _run(p)
    compare(got, oracle.attention(p), what=f"bf16 {case} poison {poison:#x}")
    assert dp.status() == 0


def test_bf16_nan_in_last_draft_token():
    p = make_dense(name="bf_n", B=1, q=8, Hq=6, Hkv=1, D=256, page_size=1728, lens=[8192], seed=74,
                   kv_format="bf16")
    t = p.max_kv_len - 1
    blk, slot, col = int(p.block_table[0, t // p.page_size]), t % p.page_size, 200
    v = p.v_cache.clone()
    v[blk, slot, 0, 2 * col] = 0xC0  # bf16 0x7FC0, little-endian
    v[blk, slot, 0, 2 * col + 1] = 0x7F
    ref = oracle.attention(p, v_cache=v)
    got, dp = _run(p, v_cache=v)
    assert dp.status() == 0
    bad = np.isnan(ref)
    assert bad[0, 7, :, col].all() and bad.sum() == 6  # row 7 (the only one that sees t), column 200
    assert np.array_equal(np.isnan(got), bad)
    compare(got[~bad], ref[~bad], what="bf16 NaN in the last draft token: finite elements")
