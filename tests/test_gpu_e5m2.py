"""GPU parity for the E5M2 cache format and for NaN bytes in seen tokens.

E5M2 workloads (dense verify on the tensor-core path, D 256 and 128; the
QSA sparse path; decode on the generic path; the generic path forced on the
verify shape) are compared with the oracle as every other workload is
(tests/_check: rel L2 <= 5e-4, <= 4 fp16 ulps).  A NaN code in a K or V byte
of a token that some row sees must make exactly the oracle's elements NaN
(all of a seeing row's output for a K byte, column d for a V byte) on both
split kernels -- padding NaNs never reach the output (tested elsewhere).
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
