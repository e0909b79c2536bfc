"""GPU parity of the fused cache write + verify (fp8kv_attn_split with new
K/V rows): the split launch quantises a verify step's new tokens into the
cache and attends over them.

Reference: the oracle's cache write of the same rows at the same positions
(slots from the block table), then the oracle's attention over that cache.
Before the call the new positions hold NaN bytes, so a row that read a
position before its write would turn NaN.  Checked: the cache bytes after the
call equal the oracle's (byte-exact), and the output matches the oracle
(tests/_check).  Cases: the query-row tensor-core kernel (8-row verify), the
CUDA-core kernel with bf16 rows and new tokens spanning two partitions, the
small-group kernel (decode: one new token per request), an E5M2 cache, and
graph replays (the write is idempotent).
"""

import numpy as np
import pytest
import torch

import oracle
from synth import make_dense, make_problem
from synth.workloads import POISON_NAN
from tests._check import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_e4m3_paged_gb300 import build_lib

    build_lib.build()
    oracle.build()


def _new_rows(p, n_new, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (p.B, n_new, p.Hkv, p.D)
    return ((torch.randn(shape, generator=g) * 1.5).to(dtype), (torch.randn(shape, generator=g) * 1.5).to(dtype))


def _positions(p, n_new):
    """(b, j, slot) of every new token: the last n_new positions of request b."""
    out = []
    for b in range(p.B):
        U = int(p.row_len[b].max())
        for j in range(n_new):
            pos = U - n_new + j
            out.append((b, j, int(p.block_table[b, pos // p.page_size]) * p.page_size + pos % p.page_size))
    return out


def _reference(p, k_new, v_new, n_new):
    kc, vc = p.k_cache.clone(), p.v_cache.clone()
    pos = _positions(p, n_new)
    k = torch.stack([k_new[b, j] for b, j, _ in pos])
    v = torch.stack([v_new[b, j] for b, j, _ in pos])
    slots = torch.tensor([s for _, _, s in pos], dtype=torch.int64)
    bad = oracle.cache_write(k, v, slots, kc, vc, p.k_scale, p.v_scale, p.page_size, kv_format=p.kv_format)
    assert bad == 0
    return kc, vc, oracle.attention(p, k_cache=kc, v_cache=vc)


def _poisoned(p, n_new):
    """The problem with NaN bytes at the new positions (their old content)."""
    kc, vc = p.k_cache.clone(), p.v_cache.clone()
    for _, _, s in _positions(p, n_new):
        kc[s // p.page_size, s % p.page_size] = POISON_NAN
        vc[s // p.page_size, s % p.page_size] = POISON_NAN
    return kc, vc


def _check(p, n_new, dtype, seed, what, **kw):
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem

    k_new, v_new = _new_rows(p, n_new, dtype, seed)
    kc_ref, vc_ref, ref = _reference(p, k_new, v_new, n_new)
    kc0, vc0 = _poisoned(p, n_new)
    dp = DeviceProblem(p, k_cache=kc0, v_cache=vc0, k_new=k_new, v_new=v_new, **kw)
    out = dp.run()
    torch.cuda.synchronize()
    assert dp.status() == 0
    assert torch.equal(dp.k_caches[0].cpu(), kc_ref), f"{what}: K cache bytes differ"
    assert torch.equal(dp.v_caches[0].cpu(), vc_ref), f"{what}: V cache bytes differ"
    compare(out.float().cpu().numpy(), ref, what=what)
    return dp, ref


@pytest.mark.parametrize("kernel", [0, 1])
def test_fused_verify_8_rows(kernel):
    p = make_problem("c2")
    dp, _ = _check(p, 8, torch.float16, 1, f"fused verify, kernel {kernel}", kernel=kernel)
    if kernel == 0:
        assert dp.plan.kernel == 2


def test_fused_bf16_rows_spanning_two_partitions():
    p = make_dense(name="fw", B=2, q=8, Hq=8, Hkv=2, D=128, page_size=64, lens=[3000, 1700], seed=81)
    # 40 new tokens over partitions of 32 tokens (forced split count)
    dp, _ = _check(p, 40, torch.bfloat16, 2, "fused, bf16 rows, two partitions", kernel=1, num_splits=94)
    assert dp.plan.num_splits == 94


def test_fused_decode_small_group():
    p = make_dense(name="fd", B=4, q=1, Hq=8, Hkv=2, D=128, page_size=16, lens=[900, 1500, 257, 4000], seed=82)
    dp, _ = _check(p, 1, torch.float16, 3, "fused decode, small group")
    assert dp.plan.kernel == 3


def test_fused_e5m2_cache():
    p = make_problem("c2", kv_format="e5m2")
    _check(p, 8, torch.float16, 4, "fused verify, E5M2 cache", kernel=2)


def test_fused_graph_replay_is_idempotent():
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem

    p = make_problem("c3_64k")
    k_new, v_new = _new_rows(p, 8, torch.float16, 5)
    kc_ref, vc_ref, ref = _reference(p, k_new, v_new, 8)
    kc0, vc0 = _poisoned(p, 8)
    dp = DeviceProblem(p, k_cache=kc0, v_cache=vc0, k_new=k_new, v_new=v_new)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dp.run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dp.run(stream=torch.cuda.current_stream().cuda_stream)
    first = None
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        got = dp.out.clone()
        first = got if first is None else first
        assert torch.equal(got, first)
    assert torch.equal(dp.k_caches[0].cpu(), kc_ref) and torch.equal(dp.v_caches[0].cpu(), vc_ref)
    compare(first.float().cpu().numpy(), ref, what="fused verify, graph replays")
    assert dp.status() == 0
