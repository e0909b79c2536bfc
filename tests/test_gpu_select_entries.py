"""GPU parity of the grouped planner (fp8kv_attn_select_to_entries).

Integer output: entry tables, masks and counts must equal the oracle's
exactly (tests/test_oracle_planner.py pins the oracle).  Covered: 1..8 query
rows, duplicate and unused slots, positions past the table (ignored, status
bit), more logical microblocks than one shared-memory chunk (a 200K-token
context), empty selections, and the planner feeding the sparse attention on
the GPU end to end (output compared with the oracle on the oracle planner's
entries).
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from synth import make_selection, make_sparse
from tests._check import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_e4m3_paged_gb300 import build_lib

    build_lib.build()
    oracle.build()


def _gpu_plan(sel, bt, max_blocks, null_block):
    from fp8_e4m3_paged_gb300 import binding as B

    Bn, q, topk = sel.shape
    stride = max(8, (q * topk + 7) // 8 * 8)
    dev = torch.device("cuda")
    tbl = torch.full((Bn, stride), -7, dtype=torch.int32, device=dev)
    msk = torch.full((Bn, stride), -7, dtype=torch.int32, device=dev)
    msk_hi = torch.full((Bn, stride), -7, dtype=torch.int32, device=dev) if q > 8 else None
    n = torch.zeros(Bn, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    a = B.make_select_args(sel=torch.as_tensor(sel, dtype=torch.int32).to(dev).contiguous(),
                           block_table=torch.as_tensor(bt, dtype=torch.int32).to(dev).contiguous(),
                           max_blocks=max_blocks, null_block=null_block, entry_tbl=tbl, entry_mask=msk,
                           n_entries=n, status=st, entry_mask_hi=msk_hi)
    B.fp8kv_attn_select_to_entries(a, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    out = (tbl.cpu().numpy(), msk.cpu().numpy().view(np.uint32), n.cpu().numpy(), int(st.item()))
    if q > 8:
        out = out + (msk_hi.cpu().numpy().view(np.uint32),)
    return out


def _same(got, ref):
    tbl, msk, n = got[:3]
    rt, rm, rn = ref[:3]
    assert np.array_equal(n, rn)
    for b in range(len(n)):
        assert np.array_equal(tbl[b, :n[b]], rt[b, :n[b]]), b
        assert np.array_equal(msk[b, :n[b]], rm[b, :n[b]]), b
        if len(got) > 4:  # rows 8..15
            assert np.array_equal(got[4][b, :n[b]], ref[4][b, :n[b]]), b
        assert bool((tbl[b, n[b]:] == -7).all())  # nothing written past the count


@pytest.mark.parametrize("q,topk,L", [(1, 100, 500), (2, 512, 8192), (4, 1000, 50000), (8, 2048, 131072),
                                     (12, 1024, 131072), (16, 512, 70000)])
def test_planner_matches_oracle(q, topk, L):
    """Rows 9..16 use two mask words and chunks of 16384 microblocks (the
    131072-token and 70000-token contexts span two and two chunks)."""
    p = make_sparse(name="pl", B=3, q=q, Hq=q, Hkv=1, D=64, L=L, topk_blocks=2, seed=q)
    bt = p.meta["block_table"].numpy()
    sel = make_selection(3, q, L, topk, seed=11 + q, past_end=2).numpy()
    got = _gpu_plan(sel, bt, bt.shape[1], 0)
    ref = oracle.select_to_entries(sel, bt, bt.shape[1], 0, with_hi=True)
    _same(got, ref if q > 8 else ref[:4])
    assert got[3] == 4 and ref[3] == 2  # FP8KV_STATUS_BAD_ENTRIES; two positions ignored


def test_planner_long_context_many_chunks():
    q, topk, L = 4, 3000, 200000  # 50000 logical microblocks: several shared-memory chunks
    bt = np.random.default_rng(0).permutation(60000)[:50000].reshape(1, -1).astype(np.int32)
    bt = np.repeat(bt, 2, axis=0)
    sel = make_selection(2, q, L, topk, seed=3).numpy()
    _same(_gpu_plan(sel, bt, 50000, 7), oracle.select_to_entries(sel, bt, 50000, 7))


def test_planner_empty_and_unused():
    sel = np.full((2, 3, 40), -1, dtype=np.int32)
    sel[1, 2, 5] = 9
    bt = np.arange(40, dtype=np.int32).reshape(2, 20)
    got = _gpu_plan(sel, bt, 20, 99)
    _same(got, oracle.select_to_entries(sel, bt, 20, 99))
    assert got[2].tolist() == [0, 8] and got[3] == 0


def test_planner_feeds_sparse_attention():
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem

    q, L, topk = 4, 131072, 2048
    p = make_sparse(name="pl", B=4, q=q, Hq=24, Hkv=2, D=128, L=L, topk_blocks=2, seed=17)
    bt = p.meta["block_table"].numpy()
    sel = make_selection(4, q, L, topk, seed=5).numpy()
    tbl, msk, n, st = _gpu_plan(sel, bt, bt.shape[1], 0)
    assert st == 0
    stride = tbl.shape[1]
    tbl = np.where(np.arange(stride)[None, :] < n[:, None], tbl, 0).astype(np.int32)
    msk = np.where(np.arange(stride)[None, :] < n[:, None], msk, 0).astype(np.uint32)
    p2 = dataclasses.replace(p, entry_tbl=torch.from_numpy(tbl), entry_mask=torch.from_numpy(msk.view(np.int32)),
                             n_entries=torch.from_numpy(n.astype(np.int32)))
    dp = DeviceProblem(p2)
    out = dp.run()
    torch.cuda.synchronize()
    rt, rm, rn, _ = oracle.select_to_entries(sel, bt, bt.shape[1], 0, entry_stride=stride)
    p3 = dataclasses.replace(p, entry_tbl=torch.from_numpy(rt), entry_mask=torch.from_numpy(rm.view(np.int32)),
                             n_entries=torch.from_numpy(rn))
    compare(out.float().cpu().numpy(), oracle.attention(p3), what="planner -> sparse attention")
    assert dp.status() == 0


def test_planner_feeds_sparse_attention_12_rows():
    """12 query rows (masks in two words) from selections to attention."""
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem

    q, L, topk = 12, 32768, 512
    p = make_sparse(name="pl", B=2, q=q, Hq=24, Hkv=2, D=128, L=L, topk_blocks=2, seed=19)
    bt = p.meta["block_table"].numpy()
    sel = make_selection(2, q, L, topk, seed=6).numpy()
    tbl, msk, n, st, msk_hi = _gpu_plan(sel, bt, bt.shape[1], 0)
    assert st == 0
    stride = tbl.shape[1]
    live = np.arange(stride)[None, :] < n[:, None]
    tbl = np.where(live, tbl, 0).astype(np.int32)
    msk = np.where(live, msk, 0).astype(np.uint32)
    msk_hi = np.where(live, msk_hi, 0).astype(np.uint32)
    p2 = dataclasses.replace(p, entry_tbl=torch.from_numpy(tbl), entry_mask=torch.from_numpy(msk.view(np.int32)),
                             entry_mask_hi=torch.from_numpy(msk_hi.view(np.int32)),
                             n_entries=torch.from_numpy(n.astype(np.int32)))
    dp = DeviceProblem(p2)
    out = dp.run()
    torch.cuda.synchronize()
    rt, rm, rn, _, rh = oracle.select_to_entries(sel, bt, bt.shape[1], 0, entry_stride=stride, with_hi=True)
    p3 = dataclasses.replace(p, entry_tbl=torch.from_numpy(rt), entry_mask=torch.from_numpy(rm.view(np.int32)),
                             entry_mask_hi=torch.from_numpy(rh.view(np.int32)), n_entries=torch.from_numpy(rn))
    compare(out.float().cpu().numpy(), oracle.attention(p3), what="planner -> sparse attention, 12 rows")
    assert dp.status() == 0
