"""GPU: context-parallel ranks simulated on one GPU, merged by the kernels.

Each simulated rank holds a page shard of one dense problem
(``dcp.shard_pages``) and runs the library's split kernel and
``fp8kv_attn_combine_lse`` on it, one rank after another on one stream (no
rank waits for another).  The ranks' (FP32 output, base-2 LSE) pairs are then
merged by ``fp8kv_attn_merge`` (the all-to-all shape's local merge) and by
``fp8kv_attn_merge_scale`` + a sum over ranks + the fp16 cast (the
all-gather + reduce-scatter shape, the sum standing in for the collective).
Both must match the oracle's attention over the whole context (tests/_check:
rel L2 <= 5e-4, <= 4 fp16 ulps).  Also: one rank reproduces the ordinary
combine bit for bit, the LSE matches the oracle's, and ranks whose shard
shows a row nothing are harmless.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from synth import make_dense, make_problem
from tests._check import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_e4m3_paged_gb300 import build_lib

    build_lib.build()
    oracle.build()


def _rank_outputs(p, R, kernel=0):
    """(o [R][B][q][Hq][D], lse [R][B][q][Hq]) of the R simulated ranks."""
    from fp8_e4m3_paged_gb300 import binding as B
    from fp8_e4m3_paged_gb300 import dcp
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem

    outs, lses = [], []
    for r in range(R):
        bt, rl, mkl = dcp.shard_pages(p.block_table, p.row_len, p.page_size, R, r)
        shard = dataclasses.replace(p, block_table=bt, row_len=rl, max_kv_len=mkl)
        dp = DeviceProblem(shard, kernel=kernel)
        o = torch.empty(p.B, p.q, p.Hq, p.D, dtype=torch.float32, device="cuda")
        lse = torch.empty(p.B, p.q, p.Hq, dtype=torch.float32, device="cuda")
        st = torch.cuda.current_stream().cuda_stream
        dp.calls[0].split(st)
        B.fp8kv_attn_combine_lse(dp.plan, dp.calls[0].args, o, lse, st)
        torch.cuda.synchronize()
        assert dp.status() == 0
        outs.append(o)
        lses.append(lse)
    return torch.stack(outs), torch.stack(lses)


def _merge(o, lse):
    from fp8_e4m3_paged_gb300 import binding as B

    R = o.shape[0]
    out = torch.empty(o.shape[1:], dtype=torch.float16, device="cuda")
    lse_out = torch.empty(lse.shape[1:], dtype=torch.float32, device="cuda")
    a = B.make_merge_args(outs=o.reshape(R, -1, o.shape[-1]), lses=lse.reshape(R, -1), out=out, lse_out=lse_out)
    B.fp8kv_attn_merge(a, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out, lse_out


def _merge_ag_rs(o, lse):
    from fp8_e4m3_paged_gb300 import binding as B

    R, D = o.shape[0], o.shape[-1]
    st = torch.cuda.current_stream().cuda_stream
    lses = lse.reshape(R, -1)
    total = torch.zeros(lses.shape[1], D, dtype=torch.float32, device="cuda")
    for r in range(R):
        scaled = torch.empty_like(total)
        a = B.make_merge_args(outs=o[r].reshape(1, -1, D), lses=lses, out_f32=scaled)
        a.num_ranks = R
        B.fp8kv_attn_merge_scale(a, r, st)
        total += scaled  # the reduce-scatter's sum
    out = torch.empty(total.shape, dtype=torch.float16, device="cuda")
    a = B.make_merge_args(outs=total.unsqueeze(0), lses=torch.zeros(1, total.shape[0], device="cuda"), out=out)
    B.fp8kv_attn_merge(a, st)
    torch.cuda.synchronize()
    return out.view(o.shape[1:])


def _decode_batch():
    return make_dense(name="dcp_decode", B=8, q=1, Hq=32, Hkv=8, D=128, page_size=16,
                      lens=(512, 1000, 2048, 3000, 4096, 700, 8192, 16384), seed=41)


@pytest.mark.parametrize("R", [2, 3, 4])
@pytest.mark.parametrize("name", ["c2", "c3_64k", "decode"])
def test_ranks_merge_to_whole(name, R):
    p = _decode_batch() if name == "decode" else make_problem(name)
    ref = oracle.attention(p)
    o, lse = _rank_outputs(p, R)
    out, _ = _merge(o, lse)
    compare(out.float().cpu().numpy(), ref, what=f"{name} merged over {R} ranks")
    out2 = _merge_ag_rs(o, lse)
    compare(out2.float().cpu().numpy(), ref, what=f"{name} scaled + summed over {R} ranks")


@pytest.mark.parametrize("kernel", [1, 2])
def test_one_rank_is_the_ordinary_combine(kernel):
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem

    p = make_problem("c2")
    dp = DeviceProblem(p, kernel=kernel)
    plain = dp.run().clone()
    torch.cuda.synchronize()
    o, lse = _rank_outputs(p, 1, kernel=kernel)
    out, lse_m = _merge(o, lse)
    assert torch.equal(out, plain)
    assert torch.equal(lse_m, lse[0])


def test_lse_matches_oracle():
    p = _decode_batch()
    _, lse_ref = oracle.attention_lse(p)
    _, lse = _rank_outputs(p, 1)
    got = lse[0].cpu().double().numpy()
    assert np.all(np.abs(got - lse_ref) <= 1e-5 * np.maximum(1.0, np.abs(lse_ref)))


def test_empty_shards_and_dead_rows():
    p = _decode_batch()
    rl = p.row_len.clone()
    rl[3, 0] = 0  # a dead row
    p = dataclasses.replace(p, row_len=rl)
    R = 8  # short requests leave most shards empty
    o, lse = _rank_outputs(p, R)
    assert bool(torch.isneginf(lse[:, 3, 0]).all())
    out, lse_m = _merge(o, lse)
    assert bool((out[3, 0] == 0).all()) and bool(torch.isneginf(lse_m[3, 0]).all())
    compare(out.float().cpu().numpy(), oracle.attention(p), what="merged with empty shards")
