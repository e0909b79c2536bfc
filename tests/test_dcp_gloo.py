"""Context-parallel exchange on CPU ranks (gloo, world sizes 2 and 4).

Each rank takes its page shard of one dense problem (``dcp.shard_pages``),
gets its shard's FP32 output and base-2 LSE from the oracle, and runs both
exchange shapes of ``fp8_e4m3_paged_gb300.dcp`` -- all-to-all, and
all-gather + reduce-scatter -- with the merge steps supplied by the test
(the oracle's merge on the host) in place of the library's kernels.  Every
rank's fp16 result must match the oracle's attention over the whole context
for the query heads that rank keeps.  No GPU is used.
"""

import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    from synth import make_dense

    return make_dense(name="dcp", B=2, q=3, Hq=4, Hkv=2, D=64, page_size=16, lens=(600, 1000), seed=21)


def _worker(rank, ws, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import oracle
        from fp8_e4m3_paged_gb300 import dcp
        from tests._check import compare

        p = _problem()
        bt, rl, mkl = dcp.shard_pages(p.block_table, p.row_len, p.page_size, ws, rank)
        shard = dataclasses.replace(p, block_table=bt, row_len=rl, max_kv_len=mkl)
        o64, l64 = oracle.attention_lse(shard, threads=1)
        o = torch.from_numpy(o64).to(torch.float32)
        lse = torch.from_numpy(l64).to(torch.float32)
        ref = oracle.attention(p, threads=1)[:, :, dcp.head_slice(p.Hq, ws, rank)]

        def merge_fn(outs, lses, out):  # the oracle's merge in place of fp8kv_attn_merge
            m, _ = oracle.merge(outs.double().numpy(), lses.double().numpy())
            out.copy_(torch.from_numpy(m).to(torch.float16))

        def scale_fn(own, lses, r, scaled):  # this rank's weight from the gathered LSEs
            _, L = oracle.merge(np.zeros((lses.shape[0],) + tuple(lses.shape[1:]) + (1,)), lses.double().numpy())
            w = np.where(np.isneginf(L), 0.0, np.exp2(lses[r].double().numpy() - L))
            scaled.copy_(torch.from_numpy(w[:, None] * own.double().numpy()).to(torch.float32))

        def cast_fn(summed, out):
            out.copy_(summed.to(torch.float16))

        a2a = dcp.merge_a2a(o, lse, merge_fn=merge_fn)
        agrs = dcp.merge_ag_rs(o, lse, scale_fn=scale_fn, cast_fn=cast_fn)
        compare(a2a.float().numpy(), ref, what=f"a2a rank {rank}")
        compare(agrs.float().numpy(), ref, what=f"ag+rs rank {rank}")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws", [2, 4])
def test_exchange_shapes_on_cpu_ranks(ws):
    import oracle

    oracle.build()  # once, before the ranks start
    mp.spawn(_worker, args=(ws, _free_port()), nprocs=ws, join=True)


def test_shards_cover_the_context_once():
    from fp8_e4m3_paged_gb300 import dcp

    p = _problem()
    for R in (1, 2, 3, 4, 7):
        total = torch.zeros_like(p.row_len)
        seen = []
        for r in range(R):
            bt, rl, mkl = dcp.shard_pages(p.block_table, p.row_len, p.page_size, R, r)
            assert bt.shape[1] * p.page_size == mkl and bool((rl <= mkl).all()) and bool((rl >= 0).all())
            total += rl
            seen.append(bt)
        assert torch.equal(total, p.row_len)
        # the shards' pages, in order, are the request's block table
        cat = torch.cat(seen, 1)[:, :p.block_table.shape[1]]
        assert torch.equal(cat, p.block_table)
