"""Context parallelism: one GPU per rank, each holding a shard of the context.

The pages' decode context parallelism ("Qualify calibrated E4M3 and disk PLE
with QSA DCP2"): every rank runs the split kernel on its own pages and
exposes, per query vector, an FP32 output and a base-2 LSE
(``fp8kv_attn_combine_lse``); one exchange then merges the ranks, either an
all-gather of the LSEs plus a reduce-scatter of the weighted outputs, or one
all-to-all of (output, LSE) head slices followed by a local merge.  Either
way each rank ends with the fp16 output of its share of the query heads.

This module is host logic only: which pages a rank holds, and the
collectives around the library's merge kernels (``fp8kv_attn_merge``,
``fp8kv_attn_merge_scale``).  The merge steps are the library calls unless a
caller passes its own (the CPU tests of the exchange pattern do).
"""

from __future__ import annotations

from typing import Callable, Optional

import torch
import torch.distributed as dist


def shard_pages(block_table: torch.Tensor, row_len: torch.Tensor, page_size: int, num_ranks: int, rank: int):
    """Rank ``rank``'s shard of a dense problem: the block-table columns
    [rank * pp, (rank + 1) * pp), pp = ceil(columns / num_ranks), with every
    row length measured from the shard's first token and clamped to it.
    Returns (block_table [B][pp] int32, row_len [B][q] int32, max_kv_len)."""
    B, P = block_table.shape
    pp = (P + num_ranks - 1) // num_ranks
    lo = rank * pp
    bt = block_table[:, lo:lo + pp]
    if bt.shape[1] < pp:  # columns past the table: no row length reaches them
        pad = torch.zeros(B, pp - bt.shape[1], dtype=block_table.dtype, device=block_table.device)
        bt = torch.cat([bt, pad], dim=1)
    rl = (row_len.to(torch.int64) - lo * page_size).clamp(min=0, max=pp * page_size).to(torch.int32)
    return bt.contiguous(), rl.contiguous(), pp * page_size


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _merge_kernel(outs: torch.Tensor, lses: torch.Tensor, out: torch.Tensor) -> None:
    from . import binding as B

    a = B.make_merge_args(outs=outs, lses=lses, out=out)
    B.fp8kv_attn_merge(a, _stream())


def _scale_kernel(own: torch.Tensor, lses: torch.Tensor, rank: int, scaled: torch.Tensor) -> None:
    from . import binding as B

    a = B.make_merge_args(outs=own.unsqueeze(0), lses=lses, out_f32=scaled)
    a.num_ranks = lses.shape[0]  # the ranks whose LSEs weigh this one
    B.fp8kv_attn_merge_scale(a, rank, _stream())


def _cast_kernel(summed: torch.Tensor, out: torch.Tensor) -> None:
    # one rank of weight 1: the merge kernel converts FP32 to fp16 (RNE)
    from . import binding as B

    zero = torch.zeros((1,) + summed.shape[:-1], dtype=torch.float32, device=summed.device)
    a = B.make_merge_args(outs=summed.unsqueeze(0), lses=zero, out=out)
    B.fp8kv_attn_merge(a, _stream())


def head_slice(num_q_heads: int, num_ranks: int, rank: int) -> slice:
    """The query heads whose merged output rank ``rank`` keeps."""
    if num_q_heads % num_ranks:
        raise ValueError(f"{num_q_heads} query heads do not split over {num_ranks} ranks")
    h = num_q_heads // num_ranks
    return slice(rank * h, (rank + 1) * h)


def merge_a2a(o: torch.Tensor, lse: torch.Tensor, group=None, *,
              merge_fn: Optional[Callable] = None) -> torch.Tensor:
    """All-to-all shape.  o: this rank's FP32 output [B][q][Hq][D], lse its
    base-2 LSE [B][q][Hq].  Head slice r of both goes to rank r, which merges
    the R slices it receives.  Returns fp16 [B][q][Hq/R][D] for this rank's
    heads (``head_slice``)."""
    R = dist.get_world_size(group)
    B_, q, Hq, D = o.shape
    h = Hq // R
    if Hq % R:
        raise ValueError(f"{Hq} query heads do not split over {R} ranks")
    send_o = o.reshape(B_ * q, R, h, D).permute(1, 0, 2, 3).contiguous()  # [dest rank][B*q][h][D]
    send_l = lse.reshape(B_ * q, R, h).permute(1, 0, 2).contiguous()
    recv_o = torch.empty_like(send_o)  # [source rank][B*q][h][D]
    recv_l = torch.empty_like(send_l)
    dist.all_to_all_single(recv_o, send_o, group=group)
    dist.all_to_all_single(recv_l, send_l, group=group)
    out = torch.empty(B_ * q, h, D, dtype=torch.float16, device=o.device)
    (merge_fn or _merge_kernel)(recv_o, recv_l, out)
    return out.view(B_, q, h, D)


def merge_ag_rs(o: torch.Tensor, lse: torch.Tensor, group=None, *,
                scale_fn: Optional[Callable] = None, cast_fn: Optional[Callable] = None) -> torch.Tensor:
    """All-gather + reduce-scatter shape.  The LSEs of all ranks are
    gathered; each rank weights its own output by 2^(lse_own - L); the
    weighted outputs are summed over the ranks by a reduce-scatter that
    leaves each rank its head slice; the FP32 sum becomes fp16.  Returns
    fp16 [B][q][Hq/R][D] for this rank's heads."""
    R = dist.get_world_size(group)
    rank = dist.get_rank(group)
    B_, q, Hq, D = o.shape
    h = Hq // R
    if Hq % R:
        raise ValueError(f"{Hq} query heads do not split over {R} ranks")
    lse_all = torch.empty(R * B_ * q * Hq, dtype=torch.float32, device=o.device)
    dist.all_gather_into_tensor(lse_all, lse.reshape(-1).contiguous(), group=group)
    lse_all = lse_all.view(R, B_ * q * Hq)
    scaled = torch.empty(B_ * q * Hq, D, dtype=torch.float32, device=o.device)
    (scale_fn or _scale_kernel)(o.reshape(B_ * q * Hq, D), lse_all, rank, scaled)
    send = scaled.view(B_ * q, R, h, D).permute(1, 0, 2, 3).contiguous().view(-1)
    recv = torch.empty(B_ * q * h * D, dtype=torch.float32, device=o.device)
    dist.reduce_scatter_tensor(recv, send, op=dist.ReduceOp.SUM, group=group)
    out = torch.empty(B_ * q, h, D, dtype=torch.float16, device=o.device)
    (cast_fn or _cast_kernel)(recv.view(B_ * q * h, D), out.view(B_ * q * h, D))
    return out.view(B_, q, h, D)
