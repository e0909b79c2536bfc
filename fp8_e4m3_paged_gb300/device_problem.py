"""Device buffers, plan and argument block for one attention problem.

Marshalling only: copies a problem's CPU tensors (see ``synth.Problem``: any
object with the same fields works) to the GPU once, plans the call, allocates
the output and the FP32 workspace, and fills the C-ABI argument struct.  The
calls themselves run in the library's kernels on the caller's stream.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class DeviceProblem:
    def __init__(self, p, *, device: str = "cuda", num_splits: int = 0, num_sms: int = 0,
                 kv_copies: int = 1, device_scales: bool = False, k_cache=None, v_cache=None,
                 kernel: int = 0, test_flags: int = 0, k_new=None, v_new=None):
        self.p = p
        dev = torch.device(device)
        self.q = p.q_fp16.to(dev).contiguous()
        kc = p.k_cache if k_cache is None else k_cache
        vc = p.v_cache if v_cache is None else v_cache
        # KV copies let a benchmark rotate through more bytes than the L2 holds.
        self.k_caches = [kc.to(dev) for _ in range(kv_copies)]
        self.v_caches = [vc.to(dev) for _ in range(kv_copies)]
        self.out = torch.zeros_like(self.q)
        # fused write of a verify step's new tokens ([B][n_new][Hkv][D] fp16/bf16)
        self.k_new = None if k_new is None else k_new.to(dev).contiguous()
        self.v_new = None if v_new is None else v_new.to(dev).contiguous()
        if p.mode == "dense":
            self.block_table = p.block_table.to(dev).contiguous()
            self.row_len = p.row_len.to(dev).contiguous()
            self.entry_tbl = self.entry_mask = self.n_entries = self.entry_mask_hi = None
            mode = B.MODE_DENSE
            max_blocks = int(p.block_table.shape[1])
            max_kv_len = int(p.max_kv_len)
        else:
            self.block_table = self.row_len = None
            self.entry_tbl = p.entry_tbl.to(dev).contiguous()
            self.entry_mask = p.entry_mask.to(dev).contiguous()
            hi = getattr(p, "entry_mask_hi", None)
            self.entry_mask_hi = None if hi is None else hi.to(dev).contiguous()
            self.n_entries = p.n_entries.to(dev).contiguous()
            mode = B.MODE_SPARSE_PAGE4
            max_blocks = int(p.entry_tbl.shape[1])
            max_kv_len = int(p.max_kv_len)
        self.desc = B.make_desc(
            mode=mode, batch=p.B, q_max=p.q, num_q_heads=p.Hq, num_kv_heads=p.Hkv,
            head_dim=p.D, page_size=p.page_size, max_kv_len=max_kv_len, max_blocks=max_blocks,
            num_kv_blocks=int(kc.shape[0]), num_sms=num_sms, num_splits=num_splits, kernel=kernel, test_flags=test_flags,
            kv_format={"e4m3": B.KV_E4M3, "e5m2": B.KV_E5M2, "bf16": B.KV_BF16}[getattr(p, "kv_format", "e4m3")])
        self.plan = B.fp8kv_attn_plan(self.desc)
        self.workspace = torch.zeros(int(self.plan.workspace_bytes), dtype=torch.uint8, device=dev)
        self.k_scale_dev = self.v_scale_dev = None
        if device_scales:
            self.k_scale_dev = torch.tensor([p.k_scale], dtype=torch.float32, device=dev)
            self.v_scale_dev = torch.tensor([p.v_scale], dtype=torch.float32, device=dev)
        self.calls = [self._make_call(i) for i in range(kv_copies)]

    def _make_call(self, i: int) -> B.Call:
        p = self.p
        args = B.make_args(
            q=self.q, k_cache=self.k_caches[i], v_cache=self.v_caches[i], out=self.out,
            workspace=self.workspace, softmax_scale=p.softmax_scale,
            k_scale=0.0 if self.k_scale_dev is not None else p.k_scale,
            v_scale=0.0 if self.v_scale_dev is not None else p.v_scale,
            block_table=self.block_table, row_kv_len=self.row_len,
            entry_tbl=self.entry_tbl, entry_mask=self.entry_mask, n_entries=self.n_entries,
            entry_mask_hi=self.entry_mask_hi, k_new=self.k_new, v_new=self.v_new,
            k_scale_dev=self.k_scale_dev, v_scale_dev=self.v_scale_dev)
        return B.Call(self.plan, args)

    def run(self, copy: int = 0, stream: Optional[int] = None) -> torch.Tensor:
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        self.calls[copy].run(s)
        return self.out

    def status(self) -> int:
        return int(self.workspace[:4].view(torch.int32).item())

    def clear_status(self) -> None:
        self.workspace[:4].zero_()
