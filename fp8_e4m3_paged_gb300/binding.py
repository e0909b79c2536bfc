"""ctypes binding of libfp8kv_attn.so (the C ABI in include/fp8kv_attn.h).

Argument marshalling only: every step of the attention runs in the library's
CUDA kernels.  Importing this module loads the in-tree shared library and
raises ImportError if it has not been built -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8kv_attn.so")

REVISION = 5
OK = 0
EINVAL = -1
EUNSUPPORTED = -2
EWORKSPACE = -3
EVERSION = -4
ECUDA = -5

MODE_DENSE = 0
MODE_SPARSE_PAGE4 = 1

KV_E4M3 = 0
KV_E5M2 = 1
KV_BF16 = 2

KERNEL_AUTO = 0
KERNEL_GENERIC = 1
KERNEL_TC = 2
KERNEL_TC_SMALL = 3

STATUS_BAD_BLOCK = 0x1
STATUS_BAD_LEN = 0x2
STATUS_BAD_ENTRIES = 0x4
STATUS_TIMEOUT = 0x8

TEST_STALL_PIPELINE = 0x1


class Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "mode", "batch", "q_max", "num_q_heads", "num_kv_heads", "head_dim", "page_size",
        "max_kv_len", "max_blocks", "num_kv_blocks", "num_sms", "num_splits", "kernel", "kv_format",
        "test_flags")]


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "revision", "mode", "batch", "q_max", "num_q_heads", "num_kv_heads", "head_dim",
        "page_size", "max_kv_len", "max_blocks", "num_kv_blocks", "group", "rows",
        "num_splits", "tile_tokens", "kernel")] + [
        ("grid", ctypes.c_int32 * 3),
        ("block_threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
        ("row_chunk", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("partial_offset", ctypes.c_int64), ("ml_offset", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
        ("kv_format", ctypes.c_int32),
        ("test_flags", ctypes.c_int32),
        ("min_part", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 13),
    ]


class Args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("k_stride_block", ctypes.c_int64), ("k_stride_token", ctypes.c_int64),
        ("k_stride_head", ctypes.c_int64),
        ("v_stride_block", ctypes.c_int64), ("v_stride_token", ctypes.c_int64),
        ("v_stride_head", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int64),
        ("row_kv_len", ctypes.c_void_p),
        ("entry_tbl", ctypes.c_void_p), ("entry_mask", ctypes.c_void_p),
        ("n_entries", ctypes.c_void_p), ("entry_stride", ctypes.c_int64),
        ("softmax_scale", ctypes.c_float), ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("k_scale_dev", ctypes.c_void_p), ("v_scale_dev", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("entry_mask_hi", ctypes.c_void_p),
        ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("k_new_stride_req", ctypes.c_int64), ("k_new_stride_token", ctypes.c_int64),
        ("k_new_stride_head", ctypes.c_int64),
        ("v_new_stride_req", ctypes.c_int64), ("v_new_stride_token", ctypes.c_int64),
        ("v_new_stride_head", ctypes.c_int64),
        ("n_new", ctypes.c_int32), ("new_dtype", ctypes.c_int32),
    ]


DTYPE_F16 = 0
DTYPE_BF16 = 1


class CacheWriteArgs(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_kv_blocks", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("k_stride_token", ctypes.c_int64), ("k_stride_head", ctypes.c_int64),
        ("v_stride_token", ctypes.c_int64), ("v_stride_head", ctypes.c_int64),
        ("slot_mapping", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("kc_stride_block", ctypes.c_int64), ("kc_stride_token", ctypes.c_int64),
        ("kc_stride_head", ctypes.c_int64),
        ("vc_stride_block", ctypes.c_int64), ("vc_stride_token", ctypes.c_int64),
        ("vc_stride_head", ctypes.c_int64),
        ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
        ("k_scale_dev", ctypes.c_void_p), ("v_scale_dev", ctypes.c_void_p),
        ("status", ctypes.c_void_p), ("kv_format", ctypes.c_int32),
    ]


MERGE_MAX_RANKS = 64


class MergeArgs(ctypes.Structure):
    _fields_ = [
        ("num_ranks", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("num_vectors", ctypes.c_int64),
        ("outs", ctypes.c_void_p), ("rank_stride_out", ctypes.c_int64),
        ("lses", ctypes.c_void_p), ("rank_stride_lse", ctypes.c_int64),
        ("out", ctypes.c_void_p), ("out_f32", ctypes.c_void_p), ("lse_out", ctypes.c_void_p),
    ]


class SelectArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("q_max", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32), ("null_block", ctypes.c_int32),
        ("sel", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int64),
        ("entry_tbl", ctypes.c_void_p), ("entry_mask", ctypes.c_void_p), ("entry_stride", ctypes.c_int64),
        ("n_entries", ctypes.c_void_p), ("status", ctypes.c_void_p),
        ("entry_mask_hi", ctypes.c_void_p),
    ]


if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m fp8_e4m3_paged_gb300.build_lib` "
        "(the CUDA library is required; there is no CPU fallback)")

lib = ctypes.CDLL(LIB_PATH)
lib.fp8kv_attn_version.restype = ctypes.c_int
lib.fp8kv_attn_version.argtypes = []
lib.fp8kv_attn_strerror.restype = ctypes.c_char_p
lib.fp8kv_attn_strerror.argtypes = [ctypes.c_int]
lib.fp8kv_attn_plan.restype = ctypes.c_int
lib.fp8kv_attn_plan.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(Plan)]
STATIC_SCRATCH_BYTES = 16 << 20

for _n in ("fp8kv_attn_split", "fp8kv_attn_combine", "fp8kv_attn_forward_static"):
    getattr(lib, _n).restype = ctypes.c_int
    getattr(lib, _n).argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Args), ctypes.c_void_p]


lib.fp8kv_attn_combine_lse.restype = ctypes.c_int
lib.fp8kv_attn_combine_lse.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Args), ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]
lib.fp8kv_attn_merge.restype = ctypes.c_int
lib.fp8kv_attn_merge.argtypes = [ctypes.POINTER(MergeArgs), ctypes.c_void_p]
lib.fp8kv_attn_merge_scale.restype = ctypes.c_int
lib.fp8kv_attn_merge_scale.argtypes = [ctypes.POINTER(MergeArgs), ctypes.c_int32, ctypes.c_void_p]
lib.fp8kv_attn_select_to_entries.restype = ctypes.c_int
lib.fp8kv_attn_select_to_entries.argtypes = [ctypes.POINTER(SelectArgs), ctypes.c_void_p]
lib.fp8kv_attn_cache_write.restype = ctypes.c_int
lib.fp8kv_attn_cache_write.argtypes = [ctypes.POINTER(CacheWriteArgs), ctypes.c_void_p]


class Fp8kvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {fp8kv_attn_strerror(code)} ({code})")


def fp8kv_attn_version() -> int:
    return lib.fp8kv_attn_version()


def fp8kv_attn_strerror(code: int) -> str:
    return lib.fp8kv_attn_strerror(code).decode()


def fp8kv_attn_plan(desc: Desc) -> Plan:
    plan = Plan()
    rc = lib.fp8kv_attn_plan(ctypes.byref(desc), ctypes.byref(plan))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_plan")
    return plan


def fp8kv_attn_split(plan: Plan, args: Args, stream: int = 0) -> None:
    rc = lib.fp8kv_attn_split(ctypes.byref(plan), ctypes.byref(args), ctypes.c_void_p(stream))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_split")


def fp8kv_attn_combine(plan: Plan, args: Args, stream: int = 0) -> None:
    rc = lib.fp8kv_attn_combine(ctypes.byref(plan), ctypes.byref(args), ctypes.c_void_p(stream))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_combine")


def fp8kv_attn_forward_static(plan: Plan, args: Args, stream: int = 0) -> None:
    """Split + combine using the library's own device scratch (no workspace)."""
    rc = lib.fp8kv_attn_forward_static(ctypes.byref(plan), ctypes.byref(args), ctypes.c_void_p(stream))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_forward_static")


# ---------------------------------------------------------------- torch glue

def make_desc(*, mode: int, batch: int, q_max: int, num_q_heads: int, num_kv_heads: int,
              head_dim: int, page_size: int, max_kv_len: int, max_blocks: int,
              num_kv_blocks: int, num_sms: int = 0, num_splits: int = 0, kernel: int = 0,
              kv_format: int = KV_E4M3, test_flags: int = 0) -> Desc:
    return Desc(mode, batch, q_max, num_q_heads, num_kv_heads, head_dim, page_size,
                max_kv_len, max_blocks, num_kv_blocks, num_sms, num_splits, kernel, kv_format,
                test_flags)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def make_args(*, q, k_cache, v_cache, out, workspace, softmax_scale: float,
              k_scale: float = 1.0, v_scale: float = 1.0,
              block_table=None, row_kv_len=None,
              entry_tbl=None, entry_mask=None, n_entries=None,
              k_scale_dev=None, v_scale_dev=None, entry_mask_hi=None, k_new=None, v_new=None) -> Args:
    """Fill an Args struct from torch CUDA tensors.

    k_cache / v_cache: uint8 tensors indexed [block][slot][kv_head][d] (any
    strides with d contiguous); q / out: fp16 [B][q_max][Hq][D] contiguous;
    workspace: a uint8 tensor of at least plan.workspace_bytes bytes.
    k_new / v_new (fused write of a verify step's new tokens): fp16 or bf16
    [B][n_new][Hkv][D], d contiguous.
    """
    a = Args()
    a.q = _ptr(q)
    a.k_cache = _ptr(k_cache)
    a.v_cache = _ptr(v_cache)
    ks = k_cache.stride()
    vs = v_cache.stride()
    eb_k = k_cache.element_size()
    eb_v = v_cache.element_size()
    a.k_stride_block, a.k_stride_token, a.k_stride_head = ks[0] * eb_k, ks[1] * eb_k, ks[2] * eb_k
    a.v_stride_block, a.v_stride_token, a.v_stride_head = vs[0] * eb_v, vs[1] * eb_v, vs[2] * eb_v
    if block_table is not None:
        a.block_table = _ptr(block_table)
        a.block_table_stride = block_table.stride(0)
    a.row_kv_len = _ptr(row_kv_len)
    if entry_tbl is not None:
        a.entry_tbl = _ptr(entry_tbl)
        a.entry_stride = entry_tbl.stride(0)
    a.entry_mask = _ptr(entry_mask)
    a.entry_mask_hi = _ptr(entry_mask_hi)
    a.n_entries = _ptr(n_entries)
    a.softmax_scale = float(softmax_scale)
    a.k_scale = float(k_scale)
    a.v_scale = float(v_scale)
    a.k_scale_dev = _ptr(k_scale_dev)
    a.v_scale_dev = _ptr(v_scale_dev)
    a.out = _ptr(out)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if k_new is not None:
        import torch

        a.k_new, a.v_new = _ptr(k_new), _ptr(v_new)
        a.k_new_stride_req, a.k_new_stride_token, a.k_new_stride_head = k_new.stride()[:3]
        a.v_new_stride_req, a.v_new_stride_token, a.v_new_stride_head = v_new.stride()[:3]
        a.n_new = k_new.shape[1]
        a.new_dtype = DTYPE_F16 if k_new.dtype == torch.float16 else DTYPE_BF16
    return a


@dataclass
class Call:
    """A planned split + combine over fixed device buffers (graph friendly)."""
    plan: Plan
    args: Args

    def split(self, stream: int) -> None:
        fp8kv_attn_split(self.plan, self.args, stream)

    def combine(self, stream: int) -> None:
        fp8kv_attn_combine(self.plan, self.args, stream)

    def run(self, stream: int) -> None:
        self.split(stream)
        self.combine(stream)


def fp8kv_attn_cache_write(args: CacheWriteArgs, stream: int = 0) -> None:
    rc = lib.fp8kv_attn_cache_write(ctypes.byref(args), ctypes.c_void_p(stream))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_cache_write")


def make_cache_write_args(*, k, v, slot_mapping, k_cache, v_cache, page_size: int,
                          k_scale: float = 1.0, v_scale: float = 1.0, k_scale_dev=None,
                          v_scale_dev=None, status=None, kv_format: int = KV_E4M3) -> CacheWriteArgs:
    """Fill a CacheWriteArgs struct from torch CUDA tensors.

    k / v: float16 or bfloat16 [N][Hkv][D] (d contiguous); slot_mapping:
    int64 [N]; k_cache / v_cache: uint8 [blocks][page_size][Hkv][D] views
    (d contiguous); status: optional int32 tensor of one element."""
    import torch

    a = CacheWriteArgs()
    N, Hkv, D = k.shape
    a.num_tokens, a.num_kv_heads, a.head_dim = N, Hkv, D
    a.page_size = page_size
    a.num_kv_blocks = k_cache.shape[0]
    a.dtype = DTYPE_F16 if k.dtype == torch.float16 else DTYPE_BF16
    a.k, a.v = _ptr(k), _ptr(v)
    a.k_stride_token, a.k_stride_head = k.stride(0), k.stride(1)
    a.v_stride_token, a.v_stride_head = v.stride(0), v.stride(1)
    a.slot_mapping = _ptr(slot_mapping)
    a.k_cache, a.v_cache = _ptr(k_cache), _ptr(v_cache)
    a.kc_stride_block, a.kc_stride_token, a.kc_stride_head = k_cache.stride()[:3]
    a.vc_stride_block, a.vc_stride_token, a.vc_stride_head = v_cache.stride()[:3]
    a.k_scale, a.v_scale = float(k_scale), float(v_scale)
    a.k_scale_dev, a.v_scale_dev = _ptr(k_scale_dev), _ptr(v_scale_dev)
    a.status = _ptr(status)
    a.kv_format = kv_format
    return a


def fp8kv_attn_combine_lse(plan: Plan, args: Args, out_f32, lse, stream: int = 0) -> None:
    """Combine one rank's shard into FP32 output [B][q][Hq][D] and base-2 LSE [B][q][Hq]."""
    rc = lib.fp8kv_attn_combine_lse(ctypes.byref(plan), ctypes.byref(args), _ptr(out_f32), _ptr(lse),
                                    ctypes.c_void_p(stream))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_combine_lse")


def make_merge_args(*, outs, lses, out=None, out_f32=None, lse_out=None) -> MergeArgs:
    """outs: FP32 [R][n..][D]; lses: FP32 [R][n..] (torch CUDA tensors; the
    vector dimensions are flattened, the rank dimension may be strided)."""
    R, D = outs.shape[0], outs.shape[-1]
    a = MergeArgs()
    a.num_ranks, a.head_dim = R, D
    a.num_vectors = lses[0].numel() if R > 0 else 0
    a.outs, a.rank_stride_out = _ptr(outs), outs.stride(0)
    a.lses, a.rank_stride_lse = _ptr(lses), lses.stride(0)
    a.out, a.out_f32, a.lse_out = _ptr(out), _ptr(out_f32), _ptr(lse_out)
    return a


def fp8kv_attn_merge(args: MergeArgs, stream: int = 0) -> None:
    rc = lib.fp8kv_attn_merge(ctypes.byref(args), ctypes.c_void_p(stream))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_merge")


def fp8kv_attn_merge_scale(args: MergeArgs, rank: int, stream: int = 0) -> None:
    rc = lib.fp8kv_attn_merge_scale(ctypes.byref(args), rank, ctypes.c_void_p(stream))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_merge_scale")


def make_select_args(*, sel, block_table, max_blocks: int, null_block: int, entry_tbl, entry_mask,
                     n_entries, status=None, entry_mask_hi=None) -> SelectArgs:
    """sel: int32 [B][q][topk]; block_table: int32 [B][>= max_blocks];
    entry_tbl / entry_mask (/ entry_mask_hi for q > 8): int32 [B][stride]
    (the mask tensors hold the uint32 bit patterns); n_entries: int32 [B]
    (torch CUDA tensors)."""
    a = SelectArgs()
    a.batch, a.q_max, a.topk = sel.shape
    a.max_blocks, a.null_block = max_blocks, null_block
    a.sel = _ptr(sel)
    a.block_table, a.block_table_stride = _ptr(block_table), block_table.stride(0)
    a.entry_tbl, a.entry_mask, a.entry_stride = _ptr(entry_tbl), _ptr(entry_mask), entry_tbl.stride(0)
    a.n_entries, a.status = _ptr(n_entries), _ptr(status)
    a.entry_mask_hi = _ptr(entry_mask_hi)
    return a


def fp8kv_attn_select_to_entries(args: SelectArgs, stream: int = 0) -> None:
    rc = lib.fp8kv_attn_select_to_entries(ctypes.byref(args), ctypes.c_void_p(stream))
    if rc != OK:
        raise Fp8kvError(rc, "fp8kv_attn_select_to_entries")
