"""Host-side tests of the C ABI (no GPU needed).

The library is built in-tree with nvcc (cross-compiling for sm_103a), loaded,
and checked to export every function include/fp8kv_attn.h declares.  Planning
is pure host code and is exercised directly; split/combine are called only
with arguments the host-side validation rejects, so no kernel is launched.
"""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8kv_attn.h")


@pytest.fixture(scope="module")
def B():
    from fp8_e4m3_paged_gb300 import build_lib

    build_lib.build()
    from fp8_e4m3_paged_gb300 import binding

    return binding


def _declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8kv_attn_\w+)\s*\(", txt)))


def test_exports_every_declared_symbol(B):
    names = _declared_functions()
    assert {"fp8kv_attn_plan", "fp8kv_attn_split", "fp8kv_attn_combine"} <= set(names)
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_strerror(B):
    assert B.fp8kv_attn_version() == B.REVISION
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(B.fp8kv_attn_strerror(code), str) and B.fp8kv_attn_strerror(code)


def _desc(B, **kw):
    base = dict(mode=B.MODE_DENSE, batch=1, q_max=8, num_q_heads=6, num_kv_heads=1, head_dim=256,
                page_size=1728, max_kv_len=131072, max_blocks=76, num_kv_blocks=77, num_sms=152)
    base.update(kw)
    return B.make_desc(**base)


def test_plan_shape_and_workspace(B):
    p = B.fp8kv_attn_plan(_desc(B))
    assert p.revision == B.REVISION
    assert p.group == 6 and p.rows == 48
    S = p.num_splits
    assert 1 <= S
    nvec = 1 * 1 * S * 48
    assert p.partial_offset >= 4
    assert p.ml_offset >= p.partial_offset + nvec * 256 * 4
    assert p.workspace_bytes >= p.ml_offset + nvec * 8
    assert p.workspace_bytes % 256 == 0
    assert p.grid[0] * p.grid[1] * p.grid[2] >= 1


def test_plan_split_override_and_batch0(B):
    p = B.fp8kv_attn_plan(_desc(B, num_splits=7))
    assert p.num_splits == 7
    p0 = B.fp8kv_attn_plan(_desc(B, batch=0))
    assert p0.workspace_bytes >= 4


@pytest.mark.parametrize("kernel,cap", [(3, 128), (2, 32), (1, None)])
def test_plan_partition_length_cap(B, kernel, cap):
    """A batch with more (request, KV head) units than SMs is split by
    length: the longest request's partitions hold at most `cap` tiles of 64
    tokens (the small-group kernel drains each pair of tiles into a
    compensated sum, so its cap is four times the others')."""
    L = 46000
    p = B.fp8kv_attn_plan(_desc(B, batch=64, q_max=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                                max_kv_len=L, max_blocks=(L + 15) // 16, num_kv_blocks=4608, kernel=kernel))
    assert p.kernel == kernel
    if cap is None:
        return
    tiles = -(-L // 64)
    assert p.num_splits == -(-tiles // cap)
    assert p.min_part == 16 * 64


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), -2),
    (dict(q_max=17), -2),
    (dict(q_max=0), -1),
    (dict(num_q_heads=5, num_kv_heads=2), -1),
    (dict(page_size=0), -1),
    (dict(max_blocks=10), -1),
    (dict(num_kv_blocks=0), -1),
    (dict(mode=7), -1),
    (dict(mode=1, page_size=16), -2),
    (dict(mode=1, page_size=4, q_max=17), -2),
    (dict(batch=-1), -1),
    (dict(num_splits=-3), -1),
])
def test_plan_rejects(B, kw, code):
    with pytest.raises(B.Fp8kvError) as ei:
        B.fp8kv_attn_plan(_desc(B, **kw))
    assert ei.value.code == code


def _fake_args(B, plan, **kw):
    a = B.Args()
    fake = 1 << 20  # 16-byte aligned non-null values; never dereferenced on the host
    a.q = a.k_cache = a.v_cache = a.out = fake
    a.k_stride_block = a.v_stride_block = 1728 * 256
    a.k_stride_token = a.v_stride_token = 256
    a.k_stride_head = a.v_stride_head = 256
    a.block_table = a.row_kv_len = fake
    a.block_table_stride = plan.max_blocks
    a.softmax_scale, a.k_scale, a.v_scale = 0.0625, 1.0, 1.0
    a.workspace = 1 << 24
    a.workspace_bytes = plan.workspace_bytes
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1),
    (dict(k_cache=(1 << 20) + 8), -1),
    (dict(k_stride_token=250), -1),
    (dict(block_table=None), -1),
    (dict(workspace=(1 << 24) + 16), -1),
    (dict(softmax_scale=float("nan")), -1),
    (dict(k_scale=float("inf")), -1),
])
def test_launch_validation(B, kw, code):
    plan = B.fp8kv_attn_plan(_desc(B))
    a = _fake_args(B, plan, **kw)
    for fn in (B.lib.fp8kv_attn_split, B.lib.fp8kv_attn_combine):
        assert fn(ctypes.byref(plan), ctypes.byref(a), None) == code


def test_sparse_rows_past_8_need_the_second_mask_words(B):
    """A sparse plan with 9..16 query rows is accepted; its launch needs
    entry_mask_hi (rows 8..15), checked on the host before any CUDA call."""
    plan = B.fp8kv_attn_plan(_desc(B, mode=1, page_size=4, q_max=12, max_kv_len=0, max_blocks=64))
    assert plan.q_max == 12 and plan.rows == 12 * plan.group
    fake = 1 << 20
    a = _fake_args(B, plan, block_table=None, row_kv_len=None, entry_tbl=fake, entry_mask=fake,
                   n_entries=fake, entry_stride=64)
    assert B.lib.fp8kv_attn_split(ctypes.byref(plan), ctypes.byref(a), None) == B.EINVAL


def test_bf16_cache_takes_the_cuda_core_kernel(B):
    plan = B.fp8kv_attn_plan(_desc(B, kv_format=B.KV_BF16))
    assert plan.kernel == 1 and plan.kv_format == B.KV_BF16
    for k in (2, 3):
        with pytest.raises(B.Fp8kvError) as ei:
            B.fp8kv_attn_plan(_desc(B, kv_format=B.KV_BF16, kernel=k))
        assert ei.value.code == -2
    with pytest.raises(B.Fp8kvError):
        B.fp8kv_attn_plan(_desc(B, kv_format=3))


@pytest.mark.parametrize("kw,plan_kw", [
    (dict(n_new=-1), {}),
    (dict(n_new=131073), {}),                                   # more than max_kv_len
    (dict(n_new=8, k_new=None), {}),                            # rows missing
    (dict(n_new=8, k_new=(1 << 20) + 8), {}),                   # misaligned
    (dict(n_new=8, k_new_stride_token=100), {}),                # stride not a multiple of 8
    (dict(n_new=8, new_dtype=2), {}),
    (dict(n_new=8), dict(kv_format=2)),                         # bf16 cache: nothing to quantise to
    (dict(n_new=8, k_scale=0.0), {}),
])
def test_fused_write_validation(B, kw, plan_kw):
    plan = B.fp8kv_attn_plan(_desc(B, **plan_kw))
    fake = 1 << 20
    base = dict(k_new=fake, v_new=fake, k_new_stride_req=8 * 256, k_new_stride_token=256, k_new_stride_head=256,
                v_new_stride_req=8 * 256, v_new_stride_token=256, v_new_stride_head=256, new_dtype=0)
    base.update(kw)
    a = _fake_args(B, plan, **base)
    assert B.lib.fp8kv_attn_split(ctypes.byref(plan), ctypes.byref(a), None) == B.EINVAL


def test_fused_write_needs_dense_mode(B):
    plan = B.fp8kv_attn_plan(_desc(B, mode=1, page_size=4, q_max=4, max_kv_len=0, max_blocks=64))
    fake = 1 << 20
    a = _fake_args(B, plan, block_table=None, row_kv_len=None, entry_tbl=fake, entry_mask=fake, n_entries=fake,
                   entry_stride=64, n_new=4, k_new=fake, v_new=fake)
    assert B.lib.fp8kv_attn_split(ctypes.byref(plan), ctypes.byref(a), None) == B.EINVAL


def test_launch_workspace_and_revision(B):
    plan = B.fp8kv_attn_plan(_desc(B))
    a = _fake_args(B, plan, workspace_bytes=plan.workspace_bytes - 1)
    assert B.lib.fp8kv_attn_split(ctypes.byref(plan), ctypes.byref(a), None) == B.EWORKSPACE
    a = _fake_args(B, plan)
    stale = B.Plan.from_buffer_copy(plan)
    stale.revision = B.REVISION + 1
    assert B.lib.fp8kv_attn_split(ctypes.byref(stale), ctypes.byref(a), None) == B.EVERSION
    assert B.lib.fp8kv_attn_combine(ctypes.byref(stale), ctypes.byref(a), None) == B.EVERSION


def test_batch0_launch_is_noop(B):
    plan = B.fp8kv_attn_plan(_desc(B, batch=0))
    a = B.Args()
    a.workspace = 1 << 24
    a.workspace_bytes = plan.workspace_bytes
    assert B.lib.fp8kv_attn_split(ctypes.byref(plan), ctypes.byref(a), None) == 0
    assert B.lib.fp8kv_attn_combine(ctypes.byref(plan), ctypes.byref(a), None) == 0


# ------------------------------------------------------------------ cache write (host validation only)

def _cw(B, **kw):
    a = B.CacheWriteArgs()
    a.num_tokens, a.num_kv_heads, a.head_dim, a.page_size, a.num_kv_blocks, a.dtype = 4, 2, 128, 16, 8, 0
    # aligned but never dereferenced: every call below is rejected on the host
    a.k = a.v = a.k_cache = a.v_cache = a.slot_mapping = 0x10000
    a.k_stride_token, a.k_stride_head = 256, 128
    a.v_stride_token, a.v_stride_head = 256, 128
    a.kc_stride_block, a.kc_stride_token, a.kc_stride_head = 4096, 256, 128
    a.vc_stride_block, a.vc_stride_token, a.vc_stride_head = 4096, 256, 128
    a.k_scale = a.v_scale = 1.0
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("bad", [
    dict(num_tokens=-1), dict(num_kv_heads=0), dict(head_dim=24), dict(head_dim=0), dict(head_dim=2048),
    dict(page_size=0), dict(num_kv_blocks=0), dict(dtype=2), dict(k=0), dict(slot_mapping=0),
    dict(v_cache=0), dict(k=0x10008), dict(k_stride_token=3), dict(v_stride_head=-8),
    dict(kc_stride_token=8), dict(vc_stride_block=-16), dict(k_scale=0.0), dict(v_scale=float("nan")),
    dict(kv_format=2), dict(kv_format=-1),
])
def test_cache_write_rejects_bad_arguments(B, bad):
    assert B.lib.fp8kv_attn_cache_write(ctypes.byref(_cw(B, **bad)), None) == B.EINVAL


def test_cache_write_empty_and_null(B):
    assert B.lib.fp8kv_attn_cache_write(None, None) == B.EINVAL
    # no tokens: nothing to launch, pointers may be null
    assert B.lib.fp8kv_attn_cache_write(ctypes.byref(_cw(B, num_tokens=0, k=0, v=0)), None) == B.OK


# ------------------------------------------------------------------ grouped planner (host validation only)

def _sel(B, **kw):
    a = B.SelectArgs()
    a.batch, a.q_max, a.topk, a.max_blocks, a.null_block = 2, 4, 16, 100, 0
    a.sel = a.block_table = a.entry_tbl = a.entry_mask = a.n_entries = 0x10000  # never dereferenced
    a.block_table_stride, a.entry_stride = 100, 64
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("bad", [
    dict(batch=-1), dict(q_max=0), dict(q_max=9), dict(q_max=17), dict(topk=-1), dict(max_blocks=0),
    dict(block_table_stride=99), dict(entry_stride=63), dict(sel=0), dict(block_table=0), dict(entry_tbl=0),
    dict(entry_mask=0), dict(n_entries=0),
])
def test_select_to_entries_rejects_bad_arguments(B, bad):
    assert B.lib.fp8kv_attn_select_to_entries(ctypes.byref(_sel(B, **bad)), None) == B.EINVAL


def test_select_to_entries_empty_batch(B):
    assert B.lib.fp8kv_attn_select_to_entries(None, None) == B.EINVAL
    assert B.lib.fp8kv_attn_select_to_entries(ctypes.byref(_sel(B, batch=0, sel=0, n_entries=0)), None) == B.OK


# ------------------------------------------------------------------ merge / combine with LSE (host validation only)

def _mg(B, **kw):
    a = B.MergeArgs()
    a.num_ranks, a.head_dim, a.num_vectors = 2, 128, 16
    a.outs = a.lses = a.out = 0x10000  # never dereferenced: every call below is rejected
    a.rank_stride_out, a.rank_stride_lse = 16 * 128, 16
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("bad", [
    dict(num_ranks=0), dict(num_ranks=65), dict(head_dim=2), dict(head_dim=130), dict(head_dim=2048),
    dict(num_vectors=-1), dict(outs=0), dict(outs=0x10008), dict(lses=0), dict(rank_stride_out=6),
    dict(rank_stride_out=-4), dict(rank_stride_lse=-1), dict(out=0x10004), dict(out=0),
])
def test_merge_rejects_bad_arguments(B, bad):
    assert B.lib.fp8kv_attn_merge(ctypes.byref(_mg(B, **bad)), None) == B.EINVAL


@pytest.mark.parametrize("rank,kw", [(-1, {}), (2, {}), (0, {"out_f32": 0})])
def test_merge_scale_rejects_bad_arguments(B, rank, kw):
    a = _mg(B, out=0, out_f32=0x10000)
    for k, v in kw.items():
        setattr(a, k, v)
    assert B.lib.fp8kv_attn_merge_scale(ctypes.byref(a), rank, None) == B.EINVAL
    # the scale step writes only out_f32
    b = _mg(B, out=0x10000, out_f32=0x10000)
    assert B.lib.fp8kv_attn_merge_scale(ctypes.byref(b), 0, None) == B.EINVAL


def test_merge_with_nothing_to_do(B):
    assert B.lib.fp8kv_attn_merge(None, None) == B.EINVAL
    assert B.lib.fp8kv_attn_merge(ctypes.byref(_mg(B, num_vectors=0, outs=0, lses=0)), None) == B.OK


def test_combine_lse_needs_its_outputs(B):
    plan = B.fp8kv_attn_plan(_desc(B))
    a = B.Args()
    a.q = a.k_cache = a.v_cache = a.block_table = a.row_kv_len = 0x10000
    a.workspace = 0x100000
    a.workspace_bytes = plan.workspace_bytes
    a.block_table_stride = 76
    a.k_stride_block = a.v_stride_block = 1728 * 256
    a.k_stride_token = a.v_stride_token = 256
    a.k_stride_head = a.v_stride_head = 256
    a.softmax_scale, a.k_scale, a.v_scale = 0.0625, 1.0, 1.0
    vp = ctypes.c_void_p
    assert B.lib.fp8kv_attn_combine_lse(ctypes.byref(plan), ctypes.byref(a), None, vp(0x10000), None) == B.EINVAL
    assert B.lib.fp8kv_attn_combine_lse(ctypes.byref(plan), ctypes.byref(a), vp(0x10008), vp(0x10000), None) == B.EINVAL
    assert B.lib.fp8kv_attn_combine_lse(ctypes.byref(plan), ctypes.byref(a), vp(0x10000), None, None) == B.EINVAL


def test_plan_records_the_cache_format(B):
    assert B.fp8kv_attn_plan(_desc(B)).kv_format == B.KV_E4M3
    assert B.fp8kv_attn_plan(_desc(B, kv_format=B.KV_E5M2)).kv_format == B.KV_E5M2
    assert B.fp8kv_attn_plan(_desc(B, kv_format=B.KV_BF16)).kv_format == B.KV_BF16
    for bad in (3, -1):
        with pytest.raises(B.Fp8kvError):
            B.fp8kv_attn_plan(_desc(B, kv_format=bad))


def test_page_division_identity():
    """The split kernels take a token's page as the high word of
    page_div * token with page_div = ceil(2^64 / page_size) (the host writes
    ~0 / page_size + 1).  Lemire, Kaser and Kurz ("Faster remainder by direct
    computation", 2019) prove it exact for every numerator below 2^32 when
    64 >= 32 + ceil(log2(page_size)); checked here on divisors and numerators
    chosen around the multiples where a truncated reciprocal would fail."""
    rng = np.random.default_rng(5)
    divisors = list(range(2, 300)) + [1728, 3296, 4099, 65536, 1000003, 2**31 - 1]
    divisors += [int(x) for x in rng.integers(2, 2**31, 200)]
    for d in divisors:
        c = (2**64 - 1) // d + 1
        ns = [0, 1, d - 1, d, d + 1, 2**31 - 1, 2**32 - 1]
        ns += [k * d + e for k in (2, 3, 1000, (2**32 - 1) // d) for e in (-1, 0, 1)]
        ns += [int(x) for x in rng.integers(0, 2**32, 50)]
        for n in ns:
            if 0 <= n < 2**32:
                assert (c * n) >> 64 == n // d, (d, n)
