"""Paged attention over an FP8 E4M3 KV cache for one GB300 (sm_103a).

The computation is the C-ABI library ``libfp8kv_attn.so`` (``include/fp8kv_attn.h``);
this package only builds it (``build_lib``), binds it (``binding``), moves a
problem's tensors to the GPU (``device_problem``) and runs the context-parallel
exchange around the library's merge kernels (``dcp``).  The
binding is imported on first use of any of its names, so that ``build_lib``
works before the library exists; using the API without the library raises
ImportError.
"""

_EXPORTS = (
    "Args", "Call", "Desc", "Fp8kvError", "Plan",
    "fp8kv_attn_combine", "fp8kv_attn_forward_static", "fp8kv_attn_plan", "fp8kv_attn_split",
    "fp8kv_attn_strerror", "fp8kv_attn_version", "make_args", "make_desc",
    # cache write, context-parallel merge, grouped planner
    "CacheWriteArgs", "MergeArgs", "SelectArgs",
    "fp8kv_attn_cache_write", "fp8kv_attn_combine_lse", "fp8kv_attn_merge", "fp8kv_attn_merge_scale",
    "fp8kv_attn_select_to_entries", "make_cache_write_args", "make_merge_args", "make_select_args",
    "KV_E4M3", "KV_E5M2",
)


def __getattr__(name):
    if name in _EXPORTS:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
