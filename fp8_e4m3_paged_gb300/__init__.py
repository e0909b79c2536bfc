"""Paged attention over an FP8 E4M3 KV cache for one GB300 (sm_103a).

The computation is the C-ABI library ``libfp8kv_attn.so`` (``include/fp8kv_attn.h``);
this package only builds it (``build_lib``) and binds it (``binding``).  The
binding is imported on first use of any of its names, so that ``build_lib``
works before the library exists; using the API without the library raises
ImportError.
"""

_EXPORTS = (
    "Args", "Call", "Desc", "Fp8kvError", "Plan",
    "fp8kv_attn_combine", "fp8kv_attn_forward_static", "fp8kv_attn_plan", "fp8kv_attn_split",
    "fp8kv_attn_strerror", "fp8kv_attn_version", "make_args", "make_desc",
)


def __getattr__(name):
    if name in _EXPORTS:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
