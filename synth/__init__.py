"""Seeded synthetic inputs for FP8 E4M3 paged attention.

This package only *makes data*: query vectors, E4M3 key/value page pools,
block tables, per-row live lengths, QSA microblock tables with visibility
masks, token-ID selections, and new fp16/bf16 K/V rows with their cache
slots.  It contains none
of the attention or quantisation arithmetic, and it is the only code shared
by the CPU oracle (``oracle/``) and the CUDA library
(``fp8_e4m3_paged_gb300``).
"""

from .workloads import (  # noqa: F401
    Problem,
    CONFIGS,
    make_problem,
    make_dense,
    make_sparse,
    quantize_e4m3,
    attended_kv_bytes,
)
from .cache_write import CacheWriteProblem, make_cache_write  # noqa: F401
from .selection import make_selection  # noqa: F401
