"""Acceptance check of a GPU fp16 output against the FP64 oracle.

Per output tensor: relative L2 <= 5e-4 (all exact zeros when the reference is
all zero), every element within 4 fp16 ulps of the reference value, where
ulp16(x) = 2^(max(floor(log2|x|), -14) - 10) (2^-24 at and below the fp16
subnormal range), and no NaN or Inf.
"""

import numpy as np

REL_L2 = 5e-4
MAX_ULPS = 4.0


def ulp16(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, e, -14.0)
    return np.exp2(np.maximum(e, -14.0) - 10.0)


def compare(gpu, ref, *, what="output"):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    stats = {"n": int(g.size)}
    bad = ~np.isfinite(g)
    stats["nonfinite"] = int(bad.sum())
    assert stats["nonfinite"] == 0, f"{what}: {stats['nonfinite']} NaN/Inf values"
    nr = float(np.linalg.norm(r))
    diff = g - r
    if nr == 0.0:
        assert np.all(g == 0.0), f"{what}: reference is all zero but output is not"
        stats["rel_l2"] = 0.0
    else:
        stats["rel_l2"] = float(np.linalg.norm(diff) / nr)
    u = ulp16(r)
    ulps = np.abs(diff) / u
    stats["max_ulps"] = float(ulps.max()) if ulps.size else 0.0
    assert stats["rel_l2"] <= REL_L2, f"{what}: rel L2 {stats['rel_l2']:.3e} > {REL_L2}"
    if stats["max_ulps"] > MAX_ULPS:
        i = np.unravel_index(np.argmax(ulps), ulps.shape)
        raise AssertionError(f"{what}: {stats['max_ulps']:.2f} fp16 ulps at {i}: gpu {g[i]!r} ref {r[i]!r}")
    return stats
