"""Acceptance check of a GPU fp16 output against the FP64 oracle.

Per output tensor: relative L2 <= 5e-4 (all exact zeros when the reference is
all zero), every element within 4 fp16 ulps of the reference value, where
ulp16(x) = 2^(max(floor(log2|x|), -14) - 10) (2^-24 at and below the fp16
subnormal range), and no NaN or Inf.

FP32 floor (only where a caller passes ``cond``): an output element that
cancels to a value far below the magnitude of its terms cannot be resolved by
any FP32-state evaluation to 4 fp16 ulps of the (tiny) result.  For such
elements the per-element bound becomes
    4 ulp16(ref) + COND_U32 * 2^-24 * cond,
cond = v_scale * sum_j w_j |V_j[d]| (the oracle's attention_abs), i.e. the
standard forward error bound of a weighted sum evaluated with unit roundoff
2^-24, with COND_U32 roundings (exponent, probability split, PV accumulation,
partition combine, normalisation).  Where cond ~ |ref| the extra term is
below 0.01 fp16 ulp, so the strict bound is unchanged there.

Logit term (where a caller also passes ``cond_qk``): an FP32 logit cannot be
better than its dot product, and with outliers in K a logit of magnitude 30
(natural units) already moves its weight by ~30 ulps when rounded once.  Both
kernel families form each logit as a TwoSum-compensated sum of partial dot
products of at most 16 exact products (FMA chunks of 8 on the CUDA cores, one
K16 MMA per part on the tensor cores), whose a priori error is gamma_16 ~ 16u
times the partial's sum of |products|.  With cond_qk = sum_j w_j a_j |v_j -
out| (the oracle's attention_logit_cond, a_j the scaled sum of |q_d k_jd|),
the bound gains COND_QK * 2^-24 * cond_qk: the first-order output change
under logit errors |dz_j| <= COND_QK 2^-24 a_j.
"""

import numpy as np

REL_L2 = 5e-4
MAX_ULPS = 4.0
COND_U32 = 16.0
COND_QK = 16.0


def ulp16(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, e, -14.0)
    return np.exp2(np.maximum(e, -14.0) - 10.0)


def compare(gpu, ref, *, what="output", cond=None, cond_qk=None, max_floor_elements=None):
    """Check gpu against ref (see the module docstring).

    cond: apply the FP32 floor to every element; cond_qk (with cond): add the
    logit term to it.  max_floor_elements (with cond): hold every element to
    the strict bound except at most this many, which must still lie within
    the FP32-floor bound; their count is returned as stats["floor_elements"]."""
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
    if cond is None:
        bound = MAX_ULPS * u
    else:
        c = np.asarray(cond, dtype=np.float64)
        bound = MAX_ULPS * u + COND_U32 * 2.0 ** -24 * c
        if cond_qk is not None:
            bound = bound + COND_QK * 2.0 ** -24 * np.asarray(cond_qk, dtype=np.float64)
        stats["max_frac_of_bound"] = float((np.abs(diff) / bound).max()) if diff.size else 0.0
        if max_floor_elements is not None:
            floor = np.abs(diff) > MAX_ULPS * u
            stats["floor_elements"] = int(floor.sum())
            assert stats["floor_elements"] <= max_floor_elements, (
                f"{what}: {stats['floor_elements']} elements beyond {MAX_ULPS} fp16 ulps "
                f"(at most {max_floor_elements} may need the FP32 floor)")
    bad = np.abs(diff) > bound
    if bad.any():
        i = np.unravel_index(np.argmax(np.abs(diff) / bound), diff.shape)
        extra = "" if cond is None else f" cond {float(np.asarray(cond)[i]):.3e}"
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of bound; worst {ulps[i]:.2f} fp16 ulps "
                             f"at {i}: gpu {g[i]!r} ref {r[i]!r}{extra}")
    return stats
