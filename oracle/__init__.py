"""FP64 CPU oracle for paged attention over an FP8 E4M3 KV cache.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use this package; the library never does.

The computation lives in ``fp8kv_oracle.cpp`` (plain C++17, double precision,
``std::thread`` over query rows).  This module compiles it with g++ and wraps
it with ctypes.  Inputs are ``synth.Problem`` objects (CPU tensors).

Parity status of each exported function (what pins it, in ``tests/``):
  e4m3 table          format definition closed form + torch float8_e4m3fn
  e5m2 table          format definition (binary16 upper byte) + torch
                      float8_e5m2, all 256 codes
  e4m3 encode         round trip of every code, exact midpoints (ties to
                      even), nearest on both sides of each midpoint,
                      saturation, signed zero, torch float8_e4m3fn in range
  attention_lse       merging the (out, lse) of disjoint context shards gives
                      the full attention and its LSE; one-token and
                      equal-logit closed forms of the LSE
  merge               one rank is the identity, an empty rank changes
                      nothing, shards of one problem merge to the whole
  select_to_entries   hand-worked golden case, invariants (every selection
                      visible exactly once, no other bit, increasing order,
                      null padding to x8), and sparse attention over the
                      result equal to a direct per-row softmax over the
                      selected tokens
  cache write         slot placement, skipped and out-of-range slots,
                      strides, decode(write(x)) within half a quantum of
                      x / scale, power-of-two scales against the encoder
  fp16 decode         all 65536 codes against numpy float16
  attention           exact-rational evaluation on tiny inputs, closed forms
                      (single token, constant keys, two tokens), invariants
                      (page permutation, split count, sparse order/padding,
                      all-visible sparse == dense causal), planted mistakes
  attention_split     equals attention within 1e-13 (split-count invariance)
  row_weights         sum to 1, two-token logistic closed form
  attention_abs       equals attention when every V byte is non-negative;
                      bounds |attention| elementwise
  attention_logit_cond
                      two-token closed form w1 w2 (a1 + a2) |v1 - v2|, zero
                      for one token and for equal values, and a bound on
                      the measured output change under relative logit
                      perturbations (k_scale scaled by 1 +- eps)
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8kv_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")

CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-pthread", "-Wall"]


def lib_path(plant: int = 0) -> str:
    name = "liboracle.so" if plant == 0 else f"liboracle_plant{plant}.so"
    return os.path.join(_BUILD, name)


def build(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle (plant != 0 builds a deliberately broken variant)."""
    out = lib_path(plant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", *CXXFLAGS, f"-DORC_PLANT={plant}", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class OrcProblem(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int), ("B", ctypes.c_int), ("q", ctypes.c_int),
        ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("q_bits", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("k_stride", ctypes.c_int64 * 3), ("v_stride", ctypes.c_int64 * 3),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int64),
        ("row_len", ctypes.c_void_p),
        ("entry_tbl", ctypes.c_void_p), ("entry_mask", ctypes.c_void_p),
        ("n_entries", ctypes.c_void_p), ("entry_stride", ctypes.c_int64),
        ("softmax_scale", ctypes.c_double), ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double), ("kv_format", ctypes.c_int),
        ("entry_mask_hi", ctypes.c_void_p),
    ]


_libs = {}


def load(plant: int = 0) -> ctypes.CDLL:
    if plant in _libs:
        return _libs[plant]
    path = build(plant)
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(OrcProblem)
    lib.orc_e4m3.restype = ctypes.c_double
    lib.orc_e4m3.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_table.argtypes = [ctypes.c_void_p]
    lib.orc_e5m2.restype = ctypes.c_double
    lib.orc_e5m2.argtypes = [ctypes.c_uint8]
    lib.orc_e5m2_table.argtypes = [ctypes.c_void_p]
    lib.orc_f16.restype = ctypes.c_double
    lib.orc_f16.argtypes = [ctypes.c_uint16]
    lib.orc_attention.argtypes = [P, ctypes.c_void_p, ctypes.c_int]
    lib.orc_attention_items.argtypes = [P, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
    lib.orc_attention_split.argtypes = [P, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
    lib.orc_attention_abs.argtypes = [P, ctypes.c_void_p, ctypes.c_int]
    lib.orc_attention_logit_cond.argtypes = [P, ctypes.c_void_p, ctypes.c_int]
    lib.orc_row_weights.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
    lib.orc_attention_lse.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.orc_merge.restype = None
    lib.orc_merge.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_void_p]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
    lib.orc_bf16.restype = ctypes.c_double
    lib.orc_bf16.argtypes = [ctypes.c_uint16]
    vp = ctypes.c_void_p
    lib.orc_cache_write.restype = ctypes.c_int
    lib.orc_cache_write.argtypes = [ctypes.c_int] * 6 + [vp, vp, vp, vp, vp, ctypes.c_float, ctypes.c_float,
                                                         vp, vp, vp, vp]
    lib.orc_cache_write_fmt.restype = ctypes.c_int
    lib.orc_cache_write_fmt.argtypes = lib.orc_cache_write.argtypes + [ctypes.c_int]
    lib.orc_e5m2_encode.restype = ctypes.c_uint8
    lib.orc_e5m2_encode.argtypes = [ctypes.c_float]
    _libs[plant] = lib
    return lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


class _Pinned:
    """Keeps the CPU tensors referenced by an OrcProblem alive."""

    def __init__(self, p, k_cache=None, v_cache=None, row_len=None):
        kc = p.k_cache if k_cache is None else k_cache
        vc = p.v_cache if v_cache is None else v_cache
        for t in (kc, vc):
            assert t.device.type == "cpu" and t.dtype == torch.uint8
        self.keep = []
        s = OrcProblem()
        s.mode = 0 if p.mode == "dense" else 1
        s.B, s.q, s.Hq, s.Hkv, s.D = p.B, p.q, p.Hq, p.Hkv, p.D
        s.page_size = p.page_size
        qb = p.q_fp16.contiguous().view(torch.int16)
        self.keep.append(qb)
        s.q_bits = qb.data_ptr()
        s.k_cache = kc.data_ptr()
        s.v_cache = vc.data_ptr()
        ks, vs = kc.stride(), vc.stride()
        s.k_stride[:] = [ks[0], ks[1], ks[2]]
        s.v_stride[:] = [vs[0], vs[1], vs[2]]
        self.keep += [kc, vc]
        if p.mode == "dense":
            bt = p.block_table.contiguous()
            rl = (p.row_len if row_len is None else torch.as_tensor(row_len, dtype=torch.int32)).contiguous()
            self.keep += [bt, rl]
            s.block_table = bt.data_ptr()
            s.bt_stride = bt.shape[1]
            s.row_len = rl.data_ptr()
        else:
            et = p.entry_tbl.contiguous()
            em = p.entry_mask.contiguous()
            ne = p.n_entries.contiguous()
            self.keep += [et, em, ne]
            s.entry_tbl = et.data_ptr()
            s.entry_mask = em.data_ptr()
            s.n_entries = ne.data_ptr()
            s.entry_stride = et.shape[1]
            hi = getattr(p, "entry_mask_hi", None)
            if hi is not None:
                hi = hi.contiguous()
                self.keep.append(hi)
                s.entry_mask_hi = hi.data_ptr()
        s.softmax_scale = p.softmax_scale
        s.k_scale = p.k_scale
        s.v_scale = p.v_scale
        s.kv_format = {"e4m3": 0, "e5m2": 1, "bf16": 2}[getattr(p, "kv_format", "e4m3")]
        self.s = s


def e4m3_table(plant: int = 0) -> np.ndarray:
    out = np.zeros(256, dtype=np.float64)
    load(plant).orc_e4m3_table(out.ctypes.data)
    return out


def e5m2_table(plant: int = 0) -> np.ndarray:
    out = np.zeros(256, dtype=np.float64)
    load(plant).orc_e5m2_table(out.ctypes.data)
    return out


def f16_value(bits: int, plant: int = 0) -> float:
    return load(plant).orc_f16(bits)


def attention(p, threads: Optional[int] = None, plant: int = 0, **over) -> np.ndarray:
    """Full output [B][q][Hq][D] in float64.  ``over`` may replace k_cache,
    v_cache or row_len with other CPU tensors of the same layout."""
    pin = _Pinned(p, **over)
    out = np.zeros((p.B, p.q, p.Hq, p.D), dtype=np.float64)
    rc = load(plant).orc_attention(ctypes.byref(pin.s), out.ctypes.data, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return out


def attention_items(p, items, threads: Optional[int] = None, plant: int = 0, **over) -> np.ndarray:
    """Outputs of the listed (b, r, h) triples only: [n][D] float64."""
    pin = _Pinned(p, **over)
    it = np.ascontiguousarray(np.asarray(items, dtype=np.int32).reshape(-1, 3))
    out = np.zeros((it.shape[0], p.D), dtype=np.float64)
    rc = load(plant).orc_attention_items(ctypes.byref(pin.s), it.ctypes.data, it.shape[0],
                                         out.ctypes.data, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the problem or an item")
    return out


def attention_abs(p, threads: Optional[int] = None, plant: int = 0, **over) -> np.ndarray:
    """Per-element condition v_scale * sum_j w_j |dec(V_j[d])| ([B][q][Hq][D])."""
    pin = _Pinned(p, **over)
    out = np.zeros((p.B, p.q, p.Hq, p.D), dtype=np.float64)
    rc = load(plant).orc_attention_abs(ctypes.byref(pin.s), out.ctypes.data, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return out


def attention_logit_cond(p, threads: Optional[int] = None, plant: int = 0, **over) -> np.ndarray:
    """Per-element logit condition sum_j w_j a_j |v_j[d] - out[d]| ([B][q][Hq][D]),
    a_j = |softmax_scale k_scale| sum_d |q[d] dec(K_j[d])|: logit errors
    |dz_j| <= eps a_j move the output by at most eps times this (first order)."""
    pin = _Pinned(p, **over)
    out = np.zeros((p.B, p.q, p.Hq, p.D), dtype=np.float64)
    rc = load(plant).orc_attention_logit_cond(ctypes.byref(pin.s), out.ctypes.data, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return out


def attention_split(p, num_splits: int, threads: Optional[int] = None, plant: int = 0, **over) -> np.ndarray:
    pin = _Pinned(p, **over)
    out = np.zeros((p.B, p.q, p.Hq, p.D), dtype=np.float64)
    rc = load(plant).orc_attention_split(ctypes.byref(pin.s), num_splits, out.ctypes.data,
                                         threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return out


def row_weights(p, b: int, r: int, h: int, plant: int = 0, **over) -> np.ndarray:
    pin = _Pinned(p, **over)
    cap = 1 << 22
    buf = np.zeros(cap, dtype=np.float64)
    n = load(plant).orc_row_weights(ctypes.byref(pin.s), b, r, h, buf.ctypes.data, cap)
    return buf[:n].copy()


def e4m3_encode(y, plant: int = 0) -> np.ndarray:
    """E4M3 bytes of float32 values (round to nearest even, saturating)."""
    lib = load(plant)
    a = np.asarray(y, dtype=np.float32).reshape(-1)
    return np.array([lib.orc_e4m3_encode(float(x)) for x in a], dtype=np.uint8).reshape(np.shape(y))


def e5m2_encode(y, plant: int = 0) -> np.ndarray:
    """E5M2 bytes of float32 values (round to nearest even, saturating to +-57344)."""
    lib = load(plant)
    a = np.asarray(y, dtype=np.float32).reshape(-1)
    return np.array([lib.orc_e5m2_encode(float(x)) for x in a], dtype=np.uint8).reshape(np.shape(y))


def bf16_value(bits: int, plant: int = 0) -> float:
    return load(plant).orc_bf16(bits)


def cache_write(k, v, slot_mapping, k_cache, v_cache, k_scale: float, v_scale: float,
                page_size: int, plant: int = 0, kv_format: str = "e4m3") -> int:
    """Write new tokens into E4M3 (or, kv_format "e5m2", E5M2) cache tensors
    in place (CPU).

    k, v: float16 or bfloat16 [N][Hkv][D] (any strides, d contiguous);
    slot_mapping: int64 [N] (slot = block * page_size + offset, < 0 = skip);
    k_cache, v_cache: uint8 [blocks][page_size][Hkv][D] views (any strides,
    d contiguous), modified in place.  Returns the number of slots whose
    block lies outside the cache (skipped)."""
    assert k.dtype == v.dtype and k.dtype in (torch.float16, torch.bfloat16)
    for t in (k, v, k_cache, v_cache):
        assert t.device.type == "cpu" and t.stride(-1) == 1
    N, Hkv, D = k.shape
    dtype = 0 if k.dtype == torch.float16 else 1
    kb, vb = k.view(torch.int16), v.view(torch.int16)
    sm = slot_mapping.to(torch.int64).contiguous()
    kes = np.array(kb.stride()[:2], dtype=np.int64)
    ves = np.array(vb.stride()[:2], dtype=np.int64)
    kbs = np.array(k_cache.stride()[:3], dtype=np.int64)
    vbs = np.array(v_cache.stride()[:3], dtype=np.int64)
    return load(plant).orc_cache_write_fmt(
        N, Hkv, D, page_size, k_cache.shape[0], dtype, kb.data_ptr(), vb.data_ptr(),
        kes.ctypes.data, ves.ctypes.data, sm.data_ptr(), float(k_scale), float(v_scale),
        k_cache.data_ptr(), v_cache.data_ptr(), kbs.ctypes.data, vbs.ctypes.data,
        {"e4m3": 0, "e5m2": 1}[kv_format])


def attention_lse(p, threads: Optional[int] = None, plant: int = 0, **over):
    """(out [B][q][Hq][D], lse [B][q][Hq]) in float64; lse is base 2."""
    pin = _Pinned(p, **over)
    out = np.zeros((p.B, p.q, p.Hq, p.D), dtype=np.float64)
    lse = np.zeros((p.B, p.q, p.Hq), dtype=np.float64)
    rc = load(plant).orc_attention_lse(ctypes.byref(pin.s), out.ctypes.data, lse.ctypes.data,
                                       threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return out, lse


def merge(outs, lses, plant: int = 0):
    """Merge R ranks' outputs [R][..][D] and base-2 LSEs [R][..]."""
    o = np.ascontiguousarray(np.asarray(outs, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(lses, dtype=np.float64))
    R, D = o.shape[0], o.shape[-1]
    n = int(np.prod(l.shape[1:]))
    m = np.zeros(o.shape[1:], dtype=np.float64)
    lm = np.zeros(l.shape[1:], dtype=np.float64)
    load(plant).orc_merge(R, n, D, o.ctypes.data, l.ctypes.data, m.ctypes.data, lm.ctypes.data)
    return m, lm


def select_to_entries(sel, block_table, max_blocks: int, null_block: int, entry_stride: Optional[int] = None,
                      with_hi: bool = False):
    """The grouped planner, from its definition ("Qualify calibrated E4M3 and
    disk PLE with QSA DCP2", commit "grouped page4 null-block padding").

    sel: int [B][q][topk] token positions of each request's query rows (< 0 =
    unused; positions at or past 4 * max_blocks are ignored and counted).
    For each request: the distinct four-token logical microblocks m = t // 4
    any row selected, in increasing order; entry_tbl = block_table[b][m];
    bit 4r + t % 4 of entry_mask set iff row r < 8 selected token t (rows
    8..15: bit 4(r - 8) + t % 4 of the second word entry_mask_hi); then null
    entries (null_block, mask 0) up to a multiple of 8.
    Returns (entry_tbl [B][stride] int32, entry_mask [B][stride] uint32,
    n_entries [B] int32, n_ignored), and entry_mask_hi [B][stride] uint32
    after them when with_hi."""
    sel = np.asarray(sel, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    B, q, _ = sel.shape
    ignored = 0
    per_req = []
    for b in range(B):
        toks = []
        for r in range(q):
            for t in sel[b, r]:
                if t < 0:
                    continue
                if t >= 4 * max_blocks:
                    ignored += 1
                    continue
                toks.append((int(t), r))
        mbs = np.unique(np.array([t // 4 for t, _ in toks], dtype=np.int64))  # sorted, distinct
        masks = {int(m): 0 for m in mbs}
        for t, r in toks:
            masks[t // 4] |= 1 << (4 * r + t % 4)
        ent = [(int(bt[b, m]), masks[int(m)]) for m in mbs]
        ent += [(null_block, 0)] * ((-len(ent)) % 8)
        per_req.append(ent)
    stride = entry_stride or max(8, max(len(e) for e in per_req))
    tbl = np.zeros((B, stride), dtype=np.int32)
    msk = np.zeros((B, stride), dtype=np.uint32)
    msk_hi = np.zeros((B, stride), dtype=np.uint32)
    n = np.zeros(B, dtype=np.int32)
    for b, ent in enumerate(per_req):
        assert len(ent) <= stride, "entries exceed the stride"
        n[b] = len(ent)
        for e, (t, m) in enumerate(ent):
            tbl[b, e] = t
            msk[b, e] = m & 0xFFFFFFFF
            msk_hi[b, e] = m >> 32
    if with_hi:
        return tbl, msk, n, ignored, msk_hi
    assert q <= 8 or not msk_hi.any(), "rows 8..15 need with_hi"
    return tbl, msk, n, ignored
