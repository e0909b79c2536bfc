"""Seeded synthetic workloads for paged attention over an FP8 E4M3 KV cache.

Everything here is *input construction*: Gaussian draws, E4M3 quantisation of
those draws (``torch.float8_e4m3fn``, round-to-nearest-even after clamping to
the finite range), page-pool layout with a seeded block permutation, poisoned
unused slots, causal live lengths and the QSA microblock selection.  No
attention arithmetic lives here.

Workload recipes (all on the CPU; Gaussian and outlier draws come from
numpy's PCG64 so that x86 and Arm hosts build identical bytes, permutations
and uniform draws from a seeded ``torch.Generator``; seeds 101..105 for the
five named configurations are a free choice of this project):

* ``c1``  one request, q=2 verify rows, Hq=6/Hkv=1, D=256, context 1024,
  page size 16, 64 pages randomly permuted; K,V ~ N(0,1) quantised with a
  per-tensor scale max|x|/448; Q fp16 ~ N(0,1); softmax scale 1/16.
* ``c2``  one request, q=8, Hq=6/Hkv=1, D=256, context 8192 in pages of 3296
  tokens (the last page partial); the stored bytes are e4m3(N(0,1)) and the
  scales are k_scale=0.37, v_scale=1.9.
* ``c3_64k`` / ``c3_128k`` / ``c3_256k``  one request, q=8, Hq=6/Hkv=1,
  D=256, page size 1728, pages relocated by a seeded permutation, values as c1.
* ``c4``  64 independent decode requests, q=1, Hq=32/Hkv=8, D=128, page 16,
  lengths round(exp(U(ln 512, ln 65536))); K,V ~ N(0,1) with 1 % of the
  elements multiplied by 20 before the per-tensor scaling.
* ``c5``  QSA sparse verify: 4 requests, q=4, Hq=24/Hkv=2, D=128, context
  131072 as 32768 four-token microblocks per request; every row picks the
  top-512 microblocks (uniform random scores) among those that start before
  its causal limit; the union is sorted and padded to a multiple of 8 with the
  null entry (microblock 0, mask 0); microblock 0 holds poison bytes.

Causal rule for verify rows: row r of a request whose context is L tokens and
which has q live rows sees tokens [0, L - q + 1 + r).

Physical block 0 is always a poisoned block that the dense tables never
reference (sparse tables reference it only through mask-0 padding), and the
unused tail slots of partially filled pages are poisoned too.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

E4M3_MAX = 448.0
E5M2_MAX = 57344.0
FMT_MAX = {"e4m3": E4M3_MAX, "e5m2": E5M2_MAX}
BF16_POISON = {0x7F: (0xC0, 0x7F),  # the NaN poison as bf16: 0x7FC0
               0x7E: (0x7F, 0x7F)}  # the largest-finite poison as bf16: 0x7F7F
POISON_NAN = 0x7F      # E4M3 NaN
POISON_MAX = 0x7E      # E4M3 +448: finite, so only true exclusion survives it


@dataclass
class Problem:
    """One attention call's inputs, all on the CPU.

    Shapes (NHD page layout, D contiguous):
      q_fp16       [B][q][Hq][D]            torch.float16
      k_cache      [num_blocks][P][Hkv][D]  torch.uint8 (E4M3/E5M2 bytes; bf16: [..][2D], LE pairs)
      v_cache      [num_blocks][P][Hkv][D]  torch.uint8
      block_table  [B][max_pages]           torch.int32   (dense)
      row_len      [B][q]                   torch.int32   (dense; 0 = dead row)
      entry_tbl    [B][max_entries]         torch.int32   (sparse)
      entry_mask   [B][max_entries]         torch.int32   (sparse; uint32 bits, rows 0..7)
      entry_mask_hi[B][max_entries]         torch.int32   (sparse, q > 8; rows 8..15)
      n_entries    [B]                      torch.int32   (sparse)
    """

    name: str
    mode: str
    B: int
    q: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    q_fp16: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    softmax_scale: float
    k_scale: float
    v_scale: float
    max_kv_len: int
    block_table: Optional[torch.Tensor] = None
    row_len: Optional[torch.Tensor] = None
    entry_tbl: Optional[torch.Tensor] = None
    entry_mask: Optional[torch.Tensor] = None
    n_entries: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)
    kv_format: str = "e4m3"       # cache format: "e4m3" (E4M3FN), "e5m2" or "bf16"
    entry_mask_hi: Optional[torch.Tensor] = None  # sparse rows 8..15 (q > 8)

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_req(self) -> int:
        if self.mode == "dense":
            return int(self.block_table.shape[1])
        return int(self.entry_tbl.shape[1])

    def strides(self, which: str = "k"):
        """Byte strides (block, token, head) of the K or V page pool."""
        t = self.k_cache if which == "k" else self.v_cache
        s = t.stride()
        return int(s[0]), int(s[1]), int(s[2])


# --------------------------------------------------------------------------
# primitives
# --------------------------------------------------------------------------

def _seed(seed: int, *salt: int) -> int:
    h = seed
    for s in salt:
        h = (h * 1_000_003 + s + 7) % (2**62)
    return h


def _gen(seed: int, *salt: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(_seed(seed, *salt))
    return g


def _f32(x: float) -> float:
    """x rounded to the nearest FP32 value.  The library's interface carries
    softmax_scale, k_scale and v_scale as FP32, so every scale a problem holds
    is an FP32 value: the oracle then computes with exactly the numbers the
    kernels receive."""
    return float(np.float32(x))


def quantize_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    """Quantise fp32 values x/scale to E4M3 bytes (RNE, clamped to +-448)."""
    y = (x / scale).clamp_(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def _poisoned(shape, poison: int, kv_format: str) -> torch.Tensor:
    """A uint8 cache tensor filled with the poison code (bf16: its two-byte
    counterpart, NaN for the NaN poison and the largest finite for 0x7E)."""
    t = torch.full(shape, poison, dtype=torch.uint8)
    if kv_format == "bf16":
        lo, hi = BF16_POISON.get(poison, (poison, poison))
        t[..., 0::2] = lo
        t[..., 1::2] = hi
    return t


def quantize_fp8(x: torch.Tensor, scale: float, kv_format: str = "e4m3") -> torch.Tensor:
    """Cache bytes of x/scale in the given format (torch's RNE conversion
    after clamping to the finite range); bf16: two bytes per element, so the
    last dimension doubles."""
    if kv_format == "e4m3":
        return quantize_e4m3(x, scale)
    if kv_format == "bf16":
        return (x / scale).to(torch.bfloat16).contiguous().view(torch.uint8)
    y = (x / scale).clamp_(-E5M2_MAX, E5M2_MAX)
    return y.to(torch.float8_e5m2).view(torch.uint8)


def _gauss(key: int, shape, outliers: bool) -> torch.Tensor:
    """N(0,1) float32 draws from numpy's PCG64 generator, which gives the
    same values on x86 and Arm hosts (torch's vectorised CPU normal sampler
    does not), so every machine builds byte-identical caches."""
    import numpy as np

    rng = np.random.Generator(np.random.PCG64(key))
    x = torch.from_numpy(rng.standard_normal(size=tuple(shape), dtype=np.float32))
    if outliers:
        sel = torch.from_numpy(rng.random(size=tuple(shape), dtype=np.float32) < 0.01)
        x[sel] *= 20.0
    return x


def causal_row_len(L: int, q_max: int, q_live: Optional[int] = None) -> list:
    """Live lengths of q_max verify rows when q_live rows are live.

    Row r < q_live sees L - q_live + 1 + r tokens; rows >= q_live are dead (0).
    """
    if q_live is None:
        q_live = q_max
    out = []
    for r in range(q_max):
        out.append(L - q_live + 1 + r if r < q_live else 0)
    return out


# --------------------------------------------------------------------------
# dense (paged verify / decode)
# --------------------------------------------------------------------------

def make_dense(
    *,
    name: str = "dense",
    B: int,
    q: int,
    Hq: int,
    Hkv: int,
    D: int,
    page_size: int,
    lens,
    seed: int,
    value_mode: str = "per_tensor",
    outliers: bool = False,
    k_scale: Optional[float] = None,
    v_scale: Optional[float] = None,
    softmax_scale: Optional[float] = None,
    poison: int = POISON_NAN,
    row_len=None,
    extra_pages: int = 0,
    kv_format: str = "e4m3",
) -> Problem:
    """Build a dense paged problem.

    lens[b] is request b's context length L_b (the longest row's view).
    ``row_len`` (optional, [B][q]) overrides the causal live lengths.
    value_mode:
      "per_tensor": x ~ N(0,1) (optional outliers), bytes = e4m3(x / s) with
                    s = max|x| / 448 over the whole K (resp. V) tensor.
      "direct":     bytes = e4m3(x), scales given by k_scale / v_scale.
    ``extra_pages`` appends unreferenced poisoned pages to the pool.
    """
    lens = [int(x) for x in lens]
    assert len(lens) == B
    pages = [max(1, math.ceil(L / page_size)) if L > 0 else 0 for L in lens]
    total_pages = sum(pages)
    num_blocks = 1 + total_pages + extra_pages
    max_pages = max(1, max(pages))

    perm = torch.randperm(total_pages + extra_pages, generator=_gen(seed, 1))
    phys = (1 + perm[:total_pages]).to(torch.int32)
    block_table = torch.zeros((B, max_pages), dtype=torch.int32)
    off = 0
    for b in range(B):
        block_table[b, : pages[b]] = phys[off: off + pages[b]]
        off += pages[b]

    Db = 2 * D if kv_format == "bf16" else D  # bytes of a token row
    k_cache = _poisoned((num_blocks, page_size, Hkv, Db), poison, kv_format)
    v_cache = _poisoned((num_blocks, page_size, Hkv, Db), poison, kv_format)

    def draw(b, which):
        return _gauss(_seed(seed, 2, b, which), (lens[b], Hkv, D), outliers)

    if value_mode == "per_tensor":
        kmax = 0.0
        vmax = 0.0
        for b in range(B):
            if lens[b] == 0:
                continue
            kmax = max(kmax, float(draw(b, 0).abs().max()))
            vmax = max(vmax, float(draw(b, 1).abs().max()))
        ks = _f32(kmax / FMT_MAX.get(kv_format, 1.0)) if kmax > 0 else 1.0
        vs = _f32(vmax / FMT_MAX.get(kv_format, 1.0)) if vmax > 0 else 1.0
        if kv_format == "bf16":  # no quantisation scale
            ks = vs = 1.0
        q_k, q_v = ks, vs
    elif value_mode == "direct":
        ks = _f32(k_scale)
        vs = _f32(v_scale)
        q_k = q_v = 1.0
    else:
        raise ValueError(value_mode)

    for b in range(B):
        L = lens[b]
        if L == 0:
            continue
        kb = quantize_fp8(draw(b, 0), q_k, kv_format)
        vb = quantize_fp8(draw(b, 1), q_v, kv_format)
        full = L // page_size
        if full:
            ids = block_table[b, :full].long()
            k_cache[ids] = kb[: full * page_size].view(full, page_size, Hkv, Db)
            v_cache[ids] = vb[: full * page_size].view(full, page_size, Hkv, Db)
        rem = L - full * page_size
        if rem:
            pid = int(block_table[b, full])
            k_cache[pid, :rem] = kb[full * page_size:]
            v_cache[pid, :rem] = vb[full * page_size:]

    q_fp16 = _gauss(_seed(seed, 3), (B, q, Hq, D), False).to(torch.float16)

    if row_len is None:
        rl = torch.tensor([causal_row_len(lens[b], q) for b in range(B)], dtype=torch.int32)
    else:
        rl = torch.as_tensor(row_len, dtype=torch.int32).reshape(B, q).clone()

    return Problem(
        name=name, mode="dense", B=B, q=q, Hq=Hq, Hkv=Hkv, D=D, page_size=page_size,
        q_fp16=q_fp16, k_cache=k_cache, v_cache=v_cache,
        softmax_scale=_f32(softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(D)),
        k_scale=float(ks), v_scale=float(vs), max_kv_len=max(lens) if lens else 0,
        block_table=block_table, row_len=rl,
        meta={"lens": lens, "seed": seed}, kv_format=kv_format,
    )


# --------------------------------------------------------------------------
# sparse (QSA four-token microblocks with per-row masks)
# --------------------------------------------------------------------------

def make_sparse(
    *,
    name: str = "sparse",
    B: int,
    q: int,
    Hq: int,
    Hkv: int,
    D: int,
    L: int,
    topk_blocks: int,
    seed: int,
    poison: int = POISON_NAN,
    outliers: bool = False,
    softmax_scale: Optional[float] = None,
    pad_to: int = 8,
    kv_format: str = "e4m3",
) -> Problem:
    """Build a QSA sparse problem over 4-token microblocks.

    Mask bit (4*r + t) set <=> query row r sees token t of that entry's
    microblock: rows 0..7 in entry_mask, rows 8..15 (bit 4*(r-8) + t) in
    entry_mask_hi (q > 8 only).  Padding entries are (microblock 0, mask 0).
    """
    assert q <= 16, "two 32-bit mask words hold 16 rows of 4 tokens"
    P = 4
    nmb = math.ceil(L / P)
    total = B * nmb
    num_blocks = 1 + total
    perm = torch.randperm(total, generator=_gen(seed, 11)).to(torch.int64)
    phys_of = (1 + perm).view(B, nmb)

    Db = 2 * D if kv_format == "bf16" else D  # bytes of a token row
    k_cache = _poisoned((num_blocks, P, Hkv, Db), poison, kv_format)
    v_cache = _poisoned((num_blocks, P, Hkv, Db), poison, kv_format)

    def draw(b, which):
        return _gauss(_seed(seed, 12, b, which), (nmb * P, Hkv, D), outliers)

    kmax = max(float(draw(b, 0).abs().max()) for b in range(B))
    vmax = max(float(draw(b, 1).abs().max()) for b in range(B))
    ks = _f32(kmax / FMT_MAX[kv_format]) if kv_format != "bf16" else 1.0
    vs = _f32(vmax / FMT_MAX[kv_format]) if kv_format != "bf16" else 1.0
    for b in range(B):
        ids = phys_of[b]
        k_cache[ids] = quantize_fp8(draw(b, 0), ks, kv_format).view(nmb, P, Hkv, Db)
        v_cache[ids] = quantize_fp8(draw(b, 1), vs, kv_format).view(nmb, P, Hkv, Db)
        # tokens past the context in the last microblock are poisoned
        tail = nmb * P - L
        if tail:
            k_cache[int(ids[-1]), P - tail:] = _poisoned((tail, Hkv, Db), poison, kv_format)
            v_cache[int(ids[-1]), P - tail:] = _poisoned((tail, Hkv, Db), poison, kv_format)

    tbls, masks = [], []
    for b in range(B):
        sel_mask = {}
        for r in range(q):
            n_r = L - q + 1 + r
            elig = math.ceil(n_r / P)
            scores = torch.rand(elig, generator=_gen(seed, 13, b, r))
            k = min(topk_blocks, elig)
            top = torch.topk(scores, k).indices.tolist()
            for m in top:
                bits = 0
                for t in range(P):
                    if m * P + t < n_r:
                        bits |= 1 << (4 * r + t)
                sel_mask[m] = sel_mask.get(m, 0) | bits
        ms = sorted(sel_mask)
        tb = [int(phys_of[b, m]) for m in ms]
        mk = [sel_mask[m] for m in ms]
        while len(tb) % pad_to:
            tb.append(0)
            mk.append(0)
        tbls.append(tb)
        masks.append(mk)
    max_e = max(len(t) for t in tbls)
    max_e = max(max_e, pad_to)
    entry_tbl = torch.zeros((B, max_e), dtype=torch.int32)
    entry_mask = torch.zeros((B, max_e), dtype=torch.int64)
    entry_mask_hi = torch.zeros((B, max_e), dtype=torch.int64)
    n_entries = torch.zeros((B,), dtype=torch.int32)
    for b in range(B):
        n = len(tbls[b])
        entry_tbl[b, :n] = torch.tensor(tbls[b], dtype=torch.int32)
        entry_mask[b, :n] = torch.tensor([m & 0xFFFFFFFF for m in masks[b]], dtype=torch.int64)
        entry_mask_hi[b, :n] = torch.tensor([m >> 32 for m in masks[b]], dtype=torch.int64)
        n_entries[b] = n
    entry_mask = _u32_bits(entry_mask)
    entry_mask_hi = _u32_bits(entry_mask_hi) if q > 8 else None

    q16 = _gauss(_seed(seed, 14), (B, q, Hq, D), False).to(torch.float16)
    return Problem(
        name=name, mode="sparse", B=B, q=q, Hq=Hq, Hkv=Hkv, D=D, page_size=P,
        q_fp16=q16, k_cache=k_cache, v_cache=v_cache,
        softmax_scale=_f32(softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(D)),
        k_scale=float(ks), v_scale=float(vs), max_kv_len=L,
        entry_tbl=entry_tbl, entry_mask=entry_mask, n_entries=n_entries, entry_mask_hi=entry_mask_hi,
        meta={"L": L, "topk_blocks": topk_blocks, "seed": seed,
              # logical microblock -> physical microblock of every request
              "block_table": phys_of.to(torch.int32)},
        kv_format=kv_format,
    )


def _u32_bits(x64: torch.Tensor) -> torch.Tensor:
    """Store unsigned 32-bit patterns in an int32 tensor (same bits)."""
    x = x64.clone()
    x[x >= 2**31] -= 2**32
    return x.to(torch.int32)


def masks_u32(p: Problem) -> torch.Tensor:
    """The sparse masks of rows 0..7 as non-negative int64 values (host-side logic)."""
    return p.entry_mask.to(torch.int64) & 0xFFFFFFFF


def masks_u64(p: Problem) -> torch.Tensor:
    """All 16 rows' sparse bits as int64 values: bit 4r + t for r < 16 (the
    second word shifted up by 32; bit 63 may make the value negative)."""
    lo = p.entry_mask.to(torch.int64) & 0xFFFFFFFF
    if p.entry_mask_hi is None:
        return lo
    return lo | (p.entry_mask_hi.to(torch.int64) << 32)


def masks_any(p: Problem) -> torch.Tensor:
    """Per entry, bit 4k + t set iff some row sees token t (both words folded)."""
    m = masks_u32(p)
    if p.entry_mask_hi is not None:
        m = m | (p.entry_mask_hi.to(torch.int64) & 0xFFFFFFFF)
    return m


# --------------------------------------------------------------------------
# named configurations
# --------------------------------------------------------------------------

def _c4_lens(seed: int, B: int = 64):
    u = torch.rand(B, generator=_gen(seed, 21), dtype=torch.float64)
    lo, hi = math.log(512.0), math.log(65536.0)
    return [int(round(math.exp(lo + (hi - lo) * float(x)))) for x in u]


CONFIGS = {
    "c1": dict(kind="dense", B=1, q=2, Hq=6, Hkv=1, D=256, page_size=16, L=1024,
               seed=101, softmax_scale=1.0 / 16.0, extra_pages=0),
    "c2": dict(kind="dense", B=1, q=8, Hq=6, Hkv=1, D=256, page_size=3296, L=8192,
               seed=102, value_mode="direct", k_scale=0.37, v_scale=1.9),
    "c3_64k": dict(kind="dense", B=1, q=8, Hq=6, Hkv=1, D=256, page_size=1728, L=65536, seed=103),
    "c3_128k": dict(kind="dense", B=1, q=8, Hq=6, Hkv=1, D=256, page_size=1728, L=131072, seed=103),
    "c3_256k": dict(kind="dense", B=1, q=8, Hq=6, Hkv=1, D=256, page_size=1728, L=262144, seed=103),
    "c4": dict(kind="dense", B=64, q=1, Hq=32, Hkv=8, D=128, page_size=16, seed=104, outliers=True),
    "c5": dict(kind="sparse", B=4, q=4, Hq=24, Hkv=2, D=128, L=131072, topk_blocks=512, seed=105),
}


def make_problem(name: str, *, poison: int = POISON_NAN, seed: Optional[int] = None, **over) -> Problem:
    """Build one of the named configurations (optionally overriding fields)."""
    cfg = dict(CONFIGS[name])
    cfg.update(over)
    kind = cfg.pop("kind")
    s = int(seed if seed is not None else cfg.pop("seed"))
    cfg.pop("seed", None)
    if kind == "dense":
        B = cfg["B"]
        if name == "c4" and "lens" not in cfg:
            lens = _c4_lens(s, B)
        else:
            lens = cfg.pop("lens", None) or [cfg["L"]] * B
        cfg.pop("L", None)
        cfg.pop("lens", None)
        return make_dense(name=name, lens=lens, seed=s, poison=poison, **cfg)
    return make_sparse(name=name, seed=s, poison=poison, **cfg)


def attended_kv_bytes(p: Problem) -> int:
    """Attended-KV bytes: per request and KV head, the union of tokens any row
    sees, times the bytes of its K and V rows (D each for E4M3/E5M2, 2D for
    bf16)."""
    row = 2 * p.D if p.kv_format == "bf16" else p.D
    if p.mode == "dense":
        tot = 0
        for b in range(p.B):
            u = int(p.row_len[b].max()) if p.q > 0 else 0
            tot += u
        return tot * p.Hkv * 2 * row
    m = masks_any(p)
    tot = 0
    for b in range(p.B):
        n = int(p.n_entries[b])
        mb = m[b, :n]
        for t in range(4):
            sel = (mb & (0x11111111 << t)) != 0
            tot += int(sel.sum())
    return tot * p.Hkv * 2 * row
