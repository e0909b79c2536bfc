"""GPU parity of the cache write (fp8kv_attn_cache_write) against the oracle.

The written cache bytes must equal the oracle's byte for byte -- the write is
integer output decided by FP32 arithmetic that both sides do in the same
precision (FP32 division, then round to nearest even with saturation) --
and every byte the write must not touch keeps its poison value.  NaN inputs
may give either NaN code (0x7F or 0xFF); both sides must give a NaN code
there.  Covered: fp16 and bf16 inputs, head dims 64/128/256, strided inputs,
caches inside a wider head layout, padding slots, out-of-range blocks (status
bit), device-side scales, exact midpoints / saturation / signed zero / NaN /
infinities, an empty write, and the full-size prefill write of the benchmark
(sampled tokens against the oracle, all untouched pages checked).
"""

import numpy as np
import pytest
import torch

import oracle
from synth import make_cache_write

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_e4m3_paged_gb300 import build_lib

    build_lib.build()
    oracle.build()


def _gpu_write(p, kc_cpu, vc_cpu, *, strided_in=False, device_scales=False, head_slice=None, fmt="e4m3"):
    from fp8_e4m3_paged_gb300 import binding as B

    dev = torch.device("cuda")
    k, v = p.k.to(dev), p.v.to(dev)
    if strided_in:  # token / head strides larger than the row, d contiguous
        N, Hkv, D = p.k.shape
        kw = torch.zeros(N, Hkv + 1, D + 16, dtype=p.k.dtype, device=dev)
        vw = torch.zeros(N + 1, Hkv, D + 32, dtype=p.k.dtype, device=dev)
        kw[:, :Hkv, :D] = k
        vw[:N, :, :D] = v
        k, v = kw[:, :Hkv, :D], vw[:N, :, :D]
    kc_full, vc_full = kc_cpu.to(dev), vc_cpu.to(dev)
    kc = kc_full if head_slice is None else kc_full[:, :, head_slice, :]
    vc = vc_full if head_slice is None else vc_full[:, :, head_slice, :]
    slots = p.slots.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ks = vs = None
    if device_scales:
        ks = torch.tensor([p.k_scale], dtype=torch.float32, device=dev)
        vs = torch.tensor([p.v_scale], dtype=torch.float32, device=dev)
    a = B.make_cache_write_args(k=k, v=v, slot_mapping=slots, k_cache=kc, v_cache=vc,
                                page_size=p.page_size, k_scale=0.0 if device_scales else p.k_scale,
                                v_scale=0.0 if device_scales else p.v_scale,
                                k_scale_dev=ks, v_scale_dev=vs, status=status,
                                kv_format=B.KV_E5M2 if fmt == "e5m2" else B.KV_E4M3)
    B.fp8kv_attn_cache_write(a, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return kc_full.cpu(), vc_full.cpu(), int(status.item())


def _oracle_write(p, kc_cpu, vc_cpu, head_slice=None, fmt="e4m3"):
    kc, vc = kc_cpu.clone(), vc_cpu.clone()
    kv = kc if head_slice is None else kc[:, :, head_slice, :]
    vv = vc if head_slice is None else vc[:, :, head_slice, :]
    bad = oracle.cache_write(p.k, p.v, p.slots, kv, vv, p.k_scale, p.v_scale, p.page_size, kv_format=fmt)
    return kc, vc, bad


def _same_bytes(got, ref, fmt="e4m3"):
    """Equal bytes, except that a NaN code may be any NaN code of the format."""
    g, r = got.numpy(), ref.numpy()
    if fmt == "e5m2":
        nan_g = ((g & 0x7C) == 0x7C) & ((g & 0x03) != 0)
        nan_r = ((r & 0x7C) == 0x7C) & ((r & 0x03) != 0)
    else:
        nan_g = (g & 0x7F) == 0x7F
        nan_r = (r & 0x7F) == 0x7F
    assert np.array_equal(nan_g, nan_r), "NaN codes differ in position"
    diff = (g != r) & ~nan_r
    assert not diff.any(), f"{int(diff.sum())} bytes differ, first at {np.argwhere(diff)[0].tolist()}"


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("scales", [(0.0078125, 0.015625), (0.0071, 0.0123)], ids=["pow2", "calibrated"])
def test_cache_write_matches_oracle(D, dtype, scales):
    p = make_cache_write(N=203, Hkv=3, D=D, page_size=16, num_blocks=20, dtype=dtype, seed=D + 1,
                         k_scale=scales[0], v_scale=scales[1])
    kc0, vc0 = p.empty_caches()
    kg, vg, st = _gpu_write(p, kc0, vc0)
    kr, vr, bad = _oracle_write(p, kc0, vc0)
    _same_bytes(kg, kr)
    _same_bytes(vg, vr)
    assert bad == 2 and st == 1  # FP8KV_STATUS_BAD_BLOCK


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_cache_write_edge_values(dtype):
    p = make_cache_write(N=96, Hkv=2, D=128, page_size=8, num_blocks=16, dtype=dtype, seed=17, edge=True,
                         k_scale=0.25, v_scale=3.0)
    kc0, vc0 = p.empty_caches()
    kg, vg, _ = _gpu_write(p, kc0, vc0)
    kr, vr, _ = _oracle_write(p, kc0, vc0)
    _same_bytes(kg, kr)
    _same_bytes(vg, vr)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("edge", [False, True])
def test_e5m2_cache_write_matches_oracle(D, dtype, edge):
    """The legacy E5M2 cache: byte-exact against the oracle's encoder, with
    calibrated scales, exact E5M2 midpoints, saturation, signed zeros,
    infinities and NaN."""
    p = make_cache_write(N=150, Hkv=2, D=D, page_size=16, num_blocks=16, dtype=dtype, seed=D + 7,
                         k_scale=0.0071, v_scale=3.3, std=200.0, edge=edge, edge_format="e5m2")
    kc0, vc0 = p.empty_caches()
    kg, vg, st = _gpu_write(p, kc0, vc0, fmt="e5m2")
    kr, vr, bad = _oracle_write(p, kc0, vc0, fmt="e5m2")
    _same_bytes(kg, kr, "e5m2")
    _same_bytes(vg, vr, "e5m2")
    assert bad == 2 and st == 1


def test_cache_write_strides_and_device_scales():
    p = make_cache_write(N=77, Hkv=2, D=128, page_size=5, num_blocks=24, seed=23)
    kc0, vc0 = p.empty_caches(extra_heads=1)  # caches inside a wider head layout
    sl = slice(1, 3)
    kg, vg, st = _gpu_write(p, kc0, vc0, strided_in=True, device_scales=True, head_slice=sl)
    kr, vr, _ = _oracle_write(p, kc0, vc0, head_slice=sl)
    _same_bytes(kg, kr)
    _same_bytes(vg, vr)
    assert st == 1


def test_cache_write_empty_is_noop():
    p = make_cache_write(N=0, Hkv=1, D=64, page_size=4, num_blocks=2, seed=1)
    kc0, vc0 = p.empty_caches()
    kg, vg, st = _gpu_write(p, kc0, vc0)
    assert torch.equal(kg, kc0) and torch.equal(vg, vc0) and st == 0


def test_cache_write_full_size_sampled():
    # the benchmark's prefill write: 65536 tokens, Hkv 8, D 128, page 16
    p = make_cache_write(N=65536, Hkv=8, D=128, page_size=16, num_blocks=4608, seed=5,
                         k_scale=0.0071, v_scale=0.0123)
    kc0, vc0 = p.empty_caches()
    kg, vg, st = _gpu_write(p, kc0, vc0)
    assert st == 1
    g = torch.Generator().manual_seed(9)
    idx = torch.randperm(p.k.shape[0], generator=g)[:256]
    sub = make_cache_write(N=0, Hkv=8, D=128, page_size=16, num_blocks=4608)
    sub.k, sub.v, sub.slots = p.k[idx], p.v[idx], p.slots[idx]
    sub.k_scale, sub.v_scale = p.k_scale, p.v_scale
    kr, vr, _ = _oracle_write(sub, kc0, vc0)
    live = [(int(s) // 16, int(s) % 16) for s in sub.slots.tolist() if 0 <= s < 4608 * 16]
    assert len(live) > 200
    for b, o in live:
        _same_bytes(kg[b, o], kr[b, o])
        _same_bytes(vg[b, o], vr[b, o])
    # pages no token names keep their poison
    used = torch.zeros(4608, dtype=torch.bool)
    s = p.slots[(p.slots >= 0) & (p.slots < 4608 * 16)]
    used[s // 16] = True
    assert bool((kg[~used] == p.poison).all()) and bool((vg[~used] == p.poison).all())
