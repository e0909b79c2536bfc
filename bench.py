#!/usr/bin/env python3
"""Benchmark: attended-KV GB/s of paged E4M3 attention (split + combine).

One step = one pass of the whole path (plan made once; split kernel + combine
kernel) over one batch of synthetic input: by default the verify workload
q=8 rows, Hq=6/Hkv=1, D=256, 131072-token context in 1728-token pages.
Inputs stay resident in HBM; several copies of the KV pool are rotated so
that each step reads bytes the L2 no longer holds.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the FP64 CPU oracle
instead, on bounded samples of the same workload.  ``--op cache_write``
measures the cache write instead (a 65536-token prefill chunk of fp16 K/V,
Hkv=8, D=128, quantised into 16-token E4M3 pages), ``--op dcp_merge`` the
context-parallel merge kernel on a decode batch, ``--op select_entries`` the
grouped planner on the sparse verify shape.

Launch: ``python bench.py [--gpus N --steps K --warmup W]``; for N > 1 under
torchrun, each rank runs an independent replica (no collective on the data
path) and the job's value is the sum of bytes over the max time over ranks.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import attended_kv_bytes, make_cache_write, make_problem  # noqa: E402

METRIC = "attended-KV GB/s and µs/step (q8 Hq6/Hkv1/D256 @128K ctx), % of HBM peak"
WORKLOAD_DESC = {
    "c3_128k": "verify q=8 rows, Hq=6/Hkv=1, D=256, context 131072, page 1728 (76 relocated pages), "
               "E4M3 K/V per-tensor scales, fp16 Q/out",
    "c3_64k": "verify q=8, Hq=6/Hkv=1, D=256, context 65536, page 1728",
    "c3_256k": "verify q=8, Hq=6/Hkv=1, D=256, context 262144, page 1728",
    "c2": "verify q=8, Hq=6/Hkv=1, D=256, context 8192, page 3296",
    "c1": "verify q=2, Hq=6/Hkv=1, D=256, context 1024, page 16",
    "c4": "64 decode requests q=1, Hq=32/Hkv=8, D=128, log-uniform contexts 512..65536, page 16",
    "c5": "QSA sparse verify 4 x q=4, Hq=24/Hkv=2, D=128, 512 four-token microblocks per row of 131072",
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampler running around the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.period = period_ms
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        win = [s for (t, s) in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = sorted(float(s[1]) for s in win if s[1].replace(".", "").isdigit())
        smax = [float(s[2]) for s in win if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in win:
            for k, n in enumerate(names):
                if s[5 + k].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(win)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_ours(args):
    import torch.distributed as dist

    from fp8_e4m3_paged_gb300 import build_lib
    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0 or ws == 1:
        build_lib.build()
    if ws > 1:
        dist.barrier()
        build_lib.build()
    from fp8_e4m3_paged_gb300.device_problem import DeviceProblem

    p = make_problem(args.workload, **_overrides(args))
    bytes_step = attended_kv_bytes(p)
    kv_bytes = p.k_cache.numel() + p.v_cache.numel()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    copies = max(2, math.ceil(3 * l2 / max(kv_bytes, 1)) + 1) if args.copies == 0 else args.copies
    k_new = v_new = None
    if args.new_tokens:
        # the verify step writes its draft tokens itself (fused cache write):
        # fp16 rows for the last new_tokens positions of every request
        if p.mode != "dense" or args.kv_format == "bf16":
            raise SystemExit("--new-tokens: dense FP8 caches only")
        g = torch.Generator().manual_seed(11)
        shape = (p.B, args.new_tokens, p.Hkv, p.D)
        k_new = torch.randn(shape, generator=g).to(torch.float16)
        v_new = torch.randn(shape, generator=g).to(torch.float16)
    dp = DeviceProblem(p, kv_copies=copies, kernel=args.kernel, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    graphs, split_graphs = [], []
    with torch.cuda.stream(s):
        for c in range(copies):
            dp.run(c)  # first launches (kernel attributes) outside capture
    torch.cuda.synchronize()
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dp.run(c)
        graphs.append(g)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=s):
            dp.calls[c].split(torch.cuda.current_stream().cuda_stream)
        split_graphs.append(g2)
    # one graph holding a step on every KV copy in turn: a serving loop
    # launches its decode steps inside larger graphs, so the per-graph launch
    # gap is amortised the same way here (every step still does all its work)
    round_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(round_graph, stream=s):
        for c in range(copies):
            dp.run(c)
    round_split = torch.cuda.CUDAGraph()
    with torch.cuda.graph(round_split, stream=s):
        for c in range(copies):
            dp.calls[c].split(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()

    def replay_steps(n, rounds_graph, singles):
        for _ in range(n // copies):
            rounds_graph.replay()
        for i in range(n % copies):
            singles[i].replay()

    def barrier():
        if ws > 1:
            dist.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(s):
        for i in range(args.warmup):
            graphs[i % copies].replay()
    torch.cuda.synchronize()

    # ---------------------------------------------------------------- timed
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(s):
        e0.record(s)
        replay_steps(args.steps, round_graph, graphs)
        e1.record(s)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    # percentiles over 50 separately timed replays of the round graph (the
    # pages' protocol reports p10 / p50 / p90); per step = replay / copies
    per_step = []
    with torch.cuda.stream(s):
        for _ in range(50):
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(s)
            round_graph.replay()
            a1.record(s)
            a1.synchronize()
            per_step.append(a0.elapsed_time(a1) * 1e3 / copies)
    per_step.sort()
    pct = {"p10": round(per_step[4], 3), "p50": round(per_step[24], 3), "p90": round(per_step[44], 3),
           "replays": 50, "steps_per_replay": copies}
    if ws > 1:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # split kernel alone (same stream, same rotation) for the roofline line
    k2 = max(args.steps // 2, 10)
    with torch.cuda.stream(s):
        for i in range(min(args.warmup, 50)):
            split_graphs[i % copies].replay()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(s)
        replay_steps(k2, round_split, split_graphs)
        f1.record(s)
    torch.cuda.synchronize()
    split_ms = f0.elapsed_time(f1) / k2
    sampler.stop()
    clocks = sampler.summary(t0, t1)

    # ---------------------------------------------------------------- e2e
    e2e = run_e2e(p, dp, args, s, bytes_step)

    status = dp.status()
    peak, peak_src = _peaks()
    value_gbs = bytes_step * ws / (ms * 1e-3) / 1e9
    alg_split = bytes_step + p.q_fp16.numel() * 2 + (p.block_table.numel() * 4 + p.row_len.numel() * 4
                                                      if p.mode == "dense" else
                                                      p.entry_tbl.numel() * 8 + p.n_entries.numel() * 4)
    achieved = alg_split / (split_ms * 1e-3) / 1e9
    traffic = _traffic_record(args.workload)
    line = {
        "metric": METRIC,
        "value": round(value_gbs, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 6),
        "us_per_step": round(ms * 1e3, 3),
        "us_per_step_percentiles": pct,
        "pct_of_hbm_peak": round(100.0 * value_gbs / ws / peak, 2),
        "hbm_peak_gbs": peak,
        "hbm_peak_source": peak_src,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; E4M3 bytes from N(0,1) with per-tensor scales)",
        "config": {
            "workload": f"{args.workload}: {WORKLOAD_DESC.get(args.workload, '')}",
            "attended_kv_bytes_per_step": bytes_step,
            "kv_format": args.kv_format,
            "fused_new_tokens": args.new_tokens,
            "kernel": {1: "generic (CUDA cores)", 2: "tcgen05 (query rows)",
                       3: "tcgen05 small group (tokens as rows)"}.get(dp.plan.kernel, str(dp.plan.kernel)),
            "num_splits": dp.plan.num_splits,
            "l2": f"inputs larger than L2: {copies} rotating KV copies, {copies * kv_bytes / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB",
            "launch": f"CUDA graphs of {copies} steps (one per KV copy), replayed back to back",
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "split",
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": alg_split,
            "avg_launch_us": round(split_ms * 1e3, 3),
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback 6.8 TB/s",
        },
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "device_status": status,
        "context_pages_v100_fp32_route_ms_at_131072": 0.7916,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p, bytes_step, budget_s=args.cpu_budget)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def _traffic_record(workload):
    """DRAM bytes per split launch from the committed ncu summary, if it
    matches the current kernel revision (else null)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(workload)
        if rec and rec.get("kernel_rev") == _kernel_rev():
            return rec.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def _kernel_rev():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_e4m3_paged_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def run_e2e(p, dp, args, s, bytes_step):
    """Same metric through the public API with host inputs: every step copies
    the step's inputs from pinned host memory (Q, the KV pool, the block table
    and row lengths), runs split + combine, and reads the fp16 output back."""
    host = {
        "q": p.q_fp16.pin_memory(),
        "k": p.k_cache.pin_memory(),
        "v": p.v_cache.pin_memory(),
    }
    if p.mode == "dense":
        host["bt"] = p.block_table.pin_memory()
        host["rl"] = p.row_len.pin_memory()
        if dp.k_new is not None:
            host["kn"] = dp.k_new.cpu().pin_memory()
            host["vn"] = dp.v_new.cpu().pin_memory()
    else:
        host["et"] = p.entry_tbl.pin_memory()
        host["em"] = p.entry_mask.pin_memory()
        host["ne"] = p.n_entries.pin_memory()
    out_h = torch.empty(dp.out.shape, dtype=dp.out.dtype).pin_memory()
    dev = {"q": dp.q, "k": dp.k_caches[0], "v": dp.v_caches[0]}
    if p.mode == "dense":
        dev["bt"], dev["rl"] = dp.block_table, dp.row_len
        if dp.k_new is not None:
            dev["kn"], dev["vn"] = dp.k_new, dp.v_new
    else:
        dev["et"], dev["em"], dev["ne"] = dp.entry_tbl, dp.entry_mask, dp.n_entries
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    steps = max(3, min(args.e2e_steps, args.steps))

    def step():
        for k, t in host.items():
            dev[k].copy_(t, non_blocking=True)
        dp.calls[0].run(torch.cuda.current_stream().cuda_stream)
        out_h.copy_(dp.out, non_blocking=True)

    with torch.cuda.stream(s):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            step()
        e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(bytes_step / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def _item_tokens(p):
    """(b, r, h) query vectors of a problem and the tokens each one attends."""
    import numpy as np

    items, toks = [], []
    if p.mode == "dense":
        for b in range(p.B):
            for r in range(p.q):
                n = int(p.row_len[b, r])
                for h in range(p.Hq):
                    items.append((b, r, h))
                    toks.append(n)
    else:
        from synth.workloads import masks_u64

        m = masks_u64(p)
        for b in range(p.B):
            mb = m[b, :int(p.n_entries[b])]
            for r in range(p.q):
                n = int(sum(((mb >> (4 * r + t)) & 1).sum() for t in range(4)))
                for h in range(p.Hq):
                    items.append((b, r, h))
                    toks.append(n)
    return items, np.asarray(toks, dtype=np.float64)


def cpu_baseline(p, bytes_step, budget_s=15.0):
    """The FP64 oracle on the host cores: whole steps of the workload when one
    fits the budget, else random subsets of its query vectors, each counted
    as the share of the step's attended tokens it covers."""
    import numpy as np

    import oracle

    threads = oracle.default_threads()
    oracle.build()
    items, toks = _item_tokens(p)
    t = time.time()
    oracle.attention_items(p, [items[int(np.argmax(toks))]], threads=1)
    per_token = max(time.time() - t, 1e-5) / max(float(toks.max()), 1.0)
    full_s = per_token * float(toks.sum()) / threads
    t0 = time.time()
    if full_s <= budget_s / 2:
        reps = 0
        while True:
            oracle.attention(p, threads=threads)
            reps += 1
            if time.time() - t0 >= budget_s:
                break
        dt = time.time() - t0
        return {"value": round(bytes_step * reps / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
                "kind": "oracle", "seconds": round(dt, 2),
                "sample": f"{reps} full step(s) of the workload (all query rows and heads)"}
    rng = np.random.default_rng(0)
    n = int(max(threads, min(len(items), budget_s / 2 * threads / (per_token * float(toks.mean()) + 1e-12))))
    frac, batches = 0.0, 0
    while time.time() - t0 < budget_s:
        pick = rng.choice(len(items), n, replace=False)
        oracle.attention_items(p, [items[i] for i in pick], threads=threads)
        frac += float(toks[pick].sum() / toks.sum())
        batches += 1
    dt = time.time() - t0
    return {"value": round(bytes_step * frac / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{batches} random subset(s) of {n} of the {len(items)} query vectors, counted by the "
                      f"share of attended tokens they cover ({frac:.3f} steps in all)"}


def _overrides(args):
    """--reqs N: the first N requests of the batched decode workload (same
    lengths and bytes as the full batch's first N), for small profiles."""
    over = {}
    if args.reqs:
        if args.workload != "c4":
            raise SystemExit("--reqs applies to the batched decode workload (c4) only")
        over["B"] = args.reqs
    if args.kv_format != "e4m3":
        over["kv_format"] = args.kv_format
    return over


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded sample (a
    subset of the workload's query vectors), sized so the whole run stays
    within a few minutes."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np

    import oracle

    oracle.build()
    threads = oracle.default_threads()
    p = make_problem(args.workload, **_overrides(args))
    bytes_step = attended_kv_bytes(p)
    allitems = [(b, r, h) for b in range(p.B) for r in range(p.q) for h in range(p.Hq)]
    # cost of one query vector
    t = time.time()
    oracle.attention_items(p, [allitems[0]], threads=1)
    per_item = max(time.time() - t, 1e-4)
    budget = args.ref_budget / max(1, args.steps + args.warmup)
    n = int(max(1, min(len(allitems), budget * threads / per_item)))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle.attention_items(p, [allitems[i] for i in rng.choice(len(allitems), n, replace=False)], threads=threads)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.attention_items(p, [allitems[i] for i in rng.choice(len(allitems), n, replace=False)], threads=threads)
    dt = time.time() - t0
    ms = dt * 1e3 / args.steps
    frac = n / len(allitems)
    value = bytes_step * frac / (ms * 1e-3) / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; E4M3 bytes from N(0,1) with per-tensor scales)",
        "config": {"workload": f"{args.workload}: {WORKLOAD_DESC.get(args.workload, '')}",
                   "attended_kv_bytes_per_step": bytes_step},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n} of {len(allitems)} query vectors per step (random subset), "
                                   f"scaled to the workload by that fraction"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


CW_METRIC = "cache-write GB/s (fp16 K/V -> E4M3 pages: 65536 tokens, Hkv=8, D=128, page 16), % of HBM peak"
CW_DESC = ("prefill chunk of 65536 new tokens (5% padding slots), Hkv=8, D=128, fp16 K and V with "
           "per-tensor scales 0.0071 / 0.0123, written into 16-token E4M3 pages of a 4608-block pool in "
           "allocator order")


def _cw_problem():
    # scales as an amax calibration gives them (not powers of two)
    return make_cache_write(N=65536, Hkv=8, D=128, page_size=16, num_blocks=4608, seed=5, bad_slots=0,
                            k_scale=0.0071, v_scale=0.0123)


def _cw_bytes(p):
    """Algorithmic bytes of one write: the slot list, and per written token
    the fp16 K and V rows read and the E4M3 K and V rows written."""
    N, Hkv, D = p.k.shape
    live = int(((p.slots >= 0) & (p.slots < p.num_blocks * p.page_size)).sum())
    return N * 8 + live * Hkv * D * (2 + 2 + 1 + 1), live


def run_cache_write(args):
    from fp8_e4m3_paged_gb300 import binding as B
    from fp8_e4m3_paged_gb300 import build_lib

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    build_lib.build()
    p = _cw_problem()
    bytes_step, live = _cw_bytes(p)
    dev = torch.device("cuda")
    k, v, slots = p.k.to(dev), p.v.to(dev), p.slots.to(dev)
    kc0, vc0 = p.empty_caches()
    kc, vc = kc0.to(dev), vc0.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    a = B.make_cache_write_args(k=k, v=v, slot_mapping=slots, k_cache=kc, v_cache=vc, page_size=p.page_size,
                                k_scale=p.k_scale, v_scale=p.v_scale, status=status)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        B.fp8kv_attn_cache_write(a, s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.fp8kv_attn_cache_write(a, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    steps = args.steps
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(steps):  # inputs (268 MB) and output (134 MB) exceed the L2
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    ms = e0.elapsed_time(e1) / steps
    # e2e: the same write through the C ABI with the step's inputs copied
    # from pinned host memory and the status word read back
    host = {"k": p.k.pin_memory(), "v": p.v.pin_memory(), "s": p.slots.pin_memory()}
    devs = {"k": k, "v": v, "s": slots}
    st_h = torch.zeros(1, dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.e2e_steps, steps))

    def e2e_step():
        for key, t in host.items():
            devs[key].copy_(t, non_blocking=True)
        B.fp8kv_attn_cache_write(a, torch.cuda.current_stream().cuda_stream)
        st_h.copy_(status, non_blocking=True)

    with torch.cuda.stream(s):
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(s)
        for _ in range(e2e_steps):
            e2e_step()
        f1.record(s)
    torch.cuda.synchronize()
    e2e_ms = f0.elapsed_time(f1) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    peak, peak_src = _peaks()
    value = bytes_step / (ms * 1e-3) / 1e9
    line = {
        "op": "cache_write",
        "metric": CW_METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": 1,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 6),
        "us_per_step": round(ms * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; N(0,1) fp16 rows with saturating outliers)",
        "config": {"workload": f"cache_write: {CW_DESC}", "written_tokens": live,
                   "l2": "inputs larger than L2: 268 MB read and 134 MB written per step",
                   "launch": "one CUDA graph per step, replayed back to back"},
        "roofline": {"bound": "hbm", "kernel": "cache_write", "achieved": round(value, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(value / peak, 4), "traffic": None,
                     "algorithmic_bytes_per_launch": bytes_step, "avg_launch_us": round(ms * 1e3, 3),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s"},
        "clocks": sampler.summary(t0, t1),
        "e2e": {"value": round(bytes_step / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
        "gpu_launches": steps,
        "device_status": int(status.item()),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cw_cpu_baseline(p, args.cpu_budget)
    print(json.dumps(line), flush=True)


def _cw_sample(p, lo, n):
    sub = make_cache_write(N=0, Hkv=p.k.shape[1], D=p.k.shape[2], page_size=p.page_size,
                           num_blocks=p.num_blocks)
    sub.k, sub.v, sub.slots = p.k[lo:lo + n], p.v[lo:lo + n], p.slots[lo:lo + n]
    sub.k_scale, sub.v_scale = p.k_scale, p.v_scale
    return sub


def cw_cpu_baseline(p, budget_s):
    """The oracle's cache write (single thread) on consecutive slices of the
    workload until the budget is spent; bytes counted like the GPU's."""
    import oracle

    oracle.build()
    kc, vc = p.empty_caches()
    n, lo, done, t0 = 256, 0, 0, time.time()
    while time.time() - t0 < budget_s:
        sub = _cw_sample(p, lo, n)
        oracle.cache_write(sub.k, sub.v, sub.slots, kc, vc, sub.k_scale, sub.v_scale, sub.page_size)
        done += _cw_bytes(sub)[0]
        lo = (lo + n) % p.k.shape[0]
    dt = time.time() - t0
    return {"value": round(done / dt / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 2), "sample": "consecutive 256-token slices of the workload, one thread"}


def run_cache_write_reference(args):
    _, rank, _ = _dist()
    if rank != 0:
        return
    import oracle

    oracle.build()
    p = _cw_problem()
    kc, vc = p.empty_caches()
    n = 64
    per = args.ref_budget / max(1, args.steps + args.warmup)
    probe = _cw_sample(p, 0, n)
    t = time.time()
    oracle.cache_write(probe.k, probe.v, probe.slots, kc, vc, p.k_scale, p.v_scale, p.page_size)
    n = int(max(16, min(p.k.shape[0], n * per / max(time.time() - t, 1e-4))))
    for _ in range(args.warmup):
        sub = _cw_sample(p, 0, n)
        oracle.cache_write(sub.k, sub.v, sub.slots, kc, vc, p.k_scale, p.v_scale, p.page_size)
    done, t0 = 0, time.time()
    for i in range(args.steps):
        sub = _cw_sample(p, (i * n) % p.k.shape[0], n)
        oracle.cache_write(sub.k, sub.v, sub.slots, kc, vc, p.k_scale, p.v_scale, p.page_size)
        done += _cw_bytes(sub)[0]
    dt = time.time() - t0
    value = done / dt / 1e9
    print(json.dumps({
        "impl": "reference", "op": "cache_write", "metric": CW_METRIC, "value": round(value, 5), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; N(0,1) fp16 rows with saturating outliers)",
        "config": {"workload": f"cache_write: {CW_DESC}"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} consecutive tokens per step, bytes counted like the GPU's"},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


DCP_METRIC = "DCP merge GB/s and µs (2048 query vectors, D=128, R ranks' FP32 outputs + base-2 LSEs -> fp16)"


def run_dcp_merge(args):
    """The cross-rank merge kernel (all-to-all shape's local merge) on a
    decode batch: 64 requests x 32 query heads, D=128, for R = 2, 4, 8 ranks.
    The value is R=2; enough input copies rotate that each merge reads bytes
    the L2 no longer holds."""
    from fp8_e4m3_paged_gb300 import binding as B
    from fp8_e4m3_paged_gb300 import build_lib

    _, _, local = _dist()
    torch.cuda.set_device(local)
    build_lib.build()
    n, D = 64 * 32, 128
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    g = torch.Generator(device="cuda").manual_seed(3)
    peak, peak_src = _peaks()
    res = {}
    for R in (2, 4, 8):
        per = R * n * (D + 1) * 4
        copies = max(2, math.ceil(3 * l2 / per))
        outs = torch.randn(copies, R, n, D, device="cuda", generator=g)
        lses = torch.randn(copies, R, n, device="cuda", generator=g) * 4
        out = torch.empty(n, D, dtype=torch.float16, device="cuda")
        argl = [B.make_merge_args(outs=outs[c], lses=lses[c], out=out) for c in range(copies)]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            B.fp8kv_attn_merge(argl[0], s.cuda_stream)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for c in range(copies):
                B.fp8kv_attn_merge(argl[c], torch.cuda.current_stream().cuda_stream)
        reps = max(3, args.steps // copies)
        with torch.cuda.stream(s):
            for _ in range(max(3, args.warmup // copies)):
                gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(reps):
                gr.replay()
            e1.record(s)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * copies)
        alg = per + n * D * 2
        res[R] = {"us": round(us, 3), "gbs": round(alg / (us * 1e-6) / 1e9, 2), "bytes": alg, "copies": copies,
                  "launches": reps * copies}
    line = {
        "op": "dcp_merge", "metric": DCP_METRIC, "value": res[2]["gbs"], "unit": "GB/s", "n_gpus": 1,
        "steps": res[2]["launches"], "warmup": args.warmup, "ms_per_step": round(res[2]["us"] / 1e3, 6),
        "us_per_step": res[2]["us"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (N(0,1) outputs, N(0,16) LSEs)",
        "config": {"workload": "dcp_merge: 64 decode requests x 32 query heads, D=128, R=2 "
                               "(R=4 and 8 under per_rank_count)",
                   "per_rank_count": res,
                   "l2": "inputs larger than L2: rotating input copies"},
        "roofline": {"bound": "hbm", "kernel": "merge", "achieved": res[2]["gbs"], "peak": peak, "unit": "GB/s",
                     "frac": round(res[2]["gbs"] / peak, 4), "traffic": None,
                     "algorithmic_bytes_per_launch": res[2]["bytes"], "avg_launch_us": res[2]["us"],
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"},
        "gpu_launches": res[2]["launches"],
    }
    print(json.dumps(line), flush=True)


SEL_METRIC = "grouped planner µs per call (token-ID selections -> microblock entries + masks)"


def run_select_entries(args):
    """The grouped planner on the QSA verify shape: 4 requests x 4 query rows
    x 2048 selected token positions over a 131072-token context."""
    import numpy as np

    from fp8_e4m3_paged_gb300 import binding as B
    from fp8_e4m3_paged_gb300 import build_lib
    from synth import make_selection

    _, _, local = _dist()
    torch.cuda.set_device(local)
    build_lib.build()
    Bn, q, topk, L = 4, 4, 2048, 131072
    mb = L // 4
    dev = torch.device("cuda")
    sel = make_selection(Bn, q, L, topk, seed=5).to(dev)
    bt = torch.from_numpy(np.random.default_rng(1).permutation(Bn * mb).astype(np.int32).reshape(Bn, mb)).to(dev)
    stride = (q * topk + 7) // 8 * 8
    tbl = torch.empty(Bn, stride, dtype=torch.int32, device=dev)
    msk = torch.empty(Bn, stride, dtype=torch.int32, device=dev)
    n = torch.empty(Bn, dtype=torch.int32, device=dev)
    a = B.make_select_args(sel=sel, block_table=bt, max_blocks=mb, null_block=0, entry_tbl=tbl, entry_mask=msk,
                           n_entries=n)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        B.fp8kv_attn_select_to_entries(a, s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(10):
            B.fp8kv_attn_select_to_entries(a, torch.cuda.current_stream().cuda_stream)
    reps = max(3, args.steps // 10)
    with torch.cuda.stream(s):
        for _ in range(max(3, args.warmup // 10)):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * 10)
    alg = sel.numel() * 4 + int(n.sum().item()) * 8 + Bn * 4
    peak, peak_src = _peaks()
    print(json.dumps({
        "op": "select_entries", "metric": SEL_METRIC, "value": round(us, 3), "unit": "us", "n_gpus": 1,
        "steps": reps * 10, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic (seeded selections: runs of "
        "neighbouring tokens, 10% unused slots, 5% duplicates)",
        "config": {"workload": "select_entries: 4 requests x 4 rows x 2048 positions, context 131072 (32768 "
                               "logical microblocks, 4 shared-memory chunks per request)",
                   "entries_per_request": n.tolist(),
                   "l2": "inputs (131 KB) stay in L2: a latency figure, not a bandwidth one"},
        "roofline": {"bound": "hbm", "kernel": "select_entries", "achieved": round(alg / (us * 1e-6) / 1e9, 2),
                     "peak": peak, "unit": "GB/s", "frac": round(alg / (us * 1e-6) / 1e9 / peak, 5),
                     "traffic": None, "algorithmic_bytes_per_launch": alg, "avg_launch_us": round(us, 3),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"},
        "gpu_launches": reps * 10,
    }), flush=True)


def run_small_reference(args, op):
    """The oracle's merge or planner on the same shapes as the GPU lines,
    whole calls, timed on the host (one thread)."""
    _, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np

    import oracle

    oracle.build()
    if op == "dcp_merge":
        n, D, R = 64 * 32, 128, 2
        rng = np.random.default_rng(3)
        outs = rng.standard_normal((R, n, D))
        lses = rng.standard_normal((R, n)) * 4

        def call():
            oracle.merge(outs, lses)
        metric, unit, alg = DCP_METRIC, "GB/s", R * n * (D + 1) * 4 + n * D * 2
    else:
        from synth import make_selection

        Bn, q, topk, L = 4, 4, 2048, 131072
        sel = make_selection(Bn, q, L, topk, seed=5).numpy()
        bt = np.random.default_rng(1).permutation(Bn * (L // 4)).astype(np.int32).reshape(Bn, L // 4)

        def call():
            oracle.select_to_entries(sel, bt, L // 4, 0)
        metric, unit, alg = SEL_METRIC, "us", None
    for _ in range(max(1, min(args.warmup, 3))):
        call()
    t0 = time.time()
    k = 0
    while k < max(1, min(args.steps, 50)) and (k == 0 or time.time() - t0 < args.ref_budget / 4):
        call()
        k += 1
    dt = (time.time() - t0) / k
    value = round(alg / dt / 1e9, 5) if unit == "GB/s" else round(dt * 1e6, 1)
    print(json.dumps({
        "impl": "reference", "op": op, "metric": metric, "value": value, "unit": unit, "n_gpus": 1,
        "steps": k, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": unit == "GB/s", "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": f"{op}: the shapes of the GPU line"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": f"{k} whole call(s)"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3_128k")
    ap.add_argument("--copies", type=int, default=0, help="KV copies to rotate (0 = enough to defeat L2)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-budget", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reqs", type=int, default=0, help="c4 only: the first N of its 64 requests")
    ap.add_argument("--new-tokens", type=int, default=0,
                    help="dense verify: the step also writes this many new tokens per request into the "
                         "cache inside the split launch (fused cache write)")
    ap.add_argument("--kernel", type=int, default=0, choices=[0, 1, 2, 3],
                    help="split kernel: 0 = the planner's choice, 1 CUDA cores, 2 tcgen05 query rows, "
                         "3 tcgen05 small group")
    ap.add_argument("--kv-format", choices=["e4m3", "e5m2", "bf16"], default="e4m3",
                    help="cache format (bf16: the unquantised cache, for A/B against the FP8 path)")
    ap.add_argument("--op", choices=["attention", "cache_write", "dcp_merge", "select_entries"], default="attention")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.op == "select_entries":
        if args.impl == "reference":
            run_small_reference(args, "select_entries")
        else:
            run_select_entries(args)
    elif args.op == "dcp_merge":
        if args.impl == "reference":
            run_small_reference(args, "dcp_merge")
        else:
            run_dcp_merge(args)
    elif args.op == "cache_write":
        if args.impl == "reference":
            run_cache_write_reference(args)
        else:
            run_cache_write(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
