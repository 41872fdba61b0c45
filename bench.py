#!/usr/bin/env python3
"""Benchmark of the paged decode attention path on GB300.

One step = one vt_paged_attn_decode call over one synthetic decode batch
(request lookup, page gather, QK^T, mask, online softmax, PV, split partials,
LSE combine, finalize: the whole hot path, one kernel launch).  Inputs sit in
HBM before timing starts.  Calls rotate over copies of the KV pool holding at
least 2x L2 of referenced KV bytes, so every call reads its pages from HBM
(no flush kernel: its dirty lines would be written back during the call).
The timed calls are launched from CUDA graphs, as a serving loop launches its
decode steps, each as a programmatic dependent of the one before (its
start-up overlaps the previous call's tail); the same calls launched one by
one from Python are reported beside them (``eager_per_call``), and ``e2e``
times the C-ABI call with host buffers and the host<->device copies.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the reference arm: a deliberately plain fp64 program on host cores).
Multi-GPU (torchrun, N > 1): every rank runs its own replica of the batch
(independent decode problems, no collective on the data path); the reported
time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "µs/call and achieved KV HBM GB/s (fraction of GB300 peak) per decode step"
UNIT = "µs/call"
# The headline is the largest single-GPU batch, the long-context skewed one
# (1.57 GB of KV per call); the other workloads are timed in the sweep.
DEFAULT_WORKLOAD = "skewed_b128_gqa4_d128"
SWEEP = ["batch1_ctx32768_gqa4_d128", "large_gqa8_b64_d128", "d256_gqa4_b16", "d256_gqa4_b16_w1024",
         "d256_gqa4_b16_f32", "d256_gqa4_b16_f32_w1024", "qwen3_1p7b_b8_gqa2_d128", "d64_gqa4_b32",
         "d64_gqa4_b32_f32", "skewed_b128_gqa4_d128_fp8", "batch1_ctx32768_gqa4_d128_fp8",
         "large_gqa8_b64_d128_fp8", "d256_gqa4_b16_fp8", "d512_gqa4_b16", "d512_gqa4_b16_w1024", "multi_q4_b64_gqa4_d128",
         "multi_q4_b64_gqa4_d128_fp8", "d64_gqa4_b32_fp8"]
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (the measured copy rate is the roofline peak)
KERNEL_SOURCES = ["decode_kernel.cuh", "kernel_variants.cuh", "vt_paged_attn_api.cu"]  # shared by every variant


def _code_only(text: str) -> str:
    """C++ source with comments and blank lines removed (the sources hold no
    comment markers inside string literals)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def variant_source(workload: str) -> str:
    """The translation unit holding the kernel variants a workload runs on."""
    from paged_attention_decode_kv_gb300 import workloads as W
    w = W.WORKLOADS[workload]
    if w.dtype == "e4m3":
        return "decode_e4m3.cu"
    return "decode_d64.cu" if w.head_dim == 64 else f"decode_d{w.head_dim}_{w.dtype}.cu"


def kernel_hash(workload: str = DEFAULT_WORKLOAD) -> str:
    """Hash of the code a workload's kernel is built from (the shared kernel
    and front end plus its variant unit; comments excluded), stamped on the
    ncu summaries so a measurement is only reused for the code it was taken
    on."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES + [variant_source(workload)]:
        h.update(_code_only((ROOT / "paged_attention_decode_kv_gb300" / "csrc" / name).read_text()).encode())
    return h.hexdigest()[:16]


def hbm_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    try:
        data = json.loads(p.read_text())
    except Exception:
        return None
    entry = data.get(workload)
    if not entry or entry.get("kernel_hash") != kernel_hash(workload):
        return None
    return entry.get("dram_bytes_per_launch")


def clocks_acceptable(clk: dict) -> bool:
    """False when the timed region ran throttled by hardware or thermals, or
    with SM clocks well below their maximum and no reason given (a leftover
    clock lock); power capping is kept (and shows in the reasons)."""
    if {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"} & set(clk.get("reasons") or []):
        return False
    sm, top = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    if sm and top and sm < 0.85 * top and not clk.get("reasons"):
        return False
    return True


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.1)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.file.flush()
        rows = []
        for line in Path(self.file.name).read_text().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, _, p in rows for k in range(4) if p[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


ROTATE_BYTES = 256 << 20  # distinct KV bytes read between two uses of the same pool copy (2x L2)


def make_device_case(name: str, seed: int, device, pool_blocks: int = 0, copies: int = 0):
    """The workload on the device, with enough copies of its KV pool that
    consecutive calls never find their pages in L2: copy c serves calls
    c, c + n, ..., and n copies hold >= 2x L2 of referenced KV bytes.
    pool_blocks > 0 shrinks the page pool (same contexts and pages used);
    copies > 0 fixes the number of pool copies (profiler runs, where the
    profiler cleans the caches before each captured launch, use one)."""
    from paged_attention_decode_kv_gb300 import workloads as W
    w = W.WORKLOADS[name]
    if pool_blocks > 0:
        w = w.with_(pool_blocks=pool_blocks)
    case = W.make_case(w, seed)
    k, v = case.pool(device)
    n_copies = copies if copies > 0 else max(2, -(-ROTATE_BYTES // max(case.kv_bytes(), 1)) + 1)
    pools = [(k, v)] + [(k.clone(), v.clone()) for _ in range(n_copies - 1)]
    t = {"q": case.q.to(device), "pools": pools, "k": k, "v": v,
         "bt": case.block_tables.to(device), "cl": case.context_lens.to(device)}
    if case.fp8:
        t["ks"], t["vs"] = case.scales(device)
    return case, t


def decode_step(vt, case, t, q, k, v, bt, cl, out):
    """One decode call through the entry point for the workload's storage
    (FP8 caches take their per-kv-head scales from ``t``)."""
    w = case.workload
    if case.fp8:
        return vt.decode_fp8(q, k, v, t["ks"], t["vs"], bt, cl, w.scale, w.window, out=out)
    if w.q_len > 1:
        return vt.decode_multi(q, k, v, bt, cl, w.scale, w.window, out=out)
    return vt.decode(q, k, v, bt, cl, w.scale, w.window, out=out)


def time_calls(vt, case, t, steps, warmup):
    """Per-call CUDA-event times (s) on the launching stream; call s reads pool
    copy s mod n, so its KV pages come from HBM, not L2."""
    import torch
    w = case.workload
    out = torch.empty_like(t["q"])
    stream = torch.cuda.current_stream()
    pools = t["pools"]
    for i in range(warmup):
        k, v = pools[i % len(pools)]
        decode_step(vt, case, t, t["q"], k, v, t["bt"], t["cl"], out)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for s in range(steps):
        k, v = pools[(warmup + s) % len(pools)]
        starts[s].record(stream)
        decode_step(vt, case, t, t["q"], k, v, t["bt"], t["cl"], out)
        ends[s].record(stream)
    torch.cuda.synchronize()
    status = vt.vt_paged_attn_device_status()
    if status:
        raise RuntimeError(f"device status {status:#x} after timed calls")
    return [a.elapsed_time(b) * 1e-3 for a, b in zip(starts, ends)]


def time_graph(vt, case, t, steps, warmup):
    """Mean device time (s) per call of exactly `steps` calls launched from
    CUDA graphs, as a serving loop would launch its decode steps.  One graph
    holds a whole number of rotations over the pool copies (>= 32 calls); it is
    replayed steps // chunk times, then a graph of the remaining calls runs.
    One event pair on the launching stream brackets all of them."""
    import torch
    w = case.workload
    out = torch.empty_like(t["q"])
    pools = t["pools"]
    n = len(pools)
    chunk = n * -(-32 // n)

    def calls(count):
        for i in range(count):
            k, v = pools[i % n]
            decode_step(vt, case, t, t["q"], k, v, t["bt"], t["cl"], out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls(max(warmup, 3))
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    full, rem = divmod(steps, chunk)
    g_full, g_rem = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full):
        calls(chunk)
    if rem:
        with torch.cuda.graph(g_rem):
            calls(rem)
    for _ in range(max(1, warmup // chunk)):
        g_full.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(full):
        g_full.replay()
    if rem:
        g_rem.replay()
    b.record(stream)
    torch.cuda.synchronize()
    status = vt.vt_paged_attn_device_status()
    if status:
        raise RuntimeError(f"device status {status:#x} after graph-launched calls")
    return a.elapsed_time(b) * 1e-3 / steps, chunk


def time_e2e(vt, case, t, steps, warmup):
    """Through the C-ABI with host buffers, every step: one pinned host->device
    copy of the step's inputs (q, block table and context lengths packed in
    one buffer), the decode, and a device->host copy of the output.  The KV
    pool is resident state (rotated across copies as in time_graph).  Steps
    are launched from CUDA graphs like the device-only timing; one event pair
    brackets all of them.  Returns (mean seconds per step, h2d bytes, d2h bytes)."""
    import torch
    w = case.workload

    def align(x):
        return (x + 255) // 256 * 256

    parts = [case.q.contiguous(), case.block_tables.contiguous(), case.context_lens.contiguous()]
    sizes = [p.numel() * p.element_size() for p in parts]
    offs = [0, align(sizes[0]), align(sizes[0]) + align(sizes[1])]
    total = offs[2] + sizes[2]
    hbuf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for p, o, n in zip(parts, offs, sizes):
        hbuf[o:o + n].copy_(p.view(-1).view(torch.uint8))
    dbuf = torch.empty(total, dtype=torch.uint8, device=t["q"].device)
    dq, dbt, dcl = (dbuf[o:o + n].view(p.dtype).view(p.shape) for p, o, n in zip(parts, offs, sizes))
    hout = torch.empty_like(case.q).pin_memory()
    out = torch.empty_like(t["q"])
    pools = t["pools"]
    n = len(pools)
    chunk = n * -(-16 // n)

    def steps_of(count):
        for i in range(count):
            k, v = pools[i % n]
            dbuf.copy_(hbuf, non_blocking=True)
            decode_step(vt, case, t, dq, k, v, dbt, dcl, out)
            hout.copy_(out, non_blocking=True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        steps_of(max(warmup, 3))
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    full, rem = divmod(steps, chunk)
    g_full, g_rem = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full):
        steps_of(chunk)
    if rem:
        with torch.cuda.graph(g_rem):
            steps_of(rem)
    g_full.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(full):
        g_full.replay()
    if rem:
        g_rem.replay()
    b.record(stream)
    torch.cuda.synchronize()
    if not torch.equal(hout, out.cpu()):
        raise RuntimeError("end-to-end output differs from the device output")
    return a.elapsed_time(b) * 1e-3 / steps, sum(sizes), hout.numel() * hout.element_size()


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_baseline(case, budget_s: float, threads: int = 1):
    """The oracle, as it stands, on `threads` host cores: whole calls of this
    workload, or a row sample of one call when a whole call exceeds the
    budget (rows spread evenly over the batch, shuffled so every thread gets
    a similar mix of long and short sequences, and the time scaled by rows).
    Returns (seconds per call, sample description)."""
    import numpy as np
    import oracle
    from paged_attention_decode_kv_gb300 import workloads as W
    o = oracle.default_oracle()
    w = case.workload
    k, v, bt = case.compact()
    qa, ka, va = W.to_oracle_array(case.q), W.to_oracle_array(k), W.to_oracle_array(v)
    if case.fp8 and w.q_len > 1:
        # the oracle's multi-token rows take the FP8 cache as its fp64 values
        import torch
        ks, vs = case.scales()
        ka = (k.view(torch.float8_e4m3fn).to(torch.float64) * ks.double()[None, None, :, None]).numpy()
        va = (v.view(torch.float8_e4m3fn).to(torch.float64) * vs.double()[None, None, :, None]).numpy()
        qa = case.q.to(torch.float64).numpy()  # bf16 -> fp64 is exact; one storage type for all three
    tail = (bt.numpy(), case.context_lens.numpy(), w.scale, w.window)

    def decode_rows(rows, threads=1):
        if w.q_len > 1:
            return o.decode_multi_rows(rows, qa, ka, va, *tail, threads=threads)
        if case.fp8:
            ks, vs = case.scales()
            return o.decode_rows_e4m3(rows, qa, ka, va, ks.numpy(), vs.numpy(), *tail, threads=threads)
        return o.decode_rows(rows, qa, ka, va, *tail, threads=threads)

    if w.q_len > 1:
        rows_all = [(b, j, i) for b in range(w.num_seqs) for j in range(w.q_len) for i in range(w.num_q_heads)]
    else:
        rows_all = [(b, i) for b in range(w.num_seqs) for i in range(w.num_q_heads)]
    # cost of a whole call from a probe of 8 rows: oracle time grows with the
    # tokens a row attends to, so the probe's time is scaled by tokens
    L = case.context_lens.numpy().astype(np.int64)
    L_eff = np.minimum(L, w.window) if w.window > 0 else L
    tokens_all = float(L_eff.sum()) * w.num_q_heads * w.q_len
    probe = [rows_all[j] for j in np.linspace(0, len(rows_all) - 1, 8).astype(int)]
    t0 = time.perf_counter()
    decode_rows(probe)
    probe_s = time.perf_counter() - t0
    tokens_probe = float(sum(L_eff[r[0]] for r in probe))
    whole_est = max(probe_s, 1e-7) * tokens_all / max(tokens_probe, 1.0)
    who = "single thread" if threads == 1 else f"{threads} threads"
    if whole_est / threads <= budget_s:
        calls, t0 = 0, time.perf_counter()
        while True:
            decode_rows(rows_all, threads)
            calls += 1
            el = time.perf_counter() - t0
            if el >= budget_s or calls >= 1000:
                break
        return el / calls, f"{calls} whole calls ({len(rows_all)} rows each) of {w.name}, {who}"
    n = max(threads, int(len(rows_all) * budget_s * threads / whole_est))
    pick = np.linspace(0, len(rows_all) - 1, min(n, len(rows_all))).astype(int)
    pick = np.random.default_rng(0).permutation(pick)
    rows = [rows_all[p] for p in pick]
    t0 = time.perf_counter()
    decode_rows(rows, threads)
    el = time.perf_counter() - t0
    return el / len(rows) * len(rows_all), (f"{len(rows)} of {len(rows_all)} rows of one call of {w.name} "
                                            f"(spread evenly over the batch), {who}, scaled to a whole call")


def run_reference(args, rank, world):
    from paged_attention_decode_kv_gb300 import workloads as W
    if rank != 0:
        return 0
    case = W.make_case(W.WORKLOADS[args.workload], 0)
    cores = host_cores()
    # each step is a bounded sample: the whole run stays within a few minutes
    budget = min(args.ref_budget, 120.0 / max(args.steps, 1))
    for _ in range(args.warmup):
        oracle_baseline(case, 0.0, cores)
    times = []
    sample = ""
    for _ in range(args.steps):
        t, sample = oracle_baseline(case, budget, cores)
        times.append(t)
    us = statistics.mean(times) * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "storage_dtype": case.workload.dtype},
            "cpu_baseline": {"kind": "oracle", "value": us, "unit": UNIT, "cores": cores, "sample": sample},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks(x: float, dist, device) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def summarize(times):
    s = sorted(times)
    return {"mean_us": statistics.mean(s) * 1e6, "median_us": s[len(s) // 2] * 1e6,
            "p10_us": s[len(s) // 10] * 1e6, "p90_us": s[(9 * len(s)) // 10] * 1e6}


def run_profile_only(args):
    """A short, fixed run of one workload for ncu captures (no timing and no
    JSON line): warm-up calls plus --steps calls, pools rotated as in the bench."""
    import torch
    import paged_attention_decode_kv_gb300 as vt
    from paged_attention_decode_kv_gb300 import build_lib
    build_lib.build()
    dev = torch.device("cuda", 0)
    case, t = make_device_case(args.workload, args.seed, dev, args.pool_blocks, copies=1)
    w = case.workload
    out = torch.empty_like(t["q"])
    for i in range(args.warmup + args.steps):
        k, v = t["pools"][i % len(t["pools"])]
        decode_step(vt, case, t, t["q"], k, v, t["bt"], t["cl"], out)
    torch.cuda.synchronize()
    status = vt.vt_paged_attn_device_status()
    print(f"profile-only {w.name}: {args.warmup} + {args.steps} calls, kv bytes {case.kv_bytes()}, "
          f"status {status}, plan {vt.vt_paged_attn_last_plan()}")
    return 1 if status else 0


def run_ours(args, rank, world, dist):
    import torch
    import paged_attention_decode_kv_gb300 as vt
    from paged_attention_decode_kv_gb300 import build_lib
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not build_lib.up_to_date():
        build_lib.build()
    if dist is not None:
        dist.barrier()
    vt.library()
    # decode after decode on one stream: each call's start-up (context
    # lengths, partition, block table) overlaps the previous call's tail
    vt.vt_paged_attn_set_overlap(True)
    peak, peak_src = hbm_peak()

    case, t = make_device_case(args.workload, args.seed + rank, dev)
    w = case.workload
    kv = case.kv_bytes()
    algo = kv + case.qo_bytes()
    context_tokens = int(case.context_lens.sum())

    # timed region: barrier + synchronize on both sides, clocks sampled during it
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    def timed_region():
        with ClockSampler(local) as clocks:
            g_s, ch = time_graph(vt, case, t, args.steps, args.warmup)
        torch.cuda.synchronize()
        return g_s, ch, clocks.summary()

    graph_s, chunk, clk = timed_region()
    remeasured = not clocks_acceptable(clk)
    if remeasured:  # a throttled or clock-locked run is taken once more
        graph_s, chunk, clk = timed_region()
    if dist is not None:
        dist.barrier()
    plan = vt.vt_paged_attn_last_plan()
    mean_s = max_over_ranks(graph_s, dist, dev)
    # the same calls launched one by one from Python (per-call event pairs)
    times = time_calls(vt, case, t, max(200, args.steps // 10), args.warmup)
    e2e_step_s, h2d, d2h = time_e2e(vt, case, t, max(200, args.steps // 5), args.warmup)
    e2e_s = max_over_ranks(e2e_step_s, dist, dev)

    host_case = case
    n_pool_copies = len(t["pools"])
    del t
    torch.cuda.empty_cache()
    sweep = []
    if not args.no_sweep and rank == 0:
        for name in SWEEP:
            if name == args.workload:
                continue
            case_s, t_s = make_device_case(name, args.seed, dev)
            m, _ = time_graph(vt, case_s, t_s, args.sweep_steps, 3)
            ts = time_calls(vt, case_s, t_s, max(50, args.sweep_steps // 4), 3)
            a_bytes = case_s.kv_bytes() + case_s.qo_bytes()
            tr = recorded_traffic(name)
            sweep.append({"workload": name, "us_per_call": m * 1e6, "eager_per_call": summarize(ts),
                          "kv_gbs": case_s.kv_bytes() / m / 1e9,
                          "achieved_gbs": a_bytes / m / 1e9, "frac": a_bytes / m / 1e9 / peak,
                          "frac_of_nominal": a_bytes / m / 1e9 / NOMINAL_HBM_GBS,
                          "algorithmic_bytes": a_bytes, "ideal_us_at_peak": a_bytes / (peak * 1e9) * 1e6,
                          "traffic": tr, "traffic_over_algorithmic": (tr / a_bytes) if tr else None,
                          "plan": vt.vt_paged_attn_last_plan()})
            del case_s, t_s
            torch.cuda.empty_cache()

    if rank != 0:
        return 0
    cores = host_cores()
    cpu1_s, cpu1_sample = oracle_baseline(host_case, args.ref_budget, 1)
    cpun_s, cpun_sample = oracle_baseline(host_case, args.ref_budget, cores)
    achieved = algo / mean_s / 1e9
    traffic = recorded_traffic(w.name)
    line = {
        "metric": METRIC, "value": mean_s * 1e6, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_s * 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "num_seqs": w.num_seqs,
                   "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "storage_dtype": w.dtype, "window": w.window,
                   "context_tokens": context_tokens,
                   "l2": f"inputs larger than L2: calls rotate over {n_pool_copies} copies of the KV pool "
                         f"(>= 256 MiB of distinct KV between reuses)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": f"CUDA graphs of {chunk} calls, replayed; one event pair around all "
                             f"{args.steps} timed calls; programmatic dependent launch between consecutive "
                             "calls (vt_paged_attn_set_overlap)"},
        "eager_per_call": summarize(times),
        "kv_gbs": kv / mean_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS, "traffic": traffic,
                     "traffic_over_algorithmic": (traffic / algo) if traffic else None,
                     "ideal_us_at_peak": algo / (peak * 1e9) * 1e6,
                     "algorithmic_bytes_per_launch": algo, "peak_source": peak_src,
                     "kernel": "vt::paged_decode_kernel"},
        "cpu_baseline": {"value": cpun_s * 1e6, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": cpun_sample,
                         "single_core": {"value": cpu1_s * 1e6, "unit": UNIT, "cores": 1, "sample": cpu1_sample}},
        "e2e": {"value": e2e_s * 1e6, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"], "remeasured": remeasured},
        "plan": plan,
        "kernel_hash": kernel_hash(w.name),
        "sweep": sweep,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sweep-steps", type=int, default=300)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=10.0, help="seconds of oracle work per reference sample")
    ap.add_argument("--profile-only", action="store_true",
                    help="run --warmup + --steps calls of --workload for a profiler; no timing, no JSON line")
    ap.add_argument("--pool-blocks", type=int, default=0, help="shrink the page pool (profile-only runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.profile_only:
        return run_profile_only(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group(backend=backend)
        dist = tdist
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
