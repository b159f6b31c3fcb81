#!/usr/bin/env python
"""Benchmark of one batched prompt-lookup draft step on GB300.

A step is one call of the library's public entry point, lookup_draft: the
split-history scan over every request's history plus the draft fill, for one
batch of synthetic histories (default: the 25k-token recitation workload, B=64
requests of 25,000 tokens, 6.4 MB of int32 history).  Prints one JSON line.

  value         microseconds per step on the device, inputs resident in HBM.  The
                K timed steps are public-API calls captured into CUDA graphs
                (replayed back to back); consecutive steps read different copies
                of the batch whose total size is over twice the L2 cache, so
                every step reads its history from HBM.
  eager_us_per_step
                the same K steps as direct calls from Python (host launch cost
                included), for reference.
  roofline      the scan kernel alone: 4 bytes per history token (each read once)
                divided by its mean duration per launch, from CUDA events around
                back-to-back scan launches (captured in a CUDA graph, inputs
                rotating as above) on their stream, against the measured HBM copy
                bandwidth.  scan_us_isolated: events around single launches.
                read_floor: a launch that only streams the same bytes, timed the
                same way (the best of 16-byte loads in three launch shapes and
                bulk copies into shared memory): what one launch reading them
                once reaches here.
  e2e           lookup_draft_host: pinned host buffers in, the step, outputs back
                to the host, every step.
  cpu_baseline  the CPU oracle (brute force, one thread per slice of requests) on
                this machine's host cores, on the same batch, and on one thread
                (median of up to 5 whole batches); `value` is the faster of the
                two, `cores` the threads it used.  Also the CPU model.
  loop_steps    microseconds per call of the decode-loop steps around the draft
                (fusion, scheduling, greedy and sampled verification, append of
                the committed tokens), the append's GB/s, and one whole
                draft-to-append loop step, on the same batch.
  index         the incremental n-gram index on the same batch: build time and
                size, the draft from the index (checked against the oracle), the
                in-place append, and the decode-loop step on the index.
  context_cache context-cache drafting (llama.cpp's rule) on the same batch:
                build time and size, the draft (checked against the oracle) and
                the in-place append.
  workloads     the step and the scan on each of the five workloads (tiny,
                recitation25k, periodic, ragged262k, chats), timed as above, with
                the scan's GB/s and fraction of the measured copy bandwidth and a
                whole-batch check of the outputs against the oracle.

--impl reference times that oracle as the comparison arm on the same workload.
Multi-GPU (torchrun, one rank per GPU): every rank drafts its own batch (weak
scaling, no data exchange); the step time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs per batched draft step; history GB/s scanned vs GB300 HBM roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
SCAN_SOURCE = os.path.join(ROOT, "prompt_lookup_speculative_gb300", "csrc", "lookup_draft.cu")
PROFILES = os.path.join(ROOT, "profiles")
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", default="recitation25k")
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-budget-s", type=float, default=2.0,
                    help="wall-clock budget of the CPU-baseline sample")
    ap.add_argument("--reference-budget-s", type=float, default=90.0,
                    help="wall-clock budget of the whole --impl reference run")
    ap.add_argument("--settle-s", type=float, default=0.5,
                    help="untimed graph replays before the timed region, so clocks settle")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-loop", action="store_true",
                    help="skip the timing of the decode-loop steps (fusion, scheduling, verification, append)")
    ap.add_argument("--no-index", action="store_true",
                    help="skip the timing of the incremental n-gram index")
    ap.add_argument("--no-ctx", action="store_true", help="skip the timing of context-cache drafting")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the step and scan timings of every workload")
    ap.add_argument("--loop-only", action="store_true",
                    help="time only the decode-loop steps (replays = steps / copies of the batch)")
    ap.add_argument("--size-sweep", action="store_true",
                    help="time the step, the scan and the read floor on the recitation recipe at history "
                         "lengths 4,096 to 400,000 tokens (B = 64) and fit a fixed cost plus a rate to each")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- ranks ----
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank drafts its own batch: same workload recipe, its own seed."""
    return int(base_seed) + 1000 * int(rank)


def max_over_ranks(value: float, dist, device=None) -> float:
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi sampled every 100 ms while the GPU work runs."""

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.proc = None
        self.rows = []
        if not enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for ln in out.splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) >= 10:
                self.rows.append(parts)

    def summary(self) -> dict:
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        util = [num(r[4]) or 0.0 for r in self.rows]
        loaded = [num(r[1]) for r, u in zip(self.rows, util) if u > 0 and num(r[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[6:10]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(loaded or sm) if (loaded or sm) else None,
                "sm_max_mhz": num(self.rows[0][2]),
                "reasons": reasons,
                "samples": len(self.rows),
                "samples_under_load": len(loaded),
                "power_w_max": max((num(r[3]) or 0.0) for r in self.rows)}


# ------------------------------------------------------------- roofline ----
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


HOST_SIDE_MARKER = b"// ------------------------------------------------------------- host side ----"


def scan_source_hash() -> str:
    """sha256 (16 hex) of the device code of csrc/lookup_draft.cu: the file up to
    its host-side marker, with comments and layout removed, so host-only and
    comment-only edits keep a kernel capture valid."""
    with open(SCAN_SOURCE, "rb") as f:
        src = f.read()
    cut = src.find(HOST_SIDE_MARKER)
    code = (src if cut < 0 else src[:cut]).decode("utf-8")
    code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)          # block comments
    code = re.sub(r"//[^\n]*", " ", code)                         # line comments
    code = " ".join(code.split())                                  # layout
    return hashlib.sha256(code.encode("utf-8")).hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per scan launch from the committed ncu summary of this workload
    (profiles/scan_kernel_<workload>.md), if it was taken on this exact kernel
    source (else None)."""
    try:
        text = open(os.path.join(PROFILES, f"scan_kernel_{workload}.md"), encoding="utf-8").read()
    except OSError:
        return None
    src = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    wl = re.search(r"workload:\s*(\S+)", text)
    tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not (src and wl and tr) or src.group(1) != scan_source_hash() or wl.group(1) != workload:
        return None
    return int(tr.group(1))


# ------------------------------------------------------------------ GPU ----
def run_gpu(args, rank: int, world: int, local_rank: int):
    import numpy as np
    import torch

    import gen
    import prompt_lookup_speculative_gb300 as pkg

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU fallback)")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = dist_init(world, "nccl")
    lib = pkg.load_library()

    if args.size_sweep:
        if rank == 0:
            print(json.dumps(size_sweep(lib, pkg, dev, max(10, min(200, args.steps)))), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    seed = rank_seed(gen.DEFAULT_SEED[args.workload] if args.seed is None else args.seed, rank)
    w = gen.make_workload(args.workload, seed)
    B, K, min_m, max_m = w.B, w.K, w.min_m, w.max_m
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    ncopy = max(3, math.ceil(2 * l2 / max(w.history_bytes, 1)) + 1)
    stream = torch.cuda.Stream(dev)
    h = int(stream.cuda_stream)

    tok_host = torch.from_numpy(w.tokens)
    off_host = torch.from_numpy(w.offsets)
    toks = [tok_host.to(dev) for _ in range(ncopy)]
    offs = [off_host.to(dev) for _ in range(ncopy)]
    tok_p = [t.data_ptr() for t in toks]
    off_p = [o.data_ptr() for o in offs]
    draft = torch.empty((B, K), dtype=torch.int32, device=dev)
    length = torch.empty(B, dtype=torch.int32, device=dev)
    pos = torch.empty(B, dtype=torch.int32, device=dev)
    dp, lp, pp = draft.data_ptr(), length.data_ptr(), pos.data_ptr()
    ws_bytes = pkg.workspace_bytes(B, dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    wsp = ws.data_ptr()

    if args.loop_only:
        loop = measure_loop(lib, pkg, w, dev, stream, toks, offs, max(1, args.steps // ncopy))
        index = None
        if not args.no_index:
            import oracle
            want = oracle.lookup_draft(w.tokens, w.offsets, min_m, max_m, K, threads=os.cpu_count() or 1)
            index = measure_index(lib, pkg, w, dev, stream, want)
        ctx = None if args.no_ctx else measure_ctx(lib, pkg, w, dev, stream)
        if rank == 0:
            print(json.dumps({"metric": "µs per decode-loop step (draft, schedule, fuse, verify, append)",
                              "value": loop["loop_step_us"], "unit": "us/step", "n_gpus": world,
                              "higher_is_better": False, "data": "synthetic",
                              "config": {"workload": args.workload, "B": B, "history_tokens": w.total_tokens,
                                         "seed": seed},
                              "loop_steps": loop, "index": index, "context_cache": ctx}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    def step(i: int, handle: int):
        j = i % ncopy
        rc = lib.lookup_draft(tok_p[j], off_p[j], B, min_m, max_m, K, dp, lp, pp, handle)
        if rc != 0:
            raise pkg.LookupDraftError(rc, lib)

    clocks = ClockSampler(dev.index, enabled=not args.no_clocks)
    torch.cuda.synchronize(dev)

    # warm-up: eager steps, then graph capture (one graph per rotation of the copies)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i, h)
    stream.synchronize()
    # graphs: one whole rotation (steps over copies 0 .. ncopy-1) and, for K not a
    # multiple of ncopy, the first K mod ncopy steps of one.  The untimed replays
    # run whole rotations only, so the timed region starts at copy 0, the least
    # recently read: every timed step reads a copy last read ncopy steps earlier,
    # with (ncopy - 1) other copies (> 2x L2) read in between.
    full_reps, tail = divmod(args.steps, ncopy)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            hc = int(torch.cuda.current_stream().cuda_stream)
            for i in range(n):
                step(i, hc)
        return g

    # the library counts the launches it enqueues; a capture enqueues each once
    n0 = lib.lookup_draft_launch_count()
    g_full = capture(ncopy)
    n1 = lib.lookup_draft_launch_count()
    g_tail = capture(tail) if tail else None
    n2 = lib.lookup_draft_launch_count()
    timed_launches = int((n1 - n0) * full_reps + (n2 - n1))
    clock_hz = float(getattr(torch.cuda.get_device_properties(dev), "clock_rate", 2_000_000)) * 1000.0
    with torch.cuda.stream(stream):
        for _ in range(3):                           # first launches upload the graphs
            for g in (g_tail, g_full):
                if g is not None:
                    g.replay()
        t_end = time.perf_counter() + args.settle_s  # untimed replays: clocks settle under load
        while True:
            g_full.replay()
            stream.synchronize()
            if time.perf_counter() >= t_end:
                break

    # timed region: exactly K steps.  A short device-side sleep ahead of the start
    # event lets the host enqueue the replays first, so the events time the steps
    # on the device, not the host's graph submission.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(200e-6 * clock_hz))
        ev0.record(stream)
        for _ in range(full_reps):
            g_full.replay()
        if g_tail is not None:
            g_tail.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    us_per_step = 1000.0 * ms_total / args.steps

    # spread: whole rotations replayed one by one, each between its own events
    n_spread = 40
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_spread)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(200e-6 * clock_hz))
        for a, b in evs:
            a.record(stream)
            g_full.replay()
            b.record(stream)
    torch.cuda.synchronize(dev)
    per_rep = sorted(1000.0 * a.elapsed_time(b) / ncopy for a, b in evs)
    spread = {q: round(max_over_ranks(float(np.percentile(per_rep, v)), dist, dev), 3)
              for q, v in (("p10", 10), ("p50", 50), ("p90", 90))}
    spread.update({"replays": n_spread, "steps_per_replay": ncopy,
                   "what": "us per step of single whole-rotation graph replays, each between its own CUDA events"})
    del g_full, g_tail

    # eager: the same K steps as direct calls
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            step(i, h)
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    eager_us = 1000.0 * max_over_ranks(ev0.elapsed_time(ev1), dist, dev) / args.steps

    # roofline: the scan kernel alone.  (a) back to back: ncopy scan launches over
    # the rotating copies captured in one CUDA graph, replayed; CUDA events around
    # the replays on the launching stream give the mean duration per launch.
    # (b) isolated: events around each single launch (includes the event gaps).
    def scan_call(j: int, handle: int):
        rc = lib.lookup_draft_scan(tok_p[j], off_p[j], B, min_m, max_m, wsp, ws_bytes, handle)
        if rc != 0:
            raise pkg.LookupDraftError(rc, lib)

    def fill_call(j: int, handle: int):
        rc = lib.lookup_draft_fill(tok_p[j], off_p[j], B, min_m, max_m, K, wsp, ws_bytes,
                                   dp, lp, pp, None, handle)
        if rc != 0:
            raise pkg.LookupDraftError(rc, lib)

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            hc = int(torch.cuda.current_stream().cuda_stream)
            for j in range(ncopy):
                fn(j, hc)
        return g

    def time_graph(g, reps: int) -> float:
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return 1000.0 * ev0.elapsed_time(ev1) / (reps * ncopy)

    reps = max(10, min(200, args.steps // ncopy))
    scan_us = max_over_ranks(time_graph(graph_of(scan_call), reps), dist, dev)
    floor = time_read_floor(lib, pkg, toks, w.history_bytes, dev, stream, reps)
    floor_us = max_over_ranks(floor["us"], dist, dev)
    fill_us = max_over_ranks(time_graph(graph_of(fill_call), reps), dist, dev)
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(ncopy)]
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(ncopy)]
    iso_ms = []
    for rep in range(4):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(2e-3 * clock_hz))   # host runs ahead: no gaps between launches
            for j in range(ncopy):
                ea[j].record(stream)
                scan_call(j, h)
                eb[j].record(stream)
                fill_call(j, h)
        stream.synchronize()
        if rep:
            iso_ms += [ea[j].elapsed_time(eb[j]) for j in range(ncopy)]
    scan_iso_us = 1000.0 * max_over_ranks(statistics.fmean(iso_ms), dist, dev)

    loop = None
    if not args.no_loop:
        loop = measure_loop(lib, pkg, w, dev, stream, toks, offs, reps)
    index = None
    if not args.no_index:
        import oracle
        want = oracle.lookup_draft(w.tokens, w.offsets, min_m, max_m, K, threads=os.cpu_count() or 1)
        index = measure_index(lib, pkg, w, dev, stream, want)
    ctx = None if args.no_ctx else measure_ctx(lib, pkg, w, dev, stream)
    workloads = None
    if not args.no_workloads:
        workloads = measure_workloads(lib, pkg, dev, stream, list(gen.DEFAULT_SEED), 1000 * rank, reps)

    # e2e: host buffers through lookup_draft_host, copies inside every step
    h_tok = tok_host.pin_memory()
    h_off = off_host.pin_memory()
    h_draft = torch.empty((B, K), dtype=torch.int32).pin_memory()
    h_len = torch.empty(B, dtype=torch.int32).pin_memory()
    h_pos = torch.empty(B, dtype=torch.int32).pin_memory()
    args_host = (h_tok.data_ptr(), h_off.data_ptr(), B, min_m, max_m, K,
                 h_draft.data_ptr(), h_len.data_ptr(), h_pos.data_ptr(), h)
    for _ in range(3):
        lib.lookup_draft_host(*args_host)
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    barrier(dist, dev)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        rc = lib.lookup_draft_host(*args_host)
        if rc != 0:
            raise pkg.LookupDraftError(rc, lib)
    e2e_us = 1e6 * max_over_ranks(time.perf_counter() - t0, dist, dev) / n_e2e
    clocks.stop()

    # outputs must be the oracle's (checked on request 0..B of the last step's copy)
    import oracle
    o_draft, o_len, o_pos, _ = oracle.lookup_draft(w.tokens, w.offsets, min_m, max_m, K,
                                                   threads=os.cpu_count() or 1)
    parity = (np.array_equal(draft.cpu().numpy(), o_draft) and np.array_equal(length.cpu().numpy(), o_len)
              and np.array_equal(pos.cpu().numpy(), o_pos)
              and np.array_equal(h_draft.numpy(), o_draft) and np.array_equal(h_len.numpy(), o_len))

    cpu = None
    if rank == 0:
        cpu = cpu_baseline(w, args.cpu_budget_s)
    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return

    hist_bytes = w.history_bytes
    peak, peak_kind = measured_hbm_peak()
    achieved = hist_bytes / (scan_us * 1e-6) / 1e9
    traffic = recorded_traffic(args.workload)
    line = {
        "metric": METRIC,
        "value": round(us_per_step, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us_per_step / 1000.0, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "data": "synthetic",
        "config": {
            "workload": args.workload,
            "description": gen.DESCRIPTION[args.workload],
            "B": B, "history_tokens": w.total_tokens, "history_bytes": hist_bytes,
            "min_m": min_m, "max_m": max_m, "K": K, "seed": seed,
            "l2": f"inputs larger than L2 in rotation: the {args.steps} timed steps read device copies "
                  f"0, 1, ... (mod {ncopy}) of the batch, each last read {ncopy} steps earlier with "
                  f"{(ncopy - 1) * hist_bytes / 2**20:.0f} MiB of other copies read in between "
                  f"(> 2x L2 of {l2 / 2**20:.0f} MiB); {ncopy} copies, "
                  f"{ncopy * hist_bytes / 2**20:.0f} MiB in all",
            "launch": (f"lookup_draft calls captured in a CUDA graph of {ncopy} steps (one rotation), "
                       f"replayed {full_reps}x" + (f", then a graph of the first {tail}" if tail else "")),
            "parallelism": f"replicas x{world} (one batch per GPU, no exchange)",
        },
        "history_gbs_per_step": round(world * hist_bytes / (us_per_step * 1e-6) / 1e9, 1),
        "step_us_spread": spread,
        "eager_us_per_step": round(eager_us, 3),
        "scan_us": round(scan_us, 3),
        "scan_us_isolated": round(scan_iso_us, 3),
        "fill_us": round(fill_us, 3),
        "roofline": {
            "bound": "hbm",
            "kernel": "scan_kernel",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_kind": f"{peak_kind} copy bandwidth",
            "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "algorithmic_bytes_per_launch": hist_bytes,
            "traffic": traffic,
            "read_floor": {
                "kernel": "read_floor_bulk_kernel" if floor["shape"].startswith("bulk") else "read_floor_kernel",
                "us": round(floor_us, 3),
                "achieved": round(hist_bytes / (floor_us * 1e-6) / 1e9, 1),
                "frac": round(hist_bytes / (floor_us * 1e-6) / 1e9 / peak, 4),
                "shape": floor["shape"],
                "scan_vs_read_floor": round(floor_us / scan_us, 3),
                "what": "one launch that only streams the same bytes, timed like the scan: the best of "
                        "16-byte loads and bulk copies into shared memory (" +
                        ", ".join(floor_shape_name(a, b) for a, b in FLOOR_SHAPES) + ")",
            },
        },
        "e2e": {
            "value": round(e2e_us, 3),
            "unit": "us/step",
            "h2d_bytes_per_step": int(w.tokens.nbytes + w.offsets.nbytes),
            "d2h_bytes_per_step": int(4 * B * K + 8 * B),
            "steps": n_e2e,
        },
        "cpu_baseline": cpu,
        "loop_steps": loop,
        "index": index,
        "context_cache": ctx,
        "workloads": workloads,
        "gpu_launches": timed_launches,
        "parity_with_oracle": bool(parity),
        "clocks": clocks.summary(),
        "gpu": torch.cuda.get_device_name(dev),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------- decode loop ----
LOOP_H, LOOP_T = 7, 8            # head and tail of the verify block (HyperQwen article, "第2步")


def measure_loop(lib, pkg, w, dev, stream, toks, offs, reps: int) -> dict:
    """Times of the decode-loop steps around the draft on the bench's batch.

    Each entry point is captured ncopy times back to back in one CUDA graph
    (inputs rotating over the device copies of the batch, so the append reads
    every history from HBM) and replayed; CUDA events on the launching stream
    give the mean time per call.  ``loop_step_us`` is one whole decode-loop
    step: draft with mlen (K = H + T), scheduling, fusion, greedy verification
    and the append of the committed tokens to every history;
    ``loop_step_plan_us`` the same step with scheduling and fusion in one launch
    (lookup_plan), ``loop_step_draft_plan_us`` with the draft, scheduling and
    fusion in two (lookup_draft_plan)."""
    import numpy as np
    import torch

    import gen

    H, T = LOOP_H, LOOP_T
    P = H + T
    K = H + T
    B, ncopy = w.B, len(toks)
    i32 = torch.int32
    tok_p = [t.data_ptr() for t in toks]
    off_p = [o.data_ptr() for o in offs]

    def check(rc):
        if rc != 0:
            raise pkg.LookupDraftError(rc, lib)

    # inputs: this batch's lookup drafts and match lengths, a synthetic draft model
    # that proposes the lookup head for a third of the requests, a synthetic target
    # that agrees with the block on a random prefix
    draft, length, pos, mlen = pkg.lookup_draft_ex(toks[0], offs[0], w.min_m, w.max_m, K, stream=stream)
    torch.cuda.synchronize(dev)
    rng = gen.rng_for(w.seed, 500)
    md_h = rng.integers(0, 50, size=(B, H), dtype=np.int64).astype(np.int32)
    pick = rng.random(B) < 0.33
    md_h[pick] = draft.cpu().numpy()[pick, :H]
    model_draft = torch.from_numpy(md_h).to(dev)
    state = torch.zeros((B, 3), dtype=i32, device=dev)
    long_block = torch.zeros(B, dtype=i32, device=dev)
    committed = torch.full((B,), H + T + 1, dtype=i32, device=dev)
    block = torch.empty((B, P), dtype=i32, device=dev)
    blen = torch.empty(B, dtype=i32, device=dev)
    pm = torch.empty((B, P), dtype=i32, device=dev)
    with torch.cuda.stream(stream):
        pkg.lookup_fuse(draft, mlen, model_draft, None, H, T, out=(block, blen, pm), stream=stream)
    torch.cuda.synchronize(dev)
    blk_h = block.cpu().numpy()
    tg_h = rng.integers(0, 50, size=(B, P + 1), dtype=np.int64).astype(np.int32)
    f = rng.integers(0, P + 1, size=B)
    for r in range(B):
        tg_h[r, :f[r]] = blk_h[r, :f[r]]
    target = torch.from_numpy(tg_h).to(dev)
    _, _, _, p_h, q_h, pm_h, u_h = gen.loop_verify_inputs(B, P, w.seed)
    probs, qprobs, u = (torch.from_numpy(a).to(dev) for a in (p_h, q_h, u_h))
    accepted = torch.empty(B, dtype=i32, device=dev)
    commit = torch.empty((B, P + 1), dtype=i32, device=dev)
    ncommit = torch.empty(B, dtype=i32, device=dev)
    cap = max(int(t.numel()) for t in toks) + B * (P + 1)
    out_t = [torch.empty(cap, dtype=i32, device=dev) for _ in range(ncopy)]
    out_o = [torch.empty(B + 1, dtype=torch.int64, device=dev) for _ in range(ncopy)]
    dp, lp, pp, mp = draft.data_ptr(), length.data_ptr(), pos.data_ptr(), mlen.data_ptr()

    def fuse(j, hs):
        check(lib.lookup_fuse(dp, mp, model_draft.data_ptr(), long_block.data_ptr(), B, K, H, T, 8, 6, 2, 4,
                              block.data_ptr(), blen.data_ptr(), pm.data_ptr(), hs))

    def schedule(j, hs):
        check(lib.lookup_schedule(mp, committed.data_ptr(), B, H, T, 4, 1, 2, 3, state.data_ptr(),
                                  long_block.data_ptr(), hs))

    def plan(j, hs):
        check(lib.lookup_plan(dp, mp, model_draft.data_ptr(), committed.data_ptr(), B, K, H, T, 8, 6, 2, 4, 1, 2, 3,
                              state.data_ptr(), long_block.data_ptr(), block.data_ptr(), blen.data_ptr(),
                              pm.data_ptr(), hs))

    acc = torch.full((B, 5), 0.5, dtype=torch.float32, device=dev)
    prev = torch.zeros((B, 3), dtype=i32, device=dev)
    choice = torch.empty(B, dtype=i32, device=dev)

    def policy(j, hs):                                   # the draft-source controller
        check(lib.lookup_policy(mp, accepted.data_ptr(), B, H, 3, 1.3, 1.1, 0.8, 0.125, 0.05, 6, 8, 12, acc.data_ptr(),
                                prev.data_ptr(), choice.data_ptr(), hs))

    def verify_greedy(j, hs):
        check(lib.lookup_verify(block.data_ptr(), blen.data_ptr(), target.data_ptr(), None, None, None, None,
                                B, P, accepted.data_ptr(), commit.data_ptr(), ncommit.data_ptr(), hs))

    def verify_sampled(j, hs):
        check(lib.lookup_verify(block.data_ptr(), blen.data_ptr(), target.data_ptr(), probs.data_ptr(),
                                qprobs.data_ptr(), pm.data_ptr(), u.data_ptr(), B, P, accepted.data_ptr(),
                                commit.data_ptr(), ncommit.data_ptr(), hs))

    def append(j, hs):
        check(lib.lookup_append(tok_p[j], off_p[j], commit.data_ptr(), ncommit.data_ptr(), B, P + 1,
                                out_t[j].data_ptr(), out_o[j].data_ptr(), hs))

    def draft_ex(j, hs):
        check(lib.lookup_draft_ex(tok_p[j], off_p[j], B, w.min_m, w.max_m, K, dp, lp, pp, mp, hs))

    def loop_step(j, hs):
        draft_ex(j, hs)
        schedule(j, hs)
        fuse(j, hs)
        verify_greedy(j, hs)
        append(j, hs)

    def loop_step_plan(j, hs):                          # scheduling and fusion in one launch
        draft_ex(j, hs)
        plan(j, hs)
        verify_greedy(j, hs)
        append(j, hs)

    def draft_plan(j, hs):                              # draft, scheduling and fusion in two launches
        check(lib.lookup_draft_plan(tok_p[j], off_p[j], B, w.min_m, w.max_m, model_draft.data_ptr(),
                                    committed.data_ptr(), H, T, 8, 6, 2, 4, 1, 2, 3, state.data_ptr(),
                                    long_block.data_ptr(), block.data_ptr(), blen.data_ptr(), pm.data_ptr(), mp,
                                    None, hs))

    def loop_step_draft_plan(j, hs):
        draft_plan(j, hs)
        verify_greedy(j, hs)
        append(j, hs)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = {}                                        # kernels per call, counted by the library at capture

    def timed(fn) -> float:
        with torch.cuda.stream(stream):
            for j in range(ncopy):                      # eager warm-up
                fn(j, int(stream.cuda_stream))
        g = torch.cuda.CUDAGraph()
        c0 = lib.lookup_draft_launch_count()
        with torch.cuda.graph(g, stream=stream):
            hc = int(torch.cuda.current_stream().cuda_stream)
            for j in range(ncopy):
                fn(j, hc)
        n = lib.lookup_draft_launch_count() - c0
        launches[fn.__name__] = n // ncopy if n % ncopy == 0 else n / ncopy
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return 1000.0 * ev0.elapsed_time(ev1) / (reps * ncopy)

    verify_sampled(0, int(stream.cuda_stream))            # a valid commit/ncommit before the append
    res = {
        "H": H, "T": T,
        "fuse_us": timed(fuse),
        "schedule_us": timed(schedule),
        "plan_us": timed(plan),
        "policy_us": timed(policy),
        "verify_greedy_us": timed(verify_greedy),
        "verify_sampled_us": timed(verify_sampled),
        "append_us": timed(append),
        "loop_step_us": timed(loop_step),
        "loop_step_plan_us": timed(loop_step_plan),
        "draft_plan_us": timed(draft_plan),
        "loop_step_draft_plan_us": timed(loop_step_draft_plan),
    }
    # the append's algorithmic bytes: every history token read and written once,
    # the committed tokens read and written, the counts and both offset arrays
    committed_tokens = int(ncommit.sum().item())
    res["loop_step_committed_per_request"] = round(committed_tokens / max(B, 1), 2)
    append_bytes = 8 * w.total_tokens + 8 * committed_tokens + 4 * B + 16 * (B + 1)
    res = {k: (round(v, 3) if isinstance(v, float) else v) for k, v in res.items()}
    res["append_algorithmic_bytes"] = append_bytes
    res["append_gbs"] = round(append_bytes / (res["append_us"] * 1e-6) / 1e9, 1)
    for name in ("loop_step", "loop_step_plan", "loop_step_draft_plan", "draft_plan", "append"):
        res[f"{name}_launches"] = launches[name]
    res["method"] = (f"each call captured {ncopy}x back to back in a CUDA graph over rotating input copies, "
                     f"{reps} replays, CUDA events on the launching stream")
    return res


# ------------------------------------------------------- n-gram index ----
INDEX_SPARE = 2048               # tokens of room per request for the timed appends


def measure_index(lib, pkg, w, dev, stream, want) -> dict:
    """The incremental n-gram index on the bench's batch (histories laid out in
    slabs with INDEX_SPARE tokens of room each): build time, index size, the
    draft from the index (which must equal the oracle's `want`), the in-place
    append of 8 committed tokens per request, and one whole decode-loop step on
    the index (draft, schedule, fuse, greedy verify, append) three ways: five
    entry points (``loop_step_us``), the draft with scheduling and fusion in one
    (``loop_step_plan_us``), and that plus verification with the append in one
    (``loop_step_two_call_us``), each from the same starting histories.  Each call is
    captured back to back in a CUDA graph and timed with CUDA events on its
    stream; the index is larger than L2 and its accesses are scattered."""
    import numpy as np
    import torch

    import gen

    H, T = LOOP_H, LOOP_T
    P = H + T
    B = w.B
    i32 = torch.int32
    st, base_h, len_h, cap_h = gen.slabs_from_batch(w.tokens, w.offsets, INDEX_SPARE, seed=w.seed)
    tokens = torch.from_numpy(st).to(dev)
    base = torch.from_numpy(base_h).to(dev)
    length = torch.from_numpy(len_h).to(dev)
    cap = torch.from_numpy(cap_h).to(dev)
    idx = pkg.NgramIndex(st.shape[0], w.min_m, w.max_m, device=dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def check(rc):
        if rc != 0:
            raise pkg.LookupDraftError(rc, lib)

    torch.cuda.synchronize(dev)
    builds = []
    for _ in range(3):
        with torch.cuda.stream(stream):
            ev0.record(stream)
            idx.build(tokens, base, length, stream=stream)
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        builds.append(ev0.elapsed_time(ev1))

    K = w.K
    draft = torch.empty((B, max(K, P)), dtype=i32, device=dev)
    dl, dp, dm = (torch.empty(B, dtype=i32, device=dev) for _ in range(3))
    with torch.cuda.stream(stream):
        out = pkg.lookup_index_draft(tokens, base, length, w.min_m, w.max_m, K, idx.memory, idx.slots,
                                     out=(draft[:, :K].contiguous(), dl, dp, dm), with_fallback=True, stream=stream)
    torch.cuda.synchronize(dev)
    parity = (np.array_equal(out[0].cpu().numpy(), want[0]) and np.array_equal(dl.cpu().numpy(), want[1])
              and np.array_equal(dp.cpu().numpy(), want[2]))
    fallbacks = int(out[4].sum().item())

    hs = int(stream.cuda_stream)
    tp, bp, lp, cp = tokens.data_ptr(), base.data_ptr(), length.data_ptr(), cap.data_ptr()
    mem = idx.memory.data_ptr()

    def draft_call(h, k=K):
        check(lib.lookup_index_draft(tp, bp, lp, B, w.min_m, w.max_m, k, mem, idx.slots, 64, draft.data_ptr(),
                                     dl.data_ptr(), dp.data_ptr(), dm.data_ptr(), None, h))

    launches = {}                                        # kernels per call, counted by the library at capture

    def timed(fn, per_graph: int, reps: int) -> float:
        g = torch.cuda.CUDAGraph()
        c0 = lib.lookup_draft_launch_count()
        with torch.cuda.graph(g, stream=stream):
            hc = int(torch.cuda.current_stream().cuda_stream)
            for _ in range(per_graph):
                fn(hc)
        n = lib.lookup_draft_launch_count() - c0
        launches[fn.__name__] = n // per_graph if n % per_graph == 0 else n / per_graph
        with torch.cuda.stream(stream):
            g.replay()
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return 1000.0 * ev0.elapsed_time(ev1) / (reps * per_graph)

    draft_us = timed(draft_call, 32, 20)

    # in-place append: 8 committed tokens per request per call (64 calls: 512 tokens of room)
    rng = gen.rng_for(w.seed, 501)
    W8 = 8
    commit8 = torch.from_numpy(rng.integers(0, 50, size=(B, W8)).astype(np.int32)).to(dev)
    n8 = torch.full((B,), W8, dtype=i32, device=dev)
    status = torch.empty(B, dtype=i32, device=dev)

    def append_call(h):
        check(lib.lookup_index_append(tp, bp, lp, cp, commit8.data_ptr(), n8.data_ptr(), B, W8, w.min_m, w.max_m,
                                      mem, idx.slots, 64, status.data_ptr(), h))

    append_us = timed(append_call, 16, 3)                 # 16 (capture is not run) + 16 + 48 calls

    # the decode-loop step on the index: at most P + 1 = 16 tokens per request per step
    model_draft = torch.from_numpy(rng.integers(0, 50, size=(B, H)).astype(np.int32)).to(dev)
    state = torch.zeros((B, 3), dtype=i32, device=dev)
    long_block = torch.zeros(B, dtype=i32, device=dev)
    committed = torch.full((B,), H + T + 1, dtype=i32, device=dev)   # as in the scan's loop step
    block = torch.empty((B, P), dtype=i32, device=dev)
    blen = torch.empty(B, dtype=i32, device=dev)
    pm = torch.empty((B, P), dtype=i32, device=dev)
    target = torch.from_numpy(rng.integers(0, 50, size=(B, P + 1)).astype(np.int32)).to(dev)
    # Verification by the sampled rule (u * 1 < p) with draws that accept exactly the
    # first f[r] positions, f uniform in [0, P] as the scan's loop step's target
    # agreement: the same commits per step whatever tokens the growing histories
    # put in the block (a fixed greedy target would agree with almost none).
    f = rng.integers(0, P + 1, size=B)
    probs = torch.full((B, P), 0.5, dtype=torch.float32, device=dev)
    u = torch.from_numpy(np.where(np.arange(P)[None, :] < f[:, None], 0.0, 0.75).astype(np.float32)).to(dev)
    pp, up = probs.data_ptr(), u.data_ptr()
    accepted = torch.empty(B, dtype=i32, device=dev)
    commit = torch.empty((B, P + 1), dtype=i32, device=dev)
    ncommit = torch.empty(B, dtype=i32, device=dev)

    def loop_call(h):
        draft_call(h, P)
        check(lib.lookup_schedule(dm.data_ptr(), committed.data_ptr(), B, H, T, 4, 1, 2, 3, state.data_ptr(),
                                  long_block.data_ptr(), h))
        check(lib.lookup_fuse(draft.data_ptr(), dm.data_ptr(), model_draft.data_ptr(), long_block.data_ptr(), B,
                              P, H, T, 8, 6, 2, 4, block.data_ptr(), blen.data_ptr(), pm.data_ptr(), h))
        check(lib.lookup_verify(block.data_ptr(), blen.data_ptr(), target.data_ptr(), pp, None, None, up, B, P,
                                accepted.data_ptr(), commit.data_ptr(), ncommit.data_ptr(), h))
        check(lib.lookup_index_append(tp, bp, lp, cp, commit.data_ptr(), ncommit.data_ptr(), B, P + 1, w.min_m,
                                      w.max_m, mem, idx.slots, 64, status.data_ptr(), h))

    loop_us = timed(loop_call, 16, 4)                     # 80 steps: at most 1280 tokens of room
    torch.cuda.synchronize(dev)
    room_ok = bool((status == 0).all().item())

    def restart():
        """The original histories again (lengths restored, the index rebuilt,
        untimed), so the next loop's appends have the same room."""
        length.copy_(torch.from_numpy(len_h))
        state.zero_()
        with torch.cuda.stream(stream):
            idx.build(tokens, base, length, stream=stream)
        torch.cuda.synchronize(dev)

    # the same step with the draft, scheduling and fusion in one launch
    # (lookup_index_draft_plan), from the original histories
    restart()
    dlen = torch.empty(B, dtype=i32, device=dev)
    fb = torch.empty(B, dtype=i32, device=dev)

    def loop_plan_call(h):
        check(lib.lookup_index_draft_plan(tp, bp, lp, B, w.min_m, w.max_m, mem, idx.slots, 64,
                                          model_draft.data_ptr(), committed.data_ptr(), H, T, 8, 6, 2, 4, 1, 2, 3,
                                          state.data_ptr(), long_block.data_ptr(), block.data_ptr(), blen.data_ptr(),
                                          pm.data_ptr(), dm.data_ptr(), dlen.data_ptr(), fb.data_ptr(), h))
        check(lib.lookup_verify(block.data_ptr(), blen.data_ptr(), target.data_ptr(), pp, None, None, up, B, P,
                                accepted.data_ptr(), commit.data_ptr(), ncommit.data_ptr(), h))
        check(lib.lookup_index_append(tp, bp, lp, cp, commit.data_ptr(), ncommit.data_ptr(), B, P + 1, w.min_m,
                                      w.max_m, mem, idx.slots, 64, status.data_ptr(), h))

    loop_plan_us = timed(loop_plan_call, 16, 4)           # 80 steps again
    torch.cuda.synchronize(dev)
    room_ok = room_ok and bool((status == 0).all().item())

    # and with verification and the append in one launch too (lookup_index_verify_append)
    restart()

    def loop_two_call(h):
        check(lib.lookup_index_draft_plan(tp, bp, lp, B, w.min_m, w.max_m, mem, idx.slots, 64,
                                          model_draft.data_ptr(), committed.data_ptr(), H, T, 8, 6, 2, 4, 1, 2, 3,
                                          state.data_ptr(), long_block.data_ptr(), block.data_ptr(), blen.data_ptr(),
                                          pm.data_ptr(), dm.data_ptr(), dlen.data_ptr(), fb.data_ptr(), h))
        check(lib.lookup_index_verify_append(block.data_ptr(), blen.data_ptr(), target.data_ptr(), pp, None, None,
                                             up, B, P, tp, bp, lp, cp, w.min_m, w.max_m, mem, idx.slots, 64,
                                             accepted.data_ptr(), commit.data_ptr(), ncommit.data_ptr(),
                                             status.data_ptr(), h))

    loop_two_us = timed(loop_two_call, 16, 4)             # 80 steps again
    torch.cuda.synchronize(dev)
    room_ok = room_ok and bool((status == 0).all().item())
    committed_mean = float(ncommit.float().mean().item())  # the last step's, per request

    # prompt-lookup decoding without a draft model: the block is the previous
    # step's lookup draft (P tokens), in two alternating buffers; one step is
    # verification, the append and the next draft
    drafts = [torch.full((B, P), -1, dtype=i32, device=dev) for _ in range(2)]
    dlens = [torch.zeros(B, dtype=i32, device=dev) for _ in range(2)]
    dpos, dml = torch.empty(B, dtype=i32, device=dev), torch.empty(B, dtype=i32, device=dev)
    turn = [0]

    def plain_one_call(h):
        a, b2 = turn[0] % 2, (turn[0] + 1) % 2
        turn[0] += 1
        check(lib.lookup_index_verify_append_draft(drafts[a].data_ptr(), dlens[a].data_ptr(), target.data_ptr(), pp,
                                                   None, None, up, B, P, tp, bp, lp, cp, w.min_m, w.max_m, mem,
                                                   idx.slots, 64, P, accepted.data_ptr(), commit.data_ptr(),
                                                   ncommit.data_ptr(), status.data_ptr(), drafts[b2].data_ptr(),
                                                   dlens[b2].data_ptr(), dpos.data_ptr(), dml.data_ptr(), None, h))

    def plain_two_calls(h):
        a, b2 = turn[0] % 2, (turn[0] + 1) % 2
        turn[0] += 1
        check(lib.lookup_index_verify_append(drafts[a].data_ptr(), dlens[a].data_ptr(), target.data_ptr(), pp, None,
                                             None, up, B, P, tp, bp, lp, cp, w.min_m, w.max_m, mem, idx.slots, 64,
                                             accepted.data_ptr(), commit.data_ptr(), ncommit.data_ptr(),
                                             status.data_ptr(), h))
        check(lib.lookup_index_draft(tp, bp, lp, B, w.min_m, w.max_m, P, mem, idx.slots, 64, drafts[b2].data_ptr(),
                                     dlens[b2].data_ptr(), dpos.data_ptr(), dml.data_ptr(), None, h))

    restart()
    plain_two_us = timed(plain_two_calls, 16, 4)          # 80 steps from the original histories
    torch.cuda.synchronize(dev)
    room_ok = room_ok and bool((status == 0).all().item())
    restart()
    for x in drafts:
        x.fill_(-1)
    for x in dlens:
        x.zero_()
    plain_one_us = timed(plain_one_call, 16, 4)
    torch.cuda.synchronize(dev)
    room_ok = room_ok and bool((status == 0).all().item())
    plain_committed = float(ncommit.float().mean().item())
    # the replays' last step wrote buffer 0 (16 steps per graph): the draft of the
    # grown histories, which must be the oracle's
    import oracle
    grown_t, grown_o = gen.csr_of_slabs(tokens.cpu().numpy(), base_h, length.cpu().numpy())
    want_grown = oracle.lookup_draft(grown_t, grown_o, w.min_m, w.max_m, P, threads=os.cpu_count() or 1)
    plain_parity = (np.array_equal(drafts[0].cpu().numpy(), want_grown[0])
                    and np.array_equal(dlens[0].cpu().numpy(), want_grown[1]))
    total_tokens = int(st.shape[0])
    res = {
        "layout": f"slabs with {INDEX_SPARE} tokens of room per request",
        "index_bytes": int(idx.memory.numel()),
        "index_bytes_per_token": round(idx.memory.numel() / total_tokens, 1),
        "slots": idx.slots,
        "build_ms": round(statistics.median(builds), 3),
        "draft_us": round(draft_us, 3),
        "append8_us": round(append_us, 3),
        "loop_step_us": round(loop_us, 3),
        "loop_step_launches": launches["loop_call"],
        "loop_step_plan_us": round(loop_plan_us, 3),
        "loop_step_plan_launches": launches["loop_plan_call"],
        "loop_step_two_call_us": round(loop_two_us, 3),
        "loop_step_two_call_launches": launches["loop_two_call"],
        "loop_step_committed_per_request": round(committed_mean, 2),
        "loop_step_verify": "sampled rule, draws accepting the first f positions, f uniform in [0, P]",
        "plain_lookup_step_us": round(plain_one_us, 3),
        "plain_lookup_step_launches": launches["plain_one_call"],
        "plain_lookup_step_two_call_us": round(plain_two_us, 3),
        "plain_lookup_step_two_call_launches": launches["plain_two_calls"],
        "plain_lookup_committed_per_request": round(plain_committed, 2),
        "plain_lookup_parity_with_oracle": bool(plain_parity),
        "plain_lookup": "no draft model: the block is the previous step's lookup draft (P tokens); a step is "
                        "verification, the append and the next draft (lookup_index_verify_append_draft)",
        "draft_launches": launches["draft_call"],
        "append8_launches": launches["append_call"],
        "parity_with_oracle": bool(parity),
        "fallback_requests": fallbacks,
        "appends_fit": room_ok,
        "method": "calls captured back to back in CUDA graphs (32 drafts, 16 appends, 16 loop steps per graph), "
                  "CUDA events on the launching stream",
    }
    del idx
    return res


# -------------------------------------------------------- context cache ----
CTX_K = 8                        # context-cache drafts per request


def measure_ctx(lib, pkg, w, dev, stream) -> dict:
    """Context-cache drafting on the bench's batch (slabs with INDEX_SPARE tokens
    of room): build time, size, the draft of up to CTX_K tokens (checked against
    the oracle), and the in-place append of 8 committed tokens per request."""
    import numpy as np
    import torch

    import gen
    import oracle

    B = w.B
    i32 = torch.int32
    st, base_h, len_h, cap_h = gen.slabs_from_batch(w.tokens, w.offsets, INDEX_SPARE, seed=w.seed)
    tokens = torch.from_numpy(st).to(dev)
    base = torch.from_numpy(base_h).to(dev)
    length = torch.from_numpy(len_h).to(dev)
    cap = torch.from_numpy(cap_h).to(dev)
    cc = pkg.ContextCache(st.shape[0], 1, 4, device=dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    builds = []
    for _ in range(3):
        with torch.cuda.stream(stream):
            ev0.record(stream)
            cc.build(tokens, base, length, stream=stream)
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        builds.append(ev0.elapsed_time(ev1))
    draft = torch.empty((B, CTX_K), dtype=i32, device=dev)
    dlen = torch.empty(B, dtype=i32, device=dev)
    with torch.cuda.stream(stream):
        cc.draft(tokens, base, length, CTX_K, out=(draft, dlen), stream=stream)
    torch.cuda.synchronize(dev)
    wd, wl = oracle.ctx_draft(w.tokens, w.offsets, CTX_K, threads=os.cpu_count() or 1)
    parity = bool(np.array_equal(draft.cpu().numpy(), wd) and np.array_equal(dlen.cpu().numpy(), wl))

    def timed(fn, per_graph: int, reps: int) -> float:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(per_graph):
                fn()
        with torch.cuda.stream(stream):
            g.replay()
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return 1000.0 * ev0.elapsed_time(ev1) / (reps * per_graph)

    draft_us = timed(lambda: cc.draft(tokens, base, length, CTX_K, out=(draft, dlen), stream=stream), 32, 20)
    rng = gen.rng_for(w.seed, 502)
    commit = torch.from_numpy(rng.integers(0, 50, size=(B, 8)).astype(np.int32)).to(dev)
    n8 = torch.full((B,), 8, dtype=i32, device=dev)
    status = torch.empty(B, dtype=i32, device=dev)
    append_us = timed(lambda: cc.append(tokens, base, length, cap, commit, n8, status=status, stream=stream), 16, 3)
    torch.cuda.synchronize(dev)
    res = {
        "n_range": [1, 4], "K": CTX_K, "thresholds": "count >= 1, top next token >= 1/2, every n",
        "cache_bytes": int(cc.memory.numel()),
        "cache_bytes_per_token": round(cc.memory.numel() / st.shape[0], 1),
        "build_ms": round(statistics.median(builds), 3),
        "draft_us": round(draft_us, 3),
        "mean_draft_len": round(float(wl.mean()), 3),
        "append8_us": round(append_us, 3),
        "parity_with_oracle": parity,
        "appends_fit": bool((status == 0).all().item()),
        "method": "calls captured back to back in CUDA graphs (32 drafts, 16 appends per graph), "
                  "CUDA events on the launching stream",
    }
    del cc
    return res


# ----------------------------------------------------------- read floor ----
FLOOR_SHAPES = ((2, 512), (4, 256), (8, 256), (0, 0))   # CTAs per SM x threads; (0, 0): bulk copies (TMA)


def floor_shape_name(cps: int, thr: int) -> str:
    return "bulk copies, 1x512" if cps == 0 else f"{cps}x{thr}"


def time_read_floor(lib, pkg, toks, nbytes: int, dev, stream, reps: int) -> dict:
    """The plain streaming read of the same bytes, timed the way the scan is
    (ncopy launches over the rotating copies captured in one CUDA graph, replayed
    back to back, CUDA events on the launching stream): the best over 16-byte
    loads in a few launch shapes and bulk copies into shared memory (TMA, the
    scan's own way of reading)."""
    import torch
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ncopy = len(toks)
    best = None
    for cps, thr in FLOOR_SHAPES:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            hc = int(torch.cuda.current_stream().cuda_stream)
            for j in range(ncopy):
                if cps == 0:
                    rc = lib.lookup_draft_read_floor_bulk(toks[j].data_ptr(), nbytes, out.data_ptr(), hc)
                else:
                    rc = lib.lookup_draft_read_floor(toks[j].data_ptr(), nbytes, cps, thr, out.data_ptr(), hc)
                if rc != 0:
                    raise pkg.LookupDraftError(rc, lib)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        us = 1000.0 * ev0.elapsed_time(ev1) / (reps * ncopy)
        if int(out.item()) == -1:
            raise RuntimeError("the bulk read floor's wait ran out: the measurement is invalid")
        if best is None or us < best[0]:
            best = (us, floor_shape_name(cps, thr))
        del g
    return {"us": best[0], "shape": best[1]}


# ------------------------------------------------------------ workloads ----
SPREAD_SEEDS = (6, 7, 8, 9, 10)


def time_workload(lib, pkg, w, dev, stream, l2: int, reps_cap: int, with_floor: bool) -> dict:
    """The draft step and the scan on one workload, timed the way the main line
    times its own: ncopy calls over rotating device copies (> 2x L2 in total)
    captured in one CUDA graph, replayed back to back, CUDA events on the launching
    stream; the step's outputs against the oracle's on the whole batch."""
    import numpy as np
    import torch

    import oracle

    peak, _ = measured_hbm_peak()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    B, K = w.B, w.K
    ncopy = max(3, math.ceil(2 * l2 / max(w.history_bytes, 1)) + 1)
    tok_host, off_host = torch.from_numpy(w.tokens), torch.from_numpy(w.offsets)
    toks = [tok_host.to(dev) for _ in range(ncopy)]
    offs = [off_host.to(dev) for _ in range(ncopy)]
    draft = torch.empty((B, K), dtype=torch.int32, device=dev)
    length = torch.empty(B, dtype=torch.int32, device=dev)
    pos = torch.empty(B, dtype=torch.int32, device=dev)
    ws_bytes = pkg.workspace_bytes(B, dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    reps = max(10, min(reps_cap, 20000 // ncopy))

    def step(j, hc):
        rc = lib.lookup_draft(toks[j].data_ptr(), offs[j].data_ptr(), B, w.min_m, w.max_m, K,
                              draft.data_ptr(), length.data_ptr(), pos.data_ptr(), hc)
        if rc != 0:
            raise pkg.LookupDraftError(rc, lib)

    def scan(j, hc):
        rc = lib.lookup_draft_scan(toks[j].data_ptr(), offs[j].data_ptr(), B, w.min_m, w.max_m,
                                   ws.data_ptr(), ws_bytes, hc)
        if rc != 0:
            raise pkg.LookupDraftError(rc, lib)

    def timed(fn) -> float:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            hc = int(torch.cuda.current_stream().cuda_stream)
            for j in range(ncopy):
                fn(j, hc)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        return 1000.0 * ev0.elapsed_time(ev1) / (reps * ncopy)

    step_us = timed(step)
    got = (draft.cpu().numpy(), length.cpu().numpy(), pos.cpu().numpy())
    scan_us = timed(scan)
    want = oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, K, threads=os.cpu_count() or 1)
    parity = all(np.array_equal(a, b) for a, b in zip(got, want[:3]))
    gbs = w.history_bytes / (scan_us * 1e-6) / 1e9
    res = {"B": B, "history_bytes": int(w.history_bytes), "seed": int(w.seed),
           "step_us": round(step_us, 3), "scan_us": round(scan_us, 3),
           "scan_gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
    if with_floor:
        floor = time_read_floor(lib, pkg, toks, w.history_bytes, dev, stream, reps)
        res.update({"read_floor_us": round(floor["us"], 3),
                    "read_floor_frac": round(w.history_bytes / (floor["us"] * 1e-6) / 1e9 / peak, 4),
                    "scan_vs_read_floor": round(floor["us"] / scan_us, 3)})
    res.update({"copies": ncopy, "parity_with_oracle": bool(parity)})
    del toks, offs, ws
    torch.cuda.synchronize(dev)
    return res


SWEEP_LENGTHS = (4096, 8192, 16384, 25000, 50000, 100000, 200000, 400000)


def size_sweep(lib, pkg, dev, reps_cap: int) -> dict:
    """The step, the scan and the plain-read floor against history size: the
    recitation recipe (B = 64, gen.make_workload(..., length=L)) at each length of
    SWEEP_LENGTHS, timed by time_workload like the main line, each checked
    against the oracle.  A least-squares line time = fixed + bytes / rate is fitted
    to the scan's and to the floor's times; from it, the history size at which
    each would reach 60% of the measured copy bandwidth."""
    import numpy as np
    import torch

    import gen

    peak, _ = measured_hbm_peak()
    stream = torch.cuda.Stream(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2**20))
    points = []
    for L in SWEEP_LENGTHS:
        w = gen.make_workload("recitation25k", length=L)
        r = time_workload(lib, pkg, w, dev, stream, l2, reps_cap, True)
        r["L"] = L
        points.append(r)
    mb = np.array([p["history_bytes"] for p in points], dtype=np.float64)
    fit = {}
    for name, key in (("scan", "scan_us"), ("read_floor", "read_floor_us")):
        t = np.array([p[key] for p in points], dtype=np.float64)
        slope, fixed = np.polyfit(mb, t, 1)                  # us per byte, us
        rate = 1e-3 / slope                                  # GB/s (bytes / us / 1e3)
        # bytes b with b / (fixed + b / rate) = 0.6 * peak, if the rate allows it
        want = 0.6 * peak
        b60 = (want * fixed * 1e3 / (1.0 - want / rate)) if rate > want else None
        fit[name] = {"fixed_us": round(float(fixed), 3), "rate_gbs": round(float(rate), 1),
                     "rate_frac_of_peak": round(float(rate) / peak, 4),
                     "bytes_for_60pct": None if b60 is None else int(b60)}
    return {"metric": "µs per draft step, scan and plain read against history size", "unit": "us",
            "data": "synthetic", "peak_gbs": peak,
            "config": {"workload": "recitation recipe, B = 64, L in " + ", ".join(map(str, SWEEP_LENGTHS)),
                       "l2": "each size over rotating device copies (> 2x L2)"},
            "size_sweep": points, "fit": fit}


def measure_workloads(lib, pkg, dev, stream, names, seed_offset: int, reps_cap: int) -> dict:
    """Per workload: the step and the scan on its default seed (with the read floor
    of the same bytes), then on seeds 6-10 (step, scan, parity), each timed by
    time_workload; the scan's GB/s (4 bytes per history token) against the
    measured copy bandwidth."""
    import torch

    import gen

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    peak, peak_kind = measured_hbm_peak()
    out, seeds = {}, {}
    for name in names:
        w = gen.make_workload(name, gen.DEFAULT_SEED[name] + seed_offset)
        out[name] = time_workload(lib, pkg, w, dev, stream, l2, reps_cap, True)
        rows = []
        for sd in SPREAD_SEEDS:
            r = time_workload(lib, pkg, gen.make_workload(name, sd + seed_offset), dev, stream, l2, reps_cap, False)
            rows.append({k: r[k] for k in ("seed", "history_bytes", "step_us", "scan_us", "frac",
                                           "parity_with_oracle")})
        steps = sorted(r["step_us"] for r in rows)
        scans = sorted(r["scan_us"] for r in rows)
        seeds[name] = {"per_seed": rows,
                       "step_us_median": steps[len(steps) // 2], "step_us_min": steps[0], "step_us_max": steps[-1],
                       "scan_us_median": scans[len(scans) // 2], "scan_us_min": scans[0], "scan_us_max": scans[-1],
                       "parity_with_oracle": all(r["parity_with_oracle"] for r in rows)}
    return {"peak_gbs": peak, "peak_kind": f"{peak_kind} copy bandwidth",
            "method": "per workload: calls over rotating device copies (> 2x L2) captured in one CUDA graph, "
                      "replayed back to back; CUDA events on the launching stream",
            "workloads": out,
            "seeds": seeds,
            "seeds_what": f"the same timings on seeds {', '.join(map(str, SPREAD_SEEDS))} of each workload"}


# ------------------------------------------------------------------ CPU ----
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo", encoding="utf-8"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(w, budget_s: float) -> dict:
    """The oracle, as it stands, on the host cores: whole batches until the budget;
    then on one thread, the median of up to 5 whole batches."""
    import oracle
    cores = host_cores()
    oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=cores)   # warm
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=cores)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 1000:
            break
    one = []
    t1 = time.perf_counter()
    while len(one) < 5 and (not one or time.perf_counter() - t1 < budget_s):
        ts = time.perf_counter()
        oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=1)
        one.append(time.perf_counter() - ts)
    many_us, one_us = 1e6 * el / n, 1e6 * statistics.median(one)
    use_one = one_us < many_us        # small batches: dispatching to threads costs more than it saves
    return {"value": round(one_us if use_one else many_us, 1), "unit": "us/step",
            "cores": 1 if use_one else cores, "kind": "oracle",
            "sample": (f"the whole {w.name} batch ({w.B} requests, {w.total_tokens} tokens), "
                       + (f"median of {len(one)} runs on one thread (faster than {cores} threads here)" if use_one
                          else f"x {n} runs on {cores} threads, {el:.1f} s wall")),
            "all_cores_us": round(many_us, 1),
            "single_thread_us": round(one_us, 1),
            "single_thread_sample": f"median of {len(one)} whole batches on one thread",
            "cpu": cpu_model()}


def run_reference(args, rank: int, world: int):
    """The oracle as the comparison arm: per step, a slice of the batch's requests
    sized so that the whole run fits the budget; the time is scaled to the whole
    batch by history tokens."""
    if rank != 0:
        return
    import gen
    import oracle
    seed = gen.DEFAULT_SEED[args.workload] if args.seed is None else args.seed
    w = gen.make_workload(args.workload, seed)
    cores = host_cores()
    lens = (w.offsets[1:] - w.offsets[:-1])
    t0 = time.perf_counter()
    oracle.lookup_draft(w.tokens, w.offsets, w.min_m, w.max_m, w.K, threads=cores)
    full_s = time.perf_counter() - t0
    total_steps = args.steps + args.warmup
    per_step_budget = args.reference_budget_s / max(total_steps, 1)
    frac = min(1.0, per_step_budget / max(full_s, 1e-9))
    n_req = max(1, min(w.B, int(round(frac * w.B))))
    timed_s, timed_tokens = 0.0, 0
    for i in range(total_steps):
        lo = (i * n_req) % w.B
        hi = min(w.B, lo + n_req)
        sub_off = w.offsets[lo:hi + 1]
        t = time.perf_counter()
        oracle.lookup_draft(w.tokens[sub_off[0]:sub_off[-1]], sub_off - sub_off[0],
                            w.min_m, w.max_m, w.K, threads=cores)
        dt = time.perf_counter() - t
        if i >= args.warmup:
            timed_s += dt
            timed_tokens += int(lens[lo:hi].sum())
    # time per history token over the timed steps, times the tokens of one whole batch
    us_per_step = 1e6 * timed_s * w.total_tokens / max(timed_tokens, 1)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(us_per_step, 1),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us_per_step / 1000.0, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int32",
        "data": "synthetic",
        "config": {"workload": args.workload, "description": gen.DESCRIPTION[args.workload],
                   "B": w.B, "history_tokens": w.total_tokens, "history_bytes": w.history_bytes,
                   "min_m": w.min_m, "max_m": w.max_m, "K": w.K, "seed": seed},
        "cpu_baseline": {"value": round(us_per_step, 1), "unit": "us/step", "cores": cores,
                         "kind": "oracle",
                         "sample": f"per step {n_req} of {w.B} requests of the {w.name} batch, "
                                   f"time scaled to the whole batch by history tokens"},
        "e2e": {"value": round(us_per_step, 1), "unit": "us/step",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
