#!/usr/bin/env python3
"""Benchmark: sparse-MLA decode on GB300, one JSON line on stdout.

A step is one decode call over one batch.  The default workload is the
largest single-GPU shape of the T x context matrix: 64 rows x 128 heads at a
1M-token context (64-token pages, top-k 2048 with 5% invalid slots, window
128, 262144 compressed entries per row; 16.9M attended entries per call).
Inputs are resident in HBM; L2 is flushed (a 512 MB write) before every
timed step; each step replays a CUDA graph holding the call's two launches
(the decode kernel, then the merge kernel for split rows) and is timed with
CUDA events on that stream.

The same JSON line carries ``per_config``: the same measurement on the
DeepSeek-V4-like decode (32 x 32K), the MTP decode (16 x 4 tokens, H = 64),
the long-context ragged call (contexts 4K/100K/500K/1M, one graph capture
replayed with re-drawn lengths) and the long-context sweep shapes
(T in {16, 64} x context in {100K, 500K, 1M}).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

N > 1 runs N independent replicas (one per GPU, launched by torchrun); the
only cross-rank traffic is the barrier and the max-over-ranks of the timings.
``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload instead (rank 0 only).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA decode µs/call & query-rows/s; % of HBM/tensor roofline, 1×GB300"
KERNEL_NAME = "smla_decode_kernel"
DEFAULT_WORKLOAD = "sweep_T64_ctx1048576"
PER_CONFIG = ("dsv4", "mtp", "ragged", "sweep_T16_ctx102400", "sweep_T16_ctx512000", "sweep_T16_ctx1048576",
              "sweep_T64_ctx102400", "sweep_T64_ctx512000")
LAUNCHES_PER_CALL = 2  # smla_decode enqueues the decode kernel and the merge kernel
KERNEL_SRC = os.path.join(ROOT, "sparse_mla_decode_04_gb300", "csrc", "smla_decode.cu")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def make_workload(name: str, device):
    import smla_inputs as I

    if name == "dsv4":
        return I.dsv4(device=device)
    if name == "mtp":
        return I.mtp(device=device)
    if name == "ragged":
        return I.ragged(device=device)
    if name == "tiny":
        return I.tiny(device=device)
    m = re.fullmatch(r"sweep_T(\d+)_ctx(\d+)", name)
    if m:
        return I.sweep(int(m.group(1)), int(m.group(2)), device=device)
    raise SystemExit(f"unknown workload {name}")


def workload_config(p, num_splits, name):
    lens = p.meta["seq_lens"]
    return {
        "workload": p.name,
        "rows": p.num_rows, "heads": p.num_heads, "context": lens[0] if len(set(lens)) == 1 else lens,
        "topk": p.topk, "swa": p.meta["swa"], "compressed_per_row": int(p.cmp_len.max().item()),
        "page_size": 64, "paged": p.block_table is not None, "num_splits": num_splits,
        "valid_entries": int(p.valid_entries_per_row().sum()), "l2": "flushed (512 MB write) before each timed step",
        "kv_format": "fp8-e4m3 NoPE + UE8M0/64 + bf16 RoPE", "bench_name": name,
    }


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    """Hash of the decode kernel's sources (its translation unit and the
    headers it includes): comments and whitespace are left out, so that only
    a change to the compiled kernel makes recorded counters stale."""
    h = hashlib.sha256()
    csrc = os.path.dirname(KERNEL_SRC)
    files = [os.path.join(csrc, "smla_decode.cu"), os.path.join(csrc, "sm103_ptx.cuh"),
             os.path.join(csrc, "smla_internal.h"), os.path.join(ROOT, "include", "smla.h")]
    for path in files:
        with open(path) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(os.path.basename(path).encode())
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if its recorded source hash matches the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"ncu_{KERNEL_NAME}_{workload}.txt")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_hash = re.search(r"^source_hash:\s*(\S+)", txt, re.M)
    m_bytes = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", txt, re.M)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
def replica_max(x: float, device=None) -> float:
    """Max of a per-rank number over all ranks (the replicas' step time); the
    only cross-rank operation besides the barrier.  Identity without a group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(rows_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job rows/s: every rank decodes its own batch of rows_per_rank in
    parallel; the job takes as long as the slowest rank."""
    return rows_per_rank * world / (max_ms / 1e3)


# ---------------------------------------------------------------------------
def cpu_oracle_time(p, budget_s: float, max_rows=None):
    """Time the float64 oracle, row by row, on host cores until budget_s is
    spent; returns (seconds per row, rows timed, cores)."""
    import oracle

    kw = p.oracle_kwargs()
    rows = list(range(p.num_rows if max_rows is None else min(max_rows, p.num_rows)))
    done, spent = 0, 0.0
    for r in rows:
        t0 = time.perf_counter()
        oracle.decode(rows=[r], **kw)
        spent += time.perf_counter() - t0
        done += 1
        if spent >= budget_s:
            break
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            cores = min(cores, max(n))
    except Exception:
        pass
    return spent / done, done, cores


def run_reference(args):
    import torch

    world, rank, local = dist_env()
    if rank != 0:
        return 0
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    p = make_workload(args.workload, device)
    import sparse_mla_decode_04_gb300 as smla  # planner only, for the config line

    S = smla.smla_plan_num_splits(p.num_rows, p.num_heads, p.kv_len_estimate())
    # each step: the oracle on a bounded sample (rows) of the workload
    per_row, _, cores = cpu_oracle_time(p, budget_s=2.0, max_rows=2)
    sample_rows = max(1, min(p.num_rows, int(20.0 / max(args.steps + args.warmup, 1) / per_row)))
    import oracle

    kw = p.oracle_kwargs()
    for i in range(args.warmup):
        oracle.decode(rows=[i % p.num_rows], **kw)
    times = []
    for k in range(args.steps):
        rows = [(k * sample_rows + j) % p.num_rows for j in range(sample_rows)]
        t0 = time.perf_counter()
        oracle.decode(rows=rows, **kw)
        times.append((time.perf_counter() - t0) / sample_rows)
    sec_per_row = statistics.mean(times)
    value = 1.0 / sec_per_row
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "query-rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec_per_row * p.num_rows * 1e3,
        "us_per_call": sec_per_row * p.num_rows * 1e6,
        "ms_per_step_kind": (f"extrapolated: mean oracle time per row x {p.num_rows} rows; each step ran "
                             f"{sample_rows} row(s) of the call, not the whole call"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(p, S, args.workload),
        "cpu_baseline": {"value": value, "unit": "query-rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample_rows} of {p.num_rows} rows per step (float64 NumPy oracle, "
                                   f"time per call extrapolated to all rows)"},
        "e2e": {"value": value, "unit": "query-rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def roofline(flops: float, nbytes: float, t_s: float, peaks: dict) -> dict:
    """The slower of the algorithmic bytes at HBM bandwidth and the algorithmic
    flops at the bf16 tensor peak sets the bound; achieved is the work of that
    bound divided by the measured time."""
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_tc >= t_hbm:
        achieved, peak, unit, bound = flops / t_s / 1e12, peaks["bf16_tflops"], "TFLOP/s", "tensor"
    else:
        achieved, peak, unit, bound = nbytes / t_s / 1e9, peaks["hbm_gbs"], "GB/s", "hbm"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "t_roofline_us": max(t_tc, t_hbm) * 1e6}


def time_call(p, S, ws, steps: int, warmup: int, flush_buf, stream, redraw: bool = False):
    """Capture one smla_decode call in a CUDA graph and time `steps` replays
    with CUDA events on the launching stream, L2 flushed before each.  With
    `redraw`, every replay (warm-up included) first draws new live lengths for
    all rows (the graph was captured once, at the construction-time lengths).
    Returns (per-step ms, per-step algorithmic flops, per-step bytes)."""
    import torch
    import smla_inputs as I
    import sparse_mla_decode_04_gb300 as smla

    dev = p.q_nope.device
    R, H = p.num_rows, p.num_heads
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, H), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)  # attrs + first launch outside capture
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)
    ms, flops, nbytes = [], [], []
    for i in range(warmup + steps):
        if redraw:
            I.redraw_lengths(p, seed=7000 + i)
            torch.cuda.synchronize()
        f, b = p.algorithmic_flops(), p.algorithmic_bytes()
        with torch.cuda.stream(stream):
            flush_buf.fill_(i & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        stream.synchronize()
        if i >= warmup:
            ms.append(e0.elapsed_time(e1))
            flops.append(f)
            nbytes.append(b)
    del graph
    return ms, flops, nbytes


def per_config_lines(names, dev, flush_buf, stream, peaks, steps: int, warmup: int):
    """One entry per named workload: µs per call, rows/s and the roofline."""
    import gc
    import torch
    import sparse_mla_decode_04_gb300 as smla

    res = {}
    for name in names:
        p = make_workload(name, dev)
        R, H = p.num_rows, p.num_heads
        S = smla.smla_plan_num_splits(R, H, p.kv_len_estimate())
        ws = smla.Workspace(R, H, S, device=dev)
        ms, fl, nb = time_call(p, S, ws, steps, warmup, flush_buf, stream, redraw=(name == "ragged"))
        t = statistics.mean(ms) / 1e3
        rf = roofline(statistics.mean(fl), statistics.mean(nb), t, peaks)
        flags = ws.read_error()
        res[name] = {"workload": p.name, "us_per_call": t * 1e6, "rows_per_s": R / t, "rows": R, "heads": H,
                     "num_splits": S, "valid_entries": int(round(statistics.mean(fl) / (H * 2048))),
                     "roofline": rf, "device_error": flags,
                     "timing": ("one graph capture, replayed with re-drawn lengths before each step"
                                if name == "ragged" else "graph replay, L2 flushed") + f"; {steps} steps"}
        log(f"per_config {name}: {t * 1e6:.1f} us/call, frac {rf['frac']:.3f}")
        del p, ws
        gc.collect()
        torch.cuda.empty_cache()
    return res


def next_rows_lines(dev, flush_buf, stream, peaks, steps: int, warmup: int = 3, writer_rows: int = 4 << 20,
                    topk_rows: int = 64):
    """The two producers beside the decode, each timed alone (CUDA events on
    the launching stream, L2 flushed before each step), against the HBM
    roofline of their algorithmic bytes:
      cache_write: 4M latent rows (bf16 [4M, 512]) written to a random
        permutation of 4M cache slots; 1024 B read + 584 B written + 8 B slot
        per row;
      topk_indices: the decode's largest shape, 64 rows x 1M scores, k = 2048;
        4 B read per score + 4 B written per index."""
    import gc
    import torch
    import sparse_mla_decode_04_gb300 as smla

    res = {}

    def timed(fn):
        ms = []
        for i in range(warmup + steps):
            with torch.cuda.stream(stream):
                flush_buf.fill_(i & 0xFF)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            stream.synchronize()
            if i >= warmup:
                ms.append(e0.elapsed_time(e1))
        return statistics.mean(ms) / 1e3

    g = torch.Generator(device=dev)
    g.manual_seed(77)
    n = writer_rows
    lat = (torch.randn((n, 512), generator=g, device=dev)).to(torch.bfloat16)
    slots = torch.randperm(n, generator=g, device=dev)
    pool = torch.empty((n, 576), dtype=torch.uint8, device=dev)
    sc = torch.empty((n, 8), dtype=torch.uint8, device=dev)
    st = stream.cuda_stream
    t = timed(lambda: smla.cache_write(lat, slots, pool, sc, stream=st))
    nb = n * (1024 + 584 + 8)
    res["cache_write"] = {"rows": n, "us_per_call": t * 1e6, "GB_per_s": nb / t / 1e9,
                          "roofline": {"bound": "hbm", "achieved": nb / t / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                       "frac": nb / t / 1e9 / peaks["hbm_gbs"], "algorithmic_bytes": nb}}
    log(f"next cache_write: {t * 1e6:.1f} us, {nb / t / 1e9:.0f} GB/s")
    del lat, slots, pool, sc
    gc.collect()
    torch.cuda.empty_cache()
    R, L, k = topk_rows, 1 << 20, 2048
    scores = torch.randn((R, L), generator=g, device=dev)
    lens = torch.full((R,), L, dtype=torch.int32, device=dev)
    out = torch.empty((R, k), dtype=torch.int32, device=dev)
    t = timed(lambda: smla.topk_indices(scores, lens, k, out=out, stream=st))
    nb = R * L * 4 + R * k * 4 + R * 4
    res["topk_indices"] = {"rows": R, "positions": L, "k": k, "us_per_call": t * 1e6, "GB_per_s": nb / t / 1e9,
                           "roofline": {"bound": "hbm", "achieved": nb / t / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                        "frac": nb / t / 1e9 / peaks["hbm_gbs"], "algorithmic_bytes": nb}}
    log(f"next topk_indices: {t * 1e6:.1f} us, {nb / t / 1e9:.0f} GB/s")
    del scores, lens, out
    gc.collect()
    torch.cuda.empty_cache()
    return res


def run_gpu(args):
    import gc
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import sparse_mla_decode_04_gb300 as smla

    smla.build()
    if args.next_only:  # the two producers alone, one JSON object (not a bench line)
        if rank == 0:
            fb = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
            peaks, _ = load_peaks()
            res = next_rows_lines(dev, fb, torch.cuda.Stream(device=dev), peaks, args.config_steps,
                                  writer_rows=args.next_writer_rows, topk_rows=args.next_topk_rows)
            print(json.dumps({"next_rows": res}), flush=True)
        return 0
    p = make_workload(args.workload, dev)
    if rank > 0:  # replicas draw different data
        p.q_nope.copy_(torch.randn_like(p.q_nope, dtype=torch.float32).to(torch.bfloat16))
    R, H = p.num_rows, p.num_heads
    S = args.splits or smla.smla_plan_num_splits(R, H, p.kv_len_estimate())
    ws = smla.Workspace(R, H, S, device=dev)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((R, H), dtype=torch.float32, device=dev)
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    def reduce_max(x: float) -> float:
        return replica_max(x, device=dev)

    with torch.cuda.stream(stream):
        smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)  # attrs + first launch outside capture
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)
        for _ in range(args.warmup):
            flush_buf.fill_(1)
            graph.replay()
        stream.synchronize()
    barrier()
    events = []
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        torch.cuda.nvtx.range_push("timed")
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                flush_buf.fill_(2)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                events.append((e0, e1))
        barrier()
        torch.cuda.nvtx.range_pop()
        t_wall = time.perf_counter() - t_wall
    kernel_ms = [a.elapsed_time(b) for a, b in events]
    ms_step = reduce_max(statistics.mean(kernel_ms))
    flags = ws.read_error()
    if flags:
        raise SystemExit(f"device error word set during the bench: {flags:#x}")
    del graph

    # ---- end to end through the public API with host buffers ----
    host_in = {k: getattr(p, k).cpu().pin_memory() for k in
               ("q_nope", "q_rope", "main_idx", "swa_start", "swa_len", "cmp_start", "cmp_len")}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush_buf.fill_(3)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for k, t in host_in.items():
                getattr(p, k).copy_(t, non_blocking=True)
            smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)
            e1.record(stream)
            if i >= args.warmup:
                e2e_ms.append((e0, e1))
        stream.synchronize()
    e2e_step = reduce_max(statistics.mean(a.elapsed_time(b) for a, b in e2e_ms))
    barrier()

    peaks, peak_src = load_peaks()
    flops = p.algorithmic_flops()
    nbytes = p.algorithmic_bytes()
    t_s = ms_step / 1e3
    rf = roofline(flops, nbytes, t_s, peaks)
    traffic = profiled_traffic(args.workload)
    rows_total = R * world
    line = {
        "metric": METRIC, "value": replica_throughput(R, world, ms_step), "unit": "query-rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "us_per_call": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; FP8-e4m3 N(0,1) payload, UE8M0 codes 120..134, bf16 RoPE/q)",
        "config": workload_config(p, S, args.workload) | {"parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": rf | {"traffic": traffic, "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)"
                          if peak_src == "measured" else "fallback",
                          "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                          "kernel": f"{KERNEL_NAME} (timed with smla_merge_kernel: the whole call)"},
        "e2e": {"value": rows_total / (e2e_step / 1e3), "unit": "query-rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step},
        "gpu_launches": LAUNCHES_PER_CALL * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        per_row, n_rows, cores = cpu_oracle_time(p, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": 1.0 / per_row, "unit": "query-rows/s", "cores": cores, "kind": "oracle",
                                "sample": f"{n_rows} of {R} rows of the same workload, float64 NumPy oracle "
                                          f"(~{args.cpu_budget:.0f} s budget)"}
    del p, ws, out, lse, host_in
    gc.collect()
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_per_config:
        names = [n for n in PER_CONFIG if n != args.workload]
        line["per_config"] = per_config_lines(names, dev, flush_buf, stream, peaks, args.config_steps, 3)
        line["next_rows"] = next_rows_lines(dev, flush_buf, stream, peaks, args.config_steps,
                                            writer_rows=args.next_writer_rows, topk_rows=args.next_topk_rows)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--splits", type=int, default=0, help="override the planner's split count")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time only the main workload")
    ap.add_argument("--config-steps", type=int, default=10, help="timed steps per per_config workload")
    ap.add_argument("--next-only", action="store_true",
                    help="time only the cache writer and the top-k producer (for profiling them)")
    ap.add_argument("--next-writer-rows", type=int, default=4 << 20, help="latent rows of the cache-writer line")
    ap.add_argument("--next-topk-rows", type=int, default=64, help="score rows (1M each) of the top-k line")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
