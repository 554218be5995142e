"""Benchmark of the decode-step tail on GB300.

One step = one pass of the whole hot path over one batch: pkv_decode_tail,
i.e. pkv_sample_batch (temperature / top-k / top-p / inverse-CDF sampling
with the fused token write-back) and pkv_fill_page_table (page allocation +
page-table fill) in one call, the fill running beside the sampler's second
kernel.  Workload: the mixed batch B=256, V=151936, bf16 logits N(0, 3^2),
every 3rd row greedy, pages of 16 tokens.  Logits rotate over enough
buffers to exceed twice the L2 size, so every step reads them from HBM.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica of the batch on its own GPU (rows are independent; no collective on
the data path), the timed region is bracketed by a barrier and a device
synchronise, and the step time is the maximum over ranks.

--impl reference times the CPU oracle instead (the plain fp64 definition),
on this host's cores, on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sampled tokens/s and logits GB/s vs GB300 HBM peak at B=256, V=151936 bf16"
UNIT = "tokens/s"
WORKLOAD = "mixed"
KERNEL_SOURCES = ("paged_kv_gb300/csrc/sample_common.cuh", "paged_kv_gb300/csrc/sample_stream.cuh",
                  "paged_kv_gb300/csrc/sample_finish.cuh", "paged_kv_gb300/csrc/sample_launch.cuh",
                  "paged_kv_gb300/csrc/device_common.cuh", "paged_kv_gb300/csrc/launch_config.h",
                  "paged_kv_gb300/csrc/sample_params.h", "paged_kv_gb300/csrc/page_fill.cuh")
GRAPH_LEN = 20  # steps per captured CUDA graph (at most)
MIN_REPLAYS = 5  # graph replays per timed region (at least, when there are enough steps)
# The workloads of every configuration the method is measured on; the
# headline value is the mixed batch.
CONFIG_WORKLOADS = ("pr1", "greedy", "mixed", "nucleus", "large")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "sampler_mixed_traffic.json")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    return ap.parse_args(argv)


# ----------------------------------------------------------------- distributed harness


def dist_env():
    """(rank, world, local_rank) from the torchrun environment (defaults: 0, 1, 0)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init_dist(backend: str):
    import torch.distributed as dist

    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return dist if world > 1 else None


def barrier(dist_mod, device=None):
    if dist_mod is not None:
        if device is not None and device.type == "cuda":
            dist_mod.barrier(device_ids=[device.index])
        else:
            dist_mod.barrier()


def max_over_ranks(value: float, dist_mod, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity on one rank)."""
    if dist_mod is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64,
                     device=device if device is not None and device.type == "cuda" else "cpu")
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist_mod, device=None) -> float:
    if dist_mod is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64,
                     device=device if device is not None and device.type == "cuda" else "cpu")
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.SUM)
    return float(t.item())


def timed_steps(step, steps: int, warmup: int, dist_mod=None, device=None) -> float:
    """Runs `warmup` untimed steps, then times exactly `steps` steps; returns
    milliseconds (max over ranks).  On CUDA the region is timed with events on
    the current stream, bracketed by a barrier and a synchronise."""
    import torch

    cuda = device is not None and device.type == "cuda"
    for i in range(warmup):
        step(i)
    if cuda:
        torch.cuda.synchronize(device)
    barrier(dist_mod, device)
    if cuda:
        torch.cuda.synchronize(device)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record()
        for i in range(steps):
            step(i)
        end.record()
        torch.cuda.synchronize(device)
        ms = start.elapsed_time(end)
    else:
        t0 = time.perf_counter()
        for i in range(steps):
            step(i)
        ms = (time.perf_counter() - t0) * 1e3
    barrier(dist_mod, device)
    return max_over_ranks(ms, dist_mod, device)


def make_graph(fn, n: int, device):
    """Captures n calls fn(0..n-1) into one CUDA graph (after two warm calls
    on the capture stream, so that lazy allocations happen outside it)."""
    import torch

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        for i in range(2):
            fn(i)
    torch.cuda.current_stream(device).wait_stream(s)
    torch.cuda.synchronize(device)
    with torch.cuda.graph(g, stream=s):
        for i in range(n):
            fn(i)
    torch.cuda.synchronize(device)
    return g


def timed_graph_steps(fn, steps: int, warmup: int, dist_mod, device, spread=None) -> float:
    """Times exactly `steps` calls of fn, replayed from CUDA graphs (so that
    host launch cost does not enter): graphs of up to GRAPH_LEN calls, short
    enough that there are at least MIN_REPLAYS replays, plus one graph for
    the remainder; at least `warmup` untimed calls first.  Barriers,
    synchronisation and the max over ranks as in timed_steps.  Returns the
    milliseconds of the whole region; if `spread` is a dict it receives the
    per-replay microseconds per call (median, min, max, replays), from events
    recorded between the replays inside the same region."""
    import torch

    glen = max(1, min(GRAPH_LEN, steps // MIN_REPLAYS if steps >= MIN_REPLAYS else steps))
    full = make_graph(fn, glen, device)
    rem = steps % glen
    tail = make_graph(fn, rem, device) if rem else None
    for _ in range(max(1, -(-warmup // glen))):
        full.replay()
    torch.cuda.synchronize(device)
    barrier(dist_mod, device)
    torch.cuda.synchronize(device)
    n_full = steps // glen
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_full + 2)]
    ev[0].record()
    for i in range(n_full):
        full.replay()
        ev[i + 1].record()
    if tail is not None:
        tail.replay()
    ev[-1].record()
    torch.cuda.synchronize(device)
    ms = ev[0].elapsed_time(ev[-1])
    barrier(dist_mod, device)
    if spread is not None and n_full > 0:
        us = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 / glen for i in range(n_full))
        spread.update({"median_us": round(us[len(us) // 2], 3), "min_us": round(us[0], 3),
                       "max_us": round(us[-1], 3), "replays": n_full, "calls_per_replay": glen})
    return max_over_ranks(ms, dist_mod, device)


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
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
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        sms, maxes, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sms.sort()
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


# ----------------------------------------------------------------- helpers


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def physical_gpu_index(local_rank: int) -> int:
    """nvidia-smi index of this rank's GPU (CUDA_VISIBLE_DEVICES maps them)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    items = [v.strip() for v in vis.split(",") if v.strip()]
    if local_rank < len(items) and items[local_rank].isdigit():
        return int(items[local_rank])
    return local_rank


def _code_only(text: str) -> str:
    """The source with comments and blank space removed, so that an edit of
    comments alone keeps the hash (string literals in these sources hold no
    comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_hash() -> str:
    """Hash of the kernel sources' code (comments ignored)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per sampler launch from the committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


def algorithmic_bytes(w) -> int:
    """Bytes one sampler launch must move: one read of the logits plus the
    per-row parameters, tokens and write-back (T, k, p, u, row, col, token,
    pool write)."""
    return w.B * w.V * w.elt + w.B * (4 + 4 + 4 + 4 + 4 + 8 + 4 + 4)


# ----------------------------------------------------------------- our arm


def measure_config(name: str, device, dist_mod, peak: float, warmup: int, calls: int) -> dict:
    """One workload's pkv_sample_batch (fused write-back, no debug output),
    graph-replayed with the logits rotating over enough buffers to exceed
    twice the L2 size: median and range of the per-replay time per call,
    sampled tokens/s, logits GB/s and the fraction of the HBM peak."""
    import torch

    from paged_kv_gb300 import pkv, workloads

    w = workloads.make(name)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    logit_bytes = w.B * w.V * w.elt
    nbuf = min(600, max(4, -(-2 * l2 // logit_bytes) + 1))
    base = w.logits.to(device)
    bufs = [base] + [base.clone() for _ in range(nbuf - 1)]
    d = lambda x: None if x is None else x.to(device)  # noqa: E731
    t, k, p, u = d(w.temperature), d(w.top_k), d(w.top_p), d(w.uniform)
    pool = torch.zeros(w.pool_shape, dtype=torch.int32, device=device)
    rows, cols = d(w.wb_rows), d(w.wb_cols)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    out = torch.empty(w.B, dtype=torch.int32, device=device)
    spread = {}
    timed_graph_steps(lambda i: pkv.sample_batch(bufs[i % nbuf], t, k, p, u, out_tokens=out,
                                                 token_pool=pool, wb_rows=rows, wb_cols=cols,
                                                 status=status),
                      calls, warmup, dist_mod, device, spread)
    torch.cuda.synchronize(device)
    us = spread["median_us"]
    gbs = logit_bytes / (us * 1e-6) / 1e9
    res = {"B": w.B, "V": w.V, "dtype": "bf16" if w.elt == 2 else "fp32", "us": us,
           "min_us": spread["min_us"], "max_us": spread["max_us"],
           "replays": spread["replays"], "calls_per_replay": spread["calls_per_replay"],
           "tokens_per_s": round(w.B / (us * 1e-6), 1), "logits_gbs": round(gbs, 1),
           "frac": round(gbs / peak, 4), "status": int(status.item()), "buffers": nbuf}
    del bufs, base
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch

    from paged_kv_gb300 import pkv, workloads

    rank, world, local_rank = dist_env()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist_mod = init_dist("nccl")

    w = workloads.make(WORKLOAD)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    logit_bytes = w.B * w.V * w.elt
    nbuf = max(4, -(-2 * l2 // logit_bytes) + 1)
    base = w.logits.to(device)
    bufs = [base] + [base.clone() for _ in range(nbuf - 1)]
    d = lambda x: None if x is None else x.to(device)  # noqa: E731
    t, k, p, u = d(w.temperature), d(w.top_k), d(w.top_p), d(w.uniform)
    rows, cols = d(w.wb_rows), d(w.wb_cols)
    pool = torch.zeros(w.pool_shape, dtype=torch.int32, device=device)
    cached, dev_len, tidx = d(w.cached_len), d(w.device_len), d(w.table_idx)
    free = d(w.free_slots)
    pt = torch.zeros(w.pt_shape, dtype=torch.int32, device=device)
    total = torch.zeros(1, dtype=torch.int64, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    out = torch.empty(w.B, dtype=torch.int32, device=device)

    def step(i):
        pkv.decode_tail(bufs[i % nbuf], t, k, p, u, out, pool, rows, cols, cached, dev_len, tidx,
                        w.page_size, free, pt, total, status)

    step_spread = {}
    with ClockSampler(physical_gpu_index(local_rank)) as clocks:
        ms = timed_graph_steps(step, args.steps, args.warmup, dist_mod, device, step_spread)
    torch.cuda.synchronize(device)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status word {int(status.item())} after the timed run")
    ms_per_step = ms / args.steps
    value = world * w.B / (ms_per_step * 1e-3)

    # Every configuration: one pkv_sample_batch per call (with the fused
    # write-back), graph-replayed, median and spread over the replays.  The
    # mixed batch's entry is the dominant operation of the step and gives
    # the roofline.
    peak, peak_kind = measured_peaks()
    n_k = max(MIN_REPLAYS * GRAPH_LEN, min(args.steps, 2000))
    configs = {name: measure_config(name, device, dist_mod, peak, args.warmup, n_k)
               for name in CONFIG_WORKLOADS}
    us_k = configs[WORKLOAD]["us"]
    alg = algorithmic_bytes(w)
    achieved = alg / (us_k * 1e-6) / 1e9
    # The same batch with min_p = 0.05 on every row (sampled rows then take
    # the exact path).
    minp = torch.full((w.B,), 0.05, dtype=torch.float32, device=device)
    ms_m = timed_graph_steps(lambda i: pkv.sample_batch(bufs[i % nbuf], t, k, p, u,
                                                        out_tokens=out, status=status,
                                                        min_p=minp),
                             max(50, n_k // 4), args.warmup, dist_mod, device)
    us_m = ms_m / max(50, n_k // 4) * 1e3
    # The step before the model on the same batch (pages, positions and the
    # input_ids / out_loc gathers of every token in [cached_len, device_len)).
    n_tok = int((w.device_len - w.cached_len).clamp(min=0).sum())
    prep_pool = torch.zeros(w.pool_shape, dtype=torch.int32, device=device)
    prep_out = [torch.empty(n_tok, dtype=torch.int32, device=device) for _ in range(3)]
    prep_tot = [torch.zeros(1, dtype=torch.int64, device=device) for _ in range(2)]
    ms_p = timed_graph_steps(lambda i: pkv.prepare_step(cached, dev_len, tidx, w.page_size, free,
                                                        pt, prep_pool, n_tok, *prep_out,
                                                        *prep_tot, status),
                             n_k, args.warmup, dist_mod, device)
    prep_bytes = n_tok * (3 * 4 + 4 + 4) + 12 * w.B
    ms_f = timed_graph_steps(lambda i: pkv.fill_page_table(cached, dev_len, tidx, w.page_size,
                                                           free, pt, total, status),
                             n_k, args.warmup, dist_mod, device)

    # End to end through the public API from pinned host buffers: every step
    # copies its inputs host -> device, makes the call and copies the tokens
    # and the page total back.  As a serving loop would, the inputs of step
    # i + 1 are copied on a second stream (into the other of two device
    # buffers) while step i computes; each timed step still issues exactly
    # one step's host -> device copy and one device -> host read.
    host = {name: getattr(w, name) for name in ("temperature", "top_k", "top_p", "uniform",
                                                "wb_rows", "wb_cols", "cached_len",
                                                "device_len", "table_idx")}
    h_logits = w.logits.pin_memory()
    h_in = {n: v.pin_memory() for n, v in host.items()}
    h_tok = torch.empty(w.B, dtype=torch.int32).pin_memory()
    h_total = torch.empty(1, dtype=torch.int64).pin_memory()
    d_in = [{n: torch.empty_like(v, device=device) for n, v in host.items()} for _ in range(2)]
    d_logits = [torch.empty_like(base) for _ in range(2)]
    h2d = h_logits.numel() * h_logits.element_size() + sum(
        v.numel() * v.element_size() for v in h_in.values())
    d2h = h_tok.numel() * 4 + 8
    copy_stream = torch.cuda.Stream(device)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def issue_copy(j):
        slot = j % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[slot])  # the slot's previous step is done with it
            d_logits[slot].copy_(h_logits, non_blocking=True)
            for n in d_in[slot]:
                d_in[slot][n].copy_(h_in[n], non_blocking=True)
            copied[slot].record(copy_stream)

    issue_copy(0)

    def e2e_step(i):
        slot = i % 2
        issue_copy(i + 1)
        cur = torch.cuda.current_stream(device)
        cur.wait_event(copied[slot])
        d = d_in[slot]
        pkv.decode_tail(d_logits[slot], d["temperature"], d["top_k"], d["top_p"], d["uniform"],
                        out, pool, d["wb_rows"], d["wb_cols"], d["cached_len"], d["device_len"],
                        d["table_idx"], w.page_size, free, pt, total, status)
        consumed[slot].record(cur)
        h_tok.copy_(out, non_blocking=True)
        h_total.copy_(total, non_blocking=True)
        if i == args.e2e_steps - 1:
            cur.wait_stream(copy_stream)  # every copy issued in the timed region ends in it

    ms_e2e = timed_steps(e2e_step, args.e2e_steps, 3, dist_mod, device)
    e2e_value = world * w.B / (ms_e2e / args.e2e_steps * 1e-3)

    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_baseline(w, budget_s=12.0)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "mixed decode batch: B=256, V=151936 bf16 logits N(0,3^2), "
                                   "1/3 greedy, T~U[0.5,1.5], top_k in {off,20,50}, "
                                   "top_p in {1,0.9,0.95}; pages of 16",
                       "B": w.B, "V": w.V, "page_size": w.page_size,
                       "parallelism": f"replicas x{world}",
                       "l2": f"logits rotate over {nbuf} buffers ({nbuf * logit_bytes >> 20} MiB > 2x L2)"},
            "logits_gbs": round(world * logit_bytes / (ms_per_step * 1e-3) / 1e9, 1),
            "step_spread": step_spread,
            "configs": configs,
            "page_fill_us": round(ms_f / n_k * 1e3, 3),
            "minp_us": round(us_m, 3),
            "prepare_step": {"us": round(ms_p / n_k * 1e3, 3), "tokens": n_tok,
                             "gbs": round(prep_bytes / (ms_p / n_k * 1e-3) / 1e9, 1)},
            "roofline": {"bound": "hbm", "kernel": "pkv_sample_batch (stream_kernel + finish_kernel)",
                         "achieved": round(achieved, 1),
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": recorded_traffic(),
                         "algorithmic_bytes": alg, "us_per_launch": round(us_k, 3),
                         "us_per_launch_spread": [configs[WORKLOAD]["min_us"],
                                                  configs[WORKLOAD]["max_us"]],
                         "timing": "median over graph replays of the mixed batch's "
                                   "pkv_sample_batch, logits rotating past L2"},
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                    "pipelined": "step i+1's inputs copied on a second stream during step i"},
            "gpu_launches": 2 * args.steps,  # per step: stream_kernel and finish_kernel
            "timing": f"device value and roofline: CUDA graphs of {GRAPH_LEN} steps replayed; "
                      "e2e: host-launched calls",
            "clocks": clocks.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist_mod is not None:
        dist_mod.destroy_process_group()


# ----------------------------------------------------------------- oracle arm


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_baseline(w, budget_s: float = 12.0, rows: int = 64) -> dict:
    """The oracle as it stands, on this host's cores, on a bounded sample:
    the first `rows` rows of the batch (sampling) plus the whole page fill,
    repeated until about `budget_s` seconds have passed."""
    import numpy as np

    import oracle

    cores = host_cores()
    sub = slice(0, rows)
    s = lambda x: None if x is None else x[sub]  # noqa: E731
    logits = w.logits[sub].contiguous()
    args = (s(w.temperature), s(w.top_k), s(w.top_p), s(w.uniform))
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.sample(logits, *args, threads=cores)
        pt = np.zeros(w.pt_shape, np.int32)
        oracle.fill_page_table(w.cached_len, w.device_len, w.table_idx, w.page_size,
                               w.free_slots, pt)
        done += rows
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    # The same sample on one thread (a shorter run: 16 rows per pass).
    one_rows, one_done, t1 = 16, 0, time.perf_counter()
    one_logits = w.logits[:one_rows].contiguous()
    one_args = tuple(None if x is None else x[:one_rows] for x in (w.temperature, w.top_k,
                                                                   w.top_p, w.uniform))
    while True:
        oracle.sample(one_logits, *one_args, threads=1)
        pt = np.zeros(w.pt_shape, np.int32)
        oracle.fill_page_table(w.cached_len, w.device_len, w.table_idx, w.page_size,
                               w.free_slots, pt)
        one_done += one_rows
        if time.perf_counter() - t1 >= budget_s / 4:
            break
    dt1 = time.perf_counter() - t1
    return {"value": round(done / dt, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "value_1_thread": round(one_done / dt1, 2),
            "sample": f"{done} rows of the mixed batch ({rows} per pass, with the full page fill) "
                      f"in {dt:.1f} s, fp64, {cores} threads; one thread: {one_done} rows in "
                      f"{dt1:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from paged_kv_gb300 import workloads

    w = workloads.make(WORKLOAD)
    cores = host_cores()
    import numpy as np

    import oracle

    rows = 16
    sub = slice(0, rows)
    s = lambda x: None if x is None else x[sub]  # noqa: E731
    logits = w.logits[sub].contiguous()
    params = (s(w.temperature), s(w.top_k), s(w.top_p), s(w.uniform))

    def step(i):
        oracle.sample(logits, *params, threads=cores)
        pt = np.zeros(w.pt_shape, np.int32)
        oracle.fill_page_table(w.cached_len, w.device_len, w.table_idx, w.page_size,
                               w.free_slots, pt)

    steps = min(args.steps, 20)
    warm = min(args.warmup, 3)
    ms = timed_steps(step, steps, warm)
    value = rows / (ms / steps * 1e-3)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": steps, "warmup": warm, "ms_per_step": round(ms / steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "mixed decode batch: B=256, V=151936 bf16 (oracle on a "
                               f"{rows}-row sample per step)", "B": w.B, "V": w.V,
                   "page_size": w.page_size},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{rows} rows of the mixed batch per step plus the full page "
                                   f"fill, {steps} steps"},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
