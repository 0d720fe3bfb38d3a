"""Benchmark of the DSA lightning-indexer hot path (index logits + masked top-k).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline]

One step = one call of the composed entry point dsa_indexer_topk (or
dsa_indexer_topk_paged) over one batch of synthetic input resident in HBM:
the tcgen05 scoring kernel writes the fp32 logits of every in-range key tile
into the call's workspace, then the radix-select kernel takes the per-row
top-k.  The default workload is the long single-sequence causal prefill with
e4m3 keys and queries: T=S=32768, H=64, D=128, index_topk=2048, per-row UE8M0
scales, fp32 weights -- the largest configuration of the path that runs on
one GPU.  L2 is flushed (a 256 MiB write) before every timed step, outside
the step's own event pair.

A second timed pass runs the two stages as separate calls with an event
between them: the scoring kernel's duration there gives the roofline line,
the top-k's its share.  Both passes check, before timing, that the composed
call and the separate calls give the same indices bit for bit.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the path has no exchange step): the K steps are bracketed by a
barrier + synchronize, the per-step time is the max over ranks, and `value`
is the rows all ranks processed divided by that time.

--impl reference times the CPU oracle (the only other implementation of this
path) on the host cores, on a bounded row sample of the same workload.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("indexer+top-k query rows/sec and TFLOP/s (prefill), GB/s (decode) "
          "vs GB300 roofline")
L2_FLUSH_BYTES = 256 << 20
# The committed ncu summary that gives the scoring kernel's DRAM traffic per
# launch, and the sources it was taken on, per workload.
PROFILES = {
    "prefill_fp8": ("score_prefill_fp8_T32768_H64_D128.md",
                    ("top_selection_dsa_gb300/csrc/dsa_score.cuh",
                     "top_selection_dsa_gb300/csrc/dsa_common.cuh",
                     "top_selection_dsa_gb300/csrc/dsa_score_prefill_fp8.cu")),
    "prefill_causal": ("score_prefill_bf16_T4096_H64_D128.md",
                       ("top_selection_dsa_gb300/csrc/dsa_score.cuh",
                        "top_selection_dsa_gb300/csrc/dsa_common.cuh",
                        "top_selection_dsa_gb300/csrc/dsa_score_prefill_bf16.cu")),
    "prefill_mxfp4": ("score_prefill_mxfp4_T32768_H64_D128.md",
                      ("top_selection_dsa_gb300/csrc/dsa_score_mx.cuh",
                       "top_selection_dsa_gb300/csrc/dsa_score.cuh",
                       "top_selection_dsa_gb300/csrc/dsa_common.cuh",
                       "top_selection_dsa_gb300/csrc/dsa_score_prefill_mxfp4.cu")),
}
# Rows of the CPU oracle sample for cpu_baseline (about 10-30 s of the host's
# cores); the reference arm times an eighth of it per step.
ORACLE_ROWS = {"prefill_fp8": 2048, "prefill_causal": 4096, "prefill_thd": 4096,
               "paged_decode": 128, "tiny_causal": 256, "prefill_mxfp4": 2048}
# Dense tensor peak per element type, as a multiple of the measured bf16 one
# (the nominal ratios: e4m3 2x, E2M1 with block scales 6x).
PEAK_RATIO = {0: 1.0, 1: 2.0, 2: 6.0}
DTYPE_NAME = {0: "bf16", 1: "e4m3", 2: "mxfp4 (e2m1 + e8m0 per 32)"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="prefill_fp8",
                    choices=("prefill_causal", "prefill_thd", "prefill_fp8", "paged_decode",
                             "tiny_causal", "prefill_mxfp4"))
    ap.add_argument("--prologue", action="store_true",
                    help="time the steps before the indexer (query quantisation + weight "
                         "fold, key LayerNorm + e4m3 paged insert) at the e4m3 workload's "
                         "sizes instead of the hot path; one JSON line per step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true",
                    help="skip the clock-sampling load window (for profiler runs)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T = S of the prefill workloads (smaller profiler captures)")
    ap.add_argument("--oracle-rows", type=int, default=0,
                    help="rows of the CPU oracle sample for cpu_baseline (default per "
                         "workload, 10-30 s of the host's cores; the reference arm times an "
                         "eighth of it per step)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def launches_per_step(p):
    """This library's kernel launches in one step: the scoring kernel, then one
    top-k kernel, or three (histogram, gather, write) when the top-k takes its
    split path -- at most 512 rows, some row longer than 16384 columns and
    none longer than 1048576 (the rule of topk_split_rows in dsa_topk.cu)."""
    rows = p.T if hasattr(p, "row_starts") else p.R
    cols = p.S if hasattr(p, "row_starts") else p.max_ctx()
    split = rows <= 512 and 16384 < cols <= 256 * 4096
    return 1 + (3 if split else 1)


def kernel_sha(sources):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """(dram read+write bytes per launch of the scoring kernel, summary file)
    from the committed ncu summary of this workload, or (None, why) when
    there is none or it was taken on other kernel sources."""
    if workload not in PROFILES:
        return None, "no committed summary for this workload"
    name, sources = PROFILES[workload]
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None, f"profiles/{name} missing"
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    s = re.search(r"kernel_sources_sha:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_sha(sources):
        return None, f"profiles/{name} taken on other kernel sources"
    return int(m.group(1)), f"profiles/{name}"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(values, world, device):
    """Element-wise max over ranks of a list of floats."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def make_workload(name, tokens=0):
    from top_selection_dsa_gb300 import workloads as wl
    if tokens and name in ("prefill_causal", "prefill_fp8", "prefill_mxfp4"):
        return wl.WORKLOADS[name](T=tokens)
    return wl.WORKLOADS[name]()


def step_flops(p):
    return 2.0 * p.valid_pairs() * p.H * p.D


# ------------------------------------------------------- CPU oracle timing

def oracle_sample_rate(p, nrows, seed=0):
    """Time the CPU oracle (logits + top-k) on a seeded row sample: rows/s."""
    import oracle
    rng = np.random.default_rng(seed)
    if hasattr(p, "row_starts"):
        rows = np.sort(rng.choice(p.T, size=min(nrows, p.T), replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        if p.dtype == 2:
            lg = oracle.logits_mxfp4(p.q, p.q_sf, p.k, p.k_sf, p.w, p.row_starts, p.row_ends,
                                     rows=rows)
        else:
            lg = oracle.logits(p.q, p.k, p.w, p.row_starts, p.row_ends, dtype=p.dtype,
                               k_scale=p.k_scale, rows=rows)
        oracle.topk(lg.astype(np.float32), p.row_starts[rows], p.row_ends[rows], p.topk,
                    S=p.S)
        dt = time.perf_counter() - t0
        sample = f"{len(rows)} of {p.T} rows, uniform without replacement (seed {seed})"
    else:
        rows = np.sort(rng.choice(p.R, size=min(nrows, p.R), replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        lg = oracle.logits_paged(p.q, p.w, p.k_cache, p.block_table, p.context_lens,
                                 next_n=p.next_n, dtype=p.dtype, k_scale=p.k_scale,
                                 ld=p.max_ctx(), rows=rows)
        rs, re_ = oracle.paged_row_ranges(p.context_lens, p.next_n)
        oracle.topk(lg.astype(np.float32), rs[rows], re_[rows], p.topk)
        dt = time.perf_counter() - t0
        sample = f"{len(rows)} of {p.R} query rows, uniform (seed {seed})"
    return len(rows) / dt, dt, sample, oracle.max_threads()


def oracle_rows(args):
    return args.oracle_rows or ORACLE_ROWS.get(args.workload, 1024)


def workload_config(p, world):
    """The `config` object both arms print for a workload."""
    paged = not hasattr(p, "row_starts")
    rows = p.R if paged else p.T
    return {"workload": p.name, "rows_per_step": rows, "valid_pairs": p.valid_pairs(),
            "index_topk": p.topk, "H": p.H, "D": p.D,
            "elements": {0: "bf16", 1: "e4m3 + UE8M0 per-row scales",
                         2: "MXFP4: E2M1 + E8M0 per 32 elements"}[p.dtype],
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    p = make_workload(args.workload, args.tokens)
    rows = max(8, oracle_rows(args) // 8)
    for _ in range(args.warmup):
        oracle_sample_rate(p, rows, seed=1)
    times, rates = [], []
    sample = cores = None
    for i in range(args.steps):
        rate, dt, sample, cores = oracle_sample_rate(p, rows, seed=2 + i)
        times.append(dt)
        rates.append(rate)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * float(np.mean(times)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(p, 1),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {sample}"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- our path

def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from top_selection_dsa_gb300 import api

    p = make_workload(args.workload, args.tokens)
    paged = not hasattr(p, "row_starts")
    cuda = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731

    def elems(x):
        if p.dtype == 0:
            return cuda(x.view(np.int16)).view(torch.bfloat16)
        return cuda(x).view(torch.float8_e4m3fn)

    stream = torch.cuda.current_stream(device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    mx = (not paged) and p.dtype == 2
    if mx:
        q, qsf, k, ksf, w = cuda(p.q), cuda(p.q_sf), cuda(p.k), cuda(p.k_sf), cuda(p.w)
        rs, re_ = cuda(p.row_starts), cuda(p.row_ends)
        rows_per_step = p.T
        ld = (p.S + 3) // 4 * 4
        ws = torch.empty(api.workspace_bytes(api.DSA_OP_INDEXER_TOPK, p.T, p.S, p.topk),
                         dtype=torch.uint8, device=device)
        lg_bytes = (p.T * ld * 4 + 255) // 256 * 256
        logits = ws[:p.T * ld * 4].view(torch.float32).view(p.T, ld)
        ws_topk = ws[lg_bytes:]
        out = torch.empty((p.T, p.topk), dtype=torch.int32, device=device)

        def score():
            api.indexer_logits_mxfp4(q, qsf, k, ksf, w, rs, re_, logits=logits)

        def select():
            api.topk(logits, rs, re_, p.topk, S=p.S, out=out, workspace=ws_topk)

        def fused(o):
            return api.indexer_topk_mxfp4(q, qsf, k, ksf, w, rs, re_, p.topk, out=o,
                                          workspace=ws)
    elif not paged:
        q, k, w = elems(p.q), elems(p.k), cuda(p.w)
        rs, re_ = cuda(p.row_starts), cuda(p.row_ends)
        ks = cuda(p.k_scale) if p.k_scale is not None else None
        rows_per_step = p.T
        ld = (p.S + 3) // 4 * 4
        # One workspace as the composed call lays it out: logits, then (few
        # long rows only) the split top-k scratch.  The separate calls of the
        # breakdown pass use the same regions.
        ws = torch.empty(api.workspace_bytes(api.DSA_OP_INDEXER_TOPK, p.T, p.S, p.topk),
                         dtype=torch.uint8, device=device)
        lg_bytes = (p.T * ld * 4 + 255) // 256 * 256
        logits = ws[:p.T * ld * 4].view(torch.float32).view(p.T, ld)
        ws_topk = ws[lg_bytes:]
        out = torch.empty((p.T, p.topk), dtype=torch.int32, device=device)

        def score():
            api.indexer_logits(q, k, w, rs, re_, k_scale=ks, logits=logits)

        def select():
            api.topk(logits, rs, re_, p.topk, S=p.S, out=out, workspace=ws_topk)

        def fused(o):
            return api.indexer_topk(q, k, w, rs, re_, p.topk, k_scale=ks, out=o, workspace=ws)
    else:
        q, w, kc = elems(p.q), cuda(p.w), elems(p.k_cache)
        bt, cl = cuda(p.block_table), cuda(p.context_lens)
        ks = cuda(p.k_scale.reshape(-1)) if p.k_scale is not None else None
        rows_per_step = p.R
        ld = p.max_ctx()
        ws = torch.empty(api.workspace_bytes(api.DSA_OP_INDEXER_TOPK_PAGED, p.R, ld, p.topk),
                         dtype=torch.uint8, device=device)
        lg_bytes = (p.R * ld * 4 + 255) // 256 * 256
        logits = ws[:p.R * ld * 4].view(torch.float32).view(p.R, ld)
        ws_topk = ws[lg_bytes:]
        out = torch.empty((p.R, p.topk), dtype=torch.int32, device=device)
        rs_np, re_np = (np.zeros(p.R, np.int32),
                        np.array([max(int(p.context_lens[r // p.next_n]) - p.next_n
                                      + r % p.next_n + 1, 0) for r in range(p.R)], np.int32))
        rs, re_ = cuda(rs_np), cuda(re_np)

        def score():
            api.indexer_logits_paged(q, w, kc, bt, cl, next_n=p.next_n, k_scale=ks,
                                     logits=logits)

        def select():
            api.topk(logits, rs, re_, p.topk, out=out, workspace=ws_topk)

        def fused(o):
            return api.indexer_topk_paged(q, w, kc, bt, cl, p.topk, next_n=p.next_n,
                                          k_scale=ks, out=o, workspace=ws)

    # The composed call is the same two kernels: check bit-identity once.
    score()
    select()
    ref_out = out.clone()
    fused_out = torch.empty_like(out)
    fused(fused_out)
    torch.cuda.synchronize(device)
    if not torch.equal(fused_out, ref_out):
        raise RuntimeError("composed entry point differs from logits + top-k")
    if api.last_device_error() != api.DSA_OK:
        raise RuntimeError("device error word set during warm-up")

    def composed_step():
        fused(fused_out)

    def split_step():
        score()
        select()

    for _ in range(args.warmup):
        flush.zero_()
        composed_step()
        flush.zero_()
        split_step()
    torch.cuda.synchronize(device)

    # Timed pass 1 (the step): K composed calls, one event pair each.
    # Timed pass 2 (the breakdown): K steps of the two separate calls with an
    # event between them.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clocks:
        # nvidia-smi samples every 100 ms while a timed pass may last only a
        # few ms: keep the same load running for ~1 s right before it, so the
        # samples describe the clocks the steps run at.
        t_end = time.perf_counter() + (0.0 if args.no_clocks else 1.0)
        while time.perf_counter() < t_end:
            for _ in range(4):
                flush.zero_()
                composed_step()
            torch.cuda.synchronize(device)
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            composed_step()
            ev[i][1].record(stream)
        torch.cuda.synchronize(device)
        wall = time.perf_counter() - wall0
        for i in range(args.steps):
            flush.zero_()
            ev2[i][0].record(stream)
            score()
            ev2[i][1].record(stream)
            select()
            ev2[i][2].record(stream)
        torch.cuda.synchronize(device)
    barrier(world)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    score_ms = [e[0].elapsed_time(e[1]) for e in ev2]
    topk_ms = [e[1].elapsed_time(e[2]) for e in ev2]
    split_ms = [e[0].elapsed_time(e[2]) for e in ev2]
    if api.last_device_error() != api.DSA_OK:
        raise RuntimeError("device error word set during the timed steps")
    if not torch.equal(fused_out, ref_out):
        raise RuntimeError("timed composed calls changed their result")
    ms, s_ms, t_ms, sp_ms = reduce_max([statistics.mean(step_ms), statistics.mean(score_ms),
                                        statistics.mean(topk_ms), statistics.mean(split_ms)],
                                       world, device)

    # End to end through the C ABI from pinned host buffers, every step.
    # Prefill: dsa_indexer_topk_host takes the host pointers and overlaps the
    # uploads, the kernels and the download of the indices over row chunks.
    # Paged decode: the step's inputs are copied up, the fused call runs, the
    # indices are copied down (the K cache stays resident: it is the serving
    # system's state, not an input).
    e2e = None
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        host_out = torch.empty(out.shape, dtype=torch.int32).pin_memory()
        if mx:
            host_in = [pin(a) for a in (p.q, p.q_sf, p.k, p.k_sf, p.w, p.row_starts, p.row_ends)]
            dev_in = [q, qsf, k, ksf, w, rs, re_]

            def e2e_step():
                for d, h in zip(dev_in, host_in):
                    d.view(-1).copy_(h.view(-1), non_blocking=True)
                fused(out)
                host_out.copy_(out, non_blocking=True)
        elif not paged:
            if p.dtype == 0:
                hq, hk = pin(p.q.view(np.int16)).view(torch.bfloat16), \
                    pin(p.k.view(np.int16)).view(torch.bfloat16)
            else:
                hq, hk = pin(p.q).view(torch.float8_e4m3fn), pin(p.k).view(torch.float8_e4m3fn)
            hw, hrs, hre = pin(p.w), pin(p.row_starts), pin(p.row_ends)
            hks = pin(p.k_scale) if p.k_scale is not None else None
            host_in = [t for t in (hq, hk, hw, hrs, hre, hks) if t is not None]
            # The resident-input workspace is not needed any more: the host
            # pipeline takes its own device buffer.
            del ws, logits, ws_topk
            hbuf = torch.empty(api.indexer_topk_host_bytes(p.T, p.S, q.shape[1], q.shape[2],
                                                           p.topk, p.dtype),
                               dtype=torch.uint8, device=device)

            def e2e_step():
                api.indexer_topk_host(hq, hk, hw, hrs, hre, p.topk, k_scale=hks, out=host_out,
                                      device_buffer=hbuf, device=device)
        else:
            host_in = [pin(a) for a in
                       (p.q.view(np.uint8), p.w, p.block_table, p.context_lens)]
            dev_in = [q.view(torch.uint8), w, bt, cl]
            if ks is not None:
                host_in.append(pin(p.k_scale.reshape(-1)))
                dev_in.append(ks)

            def e2e_step():
                for d, h in zip(dev_in, host_in):
                    d.view(-1).copy_(h.view(-1), non_blocking=True)
                fused(out)
                host_out.copy_(out, non_blocking=True)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = host_out.numel() * 4
        e2e_ms = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step()
            b.record(stream)
            b.synchronize()
            if i >= args.warmup:
                e2e_ms.append(a.elapsed_time(b))
        if not torch.equal(host_out, ref_out.cpu()):
            raise RuntimeError("end-to-end result differs from the resident-input result")
        # The copies alone, one direction at a time, on the same stream: the
        # floor an overlapped pipeline approaches is the larger of the two.
        up_dst = torch.empty(h2d, dtype=torch.uint8, device=device)
        h2d_ms, d2h_ms = [], []
        for i in range(args.warmup + args.steps):
            evc = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            evc[0].record(stream)
            off = 0
            for h in host_in:
                n = h.numel() * h.element_size()
                up_dst[off:off + n].copy_(h.view(-1).view(torch.uint8), non_blocking=True)
                off += n
            evc[1].record(stream)
            host_out.copy_(out, non_blocking=True)
            evc[2].record(stream)
            evc[2].synchronize()
            if i >= args.warmup:
                h2d_ms.append(evc[0].elapsed_time(evc[1]))
                d2h_ms.append(evc[1].elapsed_time(evc[2]))
        del up_dst
        em, hm, dm = reduce_max([statistics.mean(e2e_ms), statistics.mean(h2d_ms),
                                 statistics.mean(d2h_ms)], world, device)
        e2e = {"value": world * rows_per_step / (em / 1e3), "unit": "rows/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": em,
               "entry_point": ("copies + dsa_indexer_topk_mxfp4 + copy" if mx else
                               "dsa_indexer_topk_host" if not paged else
                               "copies + dsa_indexer_topk_paged + copy"),
               "copies_alone_ms": {"h2d": hm, "d2h": dm,
                                   "h2d_gbs": h2d / hm / 1e6, "d2h_gbs": d2h / dm / 1e6}}

    if rank != 0:
        return 0

    peaks, peak_src = measured_peaks()
    flops = step_flops(p)
    if not paged:
        ratio = PEAK_RATIO[p.dtype]
        peak = peaks["bf16_tflops"] * ratio
        achieved = flops / (s_ms / 1e3) / 1e12
        traffic, traffic_src = profiled_traffic(args.workload if not args.tokens else "")
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "traffic_source": traffic_src,
                "kernel": ("score_mx_kernel (tcgen05 kind::mxf4 block-scaled scoring)" if mx else
                           "score_kernel (tcgen05 scoring, writes fp32 logits)"),
                "algorithmic_flops_per_launch": flops,
                "duration_ms": s_ms,
                "peak_source": f"{peak_src} bf16 burst" + (
                    f" x{ratio:g} (the nominal {DTYPE_NAME[p.dtype]}:bf16 dense ratio)"
                    if ratio != 1.0 else "")}
    else:
        kbytes = int(sum(int(L) for L in p.context_lens)) * p.D * (2 if p.dtype == 0 else 1)
        other = p.R * p.H * p.D * (2 if p.dtype == 0 else 1) + p.R * p.H * 4 \
            + int(sum(-(-int(L) // p.block_size) for L in p.context_lens)) * 4 \
            + p.valid_pairs() * 4
        alg = kbytes + other
        achieved = alg / (s_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": None,
                "kernel": "score_kernel (paged, writes fp32 logits)",
                "algorithmic_bytes_per_launch": alg, "duration_ms": s_ms,
                "peak_source": f"{peak_src} hbm copy"}
    # top-k pass: reads each valid logit once, writes the indices.
    topk_bytes = p.valid_pairs() * 4 + rows_per_step * p.topk * 4
    launches = launches_per_step(p)
    cfg = workload_config(p, world)
    cfg.update({"step": ("one dsa_indexer_topk_mxfp4 call" if mx else
                         "one dsa_indexer_topk call" if not paged
                         else "one dsa_indexer_topk_paged call"),
                "l2": "flushed before every step (256 MiB write, outside the step events)",
                "clock_window": "nvidia-smi every 100 ms over a 1 s window of the same "
                                "steps right before the timed ones, and over both timed "
                                "passes"})
    line = {
        "metric": METRIC,
        "value": world * rows_per_step / (ms / 1e3),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {0: "bf16", 1: "e4m3", 2: "mxfp4"}[p.dtype],
        "data": "synthetic",
        "config": cfg,
        "tflops": flops / (ms / 1e3) / 1e12,
        "kernels": {"pass": "separate calls, an event between the stages, L2 flushed",
                    "score_ms": s_ms, "topk_ms": t_ms, "score_plus_topk_ms": sp_ms,
                    "topk_gbs": topk_bytes / (t_ms / 1e3) / 1e9,
                    "topk_hbm_frac": topk_bytes / (t_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                    "topk_algorithmic_bytes": topk_bytes},
        "roofline": roof,
        "gpu_launches": launches * args.steps,
        "gpu_launches_note": f"{launches} per composed call in the timed step pass; the "
                             f"breakdown pass launches the same kernels again",
        "wall_s_timed_region": wall,
    }
    if e2e is not None:
        line["e2e"] = e2e
    cs = clocks.summary()
    line["clocks"] = cs
    if not args.no_cpu_baseline and world == 1:
        rate, dt, sample, cores = oracle_sample_rate(p, oracle_rows(args))
        line["cpu_baseline"] = {"value": rate, "unit": "rows/s", "cores": cores,
                                "kind": "oracle", "sample": sample, "seconds": dt}
    print(json.dumps(line), flush=True)
    return 0


def run_prologue(args):
    """The two steps before the indexer, each timed alone with CUDA events on
    inputs in HBM (L2 flushed before every step), against the measured HBM
    copy bandwidth: bytes = every input read once + every output written."""
    import torch
    from top_selection_dsa_gb300 import api
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    T, H, D = (args.tokens or 32768), 64, 128
    g = torch.Generator(device=device)
    g.manual_seed(0)
    q = (torch.randn((T, H, D), device=device, generator=g) / D ** 0.5).to(torch.bfloat16)
    w = torch.randn((T, H), device=device, generator=g) / 8
    q8 = torch.empty((T, H, D), dtype=torch.uint8, device=device)
    wo = torch.empty((T, H), dtype=torch.float32, device=device)
    k = (torch.randn((T, D), device=device, generator=g) * 0.5).to(torch.bfloat16)
    gamma = torch.ones(D, device=device)
    beta = torch.zeros(D, device=device)
    bs = 64
    nb = (T + bs - 1) // bs
    slots = torch.randperm(nb * bs, device=device, generator=g)[:T].to(torch.int64)
    cache = torch.empty((nb, bs, D), dtype=torch.uint8, device=device)
    scale = torch.empty(nb * bs, dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    ws = float(D ** -0.5 * H ** -0.5)
    ops = {
        "q_quant_fold_weights": (lambda: api.q_quant_fold_weights(q, w, ws, H, q_fp8=q8,
                                                                  weights_out=wo),
                                 T * H * (D * 2 + 4 + D + 4)),
        "k_norm_quant_insert": (lambda: api.k_norm_quant_insert(k, gamma, beta, 1e-6, slots,
                                                                cache, scale),
                                T * (D * 2 + 8 + D + 4) + 2 * D * 4),
    }
    peaks, src = measured_peaks()
    stream = torch.cuda.current_stream(device)
    for name, (fn, nbytes) in ops.items():
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        times = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        gbs = nbytes / (ms / 1e3) / 1e9
        print(json.dumps({"metric": f"{name} GB/s vs HBM (before the indexer)", "value": gbs,
                          "unit": "GB/s", "ms_per_step": ms, "steps": args.steps,
                          "warmup": args.warmup, "higher_is_better": True,
                          "config": {"tokens": T, "H": H, "D": D, "bytes_per_step": nbytes,
                                     "l2": "flushed before every step"},
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                                       "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                                       "peak_source": f"{src} hbm copy"}}))
    if api.last_device_error() != api.DSA_OK:
        raise RuntimeError("device error word set")
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.prologue:
        return run_prologue(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
