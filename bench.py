#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300: prefill tokens/s and decode steps/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kda|reference]

One JSON line on stdout (rank 0).  The headline ``value`` is chunked-prefill
throughput on one 8192-token sequence with 32 heads of d = 128 (bf16 q/k/v,
fp32 state), inputs resident in HBM.  The same line carries the single-token
decode step (256 sequences x 32 heads, fp32 state updated in place, a fresh
token set every step) under ``decode``, the end-to-end number through the C
ABI from pinned host buffers under ``e2e``, the roofline of the dominant
kernel, the clocks seen during the timed region and the fp64 CPU oracle timed
on this host's cores.  Every (sequence, head) chain is independent, so N > 1
runs N replicas (one per GPU) with no collective ("replicas only").

``--impl reference`` times the fp64 CPU oracle (the reference arm of this
build) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PREFILL = "prefill_bf16_T8192_H32_D128"
DECODE = "decode_bf16_N256_H32_D128"
METRIC = "KDA prefill tokens/s and decode steps/s (H=32,d=128) on 1 GB300; % roofline"
# compulsory bytes per token-head: bf16 q, k, v, O + fp32 log_alpha + fp32 beta
BYTES_TOKEN_HEAD = 3 * 256 + 512 + 4 + 256
# contraction flops per token-head (8 C D + 6 D^2 with C = 64, D = 128), without the inverse
FLOPS_TOKEN_HEAD = 8 * 64 * 128 + 6 * 128 * 128
# the same with the chunk inverse counted as 12 C^2 per token-head
FLOPS_TOKEN_HEAD_INV = FLOPS_TOKEN_HEAD + 12 * 64 * 64
# the nominal HBM3e bandwidth, reported beside the measured peak for the decode step
HBM_NOMINAL_GBS = 8000.0
# one fp32 state of one (sequence, head), d_k = d_v = 128
STATE_BYTES = 128 * 128 * 4
PARTS = ("prefill", "decode", "verify", "few", "varlen", "long", "e2e")


# DRAM bytes per launch (dram__bytes_read.sum, dram__bytes_write.sum, in MB) of
# the ncu captures summarised under profiles/, taken on the workloads this
# script times.  An entry counts only while every source it was built from
# still hashes to the recorded prefix (sha256 of the file); after any edit to
# them the traffic reads null until a new capture replaces the entry.
PROFILED_TRAFFIC = {
    "kda_tc_prep": {
        "read_mb": 336.866304, "write_mb": 482.202112, "profile": "profiles/prefill_tc_T8192_H32_D128.md",
        "sources": {"csrc/prefill_tc.cu": "e7098c99976f671c", "csrc/umma.cuh": "351aa210ce878847",
                    "csrc/common.cuh": "cef06e6ff0b08c46"}},
    "kda_decode_kernel": {
        "read_mb": 547.411712, "write_mb": 477.935616, "profile": "profiles/decode_N256_H32_D128.md",
        "sources": {"csrc/decode.cu": "ca2b6a97d7eeaad3", "csrc/common.cuh": "cef06e6ff0b08c46"}},
    "kda_decode_multi_kernel": {
        "read_mb": 621.051648, "write_mb": 492.077056, "profile": "profiles/decode_N256_H32_D128.md",
        "sources": {"csrc/decode.cu": "ca2b6a97d7eeaad3", "csrc/common.cuh": "cef06e6ff0b08c46"}},
}


def profiled_traffic(kernel, table=None):
    """(bytes per launch, profile path) for ``kernel`` if its capture matches
    the current sources, else (None, reason)."""
    e = (PROFILED_TRAFFIC if table is None else table).get(kernel)
    if e is None:
        return None, "no capture"
    for rel, sha in e["sources"].items():
        path = os.path.join(ROOT, "kimi_delta_attention_chunked_gb300", rel)
        if not os.path.exists(path) or hashlib.sha256(open(path, "rb").read()).hexdigest()[:len(sha)] != sha:
            return None, f"{rel} changed since the capture"
    return (e["read_mb"] + e["write_mb"]) * 1e6, e["profile"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier_max(t, world, device):
    """Max of a per-rank time over all ranks (the job is as slow as its slowest replica)."""
    if world == 1:
        return t
    import torch.distributed as dist
    x = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return float(x.item())


def replica_throughput(units_per_rank, steps, world, max_ms):
    """Whole-job throughput of N independent replicas: every rank processes
    units_per_rank units per step; the job takes the slowest rank's time."""
    return units_per_rank * world * steps / (max_ms / 1e3)


def sync_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- oracle baseline
def oracle_sample(n_tokens, seed=0, min_seconds=0.0, max_repeats=1):
    """Time the fp64 oracle on the first n_tokens of the prefill workload, all 32
    heads, repeated until min_seconds have passed (at most max_repeats runs)."""
    import oracle
    from kimi_delta_attention_chunked_gb300 import inputs
    w = inputs.WORKLOADS[PREFILL]
    d = inputs.make_prefill(w, device="cpu", seed=seed, lengths=[n_tokens])
    args = [d[x].contiguous() for x in ("q", "k", "v", "log_alpha", "beta")]
    oracle.build()
    oracle.prefill(*[a[:8] for a in args])                      # load + warm
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.prefill(*args)
        runs += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or runs >= max_repeats:
            break
    return runs * n_tokens / dt, dt, oracle.max_threads(), runs


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    n_tok = 8192                                    # the whole workload per step (~0.5 s on 16 cores)
    for _ in range(args.warmup):
        oracle_sample(n_tok)
    t_all = 0.0
    cores = 1
    for _ in range(args.steps):
        _, dt, cores, _ = oracle_sample(n_tok)
        t_all += dt
    value = args.steps * n_tok / t_all
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_all / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL, "T": 8192, "H": 32, "dk": 128, "dv": 128, "chunk": 64,
                   "sample": f"all {n_tok} tokens x 32 heads per step"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"all {n_tok} tokens x 32 heads of the workload, once per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def time_prefill(kda, d, steps, warmup, stream, dev):
    q, k, v, g, b = d["q"], d["k"], d["v"], d["log_alpha"], d["beta"]
    T, H, dk = q.shape
    ws = torch.empty(kda.kda_prefill_workspace_size(1, T, H, dk, v.shape[-1], 64, q.dtype), dtype=torch.uint8,
                     device=dev)
    O = torch.empty_like(v)
    Sf = torch.empty((1, H, dk, v.shape[-1]), dtype=torch.float32, device=dev)
    call = lambda: kda.kda_prefill(q, k, v, g, b, O=O, S_final=Sf, workspace=ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        # the timed steps: the calls alone between two events
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(steps):
            call()
        end.record(stream)
        torch.cuda.synchronize()
        # then as many calls again with the library's trace events, per call
        # [start, every chunk-prep launch done, state pass joined], for the
        # split between the two kernels: an event between two kernels costs
        # each call a few microseconds, so these calls are not the timed ones
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for row in evs:
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
        for i in range(steps):
            kda.kda_set_trace_events(evs[i])
            call()
        kda.kda_set_trace_events(None)
        torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    prep_ms = [r[0].elapsed_time(r[1]) for r in evs]
    chain_ms = [r[1].elapsed_time(r[2]) for r in evs]
    return total_ms, statistics.mean(prep_ms), statistics.mean(chain_ms), 2 * steps


def time_decode(kda, w, inputs, steps, warmup, stream, dev, seed=0):
    n_sets = steps + warmup
    d = inputs.make_decode(w, device=dev, seed=seed, n_token_sets=n_sets)
    S = d["S"]
    o = torch.empty((w.B, w.H, w.dv), dtype=w.dtype, device=dev)
    with torch.cuda.stream(stream):
        for t in range(warmup):
            kda.kda_decode(d["q"][t], d["k"][t], d["v"][t], d["log_alpha"][t], d["beta"][t], S, o=o, stream=stream)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for t in range(warmup, n_sets):
            kda.kda_decode(d["q"][t], d["k"][t], d["v"][t], d["log_alpha"][t], d["beta"][t], S, o=o, stream=stream)
        end.record(stream)
        torch.cuda.synchronize()
    return start.elapsed_time(end), steps


def time_verify(kda, inputs, steps, warmup, stream, dev, K=8, N=256, H=32, D=128, seed=0):
    """Multi-token verify: K proposed tokens per sequence, all committed."""
    w = inputs.Workload("verify", "prefill", H=H, dk=D, dv=D, dtype=torch.bfloat16, T=K, B=N)
    d = inputs.make_prefill(w, device=dev, seed=seed, lengths=[K] * N)
    rs = lambda x, last: x.view(N, K, H, last).contiguous()
    q, k, v, g = rs(d["q"], D), rs(d["k"], D), rs(d["v"], D), rs(d["log_alpha"], D)
    b = d["beta"].view(N, K, H).contiguous()
    S = (torch.randn((N, H, D, D), device=dev, dtype=torch.float32) * 0.02).contiguous()
    o = torch.empty((N, K, H, D), dtype=torch.bfloat16, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            kda.kda_decode_multi(q, k, v, g, b, S, o=o, stream=stream)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            kda.kda_decode_multi(q, k, v, g, b, S, o=o, stream=stream)
        end.record(stream)
        torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    bytes_call = N * H * (8 * D * D + K * (3 * 2 * D + 4 * D + 4 + 2 * D))
    return ms, bytes_call


def time_few_heads(kda, inputs, steps, warmup, stream, dev, H=2, T=262144, seed=0):
    """One long sequence with few heads (the per-GPU share under head
    parallelism): the state pass is cut into segments and scanned."""
    w = inputs.Workload("few_heads", "prefill", T=T, B=1, H=H, dk=128, dv=128, dtype=torch.bfloat16, chunk=64)
    d = inputs.make_prefill(w, device=dev, seed=seed)
    ws = torch.empty(kda.kda_prefill_workspace_size(1, T, H, 128, 128, 64, torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    O = torch.empty_like(d["v"])
    Sf = torch.empty((1, H, 128, 128), dtype=torch.float32, device=dev)
    call = lambda: kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], O=O, S_final=Sf,
                                   workspace=ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            call()
        end.record(stream)
        torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    out = {"workload": f"prefill_bf16_T{T}_H{H}_D128", "value": T / (ms / 1e3), "unit": "tokens/s",
           "ms_per_step": ms, "note": "segment scan of the state pass (few chains, long sequence)"}
    out["roofline"] = step_roofline(T * H * BYTES_TOKEN_HEAD + H * STATE_BYTES, ms)
    return out


def step_roofline(bytes_per_step, ms, hbm=None):
    """HBM roofline of one whole prefill call: compulsory bytes (inputs, O,
    states) over the measured time, against the measured copy bandwidth."""
    hbm = hbm or peaks()[0]
    achieved = bytes_per_step / (ms / 1e3) / 1e9
    return {"bound": "hbm", "bytes_per_step": bytes_per_step, "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "floor_ms": bytes_per_step / (hbm * 1e9) * 1e3}


def time_prefill_workload(kda, inputs, name, steps, warmup, stream, dev, seed=0):
    """One of the larger prefill workloads (packed varlen with random initial
    states; the 1,048,576-token sequence), inputs resident in HBM, the same
    call a user makes.  Each workload's tensors are freed before returning."""
    w = inputs.WORKLOADS[name]
    d = inputs.make_prefill(w, device=dev, seed=seed)
    T, H, n_seq = d["T"], w.H, len(d["lengths"])
    ws = torch.empty(kda.kda_prefill_workspace_size(n_seq, T, H, 128, 128, 64, torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    O = torch.empty_like(d["v"])
    Sf = torch.empty((n_seq, H, 128, 128), dtype=torch.float32, device=dev)
    call = lambda: kda.kda_prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"],
                                   cu_seqlens=d["cu_seqlens"] if w.varlen else None,
                                   cu_seqlens_host=d["cu_seqlens_host"] if w.varlen else None,
                                   O=O, S_final=Sf, workspace=ws, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            call()
        end.record(stream)
        torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    state_io = (2 if d["S0"] is not None else 1) * n_seq * H * STATE_BYTES
    out = {"workload": name, "value": T / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
           "tokens": T, "sequences": n_seq, "lengths": d["lengths"] if w.varlen else None,
           "roofline": step_roofline(T * H * BYTES_TOKEN_HEAD + state_io, ms)}
    del d, ws, O, Sf
    torch.cuda.empty_cache()
    return out


def link_bandwidth(dev, nbytes=1 << 30, reps=3):
    """Pinned host <-> device copy rates (GB/s) on this machine, each direction
    alone, best of ``reps``: the roofline of the end-to-end number."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    g = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, (dst, src) in (("h2d_gbs", (g, h)), ("d2h_gbs", (h, g))):
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        out[name] = nbytes / (best / 1e3) / 1e9
    del h, g
    return out


def time_e2e(kda, d, steps, stream, dev):
    """Through the C ABI from pinned host buffers: every step uploads its inputs,
    runs the prefill and reads O and S_final back.  Steps are pipelined the way
    a serving loop would run them: two sets of device buffers, uploads on two
    copy streams, downloads on a third, so the upload of step i + 1 overlaps
    the prefill of step i."""
    names = ("q", "k", "v", "log_alpha", "beta")
    up_streams = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
    up_of = {"q": 0, "k": 0, "v": 0, "log_alpha": 1, "beta": 1}
    down = torch.cuda.Stream(device=dev)
    host = {n: d[n].cpu().pin_memory() for n in names}
    T, H, dk = d["q"].shape
    dv = d["v"].shape[-1]
    ws = torch.empty(kda.kda_prefill_workspace_size(1, T, H, dk, dv, 64, d["q"].dtype), dtype=torch.uint8,
                     device=dev)
    sets = []
    for _ in range(2):
        sets.append({
            "in": {n: torch.empty_like(d[n]) for n in names},
            "O": torch.empty_like(d["v"]), "Sf": torch.empty((1, H, dk, dv), dtype=torch.float32, device=dev),
            "O_h": torch.empty(d["v"].shape, dtype=d["v"].dtype).pin_memory(),
            "Sf_h": torch.empty((1, H, dk, dv), dtype=torch.float32).pin_memory(),
            "free": torch.cuda.Event(), "done": torch.cuda.Event(), "read": torch.cuda.Event()})
        sets[-1]["free"].record(stream)
        sets[-1]["read"].record(down)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sets[0]["O"].numel() * sets[0]["O"].element_size() + sets[0]["Sf"].numel() * 4

    def step(i):
        b = sets[i % 2]
        ups = []
        for j, us in enumerate(up_streams):
            us.wait_event(b["free"])                    # the prefill that last used this set is done
            with torch.cuda.stream(us):
                for n in names:
                    if up_of[n] == j:
                        b["in"][n].copy_(host[n], non_blocking=True)
            e = torch.cuda.Event()
            e.record(us)
            ups.append(e)
        for e in ups:
            stream.wait_event(e)
        stream.wait_event(b["read"])                    # its outputs have been read back
        kda.kda_prefill(b["in"]["q"], b["in"]["k"], b["in"]["v"], b["in"]["log_alpha"], b["in"]["beta"],
                        O=b["O"], S_final=b["Sf"], workspace=ws, stream=stream)
        b["free"].record(stream)
        b["done"].record(stream)
        down.wait_event(b["done"])
        with torch.cuda.stream(down):
            b["O_h"].copy_(b["O"], non_blocking=True)
            b["Sf_h"].copy_(b["Sf"], non_blocking=True)
        b["read"].record(down)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for us in up_streams:
        us.wait_event(start)
    for i in range(steps):
        step(i)
    fin = torch.cuda.Event()
    fin.record(down)
    stream.wait_event(fin)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end), h2d, d2h


def run_gpu(args):
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import kimi_delta_attention_chunked_gb300 as kda
    from kimi_delta_attention_chunked_gb300 import build, inputs
    build.build()
    kda.load()
    hbm, bf16_tf, peak_src = peaks()
    stream = torch.cuda.Stream(device=dev)
    parts = set(getattr(args, "parts", None) or PARTS)

    wp = inputs.WORKLOADS[PREFILL]
    d = inputs.make_prefill(wp, device=dev, seed=rank)
    d["S0"] = None
    T, H = d["T"], wp.H
    in_bytes = sum(d[n].numel() * d[n].element_size() for n in ("q", "k", "v", "log_alpha", "beta"))
    traffic = {name: profiled_traffic(name) for name in ("kda_tc_prep", "kda_decode_kernel", "kda_decode_multi_kernel")}
    line = {"metric": METRIC, "value": None, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": PREFILL, "B": 1, "T": T, "H": H, "dk": 128, "dv": 128, "chunk": 64,
                       "state": "fp32, S0 = 0", "parallelism": "replicas" if world > 1 else "single",
                       "l2": f"inputs {in_bytes / 1e6:.0f} MB per step > 129 MB L2 (no flush)"}}
    if parts != set(PARTS):
        line["parts"] = sorted(parts)

    sync_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        if "prefill" in parts:
            ms, prep_ms, chain_ms, launches = time_prefill(kda, d, args.steps, args.warmup, stream, dev)
            ms = barrier_max(ms, world, dev)
            ms_step = ms / args.steps
            # roofline of the dominant kernel: the chunk-prep launches, which run
            # back to back on the caller's stream, timed from the first prep
            # launch to the last one's end
            prep_bytes = T * H * (3 * 256 + 512 + 4)               # q, k, v, log_alpha, beta read once
            achieved = prep_bytes / (prep_ms / 1e3) / 1e9
            step_bytes = T * H * BYTES_TOKEN_HEAD + H * STATE_BYTES
            line.update({
                "value": replica_throughput(T, args.steps, world, ms), "ms_per_step": ms_step,
                "roofline": {"bound": "hbm", "kernel": "kda_tc_prep", "achieved": achieved, "peak": hbm,
                             "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic["kda_tc_prep"][0],
                             "traffic_source": traffic["kda_tc_prep"][1], "peak_source": peak_src,
                             "bytes_per_launch": prep_bytes, "launch_ms": prep_ms},
                "step_roofline": dict(step_roofline(step_bytes, ms_step, hbm),
                                      tflops=T * H * FLOPS_TOKEN_HEAD / (ms_step / 1e3) / 1e12,
                                      tflops_with_inverse=T * H * FLOPS_TOKEN_HEAD_INV / (ms_step / 1e3) / 1e12,
                                      kernel_ms={"kda_tc_prep_span": prep_ms, "state_pass_tail": chain_ms}),
                "gpu_launches": launches * world})
            sync_barrier(world)
        if "decode" in parts:
            wd = inputs.WORKLOADS[DECODE]
            dms, dsteps = time_decode(kda, wd, inputs, max(args.steps, args.decode_steps), args.warmup, stream, dev,
                                      seed=rank)
            dms = barrier_max(dms, world, dev)
            dec_bytes_step = wd.B * wd.H * (8 * wd.dk * wd.dv + 3 * 256 + 512 + 4 + 256)
            dec_ms_step = dms / dsteps
            dec_achieved = dec_bytes_step / (dec_ms_step / 1e3) / 1e9
            line["decode"] = {
                "workload": DECODE, "value": replica_throughput(1, dsteps, world, dms), "unit": "steps/s",
                "steps": dsteps, "ms_per_step": dec_ms_step,
                "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel", "achieved": dec_achieved,
                             "peak": hbm, "unit": "GB/s", "frac": dec_achieved / hbm,
                             "frac_of_nominal_8tbs": dec_achieved / HBM_NOMINAL_GBS,
                             "traffic": traffic["kda_decode_kernel"][0],
                             "traffic_source": traffic["kda_decode_kernel"][1], "bytes_per_launch": dec_bytes_step},
                "l2": "fp32 state 537 MB > L2; fresh token set per step"}
            torch.cuda.empty_cache()
        if "verify" in parts:
            vms, vbytes = time_verify(kda, inputs, max(args.steps, 50), args.warmup, stream, dev, seed=rank)
            vms = barrier_max(vms, world, dev)
            line["verify"] = {
                "workload": "verify_bf16_N256_K8_H32_D128", "value": replica_throughput(1, 1, world, vms),
                "unit": "calls/s", "ms_per_call": vms,
                "roofline": {"bound": "hbm", "kernel": "kda_decode_multi_kernel",
                             "achieved": vbytes / (vms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                             "frac": vbytes / (vms / 1e3) / 1e9 / hbm,
                             "traffic": traffic["kda_decode_multi_kernel"][0],
                             "traffic_source": traffic["kda_decode_multi_kernel"][1], "bytes_per_launch": vbytes}}
        if "few" in parts:
            line["few_heads_long"] = time_few_heads(kda, inputs, max(3, args.steps // 4), args.warmup, stream, dev,
                                                    seed=rank)
        if "varlen" in parts:
            line["varlen"] = time_prefill_workload(kda, inputs, "varlen_bf16_8seq_1K_32K_H32_D128",
                                                   max(3, args.steps // 4), args.warmup, stream, dev, seed=rank)
        if "long" in parts:
            line["long_1M"] = time_prefill_workload(kda, inputs, "long_bf16_T1M_H32_D128", args.long_steps,
                                                    min(args.warmup, 2), stream, dev, seed=rank)
    line["clocks"] = clk.summary()
    if "e2e" in parts:
        e2e_steps = max(6, args.steps // 2)
        e2e_ms, h2d, d2h = time_e2e(kda, d, e2e_steps, stream, dev)
        e2e_ms = barrier_max(e2e_ms, world, dev)
        link = link_bandwidth(dev)
        e2e_step_ms = e2e_ms / e2e_steps
        # with uploads and downloads on separate copy streams the copies of one
        # step can at best run at the link's one-direction rates, in parallel
        copy_floor_ms = max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9)) * 1e3
        line["e2e"] = {"value": replica_throughput(T, e2e_steps, world, e2e_ms), "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step_ms,
                       "pipelining": "2 buffer sets; uploads on 2 copy streams overlap the previous step's prefill",
                       "roofline": {"bound": "host link", "link_gbs": link, "copy_floor_ms": copy_floor_ms,
                                    "frac": copy_floor_ms / e2e_step_ms}}
    if rank == 0 and not args.no_cpu_baseline:
        v, dt, cores, runs = oracle_sample(args.oracle_tokens, min_seconds=args.oracle_seconds, max_repeats=40)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{args.oracle_tokens} of 8192 tokens x 32 heads, {runs} runs ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--oracle-tokens", type=int, default=8192)
    ap.add_argument("--oracle-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--long-steps", type=int, default=3, help="timed steps of the 1,048,576-token prefill")
    ap.add_argument("--parts", type=lambda x: [p for p in x.split(",") if p], default=None,
                    help="comma list of " + ",".join(PARTS) + " (default: all)")
    args = ap.parse_args()
    for p in args.parts or ():
        if p not in PARTS:
            ap.error(f"unknown part {p}")
    if args.warmup < 3 and args.impl == "kda":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
