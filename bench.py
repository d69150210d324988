#!/usr/bin/env python3
"""Benchmark of the Engram conditional-memory hot path on GB300.

One step = one pass of the whole hot path over one batch of 16 sequences x 4096
tokens (65,536 tokens):
  1. hash + gather of every token's 16 table rows (orders {2, 3} x 8 heads,
     ~2.0M-row prime tables, 64 bf16 per row, 4.1 GB resident) -> e [65536, 1024];
  2. the context-aware gate, forward + backward on four micro-batches of
     T = 16384 tokens at d = 4096 (bf16), the first forward also forming the
     weight fold w = w_h * w_k that the others use, the backwards adding into
     one array of weight-gradient partials (the first writes it), then one
     ordered reduction of those partials, accumulating into fp32 grad_w_h /
     grad_w_k (10 kernel launches: the hash + gather is one).
The reported value is tokens/s through the whole step (whole job, all ranks).
The same line also carries the gate on its own workloads (`configs`: forward
alone at T = 8192, d = 2048; fwd + bwd + reduce at d = 7168 for three token
counts and a ragged pack) and the NEXT rows' kernels on theirs (`next_rows`).
Inputs are resident in HBM (the device-timed value) or copied from pinned host
memory every step (the `e2e` value).  The per-step working set (4.1 GB table,
2 GB of gate inputs) is far larger than L2, so no flush is needed.

`--impl reference` times the CPU oracle (the correctness reference, plain C,
fp64) on the host cores instead: every timed step is one whole step of the same
workload, nothing sampled or scaled.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import json
import math
import os
import statistics
import subprocess
import sys
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "gate fwd+bwd tokens/s and HBM GB/s (% of roofline); hash-gather rows/s"
SEQS, SEQ_LEN = 16, 4096
MICRO_T, D = 16384, 4096
EPS = 1e-6
STEP_LAUNCHES = 10
WORKLOAD = (f"engram step: hash+gather {SEQS}x{SEQ_LEN} tokens (Zipf(1.1) ids over V=128000 -> V'=98560, "
            f"16 tables of ~2.0M x 64 bf16 = 4.1 GB) + weight fold + gate fwd/bwd/grad_w_reduce on "
            f"4 micro-batches T={MICRO_T} d={D} bf16")


# ----------------------------------------------------------------------------- host-side plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return rank, local, world


def aggregate_max(value: float, group_backend_device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=group_backend_device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def load_traffic(kernel: str):
    """ncu DRAM bytes per launch recorded for `kernel`, or None when its source changed since the capture."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return rec["dram_bytes_per_launch"] if h.hexdigest() == rec["sources_sha256"] else None


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) taken while the timed region runs."""

    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", f"engram_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t0: _dt.datetime, t1: _dt.datetime):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != len(self.FIELDS):
                    continue
                try:
                    ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if len(inside) < 3:  # short timed region: widen to the samples around it
            pad = _dt.timedelta(seconds=0.5)
            inside = [r for r in rows if t0 - pad <= r[0] <= t1 + pad]
            window = "timed region +- 0.5 s"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------- the workload

def algorithmic_bytes(P: int):
    """Algorithmic HBM bytes per launch of each kernel in one step (see the design notes)."""
    T_all = SEQS * SEQ_LEN
    tables, row_bytes = 16, 128
    return {
        "hash_gather": T_all * (4 + 4 + 2 * tables * row_bytes),  # id, compressed id, 16 rows read + e_t written
        "gate_fwd_fold": MICRO_T * (8 * D + 16) + 3 * 4 * D,      # the forward + w_h, w_k read, w_fused written
        "gate_fwd": MICRO_T * (8 * D + 16),                       # h, k, v read, out written, 4 fp32 stats
        "gate_bwd": MICRO_T * (14 * D + 16) + P * D * 4,         # dout, v, h, k, stats read; dh, dk, dv, partials
        "gate_bwd_accumulate": MICRO_T * (14 * D + 16) + 2 * P * D * 4,  # the same + the partials read back
        "grad_w_reduce": P * D * 4 + 7 * D * 4,                   # the accumulated partials, w_h, w_k, grads, dweight
    }


def make_workload(device):
    import torch

    from synth import device as SD
    from synth import workloads as W

    hw = W.hash_gather_64k(num_seqs=SEQS, seq_len=SEQ_LEN)
    gates = [W.GateWorkload(name=f"mb{i}", T=MICRO_T, d=D, dtype="bf16", seed=3 * 101 + 7 + 1000003 * i)
             for i in range(4)]
    import engram_conditional_memory_gb300 as ecm

    s = hw.spec
    wk = {
        "hw": hw,
        "spec": ecm.HashSpec(s.min_order, s.num_orders, s.heads, s.multipliers, s.primes),
        "ids": torch.from_numpy(hw.token_ids).to(device),
        "offs": torch.from_numpy(hw.seq_offsets).to(device),
        "cmap": torch.from_numpy(hw.compress_map).to(device),
        "table": SD.hash_table(hw, device),
        "mb": [SD.gate_device_inputs(g, device) for g in gates],
    }
    w0 = wk["mb"][0]
    wk["w_h"], wk["w_k"] = w0["w_h"], w0["w_k"]
    T_all = hw.T
    wk["rows"] = torch.empty((T_all, s.tables * hw.row_dim), dtype=torch.bfloat16, device=device)
    wk["w_fused"] = torch.empty(D, dtype=torch.float32, device=device)
    P = ecm.gate_bwd_num_partials(MICRO_T, D)
    wk["P"] = P
    wk["out"] = [torch.empty((MICRO_T, D), dtype=torch.bfloat16, device=device) for _ in range(4)]
    wk["dh"] = [torch.empty_like(o) for o in wk["out"]]
    wk["dk"] = [torch.empty_like(o) for o in wk["out"]]
    wk["dv"] = [torch.empty_like(o) for o in wk["out"]]
    wk["stats"] = [tuple(torch.empty(MICRO_T, dtype=torch.float32, device=device) for _ in range(4))
                   for _ in range(4)]
    # one array of weight-gradient partials: micro-batch 0 writes it, 1-3 add to it, one reduction
    wk["part"] = torch.empty((P, D), dtype=torch.float32, device=device)
    wk["dweight"] = torch.empty(D, dtype=torch.float32, device=device)
    wk["grad_w_h"] = torch.zeros(D, dtype=torch.float32, device=device)
    wk["grad_w_k"] = torch.zeros(D, dtype=torch.float32, device=device)
    wk["num_sms"] = torch.cuda.get_device_properties(device).multi_processor_count
    return wk


def gate_forward(wk, i):
    """Micro-batch i's forward; the first one also forms the weight fold the later calls use."""
    import engram_conditional_memory_gb300 as ecm

    m, st = wk["mb"][i], wk["stats"][i]
    if i == 0:
        ecm.gate_fwd_fold(m["h"], m["k"], m["v"], wk["w_h"], wk["w_k"], EPS, out=wk["out"][i], stats=st,
                          w_fused_out=wk["w_fused"])
    else:
        ecm.gate_fwd(m["h"], m["k"], m["v"], wk["w_fused"], EPS, out=wk["out"][i], stats=st)


def run_step(wk, mark=None, gather_stream=None):
    """Launch one step (10 kernels) on the current stream; `mark(name)` is called after each call.

    With `gather_stream`, the hash + gather runs there, beside the gate work, with one CTA per SM (so
    that each SM also holds the gate's CTAs), and the current stream waits for it at the end.  The
    rows a token needs follow from its ids alone, so a pipelined step gathers while the gate work runs:
    across steps that is the same throughput as gathering the next batch during this one's gate work.
    The gather's latency-bound DRAM traffic (random 128-byte rows) then shares HBM with the gate's
    streaming instead of running alone."""
    import torch

    import engram_conditional_memory_gb300 as ecm

    hw = wk["hw"]
    main = torch.cuda.current_stream()
    if gather_stream is not None:
        gather_stream.wait_stream(main)
        with torch.cuda.stream(gather_stream):
            prev = ecm.set_max_ctas(wk["num_sms"])
            try:
                ecm.hash_gather(wk["spec"], wk["ids"], wk["offs"], wk["table"], wk["cmap"], hw.vocab, hw.vocab_c,
                                out_rows=wk["rows"])
            finally:
                ecm.set_max_ctas(prev)
    else:
        ecm.hash_gather(wk["spec"], wk["ids"], wk["offs"], wk["table"], wk["cmap"], hw.vocab, hw.vocab_c,
                        out_rows=wk["rows"])
        mark and mark("hash_gather")
    for i, m in enumerate(wk["mb"]):
        st = wk["stats"][i]
        gate_forward(wk, i)
        mark and mark("gate_fwd_fold" if i == 0 else "gate_fwd")
        ecm.gate_bwd(m["dout"], m["h"], m["k"], m["v"], wk["w_fused"], *st, P=wk["P"], dh=wk["dh"][i],
                     dk=wk["dk"][i], dv=wk["dv"][i], dw_partial=wk["part"], accumulate=i > 0)
        mark and mark("gate_bwd_accumulate" if i else "gate_bwd")
    reduce_step(wk)
    mark and mark("grad_w_reduce")
    if gather_stream is not None:
        main.wait_stream(gather_stream)
    return STEP_LAUNCHES


def reduce_step(wk):
    """The step's weight gradient: one ordered reduction of the partials the four micro-batches
    added into, accumulated into grad_w_h and grad_w_k as gradient accumulation would."""
    import engram_conditional_memory_gb300 as ecm

    ecm.grad_w_reduce(wk["part"], dweight_fused=wk["dweight"], w_h=wk["w_h"], w_k=wk["w_k"],
                      grad_w_h=wk["grad_w_h"], grad_w_k=wk["grad_w_k"])


# ----------------------------------------------------------------------------- device timing

def capture_step(wk, device):
    """The step as one CUDA graph (10 kernel nodes, the hash + gather on a branch of its own beside
    the gate work).  The library's per-device set-up and each kernel's shared-memory attribute are
    done by an eager step first; device-pointer checks are off during capture (they were made by
    that eager step on the same buffers)."""
    import torch

    import engram_conditional_memory_gb300 as ecm

    side = torch.cuda.Stream(device)
    gather = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run_step(wk, gather_stream=gather)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    prev = ecm.set_validation(0)
    try:
        with torch.cuda.graph(graph):
            run_step(wk, gather_stream=gather)
    finally:
        ecm.set_validation(prev)
    return graph


def time_graph(graph, steps, warmup, device):
    """Device time of `steps` replays of the step graph (CUDA events on the replaying stream)."""
    import torch

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(device)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    wall0 = _dt.datetime.now()
    start.record(stream)
    for _ in range(steps):
        graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    wall1 = _dt.datetime.now()
    barrier(device)
    return start.elapsed_time(end), STEP_LAUNCHES * steps, wall0, wall1


def time_device(wk, steps, warmup, device):
    """Eager steps with a CUDA event between consecutive launches: the per-kernel durations."""
    import torch

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        run_step(wk)
    torch.cuda.synchronize()
    # events between consecutive launches: per-kernel durations inside the timed region
    bounds = []

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        bounds.append((name, e))

    barrier(device)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    wall0 = _dt.datetime.now()
    start.record(stream)
    prev = start
    launches = 0
    for _ in range(steps):
        launches += run_step(wk, mark)
    end.record(stream)
    torch.cuda.synchronize()
    wall1 = _dt.datetime.now()
    barrier(device)
    elapsed = start.elapsed_time(end)
    per = {}
    for name, e in bounds:
        per.setdefault(name, []).append(prev.elapsed_time(e))
        prev = e
    return elapsed, per, launches, wall0, wall1


def time_e2e(wk, steps, warmup, device):
    """Same step through the public API, with each step's inputs copied from pinned host memory and
    the step's result (the accumulated fp32 weight gradients) read back to the host.

    Copies run on a copy stream into the four micro-batch buffers, so micro-batch i+1 crosses the
    host link while micro-batch i computes; events order every reuse of a buffer or of the ids.
    """
    import torch

    import engram_conditional_memory_gb300 as ecm

    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device)
    names = ("h", "k", "v", "dout")
    host_ids = wk["ids"].cpu().pin_memory()
    host_mb = [{n: m[n].cpu().pin_memory() for n in names} for m in wk["mb"]]
    res_h = torch.empty(2 * D, dtype=torch.float32, pin_memory=True)
    h2d = host_ids.numel() * 4 + sum(t.numel() * t.element_size() for m in host_mb for t in m.values())
    d2h = res_h.numel() * 4
    ready = [torch.cuda.Event() for _ in range(4)]   # micro-batch i's inputs are on the device
    done = [torch.cuda.Event() for _ in range(4)]    # compute has finished reading micro-batch i
    ids_ready, hash_done = torch.cuda.Event(), torch.cuda.Event()
    hw = wk["hw"]

    def step():
        with torch.cuda.stream(copy):
            copy.wait_event(hash_done)  # the previous step's hash has read the id buffer
            wk["ids"].copy_(host_ids, non_blocking=True)
            ids_ready.record(copy)
            for i, m in enumerate(wk["mb"]):
                copy.wait_event(done[i])  # the previous step has finished with this buffer
                for n in names:
                    m[n].copy_(host_mb[i][n], non_blocking=True)
                ready[i].record(copy)
        comp.wait_event(ids_ready)
        ecm.hash_gather(wk["spec"], wk["ids"], wk["offs"], wk["table"], wk["cmap"], hw.vocab, hw.vocab_c,
                        out_rows=wk["rows"])
        hash_done.record(comp)
        for i, m in enumerate(wk["mb"]):
            comp.wait_event(ready[i])
            st = wk["stats"][i]
            gate_forward(wk, i)
            ecm.gate_bwd(m["dout"], m["h"], m["k"], m["v"], wk["w_fused"], *st, P=wk["P"], dh=wk["dh"][i],
                         dk=wk["dk"][i], dv=wk["dv"][i], dw_partial=wk["part"], accumulate=i > 0)
            done[i].record(comp)
        reduce_step(wk)
        res_h[:D].copy_(wk["grad_w_h"], non_blocking=True)
        res_h[D:].copy_(wk["grad_w_k"], non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(comp)
    copy.wait_event(start)  # no copy of the timed region starts before the start event
    for _ in range(steps):
        step()
    end.record(comp)
    torch.cuda.synchronize()
    barrier(device)
    return start.elapsed_time(end), h2d, d2h


# ----------------------------------------------------------------------------- the CPU oracle

def _oracle_threads():
    return max(1, os.cpu_count() or 1)


def _ranges(n: int, parts: int):
    parts = max(1, min(parts, n)) if n else 1
    return [(n * i // parts, n * (i + 1) // parts) for i in range(parts)]


ORACLE_GATE_CHUNK = 256  # tokens per oracle call in the gate legs (bounds each call's fp64 outputs)


def oracle_step(pool, threads, hw, table_host, mbs_host, w_h, w_k):
    """Seconds of ONE WHOLE step computed by the oracle over the full workload, nothing sampled
    or scaled: hash + gather of all 65,536 tokens from the full 4.1 GB table, the fold, gate
    forward + backward of all four micro-batches (4 x 16384 tokens), then the ordered reduction of
    the per-range weight-gradient sums into both weight gradients.  Token ranges run on `threads`
    host threads (ctypes releases the GIL inside each oracle call)."""
    import oracle

    s = hw.spec

    def hash_part(b):
        idx = oracle.hash_indices(hw.token_ids, hw.seq_offsets, hw.compress_map, hw.vocab, s.min_order,
                                  s.num_orders, s.heads, s.multipliers, s.primes, b[0], b[1])
        oracle.gather_rows(table_host, s.primes, idx)

    def gate_part(args):
        m, (t0, t1) = args
        oracle.gate_fwd(m["h"], m["k"], m["v"], w_h, w_k, EPS, t0, t1)
        return oracle.gate_bwd(m["dout"], m["h"], m["k"], m["v"], w_h, w_k, EPS, t0, t1)["dweight"]

    t0 = time.perf_counter()
    list(pool.map(hash_part, _ranges(hw.T, 4 * threads)))
    oracle.fuse_weight(w_h, w_k)
    work = [(m, b) for m in mbs_host
            for b in _ranges(m["h"].shape[0], max(1, m["h"].shape[0] // ORACLE_GATE_CHUNK))]
    partials = np.stack(list(pool.map(gate_part, work)))
    oracle.grad_w_reduce(partials, w_h, w_k)
    return time.perf_counter() - t0


def _bf16_bits(t):
    """Host numpy view (raw uint16 bits) of a CPU bf16 tensor, no copy."""
    import torch

    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_inputs_from_device(wk):
    """Host copies of the step's device inputs: the full table and all four micro-batches."""
    table_host = _bf16_bits(wk["table"].cpu())
    mbs = [{n: _bf16_bits(m[n].cpu()) for n in ("h", "k", "v", "dout")} for m in wk["mb"]]
    return table_host, mbs, wk["w_h"].cpu().numpy(), wk["w_k"].cpu().numpy()


def oracle_inputs_on_host(hw):
    """The same workload drawn on the host with torch's CPU generator from the same seeds and recipe
    (values differ from the device draws; sizes and distributions are the same).  Every page of the
    4.1 GB table and of the 2.1 GB of gate inputs is written, so the oracle reads real memory."""
    from synth import device as SD
    from synth import workloads as W

    table_host = _bf16_bits(SD.hash_table(hw, "cpu"))
    mbs = []
    for i in range(4):
        g = W.GateWorkload(name=f"mb{i}", T=MICRO_T, d=D, dtype="bf16", seed=3 * 101 + 7 + 1000003 * i)
        t = SD.gate_device_inputs(g, "cpu")
        mbs.append({n: _bf16_bits(t[n]) for n in ("h", "k", "v", "dout")})
        if i == 0:
            w_h, w_k = t["w_h"].numpy(), t["w_k"].numpy()
    return table_host, mbs, w_h, w_k


def time_oracle_steps(hw, table_host, mbs, w_h, w_k, steps: int, warmup: int):
    """Wall seconds of each of `steps` whole oracle steps after `warmup` untimed ones."""
    threads = _oracle_threads()
    times = []
    with ThreadPoolExecutor(threads) as pool:
        for i in range(warmup + steps):
            t = oracle_step(pool, threads, hw, table_host, mbs, w_h, w_k)
            if i >= warmup:
                times.append(t)
    return times, threads


def oracle_sample_text(steps: int, threads: int) -> str:
    return (f"{steps} whole steps timed one by one (none sampled or scaled): hash+gather of all {SEQS * SEQ_LEN} "
            f"tokens from the full 4.1 GB table, fold, gate fwd+bwd of all 4 x {MICRO_T} tokens, ordered "
            f"weight-gradient reduction; {threads} host threads")


ORACLE_CONFIG_SAMPLE = 4096  # tokens the per-config oracle rates are measured on (whole T where smaller)


def _rates(run_part, reduce, ranges, n_tokens: int, what: str) -> dict:
    """tokens/s of the oracle over `ranges` (then `reduce` of the parts), first on one core (one call
    after another), then on every core (the same calls on a thread pool)."""
    t0 = time.perf_counter()
    reduce([run_part(b) for b in ranges])
    t1 = time.perf_counter() - t0
    threads = _oracle_threads()
    with ThreadPoolExecutor(threads) as pool:
        t0 = time.perf_counter()
        reduce(list(pool.map(run_part, ranges)))
        t2 = time.perf_counter() - t0
    return {"single_core": {"tokens_per_s": n_tokens / t1, "cores": 1, "seconds": t1},
            "all_cores": {"tokens_per_s": n_tokens / t2, "cores": threads, "seconds": t2},
            "sample": what}


def oracle_gate_rates(x: dict, fwd_only: bool, T_config: int) -> dict:
    """The oracle's gate on host copies of a config's first tokens: the forward, or forward +
    backward of every token then the ordered reduction of the per-call weight-gradient sums."""
    import oracle

    n = x["h"].shape[0]
    ranges = _ranges(n, max(1, n // ORACLE_GATE_CHUNK))

    def part(b):
        oracle.gate_fwd(x["h"], x["k"], x["v"], x["w_h"], x["w_k"], EPS, b[0], b[1])
        if not fwd_only:
            return oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], EPS, b[0], b[1])["dweight"]

    def reduce(parts):
        if not fwd_only:
            oracle.grad_w_reduce(np.stack(parts), x["w_h"], x["w_k"])

    ops = "gate fwd" if fwd_only else "gate fwd + bwd + ordered reduction"
    what = (f"{ops} of all {n} tokens" if n == T_config else
            f"{ops} of the first {n} of the {T_config} tokens (the oracle's cost per token does not depend on T)")
    return _rates(part, reduce, ranges, n, what + f", in {len(ranges)} calls")


def oracle_hash_rates(hw, table_host) -> dict:
    """The oracle's hash + gather of every token of the step's batch from the full host table."""
    import oracle

    s = hw.spec

    def part(b):
        idx = oracle.hash_indices(hw.token_ids, hw.seq_offsets, hw.compress_map, hw.vocab, s.min_order,
                                  s.num_orders, s.heads, s.multipliers, s.primes, b[0], b[1])
        oracle.gather_rows(table_host, s.primes, idx)

    ranges = _ranges(hw.T, 4 * _oracle_threads())
    return _rates(part, lambda parts: None, ranges, hw.T,
                  f"hash + gather of all {hw.T} tokens from the full 4.1 GB table, in {len(ranges)} calls")


# ----------------------------------------------------------------------------- the gate at every workload size

L2_BYTES = 129 * 2 ** 20


def _gate_config_entry(wl, device, steps: int, warmup: int, peak: float, fwd_only: bool, with_oracle: bool = False):
    """Gate kernels of one workload, each timed on its own over rotating input sets (so a launch
    never finds its inputs in L2 from the previous use), plus the fwd -> bwd -> grad_w_reduce
    sequence for training workloads.  Every timing is a CUDA-graph replay with events between
    replays on the replaying stream; per launch = median replay time / launches per replay."""
    import torch

    import engram_conditional_memory_gb300 as ecm
    from synth import device as SD

    T, d = wl.T, wl.d
    fwd_b = T * (8 * d + 16)
    sets = max(2, min(8, math.ceil(6 * L2_BYTES / fwd_b)))
    P = ecm.gate_bwd_num_partials(T, d)
    bwd_b = T * (14 * d + 16) + 4 * d * P
    red_b = 4 * d * P + 28 * d
    S = []
    for j in range(sets):
        w = wl if j == 0 else type(wl)(**{**wl.__dict__, "seed": wl.seed + 7919 * j})
        t = SD.gate_device_inputs(w, device, with_dout=not fwd_only)
        s = {"in": t, "wf": ecm.fuse_weight(t["w_h"], t["w_k"]), "out": torch.empty_like(t["v"]),
             "st": tuple(torch.empty(T, dtype=torch.float32, device=device) for _ in range(4))}
        if not fwd_only:
            s.update(dh=torch.empty_like(t["h"]), dk=torch.empty_like(t["k"]), dv=torch.empty_like(t["v"]),
                     part=torch.empty((P, d), dtype=torch.float32, device=device),
                     dw=torch.empty(d, dtype=torch.float32, device=device),
                     gh=torch.zeros(d, dtype=torch.float32, device=device),
                     gk=torch.zeros(d, dtype=torch.float32, device=device))
        S.append(s)

    def fwd(s):
        t = s["in"]
        ecm.gate_fwd(t["h"], t["k"], t["v"], s["wf"], wl.eps, out=s["out"], stats=s["st"])

    def bwd(s):
        t = s["in"]
        ecm.gate_bwd(t["dout"], t["h"], t["k"], t["v"], s["wf"], *s["st"], P=P, dh=s["dh"], dk=s["dk"],
                     dv=s["dv"], dw_partial=s["part"])

    def red(s):
        t = s["in"]
        ecm.grad_w_reduce(s["part"], dweight_fused=s["dw"], w_h=t["w_h"], w_k=t["w_k"], grad_w_h=s["gh"],
                          grad_w_k=s["gk"])

    def seq(s):
        fwd(s)
        bwd(s)
        red(s)

    stream = torch.cuda.current_stream()

    def graph_time(fn, per_replay: int):
        for s in S:  # eager first: per-device set-up and pointer checks outside the capture
            fn(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        prev = ecm.set_validation(0)
        try:
            with torch.cuda.graph(g):
                for s in S:
                    fn(s)
        finally:
            ecm.set_validation(prev)
        for _ in range(warmup):
            g.replay()
        reps = max(3, math.ceil(steps / sets))
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(reps):
            g.replay()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        ms = statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(reps))
        return ms / (sets * per_replay), reps * sets * per_replay

    def entry(ms, nbytes, launches):
        gbs = nbytes / (ms / 1e3) / 1e9
        return {"avg_us": ms * 1e3, "bytes": nbytes, "GBps": gbs, "frac": gbs / peak, "launches_timed": launches}

    res = {"T": T, "d": d, "dtype": wl.dtype, "sets": sets,
           "l2": f"{sets} rotating input sets: {sets - 1} other launches' inputs between reuses of one set"}
    if wl.seq_lengths is not None:
        res["ragged"] = {"sequences": int(len(wl.seq_lengths)), "min_len": int(wl.seq_lengths.min()),
                         "max_len": int(wl.seq_lengths.max()), "packed_as_one_T": T}
    ms, n = graph_time(fwd, 1)
    res["gate_fwd"] = entry(ms, fwd_b, n)
    res["gate_fwd"]["tokens_per_s"] = T / (ms / 1e3)
    if not fwd_only:
        res["P"] = P
        ms, n = graph_time(bwd, 1)
        res["gate_bwd"] = entry(ms, bwd_b, n)
        ms, n = graph_time(red, 1)
        res["grad_w_reduce"] = entry(ms, red_b, n)
        res["grad_w_reduce"]["note"] = "alone, partials read from HBM"
        ms, n = graph_time(seq, 3)
        step = entry(3 * ms, fwd_b + bwd_b + red_b, n)
        step["tokens_per_s"] = T / (3 * ms / 1e3)
        step["launches_per_step"] = 3
        res["fwd_bwd_reduce"] = step
    if with_oracle:  # the oracle on host copies of set 0's first tokens, on one core and on all
        n = min(T, ORACLE_CONFIG_SAMPLE) if T > 2 * ORACLE_CONFIG_SAMPLE else T
        t = S[0]["in"]
        host = (lambda a: _bf16_bits(a)) if t["h"].dtype == torch.bfloat16 else (lambda a: a.contiguous().numpy())
        x = {nm: host(t[nm][:n].cpu()) for nm in (("h", "k", "v") if fwd_only else ("h", "k", "v", "dout"))}
        x["w_h"], x["w_k"] = t["w_h"].cpu().numpy(), t["w_k"].cpu().numpy()
        res["oracle"] = oracle_gate_rates(x, fwd_only, T)
    del S
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def time_gate_configs(device, steps: int, warmup: int, peak: float, with_oracle: bool = False):
    """The gate-only workloads: forward at T = 8192, d = 2048, and fwd + bwd + grad_w_reduce at
    d = 7168 for T in {4096, 32768, 131072} and a ragged pack of 64 sequences (the gate sees one T);
    with_oracle: also the oracle's rate on each, on one core and on all host cores."""
    from synth import workloads as W

    out = {}
    wl = W.gate_fwd_2k()
    out[wl.name] = _gate_config_entry(wl, device, steps, warmup, peak, fwd_only=True, with_oracle=with_oracle)
    for wl in (W.gate_sweep_7k(4096), W.gate_sweep_7k(32768), W.gate_sweep_7k(131072), W.gate_ragged_7k()):
        out[wl.name] = _gate_config_entry(wl, device, steps, warmup, peak, fwd_only=False, with_oracle=with_oracle)
    return out


# ----------------------------------------------------------------------------- single-op runs (profiling)

def time_only(op: str, steps: int, warmup: int, device) -> dict:
    """Time one kernel (or one fixed sequence of kernels) alone on its workload, as CUDA-graph replays
    with an event between replays (eager where capture is refused): the NEXT rows' workloads and the
    small cases the ncu captures are taken on."""
    import types

    import torch

    import engram_conditional_memory_gb300 as ecm
    from synth import device as SD
    from synth import workloads as W

    args = types.SimpleNamespace(only=op, steps=steps, warmup=warmup)
    stream = torch.cuda.current_stream()
    if op.startswith("hash_gather"):
        if op == "hash_gather_small":  # 4 x 4096 tokens, 16 tables of ~200k rows (0.41 GB, > L2)
            hw = W.hash_gather_64k(num_seqs=4, seq_len=SEQ_LEN)
            hw = W.HashGatherWorkload(**{**hw.__dict__, "spec": W.hash_spec(4 * 7919 + 11, 2, 2, 8, 200_003)})
        else:
            hw = W.hash_gather_64k(num_seqs=SEQS, seq_len=SEQ_LEN)
        s = hw.spec
        spec = ecm.HashSpec(s.min_order, s.num_orders, s.heads, s.multipliers, s.primes)
        ids, offs = torch.from_numpy(hw.token_ids).to(device), torch.from_numpy(hw.seq_offsets).to(device)
        cmap, table = torch.from_numpy(hw.compress_map).to(device), SD.hash_table(hw, device)
        if op == "hash_gather_host":  # the same 4.1 GB table, page-locked in host memory
            table = table.cpu().pin_memory()
        rows = torch.empty((hw.T, s.tables * hw.row_dim), dtype=table.dtype, device=device)
        nbytes = hw.T * (8 + 2 * s.tables * hw.row_dim * 2)

        def launch():
            ecm.hash_gather(spec, ids, offs, table, cmap, hw.vocab, hw.vocab_c, out_rows=rows)
    elif op.startswith("gate_hc"):
        # the multi-branch gate at its production shape: T = 8192, hc = 4, d = 4096, bf16; the _d7168
        # ops take rows too large for a whole token (T = 4096, hc = 4, d = 7168), run branch by branch
        wl = W.gate_hc_4x4k()
        if op.endswith("_d7168"):
            wl = W.GateHcWorkload(name="gate_hc4_T4096_d7168", T=4096, hc=4, d=7168, dtype="bf16", seed=wl.seed)
        T, hc, d = wl.T, wl.hc, wl.d
        x = SD.normal_tensor((T * hc, d), wl.seed + 1, 0.0, 1.0, "bf16", device).reshape(T, hc, d)
        kv = SD.normal_tensor((T * (hc + 1), d), wl.seed + 2, 0.0, 1.0, "bf16", device).reshape(T, hc + 1, d)
        g = SD.normal_tensor((T * hc, d), wl.seed + 3, 0.0, 1.0, "bf16", device).reshape(T, hc, d)
        w_h = SD.normal_tensor((1, hc * d), wl.seed + 4, 1.0, 0.1, "f32", device).reshape(-1)
        w_k = SD.normal_tensor((1, hc * d), wl.seed + 5, 1.0, 0.1, "f32", device).reshape(-1)
        wf = ecm.fuse_weight(w_h, w_k).reshape(hc, d)
        out, *st = ecm.gate_hc_fwd(x, kv, wf, wl.eps, wl.clamp)
        P = ecm.gate_bwd_num_partials(T, hc * d)
        dx, dkv, part = ecm.gate_hc_bwd(g, x, kv, wf, *st, clamp=wl.clamp, P=P)
        if op.startswith("gate_hc_bwd"):
            nbytes = T * ((5 * hc + 2) * 2 * d + 16 * hc) + P * hc * d * 4

            def launch():
                ecm.gate_hc_bwd(g, x, kv, wf, *st, clamp=wl.clamp, P=P, dx=dx, dkv=dkv, dw_partial=part)
        else:
            nbytes = T * ((3 * hc + 1) * 2 * d + 16 * hc)

            def launch():
                ecm.gate_hc_fwd(x, kv, wf, wl.eps, wl.clamp, out=out, stats=st)
    elif op.startswith("short_conv"):
        # the short conv after the gate's micro-batch: 4 x 4096 tokens, d = 4096 bf16, width 4, dilation 3
        cw = W.short_conv_4x4k()
        T, d = cw.T, cw.d
        v = SD.normal_tensor((T, d), cw.seed + 1, 0.0, 0.5, "bf16", device)
        h = SD.normal_tensor((T, d), cw.seed + 2, 0.0, 1.0, "bf16", device)
        g = SD.normal_tensor((T, d), cw.seed + 3, 0.0, 1.0, "bf16", device)
        nw = SD.normal_tensor((1, d), cw.seed + 4, 1.0, 0.1, "f32", device).reshape(-1)
        cwt = SD.normal_tensor((d, cw.width), cw.seed + 5, 0.0, 0.5, "f32", device)
        bias = SD.normal_tensor((1, d), cw.seed + 6, 0.0, 0.1, "f32", device).reshape(-1)
        offs = torch.arange(0, T + 1, 4096, dtype=torch.int64, device=device)
        out, rstd = ecm.short_conv_fwd(v, nw, cwt, offs, cw.dilation, h=h, bias=bias)
        dv, part = ecm.short_conv_bwd(g, v, nw, cwt, rstd, offs, cw.dilation, bias=bias)
        red = ecm.short_conv_grad_reduce(part, cw.width, d)
        P = part.shape[0]
        if op == "short_conv_fwd":  # the op's own bytes: V~ and H read, out written, rstd written
            nbytes = 3 * T * d * 2 + 4 * T

            def launch():
                ecm.short_conv_fwd(v, nw, cwt, offs, cw.dilation, h=h, bias=bias, out=out, rstd=rstd)
        elif op == "short_conv_fwd_given":  # the same with rstd given (made by the gate): rstd read
            nbytes = 3 * T * d * 2 + 4 * T

            def launch():
                ecm.short_conv_fwd(v, nw, cwt, offs, cw.dilation, h=h, bias=bias, out=out, given_rstd=rstd)
        elif op == "short_conv_bwd":  # dout, V~, rstd read; dv and the partials written
            nbytes = 3 * T * d * 2 + 4 * T + P * (cw.width + 2) * d * 4

            def launch():
                ecm.short_conv_bwd(g, v, nw, cwt, rstd, offs, cw.dilation, bias=bias, dv=dv, dw_partial=part)
        else:
            nbytes = P * (cw.width + 2) * d * 4 + (cw.width + 2) * d * 4

            def launch():
                ecm.short_conv_grad_reduce(part, cw.width, d, out=red)
    elif op.startswith("sinkhorn"):
        # the Engram Sinkhorn on 16384 x 5120 fp32 (bf16 gradient): 335 MB per matrix, > L2
        sw = W.sinkhorn_16k_x_5120()
        R, D = sw.rows, sw.head_dim
        grad = SD.normal_tensor((R, D), sw.seed + 1, 0.0, 1.0, "bf16", device)
        mom = SD.normal_tensor((R, D), sw.seed + 2, 0.0, 0.5, "f32", device)
        rs = torch.ones(R, dtype=torch.float32, device=device)
        cs = torch.ones(D, dtype=torch.float32, device=device)
        inp = ecm.sinkhorn_momentum_update(grad, mom, sw.beta1, sw.nesterov)
        P = ecm.sinkhorn_num_partials(R, D)
        nrm, part = ecm.sinkhorn_step(inp, rs, cs, sw.eps, P=P)
        csum = ecm.sinkhorn_step_reduce(part, col_scale=cs, eps=sw.eps)
        out = ecm.sinkhorn_finalize(inp, rs, cs, sw.eps, math.sqrt(D))
        b_mom = R * D * (2 + 4 + 4 + 4)
        b_step = R * D * 4 + R * 12 + D * 4 + P * D * 4
        b_red = P * D * 4 + 3 * D * 4
        b_fin = 2 * R * D * 4 + R * 4 + D * 4
        fns = {
            "sinkhorn_momentum": (b_mom, lambda: ecm.sinkhorn_momentum_update(grad, mom, sw.beta1, sw.nesterov,
                                                                               sinkhorn_input=inp)),
            "sinkhorn_step": (b_step, lambda: ecm.sinkhorn_step(inp, rs, cs, sw.eps, P=P, row_norm=nrm,
                                                                col_sumsq_partial=part)),
            "sinkhorn_reduce": (b_red, lambda: ecm.sinkhorn_step_reduce(part, col_sumsq=csum, col_scale=cs,
                                                                        eps=sw.eps)),
            "sinkhorn_finalize": (b_fin, lambda: ecm.sinkhorn_finalize(inp, rs, cs, sw.eps, math.sqrt(D), out=out)),
        }
        if op == "sinkhorn":  # one optimizer pass: momentum, one row + column step, finalize
            nbytes = b_mom + b_step + b_red + b_fin

            def launch():
                for k in ("sinkhorn_momentum", "sinkhorn_step", "sinkhorn_reduce", "sinkhorn_finalize"):
                    fns[k][1]()
        else:
            nbytes, launch = fns[op]
    elif op.startswith("gate_conv"):
        # the gate's forward and the short conv after it, T = 16384, d = 4096 bf16: with the conv's own
        # statistic pass (gate_conv_fwd) or with the statistic made by the gate (gate_conv_fwd_fused)
        wl, cw = W.gate_train_4k(), W.short_conv_4x4k()
        t = SD.gate_device_inputs(wl, device)
        T, d = wl.T, wl.d
        wf = ecm.fuse_weight(t["w_h"], t["w_k"])
        h = SD.normal_tensor((T, d), cw.seed + 2, 0.0, 1.0, "bf16", device)
        nw = SD.normal_tensor((1, d), cw.seed + 4, 1.0, 0.1, "f32", device).reshape(-1)
        cwt = SD.normal_tensor((d, cw.width), cw.seed + 5, 0.0, 0.5, "f32", device)
        bias = SD.normal_tensor((1, d), cw.seed + 6, 0.0, 0.1, "f32", device).reshape(-1)
        offs = torch.arange(0, T + 1, 4096, dtype=torch.int64, device=device)
        vt, *st = ecm.gate_fwd(t["h"], t["k"], t["v"], wf, EPS)
        _, *_, vstat = ecm.gate_fwd_rms(t["h"], t["k"], t["v"], wf, EPS, out_eps=cw.eps, stats=st)
        out, rstd = ecm.short_conv_fwd(vt, nw, cwt, offs, cw.dilation, h=h, bias=bias, eps=cw.eps)
        nbytes = T * (8 * d + 16) + 3 * T * d * 2 + 4 * T  # the two ops' own bytes

        if op == "gate_conv_fwd_fused":
            def launch():
                ecm.gate_fwd_rms(t["h"], t["k"], t["v"], wf, EPS, out_eps=cw.eps, out=vt, stats=st, out_rstd=vstat)
                ecm.short_conv_fwd(vt, nw, cwt, offs, cw.dilation, h=h, bias=bias, out=out, given_rstd=vstat)
        else:
            def launch():
                ecm.gate_fwd(t["h"], t["k"], t["v"], wf, EPS, out=vt, stats=st)
                ecm.short_conv_fwd(vt, nw, cwt, offs, cw.dilation, h=h, bias=bias, eps=cw.eps, out=out, rstd=rstd)
    else:
        # gate_fwd_2k: T=8192 d=2048; gate_fwd_7k / gate_bwd_7k: T=131072 d=7168; otherwise T=16384 d=4096
        wl = {"gate_fwd_2k": W.gate_fwd_2k(), "gate_fwd_7k": W.gate_sweep_7k(131072),
              "gate_bwd_7k": W.gate_sweep_7k(131072)}.get(op, W.gate_train_4k())
        t = SD.gate_device_inputs(wl, device)
        wf = ecm.fuse_weight(t["w_h"], t["w_k"])
        out, *st = ecm.gate_fwd(t["h"], t["k"], t["v"], wf, EPS)
        P = ecm.gate_bwd_num_partials(wl.T, wl.d)
        dh, dk, dv, part = ecm.gate_bwd(t["dout"], t["h"], t["k"], t["v"], wf, *st, P=P)
        if op in ("gate_bwd", "gate_bwd_7k"):
            nbytes = wl.T * (14 * wl.d + 16) + P * wl.d * 4

            def launch():
                ecm.gate_bwd(t["dout"], t["h"], t["k"], t["v"], wf, *st, P=P, dh=dh, dk=dk, dv=dv, dw_partial=part)
        elif op == "gate_bwd_accumulate":  # the step's later backwards: partials read back and added to
            nbytes = wl.T * (14 * wl.d + 16) + 2 * P * wl.d * 4

            def launch():
                ecm.gate_bwd(t["dout"], t["h"], t["k"], t["v"], wf, *st, P=P, dh=dh, dk=dk, dv=dv, dw_partial=part,
                             accumulate=True)
        elif op == "grad_w_reduce":  # the step's launch: the accumulated partials, both weight gradients
            gh, gk = torch.zeros_like(t["w_h"]), torch.zeros_like(t["w_k"])
            nbytes = P * wl.d * 4 + 7 * wl.d * 4

            def launch():
                ecm.grad_w_reduce(part, dweight_fused=wf, w_h=t["w_h"], w_k=t["w_k"], grad_w_h=gh, grad_w_k=gk)
        else:  # gate_fwd on T=16384 d=4096, gate_fwd_2k on T=8192 d=2048, gate_fwd_7k on T=131072 d=7168
            nbytes = wl.T * (8 * wl.d + 16)

            def launch():
                ecm.gate_fwd(t["h"], t["k"], t["v"], wf, EPS, out=out, stats=st)
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()

    def timed(run_one):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        ev[0].record(stream)
        for i in range(args.steps):
            run_one()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]

    eager = timed(launch)
    # the same launches replayed from a CUDA graph: no host work between them (pointer checks were
    # made by the eager launches on the same buffers); eager timing stands where capture is refused
    graph_times = None
    if op != "hash_gather_host":
        graph = torch.cuda.CUDAGraph()
        prev = ecm.set_validation(0)
        try:
            with torch.cuda.graph(graph):
                launch()
        except RuntimeError:
            graph = None
        finally:
            ecm.set_validation(prev)
        if graph is not None:
            for _ in range(args.warmup):
                graph.replay()
            graph_times = timed(graph.replay)
    times = graph_times or eager
    peak, kind = load_peaks()
    med = statistics.median(times)
    gbs = nbytes / (med / 1e3) / 1e9
    return {"only": op, "median_ms": med, "min_ms": min(times), "eager_median_ms": statistics.median(eager),
            "timing": "graph" if graph_times else "eager", "bytes": nbytes, "GBps": gbs, "frac": gbs / peak,
            "peak": peak, "peak_kind": kind, "launches": args.steps}


def main_only(args, device):
    print(json.dumps(time_only(args.only, args.steps, args.warmup, device)), flush=True)
    return 0


# The NEXT rows' own workloads, timed in the default run: the multi-branch gate (whole token at d = 4096,
# clusters at d = 7168), the short convolution after the gate, the Engram Sinkhorn and the gather from a
# host-resident table.  Whether consecutive launches find their inputs in L2: the reductions' (19-21 MB)
# do, every other workload here is far larger than the 129 MB L2.
NEXT_OPS = [
    ("gate_hc_fwd", "hc=4 T=8192 d=4096 bf16, whole token per CTA", False),
    ("gate_hc_bwd", "hc=4 T=8192 d=4096 bf16, whole token per CTA", False),
    ("gate_hc_fwd_d7168", "hc=4 T=4096 d=7168 bf16, clusters of 2 CTAs", False),
    ("gate_hc_bwd_d7168", "hc=4 T=4096 d=7168 bf16, clusters of 4 CTAs", False),
    ("short_conv_fwd", "4x4096 tokens d=4096 bf16 width 4 dilation 3, rstd pass + sweep", False),
    ("short_conv_fwd_given", "the same with rstd made by the gate (the sweep alone)", False),
    ("gate_conv_fwd_fused", "gate_fwd_rms then short_conv_fwd_given, T=16384 d=4096", False),
    ("short_conv_bwd", "4x4096 tokens d=4096 bf16, one pass on clusters of 8", False),
    ("short_conv_reduce", "P=192 partials of (width+2) x 4096", True),
    ("sinkhorn", "16384 x 5120 fp32: momentum + row step + reduce + finalize", False),
    ("sinkhorn_momentum", "16384 x 5120, bf16 gradient, Nesterov", False),
    ("sinkhorn_step", "16384 x 5120, P=1024", False),
    ("sinkhorn_reduce", "P=1024 x 5120 + column step", True),
    ("sinkhorn_finalize", "16384 x 5120", False),
    ("hash_gather_host", "the 65,536-token gather from the 4.1 GB table in pinned host memory", False),
]


def time_next_rows(device, steps: int, warmup: int) -> dict:
    import torch

    out = {}
    for op, what, l2_resident in NEXT_OPS:
        r = time_only(op, steps, warmup, device)
        out[op] = {"workload": what, "median_us": r["median_ms"] * 1e3, "bytes": r["bytes"], "GBps": r["GBps"],
                   "frac": r["frac"], "timing": r["timing"], "launches": r["launches"],
                   "inputs_in_l2_between_launches": l2_resident}
        if op == "hash_gather_host":  # bound by the host link, not HBM: the rows cross it once
            link = SEQS * SEQ_LEN * 16 * 128
            out[op].update(bound="host link", link_bytes=link, link_GBps=link / (r["median_ms"] / 1e3) / 1e9,
                           frac_note="frac is against the HBM peak; the rows cross the host link at link_GBps")
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- table offload

def main_offload(args, device):
    """The step with its tables in host memory: the hash + gather of the next batch (its rows follow
    from the ids alone, so it can run ahead) reads the page-locked host table on a side stream, with
    a few CTAs, while this step's gate work runs; versus the step with the table in HBM."""
    import torch

    import engram_conditional_memory_gb300 as ecm

    wk = make_workload(device)
    host_table = wk["table"].cpu().pin_memory()
    hw = wk["hw"]
    comp = torch.cuda.current_stream()
    side = torch.cuda.Stream(device)
    rows_next = torch.empty_like(wk["rows"])
    fetched = torch.cuda.Event()

    def gate_part():
        for i, m in enumerate(wk["mb"]):
            st = wk["stats"][i]
            gate_forward(wk, i)
            ecm.gate_bwd(m["dout"], m["h"], m["k"], m["v"], wk["w_fused"], *st, P=wk["P"], dh=wk["dh"][i],
                         dk=wk["dk"][i], dv=wk["dv"][i], dw_partial=wk["part"], accumulate=i > 0)
        reduce_step(wk)

    def offload_step():
        side.wait_event(fetched)  # rows_next is free once the previous step's prefetch was consumed
        with torch.cuda.stream(side):
            prev = ecm.set_max_ctas(args.offload_ctas)
            ecm.hash_gather(wk["spec"], wk["ids"], wk["offs"], host_table, wk["cmap"], hw.vocab, hw.vocab_c,
                            out_rows=rows_next)
            ecm.set_max_ctas(prev)
        gate_part()
        comp.wait_stream(side)  # the next step's rows are in HBM by the end of this step
        fetched.record(comp)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        side.wait_event(a)
        for _ in range(args.steps):
            fn()
        b.record(comp)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    dev_ms = timed(lambda: run_step(wk))
    off_ms = timed(offload_step)
    host_alone = timed(lambda: ecm.hash_gather(wk["spec"], wk["ids"], wk["offs"], host_table, wk["cmap"], hw.vocab,
                                               hw.vocab_c, out_rows=rows_next))
    # the prefetched rows equal the ones gathered from HBM
    ecm.hash_gather(wk["spec"], wk["ids"], wk["offs"], host_table, wk["cmap"], hw.vocab, hw.vocab_c, out_rows=rows_next)
    run_step(wk)
    torch.cuda.synchronize()
    same = bool(torch.equal(rows_next, wk["rows"]))
    print(json.dumps({"offload": {"step_ms_table_in_hbm": dev_ms, "step_ms_table_in_host_memory": off_ms,
                                  "overhead": off_ms / dev_ms - 1.0, "host_gather_alone_ms": host_alone,
                                  "offload_ctas": args.offload_ctas, "rows_identical": same,
                                  "workload": WORKLOAD}}), flush=True)
    return 0


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end timing (profiling runs)")
    ap.add_argument("--cpu-steps", type=int, default=3, help="whole oracle steps timed for cpu_baseline")
    ap.add_argument("--no-configs", action="store_true", help="skip the gate-only workloads (profiling runs)")
    ap.add_argument("--no-next", action="store_true", help="skip the NEXT rows' workloads (profiling runs)")
    ap.add_argument("--offload", action="store_true",
                    help="the step with the tables in host memory, prefetched on a side stream (vs in HBM)")
    ap.add_argument("--offload-ctas", type=int, default=32, help="CTAs of the host-table gather in --offload")
    ap.add_argument("--only", choices=["hash_gather", "hash_gather_small", "hash_gather_host", "gate_fwd",
                                       "gate_fwd_2k", "gate_fwd_7k", "gate_bwd", "gate_bwd_7k",
                                       "gate_bwd_accumulate", "grad_w_reduce",
                                       "gate_hc_fwd", "gate_hc_bwd",
                                       "sinkhorn", "sinkhorn_momentum", "sinkhorn_step", "sinkhorn_reduce",
                                       "sinkhorn_finalize", "short_conv_fwd", "short_conv_fwd_given", "short_conv_bwd",
                                       "short_conv_reduce", "gate_conv_fwd", "gate_conv_fwd_fused", "gate_hc_fwd_d7168",
                                       "gate_hc_bwd_d7168"],
                    help="time one kernel alone on its workload (consecutive launches, L2 not flushed)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, local, world = dist_env()
    if args.impl == "reference":
        return main_reference(args, rank, world)
    return main_native(args, rank, local, world)


def main_reference(args, rank, world):
    """The CPU oracle on the host cores, one whole step of the workload per timed step; rank 0 alone
    works and prints under torchrun."""
    if rank != 0:
        return 0
    from synth import workloads as W

    hw = W.hash_gather_64k(num_seqs=SEQS, seq_len=SEQ_LEN)
    table_host, mbs, w_h, w_k = oracle_inputs_on_host(hw)
    times, threads = time_oracle_steps(hw, table_host, mbs, w_h, w_k, args.steps, args.warmup)
    T_all = hw.T
    mean_s = sum(times) / len(times)
    value = T_all / mean_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": T_all, "parallelism": "replicas",
                   "inputs": "drawn on the host (torch CPU generator, same seeds and recipe as the device draws)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": oracle_sample_text(args.steps, threads),
                         "step_ms_min": min(times) * 1e3, "step_ms_max": max(times) * 1e3},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main_native(args, rank, local, world):
    import torch
    import torch.distributed as dist

    import engram_conditional_memory_gb300 as ecm

    if not torch.cuda.is_available():
        print("bench.py: no CUDA device", file=sys.stderr)
        return 2
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=device)
    ecm.load_library()
    if args.only:
        return main_only(args, device)
    if args.offload:
        return main_offload(args, device)
    wk = make_workload(device)
    props = torch.cuda.get_device_properties(device)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local)
    graph = capture_step(wk, device)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    elapsed, launches, w0, w1 = time_graph(graph, args.steps, args.warmup, device)
    clocks = sampler.stop(w0, w1)
    max_ms = aggregate_max(elapsed, device)
    _, per, _, _, _ = time_device(wk, args.steps, args.warmup, device)
    T_all = wk["hw"].T
    value = world * T_all * args.steps / (max_ms / 1e3)
    peak, peak_kind = load_peaks()
    ab = algorithmic_bytes(wk["P"])
    ops = {}
    tokens_per_launch = {"hash_gather": T_all, "gate_fwd_fold": MICRO_T, "gate_fwd": MICRO_T, "gate_bwd": MICRO_T,
                         "gate_bwd_accumulate": MICRO_T}
    for name, times in per.items():
        avg = sum(times) / len(times)
        gbs = ab[name] / (avg / 1e3) / 1e9
        ops[name] = {"avg_ms": avg, "launches": len(times), "bytes": ab[name], "GBps": gbs, "frac": gbs / peak}
        if name in tokens_per_launch:
            ops[name]["tokens_per_s"] = tokens_per_launch[name] / (avg / 1e3)
    step_bytes = (ab["hash_gather"] + ab["gate_fwd_fold"] + 3 * ab["gate_fwd"] + ab["gate_bwd"]
                  + 3 * ab["gate_bwd_accumulate"] + ab["grad_w_reduce"])
    dom = "gate_bwd_accumulate"  # three of the four backward launches
    roof = {"bound": "hbm", "kernel": dom, "achieved": ops[dom]["GBps"], "peak": peak, "unit": "GB/s",
            "frac": ops[dom]["GBps"] / peak, "peak_kind": f"{peak_kind} (copy bandwidth)",
            "traffic": load_traffic(dom), "algorithmic_bytes_per_launch": ab[dom]}
    e2e = None
    if not args.no_e2e:
        e_ms, h2d, d2h = time_e2e(wk, args.steps, args.warmup, device)
        e_max = aggregate_max(e_ms, device)
        e2e = {"value": world * T_all * args.steps / (e_max / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    # per-GPU measurements of the gate's and the NEXT rows' own workloads: at N = 1 only (each replica
    # would repeat them), after the timed step
    configs = None if args.no_configs or world > 1 else time_gate_configs(
        device, args.steps, args.warmup, peak, with_oracle=rank == 0 and not args.no_cpu_baseline)
    next_rows = None if args.no_next or world > 1 else time_next_rows(device, args.steps, args.warmup)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        table_host, mbs, w_h, w_k = oracle_inputs_from_device(wk)
        times, threads = time_oracle_steps(wk["hw"], table_host, mbs, w_h, w_k, args.cpu_steps, 1)
        hash_rates = oracle_hash_rates(wk["hw"], table_host)
        del table_host, mbs
        mean_s = sum(times) / len(times)
        cpu = {"value": T_all / mean_s, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": oracle_sample_text(args.cpu_steps, threads) + "; inputs copied from the device",
               "step_ms_mean": mean_s * 1e3, "step_ms_min": min(times) * 1e3,
               "hash_gather_64k": hash_rates}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "math": "fp32 accumulate; uint64 hash",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step": T_all, "global_batch": world * T_all,
                       "seq_len": SEQ_LEN, "parallelism": f"replicas x{world}",
                       "l2": "no flush: per-step working set 6.1 GB >> 129 MB L2",
                       "timing": "value: CUDA-graph replays of the 10-launch step, the hash + gather on a branch "
                                 "beside the gate work; ops/roofline: eager serial steps "
                                 "with an event between launches; e2e: eager calls with host copies"},
            "hbm_gbs": step_bytes / (max_ms / args.steps / 1e3) / 1e9,
            "hash_gather_rows_per_s": 16 * T_all / (ops["hash_gather"]["avg_ms"] / 1e3),
            "roofline": roof, "ops": ops, "configs": configs, "next_rows": next_rows, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
