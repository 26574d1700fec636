#!/usr/bin/env python3
"""Benchmark of the SSD layer forward scan on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one full forward (every kernel of the chunked scan) over one batch of
the workload.  ``value`` is tokens/s (batch*seqlen per step) with inputs already
resident in HBM; ``e2e`` is the same metric through the host-buffer entry point
(ssd_fwd_host) with the input copies in and the output copies out inside the
timed region.  Inputs rotate over several device copies whose total exceeds the
126 MB L2, so every step reads cold data.

With N > 1 (torchrun) every rank runs its own copy of the workload on its own
GPU (the batch dimension shards with no exchange: weak scaling); rank 0 prints
the line with the max-over-ranks time.  ``--impl reference`` times the fp64
CPU oracle instead (on the host cores, bounded samples of the same workload).

The headline line also carries sub-records measured after the timed region:
the single-token decode step, the forward with the dt pre-step, packed
variable-length sequences, the backward (ssd_bwd) on the same workload, and
the other large workloads.
"""
from __future__ import annotations

import argparse
import dataclasses
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from structured_state_space_03_b300 import workloads as wl  # noqa: E402

METRIC = "SSD fwd tokens/s (batch·seqlen/s) at 1 B300; % of HBM/tensor roofline"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: enough for ~3 s)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.HEADLINE.name, choices=[w.name for w in wl.WORKLOADS])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the sub-record of the other large workloads (headline run only)")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward sub-record (headline run only)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip every sub-record (decode, pre-step, packed, backward, other workloads)")
    ap.add_argument("--seqlen", type=int, default=0,
                    help="run the named workload at this sequence length instead (a scaled-down case for "
                         "profilers; the record's workload name gains the new length)")
    ap.add_argument("--ref-seconds", type=float, default=0.0,
                    help="oracle seconds per step of --impl reference (0: spread ~150 s over the steps)")
    return ap.parse_args()


# -- environment ------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's `value` (a no-op with one rank): the job's
    time is its slowest rank's."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest(kernel=None):
    """Digest of the device sources: the headers and every translation unit that
    defines a kernel (host-only files such as the C-ABI entry points are left out).
    With `kernel`, only the headers and the file that defines that kernel, so a
    change to another kernel's file does not retire its recorded counters."""
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "structured_state_space_03_b300", "csrc", "*"))):
        with open(f, "rb") as fh:
            data = fh.read()
        if f.endswith(".cuh") or (b"__global__" in data and (kernel is None or kernel.encode() in data)):
            h.update(os.path.basename(f).encode() + data)
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summaries, if they were taken on the current sources of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    ent = rec.get(f"{kernel}@{workload}")
    if not ent or ent.get("source_digest") != source_digest(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of the SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.rows = []
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            target = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={target}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, RuntimeError, AttributeError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def mark(self):
        return len(self.rows)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, start, end):
        rows = self.rows[start:end] or self.rows[-3:]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# -- workload bookkeeping ---------------------------------------------------------------

def unavoidable_bytes(w):
    """x, y, dt, B, C, A, D and the states that cross HBM once per step."""
    e = 2 if w.dtype == "bf16" else 4
    tok = w.batch * w.seqlen
    xy = 2 * tok * w.nheads * w.headdim * e
    bc = 2 * tok * w.ngroups * w.dstate * e
    dt = tok * w.nheads * 4
    states = w.batch * w.nheads * w.headdim * w.dstate * 4 * (2 if w.with_init else 1)
    return xy + bc + dt + states + 2 * w.nheads * 4


def causal_flops(w):
    """Algorithmic tensor-core FLOPs of the chunked scan (upper triangle excluded):
    per (batch, chunk): G*N*Q(Q+1) + H*[P*Q(Q+1) + 4*Q*N*P]; the last chunk is partial."""
    total = 0
    for c in range(math.ceil(w.seqlen / w.chunk)):
        q = min(w.chunk, w.seqlen - c * w.chunk)
        total += w.ngroups * w.dstate * q * (q + 1) + w.nheads * (w.headdim * q * (q + 1)
                                                                   + 4 * q * w.dstate * w.headdim)
    return total * w.batch


def kernel_algorithmic_bytes(w, name):
    """Bytes a kernel must move to do its own share of the step, counting the
    workspace states it exchanges with the other kernels (fp32)."""
    e = 2 if w.dtype == "bf16" else 4
    tok = w.batch * w.seqlen
    x = tok * w.nheads * w.headdim * e
    bc = tok * w.ngroups * w.dstate * e
    dt = tok * w.nheads * 4
    nc = math.ceil(w.seqlen / w.chunk)
    st = w.batch * w.nheads * nc * w.headdim * w.dstate * 4
    fin = w.batch * w.nheads * w.headdim * w.dstate * 4
    if name.startswith("chunk_state"):
        return x + bc + dt + st
    if name.startswith("state_pass"):
        return 2 * st + fin * (2 if w.with_init else 1)
    if name.startswith("chunk_out"):
        return x + 2 * bc + dt + st + x
    if name.startswith("ssd_fused") or name.startswith("chunk_scan"):
        return unavoidable_bytes(w)
    return unavoidable_bytes(w)


# -- the CPU oracle (baseline leg and reference arm) ------------------------------------

def decode_step_measurement(dev, peaks, stream, batch=64, steps=400):
    """The recurrent single-token step (ssd_step) on the 2.7B-shaped heads at a
    serving batch: 80 heads x headdim 64, dstate 64, 1 group, bf16.  Two state
    sets (2 x 84 MB) alternate so every step's state traffic goes to HBM."""
    import structured_state_space_03_b300 as ssd
    H, P, N, G = 80, 64, 64, 1
    gen = torch.Generator(device="cpu").manual_seed(777)
    mk = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16).to(dev)
    x, B, C = mk(batch, H, P), mk(batch, G, N), mk(batch, G, N)
    dt = (torch.rand(batch, H, generator=gen) * 0.099 + 0.001).to(dev)
    A = -torch.exp(torch.rand(H, generator=gen) * math.log(16.0)).to(dev)
    D = torch.randn(H, generator=gen).to(dev)
    states = [(torch.randn(batch, H, P, N, generator=gen) * 0.1).to(dev) for _ in range(2)]
    y = torch.empty_like(x)
    for k in range(10):
        ssd.ssd_step(x, dt, A, B, C, D, state=states[k % 2], y=y, stream=stream)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for k in range(steps):
        ssd.ssd_step(x, dt, A, B, C, D, state=states[k % 2], y=y, stream=stream)
    e.record(stream)
    torch.cuda.synchronize()
    ssd.ssd_check_device_status(stream)
    us = s.elapsed_time(e) / steps * 1e3
    nbytes = 2 * batch * H * P * N * 4 + 2 * batch * H * P * 2 + 2 * batch * G * N * 2 + batch * H * 4 + 2 * H * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"workload": f"decode_b{batch}_H{H}_P{P}_N{N}_G{G}", "us_per_step": us,
            "tokens_per_s": batch / (us * 1e-6), "bytes_per_step": nbytes, "achieved_gbs": gbs,
            "peak_gbs": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"], "kernel": "ssd_step_vec_kernel",
            "l2": "two state sets of 84 MB alternate (> 126 MB L2)"}


def pre_step_measurement(sets, w, stream, steps=100):
    """The headline forward through ssd_fwd_pre (softplus of dt + bias and the
    zero-order-hold input scale, applied on the device) against ssd_fwd on the
    same inputs; both allocate their workspace per call the same way."""
    import structured_state_space_03_b300 as ssd
    dev = sets[0]["x"].device
    # softplus(dt + bias) with bias = log(expm1(0.01)): steps of about 0.01 to 0.11,
    # the dt scale of the workload itself
    bias = torch.full((w.nheads,), math.log(math.expm1(0.01)), device=dev)

    def timed(fn):
        for k in range(5):
            fn(k)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for k in range(steps):
            fn(k)
        e.record(stream)
        torch.cuda.synchronize()
        ssd.ssd_check_device_status(stream)
        return s.elapsed_time(e) / steps * 1e3

    def plain(k):
        d = sets[k % len(sets)]
        ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk=w.chunk, y=d["y"],
                    final_state=d["final"], stream=stream)

    def pre(k):
        d = sets[k % len(sets)]
        ssd.ssd_fwd_pre(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk=w.chunk,
                        dt_bias=bias, softplus=True, zoh=True, y=d["y"], final_state=d["final"], stream=stream)

    t_plain, t_pre = timed(plain), timed(pre)
    return {"workload": w.name, "modes": "softplus(dt + bias), bias = log(expm1(0.01)); zero-order hold",
            "us_per_step_ssd_fwd": t_plain,
            "us_per_step_ssd_fwd_pre": t_pre, "overhead_us": t_pre - t_plain,
            "tokens_per_s": w.tokens / (t_pre * 1e-6),
            "kernels": ["pre_kernel"] + ssd.ssd_fwd_kernels(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate,
                                                            w.chunk, wl.torch_dtype(w.dtype))}


def varlen_step_measurement(sets, w, stream, peaks, steps=100, nseq=12, seed=5):
    """Packed variable-length sequences (ssd_fwd_varlen): the headline's
    batch x seqlen tokens repacked as nseq sequences of seeded mixed lengths
    (log-uniform over a 64x range), on the same heads, against ssd_fwd on the
    batch layout of the same tokens.  Both allocate their workspace per call;
    the packed call also builds and uploads its chunk table."""
    import structured_state_space_03_b300 as ssd
    total = w.batch * w.seqlen
    lengths = wl.varlen_lengths(total, nseq, seed)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    packed = [{k: d[k].reshape(total, *d[k].shape[2:]) for k in ("x", "dt", "B", "C", "y")} for d in sets]

    def timed(fn):
        for k in range(5):
            fn(k)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for k in range(steps):
            fn(k)
        e.record(stream)
        torch.cuda.synchronize()
        ssd.ssd_check_device_status(stream)
        return s.elapsed_time(e) / steps * 1e3

    def batch(k):
        d = sets[k % len(sets)]
        ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], None, chunk=w.chunk, y=d["y"],
                    return_final=False, stream=stream)

    def varlen(k):
        d, q = sets[k % len(sets)], packed[k % len(sets)]
        ssd.ssd_fwd_varlen(q["x"], q["dt"], d["A"], q["B"], q["C"], d["D"], None, cu_seqlens=cu, chunk=w.chunk,
                           y=q["y"], return_final=False, stream=stream)

    t_batch, t_var = timed(batch), timed(varlen)
    nbytes = unavoidable_bytes(w) - w.batch * w.nheads * w.headdim * w.dstate * 4  # no states in or out
    return {"tokens": total, "sequences": nseq, "lengths": lengths, "chunk": w.chunk,
            "heads": f"{w.nheads} x {w.headdim}, dstate {w.dstate}, {w.ngroups} group(s), {w.dtype}",
            "us_per_step_ssd_fwd_varlen": t_var, "us_per_step_ssd_fwd_batch": t_batch,
            "tokens_per_s": total / (t_var * 1e-6), "algorithmic_bytes": nbytes,
            "frac_of_hbm": nbytes / (t_var * 1e-6) / (peaks["hbm_gbs"] * 1e9),
            "kernels": ["ssd_fused_pipe_tc"]}


def plan_oracle_rows(w, inp, cores, seconds_per_call):
    """The (batch, head, headdim) rows one timed oracle call covers: every row
    when they fit in ``seconds_per_call`` on ``cores`` threads, else a seeded
    subset sized from a short calibration call (a multiple of ``cores``)."""
    import oracle
    total = w.batch * w.nheads * w.headdim
    order = torch.randperm(total, generator=torch.Generator().manual_seed(3)).tolist()
    probe = order[:min(total, 2 * cores)]
    t0 = time.perf_counter()
    oracle.recurrence(**inp, rows=probe, nthreads=cores)
    per_row = (time.perf_counter() - t0) / len(probe) * cores  # thread-seconds per row
    fit = int(seconds_per_call * cores / max(per_row, 1e-9))
    n = total if fit >= total else max(cores, fit // cores * cores)
    return sorted(order[:n])


def oracle_rate(w, inp, rows, cores):
    """One timed oracle call over ``rows``: tokens/s, scaled by the row fraction."""
    import oracle
    t0 = time.perf_counter()
    oracle.recurrence(**inp, rows=rows, nthreads=cores)
    el = time.perf_counter() - t0
    return w.batch * w.seqlen * len(rows) / (w.batch * w.nheads * w.headdim) / el, el


def oracle_sample_text(w, rows, calls, per_call_s):
    total = w.batch * w.nheads * w.headdim
    what = "every" if len(rows) == total else f"a seeded subset of {len(rows)} of the {total}"
    return (f"the sequential fp64 recurrence over {what} (batch, head, headdim) rows for the full sequence, "
            f"one threaded call per sample, median of {calls} calls (~{per_call_s:.2f} s each); "
            f"tokens/s scaled by the row fraction")


def cpu_baseline(w, inp, seconds):
    """The oracle timed on the host cores: the same rows and method as the
    reference arm, repeated for ``seconds``; the median call."""
    cores = len(os.sched_getaffinity(0))
    rows = plan_oracle_rows(w, inp, cores, min(seconds, 3.0))
    vals, secs = [], 0.0
    while secs < seconds or len(vals) < 3:
        v, el = oracle_rate(w, inp, rows, cores)
        vals.append(v)
        secs += el
    value = statistics.median(vals)
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": oracle_sample_text(w, rows, len(vals), secs / len(vals))}


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    inp = wl.workload_inputs(w)
    cores = len(os.sched_getaffinity(0))
    steps = args.steps or 5
    per_step = args.ref_seconds or max(0.5, min(3.0, 150.0 / max(1, steps + args.warmup)))
    rows = plan_oracle_rows(w, inp, cores, per_step)
    for _ in range(args.warmup):
        oracle_rate(w, inp, rows, cores)
    vals, secs = [], 0.0
    for _ in range(steps):
        v, el = oracle_rate(w, inp, rows, cores)
        vals.append(v)
        secs += el
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": oracle_sample_text(w, rows, steps, secs / steps)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w):
    """The workload as both arms name it."""
    return {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
            "dstate": w.dstate, "ngroups": w.ngroups, "chunk": w.chunk}


# -- the GPU arm ------------------------------------------------------------------------

def device_sets(w, inp, dev):
    """Device copies of one input set, enough that the steps rotating over them
    read more than three times the L2 between two uses of one copy."""
    per_set = unavoidable_bytes(w)
    nsets = max(2, math.ceil(3 * L2_BYTES / per_set))
    sets = []
    for _ in range(nsets):
        d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        d["y"] = torch.empty_like(d["x"])
        d["final"] = torch.empty(w.batch, w.nheads, w.headdim, w.dstate, dtype=torch.float32, device=dev)
        sets.append(d)
    return sets, per_set


def make_step(w, sets, ws):
    import structured_state_space_03_b300 as ssd

    def step(k, stream):
        d = sets[k % len(sets)]
        ssd.ssd_fwd_ws(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], chunk=w.chunk,
                       workspace=ws, y=d["y"], final_state=d["final"], stream=stream)
    return step


def capture(step, first, count):
    """A CUDA graph of ``count`` consecutive steps (rotation index from ``first``)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for k in range(first, first + count):
            step(k, cs)
    return g


def graph_plan(steps, max_nodes=200):
    """Graphs replayed in the timed region: (steps per graph, replays) pairs
    covering exactly ``steps`` steps."""
    per = min(steps, max_nodes)
    plan = [(per, steps // per)]
    if steps % per:
        plan.append((steps % per, 1))
    return plan


def per_kernel_times(step, nk, stream, count):
    """Device time of each kernel of a step, from events the library records
    right around each launch: ``count`` profiled steps captured in a CUDA graph
    and replayed (untimed otherwise), so host-side launch work does not sit
    between an event and its kernel.  Returns (ms per launch per kernel, how)."""
    import structured_state_space_03_b300 as ssd
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)] for _ in range(count)]
    for row in evs:  # create the underlying CUDA events
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    how = "event pairs around each launch, in a CUDA graph of the profiled steps"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for k in range(count):
                ssd.ssd_profile_events(evs[k])
                step(k, cs)
                ssd.ssd_profile_events(None)
        g.replay()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        out = [0.0] * nk
        for row in evs:
            for i in range(nk):
                out[i] += row[2 * i].elapsed_time(row[2 * i + 1])
        del g
    except RuntimeError:
        ssd.ssd_profile_events(None)
        torch.cuda.synchronize()
        how = "event pairs around each launch, steps issued one by one"
        for k in range(count):
            ssd.ssd_profile_events(evs[k])
            step(k, stream)
            ssd.ssd_profile_events(None)
        torch.cuda.synchronize()
        out = [0.0] * nk
        for row in evs:
            for i in range(nk):
                out[i] += row[2 * i].elapsed_time(row[2 * i + 1])
    ssd.ssd_check_device_status(stream)
    return [v / count for v in out], how


def workload_record(w, dev, stream, peaks, steps=20):
    """One workload measured the way the headline is: ms per step over a graph
    of ``steps`` steps, the roofline of the step and each kernel's share."""
    import structured_state_space_03_b300 as ssd
    dtype = wl.torch_dtype(w.dtype)
    dims = (w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk)
    kernels = ssd.ssd_fwd_kernels(*dims, dtype)
    inp = wl.workload_inputs(w)
    sets, per_set = device_sets(w, inp, dev)
    ws = torch.empty(ssd.ssd_fwd_workspace_size(*dims, dtype), dtype=torch.uint8, device=dev)
    step = make_step(w, sets, ws)
    for k in range(3):
        step(k, stream)
    torch.cuda.synchronize()
    ssd.ssd_check_device_status(stream)
    g = capture(step, 0, steps)
    g.replay()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    g.replay()
    s1.record(stream)
    torch.cuda.synchronize()
    ssd.ssd_check_device_status(stream)
    ms = s0.elapsed_time(s1) / steps
    pk, _ = per_kernel_times(step, len(kernels), stream, 5)
    t_hbm = unavoidable_bytes(w) / (peaks["hbm_gbs"] * 1e9)
    t_tc = causal_flops(w) / (peaks["bf16_tflops"] * 1e12)
    rec = {"ms_per_step": ms, "tokens_per_s": w.tokens / (ms * 1e-3), "path": ssd.ssd_fwd_path(*dims, dtype),
           "block": ssd.ssd_fwd_block(*dims, dtype),  # the chunk length evaluated (exact for any length)
           "unavoidable_bytes": unavoidable_bytes(w), "causal_flops": causal_flops(w),
           "roofline_ms": max(t_hbm, t_tc) * 1e3, "bound": "hbm" if t_hbm >= t_tc else "tensor",
           "frac": max(t_hbm, t_tc) * 1e3 / ms, "steps": steps,
           "kernels": {kernels[i]: pk[i] for i in range(len(kernels))}}
    del sets, ws, g
    torch.cuda.empty_cache()
    return rec


FP32_LANES_PER_SM = 128  # fp32 FMA lanes per SM (4 sub-partitions x 32)


def fp32_fma_peak_tflops(peaks):
    """Peak fp32 FMA throughput of the plain ALU path: SMs x lanes x 2 flops x
    the maximum SM clock (148 x 128 x 2 x 2.032 GHz = 77.0 TFLOP/s on B300)."""
    return 148 * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2032.0) * 1e6 / 1e12


def bwd_flops(w, q=64):
    """Algorithmic FLOPs of the chunked backward (64-token chunks), masked
    (lower-triangular) products counted on their triangle: per (batch, chunk of
    q tokens) G * q(q+1)N for C B^T, and per head 2q(q+1)P (dy x^T, M^T dy) +
    2q(q+1)N (K^T C, K dt B) + 10qPN (B g^T, dy h, x g, the two chunk states)."""
    total = 0
    for c in range(math.ceil(w.seqlen / q)):
        n = min(q, w.seqlen - c * q)
        total += w.ngroups * n * (n + 1) * w.dstate + w.nheads * (
            2 * n * (n + 1) * w.headdim + 2 * n * (n + 1) * w.dstate + 10 * n * w.headdim * w.dstate)
    return total * w.batch


def bwd_unavoidable_bytes(w):
    """x, dy, B, C, dt read and dx, ddt, dB, dC (fp32) written once, plus the
    states (init, dfinal in; dinit out) and A, D, dA, dD."""
    e = 2 if w.dtype == "bf16" else 4
    tok = w.batch * w.seqlen
    ins = 2 * tok * w.nheads * w.headdim * e + 2 * tok * w.ngroups * w.dstate * e + tok * w.nheads * 4
    outs = tok * w.nheads * w.headdim * 4 + tok * w.nheads * 4 + 2 * tok * w.ngroups * w.dstate * 4
    states = 3 * w.batch * w.nheads * w.headdim * w.dstate * 4
    return ins + outs + states + 4 * w.nheads * 4


def bwd_chunk_bytes(w, q):
    """Bytes the in-chunk backward kernel must move per launch: x, dy, B, C and dt
    in, one recomputed and one adjoint fp32 state per (batch, head, q-token chunk)
    in, dx, ddt, dB and dC (fp32) out."""
    e = 2 if w.dtype == "bf16" else 4
    tok = w.batch * w.seqlen
    nc = math.ceil(w.seqlen / q)
    ins = 2 * tok * w.nheads * w.headdim * e + 2 * tok * w.ngroups * w.dstate * e + tok * w.nheads * 4
    states = 2 * w.batch * w.nheads * nc * w.headdim * w.dstate * 4
    outs = tok * w.nheads * w.headdim * 4 + tok * w.nheads * 4 + 2 * tok * w.ngroups * w.dstate * 4
    return ins + states + outs


def backward_measurement(w, dev, stream, peaks, steps=20):
    """The backward (ssd_bwd) on the workload: ms per step over a CUDA graph of
    ``steps`` backward calls rotating over input sets larger than L2, each
    kernel's device time, the step against its roofline and the dominant
    kernel against the fp32 FMA peak it runs on."""
    import structured_state_space_03_b300 as ssd
    dtype = wl.torch_dtype(w.dtype)
    names = ssd.ssd_bwd_kernels(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, dtype)
    inp = wl.workload_inputs(w)
    dy, dfinal = wl.make_cotangents(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.dtype, seed=w.seed)
    per_set = bwd_unavoidable_bytes(w)
    nsets = max(2, math.ceil(3 * L2_BYTES / per_set))
    sets = []
    for _ in range(nsets):
        d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
        d["dy"], d["dfinal"] = dy.to(dev), dfinal.to(dev)
        sets.append(d)

    def step(k, st):
        d = sets[k % nsets]
        ssd.ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init_state"], dy=d["dy"],
                    dfinal_state=d["dfinal"], stream=st)

    for k in range(3):
        step(k, stream)
    torch.cuda.synchronize()
    ssd.ssd_check_device_status(stream)
    g = capture(step, 0, steps)
    g.replay()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    g.replay()
    s1.record(stream)
    torch.cuda.synchronize()
    ssd.ssd_check_device_status(stream)
    ms = s0.elapsed_time(s1) / steps
    pk, how = per_kernel_times(step, len(names), stream, 5)
    dom = max(range(len(names)), key=lambda i: pk[i])
    flops = bwd_flops(w)
    # the in-chunk kernel's share of the FLOPs: everything but the two chunk states
    states_flops = 4 * w.batch * w.seqlen * w.nheads * w.headdim * w.dstate
    kflops = {"bwd_chunk": flops - states_flops, "bwd_chunk_tc": flops - states_flops,
              "bwd_chunk_states": states_flops}
    alu_peak = fp32_fma_peak_tflops(peaks)
    t_hbm = per_set / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    # a kernel that runs twice in a step (the chunk-state kernel: S_c, then G_c) is listed as name#2
    keys = [n if names[:k].count(n) == 0 else f"{n}#{names[:k].count(n) + 1}" for k, n in enumerate(names)]
    rec = {"workload": w.name, "ms_per_step": ms, "tokens_per_s": w.tokens / (ms * 1e-3), "steps": steps,
           "kernels": {keys[i]: {"ms_per_launch": pk[i], "share": pk[i] / (sum(pk) or 1.0)}
                       for i in range(len(names))},
           "kernel_timing": how,
           "step_roofline": {"unavoidable_bytes": per_set, "algorithmic_flops": flops,
                             "roofline_ms": max(t_hbm, t_tc) * 1e3, "bound": "hbm" if t_hbm >= t_tc else "tensor",
                             "frac": max(t_hbm, t_tc) * 1e3 / ms},
           "l2": f"inputs rotate over {nsets} device copies ({nsets * per_set / 2**20:.0f} MiB > 126 MB L2)"}
    if names[dom] == "bwd_chunk_tc":
        # tensor cores: its FLOPs take ~8 us at the bf16 peak, so the bound is its bytes
        nbytes = bwd_chunk_bytes(w, 128)
        ach = nbytes / (pk[dom] * 1e-3) / 1e9
        rec["roofline"] = {"bound": "hbm", "kernel": names[dom], "achieved": ach, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": ach / peaks["hbm_gbs"], "traffic": recorded_traffic(names[dom], w.name),
                           "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": kflops[names[dom]],
                           "launch_ms": pk[dom], "peak_source": "measured (copy bandwidth)"}
    elif names[dom] in kflops:
        ach = kflops[names[dom]] / (pk[dom] * 1e-3) / 1e12
        rec["roofline"] = {"bound": "alu", "kernel": names[dom], "achieved": ach, "peak": alu_peak,
                           "unit": "TFLOP/s", "frac": ach / alu_peak, "traffic": recorded_traffic(names[dom], w.name),
                           "algorithmic_flops_per_launch": kflops[names[dom]], "launch_ms": pk[dom],
                           "peak_source": "148 SMs x 128 fp32 lanes x 2 flops x max SM clock"}
    del sets, g
    torch.cuda.empty_cache()
    return rec


def main():
    args = parse_args()
    world, rank, local = dist_env()
    w = wl.by_name(args.workload)
    if args.seqlen > 0 and args.seqlen != w.seqlen:
        w = dataclasses.replace(w, seqlen=args.seqlen, name=f"{w.name}_at_L{args.seqlen}")
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import structured_state_space_03_b300 as ssd
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssd.lib()
    dtype = wl.torch_dtype(w.dtype)
    dims = (w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.chunk)
    kernels = ssd.ssd_fwd_kernels(*dims, dtype)
    path = ssd.ssd_fwd_path(*dims, dtype)
    nk = len(kernels)

    inp = wl.workload_inputs(w)
    sets, per_set = device_sets(w, inp, dev)
    nsets = len(sets)
    ws = torch.empty(ssd.ssd_fwd_workspace_size(*dims, dtype), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = make_step(w, sets, ws)

    warmup = max(3, args.warmup)
    for k in range(warmup):
        step(k, stream)
    torch.cuda.synchronize()
    ssd.ssd_check_device_status(stream)

    steps = args.steps
    if steps <= 0:  # enough steps for a ~3 s timed region
        t0 = time.perf_counter()
        for k in range(20):
            step(k, stream)
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 20
        steps = int(min(200000, max(50, 3.0 / max(per, 1e-6))))

    # The timed region replays CUDA graphs of the steps, so host-side launch
    # work (Python, argument checks) does not leave the GPU idle between steps.
    plan = graph_plan(steps)
    graphs = []
    first = 0
    for per, reps in plan:
        graphs.append((capture(step, first, per), reps))
        first += per
    for g, _ in graphs:  # upload and warm each graph once
        g.replay()
    torch.cuda.synchronize()
    ssd.ssd_check_device_status(stream)

    sampler = ClockSampler(local)
    time.sleep(0.3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    mark0 = sampler.mark()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for g, reps in graphs:
        for _ in range(reps):
            g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    mark1 = sampler.mark()
    if world > 1:
        dist.barrier()
    elapsed_ms = start.elapsed_time(end)
    time.sleep(0.25)
    sampler.stop()
    ssd.ssd_check_device_status(stream)
    elapsed_ms = max_over_ranks(elapsed_ms, dev)

    # the same steps issued one call at a time from Python, the stream kept
    # busy by `warmup` queued steps (for reference; not the headline)
    for k in range(warmup):
        step(k, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        step(k, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ssd.ssd_check_device_status(stream)
    eager_ms = e0.elapsed_time(e1) / steps

    # each kernel's own device time, in a separate untimed pass
    per_kernel, kernel_timing = per_kernel_times(step, nk, stream, max(5, min(steps, 100)))
    tot_k = sum(per_kernel) or 1.0
    dom = max(range(nk), key=lambda i: per_kernel[i])
    dom_name = kernels[dom]
    peaks, peak_src = load_peaks()
    dom_bytes = kernel_algorithmic_bytes(w, dom_name)
    dom_gbs = dom_bytes / (per_kernel[dom] * 1e-3) / 1e9
    traffic = recorded_traffic(dom_name, w.name)

    ms_per_step = elapsed_ms / steps
    tokens = w.tokens
    value = tokens * steps * world / (elapsed_ms * 1e-3)
    t_hbm = unavoidable_bytes(w) / (peaks["hbm_gbs"] * 1e9)
    t_tc = causal_flops(w) / (peaks["bf16_tflops"] * 1e12)
    t_roof = max(t_hbm, t_tc)

    # end to end through the host-buffer entry point, pinned host memory
    host = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    y_host = torch.empty_like(host["x"]).pin_memory()
    f_host = torch.empty(w.batch, w.nheads, w.headdim, w.dstate, dtype=torch.float32).pin_memory()
    e2e_steps = max(5, min(steps, 100))

    def host_step():
        ssd.ssd_fwd_host(host["x"], host["dt"], host["A"], host["B"], host["C"], host["D"], host["init_state"],
                         chunk=w.chunk, y=y_host, final_state=f_host, stream=stream)

    for _ in range(3):
        host_step()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        host_step()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, dev)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = y_host.numel() * y_host.element_size() + f_host.numel() * 4

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w),
        "run": {"path": path, "block": ssd.ssd_fwd_block(*dims, dtype), "kernels": kernels,
                "timing": f"CUDA events around graph replays of the {steps} steps ({len(graphs)} graph(s))",
                "l2": f"inputs rotate over {nsets} device copies ({nsets * per_set / 2**20:.0f} MiB > 126 MB L2)"},
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": dom_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": dom_gbs / peaks["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": dom_bytes, "launch_ms": per_kernel[dom],
                     "launch_timing": kernel_timing,
                     "peak_source": f"{peak_src} (copy bandwidth)"},
        "step_roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor", "unavoidable_bytes": unavoidable_bytes(w),
                          "causal_flops": causal_flops(w), "roofline_ms": t_roof * 1e3,
                          "frac": t_roof * 1e3 / ms_per_step, "peak_source": peak_src},
        "kernels": {kernels[i]: {"ms_per_launch": per_kernel[i], "share": per_kernel[i] / tot_k}
                    for i in range(nk)},
        "eager": {"ms_per_step": eager_ms, "tokens_per_s": tokens * world / (eager_ms * 1e-3),
                  "how": "ssd_fwd_ws called once per step from Python, stream pre-filled"},
        "e2e": {"value": tokens * e2e_steps * world / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "entry": "ssd_fwd_host"},
        "gpu_launches": nk * steps,
        "clocks": sampler.summary(mark0, mark1),
    }
    del graphs
    if rank == 0 and world == 1 and not args.no_extras:
        line["decode_step"] = decode_step_measurement(dev, peaks, stream)
        if w is wl.HEADLINE:
            line["pre_step"] = pre_step_measurement(sets, w, stream)
            line["varlen_step"] = varlen_step_measurement(sets, w, stream, peaks)
            if not args.no_backward:
                line["backward"] = backward_measurement(w, dev, stream, peaks)
            if not args.no_workloads:
                del sets
                torch.cuda.empty_cache()
                line["workloads"] = {o.name: workload_record(o, dev, stream, peaks)
                                     for o in wl.WORKLOADS[2:]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
