#!/usr/bin/env python
"""Benchmark of the KDA backward pass on GB300.

One step = one full backward (kda_bwd with the chunk states recomputed inside:
forward-state scan + reverse dS scan, per-chunk gradients, dA_log reduction)
over one batch of the main workload, B=4 T=8192 H=32 K=V=128 bf16, inputs
already resident in HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs as one process per GPU under torchrun: every rank processes its
own batch (independent problems, no collective on the data path), the
reported time is the max over ranks and the value counts the tokens of all
ranks ("weak" scaling).  `--impl reference` times the fp64 CPU oracle (the
only reference there is for this path) on a bounded sample of the same
workload, on the host cores, rank 0 only.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA backward tokens/s on 1×GB300 and % of bf16-TC/HBM roofline; vs CPU oracle"
WORKLOAD = "main_bf16"

# Algorithmic HBM bytes per (token, head) for K = V = 128, bf16 (chunk 64):
#   path: read q, k, v, dO, g (5 x 256 B) and beta (2 B); write dq, dk, dv, dg
#   (4 x 256 B) and dbeta (2 B); write and read the bf16 chunk states S_n once
#   each (2 x 32 KiB per 64 tokens = 1024 B)                       -> 3332 B
#   gradient kernel: the same inputs and outputs, plus S_n and dS_{n+1}
#   (2 x 512 B) read                                               -> 3332 B
ALG_BYTES = {"grads": 3332, "path": 3332}
# Algorithmic FLOP per (token, head): each product of a 64-token chunk (C = 64,
# D = 128) at its useful size, 2 m n k, triangular ones (the strictly lower or
# lower pair matrices and inverse, the masked dMqk / dAkk) at half:
#   prep   G, Mqk 2 x 0.52 M, W, U0, Mqk W 3 x 0.52 M, WY inverse 0.17 M  -> 2.8 M
#   forward scan   W S_n, kr^T U                 2 x 2.1 M              -> 4.2 M
#   reverse scan   kr dS, W^T (.), QE^T dO       3 x 2.1 M              -> 6.3 M
#   gradients  kd S 2.1, INVb Xr 1.05, Mqk^T dO 1.05, kr dS 2.1, U dS^T 2.1,
#              INV^T dU 1.05, [dO; dvcorr] U^T 1.05, S [dO; dvcorr]^T 4.2,
#              the four intra-chunk terms 2.1                             -> 16.8 M
#   path                                                                 -> 30.1 M
ALG_FLOP = {"grads": 16.8e6 / 64, "path": 30.1e6 / 64}
# phases recorded by kda_bwd_timed (5 events) and the kernel each one runs
PHASES = ("prep", "scan", "grads", "reduce")
KERNEL_NAMES = {"prep": "kda_prep_tc_kernel", "scan": "kda_scan_tc_kernel",
                "grads": "kda_grads_tc_kernel", "reduce": "kda_dalog_reduce_kernel"}
# kernels of one kda_bwd call: prep, scans, gradients, dA_log reduction; a
# varlen call adds the sequence-order kernel, context-parallel scans (few
# (sequence, head) chains) add their combine kernel and second scan pass, and
# the tensor-core path (bf16, K = V = 128) its two exact kernels for gates
# past the block range (one after the prep, one after the gradients; each
# walks the chunk flags and works only on flagged chunks)
LAUNCHES_PER_STEP = 4


def launches_per_step(shape, cu, forward=False):
    import linear_attention_backward_gb300 as kda
    n = (3 if forward else LAUNCHES_PER_STEP) + (0 if cu is None else 1)
    if shape.dtype == kda.KDA_BF16 and shape.K == 128:
        n += 1 if forward else 2
    return n + (2 if kda.scan_segments(shape) > 0 else 0)

# DRAM traffic per launch of the gradient kernel from ncu
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by the hash of the
# kernel sources it was taken from; a changed kernel reports null until it
# is measured again.
NCU_TRAFFIC = {
    # ncu on main_b1_bf16 (B=1: 4096 chunk-heads per launch), DRAM read 841.4 MB +
    # write 244.7 MB (profiles/traffic_main_b1_bf16.md), scaled by 4 to the main
    # workload's 16384 chunk-heads (the kernel's traffic is proportional to them)
    "kda_grads_tc_kernel": {"sha": "523e956effe5a3d3", "workload": "main_bf16",
                            "bytes_per_launch": 4344210432},
}

KERNEL_SOURCES = {
    "grads": ["kda_grads_tc.cu", "kda_tc_tiles.cuh", "kda_umma.cuh", "kda_chunk.cuh",
              "kda_device.cuh", "kda_params.h"],
}


def src_hash(kernel):
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "linear_attention_backward_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms, each sample
    stamped with the host clock on arrival, so that the samples taken during
    the timed region can be kept alone (``window``)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []  # (host time, line)
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def running(self):
        """True once the first sample has arrived (or sampling is unavailable)."""
        return self.proc is None or len(self.lines) > 0

    def mark(self, t0, t1):
        """Keep only samples that arrived in [t0, t1] (host clock)."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if self.window is not None:
            inside = [ln for t, ln in lines if self.window[0] <= t <= self.window[1]]
            lines = inside if inside else [ln for _, ln in lines[-3:]]
        else:
            lines = [ln for _, ln in lines]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "interval_ms": 20,
                "window": "samples that arrived during the timed region" if self.window else
                          "all samples", "reasons": sorted(reasons)}


def max_over_ranks(ms, pg, device):
    """The slowest rank's time: every rank's timed region counts, and the job
    is done when the last rank is (pg None: one process)."""
    if pg is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world_size, ms):
    """Whole-job throughput: the units all ranks processed (each rank its own
    batch of the same size: weak scaling) over the slowest rank's time."""
    return units_per_rank * world_size / (ms * 1e-3)


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def oracle_sample(x, n_units, t_sample, nthreads):
    """Run the fp64 oracle on n_units (sequence, head) units, each the first
    t_sample tokens of its sequence; returns seconds."""
    import numpy as np
    import oracle
    B, T, H, K = x["q"].shape
    units = [(b, h) for b in range(B) for h in range(H)]
    units = (units * (n_units // len(units) + 1))[:n_units]
    t_sample = min(t_sample, T)
    pick = lambda t, b, h: t[b, :t_sample, h:h + 1].double().numpy()
    cat = lambda name: np.concatenate([pick(x[name], b, h) for b, h in units], 0)
    q, k, v, g, dO = (cat(n) for n in ("q", "k", "v", "g", "dO"))
    beta = np.concatenate([x["beta"][b, :t_sample, h:h + 1].double().numpy()
                           for b, h in units], 0)
    # per-unit A_log differs; a one-head batch shares A_log, so take the mean
    # head's value: the oracle's cost does not depend on it
    A_log = x["A_log"][:1].double().numpy()
    cu = [i * t_sample for i in range(n_units + 1)]
    h0 = x["h0"][:1, :1].double().numpy().repeat(n_units, 0)
    dhT = x["dhT"][:1, :1].double().numpy().repeat(n_units, 0)
    t0 = time.perf_counter()
    oracle.backward(q, k, v, g, beta, A_log, h0, dO, dhT, cu_seqlens=cu, nthreads=nthreads)
    return time.perf_counter() - t0, n_units * t_sample


def cpu_baseline(x, steps=1):
    """The oracle on the whole workload (every (sequence, head) unit, all
    tokens): about 10 s of fp64 work on 16 host cores."""
    cores = os.cpu_count() or 1
    B, T, H, _ = x["q"].shape
    n_units = B * H
    t_sample = T
    times = []
    head_tokens = 0
    for _ in range(steps):
        dt, head_tokens = oracle_sample(x, n_units, t_sample, cores)
        times.append(dt)
    sec = statistics.median(times)
    return {"value": (head_tokens / H) / sec, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"the whole {WORKLOAD} workload: all {n_units} (sequence, head) units x "
                      f"{t_sample} tokens (= {head_tokens} head-tokens), fp64, {cores} OpenMP "
                      f"threads, one run; tokens = head-tokens / H",
            "seconds": sec}


def run_reference(args, ws, rank):
    import oracle
    from linear_attention_backward_gb300 import workloads as wl
    if rank != 0:
        return 0
    oracle.build()
    x = wl.make_inputs(wl.WORKLOADS[WORKLOAD], seed=0)
    w = wl.WORKLOADS[WORKLOAD]
    for _ in range(args.warmup):
        oracle_sample(x, 1, 256, 1)
    cores = os.cpu_count() or 1
    t_sample = 1024
    t_all = 0.0
    ht = 0
    for _ in range(args.steps):
        dt, n = oracle_sample(x, cores, t_sample, cores)
        t_all += dt
        ht += n
    value = (ht / w.H) / t_all
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_all / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {cores} (sequence, head) units x first "
                                   f"{t_sample} tokens, fp64, {cores} threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129 << 20  # GB300 L2


def flushes_l2(w):
    """Workloads whose input tensors fit in L2 get a 256 MB write between
    timed steps, and only the calls themselves are timed."""
    return w.B * w.T * w.H * w.K * 2 < L2_BYTES if not w.varlen else False


def workload_config(w):
    shape = (f"{w.varlen[0]} packed sequences of U[{w.varlen[1]}, {w.varlen[2]}] tokens"
             if w.varlen else f"B={w.B} T={w.T}")
    return {"workload": f"{w.name}: KDA chunked backward, {shape} H={w.H} "
                        f"K={w.K} V={w.V} chunk={w.chunk}, states recomputed in the call",
            "global_batch": w.B, "seq_len": w.T, "heads": w.H, "head_dim": w.K,
            "parallelism": "replicas (one independent batch per GPU)",
            "l2": ("L2 flushed between timed steps (a 256 MB buffer written outside the "
                   "timed calls; each input tensor is B*T*H*128*2 bytes, below the 129 MB L2)"
                   if flushes_l2(w) else
                   "inputs larger than L2 (each input tensor is B*T*H*128*2 bytes; "
                   "268 MB at B=4), no flush")}


def run_forward(args, w, xh, dev, ws, pg):
    """The forward pass (prep, forward state scan, chunk outputs) on the
    workload's inputs, resident in HBM: one JSON line."""
    import torch
    import linear_attention_backward_gb300 as kda
    d = {n: (t.to(dev) if t is not None else None) for n, t in xh.items()}
    cu = d["cu_seqlens"]
    shape = kda.make_shape(d["q"], d["v"], cu_seqlens=cu)
    wsb = torch.empty((kda.workspace_bytes(shape),), dtype=torch.uint8, device=dev)
    o = torch.empty_like(d["v"])
    nseq = w.B if cu is None else cu.numel() - 1
    hT = torch.empty((nseq, w.H, w.K, w.V), dtype=torch.float32, device=dev)

    def step():
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d.get("h0"),
                cu_seqlens=cu, o=o, hT=hT, want_hT=True, workspace=wsb)

    for _ in range(args.warmup):
        step()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev) if flushes_l2(w) else None
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    s0.record()
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 255)
        pairs[i][0].record()
        step()
        pairs[i][1].record()
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / args.steps
    if flush is not None:  # the calls alone
        ms = sum(a.elapsed_time(b) for a, b in pairs) / args.steps
    ms = max_over_ranks(ms, pg, dev)
    assert kda.get_device_status() == 0
    tokens = int(xh["q"].shape[0] * xh["q"].shape[1])
    cfg = workload_config(w)
    cfg["workload"] = cfg["workload"].replace("chunked backward", "chunked forward").replace(
        "states recomputed in the call", "o and hT")
    line = {"metric": "KDA forward tokens/s (kda_fwd: o and hT)", "value": job_rate(tokens, ws, ms),
            "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": cfg,
            "gpu_launches": launches_per_step(shape, cu, forward=True) * args.steps,
            "scan_segments": kda.scan_segments(shape)}
    if int(os.environ.get("RANK", "0")) == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name (default: the main B=4 T=8192 H=32 batch)")
    ap.add_argument("--forward", action="store_true",
                    help="time the forward pass (kda_fwd: o and hT) instead of the backward")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws, rank, local = dist_setup()

    if args.impl == "reference":
        return run_reference(args, ws, rank)

    import torch
    import __graft_entry__
    __graft_entry__.build()
    import linear_attention_backward_gb300 as kda
    from linear_attention_backward_gb300 import workloads as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    w = wl.WORKLOADS[args.workload]
    xh = wl.make_inputs(w, seed=rank)
    if args.forward:
        return run_forward(args, w, xh, dev, ws, pg)
    names_in = ["q", "k", "v", "g", "beta", "dO", "A_log"]
    if w.with_h0:
        names_in.append("h0")
    if w.with_dhT:
        names_in.append("dhT")
    if xh["cu_seqlens"] is not None:  # varlen: the packed sequences' bounds
        names_in.append("cu_seqlens")
    d = {n: xh[n].to(dev) for n in names_in}
    h0 = d.get("h0")
    dhT = d.get("dhT")
    cu = d.get("cu_seqlens")
    nseq = w.B if cu is None else cu.numel() - 1
    shape = kda.make_shape(d["q"], d["v"], cu_seqlens=cu)
    wsb = torch.empty((kda.workspace_bytes(shape),), dtype=torch.uint8, device=dev)
    out = {n: torch.empty_like(d[m]) for n, m in
           (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dg", "g"), ("dbeta", "beta"))}
    out["dA_log"] = torch.empty((w.H,), dtype=torch.float32, device=dev)
    out["dh0"] = torch.empty((nseq, w.H, w.K, w.V), dtype=torch.float32, device=dev)

    def step(events=None):
        kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], h0, d["dO"], dhT,
                cu_seqlens=cu, out=out, workspace=wsb, events=events)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert kda.get_device_status() == 0

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    for e4 in evs:  # materialise the events (created lazily by torch)
        for e in e4:
            e.record()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev) if flushes_l2(w) else None
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local])
    sampler.start()
    # untimed steps until the sampler is live (nvidia-smi takes a moment to
    # start), so that its samples cover the timed region
    t_wait = time.perf_counter()
    while not sampler.running() and time.perf_counter() - t_wait < 10.0:
        step()
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record()
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 255)
        step(evs[i])
    end.record()
    torch.cuda.synchronize()
    sampler.mark(t0, time.perf_counter())
    clocks = sampler.stop()
    if pg:
        pg.barrier()
    ms = start.elapsed_time(end)
    if flush is not None:  # the calls alone, from their first to their last event
        ms = sum(e5[0].elapsed_time(e5[4]) for e5 in evs)
    phase = {n: [] for n in PHASES}
    for e5 in evs:
        for j, n in enumerate(PHASES):
            phase[n].append(e5[j].elapsed_time(e5[j + 1]))
    ms = max_over_ranks(ms, pg, dev)
    ms_step = ms / K
    tokens = int(xh["q"].shape[0] * xh["q"].shape[1])  # B * T, or the packed total (varlen)
    value = job_rate(tokens, ws, ms_step)
    assert kda.get_device_status() == 0

    # ---- with the chunk states given: kda_fwd_states, then kda_bwd on them ----
    def timed(fn, n=10):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    states = kda.fwd_states(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], h0,
                            cu_seqlens=cu, workspace=wsb)
    states_given = {
        "fwd_states_ms": timed(lambda: kda.fwd_states(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                      d["A_log"], h0, cu_seqlens=cu,
                                                      states=states, workspace=wsb)),
        "bwd_ms": timed(lambda: kda.bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"],
                                        h0, d["dO"], dhT, cu_seqlens=cu, out=out, workspace=wsb,
                                        states=states)),
        "what": "kda_fwd_states (chunk-parallel prep and the forward tcgen05 scan, packed "
                "chunk states) and kda_bwd given those states (prep, reverse scan, gradients), "
                "CUDA events, 10 calls each"}
    del states
    assert kda.get_device_status() == 0

    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs up from pinned host memory, runs the
    # backward and reads every gradient back.  Steps are pipelined over three
    # streams with two device buffer sets: step i + 1's inputs go up while step
    # i computes and step i - 1's gradients come down (the two directions use
    # separate copy engines).
    pin = {n: xh[n].pin_memory() for n in names_in}
    host_out = {n: torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for n, o in out.items()}
    bi = sum(t.numel() * t.element_size() for t in pin.values())
    bo = sum(t.numel() * t.element_size() for t in host_out.values())
    E = max(1, args.e2e_steps)
    dsets = [d, {n: torch.empty_like(t) for n, t in d.items()}]
    osets = [out, {n: torch.empty_like(t) for n, t in out.items()}]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n_steps, after=None):
        done_c = [None, None]  # per buffer set: its last step has computed
        done_o = [None, None]  # per buffer set: its gradients are down
        if after is not None:
            s_in.wait_event(after)
        for i in range(n_steps):
            b = i % 2
            di, oi = dsets[b], osets[b]
            with torch.cuda.stream(s_in):
                if done_c[b] is not None:
                    s_in.wait_event(done_c[b])
                for n in names_in:
                    di[n].copy_(pin[n], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            comp.wait_event(ready)
            if done_o[b] is not None:
                comp.wait_event(done_o[b])
            kda.bwd(di["q"], di["k"], di["v"], di["g"], di["beta"], di["A_log"], di.get("h0"),
                    di["dO"], di.get("dhT"), cu_seqlens=di.get("cu_seqlens"), out=oi,
                    workspace=wsb)
            done_c[b] = torch.cuda.Event()
            done_c[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_c[b])
                for n, o in oi.items():
                    host_out[n].copy_(o, non_blocking=True)
                done_o[b] = torch.cuda.Event()
                done_o[b].record(s_out)
        comp.wait_stream(s_out)

    e2e_run(2)  # warm-up (first use of the second buffer set and of the pinned buffers)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    s0.record(comp)
    e2e_run(E, after=s0)
    s1.record(comp)
    torch.cuda.synchronize()
    e2e_ms = s0.elapsed_time(s1) / E
    e2e_ms = max_over_ranks(e2e_ms, pg, dev)
    # the same copies without the backward, for the host link's own time per
    # step on this machine (the link differs between boxes)
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    c0.record(comp)
    s_in.wait_event(c0)
    s_out.wait_event(c0)
    for i in range(E):
        di, oi = dsets[i % 2], osets[i % 2]
        with torch.cuda.stream(s_in):
            for n in names_in:
                di[n].copy_(pin[n], non_blocking=True)
        with torch.cuda.stream(s_out):
            for n, o in oi.items():
                host_out[n].copy_(o, non_blocking=True)
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    c1.record(comp)
    torch.cuda.synchronize()
    copies_ms = max_over_ranks(c0.elapsed_time(c1) / E, pg, dev)
    e2e = {"value": job_rate(tokens, ws, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms,
           "copies_only_ms_per_step": copies_ms,
           "steps": E, "pipeline": "H2D / backward / D2H on three streams, two device "
                                   "buffer sets, every step's inputs up and gradients down"}

    # ---- roofline of the dominant kernel, and of the whole step ----
    hbm, tflops, src = load_peaks()
    kern_ms = {k: statistics.mean(v) for k, v in phase.items()}
    dom = "grads"  # the largest phase on every workload measured
    head_tokens = tokens * w.H
    alg = ALG_BYTES[dom] * head_tokens
    achieved = alg / (kern_ms[dom] * 1e-3) / 1e9
    tr = NCU_TRAFFIC.get(KERNEL_NAMES[dom])
    traffic = None
    if tr and tr.get("sha") == src_hash(dom) and tr.get("workload") == args.workload:
        traffic = tr["bytes_per_launch"]
    roofline = {"kernel": KERNEL_NAMES[dom], "bound": "hbm", "achieved": achieved,
                "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                "alg_bytes_per_launch": alg,
                "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                "tensor_frac": (ALG_FLOP[dom] * head_tokens / (kern_ms[dom] * 1e-3) / 1e12)
                / tflops}
    path_alg = ALG_BYTES["path"] * head_tokens
    path = {"alg_bytes_per_step": path_alg,
            "achieved_gbs": path_alg / (ms_step * 1e-3) / 1e9,
            "frac_hbm": path_alg / (ms_step * 1e-3) / 1e9 / hbm,
            "frac_tensor": ALG_FLOP["path"] * head_tokens / (ms_step * 1e-3) / 1e12 / tflops}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w), "clocks": clocks, "e2e": e2e,
        "gpu_launches": launches_per_step(shape, cu) * K, "scan_segments": kda.scan_segments(shape),
        "roofline": roofline, "path_roofline": path,
        "kernels_ms": kern_ms, "kernels": KERNEL_NAMES, "states_given": states_given,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = {k: v for k, v in cpu_baseline(xh).items() if k != "seconds"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
