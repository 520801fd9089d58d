#!/usr/bin/env python
"""Benchmark of HSTU jagged attention, forward + backward, on one GB300.

Workload: the heavy-tailed training batch -- 64 jagged sequences with
Zipf(1.2) history lengths on [1, 8192] after stochastic-length sampling, plus
32 candidates each; 4 heads of 128; BF16 inputs, FP32 outputs; causal +
candidate mask; relative-position (128) and log2 time-gap (64) bias.  One
step = forward (attention + LayerNorm gate) and backward (dq, dk, dv, du,
d_rab) of one batch.  16 distinct seeded batches are resident in HBM and
taken in turn, so consecutive steps never find their inputs in L2.

Metric: useful TFLOP/s, counting allowed (unmasked) query-key pairs only:
forward 2 (d_qk + d_v) and backward 2 (3 d_qk + 2 d_v) FLOPs per pair.

With --workload layer it measures the full HSTU layer instead (x W1, SiLU
split, the same attention, LayerNorm gate, y W2 + x, forward + backward on 8
sequences of 8K-32K tokens at D = 512), counting the projections' FLOPs too.

The e2e figure runs the same steps through the C ABI from pinned host
buffers, every step's inputs uploaded and its result read back (a training
step's parameter gradients, an inference request's candidate outputs), the
copies on two streams overlapping the neighbouring steps' compute;
e2e.all_outputs reads back every output and gradient instead.  A heavy-tailed
batch's inputs sit in one buffer (one transfer per step, as a data loader
delivers a batch).

With --graph the K timed steps are captured once as a CUDA graph and the
timed region replays it (the per-kernel events of the library's timing hook
are part of the graph); by default they are launched one by one.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload layer] [--graph]
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
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from hstu_jagged_attention_02_gb300 import synth  # noqa: E402

METRIC = "HSTU jagged attention useful TFLOP/s (fwd+bwd), % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"
WORKLOAD = ("heavy_tailed: 64 jagged sequences, Zipf(1.2) history lengths on [1,8192] with "
            "stochastic-length sampling + 32 candidates, 4 heads x 128, BF16 in / FP32 out, "
            "causal + candidate mask, position + time rab, forward + backward")
N_SEEDS = 16
# algorithmic DRAM bytes per (token, head, dim) of each attention kernel, BF16 in / FP32 out
KERNEL_BYTES_PER_ELEM = {"fwd": 3 * 2 + 4, "bwd": 3 * 2 + 2 * 2 + 3 * 4}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def allowed_pairs(b) -> int:
    """Allowed (i, j) pairs of a batch summed over sequences and heads."""
    n = b.lengths.astype(np.int64)
    c = b.num_contexts.astype(np.int64) if b.num_contexts is not None else np.zeros_like(n)
    m = b.num_targets.astype(np.int64) if b.num_targets is not None else np.zeros_like(n)
    h_end = n - m
    per_seq = h_end * (h_end + 1) // 2 + c * (c - 1) // 2 + m * (h_end + 1)
    return int(per_seq.sum()) * b.H


def useful_flops(b):
    p = allowed_pairs(b)
    fwd = 2 * (b.d_qk + b.d_v) * p
    bwd = 2 * (3 * b.d_qk + 2 * b.d_v) * p
    return fwd, bwd


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons.  mark_load()
    and stop() bracket the loaded span (the soak steps and the timed steps,
    back to back on the stream); only samples whose timestamps fall inside it
    enter the summary."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.f = None
        self.t_load = None

    def mark_load(self):
        self.t_load = time.time()

    @staticmethod
    def _epoch(stamp):
        # nvidia-smi prints local time as "YYYY/MM/DD HH:MM:SS.mmm"
        try:
            day, frac = stamp.rsplit(".", 1) if "." in stamp else (stamp, "0")
            return time.mktime(time.strptime(day.strip(), "%Y/%m/%d %H:%M:%S")) + float("0." + frac.strip())
        except ValueError:
            return None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:   # no nvidia-smi: the line says so
            self.proc = None

    def stop(self):
        t_end = time.time()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()   # the sampler this object started
        self.f.flush()
        self.f.seek(0)
        rows = [ln.strip().split(",") for ln in self.f.read().splitlines() if ln.strip()]
        self.f.close()
        os.unlink(self.f.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0 = self.t_load if self.t_load is not None else 0.0
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 10:
                continue
            ts = self._epoch(r[0])
            if ts is not None and not (t0 <= ts <= t_end):
                continue   # before the load or after it
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
            except ValueError:
                continue
            try:
                power.append(float(r[4]))
            except ValueError:
                pass
            for nm, val in zip(names, r[6:10]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_min_mhz": min(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "power_w_max": max(power) if power else None,
                "samples": len(sm)}


# the translation unit of each timed attention kernel plus the headers it includes
KERNEL_SOURCES = {
    "fwd": ("hstu_tc_fwd.cu", "tc_ptx.cuh", "hstu_common.cuh"),
    "bwd": ("hstu_tc_bwd.cu", "tc_ptx.cuh", "hstu_common.cuh"),
}


def _code_only(text: str) -> str:
    """Source text without comments and blank lines."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_sources_sha(role: str):
    """Hash of the code an attention kernel is compiled from: its translation
    unit and device headers, the kernel parameter block of hstu_internal.h
    and the public header's declarations (comments left out)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hstu_jagged_attention_02_gb300", "csrc")
    for fn in KERNEL_SOURCES[role]:
        h.update(_code_only(open(os.path.join(csrc, fn)).read()).encode())
    internal = open(os.path.join(csrc, "hstu_internal.h")).read()
    i = internal.index("struct AttnParams {")
    h.update(_code_only(internal[i:internal.index("};", i)]).encode())
    h.update(_code_only(open(os.path.join(ROOT, "include", "hstu_attn.h")).read()).encode())
    return h.hexdigest()[:16]


def traffic_record(kernel_role: str):
    """DRAM bytes per token of the dominant kernel from the committed ncu
    capture, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):   # unreadable or malformed record: no traffic figure
        return None
    rec = d.get(kernel_role)
    if rec and rec.get("sources_sha") == kernel_sources_sha(kernel_role.split(":")[1]):
        return rec
    return None


# ------------------------------------------------------------ workloads

class AttentionWorkload:
    """The heavy-tailed attention batch (the default line)."""
    name = "heavy_tailed"
    has_backward = True
    metric = METRIC
    description = WORKLOAD
    n_batches = N_SEEDS
    dropout_p = 0.0   # --dropout: the fused dropout on y (fixed seed and offset)
    plan_once = True  # the forward plans the backward too (--plan-each-call: each call plans for itself)

    def dropout(self):
        return None if not self.dropout_p else (self.dropout_p, 20240601, 0)

    def batches(self, rank):
        return [synth.heavy_tailed(rank * N_SEEDS + s) for s in range(N_SEEDS)]

    def problem(self, b, dev):
        from hstu_jagged_attention_02_gb300.attention import Problem
        return Problem(b, device=dev, out_dtype="fp32", dropout=self.dropout(), plan_once=self.plan_once,
                       packed_inputs=True)

    def flops(self, b):
        """(attention fwd, attention bwd, whole step) useful FLOPs."""
        f, bw = useful_flops(b)
        return f, bw, f + bw

    def kernel_bytes(self, b, role):
        """Algorithmic DRAM bytes of one launch of the attention kernel of a role."""
        return KERNEL_BYTES_PER_ELEM[role] * b.T * b.H * b.d_qk

    def host_io(self, pr):
        # a batch's inputs sit in one device buffer, as a data loader would
        # deliver them: one host-to-device transfer per step
        ins = [pr.input_buffer]
        outs = [t for t in (pr.y, pr.dq, pr.dk, pr.dvv, pr.du, pr.d_rab_pos, pr.d_rab_time)
                if t is not None]
        return ins, outs

    def result(self, pr):
        # what a training step reads back: the gradients of the attention's own
        # parameters (the bias tables); the activation gradients stay on the
        # device for the layer below
        return [t for t in (pr.d_rab_pos, pr.d_rab_time) if t is not None]

    def oracle_step(self, b):
        from oracle import oracle as O
        d = self.dropout()
        O.backward(b, o=O.forward(b, dropout=d)["o"], dropout=d)

    def cpu_samples(self, batches):
        return [sub_batch(b, 16) for b in batches], "fwd+bwd of the first 16 of the 64 sequences of a batch"

    def shrink_samples(self, samples, frac, what):
        """Each sample cut to its longest prefix of sequences with at most frac
        of its useful FLOPs (at least one sequence)."""
        out = []
        for b in samples:
            full, keep = self.flops(b)[2], 1
            for n in range(2, b.B + 1):
                if self.flops(sub_batch(b, n))[2] <= frac * full:
                    keep = n
            out.append(sub_batch(b, keep))
        return out, f"{what}, each cut to the prefix of sequences with <= {frac:.2f} of its FLOPs (time budget)"

    def config(self):
        return {"batches": N_SEEDS, "seeds": f"0..{N_SEEDS - 1} (+rank*{N_SEEDS})",
                "l2": "inputs larger than L2: 16 distinct resident batches taken in turn",
                "planner": ("one launch per step (the forward plans the backward too)" if self.plan_once
                            else "one launch per call")}


class LayerWorkload(AttentionWorkload):
    """The full HSTU layer: 8 sequences of U[8192, 32768] history + 128
    candidates, D = 512 (4 heads of 128); x W1 -> SiLU -> attention -> y W2 + x,
    forward and backward."""
    name = "layer"
    metric = "HSTU layer useful TFLOP/s (fwd+bwd: attention + the two projections)"
    description = ("layer: 8 jagged sequences, history U[8192,32768] + 128 candidates, D=512 = 4 heads x 128, "
                   "BF16 x/W1/W2, FP32 outputs; Z1 = x W1, SiLU split U|V|Q|K, causal + candidate mask, "
                   "position + time rab, LayerNorm gate, out = x + y W2; forward + backward")
    n_batches = 2

    def batches(self, rank):
        return [synth.layer(rank * 2 + s) for s in range(2)]

    def problem(self, b, dev):
        from hstu_jagged_attention_02_gb300.layer import LayerProblem
        return LayerProblem(b, device=dev, dropout=self.dropout())

    def flops(self, b):
        f, bw = useful_flops(b)
        D = b.H * b.d_v
        gemm = 3 * (2 * b.T * D * 4 * D + 2 * b.T * D * D)   # forward 2 GEMMs, backward 4
        return f, bw, f + bw + gemm

    def host_io(self, pr):
        ins = [t for t in (pr.offsets, pr.num_targets, pr.num_contexts, pr.timestamps, pr.rab_pos,
                           pr.rab_time, pr.x, pr.w1, pr.w2, pr.dout) if t is not None]
        outs = [t for t in (pr.out, pr.dx, pr.dw1, pr.dw2, pr.d_rab_pos, pr.d_rab_time) if t is not None]
        return ins, outs

    def result(self, pr):
        # the layer's parameter gradients (W1, W2, the bias tables)
        return [t for t in (pr.dw1, pr.dw2, pr.d_rab_pos, pr.d_rab_time) if t is not None]

    def oracle_step(self, b):
        from oracle import oracle as O
        O.layer_backward(b, dropout=self.dropout())

    def cpu_samples(self, batches):
        return ([synth.layer(100 + s, n_lo=1024, n_hi=1024, B=1) for s in range(2)],
                "layer fwd+bwd of one sequence of 1024 history + 128 candidates at D=512")

    def shrink_samples(self, samples, frac, what):
        return samples, what   # one sequence per sample already

    def config(self):
        return {"batches": 2, "seeds": "0..1 (+rank*2)",
                "l2": "inputs larger than L2: each batch holds several GB of activations"}


class DeltaWorkload(AttentionWorkload):
    """KV-cached candidate scoring (the delta forward): 32 sequences whose
    2K-8K cached tokens (context + history) are kept as K/V, each scoring 128
    new candidates; forward only."""
    name = "delta"
    metric = "HSTU delta-forward useful TFLOP/s (KV-cached candidates vs history)"
    description = ("delta: 32 sequences, cached history U[2048,8192] tokens (K/V kept), 128 candidates each, "
                   "4 heads x 128, BF16 in / FP32 out, candidates see the cache and themselves, position + time "
                   "rab, LayerNorm gate; forward only")
    n_batches = 4
    has_backward = False

    def batches(self, rank):
        out = []
        for s in range(4):
            rng = np.random.default_rng(1000 + rank * 4 + s)
            hist = rng.integers(2048, 8192, size=32, endpoint=True)
            out.append(synth.make_batch(hist, H=4, d_qk=128, d_v=128, dtype="bf16", num_targets=128,
                                        seed=1000 + rank * 4 + s, backward=False))
        return out

    def problem(self, b, dev):
        from hstu_jagged_attention_02_gb300.delta import DeltaProblem
        return DeltaProblem(b, device=dev)

    def flops(self, b):
        m = b.num_targets.astype(np.int64)
        cached = b.lengths.astype(np.int64) - m
        pairs = int((m * (cached + 1)).sum()) * b.H
        f = 2 * (b.d_qk + b.d_v) * pairs
        return f, 0, f

    def kernel_bytes(self, b, role):
        # cached tokens supply K and V (BF16); candidates read q, k, v and write o (FP32)
        m = int(b.num_targets.sum())
        return (4 * (b.T - m) + 10 * m) * b.H * b.d_qk

    def host_io(self, pr):
        # the KV cache (cached K, V and their timestamps) is resident device
        # state between requests; a request uploads its candidates
        ins = [t for t in (pr.cand_offsets, pr.cache_offsets, pr.cand_ts, pr.rab_pos, pr.rab_time,
                           pr.q, pr.k, pr.v, pr.u) if t is not None]
        return ins, [pr.o, pr.y]

    def result(self, pr):
        return [pr.y]   # the candidates' outputs: the response to the request

    def oracle_step(self, b):
        from oracle import oracle as O
        from hstu_jagged_attention_02_gb300.delta import split_rows
        rows = np.zeros(b.T, bool)
        rows[split_rows(b)[1]] = True
        O.forward(b, rows=rows)

    def cpu_samples(self, batches):
        return [sub_batch(b, 2) for b in batches], "delta forward of the first 2 of 32 sequences of a batch"

    def config(self):
        return {"batches": 4, "seeds": "1000..1003 (+rank*4)",
                "l2": "inputs larger than L2: each batch holds ~300 MB of cached K/V"}


WORKLOADS = {"heavy_tailed": AttentionWorkload, "layer": LayerWorkload, "delta": DeltaWorkload}


# ------------------------------------------------------------ CPU oracle arm

def time_oracle(wl, samples, budget_s):
    """Runs the FP64 oracle over samples until budget_s is spent; returns
    (useful flops, seconds, batches used, threads)."""
    from oracle import oracle as O
    done_flops, t0, used = 0, time.perf_counter(), 0
    for b in samples:
        wl.oracle_step(b)
        done_flops += wl.flops(b)[2]
        used += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return done_flops, time.perf_counter() - t0, used, O.num_threads()


def sub_batch(b, n_seq):
    """The first n_seq sequences of a batch (a bounded sample of the workload)."""
    end = int(b.offsets[n_seq])
    sl = slice(0, end)
    return synth.Batch(
        name=b.name, seed=b.seed, dtype=b.dtype, B=n_seq, H=b.H, d_qk=b.d_qk, d_v=b.d_v,
        lengths=b.lengths[:n_seq].copy(), offsets=b.offsets[: n_seq + 1].copy(),
        num_targets=None if b.num_targets is None else b.num_targets[:n_seq].copy(),
        num_contexts=None if b.num_contexts is None else b.num_contexts[:n_seq].copy(),
        timestamps=None if b.timestamps is None else b.timestamps[sl].copy(),
        q=b.q[sl], k=b.k[sl], v=b.v[sl], u=None if b.u is None else b.u[sl],
        dy=None if b.dy is None else b.dy[sl], rab_pos=b.rab_pos, rab_time=b.rab_time,
        alpha=b.alpha, max_seq_len=b.max_seq_len, norm=b.norm, eps=b.eps)


REFERENCE_BUDGET_S = 150.0   # the whole --impl reference run, warm-up included


def run_reference(args, wl, rank, world):
    if rank != 0:
        return
    from oracle import oracle as O
    samples, what = wl.cpu_samples(wl.batches(0))
    # The first warm-up step times the sample; if K + W steps of it would
    # overrun the budget, every step takes a smaller sample (fewer sequences,
    # sized by allowed pairs, which the oracle's time follows).
    n_steps = args.steps + max(args.warmup, 1)
    t0 = time.perf_counter()
    wl.oracle_step(samples[0])
    t_first = time.perf_counter() - t0
    cost = [wl.flops(b)[2] for b in samples]
    est = t_first / cost[0] * sum(cost[k % len(samples)] for k in range(n_steps))
    if est > REFERENCE_BUDGET_S:
        samples, what = wl.shrink_samples(samples, REFERENCE_BUDGET_S / est, what)
    for w in range(1, args.warmup):
        wl.oracle_step(samples[w % len(samples)])
    flops, t0 = 0, time.perf_counter()
    for k in range(args.steps):
        b = samples[k % len(samples)]
        wl.oracle_step(b)
        flops += wl.flops(b)[2]
    dt = time.perf_counter() - t0
    val = flops / dt / 1e12
    line = {"impl": "reference", "metric": wl.metric, "value": val, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict({"workload": wl.description, "sample": what}, **wl.config()),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": O.num_threads(), "kind": "oracle",
                             "sample": f"per step: {what}"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def run_gpu(args, wl, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from hstu_jagged_attention_02_gb300 import binding as C

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    batches = wl.batches(rank)
    nb = len(batches)
    probs = [wl.problem(b, dev) for b in batches]
    flops = [wl.flops(b) for b in batches]
    stream = torch.cuda.current_stream()

    # The timed steps record the library's kernel events around the dominant
    # kernel only: each recorded pair costs the step 2-4 us (an event between
    # two launches also turns a programmatic launch edge into a plain stream
    # dependency).  The other attention kernel is timed in a separate pass.
    dom = "bwd" if wl.has_backward else "fwd"

    def step(i, ev=None, roles=(dom,)):
        pr = probs[i % nb]
        if ev is not None and "fwd" in roles:
            C.hstu_time_next_attention_kernel(ev[0].cuda_event, ev[1].cuda_event)
        pr.forward()
        n = C.hstu_last_launch_count()
        if not wl.has_backward:   # no backward kernel: its interval is reported as 0
            return n
        if ev is not None and "bwd" in roles:
            C.hstu_time_next_attention_kernel(ev[2].cuda_event, ev[3].cuda_event)
        pr.backward()
        return n + C.hstu_last_launch_count()

    t_w = time.perf_counter()
    for w in range(max(args.warmup, 0)):
        step(w)
    torch.cuda.synchronize()
    t_step = (time.perf_counter() - t_w) / max(args.warmup, 1)
    for pr in probs:
        assert pr.device_error() == 0, "device error during warm-up"
    # Soak: untimed steps queued directly before the timed ones, so the clock
    # record covers about args.soak_s seconds of sustained load ending with the
    # timed region (a timed region of a few milliseconds alone falls between
    # two clock samples).
    n_soak = int(min(20000, math.ceil(args.soak_s / max(t_step, 1e-5)))) if args.soak_s > 0 else 0

    # ---- timed region: K steps, kernel events on the launching stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for e4 in evs:   # torch only times events it has recorded once; the library re-records them
        for e in e4:
            e.record(stream)
    # With --graph the K steps are captured once into a CUDA graph (the
    # library's calls, their kernel-timing events and programmatic launch
    # edges included) and the timed region replays it; by default they are
    # launched one by one.
    graph = None
    launches = 0
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for k in range(args.steps):
                    launches += step(k, evs[k])
        torch.cuda.synchronize()
    clock = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clock.start()
    time.sleep(0.3)  # let the sampler start before the load
    clock.mark_load()
    for k in range(n_soak):
        step(k)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for k in range(args.steps):
            launches += step(k, evs[k])
    end.record(stream)
    torch.cuda.synchronize()
    clocks = clock.stop()
    if world > 1:
        dist.barrier()
    elapsed_ms = start.elapsed_time(end)
    dom_i = 2 if dom == "bwd" else 0
    dom_ms = [e[dom_i].elapsed_time(e[dom_i + 1]) for e in evs]
    # the other attention kernel: one untimed pass over the resident batches
    # with its events (the forward of a training step; none for the delta
    # forward, which has no backward)
    # The same pass gives the per-batch spread: events at each step's
    # boundaries (between steps, where no programmatic edge is crossed).
    other_ms = [0.0]
    oev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nb)]
    sev = [torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)]
    for e in [x for e4 in oev for x in e4] + sev:
        e.record(stream)
    sev[0].record(stream)
    for k in range(nb):
        step(k, oev[k], roles=("fwd",) if wl.has_backward else ())
        sev[k + 1].record(stream)
    torch.cuda.synchronize()
    if wl.has_backward:
        other_ms = [e[0].elapsed_time(e[1]) for e in oev]
    per_batch = sorted(flops[k][2] / (sev[k].elapsed_time(sev[k + 1]) * 1e-3) / 1e12 for k in range(nb))
    step_flops = [flops[k % nb] for k in range(args.steps)]
    tot_flops = sum(f[2] for f in step_flops)
    for pr in probs:
        assert pr.device_error() == 0, "device error in the timed region"

    if world > 1:
        from hstu_jagged_attention_02_gb300 import dp
        elapsed_ms, tot_flops = dp.reduce_step_time(elapsed_ms, tot_flops, device=dev)

    # ---- end to end through the C ABI with host buffers
    e2e = run_e2e(args, wl, probs, flops, stream, world)
    e2e["read_back"] = "the step's result: " + ("the candidates' outputs" if not wl.has_backward
                                                 else "the parameter gradients (activation gradients stay on the device)")
    e2e_all = run_e2e(args, wl, probs, flops, stream, world, all_outputs=True)
    e2e["all_outputs"] = {k: e2e_all[k] for k in ("value", "d2h_bytes_per_step", "ms_per_step", "repeats")}

    if rank != 0:
        return
    pk, pk_kind = peaks()
    value = tot_flops / (elapsed_ms * 1e-3) / 1e12
    dom_flops = [f[1] if dom == "bwd" else f[0] for f in step_flops]
    peak_sust = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_burst = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak_bw = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    # algorithmic bytes of the kernel per launch: forward reads q, k, v (BF16) and
    # writes o (FP32); backward reads q, k, v and dO as a BF16 pair and writes dk,
    # dv and the dq reduction (FP32)
    dom_bytes = [wl.kernel_bytes(batches[k % nb], dom) for k in range(args.steps)]
    secs = sum(dom_ms) * 1e-3
    t_tensor = sum(dom_flops) / (peak_sust * 1e12)
    t_hbm = sum(dom_bytes) / (peak_bw * 1e9)
    tr = traffic_record(f"{wl.name}:{dom}")
    # DRAM bytes of one launch, from the committed ncu capture of one batch,
    # scaled to this run's mean batch by the token count
    mean_tokens = float(np.mean([batches[k % nb].T for k in range(args.steps)]))
    traffic = tr["dram_bytes_per_token"] * mean_tokens if tr else None
    common = {"traffic": traffic, "kernel": f"attention {dom} kernel",
              "traffic_source": (f"ncu capture `{tr['capture']}` of {tr['capture_tokens']} tokens, sources "
                                 f"{tr['sources_sha']} (per-token DRAM bytes x {mean_tokens:.0f} tokens)" if tr else
                                 "no capture on the current kernel sources"),
              "avg_launch_ms": sum(dom_ms) / len(dom_ms), "share_of_step": sum(dom_ms) / elapsed_ms,
              "algorithmic_bytes_per_launch": sum(dom_bytes) / len(dom_bytes),
              "useful_flops_per_launch": sum(dom_flops) / len(dom_flops)}
    if t_tensor >= t_hbm:
        achieved = sum(dom_flops) / secs / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_sust, "unit": "TFLOP/s",
                    "frac": achieved / peak_sust,
                    "peak_source": f"{pk_kind} bf16_tflops_sustained (kernel timed inside the step loop)"}
    else:
        achieved = sum(dom_bytes) / secs / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak_bw, "unit": "GB/s",
                    "frac": achieved / peak_bw, "peak_source": f"{pk_kind} hbm_gbs"}
    roofline.update(common)
    # CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        samples, what = wl.cpu_samples(batches)
        cf, cdt, used, cores = time_oracle(wl, samples, budget_s=args.cpu_budget)
        cpu = {"value": cf / cdt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{used} x {what}", "seconds": cdt}
    cfg = {"workload": wl.description}
    cfg.update(wl.config())
    cfg["launch"] = ("the K timed steps captured once as a CUDA graph and replayed" if args.graph
                     else "stream launches")
    if wl.dropout_p:
        cfg["dropout_p"] = wl.dropout_p
    cfg.update({"per_rank_batches": nb, "mean_tokens_per_batch": float(np.mean([b.T for b in batches]))})
    line = {"metric": wl.metric, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": cfg,
            "pct_of_bf16_peak": 100.0 * value / peak_burst,
            "peak_bf16_tflops": {"burst": peak_burst, "sustained": peak_sust, "source": pk_kind},
            "fwd_kernel_ms_avg": (sum(dom_ms) / len(dom_ms) if dom == "fwd" else sum(other_ms) / len(other_ms)),
            "bwd_kernel_ms_avg": (sum(dom_ms) / len(dom_ms) if dom == "bwd" else 0.0),
            "kernel_times": (f"{dom}: events around every launch in the timed region; "
                             + ("fwd: a separate untimed pass over the resident batches" if dom == "bwd"
                                else "no backward kernel")),
            "per_batch": {"unit": UNIT, "min": per_batch[0], "median": statistics.median(per_batch),
                          "max": per_batch[-1],
                          "note": "each resident batch once, in a separate untimed pass with step-boundary events"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": dict(clocks, span=f"{n_soak} untimed steps queued directly before the timed ones, then the timed steps")}
    print(json.dumps(line), flush=True)


def run_e2e(args, wl, probs, flops, stream, world, all_outputs=False):
    """Same metric through the public C ABI with pinned host buffers: each step
    copies its inputs host -> device, runs forward + backward and copies the
    step's result back: the parameter gradients of a training step (the
    activation gradients stay on the device for the layer below), the
    candidates' outputs of an inference request, or with all_outputs every
    output and gradient.  The copies run on two copy streams and overlap the compute
    of the neighbouring steps, as a training loop's input prefetch and result
    drain would (each batch has its own device buffers; a step's upload waits
    until the download of the previous step that used those buffers is done,
    and its compute waits for its upload).  The timed region runs from before
    the first upload to after the last download; it covers at least 100 ms of
    steps and is timed three times (the median is the value, all three are
    reported).  Returns the e2e dict."""
    import torch
    nb = len(probs)
    hosts = []
    for pr in probs:
        ins, outs = wl.host_io(pr)
        if not all_outputs:
            outs = wl.result(pr)
        h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in ins]
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        hosts.append((ins, h_in, outs, h_out))
    bi = sum(t.numel() * t.element_size() for t in hosts[0][1])
    bo = sum(t.numel() * t.element_size() for t in hosts[0][3])
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    drained = [None] * nb          # event: the last download from batch slot j is done

    def one(i):
        j = i % nb
        pr = probs[j]
        ins, h_in, outs, h_out = hosts[j]
        with torch.cuda.stream(up):
            if drained[j] is not None:
                up.wait_event(drained[j])
            for d, h in zip(ins, h_in):
                d.copy_(h, non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(up)
        stream.wait_event(uploaded)
        pr.forward(stream)
        if wl.has_backward:
            pr.backward(stream)
        computed = torch.cuda.Event()
        computed.record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed)
            for d, h in zip(outs, h_out):
                h.copy_(d, non_blocking=True)
            drained[j] = torch.cuda.Event()
            drained[j].record(down)

    for w in range(max(args.warmup, 1)):
        one(w)
    torch.cuda.synchronize()

    def timed(k):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        up.wait_stream(stream)
        down.wait_stream(stream)
        for i in range(k):
            one(i)
        stream.wait_stream(down)
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    # The host link and the host thread that issues the copies are shared
    # with the rest of the machine, so a region of a few milliseconds can
    # catch a stall: the region is stretched to at least 100 ms of steps and
    # timed three times, and the median is reported with all three.
    k = args.steps
    ms_first = timed(k)
    if world == 1 and ms_first < 100.0:   # ranks keep one step count
        k = min(2000, max(k, int(k * 100.0 / max(ms_first, 1e-3)) + 1))
    runs = []
    for _ in range(3):
        ms = timed(k)
        fl = sum(flops[i % nb][2] for i in range(k))
        if world > 1:
            from hstu_jagged_attention_02_gb300 import dp
            ms, fl = dp.reduce_step_time(ms, fl, device=torch.device("cuda", torch.cuda.current_device()))
        runs.append((fl / (ms * 1e-3) / 1e12, ms))
    value, ms = sorted(runs)[1]
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": ms / k, "steps": k, "repeats": [round(v, 2) for v, _ in runs]}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--soak-s", type=float, default=1.5,
                    help="seconds of untimed steps queued right before the timed ones, under the clock sampler")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="heavy_tailed", choices=sorted(WORKLOADS),
                    help="heavy_tailed attention (the default line) or the full layer")
    ap.add_argument("--graph", action="store_true",
                    help="capture the timed steps as a CUDA graph and time its replay")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="fused dropout probability on y (heavy_tailed and layer workloads)")
    ap.add_argument("--plan-each-call", action="store_true",
                    help="heavy_tailed: the forward and the backward each run their own planner")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]()
    if args.plan_each_call:
        wl.plan_once = False
    if args.dropout:
        if not wl.has_backward:
            ap.error("--dropout applies to training workloads only")
        wl.dropout_p = args.dropout
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, wl, rank, world)
        else:
            run_gpu(args, wl, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
