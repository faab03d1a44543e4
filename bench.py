#!/usr/bin/env python
"""Benchmark of the GB300 Gated DeltaNet hot path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

One step is one single-layer prefill of the 4096-token workload (16 q/k heads,
32 value heads, d = 128, chunk 64) through the chunked tcgen05 path: the
per-chunk preparation kernel followed by the state-passing kernel.  `value`
is prefill tokens/s over all ranks, device-timed with CUDA events over exactly
K back-to-back steps whose inputs are already in HBM.  Input replicas are
rotated so that the data each step reads (about 4 x 97 MiB in total) does not
sit in the 126 MiB L2 from the previous step.

Also measured and reported on the same line:
  * per-kernel CUDA-event durations inside the timed region and the roofline
    of the dominant kernel (algorithmic FLOPs / duration against the measured
    bf16 tensor peak);
  * the 30-layer batch-1 decode step (us per step and HBM GB/s of the state
    read+write, rotating 5 replicas of the 60 MiB state), as one batched
    launch per step and as 30 single-layer launches per step;
  * the direct-scan prefill on the same 4K workload (the scan vs. blocks
    comparison);
  * e2e: the same prefill metric through the library's host-buffer call
    gdn_prefill_host (pinned host -> device copies of the inputs and device ->
    host copies of the outputs and final state inside the timed region, every
    step), three calls in flight on three streams so that copies and kernels of
    consecutive steps overlap; the serial figure (one stream) is reported too;
  * cpu_baseline: the fp64 CPU oracle timed on this host's cores;
  * SM clocks sampled with nvidia-smi while the GPU is under load.

--impl reference times the CPU oracle (the only reference this method has) on
the same workload, metric and unit.  Multi-GPU runs (torchrun) run independent
replicas of the workload on every rank (no collective on the data path) and
report the aggregate over ranks with max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN prefill tok/s @4K; decode step µs (30 layers); % tensor/HBM roofline"
UNIT = "tok/s"
T_TOKENS = 4096
HK, HV, D, C = 16, 32, 128, 64
WORKLOAD = ("single-layer Gated DeltaNet prefill, 1 sequence x 4096 tokens, 16 q/k heads, 32 v heads, "
            "dk=dv=128, chunk 64, bf16 q/k/v, fp32 gates and state, bf16 out")

# Algorithmic work per token per value head (dense-equivalent, no split-precision passes):
#   preparation: K K^T and Q K^T (4 C d) + triangular solve (C^2 / 3) + P = K^T Gamma T (2 d C) + R = Aqk T (2 C^2)
#   state pass:  Q S^T and K S^T (4 d^2) + P X (2 d^2) + R X (2 C d)
FLOPS_PREP = 4 * C * D + C * C / 3 + 2 * D * C + 2 * C * C
FLOPS_PASS = 4 * D * D + 2 * D * D + 2 * C * D
FLOPS_SCAN = 6 * D * D
DECODE_LAYERS = 30
DECODE_STATE_BYTES = DECODE_LAYERS * HV * D * D * 4 * 2   # fp32 state read + written per 30-layer step


# --------------------------------------------------------------------------- distributed helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def aggregate(local_seconds: float, local_units: float, group=None):
    """Max of the timed seconds and sum of the units over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_seconds, local_units
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------- peaks and clocks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="gdn_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path:
                try:
                    os.unlink(self.path)
                except OSError:
                    pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        loaded = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in loaded if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": reasons, "samples": len(rows),
                "samples_under_load": len(loaded),
                "power_w_max": max((num(r[3]) or 0) for r in loaded)}


# --------------------------------------------------------------------------- workloads
def make_prefill_replicas(n_rep: int, dev):
    import torch
    from gated_deltanet_linear_03_gb300 import gdn, synth
    inp = synth.prefill_4k()
    cu_host = inp.cu_seqlens.tolist()
    host = {"q": inp.q, "k": inp.k, "v": inp.v, "la": inp.log_alpha, "b": inp.beta, "cu": inp.cu_seqlens}
    base = {k: v.to(dev) for k, v in host.items()}
    ws_bytes = gdn.workspace_size(1, T_TOKENS, HK, HV, D, D, cu_host, "chunked")
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)       # one workspace, reused every step
    plans = []
    for r in range(n_rep):
        t = base if r == 0 else {k: v.clone() for k, v in base.items()}
        plans.append(gdn.PrefillPlan(t["q"], t["k"], t["v"], t["la"], t["b"], t["cu"], workspace=ws,
                                     cu_seqlens_host=cu_host))
    return inp, host, plans, cu_host


def time_prefill_steps(plans, steps, warmup, stream):
    """Exactly `steps` prefill steps, events only around them (the timed region of `value`); then the same
    number of steps again with events between the two kernels, for the per-kernel durations."""
    import torch
    R = len(plans)
    for i in range(warmup):
        plans[i % R].run(stream=stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            p = plans[i % R]
            p.run_phase("prep", stream=stream)
            p.run_phase("pass", stream=stream)
        end.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    # per-kernel split (not part of the timed region above)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            p = plans[i % R]
            ev[i][0].record(stream)
            p.run_phase("prep", stream=stream)
            ev[i][1].record(stream)
            p.run_phase("pass", stream=stream)
            ev[i][2].record(stream)
    torch.cuda.synchronize()
    prep = [e[0].elapsed_time(e[1]) for e in ev]
    pas = [e[1].elapsed_time(e[2]) for e in ev]
    return total_ms, statistics.mean(prep), statistics.mean(pas)


def soak(fn, seconds: float):
    import torch
    t0 = time.time()
    while time.time() - t0 < seconds:
        for _ in range(20):
            fn()
        torch.cuda.synchronize()


def time_decode(dev, stream, steps=256, n_rep=5, norm=False):
    """30-layer decode steps (one batched launch per step over the 30 layer states), rotating n_rep
    state replicas so that no step finds its 60 MiB of state in L2.  The `steps` launches are captured
    in one CUDA graph, as a model's decode step would be, so host launch overhead is not measured."""
    import torch
    from gated_deltanet_linear_03_gb300 import gdn, synth
    di = synth.decode_30(steps=steps)
    states = [di.state.to(dev) for _ in range(n_rep)]
    q, k, v = di.q.to(dev), di.k.to(dev), di.v.to(dev)
    la, b = di.log_alpha.to(dev), di.beta.to(dev)
    out = torch.empty(DECODE_LAYERS, HV, D, dtype=torch.bfloat16, device=dev)
    w = torch.linspace(0.5, 2.0, D, device=dev) if norm else None

    def step(i):
        gdn.decode_step(states[i % n_rep], q[i], k[i], v[i], la[i], b[i], out=out, stream=stream, norm_weight=w)
    with torch.cuda.stream(stream):
        for i in range(5):
            step(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            step(i)
    with torch.cuda.stream(stream):
        graph.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        graph.replay()
        e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / steps


def time_decode_per_layer(dev, stream, steps=64, n_rep=5):
    """The same 30-layer decode step issued as 30 single-layer launches (one per layer, as a model that
    interleaves the recurrence with its other layers would), captured in one CUDA graph."""
    import torch
    from gated_deltanet_linear_03_gb300 import gdn, synth
    di = synth.decode_30(steps=steps)
    states = [di.state.to(dev) for _ in range(n_rep)]
    q, k, v = di.q.to(dev), di.k.to(dev), di.v.to(dev)
    la, b = di.log_alpha.to(dev), di.beta.to(dev)
    out = torch.empty(DECODE_LAYERS, HV, D, dtype=torch.bfloat16, device=dev)

    def step(i):
        st = states[i % n_rep]
        for l in range(DECODE_LAYERS):
            gdn.decode_step(st[l:l + 1], q[i, l:l + 1], k[i, l:l + 1], v[i, l:l + 1], la[i, l:l + 1],
                            b[i, l:l + 1], out=out[l:l + 1], stream=stream)
    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            step(i)
    with torch.cuda.stream(stream):
        graph.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        graph.replay()
        e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / steps


def time_qk_prep(dev, stream, iters=20):
    """The 4K layer from raw q/k projections: L2 normalisation and q scaling fused into the kernels
    (qk_norm), against the same done as a separate PyTorch pass before the plain call; then also from raw
    gate projections (log_alpha = -c softplus(a + b), beta = sigmoid(y) formed in the kernels), against
    PyTorch computing q/k and the gates before the plain call."""
    import torch
    import torch.nn.functional as F
    from gated_deltanet_linear_03_gb300 import gdn, synth
    inp = synth.prefill_inputs([T_TOKENS], hk=HK, hv=HV, dk=D, dv=D, seed=1001, raw_qk=True)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    la, b, cu = inp.log_alpha.to(dev), inp.beta.to(dev), inp.cu_seqlens.to(dev)
    cu_host = inp.cu_seqlens.tolist()
    scale = 1.0 / math.sqrt(D)
    fused = gdn.PrefillPlan(q, k, v, la, b, cu, cu_seqlens_host=cu_host, qk_norm=True, q_scale=scale)
    qn, kn = torch.empty_like(q), torch.empty_like(k)
    plain = gdn.PrefillPlan(qn, kn, v, la, b, cu, cu_seqlens_host=cu_host)

    def separate():
        qn.copy_((F.normalize(q.float(), dim=-1, eps=1e-3) * scale).to(torch.bfloat16))
        kn.copy_(F.normalize(k.float(), dim=-1, eps=1e-3).to(torch.bfloat16))
        plain.run(stream=stream)

    w = torch.linspace(0.5, 2.0, D, device=dev)
    normed = gdn.PrefillPlan(q, k, v, la, b, cu, cu_seqlens_host=cu_host, qk_norm=True, q_scale=scale, norm_weight=w)
    # raw gates with the model recipe's parameters (c = 0.5, b = 2 on every value head)
    rg = synth.prefill_inputs([T_TOKENS], hk=HK, hv=HV, dk=D, dv=D, seed=1001, raw_qk=True, raw_gates="config")
    ga, gy = rg.log_alpha.to(dev), rg.beta.to(dev)
    gc, gbias = rg.gate_scale.to(dev), rg.gate_bias.to(dev)
    gated = gdn.PrefillPlan(q, k, v, ga, gy, cu, cu_seqlens_host=cu_host, qk_norm=True, q_scale=scale,
                            gate_scale=gc, gate_bias=gbias)
    la_s, b_s = torch.empty_like(ga), torch.empty_like(gy)
    plain_g = gdn.PrefillPlan(qn, kn, v, la_s, b_s, cu, cu_seqlens_host=cu_host)

    def separate_gates():
        qn.copy_((F.normalize(q.float(), dim=-1, eps=1e-3) * scale).to(torch.bfloat16))
        kn.copy_(F.normalize(k.float(), dim=-1, eps=1e-3).to(torch.bfloat16))
        la_s.copy_(-gc * F.softplus(ga + gbias))
        b_s.copy_(torch.sigmoid(gy))
        plain_g.run(stream=stream)

    res = {}
    for name, fn in (("fused_us", lambda: fused.run(stream=stream)), ("separate_pass_us", separate),
                     ("fused_with_output_norm_us", lambda: normed.run(stream=stream)),
                     ("fused_with_gates_us", lambda: gated.run(stream=stream)),
                     ("separate_pass_with_gates_us", separate_gates)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(iters):
                fn()
            e0.record(stream)
        torch.cuda.synchronize()
        res[name] = s0.elapsed_time(e0) * 1e3 / iters
    res["workload"] = ("4K layer from raw q/k projections (L2-normalise q and k, q / sqrt(d)); "
                       "fused_with_output_norm_us also fuses the output normalisation; *_with_gates_us start from "
                       "raw gate projections too (log_alpha = -0.5 softplus(a + 2), beta = sigmoid(y))")
    return res


def run_each_kernel_once(args):
    """Two passes of every kernel of the path on the bench workload (chunk preparation, state pass,
    direct scan, 30-layer decode), nothing timed: the target for profiler captures."""
    import torch
    from gated_deltanet_linear_03_gb300 import gdn, synth
    dev = torch.device("cuda", 0)
    gdn.load_library()
    _, _, plans, cu_host = make_prefill_replicas(1, dev)
    t = plans[0].tensors
    plan_scan = gdn.PrefillPlan(t[0], t[1], t[2], t[3], t[4], t[5], algo="scan", cu_seqlens_host=cu_host)
    di = synth.decode_30(steps=2)
    st = di.state.to(dev)
    dq, dk_, dv = di.q.to(dev), di.k.to(dev), di.v.to(dev)
    dla, db = di.log_alpha.to(dev), di.beta.to(dev)
    for i in range(2):
        plans[0].run_phase("prep")
        plans[0].run_phase("pass")
        plan_scan.run()
        gdn.decode_step(st, dq[i], dk_[i], dv[i], dla[i], db[i])
    err = gdn.device_error()
    print(json.dumps({"profile_target": "prep, pass, scan, decode x 2", "device_error": err}))
    return 0 if err == 0 else 1


def run_decode_replicas(args):
    """Profiler target for the decode step's DRAM traffic: the batched 30-layer step on five 60 MiB state
    replicas (300 MiB, more than L2), three untimed warm-up rounds, then five consecutive launches, one per
    replica, as in the timed decode measurement.  Nothing is timed."""
    import torch
    from gated_deltanet_linear_03_gb300 import gdn, synth
    dev = torch.device("cuda", 0)
    gdn.load_library()
    di = synth.decode_30(steps=4)
    states = [di.state.to(dev) for _ in range(5)]
    q, k, v = di.q.to(dev), di.k.to(dev), di.v.to(dev)
    la, b = di.log_alpha.to(dev), di.beta.to(dev)
    out = torch.empty(DECODE_LAYERS, HV, D, dtype=torch.bfloat16, device=dev)
    for r in range(4):
        for i in range(5):
            gdn.decode_step(states[i], q[r], k[r], v[r], la[r], b[r], out=out)
    err = gdn.device_error()
    print(json.dumps({"profile_target": "decode step, 3 warm-up rounds then 5 launches on 5 rotating state replicas",
                      "bytes_per_launch_algorithmic": DECODE_STATE_BYTES, "device_error": err}))
    return 0 if err == 0 else 1


def run_crossover(args):
    """Short-to-long prefill sweep: device time per call of the direct scan and of the chunked path (and, for
    a few tokens, of that many batched decode steps) for N sequences of T tokens each, continuing from a
    nonzero state as a speculative verify or a prompt segment would.  Each call is replayed from a CUDA
    graph, so host launch overhead is not counted.  Prints one JSON line per (N, T)."""
    import torch
    from gated_deltanet_linear_03_gb300 import gdn, synth
    dev = torch.device("cuda", 0)
    gdn.load_library()
    stream = torch.cuda.Stream(dev)

    def graph_us(fn, reps=20):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            g.replay()
            e0.record(stream)
        torch.cuda.synchronize()
        return s0.elapsed_time(e0) * 1e3 / reps

    for n in (1, 8):
        for t in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096):
            inp = synth.prefill_inputs([t] * n, seed=1005, init_std=0.02)
            d = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens)]
            s0 = inp.init_state.to(dev)
            cu = inp.cu_seqlens.tolist()
            row = {"n_seqs": n, "tokens_per_seq": t}
            for algo in ("scan", "chunked"):
                plan = gdn.PrefillPlan(*d, init_state=s0, algo=algo, cu_seqlens_host=cu)
                row[algo + "_us"] = graph_us(lambda: plan.run(stream=stream))
            if t <= 8:
                st = s0.clone()
                q = d[0].view(n, t, HK, D).transpose(0, 1).contiguous()
                k = d[1].view(n, t, HK, D).transpose(0, 1).contiguous()
                v = d[2].view(n, t, HV, D).transpose(0, 1).contiguous()
                la = d[3].view(n, t, HV).transpose(0, 1).contiguous()
                b = d[4].view(n, t, HV).transpose(0, 1).contiguous()
                out = torch.empty(n, HV, D, dtype=torch.bfloat16, device=dev)

                def steps():
                    for i in range(t):
                        gdn.decode_step(st, q[i], k[i], v[i], la[i], b[i], out=out, stream=stream)
                row["decode_steps_us"] = graph_us(steps)
            row["best"] = min((k for k in row if k.endswith("_us")), key=lambda k: row[k])[:-3]
            print(json.dumps(row), flush=True)
    return 0


def time_scan(plan_scan, stream, iters=5):
    import torch
    with torch.cuda.stream(stream):
        plan_scan.run(stream=stream)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(iters):
            plan_scan.run(stream=stream)
        e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters


def time_plan(plan, stream, iters):
    """Device time (ms) of one call of a prefill plan: one untimed call, then the mean of `iters`."""
    import torch
    with torch.cuda.stream(stream):
        plan.run(stream=stream)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(iters):
            plan.run(stream=stream)
        e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / iters


def time_long_context(dev, stream, decode_steps=64):
    """The 128K-token single-layer prefill (model shape and gates), by the chunked path and by the direct
    scan on the same inputs, each emitting the final state; then `decode_steps` batch-1 decode steps that
    continue from the chunked path's final state (one layer, captured in one CUDA graph).  The inputs are
    drawn on the device (same recipe, its own seed stream): drawing 3 GiB on the host takes minutes."""
    import torch
    from gated_deltanet_linear_03_gb300 import gdn, synth
    T = 131072
    inp = synth.prefill_inputs([T], seed=1003, device=dev)
    args = (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens.to(dev))
    res = {"workload": "1 sequence x 131072 tokens, 16 q/k heads, 32 v heads, d=128, bf16 q/k/v, "
                       "final state emitted",
           "protocol": "chunked and scan runs interleaved (chunked, scan, chunked, scan, ...), 3 of each after one "
                       "untimed run of each; medians"}
    plans = {algo: gdn.PrefillPlan(*args, algo=algo, cu_seqlens_host=[0, T]) for algo in ("chunked", "scan")}
    times = {"chunked": [], "scan": []}
    for algo in ("chunked", "scan"):
        time_plan(plans[algo], stream, 1)
    for _ in range(3):   # alternate the two paths so that clock or thermal drift affects both alike
        for algo in ("chunked", "scan"):
            times[algo].append(time_plan(plans[algo], stream, 1))
    for algo in ("chunked", "scan"):
        ms = statistics.median(times[algo])
        res[algo] = {"ms": ms, "tok_per_s": T / (ms * 1e-3), "runs_ms": times[algo]}
    state = plans["chunked"].final_state.clone()
    del plans
    res["chunked_over_scan_speedup"] = res["scan"]["ms"] / res["chunked"]["ms"]
    di = synth.decode_inputs(1, decode_steps, seed=1006, device=dev)
    out = torch.empty(1, HV, D, dtype=torch.bfloat16, device=dev)

    def step(i):
        gdn.decode_step(state, di.q[i], di.k[i], di.v[i], di.log_alpha[i], di.beta[i], out=out, stream=stream)
    work = state.clone()
    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
    torch.cuda.synchronize()
    state.copy_(work)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(decode_steps):
            step(i)
    with torch.cuda.stream(stream):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        graph.replay()
        e.record(stream)
    torch.cuda.synchronize()
    us = s.elapsed_time(e) * 1e3 / decode_steps
    res["decode_after_prefill"] = {"steps": decode_steps, "us_per_step": us, "tok_per_s": 1e6 / us,
                                   "launch": f"{decode_steps} single-layer steps in one CUDA graph, "
                                             "continuing in place from the 128K final state (2 MiB, L2-resident)"}
    return res


def time_ragged(dev, stream, iters=5):
    """Eight packed sequences, lengths log-uniform in [256, 32768] (seed 1004), nonzero initial states,
    by the chunked path and by the direct scan (inputs drawn on the device, as for the 128K case)."""
    from gated_deltanet_linear_03_gb300 import gdn, synth
    lengths = synth.log_uniform_lengths(8, 256, 32768, 1004)
    inp = synth.prefill_inputs(lengths, seed=1004, init_std=0.02, device=dev)
    cu_host = inp.cu_seqlens.tolist()
    args = (inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.cu_seqlens.to(dev))
    T = cu_host[-1]
    res = {"workload": f"8 packed sequences {lengths} ({T} tokens), 16 q/k heads, 32 v heads, d=128, "
                       "initial states ~N(0, 0.02^2)",
           "auto_picks": gdn.resolve_algo(len(lengths), T, HK, HV, D, D, cu_host)}
    for algo in ("chunked", "scan"):
        plan = gdn.PrefillPlan(*args, init_state=inp.init_state, algo=algo, cu_seqlens_host=cu_host)
        ms = time_plan(plan, stream, iters)
        res[algo] = {"ms": ms, "tok_per_s": T / (ms * 1e-3)}
        del plan
    return res


def time_e2e(host, cu_host, dev, stream, steps):
    """End to end through the library's host-buffer call (gdn_prefill_host): every step copies its inputs
    from pinned host memory, runs the prefill and copies the outputs and the final state back to pinned host
    memory.  Pipelined: three plans, each with its own device staging and host outputs, take turns on three
    streams, so one step's copies run under another step's kernels (H2D and D2H use separate copy engines;
    three in flight measured 2% above two).  Also timed serially: one plan on one stream, nothing
    overlapped."""
    import torch
    from gated_deltanet_linear_03_gb300 import gdn
    ins = [host[k].pin_memory() for k in ("q", "k", "v", "la", "b")]
    plans = [gdn.HostPrefillPlan(*ins, cu_host, device=dev) for _ in range(3)]
    streams = [stream, torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

    def timed(n_streams):
        for i in range(3):
            plans[i % n_streams].run(streams[i % n_streams])
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_streams)]
        start.record(streams[0])
        for s in streams[1:n_streams]:
            s.wait_event(start)
        for i in range(steps):
            plans[i % n_streams].run(streams[i % n_streams])
        for e, s in zip(ends, streams):
            e.record(s)
        torch.cuda.synchronize()
        return max(start.elapsed_time(e) for e in ends) / steps
    ms_pipe = timed(3)
    ms_serial = timed(1)
    return T_TOKENS / (ms_pipe * 1e-3), T_TOKENS / (ms_serial * 1e-3), plans[0].h2d_bytes, plans[0].d2h_bytes


def cpu_baseline(budget_s: float = 20.0):
    """The fp64 oracle (as it stands) on the 4K workload, all host cores."""
    import oracle
    from gated_deltanet_linear_03_gb300 import synth
    inp = synth.prefill_4k()
    args = (inp.q.float().numpy(), inp.k.float().numpy(), inp.v.float().numpy(), inp.log_alpha.numpy(),
            inp.beta.numpy(), inp.cu_seqlens.numpy())
    cores = os.cpu_count() or 1
    times = []
    t_start = time.time()
    while True:
        t0 = time.perf_counter()
        oracle.prefill(*args, n_threads=cores)
        times.append(time.perf_counter() - t0)
        if len(times) >= 3 or time.time() - t_start > budget_s:
            break
    t = statistics.median(times)
    # single core: the same 4K layer once, and the 64-token tiny case (2 heads, d = 32) repeated for ~0.5 s
    t0 = time.perf_counter()
    oracle.prefill(*args, n_threads=1)
    t_one = time.perf_counter() - t0
    tiny = synth.tiny_case()
    targs = (tiny.q.float().numpy(), tiny.k.float().numpy(), tiny.v.float().numpy(), tiny.log_alpha.numpy(),
             tiny.beta.numpy(), tiny.cu_seqlens.numpy())
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < 0.5:
        oracle.prefill(*targs, n_threads=1)
        reps += 1
    t_tiny = (time.perf_counter() - t0) / reps
    return {"value": T_TOKENS / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"full 4096-token layer, all 32 value heads, fp64, median of {len(times)} runs "
                      f"({t:.2f} s each)",
            "single_core": {"value": T_TOKENS / t_one, "unit": UNIT, "cores": 1,
                            "sample": f"the same 4K layer once ({t_one:.2f} s)"},
            "single_core_tiny": {"value": 64 / t_tiny, "unit": UNIT, "cores": 1,
                                 "sample": f"64 tokens, 2 heads, d = 32, fp32 inputs, {reps} runs"}}


# --------------------------------------------------------------------------- arms
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from gated_deltanet_linear_03_gb300 import synth
    inp = synth.prefill_4k()
    a = (inp.q.float().numpy(), inp.k.float().numpy(), inp.v.float().numpy(), inp.log_alpha.numpy(),
         inp.beta.numpy(), inp.cu_seqlens.numpy())
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle.prefill(*a, n_threads=cores, want_out=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.prefill(*a, n_threads=cores)
    dt = time.perf_counter() - t0
    value = T_TOKENS * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "each step: the full 4096-token layer, all 32 value heads, fp64"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_gb300(args):
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    from gated_deltanet_linear_03_gb300 import gdn
    gdn.load_library()
    stream = torch.cuda.Stream(dev)
    peaks = load_peaks()

    n_rep = 4
    inp, host, plans, cu_host = make_prefill_replicas(n_rep, dev)
    plan_scan = gdn.PrefillPlan(plans[0].tensors[0], plans[0].tensors[1], plans[0].tensors[2],
                                plans[0].tensors[3], plans[0].tensors[4], plans[0].tensors[5], algo="scan",
                                cu_seqlens_host=cu_host)

    gpu_index = dev.index if dev.index is not None else 0
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[gpu_index])
        except ValueError:
            pass
    with ClockSampler(gpu_index) as clk:
        with torch.cuda.stream(stream):
            soak(lambda: plans[0].run(stream=stream), 1.5)
        total_ms, prep_ms, pass_ms = time_prefill_steps(plans, args.steps, args.warmup, stream)
        decode_us = time_decode(dev, stream)
        decode_norm_us = time_decode(dev, stream, norm=True)
        decode_layer_us = time_decode_per_layer(dev, stream)
        scan_ms = time_scan(plan_scan, stream)
        qk_prep = time_qk_prep(dev, stream)
        long_ctx = time_long_context(dev, stream)
        ragged = time_ragged(dev, stream)
    clocks = clk.summary()
    e2e_tps, e2e_serial_tps, h2d, d2h = time_e2e(host, cu_host, dev, stream, max(4, min(args.steps, 20)))
    err = gdn.device_error(stream)

    seconds, units = aggregate(total_ms * 1e-3, float(T_TOKENS * args.steps))
    value = units / seconds
    e2e_secs, e2e_units = aggregate(T_TOKENS / e2e_tps, float(T_TOKENS))

    flops_prep = FLOPS_PREP * T_TOKENS * HV
    flops_pass = FLOPS_PASS * T_TOKENS * HV
    kernels = {
        "chunk_prep_kernel": {"ms": prep_ms, "tflops": flops_prep / (prep_ms * 1e-3) / 1e12},
        "state_pass_kernel": {"ms": pass_ms, "tflops": flops_pass / (pass_ms * 1e-3) / 1e12},
    }
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    ach = kernels[dom]["tflops"]
    traffic = load_traffic(dom)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": traffic,
                "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)",
                "flops_per_launch": flops_prep if dom == "chunk_prep_kernel" else flops_pass}
    # the whole prefill call (both kernels) against both rooflines: dense-equivalent FLOPs and the algorithmic
    # bytes (q, k, v, gates read once, outputs written once, the final state written; no initial state)
    step_s = total_ms * 1e-3 / args.steps
    call_bytes = T_TOKENS * (2 * HK * D * 2 + HV * D * 2 + 2 * HV * 4 + HV * D * 2) + HV * D * D * 4
    roofline["whole_call"] = {
        "tflops": (flops_prep + flops_pass) / step_s / 1e12,
        "frac_tensor": (flops_prep + flops_pass) / step_s / 1e12 / peaks["bf16_tflops"],
        "hbm_gbs": call_bytes / step_s / 1e9, "frac_hbm": call_bytes / step_s / 1e9 / peaks["hbm_gbs"],
        "bytes": call_bytes, "flops": flops_prep + flops_pass}
    dec_gbs = DECODE_STATE_BYTES / (decode_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD},
        "setup": {"algo": "chunked (tcgen05)", "parallelism": f"replicas x{world}",
                  "l2": f"{n_rep} rotating input replicas (~{n_rep * 97} MiB) > L2"},
        "roofline": roofline,
        "kernels": kernels,
        "decode": {"workload": "batch-1 decode step, 30 layers x 32 v heads x 128x128 fp32 state, bf16 q/k/v",
                   "us_per_step": decode_us, "hbm_gbs": dec_gbs,
                   "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": dec_gbs / peaks["hbm_gbs"], "traffic": load_traffic("decode_step_kernel")},
                   "l2": "5 rotating state replicas (300 MiB)", "launch": "256 steps replayed as one CUDA graph",
                   "with_output_norm": {"us_per_step": decode_norm_us,
                                        "hbm_gbs": DECODE_STATE_BYTES / (decode_norm_us * 1e-6) / 1e9,
                                        "fused": "root-mean-square output norm with per-channel weight"},
                   "per_layer_launches": {"us_per_step": decode_layer_us,
                                          "hbm_gbs": DECODE_STATE_BYTES / (decode_layer_us * 1e-6) / 1e9,
                                          "launch": "30 single-layer launches per step, 64 steps in one "
                                                    "CUDA graph"}},
        "scan": scan_line(scan_ms, clocks, dev),
        "qk_prep": qk_prep,
        "long_context": long_ctx,
        "ragged": ragged,
        "e2e": {"value": e2e_units / e2e_secs, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "gdn_prefill_host (pinned host inputs and outputs), three plans in turn on three streams",
                "serial_value": e2e_serial_tps},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "device_error": err,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def scan_line(scan_ms, clocks, dev):
    """The direct scan on the 4K layer against the FP32 pipe: 6 d^2 FLOP per token per head on the CUDA cores;
    peak = SMs x 128 FP32 lanes x 2 FLOP (one FMA) x the median SM clock sampled during the run."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
    peak = sms * 128 * 2 * mhz * 1e6 / 1e12
    tflops = FLOPS_SCAN * T_TOKENS * HV / (scan_ms * 1e-3) / 1e12
    return {"tok_per_s": T_TOKENS / (scan_ms * 1e-3), "ms": scan_ms, "fp32_tflops": tflops,
            "roofline": {"bound": "alu", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "peak_source": f"{sms} SMs x 128 FP32 lanes x 2 FLOP x {mhz:.0f} MHz (median SM clock "
                                        "sampled during the run)"}}


def load_traffic(kernel: str):
    """DRAM bytes (read + write) per launch from the committed ncu capture of this kernel, or None
    when there is none or the kernel's source changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
        src = os.path.join(ROOT, "gated_deltanet_linear_03_gb300", "csrc", rec["source"])
        if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != rec["source_sha"]:
            return None
        return rec["bytes"]
    except Exception:
        return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--each-kernel-once", action="store_true",
                    help="run every kernel of the path twice on the bench workload, untimed (profiler target)")
    ap.add_argument("--decode-replicas", action="store_true",
                    help="decode step on 5 rotating state replicas after warm-up, untimed (profiler target)")
    ap.add_argument("--crossover", action="store_true",
                    help="sweep short to long sequences: scan vs chunked (vs decode steps) device time per call")
    args = ap.parse_args(argv)
    if args.each_kernel_once:
        return run_each_kernel_once(args)
    if args.crossover:
        return run_crossover(args)
    if args.decode_replicas:
        return run_decode_replicas(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
