#!/usr/bin/env python3
"""Benchmark of the Q4NX dequant-GEMV hot path on GB300: one JSON line.

Workload (one "step"): a Qwen3-0.6B-shaped decode step at batch 1 -- 28 layers
x 7 q4_1 projections (q 2048x1024, k/v 1024x1024, o 1024x2048, gate/up
3072x1024, down 1024x3072), distinct seeded weights per (layer, matrix),
275.25 MB of chunks, each matrix with its own bf16 N(0,1) activation vector.
Every step streams all weights once (more than the 129 MB L2, so no step
reuses L2-resident weights).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

value      = weight GB/s of the whole job (chunk bytes / s), inputs resident in HBM,
             timed with CUDA events on the launching stream over exactly K steps
             (CUDA-graph replays of the step), max over ranks.
e2e        = the same metric through the public API with host buffers: per step
             the activations go host->device from pinned memory, the step runs,
             the outputs come back device->host (copies on a second stream,
             double-buffered, overlapping the neighbouring steps' launches),
             and the host waits for each step's outputs, one step behind.
roofline   = the dominant kernel (q4nx GEMV): algorithmic bytes per launch
             (chunks + x + y) / mean launch duration, against the measured HBM
             copy bandwidth.
repeats    = the same K-step region timed again back to back (min / median / max).
secondary  = every configuration's kernels timed on their own over rotated weight
             copies (>= 512 MB, back to back): q4_1 1024x1024 GEMV and decode;
             Q4_K 9728x2560 / 2560x9728 GEMV and repack; q4_1 12288x4096 /
             4096x12288 at one token (fraction of the HBM copy peak) and at 64
             tokens (TFLOP/s, fraction of the bytes-or-tensor roofline); the Q8
             lm_head 151936x2560 in both layouts (GEMV, GEMV + top-1, 64-token
             GEMM) and the argmax of 1 and 64 logit rows.
cpu_baseline / --impl reference = the oracle (plain C, binary64, one core)
             on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own replica of the workload (weak
scaling, no collective on the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q4NX fused dequant-GEMV weight GB/s (% of HBM peak); M=64 GEMM TFLOPS"
WORKLOAD = "Qwen3-0.6B-shaped decode layer x28, q4_1, batch 1"
WORKLOAD_ID = 2
CHUNK = synth.CHUNK_BYTES[synth.Q4_1]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _traffic_if_current():
    """DRAM bytes (read + write) of one GEMV launch from the committed ncu capture,
    or None when the kernel's source has changed since that capture."""
    import hashlib

    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tp):
        return None
    with open(tp) as f:
        d = json.load(f)
    h = hashlib.sha256()
    for rel in d.get("source_files", []):
        p = os.path.join(ROOT, rel)
        if not os.path.exists(p):
            return None
        with open(p, "rb") as fh:
            h.update(fh.read())
    return d.get("gemv_q4_1_bytes_per_launch") if h.hexdigest() == d.get("source_sha256") else None


def _matrices():
    """(layer, matrix_id, N, K) of one step."""
    return [(l, mi, n, k) for l in range(synth.QWEN3_06B_LAYERS) for mi, (_, n, k) in enumerate(synth.QWEN3_06B_LAYER)]


def _gen(layer, mi, N, K):
    f, w = synth.workload_weight(WORKLOAD_ID, mi, layer=layer, shape=(N, K))
    x = synth.workload_activations(WORKLOAD_ID, mi, 1, K, layer=layer)[0]
    return w, x


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, fl in enumerate(flags) if fl.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- CPU arms --

def cpu_oracle_sample(mats, gen, budget_s: float, start: int = 0):
    """Run the oracle over matrices of the workload until `budget_s` is spent.
    Returns (weight bytes, seconds, matrices done)."""
    import oracle

    done, nbytes, t_used = 0, 0, 0.0
    i = start
    while t_used < budget_s and done < len(mats):
        l, mi, N, K = mats[i % len(mats)]
        w, x = gen(l, mi, N, K)
        t0 = time.perf_counter()
        oracle.matmul(w, oracle.Q4_1, N, K, x)
        t_used += time.perf_counter() - t0
        nbytes += w.size
        done += 1
        i += 1
    return nbytes, t_used, done


def run_reference(args, rank: int):
    if rank != 0:
        return
    mats = _matrices()
    steps, warm = args.steps, args.warmup
    per_step = max(0.02, min(10.0, 150.0 / (steps + warm)))
    for s in range(warm):
        cpu_oracle_sample(mats, _gen, per_step, start=s)
    tot_b, tot_t, tot_m = 0, 0.0, 0
    for s in range(steps):
        b, t, m = cpu_oracle_sample(mats, _gen, per_step, start=warm + s)
        tot_b += b
        tot_t += t
        tot_m += m
    gbs = tot_b / tot_t / 1e9
    sample = (f"oracle binary64 matvec (plain C, 1 thread) over {tot_m} matrices of the workload "
              f"(~{per_step:.2f} s per step, {tot_b / 1e6:.1f} MB of chunks)")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * tot_t / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": synth.QWEN3_06B_LAYERS, "matrices_per_step": len(mats),
                       "weight_bytes_per_step": sum((n // 32) * (k // 256) * 5120 for _, _, n, k in mats),
                       "kind": "q4_1", "batch": 1, "sample": "bounded per step"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm --

def max_over_ranks(v: float, world: int, device=None) -> float:
    """The largest of every rank's v (each rank's own v when world == 1)."""
    if world <= 1:
        return float(v)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, bytes_per_rank_step: float, steps: int, seconds: float) -> float:
    """Whole-job GB/s: every rank streams its own copy of the step (weak scaling),
    timed by the slowest rank."""
    return world * bytes_per_rank_step * steps / seconds / 1e9


def run_gpu(args, rank: int, world: int):
    import torch

    import dequant_gemv_gb300 as q

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mats = _matrices()

    # inputs: all weights in one device buffer, all x in one, all y in one
    offs, xoffs, yoffs = [], [], []
    wtot = xtot = ytot = 0
    for (_, _, N, K) in mats:
        offs.append(wtot)
        xoffs.append(xtot)
        yoffs.append(ytot)
        wtot += (N // 32) * (K // 256) * CHUNK
        xtot += K
        ytot += N
    wdev = torch.empty(wtot, dtype=torch.uint8, device=dev)
    x_host = torch.empty(xtot, dtype=torch.bfloat16, pin_memory=True)
    for i, (l, mi, N, K) in enumerate(mats):
        w, x = _gen(l, mi, N, K)
        wdev[offs[i]:offs[i] + w.size].copy_(torch.from_numpy(w))
        x_host[xoffs[i]:xoffs[i] + K].copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
    xdev = x_host.to(dev)
    ydev = torch.empty(ytot, dtype=torch.bfloat16, device=dev)
    y_host = torch.empty(ytot, dtype=torch.bfloat16, pin_memory=True)
    weights = [q.Weight(wdev[offs[i]:offs[i] + (N // 32) * (K // 256) * CHUNK], q.Q4NX_Q4_1, N, K)
               for i, (_, _, N, K) in enumerate(mats)]
    xs = [xdev[xoffs[i]:xoffs[i] + K] for i, (_, _, N, K) in enumerate(mats)]
    ys = [ydev[yoffs[i]:yoffs[i] + N] for i, (_, _, N, K) in enumerate(mats)]
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        items = [(weights[i], xs[i], ys[i]) for i in range(len(mats))]
        ws_need = int(q.lib.q4nx_gemv_batch_workspace((q.q4nx_gemv_item * len(items))(
            *[q.q4nx_gemv_item(W.c(), x.data_ptr(), y.data_ptr()) for W, x, y in items]), len(items)))
        ws = torch.zeros(max(ws_need, 1 << 20), dtype=torch.uint8, device=dev)
        # the step: every matrix of the 28 layers in one batched launch
        step_batch = q.GemvBatch(items, "bf16", ws)
        # the same work respecting a decode layer's data dependencies: {q,k,v}, {o}, {gate,up}, {down}
        per_layer = []
        for l in range(synth.QWEN3_06B_LAYERS):
            base = 7 * l
            for grp in ((0, 1, 2), (3,), (4, 5), (6,)):
                per_layer.append(q.GemvBatch([items[base + j] for j in grp], "bf16", ws))
        # the same schedule with the matrices that read the same activations
        # stored as one weight (q|k|v and gate|up: adjacent chunk arrays, same
        # K), so that each phase is one matrix on one x; k, v and up then read
        # q's and gate's activations, as in a real layer
        per_layer_merged = []
        for l in range(synth.QWEN3_06B_LAYERS):
            base = 7 * l
            for grp in ((0, 1, 2), (3,), (4, 5), (6,)):
                i0, i1 = base + grp[0], base + grp[-1]
                N = sum(mats[base + j][2] for j in grp)
                K = mats[i0][3]
                Wm = q.Weight(wdev[offs[i0]:offs[i1] + (mats[i1][2] // 32) * (K // 256) * CHUNK], q.Q4NX_Q4_1, N, K)
                per_layer_merged.append(q.GemvBatch([(Wm, xs[i0], ydev[yoffs[i0]:yoffs[i0] + N])], "bf16", ws))
    torch.cuda.synchronize()

    def capture(fn):
        with torch.cuda.stream(stream):
            fn()                                     # eager run once (kernel attributes)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    graph = capture(step_batch)                 # one step (used for the end-to-end leg)
    # the end-to-end leg's second set of device x / y buffers (double buffering)
    xdev2 = torch.empty_like(xdev)
    ydev2 = torch.empty_like(ydev)
    y_host2 = torch.empty(ytot, dtype=torch.bfloat16, pin_memory=True)
    step_batch2 = q.GemvBatch([(weights[i], xdev2[xoffs[i]:xoffs[i] + K], ydev2[yoffs[i]:yoffs[i] + N])
                               for i, (_, _, N, K) in enumerate(mats)], "bf16", ws)
    graph2 = capture(step_batch2)
    # the timed loop replays graphs of several consecutive steps, so that each
    # step's launch overlaps the previous one (programmatic dependent launch)
    # as in a decode loop; a step is still one launch over all 196 matrices
    per_graph = max(1, min(8, args.steps))
    graph_many = capture(lambda: [step_batch() for _ in range(per_graph)])
    rem = args.steps % per_graph
    graph_rem = capture(lambda: [step_batch() for _ in range(rem)]) if rem else None
    launches_per_step = 1

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # warm-up
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
        graph_many.replay()
    stream.synchronize()

    gpu_uuid = None
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    clocks = ClockSampler(gpu_uuid)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)                              # let the sampler start before the timed region
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps // per_graph):
            graph_many.replay()
        if graph_rem is not None:
            graph_rem.replay()
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    ms_per_step = ms / args.steps
    value = job_throughput(world, wtot, args.steps, ms / 1e3)

    # the same K-step region timed again, for its spread (the line's value is the first timing)
    rep_ms = [ms_per_step]
    for _ in range(args.repeats):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        with torch.cuda.stream(stream):
            a_.record(stream)
            for _ in range(args.steps // per_graph):
                graph_many.replay()
            if graph_rem is not None:
                graph_rem.replay()
            b_.record(stream)
        stream.synchronize()
        rep_ms.append(max_over_ranks(a_.elapsed_time(b_), world, dev) / args.steps)
    clk = clocks.stop()

    # other schedules of the same step, for context (not the headline)
    def time_graph(g, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            a.record(stream)
            for _ in range(n):
                g.replay()
            b.record(stream)
        stream.synchronize()
        return a.elapsed_time(b) / n
    alt = {}
    if not args.no_alt:
        g_layer = capture(lambda: [b() for b in per_layer])
        t_layer_ms = time_graph(g_layer, 200)
        alt["per_layer_4_launches_gbs"] = wtot / (t_layer_ms / 1e3) / 1e9
        alt["us_per_layer_dependent"] = t_layer_ms * 1e3 / synth.QWEN3_06B_LAYERS
        g_merged = capture(lambda: [b() for b in per_layer_merged])
        t_merged_ms = time_graph(g_merged, 200)
        alt["us_per_layer_dependent_merged_qkv_gate_up"] = t_merged_ms * 1e3 / synth.QWEN3_06B_LAYERS
        del g_merged
        g_single = capture(lambda: [q.q4nx_gemv(weights[i], xs[i], out=ys[i], ws=ws) for i in range(len(mats))])
        alt["one_launch_per_matrix_gbs"] = wtot / (time_graph(g_single, 100) / 1e3) / 1e9
        del g_layer, g_single

    # roofline of the dominant kernel (every launch of the step is the GEMV)
    alg_bytes_step = wtot + 2 * xtot + 2 * ytot
    launch_us = ms_per_step * 1e3 / launches_per_step
    achieved = alg_bytes_step / launches_per_step / (launch_us * 1e-6) / 1e9
    peak, peak_kind = _peaks()
    traffic = _traffic_if_current()

    # end to end through the public API with host buffers.  Every step copies
    # its activations host -> device from pinned memory and reads its outputs
    # back device -> host, each on a stream of its own and double-buffered, so
    # that step i+1's input copy and step i's output read overlap the GEMV
    # launches on the compute stream; the host waits for each step's outputs
    # one step behind, and for the last step's before the clock stops.
    e2e_steps = max(3, min(args.steps, 200))
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = ((xdev, ydev, y_host, graph), (xdev2, ydev2, y_host2, graph2))

    def e2e_run(n):
        x_ready = [torch.cuda.Event() for _ in range(2)]
        k_done = [torch.cuda.Event() for _ in range(2)]
        y_read = [None, None]
        for i in range(n):
            b = i % 2
            xd, yd, yh, g = bufs[b]
            with torch.cuda.stream(h2d_stream):
                if i >= 2:
                    h2d_stream.wait_event(k_done[b])           # step i-2 has read this x buffer
                xd.copy_(x_host, non_blocking=True)
                x_ready[b].record(h2d_stream)
            with torch.cuda.stream(stream):
                stream.wait_event(x_ready[b])
                g.replay()                                     # (yd's step i-2 outputs reached the host first)
                k_done[b].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(k_done[b])
                yh.copy_(yd, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(d2h_stream)
                y_read[b] = ev
            if i >= 1:
                y_read[1 - b].synchronize()                    # step i-1's outputs are on the host
        y_read[(n - 1) % 2].synchronize()

    e2e_run(4)
    barrier()
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    t_e2e = time.perf_counter() - t0
    t_e2e = max_over_ranks(t_e2e, world, dev)
    e2e_value = job_throughput(world, wtot, e2e_steps, t_e2e)

    secondary = None
    if rank == 0 and not args.no_secondary:
        secondary = secondary_configs(q, Kit(torch, dev, stream))

    cpu = None
    if rank == 0 and not args.no_cpu:
        b, t, m = cpu_oracle_sample(mats, _gen, args.cpu_seconds)
        cpu = {"value": b / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"oracle binary64 matvec (plain C, 1 thread) over the first {m} of the step's "
                         f"{len(mats)} matrices ({b / 1e6:.1f} MB of chunks, {t:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": synth.QWEN3_06B_LAYERS, "matrices_per_step": len(mats),
                       "weight_bytes_per_step": wtot, "kind": "q4_1", "batch": 1,
                       "l2": "inputs larger than L2 (275 MB of weights streamed per step)",
                       "launch": "one q4nx_gemv_batch launch of all 196 matrices per step; CUDA graphs of "
                                 f"{per_graph} consecutive steps, replayed back to back",
                       "us_per_layer": ms_per_step * 1e3 / synth.QWEN3_06B_LAYERS,
                       "us_per_layer_note": "all 28 layers' GEMVs in one launch (independent x per matrix); "
                                            "the dependent schedule ({q,k,v} -> o -> {gate,up} -> down, each "
                                            "phase one batched launch) is other_schedules.us_per_layer_dependent",
                       "other_schedules": alt,
                       "hbm_frac_of_nominal_8tbs": value / 8000.0},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
                         "traffic_source": "stored ncu capture of this kernel (profiles/traffic.json, "
                                           "dram read + write per launch); null when the kernel's sources "
                                           "differ from the captured ones",
                         "bytes_per_launch": alg_bytes_step / launches_per_step,
                         "launch_us": launch_us},
            "repeats": {"n": len(rep_ms), "ms_per_step_min": min(rep_ms),
                        "ms_per_step_median": statistics.median(rep_ms), "ms_per_step_max": max(rep_ms),
                        "note": "the K-step timed region, timed again back to back; value uses the first"},
            "secondary": secondary,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": 2 * xtot,
                    "d2h_bytes_per_step": 2 * ytot},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "clocks_window": "sampled over the timed region and its repeats",
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------ timing kit --

class Kit:
    """Back-to-back timing of launches: CUDA graphs over rotated input copies
    (together at least 512 MB, so that no launch finds its weights in L2),
    CUDA events on the launching stream."""

    def __init__(self, torch, dev, stream):
        self.torch, self.dev, self.stream = torch, dev, stream
        self.hbm, _ = _peaks()
        self.tc_peak = 1971.6
        p = os.path.join(ROOT, "MEASURED_PEAKS.json")
        if os.path.exists(p):
            with open(p) as f:
                self.tc_peak = float(json.load(f).get("bf16_tflops", self.tc_peak))

    @staticmethod
    def copies_for(nbytes):
        return max(2, min(1024, (512 << 20) // max(nbytes, 1) + 1))

    def timeit(self, fns, iters):
        """us per launch of `iters` launches cycling over the callables in `fns` (one per copy)."""
        torch, stream = self.torch, self.stream
        with torch.cuda.stream(stream):
            for f in fns:
                f()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        per_graph = len(fns) * max(1, 64 // len(fns))
        with torch.cuda.graph(g, stream=stream):
            for i in range(per_graph):
                fns[i % len(fns)]()
        reps = max(1, iters // per_graph)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        stream.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * per_graph)

    def dev_bytes(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def dev_bf16(self, bits):
        t = self.torch
        return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(self.dev).view(t.bfloat16)

    def hbm_frac(self, nbytes, us):
        return nbytes / us / 1e3 / self.hbm

    def roofline_us(self, nbytes, flops):
        """The bytes-or-tensor roofline time of one launch (HBM copy peak, bf16 tensor burst peak)."""
        return max(nbytes / (self.hbm * 1e3), flops / (self.tc_peak * 1e6))


def secondary_configs(q, kit):
    """The five configurations' kernels, each timed on its own (rotated weight
    copies, back to back): one-token GEMVs with their fraction of the measured
    HBM copy bandwidth; 64-token GEMMs with TFLOP/s and their fraction of the
    bytes-or-tensor roofline; the decode, repack and top-1 kernels."""
    import ctypes

    torch = kit.torch
    dev = kit.dev
    out = {}

    def weights(kind, N, K, wid, f=None):
        if f is None:
            f, w = synth.make(kind, N, K, synth.rng(wid, 0, 0))
        else:
            f.kind = kind
            w = synth.pack(f)
        base = kit.dev_bytes(w)
        Ws = [q.Weight(base if r == 0 else base.clone(), kind, N, K) for r in range(kit.copies_for(w.size))]
        return f, w.size, Ws

    def gemv(Ws, N, K, nb, wid, out_f32):
        x = kit.dev_bf16(synth.workload_activations(wid, 0, 1, K)[0])
        y = torch.empty(N, dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
        with torch.cuda.stream(kit.stream):
            ws = torch.zeros(int(q.lib.q4nx_gemv_workspace(ctypes.byref(Ws[0].c()))), dtype=torch.uint8, device=dev)
        od = "f32" if out_f32 else "bf16"
        us = kit.timeit([lambda W=W: q.q4nx_gemv(W, x, out=y, out_dtype=od, ws=ws) for W in Ws], 400)
        alg = nb + 2 * K + (4 if out_f32 else 2) * N
        return {"gemv_us": round(us, 3), "gemv_frac": round(kit.hbm_frac(alg, us), 4), "_x": x, "_ws": ws}

    def gemm(Ws, N, K, nb, wid, out_f32, M=64):
        X = kit.dev_bf16(synth.workload_activations(wid, 0, M, K))
        Y = torch.empty((M, N), dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
        with torch.cuda.stream(kit.stream):
            ws = torch.zeros(int(q.lib.q4nx_gemm_workspace(ctypes.byref(Ws[0].c()), M)), dtype=torch.uint8, device=dev)
        od = "f32" if out_f32 else "bf16"
        us = kit.timeit([lambda W=W: q.q4nx_gemm_m64(W, X, out=Y, out_dtype=od, ws=ws) for W in Ws], 200)
        flops = 2.0 * M * N * K
        alg = nb + 2 * M * K + (4 if out_f32 else 2) * M * N
        t_roof = kit.roofline_us(alg, flops)
        return {"gemm_m64_us": round(us, 3), "gemm_m64_tflops": round(flops / us / 1e6, 1),
                "gemm_m64_frac": round(t_roof / us, 4),
                "gemm_m64_bound": "hbm" if alg / (kit.hbm * 1e3) >= flops / (kit.tc_peak * 1e6) else "tensor"}

    def clean(d):
        return {k: v for k, v in d.items() if not k.startswith("_")}

    # 1: q4_1 1024x1024, decode + GEMV
    f, nb, Ws = weights(synth.Q4_1, 1024, 1024, 1)
    d = gemv(Ws, 1024, 1024, nb, 1, False)
    outs = [torch.empty((1024, 1024), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    us = kit.timeit([lambda W=W, o=outs[i % 2]: q.q4nx_decode(W, out=o) for i, W in enumerate(Ws)], 200)
    d.update({"decode_us": round(us, 3), "decode_frac": round(kit.hbm_frac(nb + 2 * 1024 * 1024, us), 4)})
    out["q4_1_1024x1024"] = clean(d)
    del Ws, outs
    # 3: Q4_K GEMV and the repack, both shapes
    for N, K in ((9728, 2560), (2560, 9728)):
        f, nb, Ws = weights(synth.Q4_K, N, K, 3)
        d = gemv(Ws, N, K, nb, 3, False)
        rep = torch.empty((N // 32) * (K // 256) * 5120, dtype=torch.uint8, device=dev)
        us = kit.timeit([lambda W=W: q.q4nx_repack_q4k(W.chunks, N, K, out=rep) for W in Ws], 200)
        d.update({"repack_us": round(us, 3), "repack_frac": round(kit.hbm_frac(nb + rep.numel(), us), 4)})
        out[f"q4k_{N}x{K}"] = clean(d)
        del Ws, rep
    # 4: the 64-token prefill block's matrices (and the same matrices at one token)
    for N, K in ((12288, 4096), (4096, 12288)):
        f, nb, Ws = weights(synth.Q4_1, N, K, 4)
        d = gemv(Ws, N, K, nb, 4, False)
        d.update(gemm(Ws, N, K, nb, 4, False))
        out[f"q4_1_{N}x{K}"] = clean(d)
        del Ws
    # 5: the Q8 lm_head in both code layouts: logits + top-1, one token and 64
    fq = None
    for kind, name in ((synth.Q8_KR, "kr"), (synth.Q8_BLK, "blk")):
        fq, nb, Ws = weights(kind, 151936, 2560, 5, fq)
        d = gemv(Ws, 151936, 2560, nb, 5, True)
        idx1 = torch.empty(1, dtype=torch.int32, device=dev)
        us = kit.timeit([lambda W=W: q.q4nx_gemv_top1(W, d["_x"], out=idx1, ws=d["_ws"]) for W in Ws], 200)
        d.update({"gemv_top1_us": round(us, 3), "gemv_top1_frac": round(kit.hbm_frac(nb + 2 * 2560 + 4, us), 4)})
        d.update(gemm(Ws, 151936, 2560, nb, 5, True))
        out[f"q8_{name}_151936x2560"] = clean(d)
        del Ws, d
    for M in (1, 64):
        L = torch.randn((M, 151936), generator=torch.Generator(device="cpu").manual_seed(M),
                        dtype=torch.float32).to(dev)
        idx = torch.empty(M, dtype=torch.int32, device=dev)
        Ls = [L] + [L.clone() for _ in range(max(1, min(1024, (512 << 20) // L.numel() // 4)))]
        us = kit.timeit([lambda Lm=Lm: q.q4nx_argmax(Lm, out=idx) for Lm in Ls], 400)
        out[f"argmax_{M}x151936"] = {"us": round(us, 3), "frac": round(kit.hbm_frac(4 * M * 151936, us), 4)}
        del Ls, L
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------- suite --

def run_suite(args):
    """One JSON line per (workload, kernel): every kernel of the path timed on
    the workload shapes, rotating through weight copies that together exceed
    512 MB so that no launch finds its weights in L2."""
    import torch

    import dequant_gemv_gb300 as q

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    kit = Kit(torch, dev, stream)
    hbm, tc_peak = kit.hbm, kit.tc_peak
    copies_for, timeit, dev_bytes, dev_bf16 = kit.copies_for, kit.timeit, kit.dev_bytes, kit.dev_bf16

    def emit(d):
        print(json.dumps(d), flush=True)

    cases = [
        (1, "q4_1 1024x1024", synth.Q4_1, 1024, 1024),
        (3, "Q4_K 9728x2560", synth.Q4_K, 9728, 2560),
        (3, "Q4_K 2560x9728", synth.Q4_K, 2560, 9728),
        (4, "q4_1 12288x4096", synth.Q4_1, 12288, 4096),
        (4, "q4_1 4096x12288", synth.Q4_1, 4096, 12288),
        # gate and up of the same block as one weight: their chunk arrays concatenated (tile rows of
        # gate, then of up), one launch for both since they read the same activations
        (4, "q4_1 24576x4096", synth.Q4_1, 24576, 4096),
        (5, "Q8 KR 151936x2560", synth.Q8_KR, 151936, 2560),
        (5, "Q8 BLK 151936x2560", synth.Q8_BLK, 151936, 2560),
        (6, "q4_1 151936x2560", synth.Q4_1, 151936, 2560),     # an lm_head-sized q4_1 matrix (243 MB)
    ]
    only = set(args.only.split(",")) if args.only else None
    want = lambda k: only is None or k in only
    for wid, name, kind, N, K in cases:
        if args.case and args.case not in name:
            continue
        f, w = synth.make(kind, N, K, synth.rng(wid, 0, 0))
        nb = w.size
        R = copies_for(nb)
        base = dev_bytes(w)
        Ws = [q.Weight(base if r == 0 else base.clone(), kind, N, K) for r in range(R)]
        x = dev_bf16(synth.workload_activations(wid, 0, 1, K)[0])
        out_f32 = kind in (synth.Q8_KR, synth.Q8_BLK)
        y = torch.empty(N, dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
        with torch.cuda.stream(stream):
            ws = torch.zeros(max(int(q.lib.q4nx_gemv_workspace(ctypes.byref(Ws[0].c()))), 1 << 16),
                             dtype=torch.uint8, device=dev)
        od = "f32" if out_f32 else "bf16"
        if want("gemv"):
            us = timeit([lambda W=W: q.q4nx_gemv(W, x, out=y, out_dtype=od, ws=ws) for W in Ws], 400)
            alg = nb + 2 * K + (4 if out_f32 else 2) * N
            emit({"suite": "gemv", "workload": name, "M": 1, "us": us, "weight_gbs": nb / us / 1e3,
                  "roofline": {"bound": "hbm", "achieved": alg / us / 1e3, "peak": hbm, "frac": alg / us / 1e3 / hbm},
                  "frac_of_nominal_8tbs": nb / us / 1e3 / 8000.0, "copies": R})
        if wid in (5, 6) and want("top1"):
            # lm_head GEMV fused with top-1 (logits never written) vs the GEMV then the argmax kernel
            idx1 = torch.empty(1, dtype=torch.int32, device=dev)
            yl = torch.empty((1, N), dtype=torch.float32, device=dev)
            us_f = timeit([lambda W=W: q.q4nx_gemv_top1(W, x, out=idx1, ws=ws) for W in Ws], 400)
            us_s = timeit([lambda W=W: (q.q4nx_gemv(W, x, out=yl[0], out_dtype="f32", ws=ws),
                                        q.q4nx_argmax(yl, out=idx1)) for W in Ws], 400)
            alg = nb + 2 * K + 4
            emit({"suite": "gemv_top1", "workload": name, "M": 1, "us": us_f, "us_gemv_then_argmax": us_s,
                  "weight_gbs": nb / us_f / 1e3,
                  "roofline": {"bound": "hbm", "achieved": alg / us_f / 1e3, "peak": hbm, "frac": alg / us_f / 1e3 / hbm}})
        if kind == synth.Q4_1 and wid == 4 and want("pack"):
            # GGUF-type tensor of this shape -> q4_1 chunks (one-off conversion)
            for st, sname in ((synth.SRC_Q4_0, "Q4_0"), (synth.SRC_Q4_1, "Q4_1"), (synth.SRC_F16, "F16")):
                srcb, _ = synth.gguf_tensor(st, N, K, synth.rng(wid, 7, st))
                srcs = [torch.from_numpy(srcb).to(dev) for _ in range(max(2, min(64, (512 << 20) // srcb.size + 1)))]
                pout = torch.empty(nb, dtype=torch.uint8, device=dev)
                us = timeit([lambda sb=sb: q.q4nx_pack_q4_1(sb, st, N, K, out=pout) for sb in srcs], 200)
                alg = srcb.size + nb
                emit({"suite": "pack_q4_1", "workload": f"{sname} {N}x{K} -> q4_1", "us": us,
                      "roofline": {"bound": "hbm", "achieved": alg / us / 1e3, "peak": hbm, "frac": alg / us / 1e3 / hbm}})
                del srcs
        if wid in (1, 3, 4, 5) and want("decode"):
            outs = [torch.empty((N, K), dtype=torch.bfloat16, device=dev) for _ in range(min(R, 2))]
            us = timeit([lambda W=W, o=outs[i % len(outs)]: q.q4nx_decode(W, out=o) for i, W in enumerate(Ws)], 64)
            alg = nb + 2 * N * K
            emit({"suite": "decode", "workload": name, "us": us, "weight_gbs": nb / us / 1e3,
                  "roofline": {"bound": "hbm", "achieved": alg / us / 1e3, "peak": hbm, "frac": alg / us / 1e3 / hbm}})
            del outs
        if kind == synth.Q4_K and want("repack"):
            rep = torch.empty((N // 32) * (K // 256) * 5120, dtype=torch.uint8, device=dev)
            us = timeit([lambda W=W: q.q4nx_repack_q4k(W.chunks, N, K, out=rep) for W in Ws], 400)
            alg = nb + rep.numel()
            emit({"suite": "repack", "workload": name, "us": us,
                  "roofline": {"bound": "hbm", "achieved": alg / us / 1e3, "peak": hbm, "frac": alg / us / 1e3 / hbm}})
        small_ms = {synth.Q4_1: (2, 3, 4, 8, 16), synth.Q4_K: (2, 4), synth.Q8_KR: (2, 4), synth.Q8_BLK: (2,)}
        if ((kind == synth.Q4_1 and wid == 4) or kind == synth.Q4_K or wid == 5) and want("gemm_small_m"):
            # small token blocks (verify windows, multi-token prediction): q4_1 two tokens and
            # Q4_K up to four on the CUDA cores, more (and Q8 from two) on the tensor cores
            for M in small_ms[kind]:
                X = dev_bf16(synth.workload_activations(wid, 0, M, K))
                Y = torch.empty((M, N), dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
                with torch.cuda.stream(stream):
                    gws = torch.zeros(int(q.lib.q4nx_gemm_workspace(ctypes.byref(Ws[0].c()), M)), dtype=torch.uint8,
                                      device=dev)
                us = timeit([lambda W=W: q.q4nx_gemm_m64(W, X, out=Y, out_dtype=od, ws=gws) for W in Ws], 400)
                alg = nb + 2 * M * K + (4 if out_f32 else 2) * M * N
                cores = "cuda" if M <= {synth.Q4_1: 2, synth.Q4_K: 4}.get(kind, 1) else "tensor"
                emit({"suite": "gemm_small_m", "workload": name, "M": M, "path": cores, "us": us,
                      "weight_gbs": nb / us / 1e3,
                      "roofline": {"bound": "hbm", "achieved": alg / us / 1e3, "peak": hbm, "frac": alg / us / 1e3 / hbm}})
        if ((kind == synth.Q4_1 and wid in (4, 6)) or wid == 5) and want("gemm_m64"):
            M = 64
            X = dev_bf16(synth.workload_activations(wid, 0, M, K))
            Y = torch.empty((M, N), dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
            with torch.cuda.stream(stream):
                gws = torch.zeros(int(q.lib.q4nx_gemm_workspace(ctypes.byref(Ws[0].c()), M)), dtype=torch.uint8,
                                  device=dev)
            us = timeit([lambda W=W: q.q4nx_gemm_m64(W, X, out=Y, out_dtype=od, ws=gws) for W in Ws], 400)
            flops = 2.0 * M * N * K
            alg = nb + 2 * M * K + (4 if out_f32 else 2) * M * N
            t_roof = max(alg / (hbm * 1e3), flops / (tc_peak * 1e6))
            emit({"suite": "gemm_m64", "workload": name, "M": M, "us": us, "tflops": flops / us / 1e6,
                  "weight_gbs": nb / us / 1e3,
                  "roofline": {"bound": "hbm" if alg / (hbm * 1e3) >= flops / (tc_peak * 1e6) else "tensor",
                               "roofline_us": t_roof, "frac": t_roof / us, "hbm_peak": hbm, "tensor_peak": tc_peak}})
        if wid == 5 and want("argmax"):
            for M in (1, 64):
                L = torch.randn((M, N), generator=torch.Generator(device="cpu").manual_seed(M), dtype=torch.float32).to(dev)
                idx = torch.empty(M, dtype=torch.int32, device=dev)
                Ls = [L] + [L.clone() for _ in range(max(1, min(1024, (512 << 20) // L.numel() // 4)))]
                us = timeit([lambda Lm=Lm: q.q4nx_argmax(Lm, out=idx) for Lm in Ls], 400)
                emit({"suite": "argmax", "workload": f"logits {M}x{N}", "us": us,
                      "roofline": {"bound": "hbm", "achieved": 4 * M * N / us / 1e3, "peak": hbm,
                                   "frac": 4 * M * N / us / 1e3 / hbm}})
        del Ws, base
        torch.cuda.empty_cache()
    if want("block") and (not args.case or args.case in "prefill block"):
        run_block(args, q, dev, stream, timeit, emit, dev_bytes, dev_bf16, copies_for, hbm, tc_peak)


def run_block(args, q, dev, stream, timeit, emit, dev_bytes, dev_bf16, copies_for, hbm, tc_peak):
    """The 8B-width MLP block as a sequence: gate|up (24576x4096, one merged
    weight) then down (4096x12288), at M = 1 (GEMV) and M = 64 (tensor cores),
    each launch reading the weights of another copy, so the timed sequence
    streams every weight byte from HBM."""
    import torch

    shapes = [(24576, 4096), (4096, 12288)]
    mats = []
    for i, (N, K) in enumerate(shapes):
        f, w = synth.make(synth.Q4_1, N, K, synth.rng(4, 10 + i, 0))
        base = dev_bytes(w)
        R = copies_for(w.size)
        mats.append((N, K, w.size, [q.Weight(base if r == 0 else base.clone(), synth.Q4_1, N, K) for r in range(R)]))
    R = min(len(m[3]) for m in mats)
    nb = sum(m[2] for m in mats)
    for M in (1, 64):
        Xs = [dev_bf16(synth.workload_activations(4, 10 + i, M, K)) for i, (N, K, _, _) in enumerate(mats)]
        Ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (N, K, _, _) in mats]
        with torch.cuda.stream(stream):
            if M == 1:
                ws = torch.zeros(max(int(q.lib.q4nx_gemv_workspace(ctypes.byref(mats[0][3][0].c()))), 1 << 16),
                                 dtype=torch.uint8, device=dev)
            else:
                ws = torch.zeros(max(int(q.lib.q4nx_gemm_workspace(ctypes.byref(m[3][0].c()), M)) for m in mats),
                                 dtype=torch.uint8, device=dev)
        fns = []
        for r in range(R):
            for i, m in enumerate(mats):
                W = m[3][r]
                if M == 1:
                    fns.append(lambda W=W, i=i: q.q4nx_gemv(W, Xs[i][0], out=Ys[i][0], out_dtype="bf16", ws=ws))
                else:
                    fns.append(lambda W=W, i=i: q.q4nx_gemm_m64(W, Xs[i], out=Ys[i], out_dtype="bf16", ws=ws))
        us = timeit(fns, 400) * len(mats)            # per block (one launch per weight)
        flops = sum(2.0 * M * N * K for (N, K, _, _) in mats)
        alg = nb + sum(2 * M * K + 2 * M * N for (N, K, _, _) in mats)
        t_roof = max(alg / (hbm * 1e3), flops / (tc_peak * 1e6))
        emit({"suite": "block", "workload": "prefill block q4_1 8B width: gate|up 24576x4096, down 4096x12288",
              "M": M, "launches": len(mats), "us": us, "weight_gbs": nb / us / 1e3, "tflops": flops / us / 1e6,
              "roofline": {"bound": "hbm" if alg / (hbm * 1e3) >= flops / (tc_peak * 1e6) else "tensor",
                           "roofline_us": t_roof, "frac": t_roof / us}})
        del Xs, Ys, ws
    del mats
    torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-alt", action="store_true", help="skip timing the other launch schedules")
    ap.add_argument("--no-secondary", action="store_true", help="skip timing the other configurations' kernels")
    ap.add_argument("--repeats", type=int, default=6, help="extra timings of the K-step region (spread)")
    ap.add_argument("--suite", action="store_true", help="time every kernel on every workload shape (JSON lines)")
    ap.add_argument("--only", default="", help="suite: comma list of gemv,top1,decode,repack,pack,gemm_small_m,gemm_m64,argmax,block")
    ap.add_argument("--case", default="", help="suite: substring of the workload name")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.suite:
        run_suite(args)
        return
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    try:
        run_gpu(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
