#!/usr/bin/env python
"""Benchmark of the q4_0 decode path on GB300.

One step = one E2B-shaped decode weight pass at S=1: 35 layers at hidden 1536
(q/o 2048 or 4096 wide, k/v one head on L0-L14, gated MLP 6144 / 12288), q4_0
weights (1,032,486,912 weight bytes per step, more than L2 holds, so no flush
is needed between steps), fp16 activations, fp32 accumulation, run as one CUDA
graph of 141 kernel launches.  The line printed is steps/s for the whole job.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the pass
does not shard); time is the maximum over ranks.  ``--impl reference`` times
the CPU oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "q4_0 dequant-GEMV HBM GB/s vs peak; E2B-shaped decode weight-pass steps/s"
WORKLOAD = "e2b_decode_weight_pass_s1"
FALLBACK_HBM_GBS = 6800.0
SEED = 1003


# --------------------------------------------------------------- helpers ---
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Sources of the persistent decode-pass kernel and its launch: a stored DRAM
# traffic figure is used only while these are unchanged.
PASS_SOURCES = ("k_stream.cu", "q4w_device.cuh", "q4w_internal.cuh", "q4w_tc.cuh", "q4w_top2.cuh", "q4w_api.cu")


def source_hash(names=PASS_SOURCES):
    h = hashlib.sha256()
    for n in sorted(names):
        with open(os.path.join(ROOT, "int4_q4_weight_gb300", "csrc", n), "rb") as f:
            h.update(n.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel_key):
    """DRAM bytes per unit from a committed ncu summary, if the kernels have not
    changed since it was taken; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_unit")


def e2b_step_bytes(layer_dims, H=1536):
    """Algorithmic bytes of one pass: every weight byte once (codes 0.5 B and
    scales 2/32 B per weight) plus each stage's input and output vectors."""
    wbytes = 0
    abytes = 2 * H + 2 * H                          # h0 in, h out (fp16)
    for li, d in enumerate(layer_dims):
        rows = d["q"] + 2 * d["kv"]
        n = rows * H + H * d["q"] + 2 * d["mlp"] * H + H * d["mlp"]
        wbytes += n * 9 // 16
        abytes += (2 * H if li == 0 else 4 * H) + 2 * d["q"] + 4 * 2 * d["kv"]   # qkv stage
        abytes += 2 * d["q"] + 4 * H                                             # o stage
        abytes += 4 * H + 2 * d["mlp"]                                           # gate/up stage
        abytes += 2 * d["mlp"] + 4 * H                                           # down stage
    return wbytes, abytes


def parse_clock_lines(lines, t_begin=None, t_end=None):
    """Median SM clock, max clock and throttle reasons from nvidia-smi lines of
    ClockSampler.FIELDS.  Only samples stamped within [t_begin, t_end]
    (datetimes, local time) count; when none falls inside (a region shorter
    than the sampling interval) every sample counts.  None when no line parses."""
    import datetime
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    rows = []
    for line in lines:
        f = [x.strip() for x in line.split(",")]
        if len(f) < 10:
            continue
        try:
            ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
            rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
        except ValueError:
            continue
    inside = [r for r in rows if (t_begin is None or r[0] >= t_begin) and (t_end is None or r[0] <= t_end)]
    use = inside or rows
    if not use:
        return None
    reasons = {n for r in use for n, v in zip(names, r[3]) if v.lower().startswith("active")}
    return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
            "reasons": sorted(reasons), "samples": len(use)}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms (read-only)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.t_begin = self.t_end = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(device_index)
            target = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        except Exception:
            target = str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", target],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def begin(self):
        """The timed region starts (samples before it are not counted)."""
        import datetime
        self.t_begin = datetime.datetime.now()

    def end(self):
        import datetime
        self.t_end = datetime.datetime.now()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_lines(out.splitlines(), self.t_begin, self.t_end)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(seconds, world, device=None):
    """The slowest rank's time (every rank receives it); the value itself when alone."""
    if world <= 1:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_value(world, steps, seconds):
    """Whole-job steps/s: every replica ran `steps` steps within `seconds`."""
    return world * steps / seconds


def host_cores():
    """Cores this process may run on (sched_getaffinity), the oracle's thread count."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_pass_layers(C, device, threads, layer_ids=None):
    """The E2B layers quantised by the C++ oracle's own quantiser, from the
    seeded fp32 weights of the input generator (drawn on ``device``)."""
    from int4_q4_weight_gb300 import synth
    out = []
    for layer in (range(synth.E2B_N_LAYERS) if layer_ids is None else layer_ids):
        lw = {}
        for name in synth.e2b_matrix_shapes(layer):
            W = synth.e2b_weight(SEED, layer, name, device).cpu().numpy()
            lw[name] = C.quantize_q4_0(W, threads=threads)
            del W
        out.append(lw)
    return out


def layer_bytes(lw):
    return sum(c.size + s.size * 2 for c, s in lw.values())


# ------------------------------------------------------------ our arm ---
def run_ours(args, world, rank, local):
    import torch
    import int4_q4_weight_gb300 as q4w
    from int4_q4_weight_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    q4w.build()
    q4w.load()

    H = synth.E2B_HIDDEN
    layer_ids = list(range(synth.E2B_N_LAYERS - args.layers, synth.E2B_N_LAYERS))
    dims = [synth.e2b_dims(l) for l in layer_ids]
    layers = []
    for layer in layer_ids:
        g = {}
        for name in synth.e2b_matrix_shapes(layer):
            W = synth.e2b_weight(SEED, layer, name, dev)
            g[name] = q4w.q4_quantize(W)
            del W
        layers.append(g)
    torch.cuda.synchronize()
    plan = q4w.Q4DecodePlan(layers, H, device=dev)
    plan.h_in.copy_(synth.e2b_h0(SEED, dev))
    plan.capture()
    wbytes, abytes = e2b_step_bytes(dims, H)
    step_bytes = wbytes + abytes

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        plan.step_device()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        time.sleep(0.3)   # nvidia-smi starts before the timed region, not inside it
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.begin()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        plan.step_device()
    ev1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.end()
    barrier()
    clocks = sampler.stop() if sampler else None
    elapsed = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    value = replica_value(world, args.steps, elapsed)
    ms_per_step = elapsed / args.steps * 1e3

    # end to end through the public API: pinned host h -> device, one graph
    # replay, device -> pinned host result, synchronised every step
    h_host = synth.e2b_h0(SEED, dev).cpu().pin_memory()
    out_host = torch.empty(H, dtype=torch.float16).pin_memory()
    ke = min(args.steps, 2000)
    for _ in range(3):
        plan.step_host(h_host, out_host)
    barrier()
    t0 = time.perf_counter()
    for _ in range(ke):
        plan.step_host(h_host, out_host)
    te = max_over_ranks(time.perf_counter() - t0, world, dev)

    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    achieved = step_bytes / (ms_per_step * 1e-3) / 1e9
    launches = plan.launches_per_step
    traffic = stored_traffic("e2b_pass_step") if args.layers == 35 else None
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,0.02) weights quantised to q4_0 on the device, N(0,1) fp16 h0)",
        "config": {"workload": WORKLOAD if args.layers == 35 else f"{WORKLOAD}_last{args.layers}",
                   "layers": args.layers, "hidden": H, "weight_format": "q4_0",
                   "weight_bytes_per_step": wbytes, "algorithmic_bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2 (1.03 GB of weights per step)",
                   "launch": (f"one CUDA graph per step: two memsets and {launches} persistent cooperative kernel "
                              "(one CTA per SM)" if launches == 1 else
                              f"one CUDA graph per step, {launches} kernels, programmatic dependent launch"),
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(replica_value(world, ke, te), 3), "unit": "steps/s", "h2d_bytes_per_step": 2 * H,
                "d2h_bytes_per_step": 2 * H,
                "how": "pinned host h0 -> device, graph replay, device -> pinned host h, sync per step"},
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic,
                     "kernel": ("decode_pass_kernel (persistent: all stages of the pass in one launch); "
                                "timed as whole graph replays, memsets included" if launches == 1 else
                                "stage kernels of one step, all launches"),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "frac_of_nominal_8TBs": round(achieved / 8000.0, 4)},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.layers == 35:
        line["cpu_baseline"] = cpu_baseline(dev, step_bytes)
    if rank == 0 and world == 1 and not args.no_rows:
        line["rows"] = measure_rows(q4w, synth, dev, hbm, clocks, float(peaks.get("bf16_tflops", 1900.0)))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def cpu_baseline(dev, step_bytes):
    """The C++ oracle as it stands (plain loops, fp64 sums) on the host cores:
    the whole 35-layer chain with its rows split over std::thread across every
    core of sched_getaffinity, and single-threaded on a bounded sample (the
    chain over one layer of each E2B type), scaled to the step by bytes."""
    from int4_q4_weight_gb300 import synth
    from oracle import cpp_oracle
    C = cpp_oracle.oracle()
    cores = host_cores()
    layers = oracle_pass_layers(C, dev, cores)
    h0 = synth.e2b_h0(SEED, dev).cpu().numpy()
    passes, t0 = 0, time.perf_counter()
    while True:
        C.e2b_pass(h0, layers, threads=cores)
        passes += 1
        el = time.perf_counter() - t0
        if el >= 3.0:
            break
    sample_ids = [0, 4, 15, 19]
    sample = [layers[i] for i in sample_ids]
    sbytes = sum(layer_bytes(lw) for lw in sample)
    t1 = time.perf_counter()
    C.e2b_pass(h0, sample, threads=1)
    el1 = time.perf_counter() - t1
    wbytes = sum(layer_bytes(lw) for lw in layers)
    return {"value": round(passes / el, 5), "unit": "steps/s", "cores": cores, "threads": cores, "kind": "oracle",
            "sample": (f"C++ oracle (oracle/q4_oracle.cpp): {passes} full 35-layer passes of the chain in "
                       f"{el:.1f} s, rows split over {cores} std::thread"),
            "single_thread": {"value": round(sbytes / el1 / wbytes, 5), "unit": "steps/s", "threads": 1,
                              "sample": (f"the chain over layers {sample_ids} (one of each E2B layer type, "
                                         f"{sbytes} weight bytes) in {el1:.1f} s on one thread, scaled to the "
                                         f"{wbytes}-byte pass")}}


# ---------------------------------------------------------- other rows ---
def _time_graph(fn, reps, stream=None):
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(reps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def row_gemv(q4w, synth, dev, hbm, reps=10):
    """[2048, 1536] GEMV streamed over distinct weight copies totalling >= 4x L2."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    W, x = synth.gemv_inputs(seed=1001, device=dev)
    c, s = q4w.q4_quantize(W)
    per = c.numel() + s.numel() * 2
    copies = max(8, math.ceil(4 * l2 / per))
    cs = [(c.clone(), s.clone()) for _ in range(copies)]
    y = torch.empty(2048, dtype=torch.float32, device=dev)
    xv = x[0].contiguous()
    t = _time_graph(lambda: [q4w.q4_gemv(ci, si, xv, y) for ci, si in cs], reps) / copies
    b = per + 2 * 1536 + 4 * 2048
    t_iso = _time_graph(lambda: [q4w.q4_gemv(c, s, xv, y) for _ in range(100)], reps) / 100
    # the read-only-weights form: each GEMV's weight tiles stream while the one
    # before it finishes
    t_ro = _time_graph(lambda: [q4w.q4_gemv_weights_ro(ci, si, xv, y) for ci, si in cs], reps) / copies
    return {"GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / hbm, 4),
            "us_per_gemv_streamed": round(t * 1e6, 3),
            "us_per_gemv_isolated_l2_resident": round(t_iso * 1e6, 3),
            "weights_ro": {"GB/s": round(b / t_ro / 1e9, 1), "frac": round(b / t_ro / 1e9 / hbm, 4),
                           "us_per_gemv_streamed": round(t_ro * 1e6, 3)},
            "bytes": b, "copies": copies}


def row_gemv_batch(q4w, synth, dev, hbm, batch=4, reps=10):
    """[2048, 1536] GEMV of `batch` vectors (the S=4 verify shape), weights read
    once per call, streamed over distinct weight copies totalling >= 4x L2."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    W, x = synth.gemv_inputs(seed=1001, device=dev, batch=batch)
    c, s = q4w.q4_quantize(W)
    per = c.numel() + s.numel() * 2
    copies = max(8, math.ceil(4 * l2 / per))
    cs = [(c.clone(), s.clone()) for _ in range(copies)]
    y = torch.empty((batch, 2048), dtype=torch.float32, device=dev)
    t = _time_graph(lambda: [q4w.q4_gemv(ci, si, x, y) for ci, si in cs], reps) / copies
    b = per + 2 * 1536 * batch + 4 * 2048 * batch
    return {"GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / hbm, 4), "us": round(t * 1e6, 3),
            "batch": batch, "bytes": b, "copies": copies}


def row_head(q4w, synth, dev, hbm, bsz, reps=20, weights=None):
    import torch
    if weights is None:
        Wh, _ = synth.head_inputs(seed=1004, device=dev, batch=1)
        weights = q4w.q4_quantize(Wh)
        del Wh
    hc, hs = weights
    _, h = synth.head_inputs(seed=1004, device=dev, batch=bsz, V=1, K=1536)
    ws = q4w.lmhead_ws(262144, 1536, bsz, dev)
    outs = (torch.empty(bsz, dtype=torch.int32, device=dev), torch.empty(bsz, dtype=torch.float32, device=dev),
            torch.empty(bsz, dtype=torch.float32, device=dev))
    t = _time_graph(lambda: q4w.lmhead_softcap_argmax(hc, hs, h, ws=ws, idx=outs[0], top1=outs[1],
                                                      top2=outs[2]), reps)
    b = hc.numel() + hs.numel() * 2 + 2 * 1536 * bsz + 12 * bsz
    return {"GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / hbm, 4), "us": round(t * 1e6, 2),
            "bytes": b}


def row_ple(q4w, synth, dev, hbm, bf16_peak, reps=10, V=None):
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    p = synth.ple_inputs(seed=1002, device=dev, **({"V": V} if V else {}))
    ncp = max(2, math.ceil(2 * l2 / p.proj.numel() / 4))
    projs = [p.proj.clone() for _ in range(ncp)]
    out = torch.empty((64, 8960), dtype=torch.float32, device=dev)
    t = _time_graph(lambda: [q4w.ple_gather_project(p.ids, p.table, p.row_scale, pj, p.hidden,
                                                    p.norm_w, out=out) for pj in projs], reps) / ncp
    b = 64 * 8960 + 64 * 4 + p.proj.numel() * 4 + 64 * 1536 * 2 + 256 * 4 + 64 * 8960 * 4 + 64 * 4
    flops = 2 * 64 * 8960 * 1536
    # the f32 projection runs as two fp16 pieces on kind::f16: twice the
    # algorithmic flops on the tensor pipe, against the measured bf16 peak
    # (the same nominal dense rate as fp16)
    return {"GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / hbm, 4),
            "TFLOP/s": round(flops / t / 1e12, 2), "frac_f16": round(2 * flops / t / 1e12 / bf16_peak, 4),
            "bound": "hbm (f32 projection as two fp16 pieces on the tensor cores, kind::f16)",
            "us": round(t * 1e6, 2), "bytes": b, "copies": ncp}


def row_ple_q8(q4w, synth, dev, hbm, bf16_peak, reps=10, V=None):
    """The PLE with the int8 per-block-32 projection (14.6 MB instead of 55 MB)."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    p = synth.ple_inputs(seed=1002, device=dev, **({"V": V} if V else {}))
    codes, scales = q4w.q8_quantize(p.proj)
    per = codes.numel() + scales.numel() * 2
    ncp = max(2, math.ceil(2 * l2 / per))
    cs = [(codes, scales)] + [(codes.clone(), scales.clone()) for _ in range(ncp - 1)]
    out = torch.empty((64, 8960), dtype=torch.float32, device=dev)
    t = _time_graph(lambda: [q4w.ple_gather_project_q8(p.ids, p.table, p.row_scale, c, s, p.hidden,
                                                       p.norm_w, out=out) for c, s in cs], reps) / ncp
    b = 64 * 8960 + 64 * 4 + per + 64 * 1536 * 2 + 256 * 4 + 64 * 8960 * 4 + 64 * 4
    flops = 2 * 64 * 8960 * 1536
    # fp16 operands: the measured bf16 peak (the same nominal dense rate)
    return {"GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / hbm, 4),
            "TFLOP/s": round(flops / t / 1e12, 2), "frac_f16": round(flops / t / 1e12 / bf16_peak, 4),
            "bound": "hbm (int8 projection widened to fp16 in tensor memory, kind::f16)", "us": round(t * 1e6, 2), "bytes": b,
            "copies": ncp}


def row_gemm(q4w, synth, dev, hbm, bf16_peak, N, K, reps=10):
    """S=64 prefill GEMM; small weights rotate over copies beyond L2."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    W, X = synth.gemm_inputs(seed=1005, device=dev, N=N, K=K)
    c, s = q4w.q4_quantize(W)
    del W
    per = c.numel() + s.numel() * 2
    copies = max(1, math.ceil(2 * l2 / per)) if per < l2 else 1
    cs = [(c, s)] + [(c.clone(), s.clone()) for _ in range(copies - 1)]
    Y = torch.empty((64, N), dtype=torch.float32, device=dev)
    t = _time_graph(lambda: [q4w.q4_gemm_chunk(ci, si, X, Y) for ci, si in cs], reps) / copies
    b = per + 64 * K * 2 + 64 * N * 4
    flops = 2 * 64 * N * K
    return {"GB/s": round(b / t / 1e9, 1), "TFLOP/s": round(flops / t / 1e12, 2),
            "frac_hbm": round(b / t / 1e9 / hbm, 4), "frac_bf16": round(flops / t / 1e12 / bf16_peak, 4),
            "us": round(t * 1e6, 2), "bytes": b, "flops": flops, "copies": copies}


def _a8_scale(q4w, synth, dev, K):
    """w4a8 activation scale, min-max calibrated on 128 synthetic samples [128, K]."""
    cal = synth.normal_f16((128, K), synth.sub_seed(1007, K), dev)
    return float(q4w.q4_act_calibrate_a8(cal).cpu()[0])


def row_gemv_a8(q4w, synth, dev, hbm, reps=10):
    """w4a8 [2048, 1536] GEMV (activation codes under a calibrated scale),
    streamed over distinct weight copies totalling >= 4x L2."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    W, x = synth.gemv_inputs(seed=1001, device=dev)
    c, s = q4w.q4_quantize(W)
    act = _a8_scale(q4w, synth, dev, 1536)
    per = c.numel() + s.numel() * 2
    copies = max(8, math.ceil(4 * l2 / per))
    cs = [(c.clone(), s.clone()) for _ in range(copies)]
    y = torch.empty(2048, dtype=torch.float32, device=dev)
    xv = x[0].contiguous()
    t = _time_graph(lambda: [q4w.q4_gemv_a8(ci, si, xv, act, y) for ci, si in cs], reps) / copies
    b = per + 2 * 1536 + 4 * 2048
    return {"GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / hbm, 4), "us": round(t * 1e6, 3),
            "act_scale": act, "bytes": b, "copies": copies}


def row_gemm_a8(q4w, synth, dev, hbm, bf16_peak, N, K, reps=10):
    """w4a8 S=64 prefill GEMM (the token operand as activation codes)."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    W, X = synth.gemm_inputs(seed=1005, device=dev, N=N, K=K)
    c, s = q4w.q4_quantize(W)
    del W
    act = _a8_scale(q4w, synth, dev, K)
    per = c.numel() + s.numel() * 2
    copies = max(1, math.ceil(2 * l2 / per)) if per < l2 else 1
    cs = [(c, s)] + [(c.clone(), s.clone()) for _ in range(copies - 1)]
    Y = torch.empty((64, N), dtype=torch.float32, device=dev)
    t = _time_graph(lambda: [q4w.q4_gemm_chunk_a8(ci, si, X, act, Y) for ci, si in cs], reps) / copies
    b = per + 64 * K * 2 + 64 * N * 4
    flops = 2 * 64 * N * K
    return {"GB/s": round(b / t / 1e9, 1), "TFLOP/s": round(flops / t / 1e12, 2),
            "frac_hbm": round(b / t / 1e9 / hbm, 4), "frac_bf16": round(flops / t / 1e12 / bf16_peak, 4),
            "us": round(t * 1e6, 2), "act_scale": act, "bytes": b, "flops": flops, "copies": copies}


def row_q2(q4w, synth, dev, hbm, which, reps=10):
    """INT2 GEMV of the mixed-bit recipe: the FFN gate/up shape streamed over
    distinct weight copies totalling >= 4x L2, or the tied head (> L2 alone)."""
    import torch
    N, K = synth.Q2_SHAPES[which]
    codes, scales, x = synth.q2_inputs(seed=1006, device=dev, N=N, K=K)
    per = codes.numel() + 4 * N
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = 1 if per > 2 * l2 else max(8, math.ceil(4 * l2 / per))
    cs = [(codes, scales)] + [(codes.clone(), scales.clone()) for _ in range(copies - 1)]
    y = torch.empty(N, dtype=torch.float32, device=dev)
    xv = x[0].contiguous()
    t = _time_graph(lambda: [q4w.q2_gemv(c, s, xv, y) for c, s in cs], reps) / copies
    b = per + 2 * K + 4 * N
    return {"GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / hbm, 4), "us": round(t * 1e6, 3),
            "bytes": b, "copies": copies}


def measure_rows(q4w, synth, dev, hbm, clocks, bf16_peak):
    rows = {"gemv_2048x1536": row_gemv(q4w, synth, dev, hbm),
            "gemv_b4_2048x1536": row_gemv_batch(q4w, synth, dev, hbm, 4)}
    Wh, _ = synth.head_inputs(seed=1004, device=dev, batch=1)
    hw = q4w.q4_quantize(Wh)
    del Wh
    rows["lmhead_b1"] = row_head(q4w, synth, dev, hbm, 1, weights=hw)
    rows["lmhead_b8"] = row_head(q4w, synth, dev, hbm, 8, weights=hw)
    del hw
    rows["ple_s64"] = row_ple(q4w, synth, dev, hbm, bf16_peak)
    rows["ple_q8_s64"] = row_ple_q8(q4w, synth, dev, hbm, bf16_peak)
    for name, (N, K) in (("gemm_s64_up", (6144, 1536)), ("gemm_s64_down", (1536, 6144)),
                         ("gemm_s64_head", (262144, 1536))):
        rows[name] = row_gemm(q4w, synth, dev, hbm, bf16_peak, N, K)
    rows["q2_gemv_12288x1536"] = row_q2(q4w, synth, dev, hbm, "gate")
    rows["q2_gemv_head_262144x1536"] = row_q2(q4w, synth, dev, hbm, "head")
    rows["gemv_a8_2048x1536"] = row_gemv_a8(q4w, synth, dev, hbm)
    rows["gemm_a8_s64_up"] = row_gemm_a8(q4w, synth, dev, hbm, bf16_peak, 6144, 1536)
    return rows


CASES = ("gemv", "gemv_b4", "head_b1", "head_b8", "ple", "ple_q8", "gemm_up", "gemm_down", "gemm_head", "q2_gate",
         "q2_head", "gemv_a8", "gemm_a8_up", "pass_trace")


def pass_trace(q4w, synth, dev, reps):
    """Per-stage timing of the persistent pass from the device trace stamps."""
    import torch
    H = synth.E2B_HIDDEN
    layers = []
    for layer in range(synth.E2B_N_LAYERS):
        g = {}
        for name in synth.e2b_matrix_shapes(layer):
            W = synth.e2b_weight(SEED, layer, name, dev)
            g[name] = q4w.q4_quantize(W)
            del W
        layers.append(g)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nst = 4 * len(layers)
    buf = torch.zeros(nst * sms * 8, dtype=torch.int64, device=dev)
    ws = torch.empty(q4w.decode_pass_ws_bytes(layers, H), dtype=torch.uint8, device=dev)
    h0 = synth.e2b_h0(SEED, dev)
    h = torch.empty(H, dtype=torch.float16, device=dev)
    descs = q4w.make_layers(layers, H)
    for _ in range(3):
        q4w.q4_decode_pass(layers, h0, h, ws, descs=descs)
    q4w.q4_set_trace(buf)
    acc = None
    for _ in range(reps):
        q4w.q4_decode_pass(layers, h0, h, ws, descs=descs)
        torch.cuda.synchronize()
        ti = buf.view(nst, sms, 8).cpu().numpy()
        acc = ti if acc is None else acc
    q4w.q4_set_trace(None)
    ti = acc
    # stamp 0: globaltimer ns at stage entry; the others: SM cycles since entry
    # (stamp 5 shifted left by one, bit 0 = first tile had landed already)
    ghz = 2.07
    early = (ti[:, :, 5] & 1).reshape(-1, 4, sms)
    ti = ti.copy()
    ti[:, :, 0] -= ti[:, :, 0].min()   # relative ns first: float64 cannot hold absolute ns to 1 ns
    early_last = (ti[:, :, 7] & 1).reshape(-1, 4, sms)
    multi = (ti[:, :, 7] > 0).reshape(-1, 4, sms)
    ti[:, :, 5] >>= 1
    ti[:, :, 7] >>= 1
    t = ti.astype(np.float64)
    for i in range(1, 8):
        t[:, :, i] = t[:, :, 0] + t[:, :, i] / ghz
    t0 = t[0, :, 0].min()
    kinds = ["qkv", "o", "gate_up", "down"]
    # per (stage, CTA): 0 entered, 7 last tile landed (0: one tile), 1 input complete and
    # staged, 2 x built, 3 x in registers, 5 first tile landed, 6 first tile
    # usable by the whole warp, 4 own rows written
    out = {"stages": nst, "total_us": round((t[:, :, 4].max() - t0) / 1e3, 2), "sm_ghz_assumed": ghz}
    out["last_tile_already_landed_frac"] = {k: round(float(early_last[:, i][multi[:, i]].mean()), 3)
                                             if multi[:, i].any() else None for i, k in enumerate(kinds)}
    out["first_tile_already_landed_frac"] = {k: round(float(early[:, i].mean()), 3) for i, k in enumerate(kinds)}
    names = {"input_wait": (0, 1), "xform": (1, 2), "x_regs": (2, 3), "tile_wait": (3, 5),
             "warp_sync": (5, 6), "rows": (6, 4)}
    agg = {k: {n: 0.0 for n in list(names) + ["rows_max", "handoff", "next_entry", "last_tile_after_first",
                                                "rows_after_last_tile"]} for k in kinds}
    for s in range(nst):
        k = kinds[s % 4]
        for n, (i, j) in names.items():
            agg[k][n] += np.median(t[s, :, j] - t[s, :, i]) / 1e3
        agg[k]["rows_max"] += (t[s, :, 4] - t[s, :, 6]).max() / 1e3
        m = ti[s, :, 7] > 0
        if m.any():
            agg[k]["last_tile_after_first"] += np.median(t[s, m, 7] - t[s, m, 6]) / 1e3
            agg[k]["rows_after_last_tile"] += np.median(t[s, m, 4] - t[s, m, 7]) / 1e3
        if s > 0:   # last CTA done with the previous stage -> median CTA has this stage's input
            agg[k]["handoff"] += (np.median(t[s, :, 1]) - t[s - 1, :, 4].max()) / 1e3
            agg[k]["next_entry"] += np.median(t[s, :, 0] - t[s - 1, :, 4]) / 1e3
    out["per_kind_us_summed_over_layers"] = {k: {q: round(v, 2) for q, v in d.items()} for k, d in agg.items()}
    cta = int(np.argmax(t[8, :, 4]))
    cols = [0, 7, 1, 2, 3, 5, 6, 4]
    out["cta0_layer2_stages_us"] = [[round((t[s, 0, i] - t[8, 0, 0]) / 1e3, 3) for i in cols] for s in range(8, 12)]
    out["slowest_cta_layer2_stages_us"] = [[round((t[s, cta, i] - t[8, 0, 0]) / 1e3, 3) for i in cols]
                                           for s in range(8, 12)]
    return out


def run_case(args):
    """One row's workload only (used for single-kernel profiling captures)."""
    import torch
    import int4_q4_weight_gb300 as q4w
    from int4_q4_weight_gb300 import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q4w.build()
    q4w.load()
    peaks, _ = measured_peaks()
    hbm, bf16 = float(peaks["hbm_gbs"]), float(peaks.get("bf16_tflops", 1900.0))
    reps = max(1, args.steps)
    if args.case == "gemv":
        r = row_gemv(q4w, synth, dev, hbm, reps)
    elif args.case == "gemv_b4":
        r = row_gemv_batch(q4w, synth, dev, hbm, 4, reps)
    elif args.case in ("head_b1", "head_b8"):
        r = row_head(q4w, synth, dev, hbm, 1 if args.case == "head_b1" else 8, reps)
    elif args.case == "ple":
        r = row_ple(q4w, synth, dev, hbm, bf16, reps, V=args.ple_vocab)
    elif args.case == "ple_q8":
        r = row_ple_q8(q4w, synth, dev, hbm, bf16, reps, V=args.ple_vocab)
    elif args.case in ("q2_gate", "q2_head"):
        r = row_q2(q4w, synth, dev, hbm, args.case[3:], reps)
    elif args.case == "pass_trace":
        r = pass_trace(q4w, synth, dev, reps)
    elif args.case == "gemv_a8":
        r = row_gemv_a8(q4w, synth, dev, hbm, reps)
    elif args.case == "gemm_a8_up":
        r = row_gemm_a8(q4w, synth, dev, hbm, bf16, 6144, 1536, reps)
    else:
        N, K = {"gemm_up": (6144, 1536), "gemm_down": (1536, 6144), "gemm_head": (262144, 1536)}[args.case]
        r = row_gemm(q4w, synth, dev, hbm, bf16, N, K, reps)
    print(json.dumps({"case": args.case, **r}), flush=True)


# ------------------------------------------------------ reference arm ---
def run_reference(args, world, rank, local):
    """The oracle as the reference arm: the C++ oracle's chain on the host cores."""
    if rank != 0:
        return
    import torch
    from int4_q4_weight_gb300 import synth
    from oracle import cpp_oracle

    C = cpp_oracle.oracle()
    cores = host_cores()
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    layers = oracle_pass_layers(C, dev, cores)
    dims = [synth.e2b_dims(l) for l in range(synth.E2B_N_LAYERS)]
    wbytes, abytes = e2b_step_bytes(dims)
    step_bytes = wbytes + abytes
    h = synth.e2b_h0(SEED, dev).cpu().numpy()
    # one step is the full 35-layer pass when the run fits about two minutes;
    # otherwise each step runs the next few layers of the chain (cycling), and
    # the rate is scaled to the pass by weight bytes
    t0 = time.perf_counter()
    C.e2b_pass(h, layers[:1], threads=cores)
    t_layer = (time.perf_counter() - t0) * wbytes / layer_bytes(layers[0])
    per_step = synth.E2B_N_LAYERS
    if (args.steps + args.warmup) * t_layer > 120.0:
        per_step = max(1, int(synth.E2B_N_LAYERS * 120.0 / ((args.steps + args.warmup) * t_layer)))
    pos = 0

    def step():
        nonlocal pos, h
        sl = [layers[(pos + i) % len(layers)] for i in range(per_step)]
        pos = (pos + per_step) % len(layers)
        h = C.e2b_pass(h, sl, threads=cores)
        return sum(layer_bytes(lw) for lw in sl)

    for _ in range(args.warmup):
        step()
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += step()
    el = time.perf_counter() - t0
    value = done / el / wbytes
    sample = (f"each step: the C++ oracle's chain over {per_step} consecutive E2B layers "
              f"({'the full pass' if per_step == synth.E2B_N_LAYERS else 'cycling, scaled to the pass by bytes'}), "
              f"rows split over {cores} std::thread; {done} weight bytes in {el:.1f} s")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 / value, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": 35, "hidden": 1536, "weight_format": "q4_0",
                       "algorithmic_bytes_per_step": step_bytes},
            "cpu_baseline": {"value": round(value, 5), "unit": "steps/s", "cores": cores, "threads": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=CASES, default=None,
                    help="time one row's workload only (--steps = graph replays), for profiling")
    ap.add_argument("--ple-vocab", type=int, default=None,
                    help="with --case ple/ple_q8: table rows (default the full 262144; smaller for profiling captures)")
    ap.add_argument("--layers", type=int, default=35,
                    help="run only the last N E2B layers (a small case for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.case:
        run_case(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
