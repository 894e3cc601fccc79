"""Benchmark of the Hymba hybrid-head layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one hymba_layer_fwd call over the
Hymba-1.5B-shaped sliding-window layer: batch 8 x (8192 tokens + 128 meta
rows), d_model 1600, 25/5 heads of dim 64, window 1024, d_inner 3200, state
16, bf16 inputs and weights (seeded synthetic values, random init).  `value`
is real tokens per second (meta rows are computed but not counted), device
time, inputs resident in HBM.  The same line carries the decode step (batch
128 over an 8192-token history), the global-attention layer, the 4-layer
stack, the roofline of the dominant kernel, the end-to-end number through the
C ABI with host buffers, and the float64 CPU oracle timed on a bounded sample.

Multi-GPU (torchrun, one process per GPU): every rank runs its own batch
(weak scaling, no collective on the data path); the slowest rank's time is
used and `value` counts the tokens of all ranks.

--impl reference times the float64 CPU oracle (there is no other reference
implementation) on the host on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from hybrid_attention_ssm_fwd_b300 import synth  # noqa: E402

METRIC = "hybrid-head layer prefill tokens/s @8K bf16; decode tok/s; % of roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
E2E_CHUNK = 1
STAGES = ["convert", "in_proj", "kv_export", "attention", "conv", "x_proj", "dt_proj", "scan", "fuse_norm",
          "out_proj", "cache"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# SFU (MUFU) ex2 throughput of one SM per clock on B300 and the maximum SM
# clock: the roofline of the selective scan, whose algorithmic work is 16
# exponentials per (row, channel) -- one per state.
EX2_PER_CLK_PER_SM = 32
SM_COUNT = 148
SM_MAX_GHZ = 2.032
# fp32 lanes of one SM (FMA / FMUL per clock): the scan's other ALU bound.
# Per state and row it needs 4 fp32 operations: delta*A (the ex2 argument),
# decay*h + (delta*u)*B (a multiply and an FMA) and the C.h accumulation (FMA).
FP32_PER_CLK_PER_SM = 128
SCAN_FP32_OPS_PER_STATE = 4


def stage_work(s) -> dict:
    """Algorithmic work of each prefill stage: (bound, amount, unit).  Tensor
    stages count FLOPs (2 per MAC, visible attention pairs only); HBM stages
    the bytes they must move once; the scan its exponentials."""
    rows = s.B * s.L
    fl = layer_flops(s)
    Rp = (s.R + 7) // 8 * 8
    return {
        "in_proj": ("tensor", fl["in_proj"], "FLOP"),
        "attention": ("tensor", fl["attention"], "FLOP"),
        # x_proj has N = R + 2N_state = 132 columns against K = d_inner: about
        # 130 FLOP per byte, so it is HBM-bound: u in, W_x, dt (fp16) and B|C (fp32) out
        "x_proj": ("hbm", rows * (s.di * 2 + Rp * 2 + 2 * s.N * 4) + s.xproj_out * s.di * 2, "B"),
        "out_proj": ("tensor", fl["out_proj"], "FLOP"),
        "conv": ("hbm", rows * s.di * (2 + 2), "B"),                       # x in, u out (fp16)
        "fuse_norm": ("hbm", rows * s.di * (2 + 2 + 2), "B"),              # att, g in; s out
        "scan": ("alu", rows * s.di * s.N, "ex2"),                         # exp(delta A) per state
        "scan_fma": ("fma", rows * s.di * s.N * SCAN_FP32_OPS_PER_STATE, "fp32 op"),
        "scan_hbm": ("hbm", rows * (s.di * (2 + 2 + 2) + Rp * 2 + 2 * s.N * 4), "B"),  # u, z, g; dt, B|C
    }


def stage_roofline(name, work, ms, peaks):
    bound, amount, unit = work
    t = ms / 1e3
    if bound == "tensor":
        achieved, peak, u = amount / t / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    elif bound == "hbm":
        achieved, peak, u = amount / t / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "fma":
        achieved, peak, u = amount / t / 1e12, FP32_PER_CLK_PER_SM * SM_COUNT * SM_MAX_GHZ / 1e3, "Tfp32op/s"
    else:
        achieved, peak, u = amount / t / 1e12, EX2_PER_CLK_PER_SM * SM_COUNT * SM_MAX_GHZ / 1e3, "Tex2/s"
    out = {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": u,
           "frac": round(achieved / peak, 4), "ms": round(ms, 4)}
    if bound == "tensor" and peaks.get("bf16_tflops_sustained"):
        # the same work against the bf16 rate sustained for seconds under the power cap
        out["frac_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
    return out


def stage_rooflines(s, stage_ms: dict, peaks: dict):
    """Every stage against its own bound, plus the scan against its HBM and
    fp32-pipe bounds (timed as the one scan stage).  Returns the per-kernel
    rooflines and the dominant kernel: the longest stage."""
    work = stage_work(s)

    def stage(k):
        return "scan" if k.startswith("scan") else k

    kernels = {k: stage_roofline(k, w, stage_ms[stage(k)], peaks) for k, w in work.items()}
    dom = max((k for k in work if stage(k) == k), key=lambda k: stage_ms[k])
    return kernels, dom


def layer_flops(s) -> dict:
    """Algorithmic FLOPs (2 per MAC) of one prefill call, per stage; attention
    counts only visible (query, key) pairs."""
    rows = s.B * s.L
    L, M, W = s.L, s.M, s.window
    i = np.arange(L)
    if W == 0:
        vis = i + 1
    else:
        vis = np.minimum(i + 1, W) + np.minimum(M, np.maximum(0, i - W + 1))
    pairs = float(vis.sum()) * s.B
    return {
        "in_proj": 2.0 * rows * s.P_in * s.d,
        "attention": 2.0 * pairs * s.Hq * (s.dh + s.dv),
        "x_proj": 2.0 * rows * s.xproj_out * s.di,
        "dt_proj": 2.0 * rows * s.di * s.R,
        "out_proj": 2.0 * rows * s.d * s.di,
        "mean_visible_keys": float(vis.mean()),
    }


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = f"/tmp/hymba_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        under = [v for v in sm if v > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(under) if under else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def make_events(torch, n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()  # creates the underlying cudaEvent_t
    return evs


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from hybrid_attention_ssm_fwd_b300 import binding as hb
    from hybrid_attention_ssm_fwd_b300 import layer as hl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    if args.only_decode:
        return {"decode": run_decode(args, torch, hb, hl, dev, torch.cuda.current_stream(dev), peaks, peak_src)}
    s = synth.hymba15b_swa(rope_theta=10000.0, B=args.batch)
    p = synth.make_layer_inputs(s, rank_seed(rank))
    params = hl.params_to_device(p, s, dev)
    layer = hl.HymbaLayer(s, params)
    X = hl.tokens_to_device(p["Xt"], s, dev)
    Y = torch.empty(s.B, s.L, s.d, dtype=torch.float32, device=dev)
    del p
    stream = torch.cuda.current_stream(dev)
    nev = 12
    ev_sets = [make_events(torch, nev) for _ in range(args.steps)]
    evp = [(ctypes_array(e)) for e in ev_sets]

    def step():
        hb.hymba_layer_fwd(layer.desc, layer.weights, X, Y, layer.ws, status=layer.status, stream=stream)

    def step_events(i):
        hb.hymba_layer_fwd_events(layer.desc, layer.weights, X, Y, layer.ws, evp[i], nev, status=layer.status,
                                  stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if layer.check_status() != 0:
        raise RuntimeError(f"device status {layer.check_status()} after warm-up")
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # the headline: K plain calls back to back, with no event between the
    # stages of a call
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / args.steps
    if layer.check_status() != 0:
        raise RuntimeError(f"device status {layer.check_status()} in the timed region")
    # per-kernel times: a second, instrumented pass of K calls with an event
    # between every stage (the events break the launch overlap, so these
    # stages add up to more than the plain step)
    for i in range(args.steps):
        step_events(i)
    torch.cuda.synchronize()
    stage_ms = {name: statistics.mean(ev[k].elapsed_time(ev[k + 1]) for ev in ev_sets)
                for k, name in enumerate(STAGES)}
    step_each = [ev[0].elapsed_time(ev[len(STAGES)]) for ev in ev_sets]
    ms_max, value = job_throughput(ms, s.B * s.T, world, dev)

    fl = layer_flops(s)
    total_flops = fl["in_proj"] + fl["attention"] + fl["x_proj"] + fl["dt_proj"] + fl["out_proj"]
    peak = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained") or PEAKS_FALLBACK["bf16_tflops_sustained"]
    kernels, dom = stage_rooflines(s, stage_ms, peaks)
    traffic = load_traffic(dom)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, random-init weights)",
        "config": {"workload": "Hymba-1.5B-shaped SWA layer prefill, batch 8 x (8192 + 128 meta), window 1024",
                   "global_batch": s.B * world, "seq_len": s.T, "meta_tokens": s.M, "d_model": s.d,
                   "heads": f"{s.Hq}q/{s.Hkv}kv x 64", "d_inner": s.di, "d_state": s.N, "rope_theta": s.rope_theta,
                   "activations": "fp16 (fp32 accumulate; delta/B/C/state/Y fp32)",
                   "l2": "inputs larger than L2 (X~ 213 MB, projection 1.19 GB per step); no flush",
                   "parallelism": f"dp{world} (independent batches, no collective)"},
        "layer_tflops": round(total_flops / (ms_max / 1e3) / 1e12, 1),
        "roofline_layer": {"bound": "tensor", "achieved_tflops": round(total_flops / (ms_max / 1e3) / 1e12, 1),
                           "peak": peak, "frac": round(total_flops / (ms_max / 1e3) / 1e12 / peak, 4),
                           "peak_sustained": sustained,
                           "frac_sustained": round(total_flops / (ms_max / 1e3) / 1e12 / sustained, 4),
                           "note": f"all five contractions' algorithmic FLOPs / layer time, of {peak_src} bf16 "
                                   "(burst; frac_sustained: the rate held for seconds under the power cap)"},
        "roofline": dict({"kernel": dom}, **{k: v for k, v in kernels[dom].items() if k != "ms"},
                         traffic=traffic,
                         peak_source={"tensor": f"{peak_src} bf16 (burst)", "hbm": f"{peak_src} HBM copy",
                                      "alu": "SFU ex2: 32 per clock per SM x 148 SMs x 2.032 GHz",
                                      "fma": "fp32 lanes: 128 per clock per SM x 148 SMs x 2.032 GHz"}[
                                          kernels[dom]["bound"]]),
        "kernels": kernels,
        # per-stage times from the instrumented pass (events between stages)
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        # each instrumented call (its first to its last stage event)
        "instrumented_step_ms": {"median": round(statistics.median(step_each), 4), "min": round(min(step_each), 4),
                                 "max": round(max(step_each), 4)},
        "clocks": clk,
        # per layer call: W_out, W_x (bf16 -> fp16 copies) and W_dt conversions, then in_proj,
        # attention, conv, x_proj, scan, fuse_norm, out_proj (the ncu launch list shows the same)
        "gpu_launches": 10 * args.steps,
    }
    # free the prefill buffers before the other workloads
    del layer, X, Y, params
    torch.cuda.empty_cache()
    if args.only_main:
        return out
    out["e2e"] = run_e2e(args, torch, hb, hl, dev, stream)
    out["meta_prefix"] = run_meta_prefix(args, torch, hb, hl, dev, stream)
    out["block"] = run_block(args, torch, hb, hl, dev, stream)
    out["decode"] = run_decode(args, torch, hb, hl, dev, stream, peaks, peak_src)
    out["global_prefill"] = run_prefill_extra(args, torch, hb, hl, dev, stream, synth.hymba15b_global(rope_theta=10000.0),
                                              "Hymba-1.5B-shaped global-attention layer, batch 2 x (8192 + 128)")
    out["stack4"] = run_stack(args, torch, hb, hl, dev, stream)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args)
    return out


def job_throughput(ms_local: float, tokens_per_rank: int, world: int, device):
    """Whole-job throughput of a data-parallel step: every rank processes its
    own tokens_per_rank (weak scaling) and the slowest rank sets the pace, so
    the job's step time is the max over ranks.  Returns (ms_max, tokens/s)."""
    ms_max = float(ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_max], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
    return ms_max, tokens_per_rank * world / (ms_max / 1e3)


def rank_seed(rank: int) -> int:
    """Each rank draws its own batch of the workload (seeded by its rank)."""
    return 1 + rank


def ctypes_array(events):
    import ctypes
    arr = (ctypes.c_void_p * len(events))()
    for k, e in enumerate(events):
        arr[k] = e.cuda_event
    return arr


def load_traffic(kernel):
    """dram bytes per launch from the committed ncu summary, if present."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        v = d.get(kernel)
        if isinstance(v, dict):
            return v.get("bytes_per_launch")
    return None


def run_e2e(args, torch, hb, hl, dev, stream):
    """The main prefill through the C ABI from host buffers: every step copies
    X~ from pinned host memory, runs the layer and copies Y back to pinned host
    memory.  The batch goes through in chunks of E2E_CHUNK sequences on three
    streams, so the host-to-device copy of chunk i+1 and the device-to-host
    copy of chunk i-1 overlap the layer call of chunk i."""
    s = synth.hymba15b_swa(rope_theta=10000.0)
    p = synth.make_layer_inputs(s, 7)
    sc = synth.with_(s, B=E2E_CHUNK)
    layer = hl.HymbaLayer(sc, hl.params_to_device(p, sc, dev))
    Xh = torch.from_numpy(p["Xt"]).to(torch.bfloat16).pin_memory()
    Yh = torch.empty(s.B, s.L, s.d, dtype=torch.float32).pin_memory()
    Xd = torch.empty_like(Xh, device=dev)
    Yd = torch.empty(Yh.shape, dtype=torch.float32, device=dev)
    del p
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n_chunks = s.B // E2E_CHUNK
    ev_in = [torch.cuda.Event() for _ in range(n_chunks)]
    ev_done = [torch.cuda.Event() for _ in range(n_chunks)]

    def step():
        s_in.wait_stream(stream)          # the previous step's reads of Xd are done
        for c in range(n_chunks):
            sl = slice(c * E2E_CHUNK, (c + 1) * E2E_CHUNK)
            with torch.cuda.stream(s_in):
                Xd[sl].copy_(Xh[sl], non_blocking=True)
                ev_in[c].record(s_in)
        for c in range(n_chunks):
            sl = slice(c * E2E_CHUNK, (c + 1) * E2E_CHUNK)
            stream.wait_event(ev_in[c])
            hb.hymba_layer_fwd(layer.desc, layer.weights, Xd[sl], Yd[sl], layer.ws, status=layer.status,
                               stream=stream)
            ev_done[c].record(stream)
            s_out.wait_event(ev_done[c])
            with torch.cuda.stream(s_out):
                Yh[sl].copy_(Yd[sl], non_blocking=True)
        stream.wait_stream(s_out)         # the step ends when Y is on the host

    for _ in range(max(2, args.warmup)):
        step()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 10))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    out = {"value": round(s.B * s.T / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 3),
           "h2d_bytes_per_step": Xh.numel() * 2, "d2h_bytes_per_step": Yh.numel() * 4,
           "pipeline": f"{n_chunks} chunks of {E2E_CHUNK} sequences; H2D, layer and D2H on three streams",
           "status": layer.check_status()}
    del layer, Xh, Yh, Xd, Yd
    torch.cuda.empty_cache()
    return out


def run_prefill_extra(args, torch, hb, hl, dev, stream, s, name):
    p = synth.make_layer_inputs(s, 2)
    layer = hl.HymbaLayer(s, hl.params_to_device(p, s, dev))
    X = hl.tokens_to_device(p["Xt"], s, dev)
    Y = torch.empty(s.B, s.L, s.d, dtype=torch.float32, device=dev)
    del p
    for _ in range(args.warmup):
        hb.hymba_layer_fwd(layer.desc, layer.weights, X, Y, layer.ws, status=layer.status, stream=stream)
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 10))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        hb.hymba_layer_fwd(layer.desc, layer.weights, X, Y, layer.ws, status=layer.status, stream=stream)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    fl = layer_flops(s)
    tot = fl["in_proj"] + fl["attention"] + fl["x_proj"] + fl["dt_proj"] + fl["out_proj"]
    out = {"workload": name, "value": round(s.B * s.T / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "tflops": round(tot / (ms / 1e3) / 1e12, 1), "status": layer.check_status()}
    del layer, X, Y
    torch.cuda.empty_cache()
    return out


def run_meta_prefix(args, torch, hb, hl, dev, stream):
    """The main workload through the meta-prefix calls: the M meta rows once
    (hymba_meta_prefill), then the B x T real rows from that state
    (hymba_layer_fwd_meta), both inside each timed step."""
    s = synth.hymba15b_swa(rope_theta=10000.0, B=args.batch)
    p = synth.make_layer_inputs(s, 3)
    layer = hl.HymbaLayer(s, hl.params_to_device(p, s, dev))
    xm = hl.tokens_to_device(p["meta"], s, dev)
    X = hl.tokens_to_device(p["X"], s, dev)
    del p
    Y = torch.empty(s.B, s.T, s.d, dtype=torch.float32, device=dev)
    meta = layer.meta_prefill(xm)                       # allocates the meta state once
    mstruct = hb.make_meta(meta)
    ws = layer._scratch(max(hb.meta_prefill_workspace(layer.desc), hb.layer_fwd_meta_workspace(layer.desc)))

    def step():
        hb.hymba_meta_prefill(layer.desc, layer.weights, xm, mstruct, ws, status=layer.status, stream=stream)
        hb.hymba_layer_fwd_meta(layer.desc, layer.weights, mstruct, X, Y, ws, status=layer.status, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 10))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    out = {"workload": "the main workload via the meta-prefix calls (meta rows once, then B x T real rows)",
           "value": round(s.B * s.T / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "status": layer.check_status()}
    del layer, X, Y, xm, meta, ws
    torch.cuda.empty_cache()
    return out


def run_block(args, torch, hb, hl, dev, stream):
    """The full residual block around the main workload's layer (RMSNorm ->
    layer -> add, RMSNorm -> GeLU-gated MLP with F = 3 d -> add), applied in
    place to the fp32 stream each step."""
    s = synth.hymba15b_swa(rope_theta=10000.0, B=args.batch)
    d_ff = 3 * s.d
    tok, blocks = synth.make_block_inputs(s, d_ff, 4)
    blk = hl.HymbaBlock(s, hl.block_params_to_device(blocks[0], s, dev), d_ff)
    x = torch.from_numpy(tok["Xt"]).to(dev)
    del tok, blocks
    for _ in range(args.warmup):
        blk.forward(x)
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 10))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        blk.forward(x)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    fl = layer_flops(s)
    rows = s.B * s.L
    tot = fl["in_proj"] + fl["attention"] + fl["x_proj"] + fl["dt_proj"] + fl["out_proj"] + 6.0 * rows * s.d * d_ff
    out = {"workload": f"residual block around the main workload's layer, gated MLP F = {d_ff}, batch {s.B} x "
                       f"({s.T} + {s.M})",
           "value": round(s.B * s.T / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "tflops": round(tot / (ms / 1e3) / 1e12, 1), "status": blk.check_status()}
    del blk, x
    torch.cuda.empty_cache()
    return out


def run_stack(args, torch, hb, hl, dev, stream):
    """The 300M-ablation 4-layer stack, one hymba_stack_fwd call per step (the
    fp32 stream and its bf16 copy for the next layer are written by each
    layer's output projection; layer 2 reads layer 1's K/V)."""
    shapes = [synth.with_(s, rope_theta=10000.0) for s in synth.ablation300m_stack()]
    tok, layers = synth.make_stack_inputs(shapes, seed=3)
    st = hl.HymbaStack(shapes, [hl.params_to_device(p, s, dev) for p, s in zip(layers, shapes)])
    s0 = shapes[0]
    X0 = hl.tokens_to_device(tok["Xt"], s0, dev)
    y = torch.empty(s0.B, s0.L, s0.d, dtype=torch.float32, device=dev)
    del tok, layers

    def step():
        hb.hymba_stack_fwd(st.descs, st.weights, X0, y, st.ws, status=st.status, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 10))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    tot = 0.0
    for s in shapes:
        fl = layer_flops(s)
        tot += fl["in_proj"] + fl["attention"] + fl["x_proj"] + fl["dt_proj"] + fl["out_proj"]
    out = {"workload": "300M-ablation 4-layer stack (global, SWA x3, layers 1->2 share K/V), batch 32 x (2048 + 128)",
           "value": round(s0.B * s0.T / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "tflops": round(tot / (ms / 1e3) / 1e12, 1), "call": "hymba_stack_fwd", "status": st.check_status()}
    del st, X0, y
    torch.cuda.empty_cache()
    return out


def decode_bytes(s, cap):
    """Minimum HBM bytes of one decode step (weights, K/V read, state r+w)."""
    w = (s.P_in * s.d + s.d * s.di + s.xproj_out * s.di + s.di * s.R) * 2
    kv = s.B * min(cap, s.window) * s.Hkv * (s.dh + s.dv) * 2 + s.M * s.Hkv * (s.dh + s.dv) * 2
    state = s.B * s.di * s.N * 4 * 2 + s.B * s.di * (s.k - 1) * 4 * 2
    io = s.B * s.d * (2 + 4)
    return w + kv + state + io


def run_decode(args, torch, hb, hl, dev, stream, peaks, peak_src):
    s = synth.hymba15b_decode(rope_theta=10000.0)
    cap = s.window
    inp = synth.make_decode_inputs(s, 4, cap=cap, pos=8192)
    cache = hl.cache_to_device(inp, s, dev)
    layer = hl.HymbaLayer(s, hl.params_to_device(inp, s, dev), decode=True)
    xn = hl.tokens_to_device(inp["x_new"], s, dev)
    y = torch.empty(s.B, s.d, dtype=torch.float32, device=dev)
    cc = hb.make_cache(cache, cap)
    del inp

    def step():
        hb.hymba_layer_decode(layer.desc, layer.weights, xn, y, cc, layer.ws, status=layer.status, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    # per-stage times from one instrumented pass
    evs = make_events(torch, 12)
    evp = ctypes_array(evs)
    for _ in range(3):
        hb.hymba_layer_decode_events(layer.desc, layer.weights, xn, y, cc, layer.ws, evp, 12, status=layer.status,
                                     stream=stream)
    torch.cuda.synchronize()
    dstages = ["convert", "in_proj", "kv_append", "attention", "conv", "x_proj", "dt_proj", "scan", "fuse_norm",
               "out_proj", "pos"]
    stage_us = {nm: round(evs[k].elapsed_time(evs[k + 1]) * 1e3, 2) for k, nm in enumerate(dstages)}
    n = max(10, args.steps * 5)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    us = t0.elapsed_time(t1) / n * 1e3
    # CUDA-graph replay of the same call
    g_us = None
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                hb.hymba_layer_decode(layer.desc, layer.weights, xn, y, cc, layer.ws, status=layer.status,
                                      stream=side)
        stream.wait_stream(side)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(n):
            g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        g_us = t0.elapsed_time(t1) / n * 1e3
    except Exception as e:  # graph capture is an optimisation; report why it failed
        g_us = f"graph capture failed: {e}"
    best = g_us if isinstance(g_us, float) and g_us < us else us
    nbytes = decode_bytes(s, cap)
    gbs = nbytes / (best * 1e-6) / 1e9
    return {"workload": "decode step, batch 128, 8192 cached tokens (1024-slot ring + 128 meta), 1.5B shapes",
            "value": round(s.B / (best * 1e-6), 1), "unit": "tokens/s", "us_per_step": round(us, 2),
            "us_per_step_graph": round(g_us, 2) if isinstance(g_us, float) else g_us, "stage_us": stage_us,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes,
                         "traffic": load_traffic("decode_step"), "peak_source": f"{peak_src} HBM copy"},
            "status": layer.check_status()}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------


def oracle_sample(T_sample: int, seed: int):
    """One bounded sample: the float64 oracle on one sequence of T_sample
    tokens (+128 meta) at the 1.5B SWA shapes.  Returns (tokens, seconds)."""
    from oracle import hymba_ref as ref
    s = synth.hymba15b_swa(B=1, T=T_sample, rope_theta=10000.0)
    p = synth.make_layer_inputs(s, seed)
    t0 = time.perf_counter()
    ref.layer_fwd(p, p["Xt"], s)
    return s.T, time.perf_counter() - t0


def oracle_decode_sample(n_seq: int, seed: int):
    """One bounded decode sample: the float64 oracle's decode step for n_seq
    sequences at the 1.5B shapes over an 8192-token history (full 1024-slot
    ring + 128 meta K/V).  Returns (tokens, seconds)."""
    from oracle import hymba_ref as ref
    s = synth.hymba15b_decode(B=n_seq, rope_theta=10000.0)
    inp = synth.make_decode_inputs(s, seed, cap=s.window, pos=8192)
    cache = {k: inp[k] for k in ("k_ring", "v_ring", "k_meta", "v_meta", "ssm_state", "conv_state", "pos")}
    t0 = time.perf_counter()
    ref.layer_decode(inp, inp["x_new"], cache, s)
    return n_seq, time.perf_counter() - t0


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def cpu_baseline(args):
    T = args.cpu_sample_tokens
    toks, sec = oracle_sample(T, 11)
    n_dec, sec_dec = oracle_decode_sample(16, 12)
    return {"value": round(toks / sec, 2), "unit": "tokens/s", "cores": cpu_cores(), "cpu_model": cpu_model(),
            "kind": "oracle",
            "sample": f"float64 NumPy oracle, 1 sequence x ({T} + 128 meta) tokens at the 1.5B SWA shapes, "
                      f"{sec:.1f} s",
            "decode": {"value": round(n_dec / sec_dec, 2), "unit": "tokens/s",
                       "sample": f"one decode step of {n_dec} sequences over an 8192-token history "
                                 f"(1024-slot ring + 128 meta), {sec_dec:.1f} s"}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    T = args.ref_sample_tokens
    for _ in range(args.warmup):
        oracle_sample(T, 11)
    tot_tok, tot_s = 0, 0.0
    for i in range(args.steps):
        toks, sec = oracle_sample(T, 11)
        tot_tok += toks
        tot_s += sec
    v = tot_tok / tot_s
    return {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": "Hymba-1.5B-shaped SWA layer prefill (bounded sample: 1 sequence per step)",
                       "seq_len": T, "meta_tokens": 128, "parallelism": "host CPU"},
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "cores": cpu_cores(), "cpu_model": cpu_model(),
                             "kind": "oracle",
                             "sample": f"1 sequence x ({T} + 128 meta) tokens per step, float64 NumPy"},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def relaunch_ranks(args_argv, n: int, backend_env: dict = None) -> int:
    """--gpus N from a plain `python bench.py` (no torchrun around it): start
    N ranks of this script under torch.distributed.run on this node, one per
    GPU, rendezvous on 127.0.0.1, and return their exit status (rank 0 prints
    the JSON line)."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *args_argv]
    env = dict(os.environ)
    env.update(backend_env or {})
    return subprocess.call(cmd, env=env)


def run_dry_cpu(args, rank, world):
    """CPU stand-in of the multi-rank step for host-side tests (gloo): every
    rank reports a fixed step time for its own batch; the job's time is the
    slowest rank's, its throughput the tokens of all ranks."""
    import torch.distributed as dist
    ms_local = 10.0 + rank
    ms_max, value = job_throughput(ms_local, 8 * 8192, world, "cpu")
    if world > 1:
        dist.barrier()
    return {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "scaling": "weak", "dry_run": "cpu"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample-tokens", type=int, default=6144)
    ap.add_argument("--ref-sample-tokens", type=int, default=512)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-main", action="store_true",
                    help="time only the main prefill workload (used for profiler runs)")
    ap.add_argument("--batch", type=int, default=8, help="sequences in the main prefill workload")
    ap.add_argument("--only-decode", action="store_true",
                    help="time only the decode step (used for profiler runs)")
    ap.add_argument("--dry-run-cpu", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(relaunch_ranks(sys.argv[1:], args.gpus))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if args.dry_run_cpu:
        import torch.distributed as dist
        if world > 1:
            dist.init_process_group("gloo")
        out = run_dry_cpu(args, rank, world)
        if rank == 0:
            print(json.dumps(out), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
