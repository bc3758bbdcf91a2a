#!/usr/bin/env python
"""Benchmark of the tensor-parallel block hot path on GB300.

Headline (``value``): TP-sharded MLP forward + backward TFLOP/s on the Qwen3-8B-shaped
SwiGLU block with t = 8 logical shards on one GPU: X [8192, 4096], gate/up [4096, 12288]
in 1536-column shards, down [12288, 4096] in 1536-row shards.  One step is
ttl_tp_mlp_fwd + ttl_tp_mlp_bwd: fc1 (SwiGLU fused), fc2 partials, the g all-reduce,
fc2 dgrad (SwiGLU' fused), every weight gradient, the dX partials and the f all-reduce.
Algorithmic work: 9 GEMMs of 2*8192*4096*12288 FLOPs = 7.422 TFLOP per step.

The same run measures the other rows of the path on their own workloads:
  shard_reduce  reduce-scatter / all-gather / all-reduce of t in {2,4,8,16} bf16 partial
                sums [4096, 8192] (64 MiB each), HBM GB/s with L2 flushed before each launch;
  gtp_chain     8-layer GTP_remat chain (TP slice [8192, 2048] as 8 shards of 4 MiB,
                X [4096, 8192]): warm forward with side-stream prefetch, backward with
                prefetch, wgrad reduce-scatter and one-layer-deferred finalize;
  vocab_ce      LM head [151936, 4096] in 8 vocab shards + cross-entropy on 8192 tokens.

``--impl reference`` times the CPU oracle (the reference arm of this build) on a bounded
sample of the same workload.  Inputs are synthetic (seeded), drawn on the device for our
arm and on the host for the oracle.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TP-sharded MLP fwd+bwd TFLOP/s (% BF16 peak); shard-reduce HBM GB/s"
MLP = dict(t=8, T=8192, h=4096, f=12288, act="swiglu", seed=3)
MLP_FLOPS = 9 * 2.0 * MLP["T"] * MLP["h"] * MLP["f"]
WORKLOAD = "qwen3_8b_swiglu_mlp_t8_T8192_h4096_f12288_fwd_bwd"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-components", action="store_true", help="skip the shard_reduce/gtp/ce legs")
    ap.add_argument("--cpu-tokens", type=int, default=256, help="token rows of the oracle sample")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="the CPU baseline repeats the oracle sample until this much time has passed")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["sp_mlp", "shard_reduce", "gtp_chain", "vocab_ce", "vocab_embedding",
                                       "tp_attention"],
                    help="run just one secondary component (for profiling); prints its JSON object")
    ap.add_argument("--attn-small", action="store_true",
                    help="tp_attention at the profiling size: T=4096, h=4096, 8 query / 2 KV heads of 128, t=2")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing

class Dist:
    def __init__(self, want: int):
        import torch
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist
        if want != self.world and self.rank == 0:
            print(f"# note: --gpus {want} but WORLD_SIZE={self.world}; using WORLD_SIZE", file=sys.stderr)

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks and peaks

class Clocks:
    """nvidia-smi sampled every 100 ms from start() to stop(); each sample carries its own
    timestamp, so the summary can be taken over any window of the run (the headline's warm-up
    and timed region, or one component)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        self.samples = []

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait(timeout=5)
        self.f.flush()
        self.f.seek(0)
        import datetime
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            reasons = {n for n, v in zip(self.NAMES, parts[6:10]) if v.lower().startswith("active")}
            self.samples.append((ts, sm, smax, reasons))
        os.unlink(self.f.name)

    def window(self, t0=None, t1=None) -> dict:
        """Median SM clock, max clock and the throttle reasons seen between t0 and t1."""
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sel = [x for x in self.samples if (t0 is None or x[0] >= t0 - 0.05) and (t1 is None or x[0] <= t1 + 0.05)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_max_mhz": max(x[2] for x in sel),
                "samples": len(sel), "reasons": sorted(set().union(*(x[3] for x in sel)))}


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        clk = d.get("clocks_under_load", {})
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sustained_sm_mhz": clk.get("sm_mhz_median"), "sm_max_mhz": d.get("sm_max_mhz", 2070.0),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sustained_sm_mhz": None,
            "sm_max_mhz": 2070.0, "source": "fallback"}


def tensor_peak(pk: dict, clk: dict):
    """The dense bf16 peak that matches the clocks a measurement ran at.  The burst figure was
    taken at the maximum SM clock; the sustained one after seconds back to back, under the
    power cap, at a lower median clock.  A window whose median SM clock is within 5% of the
    maximum ran under burst conditions; any other window is judged against the sustained
    figure.  Returns (peak TFLOP/s, a one-line reason)."""
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz") or pk["sm_max_mhz"]
    if sm is not None and smax and sm >= 0.95 * smax:
        return pk["bf16_tflops"], (f"{pk['source']} bf16_tflops (burst): median SM clock {sm:.0f} MHz "
                                   f"within 5% of the {smax:.0f} MHz maximum")
    why = "no clock samples" if sm is None else f"median SM clock {sm:.0f} MHz below 95% of {smax:.0f} MHz"
    return pk["bf16_tflops_sustained"], f"{pk['source']} bf16_tflops_sustained (power-capped): {why}"


def roofline(bound: str, kernel: str, achieved: float, pk: dict, clk: dict, traffic=None, **extra) -> dict:
    """The roofline object of one dominant kernel: ``achieved`` in TFLOP/s (tensor) or GB/s
    (hbm), against the measured peak that fits the clocks it ran at.  For tensor-bound
    kernels it also gives the rate scaled to the maximum SM clock (time x median MHz)."""
    if bound == "tensor":
        peak, why = tensor_peak(pk, clk)
        unit = "TFLOP/s"
    else:
        peak, why, unit = pk["hbm_gbs"], f"{pk['source']} hbm_gbs (copy bandwidth)", "GB/s"
    out = {"bound": bound, "kernel": kernel, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
           "frac": round(achieved / peak, 4), "peak_source": why, "traffic": traffic}
    if bound == "tensor" and clk.get("sm_mhz"):
        out["achieved_at_max_clock"] = round(achieved * (clk["sm_max_mhz"] or pk["sm_max_mhz"]) / clk["sm_mhz"], 1)
        out["frac_of_burst_at_max_clock"] = round(out["achieved_at_max_clock"] / pk["bf16_tflops"], 4)
    out["clocks"] = clk
    out.update(extra)
    return out


def committed_traffic(kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on the current
    kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    src = os.path.join(ROOT, "tensor_transformer_layer_way_gb300", "csrc", d["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return d["bytes_per_launch"] if h == d.get("source_sha256_16") else None


# ------------------------------------------------------------------ our arm

def run_ours(args, dist):
    import torch
    import tensor_transformer_layer_way_gb300 as ttl

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    pk = peaks()
    t, T, h, f, act = MLP["t"], MLP["T"], MLP["h"], MLP["f"], MLP["act"]
    fs = f // t
    g = torch.Generator(device=dev).manual_seed(MLP["seed"] + 1000 * dist.rank)

    def rnd(shape, std):
        return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)

    X, dY = rnd((T, h), 1.0), rnd((T, h), 1.0)
    Wg = [rnd((h, fs), 0.02) for _ in range(t)]
    Wu = [rnd((h, fs), 0.02) for _ in range(t)]
    Wd = [rnd((fs, h), 0.02) for _ in range(t)]
    fo = ttl.mlp_fwd_buffers(t, act, T, h, f, dev)
    bo = ttl.mlp_bwd_buffers(t, act, T, h, f, dev)

    def step():
        ttl.tp_mlp_fwd(X, Wg, Wd, act=act, A_up=Wu, out=fo)
        ttl.tp_mlp_bwd(X, dY, Wg, Wd, fo, act=act, A_up=Wu, out=bo)

    # Clocks are sampled for the whole run; the headline's window runs from the start of the
    # warm-up to the end of the timed region, so a short timed region still has samples.
    clocks = Clocks(dist.local)
    clocks.start()
    w0 = time.time()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ttl.device_status() != 0:
        raise RuntimeError("device status set during warm-up: " + ttl.last_error())

    # Timed region: the K steps alone (no launch tracer), an event between consecutive steps.
    dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record()
    for i in range(args.steps):
        step()
        ev[i + 1].record()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    w1 = time.time()
    ms = ev[0].elapsed_time(ev[-1])
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    if ttl.device_status() != 0:
        raise RuntimeError("device status set during the timed region: " + ttl.last_error())
    ms_max = dist.max(ms)
    value = dist.world * MLP_FLOPS * args.steps / (ms_max * 1e-3) / 1e12
    med = statistics.median(per_step)

    # A separate traced pass of the same step gives every launch's duration and work.
    n_tr = min(args.steps, 20)
    ttl.trace_enable(True, 1 << 16)
    for _ in range(n_tr):
        step()
    torch.cuda.synchronize()
    recs = ttl.trace_read(1 << 16)
    ttl.trace_enable(False)
    launches_per_step = len(recs) / n_tr

    gemm = [r for r in recs if r[0] == "gemm"]
    red = [r for r in recs if r[0] == "reduce"]
    g_ms = sum(r[1] for r in gemm)
    g_fl = sum(r[2] for r in gemm)
    comps = {}
    marks = {"headline": (w0, w1)}
    e2e = bench_e2e(ttl, torch, dev, dist, args, X, dY, Wg, Wu, Wd, fo, bo)
    del fo, bo
    torch.cuda.empty_cache()
    if not args.no_components:
        for name, fn in (("sp_mlp", bench_sp_mlp), ("shard_reduce", bench_shard_reduce), ("gtp_chain", bench_gtp),
                         ("vocab_ce", bench_ce), ("vocab_embedding", bench_embedding),
                         ("tp_attention", bench_attention)):
            c0 = time.time()
            comps[name] = fn(ttl, torch, dev, pk, args)
            marks[name] = (c0, time.time())
    clocks.stop()
    clk = clocks.window(*marks["headline"])
    for name in comps:
        finish_rooflines(comps[name], pk, clocks.window(*marks[name]))

    roof = roofline("tensor", "gemm_tcgen05_kernel", g_fl / (g_ms * 1e-3) / 1e12, pk, clk,
                    traffic=committed_traffic("gemm_tcgen05_kernel"),
                    launches_per_step=len(gemm) / n_tr, flops_per_launch=g_fl / max(len(gemm), 1),
                    avg_launch_ms=g_ms / max(len(gemm), 1), share_of_step=round(g_ms / n_tr / med, 4),
                    timing=f"per-launch CUDA events in a separate traced pass of {n_tr} steps")
    r_ms = sum(r[1] for r in red)
    r_by = sum(r[3] for r in red)
    allreduce = roofline("hbm", "shard_reduce_kernel<8,AR>", r_by / (r_ms * 1e-3) / 1e9, pk, clk,
                         traffic=committed_traffic("shard_reduce_kernel<8,AR>"),
                         share_of_step=round(r_ms / n_tr / med, 4))
    # One step's launches with their FLOPs (or bytes) and times, from the traced pass.
    per = int(launches_per_step)
    roof["launches_last_step"] = [
        {"kind": r[0], "ms": round(r[1], 4), "tflops": round(r[2] / (r[1] * 1e-3) / 1e12, 1) if r[2] else None,
         "gbs": round(r[3] / (r[1] * 1e-3) / 1e9, 1) if not r[2] else None} for r in recs[-per:]]
    peak = roof["peak"]

    out = {"metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": dist.world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4),
           "median_ms_per_step": round(med, 4), "value_at_median_step": round(MLP_FLOPS / (med * 1e-3) / 1e12, 1),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded randn drawn on the device, Qwen3-8B MLP shapes)",
           "config": {"workload": WORKLOAD, "t": t, "tokens": T, "h": h, "ffn": f, "act": act,
                      "parallelism": f"{dist.world} independent replica(s), t={t} logical shards each",
                      "l2": "working set larger than L2 (288 MiB of weights + 1.5 GiB of activations); no flush",
                      "timing": "CUDA events between consecutive steps, no launch tracer in the timed region"},
           "pct_of_bf16_peak": round(value / dist.world / peak, 4), "peak_used": roof["peak_source"],
           "roofline": roof, "allreduce_in_step": allreduce,
           "e2e": e2e, "gpu_launches": int(round(launches_per_step * args.steps)), "clocks": clk}
    out.update(comps)
    return out


def finish_rooflines(comp: dict, pk: dict, clk: dict):
    """Components return their rooflines as ("pending", bound, kernel, achieved, traffic, extra)
    tuples; the peak is filled in once the component's clock window is known."""
    for k, v in list(comp.items()):
        if isinstance(v, tuple) and v and v[0] == "pending":
            _, bound, kernel, achieved, traffic, extra = v
            comp[k] = roofline(bound, kernel, achieved, pk, clk, traffic=traffic, **extra)
        elif isinstance(v, dict):
            finish_rooflines(v, pk, clk)


def pending(bound, kernel, achieved, traffic=None, **extra):
    return ("pending", bound, kernel, achieved, traffic, extra)


def bench_e2e(ttl, torch, dev, dist, args, X, dY, Wg, Wu, Wd, fo, bo):
    """The headline metric end to end through the public API with host buffers.

    Every step copies its inputs X and dY in from pinned host memory and its results (Z and
    dX, one buffer each) back out.  The copies run on a separate copy stream so that step
    i+1's inputs load and step i-1's results drain while step i computes: two input slots and
    two sets of output buffers on the device, used alternately and ordered by events (a step
    does not overwrite a set until its previous results have reached the host).  All copies
    of all K steps are inside the timed region, and the last result is checked on the host."""
    T, h, act = MLP["T"], MLP["h"], MLP["act"]
    t, f = MLP["t"], MLP["f"]
    main = torch.cuda.current_stream()
    cp = torch.cuda.Stream()
    Xin = [X, torch.empty_like(X)]
    dYin = [dY, torch.empty_like(dY)]
    fos = [fo, ttl.mlp_fwd_buffers(t, act, T, h, f, dev)]
    bos = [bo, ttl.mlp_bwd_buffers(t, act, T, h, f, dev)]
    # Two distinct host batches, alternated, so each step brings in different data.
    Xh = [X.cpu().pin_memory(), (X.cpu().float() * -1).to(torch.bfloat16).pin_memory()]
    dYh = [dY.cpu().pin_memory(), (dY.cpu().float() * -1).to(torch.bfloat16).pin_memory()]
    Zh = [torch.empty((T, h), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dXh = [torch.empty((T, h), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    ev_res = [torch.cuda.Event() for _ in range(2)]
    ev_drained = [torch.cuda.Event() for _ in range(2)]

    def load(i):
        k = i % 2
        with torch.cuda.stream(cp):
            cp.wait_event(ev_free[k])              # slot k no longer read by step i-2
            Xin[k].copy_(Xh[k], non_blocking=True)
            dYin[k].copy_(dYh[k], non_blocking=True)
            ev_in[k].record(cp)

    def run(n):
        load(0)
        for i in range(n):
            k = i % 2
            if i + 1 < n:
                load(i + 1)
            main.wait_event(ev_in[k])
            main.wait_event(ev_drained[k])         # output set k of step i-2 has reached the host
            ttl.tp_mlp_fwd(Xin[k], Wg, Wd, act=act, A_up=Wu, out=fos[k])
            ttl.tp_mlp_bwd(Xin[k], dYin[k], Wg, Wd, fos[k], act=act, A_up=Wu, out=bos[k])
            ev_free[k].record(main)
            ev_res[k].record(main)
            with torch.cuda.stream(cp):
                cp.wait_event(ev_res[k])
                Zh[k].copy_(fos[k]["Z"][0], non_blocking=True)
                dXh[k].copy_(bos[k]["dX"][0], non_blocking=True)
                ev_drained[k].record(cp)
        main.wait_stream(cp)

    run(2)
    # Three timed windows of K steps each; the median window is reported, so that one stall of
    # the host (a shared machine) does not decide the number.
    windows = []
    for _ in range(3):
        dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run(args.steps)
        e1.record()
        torch.cuda.synchronize()
        dist.barrier()
        windows.append(dist.max(e0.elapsed_time(e1)))
    ms = sorted(windows)[1]
    last = (args.steps - 1) % 2
    if not torch.equal(Zh[last].to(dev), fos[last]["Z"][0]):
        raise RuntimeError("e2e: the host copy of the last result does not match the device result")
    del fos, bos
    return {"value": round(dist.world * MLP_FLOPS * args.steps / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "h2d_bytes_per_step": 2 * T * h * 2, "d2h_bytes_per_step": 2 * T * h * 2,
            "ms_per_step": round(ms / args.steps, 4),
            "windows_ms_per_step": [round(w / args.steps, 4) for w in windows],
            "timing": "median of three timed windows of K steps each",
            "pipelining": "H2D of step i+1 and D2H of step i-1 on a copy stream during step i"}


def _flush(torch, buf):
    """Flush L2: write a buffer larger than L2, then read a second one, so the timed kernel
    starts cold and does not pay for writing back the flush's own dirty lines."""
    buf[0].add_(1)
    buf[1].sum()


def bench_shard_reduce(ttl, torch, dev, pk, args):
    T, h = 4096, 8192
    g = torch.Generator(device=dev).manual_seed(2)
    flush = [torch.zeros(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev) for _ in range(2)]
    res = {"workload": "partial_sum_reduce_T4096_h8192", "bytes_model": "RS (t+1)S, AG tS, AR 2tS; S = 64 MiB",
           "l2": "flushed before each timed launch by a 512 MiB write followed by a 512 MiB read",
           "peak_gbs": pk["hbm_gbs"]}
    reps = max(5, min(args.steps, 20))
    for t in (2, 4, 8, 16):
        bufs = [torch.randn((T, h), generator=g, device=dev).to(torch.bfloat16) for _ in range(t)]
        row = {}
        for mode, fn, kind in (("rs", ttl.shard_reduce_scatter, "reduce"), ("ag", ttl.shard_all_gather, "gather"),
                               ("ar", ttl.shard_all_reduce, "reduce")):
            for _ in range(2):
                fn(bufs)
            ttl.trace_enable(True, 1024)
            for _ in range(reps):
                _flush(torch, flush)
                fn(bufs)
            torch.cuda.synchronize()
            recs = [r for r in ttl.trace_read(1024) if r[0] == kind]
            ttl.trace_enable(False)
            ms = statistics.median(r[1] for r in recs)
            by = recs[0][3]
            gbs = by / (ms * 1e-3) / 1e9
            row[mode] = {"gbs": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 4), "us": round(ms * 1e3, 1)}
        res[f"t{t}"] = row
        del bufs
    del flush
    torch.cuda.empty_cache()
    ar8 = res["t8"]["ar"]
    res["roofline"] = pending("hbm", "shard_reduce_kernel<8,AR>", ar8["gbs"],
                              traffic=committed_traffic("shard_reduce_kernel<8,AR>"),
                              bytes_per_launch=2 * 8 * T * h * 2, median_us=ar8["us"],
                              timing=f"median of {reps} launches, L2 flushed before each")
    return res


def bench_gtp(ttl, torch, dev, pk, args):
    L, K, N, M, gdeg = 8, 8192, 2048, 4096, 8
    g = torch.Generator(device=dev).manual_seed(4)
    X = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    shards = [[(torch.randn((K // gdeg, N), generator=g, device=dev) * 0.02).to(torch.bfloat16)
               for _ in range(gdeg)] for _ in range(L)]
    dY = [torch.randn((M, N), generator=g, device=dev).to(torch.bfloat16) for _ in range(L)]
    Y = [torch.empty((M, N), device=dev, dtype=torch.bfloat16) for _ in range(L)]
    dX = torch.empty((M, K), device=dev, dtype=torch.bfloat16)
    slots = [torch.empty((K, N), device=dev, dtype=torch.bfloat16) for _ in range(2)]
    staging = [[torch.empty((K // gdeg, N), device=dev) for _ in range(gdeg)] for _ in range(L)]
    main_grad = [[torch.zeros((K // gdeg, N), device=dev) for _ in range(gdeg)] for _ in range(L)]
    from tensor_transformer_layer_way_gb300 import chain
    runner = chain.GtpChain(ttl, torch, shards, slots)

    def fwd_bwd(folded=False, fin_stream=True, wg_stream=True):
        runner.forward(X, Y, folded=folded)
        runner.backward(X, dY, dX, staging, main_grad, folded=folded, finalize_stream=fin_stream,
                        wgrad_stream=wg_stream)

    runner.forward(X, Y, cold=True)           # cold start: every first gather synchronous
    for _ in range(2):
        fwd_bwd()
    torch.cuda.synchronize()
    res = {"workload": "gtp_chain_L8_h8192_tp4_g8_T4096", "gemm_flops_per_pass": 3 * L * 2.0 * M * K * N}
    # slot_prefetch: the chain's defaults (finalizes and weight gradients on streams of their
    # own); the last variant keeps every launch on the compute stream, so its GEMM launches
    # run undisturbed and their CUDA-event durations give the kernel's own rate.
    for key, folded, fin, wgs in (("slot_prefetch", False, True, True), ("folded", True, True, True),
                                  ("slot_prefetch_wgrad_on_compute_stream", False, True, False),
                                  ("slot_prefetch_all_on_compute_stream", False, False, False)):
        # the wall time untraced (an event pair around every launch costs about 1%), then the
        # per-launch durations from a traced pass of the same passes
        reps = 3
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fwd_bwd(folded, fin, wgs)
        e1.record()
        torch.cuda.synchronize()
        wall = e0.elapsed_time(e1) / reps
        ttl.trace_enable(True, 1 << 14)
        for _ in range(reps):
            fwd_bwd(folded, fin, wgs)
        torch.cuda.synchronize()
        recs = ttl.trace_read(1 << 14)
        ttl.trace_enable(False)
        gm = [r for r in recs if r[0] == "gemm"]
        ga = [r for r in recs if r[0] == "gtp_gather"]
        fi = [r for r in recs if r[0] == "finalize"]
        gemm_ms = sum(r[1] for r in gm) / reps
        res[key] = {"ms_per_fwd_bwd": round(wall, 3),
                    "gemm_tflops": round(sum(r[2] for r in gm) / (sum(r[1] for r in gm) * 1e-3) / 1e12, 1),
                    "gemm_ms": round(gemm_ms, 3),
                    # everything the chain's wall time spends outside the GEMMs: exposed gathers,
                    # finalize work that is not hidden, launch gaps
                    "exposed_ms": round(wall - gemm_ms, 3),
                    # every GEMM FLOP of the pass over the wall time (with GEMMs on two streams
                    # their launch durations overlap, so only this rate is comparable)
                    "chain_tflops": round(res["gemm_flops_per_pass"] / (wall * 1e-3) / 1e12, 1),
                    "finalize_ms": round(sum(r[1] for r in fi) / reps, 3),
                    "finalize_gbs": round(sum(r[3] for r in fi) / (sum(r[1] for r in fi) * 1e-3) / 1e9, 1) if fi else None}
        if ga:
            res[key]["gather_gbs"] = round(sum(r[3] for r in ga) / (sum(r[1] for r in ga) * 1e-3) / 1e9, 1)
    # The gather kernel alone (in the chain it shares HBM with the GEMM it hides behind): the
    # L layers' shards gathered back to back into L distinct slots (512 MiB of traffic, beyond
    # L2), L2 flushed before each repetition, median of 5.  The L launches are replayed from a
    # CUDA graph: issued one by one from Python they arrive about 13.7 us apart, slower than
    # the kernel runs, and the measurement would time the host's launch rate.
    flush = [torch.zeros(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev) for _ in range(2)]
    dst = [torch.empty((K, N), device=dev, dtype=torch.bfloat16) for _ in range(L)]
    gather_bytes = L * 2.0 * K * N * 2
    for l in range(L):   # first calls outside the capture (one-time host set-up)
        ttl.gtp_gather(shards[l], dst[l])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g_gather = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_gather, stream=side):
        for l in range(L):
            ttl.gtp_gather(shards[l], dst[l])
    torch.cuda.synchronize()
    times = []
    for _ in range(5):
        _flush(torch, flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g_gather.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = sorted(times)[len(times) // 2]
    # the same bytes moved by torch's own device copy (one contiguous [K, N] source per layer),
    # timed the same way: the ceiling for copies of this size
    src = [torch.empty((K, N), device=dev, dtype=torch.bfloat16) for _ in range(L)]
    g_copy = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_copy, stream=side):
        for l in range(L):
            dst[l].copy_(src[l])
    torch.cuda.synchronize()
    ctimes = []
    for _ in range(5):
        _flush(torch, flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g_copy.replay()
        e1.record()
        torch.cuda.synchronize()
        ctimes.append(e0.elapsed_time(e1))
    cms = sorted(ctimes)[len(ctimes) // 2]
    del g_gather, g_copy
    res["gather_isolated"] = {"us_per_layer": round(ms * 1e3 / L, 1),
                              "gbs": round(gather_bytes / (ms * 1e-3) / 1e9, 1),
                              "frac": round(gather_bytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                              "torch_copy_same_bytes_gbs": round(gather_bytes / (cms * 1e-3) / 1e9, 1),
                              "bytes": gather_bytes, "l2": "flushed before each repetition of the 8 launches",
                              "timing": "the 8 launches replayed from a CUDA graph (device time; issued one by one "
                                        "from Python they run at the host's launch rate, about 13.7 us per call)"}
    del flush, dst, src
    res["roofline"] = pending("tensor", "gemm_tcgen05_kernel", res["slot_prefetch_all_on_compute_stream"]["gemm_tflops"],
                              path="GEMM launches of the slot_prefetch chain with every launch on the compute "
                                   "stream (the default chain overlaps them, see chain_roofline)")
    res["chain_roofline"] = pending("tensor", "whole chain (all GEMM FLOPs over the fwd+bwd wall time)",
                                    res["slot_prefetch"]["chain_tflops"],
                                    path="slot_prefetch chain, finalizes and weight gradients on their own streams")
    del X, shards, dY, Y, dX, slots, staging, main_grad, runner
    torch.cuda.empty_cache()
    return res


def bench_ce(ttl, torch, dev, pk, args):
    t, T, h, V = 8, 8192, 4096, 151936
    g = torch.Generator(device=dev).manual_seed(5)
    H = torch.randn((T, h), generator=g, device=dev).to(torch.bfloat16)
    W = [(torch.randn((V // t, h), generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(t)]
    target = torch.randint(0, V, (T,), generator=g, device=dev)
    out = ttl.ce_buffers(t, T, h, V, dev)
    res = {"workload": "vocab_parallel_ce_t8_T8192_h4096_V151936"}
    for mode, fused in (("fused_stats", True), ("separate_stats", False)):
        for _ in range(2):
            ttl.vocab_parallel_ce(H, W, target, out=out, fused_stats=fused)
        torch.cuda.synchronize()
        reps = 3
        # the wall time untraced, then the per-launch durations from a traced pass
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            ttl.vocab_parallel_ce(H, W, target, out=out, fused_stats=fused)
        e1.record()
        torch.cuda.synchronize()
        wall = e0.elapsed_time(e1) / reps
        ttl.trace_enable(True, 4096)
        for _ in range(reps):
            ttl.vocab_parallel_ce(H, W, target, out=out, fused_stats=fused)
        torch.cuda.synchronize()
        recs = ttl.trace_read(4096)
        ttl.trace_enable(False)

        def agg(kind, flops=False):
            rr = [r for r in recs if r[0] == kind]
            if not rr:
                return None
            ms = sum(r[1] for r in rr)
            if flops:
                v = sum(r[2] for r in rr) / (ms * 1e-3) / 1e12
                return {"tflops": round(v, 1), "ms": round(ms / reps, 3)}
            v = sum(r[3] for r in rr) / (ms * 1e-3) / 1e9
            return {"gbs": round(v, 1), "frac": round(v / pk["hbm_gbs"], 4), "ms": round(ms / reps, 3)}

        res[mode] = {"ms_per_fwd_bwd": round(wall, 3), "loss": float(out["loss"].item()),
                     "gemm": agg("gemm", True), "stats": agg("ce_stats"), "dlogits": agg("ce_dlogits"),
                     "combine_mean": agg("ce_small")}
    res["roofline"] = pending("tensor", "gemm_tcgen05_kernel", res["fused_stats"]["gemm"]["tflops"],
                              path="LM-head GEMM with fused statistics + dH GEMM")
    dl = res["fused_stats"]["dlogits"]
    res["roofline_hbm"] = pending("hbm", "ce_dlogits_kernel", dl["gbs"])
    del H, W, target, out
    torch.cuda.empty_cache()
    return res


def bench_sp_mlp(ttl, torch, dev, pk, args):
    """The headline workload with sequence parallelism: X and dZ as 8 token slabs of 1024 rows,
    the all-gather and reduce-scatter folded into the GEMMs (no collective kernel runs)."""
    t, T, h, f, act = MLP["t"], MLP["T"], MLP["h"], MLP["f"], MLP["act"]
    fs, slab = f // t, T // t
    g = torch.Generator(device=dev).manual_seed(MLP["seed"])

    def rnd(shape, std):
        return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)

    Xs = [rnd((slab, h), 1.0) for _ in range(t)]
    dZs = [rnd((slab, h), 1.0) for _ in range(t)]
    Wg = [rnd((h, fs), 0.02) for _ in range(t)]
    Wu = [rnd((h, fs), 0.02) for _ in range(t)]
    Wd = [rnd((fs, h), 0.02) for _ in range(t)]
    fo = ttl.sp_mlp_fwd(Xs, Wg, Wd, act=act, A_up=Wu)
    bo = ttl.sp_mlp_bwd(Xs, dZs, Wg, Wd, fo, act=act, A_up=Wu)

    def step():
        ttl.sp_mlp_fwd(Xs, Wg, Wd, act=act, A_up=Wu, out=fo)
        ttl.sp_mlp_bwd(Xs, dZs, Wg, Wd, fo, act=act, A_up=Wu, out=bo)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(10, min(args.steps, 50))
    # the wall time untraced, then the per-launch durations from a traced pass
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    ttl.trace_enable(True, 1 << 14)
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    recs = ttl.trace_read(1 << 14)
    ttl.trace_enable(False)
    gm = [r for r in recs if r[0] == "gemm"]
    res = {"workload": "qwen3_8b_swiglu_mlp_t8_T8192_sequence_parallel_fwd_bwd", "ms_per_step": round(ms, 4),
           "tflops": round(MLP_FLOPS / (ms * 1e-3) / 1e12, 1),
           "gemm_tflops": round(sum(r[2] for r in gm) / (sum(r[1] for r in gm) * 1e-3) / 1e12, 1),
           "launches_per_step": len(recs) / n, "collective_kernels_per_step": 0}
    res["roofline"] = pending("tensor", "gemm_tcgen05_kernel", res["gemm_tflops"])
    del Xs, dZs, Wg, Wu, Wd, fo, bo
    torch.cuda.empty_cache()
    return res


def bench_embedding(ttl, torch, dev, pk, args):
    """Vocab-parallel embedding: 151936 x 4096 table in 8 vocab shards, 8192 token ids."""
    t, T, h, V = 8, 8192, 4096, 151936
    g = torch.Generator(device=dev).manual_seed(6)
    E = [(torch.randn((V // t, h), generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(t)]
    ids = torch.randint(0, V, (T,), generator=g, device=dev)
    dY = torch.randn((T, h), generator=g, device=dev).to(torch.bfloat16)
    out = [torch.empty((T, h), device=dev, dtype=torch.bfloat16) for _ in range(t)]
    dE = [torch.zeros((V // t, h), device=dev) for _ in range(t)]
    flush = [torch.zeros(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev) for _ in range(2)]
    reps = 5
    res = {"workload": "vocab_parallel_embedding_t8_T8192_h4096_V151936",
           "l2": "flushed before each timed launch by a 512 MiB write followed by a 512 MiB read"}
    for name, fn in (("fwd_literal", lambda: ttl.vocab_parallel_embedding_fwd(ids, E, out=out, literal=True)),
                     ("fwd_fused", lambda: ttl.vocab_parallel_embedding_fwd(ids, E, out=out, literal=False)),
                     ("bwd", lambda: ttl.vocab_parallel_embedding_bwd(ids, dY, dE))):
        fn()
        torch.cuda.synchronize()
        ttl.trace_enable(True, 1024)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ms = 0.0
        for _ in range(reps):
            _flush(torch, flush)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
        recs = ttl.trace_read(1024)
        ttl.trace_enable(False)
        by = sum(r[3] for r in recs) / reps
        kms = sum(r[1] for r in recs) / reps
        res[name] = {"ms": round(ms / reps, 4), "kernel_gbs": round(by / (kms * 1e-3) / 1e9, 1),
                     "frac": round(by / (kms * 1e-3) / 1e9 / pk["hbm_gbs"], 4), "launches": len(recs) // reps}
    res["roofline"] = pending("hbm", "embed_gather_kernel", res["fwd_fused"]["kernel_gbs"],
                              bytes_per_launch=T * h * 2 * (1 + t))
    del E, ids, dY, out, dE, flush
    torch.cuda.empty_cache()
    return res


def bench_attention(ttl, torch, dev, pk, args):
    """Head-split TP attention block forward + backward at the Qwen3-8B shape: T=8192 tokens,
    h=4096, 32 query / 8 KV heads of 128, t=8 (4 query heads + 1 KV head per shard); with
    --attn-small the profiling case T=4096, 8 query / 2 KV heads, t=2."""
    t, T, h, n_q, n_kv, d = (2, 4096, 4096, 8, 2, 128) if args.attn_small else (8, 8192, 4096, 32, 8, 128)
    qc, kc = n_q // t * d, n_kv // t * d
    g = torch.Generator(device=dev).manual_seed(7)

    def rnd(shape, std):
        return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)

    X, dY = rnd((T, h), 1.0), rnd((T, h), 1.0)
    Wq = [rnd((h, qc), h ** -0.5) for _ in range(t)]
    Wk = [rnd((h, kc), h ** -0.5) for _ in range(t)]
    Wv = [rnd((h, kc), h ** -0.5) for _ in range(t)]
    Wo = [rnd((qc, h), (n_q * d) ** -0.5) for _ in range(t)]
    kw = dict(n_q=n_q, n_kv=n_kv, d=d)
    fo = ttl.tp_attn_fwd(X, Wq, Wk, Wv, Wo, **kw)
    bo = ttl.tp_attn_bwd(X, dY, Wq, Wk, Wv, Wo, fo, **kw)

    def step():
        ttl.tp_attn_fwd(X, Wq, Wk, Wv, Wo, out=fo, **kw)
        ttl.tp_attn_bwd(X, dY, Wq, Wk, Wv, Wo, fo, out=bo, **kw)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(5, min(args.steps, 20))
    # the wall time untraced, then the per-launch durations from a traced pass
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    ttl.trace_enable(True, 1 << 14)
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    recs = ttl.trace_read(1 << 14)
    ttl.trace_enable(False)
    flops = sum(r[2] for r in recs) / n        # algorithmic: causal contractions count their triangle
    gm = [r for r in recs if r[0] == "gemm"]
    co = [r for r in recs if r[0] == "attn_core"]
    sm = [r for r in recs if r[0] == "softmax"]
    sm_gbs = sum(r[3] for r in sm) / (sum(r[1] for r in sm) * 1e-3) / 1e9
    name = f"attention_t{t}_T{T}_h{h}_q{n_q}_kv{n_kv}_d{d}_fwd_bwd"
    res = {"workload": ("qwen3_8b_" if not args.attn_small else "") + name, "ms_per_step": round(ms, 4),
           "tflops": round(flops / (ms * 1e-3) / 1e12, 1), "flops_per_step": flops,
           "gemm_tflops": round(sum(r[2] for r in gm) / (sum(r[1] for r in gm) * 1e-3) / 1e12, 1),
           "core_tflops": round(sum(r[2] for r in co) / (sum(r[1] for r in co) * 1e-3) / 1e12, 1),
           "core_share_of_step": round(sum(r[1] for r in co) / n / ms, 4),
           "softmax_gbs": round(sm_gbs, 1), "softmax_frac_of_hbm": round(sm_gbs / pk["hbm_gbs"], 4),
           "softmax_share_of_step": round(sum(r[1] for r in sm) / n / ms, 4),
           "launches_per_step": len(recs) / n,
           "launches": [{"kind": r[0], "ms": round(r[1], 4),
                         "tflops": round(r[2] / (r[1] * 1e-3) / 1e12, 1) if r[2] else None,
                         "gbs": round(r[3] / (r[1] * 1e-3) / 1e9, 1) if not r[2] else None}
                        for r in recs[-(len(recs) // n):]]}
    res["roofline"] = pending("tensor", "attn_fwd_core_kernel + attn_bwd_core_kernel + attn_bwd_kv_kernel",
                              res["core_tflops"], share_of_step=res["core_share_of_step"])
    res["step_roofline"] = pending("tensor", "whole block step (cores, projections, row dot, all-reduces)",
                                   res["tflops"])
    del X, dY, Wq, Wk, Wv, Wo, fo, bo
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ the oracle (CPU baseline / reference arm)

def oracle_sample(tokens: int):
    import numpy as np
    import synth_inputs as si
    g = si.generator(MLP["seed"])
    X = si.randn_bf16(g, (tokens, MLP["h"])).float().numpy().astype(np.float64)
    W = {k: si.randn_bf16(g, s, 0.02).float().numpy().astype(np.float64)
         for k, s in (("Wg", (MLP["h"], MLP["f"])), ("Wu", (MLP["h"], MLP["f"])), ("Wd", (MLP["f"], MLP["h"])))}
    dY = si.randn_bf16(g, (tokens, MLP["h"])).float().numpy().astype(np.float64)
    return X, W, dY


def time_oracle(tokens: int, reps: int, warm: int = 0, min_seconds: float = 0.0):
    """Times the oracle's fwd+bwd on `tokens` rows: `warm` untimed runs, then at least `reps`
    timed ones and more until `min_seconds` of timed work has passed."""
    from oracle import tp_mlp
    X, W, dY = oracle_sample(tokens)
    times = []
    i = 0
    while i < warm + reps or sum(times) < min_seconds:
        t0 = time.perf_counter()
        fwd = tp_mlp.tp_mlp_forward(X, W, MLP["t"], MLP["act"])
        tp_mlp.tp_mlp_backward(X, W, MLP["t"], MLP["act"], dY, fwd)
        if i >= warm:
            times.append(time.perf_counter() - t0)
        i += 1
    flops = MLP_FLOPS * tokens / MLP["T"]
    return flops, times


def cpu_cores():
    """Host threads the oracle's numpy runs on: the usable cores, capped by OMP_NUM_THREADS."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count()
    omp = os.environ.get("OMP_NUM_THREADS", "")
    return min(n, int(omp)) if omp.isdigit() and int(omp) > 0 else n


def cpu_baseline(tokens: int, seconds: float) -> dict:
    """The oracle on `tokens` of the workload's token rows (full weights), repeated until
    `seconds` of wall time have passed; throughput over all repetitions."""
    flops, times = time_oracle(tokens, 1, min_seconds=seconds)
    total = sum(times)
    return {"value": round(flops * len(times) / total / 1e12, 5), "unit": "TFLOP/s", "cores": cpu_cores(),
            "kind": "oracle",
            "extrapolated_full_step_s": round(total / len(times) * MLP["T"] / tokens, 1),
            "sample": f"fp64 numpy oracle, sharded t=8 SwiGLU MLP fwd+bwd on {tokens} of 8192 tokens "
                      f"(full weights), {len(times)} repetitions, {total:.1f} s"}


def _repeat(fn, seconds: float, min_reps: int = 1) -> list:
    times = []
    while len(times) < min_reps or sum(times) < seconds:
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
    return times


def cpu_reduce(seconds: float) -> dict:
    """Config 2 in full: the oracle's all_reduce_mirror over t in {2,4,8,16} buffers of
    [4096, 8192], once on one thread and once on every core (the same function on row bands,
    one band per thread; numpy releases the GIL inside its array operations).  GB/s counts
    the same algorithmic bytes as the kernel (2 t S, S = 64 MiB of bf16)."""
    from concurrent.futures import ThreadPoolExecutor
    import synth_inputs as si
    from oracle import collectives
    n = cpu_cores()
    T, h = 4096, 8192
    by_t = {}
    for t in (2, 4, 8, 16):
        bufs = [b.float().numpy() for b in si.partial_sum_buffers(t, T, h, seed=2)]
        nbytes = 2 * t * T * h * 2
        one = _repeat(lambda: collectives.all_reduce_mirror(bufs), 0.0)
        step = max(t, (T // n) // t * t)
        bands = [slice(r, min(T, r + step)) for r in range(0, T, step)]

        def banded():
            with ThreadPoolExecutor(len(bands)) as ex:
                list(ex.map(lambda sl: collectives.all_reduce_mirror([b[sl] for b in bufs]), bands))
        many = _repeat(banded, min(seconds / 8, 2.0), 2)
        by_t[f"t{t}"] = {"gbs_1_core": round(nbytes / min(one) / 1e9, 2),
                         "gbs_all_cores": round(nbytes / min(many) / 1e9, 2),
                         "s_1_core": round(min(one), 3), "s_all_cores": round(min(many), 3)}
        del bufs
    return {"value": by_t["t8"]["gbs_all_cores"], "unit": "GB/s", "cores": n, "kind": "oracle",
            "value_1_core": by_t["t8"]["gbs_1_core"], "by_t": by_t,
            "sample": "the full workload: all_reduce_mirror (fp32 sum in buffer order, one bf16 rounding) of "
                      "t = 2, 4, 8, 16 buffers [4096, 8192], on 1 thread and on every core; value is t = 8"}


def cpu_gtp(tokens: int, seconds: float) -> dict:
    """Config 4 on a token sample: all 8 layers with the full [8192, 2048] slices as 8 row
    shards, the first `tokens` of 4096 token rows: gather + forward GEMM, gather + dgrad GEMM,
    the literal per-token-group wgrad reduce-scatter, and the deferred finalize."""
    import numpy as np
    import synth_inputs as si
    from oracle import gtp
    L, K, N, g, M = 8, 8192, 2048, 8, 4096
    inp = si.gtp_inputs(L, K, N, tokens, seed=4)
    X = inp["X"].float().numpy().astype(np.float64)
    W = [w.float().numpy().astype(np.float64) for w in inp["W"]]
    dY = [d.float().numpy().astype(np.float64) for d in inp["dY"]]
    shards = [gtp.shard_rows(w, g) for w in W]
    main_grad = [[np.zeros((K // g, N)) for _ in range(g)] for _ in range(L)]

    def fwd_bwd():
        for l in range(L):
            gtp.forward_gemm(X, gtp.gather(shards[l]))
        staging = [None] * L
        for l in range(L - 1, -1, -1):
            gtp.dgrad_gemm(dY[l], gtp.gather(shards[l]))
            staging[l] = gtp.wgrad_reduce_scatter(X, dY[l], g)
        gtp.deferred_finalize(main_grad, staging)
    times = _repeat(fwd_bwd, seconds)
    flops = 3 * L * 2.0 * tokens * K * N
    per = sum(times) / len(times)
    return {"value": round(flops / per / 1e12, 5), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "extrapolated_full_s": round(per * M / tokens, 2),
            "sample": f"fp64 numpy oracle, 8-layer GTP chain fwd+bwd on {tokens} of {M} token rows with the full "
                      f"slices; {len(times)} repetitions; the full-size time is extrapolated (x{M // tokens}, "
                      "GEMM work scales with tokens)"}


def cpu_ce(tokens: int, seconds: float) -> dict:
    """Config 5 on a token sample: the full [151936, 4096] head in 8 vocab shards, `tokens` of
    8192 token rows: logits, statistics, combine, dlogits and dH."""
    import numpy as np
    import synth_inputs as si
    from oracle import vocab_ce
    T, h, V, t = 8192, 4096, 151936, 8
    inp = si.ce_inputs(tokens, h, V, seed=5)
    H = inp["H"].float().numpy().astype(np.float64)
    W = inp["W"].float().numpy().astype(np.float64)
    target = inp["target"].numpy()
    del inp
    times = _repeat(lambda: vocab_ce.vocab_parallel_ce(H, W, target, t), seconds)
    per = sum(times) / len(times)
    flops = 2 * 2.0 * tokens * V * h
    return {"value": round(flops / per / 1e12, 5), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "extrapolated_full_s": round(per * T / tokens, 2),
            "sample": f"fp64 numpy oracle, vocab-parallel CE (t=8) on {tokens} of {T} tokens with the full head; "
                      f"{len(times)} repetitions; the full-size time is extrapolated (x{T // tokens})"}


def cpu_sp(tokens: int, seconds: float) -> dict:
    """The sequence-parallel MLP on a token sample: t = 8 slabs of tokens/8 rows, full weights."""
    from oracle import tp_mlp
    X, W, dY = oracle_sample(tokens)
    t = MLP["t"]
    w = tokens // t
    Xs = [X[r * w:(r + 1) * w] for r in range(t)]
    dZs = [dY[r * w:(r + 1) * w] for r in range(t)]

    def run():
        fwd = tp_mlp.sp_mlp_forward(Xs, W, t, MLP["act"])
        tp_mlp.sp_mlp_backward(Xs, W, t, MLP["act"], dZs, fwd)
    times = _repeat(run, seconds)
    per = sum(times) / len(times)
    flops = MLP_FLOPS * tokens / MLP["T"]
    return {"value": round(flops / per / 1e12, 5), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "extrapolated_full_s": round(per * MLP["T"] / tokens, 2),
            "sample": f"fp64 numpy oracle, sequence-parallel SwiGLU MLP fwd+bwd on {tokens} of {MLP['T']} tokens "
                      f"(8 slabs, full weights); {len(times)} repetitions; full-size time extrapolated"}


def cpu_embedding(seconds: float) -> dict:
    """The embedding lookup on a shard sample: all 8192 ids against 2 of the 8 vocab shards
    (each [18992, 4096]); the full lookup is extrapolated to 8 shards."""
    import numpy as np
    import synth_inputs as si
    from oracle import embedding
    T, h, V, t, ns = 8192, 4096, 151936, 8, 2
    Vs = V // t
    g = si.generator(6)
    E = [si.randn_bf16(g, (Vs, h), 0.02).float().numpy().astype(np.float64) for _ in range(ns)]
    import torch
    ids = torch.randint(0, V, (T,), generator=g).numpy()

    def run():
        parts = [embedding.shard_lookup(ids, E[i], i * Vs) for i in range(ns)]
        out = parts[0]
        for p in parts[1:]:
            out = out + p
    times = _repeat(run, seconds)
    full = sum(times) / len(times) * t / ns
    nbytes = T * h * 2 * (1 + t)
    return {"value": round(nbytes / full / 1e9, 3), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
            "extrapolated_full_s": round(full, 3),
            "sample": f"fp64 numpy oracle, masked lookup of all {T} ids in {ns} of {t} vocab shards and their sum; "
                      f"{len(times)} repetitions; time extrapolated to {t} shards; GB/s on the kernel's algorithmic bytes"}


def cpu_attention(seconds: float) -> dict:
    """The attention block's forward on sampled output rows at the Qwen3-8B shape: rows 127,
    255, 383 and 511 of 8192 (each needs the keys and values of the tokens up to it)."""
    import numpy as np
    import synth_inputs as si
    from oracle import attention
    T, h, n_q, n_kv, d = 512, 4096, 32, 8, 128
    inp = si.attn_inputs(T, h, n_q, n_kv, d, seed=6)
    X = inp["X"].float().numpy().astype(np.float64)
    W = {k: inp[k].float().numpy().astype(np.float64) for k in ("Wq", "Wk", "Wv", "Wo")}
    rows = [127, 255, 383, 511]
    times = _repeat(lambda: attention.forward_rows(X, W, n_q, n_kv, d, rows, t=8), seconds)
    per = sum(times) / len(times)
    m = max(rows) + 1
    flops = 2.0 * m * h * 2 * n_kv * d + sum(2.0 * h * n_q * d * 2 + 4.0 * d * (r + 1) * n_q for r in rows)
    return {"value": round(flops / per / 1e12, 5), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"fp64 numpy oracle, forward output rows {rows} of the T=8192 block (K/V projections of the "
                      f"first {m} tokens, then per-row attention and W_O); {len(times)} repetitions; forward only, "
                      "no extrapolation"}


def component_cpu_baselines(out: dict, args):
    """A cpu_baseline object for every component of the JSON line (rank 0, N = 1)."""
    sec = max(1.0, args.cpu_seconds / 4)
    legs = {"shard_reduce": lambda: cpu_reduce(sec), "gtp_chain": lambda: cpu_gtp(128, sec),
            "vocab_ce": lambda: cpu_ce(32, sec), "sp_mlp": lambda: cpu_sp(args.cpu_tokens, sec),
            "vocab_embedding": lambda: cpu_embedding(sec), "tp_attention": lambda: cpu_attention(sec)}
    for name, fn in legs.items():
        if isinstance(out.get(name), dict):
            out[name]["cpu_baseline"] = fn()


def run_reference(args, dist):
    if dist.rank != 0:
        return None
    tokens = args.cpu_tokens
    flops, times = time_oracle(tokens, args.steps, args.warmup)
    total = sum(times)
    v = flops * args.steps / total / 1e12
    return {"impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "TFLOP/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": {"workload": WORKLOAD, "t": 8, "tokens_per_step": tokens},
            "cpu_baseline": {"value": round(v, 5), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{tokens} of 8192 tokens per step, full weights"},
            "e2e": {"value": round(v, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.impl == "reference" and os.environ.get("RANK", "0") == "0":
        # Under torchrun every rank gets OMP_NUM_THREADS=1; rank 0 alone runs the oracle here (the
        # other ranks exit without work), so it takes every core.  Set before numpy is loaded.
        try:
            ncores = str(len(os.sched_getaffinity(0)))
        except AttributeError:
            ncores = str(os.cpu_count())
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
            os.environ[var] = ncores
    dist = Dist(args.gpus)
    try:
        if args.only:
            import torch
            import tensor_transformer_layer_way_gb300 as ttl
            torch.cuda.set_device(dist.local)
            fn = {"sp_mlp": bench_sp_mlp, "shard_reduce": bench_shard_reduce, "gtp_chain": bench_gtp,
                  "vocab_ce": bench_ce, "vocab_embedding": bench_embedding,
                  "tp_attention": bench_attention}[args.only]
            clocks = Clocks(dist.local)
            clocks.start()
            pk = peaks()
            comp = fn(ttl, torch, torch.device("cuda", dist.local), pk, args)
            clocks.stop()
            finish_rooflines(comp, pk, clocks.window())
            out = {"component": args.only, args.only: comp}
        elif args.impl == "reference":
            out = run_reference(args, dist)
        else:
            out = run_ours(args, dist)
            if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
                out["cpu_baseline"] = cpu_baseline(args.cpu_tokens, args.cpu_seconds)
                component_cpu_baselines(out, args)
        if dist.rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
