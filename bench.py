#!/usr/bin/env python3
"""Throughput of the GB300 FP8 delayed-scaling linear layer (fwd + bwd + update).

One step = one pass of the whole hot path over one batch: the fused amax +
scaled cast + transposed copy of X, W and dY, the fprop / dgrad / wgrad FP8
GEMMs with the dequant + amax epilogue, and the delayed-scaling update of all
five tensors (Fp8Linear.step).  The headline workload is the largest layer,
the 70B-shaped MLP (M = 8192 tokens, K = 8192, N = 28672; Student-t X with
outlier channels; HYBRID, history 1024, margin 1).  Inputs are synthetic and
seeded (fp8_workloads.py) and resident in HBM; two (X, dY) batches alternate,
each step reading more than the 129 MB L2.  Under torchrun (N > 1) each rank
is a data-parallel replica on its own tokens: the five amaxes are combined by
an all-reduce(MAX) and dW by the FP8 all-reduce (fp8_allreduce) every step.

Prints ONE JSON line (rank 0).  Metric: layer TFLOPS = 6 M N K per step over
the device time of K steps (CUDA events, max over ranks).  Added keys:
  roofline      the dominant kernel (the tcgen05 GEMM), achieved TFLOP/s vs the
                FP8 peak derived from MEASURED_PEAKS.json (bf16 x 2), and vs
                SMs x 16384 FLOP/clk x the SM clock the timed GEMM launches
                ran at, measured inside the kernel (peak_clock), and x the
                maximum SM clock (peak_boost)
  cast_roofline the fused cast kernels, achieved GB/s vs measured HBM copy
  sustained     the same step back to back for a few seconds, with its own
                clock record (the power-capped regime)
  sweep_2e28    the standalone quantize sweep's largest tensor (2^28 BF16
                elements): amax and cast + transposed copy GB/s, L2 flushed
  mlp7b         the 7B-shaped layer step (M 8192, K 4096, N 11008)
  e2e           same metric with X, dY copied in from pinned host memory and
                Y, dX, dW copied back every step
  cpu_baseline  the CPU oracle timed on a sample of the same layer
  clocks        nvidia-smi SM clocks / throttle reasons sampled while timing

``--impl reference`` times the CPU oracle (the only reference for this
method) on a bounded per-step sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fp8_workloads as wl  # noqa: E402

METRIC = "FP8 linear fwd+bwd TFLOPS & % GB300 FP8 peak; cast/amax GB/s % of HBM peak"
FP8_OVER_BF16 = 2.0       # nominal dense FP8 / BF16 tensor-core ratio (4.5 / 2.25 PFLOP/s)
FP8_FLOP_PER_CLK_SM = 16384   # dense FP8 tensor-core FLOP per clock per SM (2 x BF16's 8192)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="mlp70b", choices=["mlp7b", "mlp70b", "drift", "tiny"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--sustained-seconds", type=float, default=3.0,
                   help="length of the back-to-back sustained loop (0: skip)")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the mlp7b and sweep_2e28 keys")
    p.add_argument("--secondary", action="store_true",
                   help="also time the 70B-shaped layer, the cast sweep and the other "
                        "kernels of the path (extra keys)")
    p.add_argument("--part", action="append", default=[], choices=SECONDARY_PARTS,
                   help="with --secondary: run only these parts (repeatable)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------- distributed --

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class L2Flush:
    """L2 flush before a timed launch: a 256 MB write (larger than the 129 MB
    L2), then a 256 MB read.  The read evicts the write's dirty lines, so
    their write-back to DRAM is not charged to the launch that follows (with
    the write alone, a standalone amax timed 5 % slower than from a clean L2)."""

    def __init__(self):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.r.sum()


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling (100 ms) around a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            except Exception:
                pass
            target = f"GPU-{uuid}" if uuid and not uuid.startswith("GPU-") else uuid
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if target:
                cmd += ["-i", target]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as fh:
            lines = fh.readlines()
        os.unlink(self.path)
        return self.summarize(lines)

    @staticmethod
    def summarize(lines):
        """Median SM clock under load, the range seen, the peak power draw and
        the throttle reasons that were active in any sample, from nvidia-smi
        CSV lines in FIELDS order."""
        rows = []
        for line in lines:
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, smax = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            try:
                pw = float(parts[2])
            except ValueError:
                pw = None
            rows.append((sm, smax, pw, parts[3:]))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for *_, r in rows:
            for nm, v in zip(names, r[1:5]):
                if v.lower() == "active":
                    reasons.add(nm)
        loaded = [r[0] for r in rows if r[0] > 0.5 * rows[0][1]] or [r[0] for r in rows]
        powers = [r[2] for r in rows if r[2] is not None]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "sm_min_mhz": min(loaded), "power_w_max": max(powers) if powers else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------ our GPU path --

class EventTimer:
    def __init__(self):
        self.pairs = {}
        self.enabled = True

    def time(self, key, fn):
        if not self.enabled:
            fn()
            return
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        self.pairs.setdefault(key, []).append((s, e))

    def mean_ms(self, key):
        return statistics.mean(s.elapsed_time(e) for s, e in self.pairs[key])


def gemm_traffic(workload: str):
    """Per-launch DRAM bytes of the GEMM from the committed ncu summary, or
    None when the kernel source changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"gemm_tn_kernel.{workload}.traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    src = open(os.path.join(ROOT, "fp8_mixed_precision_amax_gb300", "csrc", "gemm.cu"), "rb").read()
    if hashlib.sha256(src).hexdigest() != d.get("gemm_cu_sha256"):
        return None
    return d.get("bytes_per_launch_mean")


def clock_peak(tflop_per_mhz: float, mhz):
    """Dense FP8 tensor peak at an SM clock, TFLOP/s (None without a clock)."""
    return None if not mhz else tflop_per_mhz * mhz


def run_layer_bench(f, w: wl.Workload, args, world, pk, peak_kind, sustained_s: float = 0.0,
                    e2e: bool = True):
    dev = torch.device("cuda")
    W = wl.layer_weight(w, dev)
    xs = [wl.layer_x(w, s, dev) for s in (0, 1)]
    dys = [wl.layer_dy(w, s, dev) for s in (0, 1)]
    lin = f.Fp8Linear(W, w.M, f.Recipe(margin=w.margin, history_len=w.history_len,
                                       hybrid=w.hybrid))
    stream = torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tflop_per_mhz = sms * FP8_FLOP_PER_CLK_SM * 1e6 / 1e12
    launches_per_step = 5
    exchange = None
    if world > 1:
        # data-parallel replicas: MAX of the five amaxes so every replica
        # derives the same scales, and the FP8 all-reduce of dW (amax, own
        # scale, MIN of the scales, cast, all-to-all of code shards,
        # decode-and-sum of this rank's shard, all-gather of BF16 shards)
        dW_sum = torch.empty_like(lin.dW)
        fg_w = f.E5M2 if w.hybrid else f.E4M3
        launches_per_step += 4          # amax, scale, cast, decode-and-sum

        def exchange():
            f.allreduce_amax(lin.meta)
            f.fp8_allreduce(lin.dW, fg_w, 0, out=dW_sum)

    def step(i):
        lin.forward(xs[i % 2])
        lin.backward(dys[i % 2])
        if exchange:
            exchange()
        lin.update()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    f.fp8_sync_status()

    def timed(run_step, steps):
        barrier(world)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            run_step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(t0.elapsed_time(t1), world)

    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.25)
    ms_eager = timed(step, args.steps)
    graphs = None
    if world == 1:
        # the same step recorded once per input batch and replayed
        graphs = [lin.capture_step(xs[k], dys[k]) for k in (0, 1)]
        for i in range(3):
            graphs[i % 2].replay()
        torch.cuda.synchronize()
        ms_graph = timed(lambda i: graphs[i % 2].replay(), args.steps)
        ms = min(ms_eager, ms_graph)
    else:
        ms_graph, ms = None, ms_eager

    # per-kernel breakdown: the same step issued as its individual kernel
    # launches through the C ABI (the grouped X+W cast, fprop, the dY cast,
    # the grouped dgrad+wgrad GEMM, the update), each between CUDA events.
    # The standalone entry points overwrite an amax (a one-word memset before
    # the kernel), so the launches are timed without amax pointers and the
    # events hold the kernels alone; the fused amax itself costs one atomic
    # per CTA.  A short
    # device-side sleep first lets the host enqueue well ahead, and the first
    # steps run without events, so the timed launches run back to back under
    # steady load and no host latency falls between an event and its kernel.
    tm = EventTimer()
    m = lin.meta
    fg = f.E5M2 if w.hybrid else f.E4M3
    E4 = f.E4M3
    nb = max(10, min(args.steps, 100))
    nb_warm = max(args.warmup, 10)
    # the SM clock the GEMM launches run at, measured inside the kernels
    # (fp8_set_clock_probe: the first CTA's %clock64 cycles over its
    # %globaltimer nanoseconds), for the clock-derived peak
    probe = torch.zeros(2, dtype=torch.int64, device=dev)
    torch.cuda.synchronize()
    torch.cuda._sleep(50_000_000)          # ~25 ms at 2 GHz: room to enqueue ahead
    for i in range(nb_warm + nb):
        tm.enabled = i >= nb_warm
        f.fp8_set_clock_probe(probe if tm.enabled else None)
        X, dY = xs[i % 2], dys[i % 2]
        tm.time("cast_XW", lambda: f.fp8_quantize_transpose_grouped(
            [(X, m.scale[0:1], lin.X8, lin.X8t, None), (W, m.scale[1:2], lin.W8, lin.W8t, None)],
            E4))
        tm.time("gemm_fprop", lambda: f.fp8_gemm_tn(lin.X8, E4, lin.W8, E4, m.scale_inv[0:1],
                                                    m.scale_inv[1:2], lin.Y, None))
        tm.time("cast_dY", lambda: f.fp8_quantize_transpose(dY, m.scale[3:4], fg, lin.dY8,
                                                            lin.dY8t))
        tm.time("gemm_bwd", lambda: f.fp8_gemm_tn_grouped(
            [(lin.dY8, fg, lin.W8t, E4, m.scale_inv[3:4], m.scale_inv[1:2], lin.dX, None),
             (lin.dY8t, fg, lin.X8t, E4, m.scale_inv[3:4], m.scale_inv[0:1], lin.dW, None)]))
        tm.time("update", lambda: lin.update())
    f.fp8_set_clock_probe(None)
    torch.cuda.synchronize()
    clk = clocks.stop()
    f.fp8_sync_status()
    pcyc, pns = (int(v) for v in probe.cpu())
    gemm_mhz = pcyc / pns * 1e3 if pns > 0 else None

    M, N, K = w.M, w.N, w.K
    flops = 6 * M * N * K
    value = world * args.steps * flops / (ms / 1e3) / 1e12
    gemm_ms = {k: tm.mean_ms(k) for k in ("gemm_fprop", "gemm_bwd")}
    gemm_flops = {"gemm_fprop": 2 * M * N * K, "gemm_bwd": 4 * M * N * K}
    cast_ms = {k: tm.mean_ms(k) for k in ("cast_XW", "cast_dY")}
    upd_ms = tm.mean_ms("update")
    fp8_peak = pk["bf16_tflops"] * FP8_OVER_BF16
    # algorithmic flops of the GEMM launches over their summed durations
    achieved = sum(gemm_flops.values()) / (sum(gemm_ms.values()) / 1e3) / 1e12
    cast_bytes = {"cast_XW": 4 * M * K + 4 * N * K, "cast_dY": 4 * M * N}
    cast_gbs = sum(cast_bytes.values()) / (sum(cast_ms.values()) / 1e3) / 1e9
    traffic = gemm_traffic(w.name)
    pc = clock_peak(tflop_per_mhz, gemm_mhz)
    pb = clock_peak(tflop_per_mhz, clk.get("sm_max_mhz"))
    res = {
        "value": value, "ms_per_step": ms / args.steps,
        "launch": "CUDA graph replay" if graphs and ms == ms_graph else "eager",
        "ms_per_step_eager": ms_eager / args.steps,
        "ms_per_step_graph": ms_graph / args.steps if ms_graph else None,
        "roofline": {"bound": "tensor", "kernel": "gemm_tn_kernel", "achieved": achieved,
                     "peak": fp8_peak, "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                     "traffic": traffic,
                     "peak_basis": f"{peak_kind} bf16 burst {pk['bf16_tflops']} x {FP8_OVER_BF16} "
                                   f"(of {peak_kind})",
                     "peak_clock": {"value": pc, "frac": achieved / pc if pc else None,
                                    "sm_mhz": gemm_mhz, "sms": sms,
                                    "basis": f"{sms} SMs x {FP8_FLOP_PER_CLK_SM} FLOP/clk x the "
                                             "SM clock the timed GEMM launches ran at, measured "
                                             "in the kernel (%clock64 cycles over %globaltimer "
                                             "ns of its first CTA, fp8_set_clock_probe)",
                                    "nvidia_smi_median_mhz": clk.get("sm_mhz")},
                     "peak_boost": {"value": pb, "frac": achieved / pb if pb else None,
                                    "sm_mhz": clk.get("sm_max_mhz")},
                     "launches_per_step": {"gemm_fprop": "fprop", "gemm_bwd": "dgrad+wgrad"},
                     "per_launch_ms": gemm_ms,
                     "per_launch_tflops": {k: gemm_flops[k] / (v / 1e3) / 1e12
                                           for k, v in gemm_ms.items()}},
        "cast_roofline": {"bound": "hbm", "kernel": "quantize_transpose_kernel",
                          "achieved": cast_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                          "frac": cast_gbs / pk["hbm_gbs"],
                          "bytes_per_element": 4,
                          "per_cast_gbs": {k: cast_bytes[k] / (v / 1e3) / 1e9
                                           for k, v in cast_ms.items()},
                          "update_us": upd_ms * 1e3},
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
        "breakdown_ms": {**gemm_ms, **cast_ms, "update": upd_ms},
    }

    if sustained_s > 0:
        # the launch mode (graph replays or eager steps) that timed faster
        res["sustained"] = run_sustained(graphs if res["launch"] != "eager" else None, step, timed,
                                         sustained_s, ms / args.steps, flops, world,
                                         tflop_per_mhz, pk)
    if e2e:
        res["e2e"] = run_e2e(f, lin, xs[0], dys[0], args, world, flops)
        res["e2e"]["full_outputs"] = {
            k: v for k, v in run_e2e(f, lin, xs[0], dys[0], args, world, flops,
                                     readback="outputs").items() if k != "overlap"}
    return res


def run_sustained(graphs, step, timed, seconds, ms_step, flops, world, tflop_per_mhz, pk):
    """The same step back to back for about ``seconds`` (graph replays or
    eager steps, whichever timed faster), timed with CUDA events around the
    whole loop, with its own clock record: the regime where the GPU runs at
    its power limit."""
    n = max(10, int(seconds * 1e3 / max(ms_step, 1e-3)))
    run = (lambda i: graphs[i % 2].replay()) if graphs else step
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.25)
    ms = timed(run, n)
    clk = clocks.stop()
    value = world * n * flops / (ms / 1e3) / 1e12
    pc = clock_peak(tflop_per_mhz, clk.get("sm_mhz"))
    return {"value": value, "unit": "TFLOPS", "ms_per_step": ms / n, "steps": n,
            "launch": "CUDA graph replay" if graphs else "eager",
            "seconds": ms / 1e3, "clocks": clk,
            "step_frac_of_peak_clock": value / world / pc if pc else None,
            "step_frac_of_sustained_bf16_x2": value / world / (pk["bf16_tflops_sustained"]
                                                               * FP8_OVER_BF16),
            "note": "whole step (casts, GEMMs, update) against the dense FP8 peak at the "
                    "sampled clock and against the measured sustained BF16 peak x 2"}


def run_e2e(f, lin, X, dY, args, world, flops, readback="metric"):
    """Same metric through the public API from pinned host buffers.  Every
    step copies its inputs X and dY in from pinned host memory inside the
    timed region, and reads its result back: with readback="metric", the
    scaling state the step's update produced (the new scales and their
    inverses, 40 B: the step's result as a training step uses it, where Y,
    dX and dW stay on the device for the neighbouring layers and the
    optimizer); with readback="outputs", Y, dX and dW themselves.  Copies run
    on their own streams, the inputs double-buffered against the compute
    stream, so step i+1's uploads and step i's downloads overlap step i's
    kernels."""
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    hX = [torch.empty_like(X, device="cpu").pin_memory() for _ in range(2)]
    hdY = [torch.empty_like(dY, device="cpu").pin_memory() for _ in range(2)]
    for h in hX:
        h.copy_(X)
    for h in hdY:
        h.copy_(dY)
    dXin = [torch.empty_like(X) for _ in range(2)]
    ddYin = [torch.empty_like(dY) for _ in range(2)]
    douts = [(torch.empty_like(lin.Y), torch.empty_like(lin.dX), torch.empty_like(lin.dW))
             for _ in range(2)]
    # what each step reads back, per slot: the outputs (two slots), or a
    # snapshot of the scaling state taken on the compute stream right after
    # the step's update (a ring of eight, so that the compute stream never
    # waits for a recent download; the snapshot is an elementwise kernel, x1.0,
    # not a memcpy, so the compute stream never queues on a copy engine that
    # an upload holds)
    nres = 2 if readback == "outputs" else 8
    dres = [tuple(douts[k]) if readback == "outputs" else
            (torch.empty_like(lin.meta.scale), torch.empty_like(lin.meta.scale_inv))
            for k in range(nres)]
    houts = [tuple(torch.empty_like(t, device="cpu").pin_memory() for t in o) for o in dres]
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]      # upload of slot done
    in_free = [ev(), ev()]       # compute done reading slot's inputs
    out_ready = [ev() for _ in range(nres)]   # compute done writing slot's results
    out_free = [ev() for _ in range(nres)]    # download of slot's results done
    for e in in_free + out_free:
        e.record(comp)
    n = max(5, min(args.steps, 50))

    def step(i):
        k, kr = i % 2, i % nres
        with torch.cuda.stream(up):
            up.wait_event(in_free[k])
            dXin[k].copy_(hX[k], non_blocking=True)
            ddYin[k].copy_(hdY[k], non_blocking=True)
            in_ready[k].record(up)
        comp.wait_event(in_ready[k])
        comp.wait_event(out_free[kr])
        lin.step(dXin[k], ddYin[k], stream=comp, outs=douts[k])
        if readback != "outputs":
            with torch.cuda.stream(comp):
                torch.mul(lin.meta.scale, 1.0, out=dres[kr][0])
                torch.mul(lin.meta.scale_inv, 1.0, out=dres[kr][1])
        in_free[k].record(comp)
        out_ready[kr].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(out_ready[kr])
            for h, d in zip(houts[kr], dres[kr]):
                h.copy_(d, non_blocking=True)
            out_free[kr].record(down)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    # the host link alone: the step's two uploads with nothing else running
    link_ms = []
    for _ in range(3):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(up):
            a0.record(up)
            dXin[0].copy_(hX[0], non_blocking=True)
            ddYin[0].copy_(hdY[0], non_blocking=True)
            a1.record(up)
        torch.cuda.synchronize()
        link_ms.append(a0.elapsed_time(a1))
    barrier(world)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(comp)
    up.wait_stream(comp)
    down.wait_stream(comp)
    for i in range(n):
        step(i)
    for k in range(nres):
        comp.wait_event(out_free[k])
    e.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(s.elapsed_time(e), world)
    h2d = X.numel() * X.element_size() + dY.numel() * dY.element_size()
    d2h = sum(t.numel() * t.element_size() for t in dres[0])
    link = min(link_ms)
    return {"value": world * n * flops / (ms / 1e3) / 1e12, "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "h2d_gbs_alone": h2d / (link / 1e3) / 1e9,
            "upload_bound_tflops": world * flops / (link / 1e3) / 1e12,
            "readback": ("Y, dX and dW" if readback == "outputs" else
                         "the step's new scales and scale_inv (its scaling state)"),
            "overlap": "uploads, compute and downloads on three streams, double-buffered"}


# ------------------------------------------------------------- CPU oracle --

def oracle_sample_step(o, w: wl.Workload, Mp: int, Np: int, state):
    """One oracle layer step on a Mp-token x Np-feature slice of the workload
    (full K): casts of the slice's X, W and dY, the three GEMMs, the update."""
    s = dataclasses.replace(w, M=Mp, N=Np)
    X = wl.bf16_bits(wl.layer_x(s, 0))
    W = wl.bf16_bits(wl.layer_weight(s))
    dY = wl.bf16_bits(wl.layer_dy(s, 0))
    rc = o.Recipe(margin=w.margin, history_len=w.history_len, hybrid=w.hybrid)
    st = state if state is not None else o.State.initial(w.history_len)
    t = time.perf_counter()
    fo = o.layer_fwd(st, rc, X, W)
    o.layer_bwd(st, rc, dY, fo["X8t"], fo["W8t"])
    o.layer_update(st, rc)
    return time.perf_counter() - t, 6 * Mp * Np * w.K, st


def cpu_baseline(w: wl.Workload, seconds: float = 12.0, Mp: int = 256, Np: int = 1024):
    import oracle as o
    st = None
    total_t, total_f, reps = 0.0, 0, 0
    while total_t < seconds or reps < 2:
        dt, fl, st = oracle_sample_step(o, w, Mp, Np, st)
        total_t += dt
        total_f += fl
        reps += 1
    line = {"value": total_f / total_t / 1e12, "unit": "TFLOPS", "cores": o.num_threads(),
            "kind": "oracle",
            "sample": f"{reps} oracle layer steps on a {Mp}-token x {Np}-feature slice of "
                      f"{w.name} (K={w.K}), {total_t:.1f} s of CPU time",
            "affinity_cores": len(os.sched_getaffinity(0))}
    # the same oracle on one thread (OpenMP), on a quarter of the slice
    try:
        import ctypes
        gomp = ctypes.CDLL("libgomp.so.1")
        n0 = o.num_threads()
        gomp.omp_set_num_threads(1)
        try:
            t1, f1, r1, st1 = 0.0, 0, 0, None
            while t1 < 4.0 or r1 < 2:
                dt, fl, st1 = oracle_sample_step(o, w, Mp // 2, Np // 2, st1)
                t1 += dt
                f1 += fl
                r1 += 1
        finally:
            gomp.omp_set_num_threads(n0)
        line["single_thread"] = {"value": f1 / t1 / 1e12, "unit": "TFLOPS", "cores": 1,
                                 "sample": f"{r1} steps on a {Mp // 2}-token x {Np // 2}-feature "
                                           f"slice, {t1:.1f} s"}
    except OSError:
        pass
    return line


def _use_all_host_cores(o) -> None:
    """Give the oracle's OpenMP loops every core this process may run on.
    torchrun sets OMP_NUM_THREADS=1 for its workers by default, which would
    otherwise time the oracle on one core whenever N > 1."""
    try:
        import ctypes
        ctypes.CDLL("libgomp.so.1").omp_set_num_threads(len(os.sched_getaffinity(0)))
    except (OSError, AttributeError):
        pass


def run_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle as o
    _use_all_host_cores(o)
    w = wl.WORKLOADS[args.workload]
    # size the per-step sample so the whole run takes about two minutes
    dt, fl, _ = oracle_sample_step(o, w, 64, 256, None)
    rate = fl / dt
    budget = 120.0 / max(1, args.steps + args.warmup)
    Mp, Np = 64, 256
    for mp, np_ in [(128, 256), (128, 512), (256, 512), (256, 1024), (512, 1024)]:
        if 6 * mp * np_ * w.K / rate <= budget:
            Mp, Np = mp, np_
    st = None
    for _ in range(args.warmup):
        _, _, st = oracle_sample_step(o, w, Mp, Np, st)
    tt, ff = 0.0, 0
    for _ in range(args.steps):
        dt, fl, st = oracle_sample_step(o, w, Mp, Np, st)
        tt += dt
        ff += fl
    value = ff / tt / 1e12
    sample = (f"each step: oracle layer step on a {Mp}-token x {Np}-feature slice of "
              f"{w.name} (full K={w.K})")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle, exact FP8 decode)", "data": "synthetic",
            "config": workload_config(w, world),
            "cpu_baseline": {"kind": "oracle", "cores": o.num_threads(), "sample": sample,
                             "value": value, "unit": "TFLOPS",
                             "affinity_cores": len(os.sched_getaffinity(0))},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def workload_config(w: wl.Workload, world: int = 1):
    return {"workload": f"{w.name}: single FP8 linear fwd+bwd+update, M={w.M} tokens, K={w.K}, "
                        f"N={w.N}, {'HYBRID' if w.hybrid else 'E4M3'}, history {w.history_len}, "
                        f"margin {w.margin}",
            "M": w.M, "K": w.K, "N": w.N, "x": w.x_kind, "history_len": w.history_len,
            "margin": w.margin, "format": "HYBRID" if w.hybrid else "E4M3",
            "l2": "inputs larger than L2: X, W, dY = %d MB read per step, two batches alternate"
                  % ((2 * w.M * w.K + 2 * w.N * w.K + 2 * w.M * w.N) // 2 ** 20),
            "parallelism": f"dp{world} replicas" + (" + amax MAX all-reduce + FP8 dW all-reduce"
                                                    if world > 1 else "")}


def sweep_line(f, pk, n: int = 28, reps: int = 12):
    """The standalone quantize sweep's largest tensor: 2^n BF16 elements
    ((2^n / 4096) x 4096, N(0, 1) with 0.1 % of elements x 100).  Timed per
    launch with CUDA events, L2 flushed (L2Flush) before each, median
    of ``reps``: the amax (2 B/element), the cast + transposed copy to E4M3
    and to E5M2 (4 B/element, scale 1), and the just-in-time sequence amax ->
    scale -> cast (fp8_quantize_transpose_current, 6 B/element)."""
    x = wl.sweep_tensor(n, device="cuda")
    rows, cols = x.shape
    ne = rows * cols
    o8 = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    o8t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    am = torch.empty(1, device="cuda")
    one = torch.ones(1, device="cuda")
    sc, si = torch.ones(1, device="cuda"), torch.ones(1, device="cuda")
    flush = L2Flush()
    ops = {"amax": (2, lambda: f.fp8_amax(x, am)),
           "cast_e4m3": (4, lambda: f.fp8_quantize_transpose(x, one, f.E4M3, o8, o8t)),
           "cast_e5m2": (4, lambda: f.fp8_quantize_transpose(x, one, f.E5M2, o8, o8t)),
           "just_in_time_e4m3": (6, lambda: f.fp8_quantize_transpose_current(
               x, f.E4M3, 0, am, sc, si, o8, o8t))}
    times = {k: [] for k in ops}
    for r in range(reps + 2):
        for k, (_, fn) in ops.items():
            flush()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            fn()
            s1.record()
            torch.cuda.synchronize()
            if r >= 2:
                times[k].append(s0.elapsed_time(s1))
    f.fp8_sync_status()
    out = {"elements": ne, "peak_gbs": pk["hbm_gbs"], "unit": "GB/s",
           "note": "event-timed per launch, L2 flushed before each (a 256 MB write, then a "
                   "256 MB read that writes its dirty lines back), median of %d" % reps}
    for k, (bpe, _) in ops.items():
        ms = statistics.median(times[k])
        gbs = bpe * ne / (ms / 1e3) / 1e9
        out[k] = {"us": ms * 1e3, "gbs": gbs, "frac": gbs / pk["hbm_gbs"],
                  "bytes_per_element": bpe}
    del x, o8, o8t, flush
    torch.cuda.empty_cache()
    return out


SECONDARY_PARTS = ("mlp70b", "cast_sweep", "layernorm_cast", "fp8_adam", "jit_scaling",
                   "fp8_allreduce", "cublaslt", "drift")


def run_secondary(f, args, pk):
    """The extra measurements: the 70B-shaped layer, the cast/amax sweep, the
    LayerNorm + cast and FP8 Adam kernels, the just-in-time scaling step, the
    FP8 all-reduce sum, the cuBLASLt context and the drift range counts.
    ``args.part`` names the ones to run (all when empty)."""
    want = lambda name: not args.part or name in args.part
    out = {}
    w7 = wl.WORKLOADS["mlp7b"]
    flush = L2Flush()
    if want("mlp70b"):
        out["mlp70b"] = secondary_mlp70b(f, args, pk)
    if want("cast_sweep"):
        out["cast_sweep"] = secondary_cast_sweep(f)
    if want("layernorm_cast"):
        out["layernorm_cast_mlp7b_X"] = secondary_layernorm_cast(f, w7, flush, pk)
    if want("fp8_adam"):
        out["fp8_adam_step_mlp7b_W"] = secondary_adam(f, w7, flush)
    if want("jit_scaling"):
        out["jit_scaling_layer_step_mlp7b"] = secondary_jit_scaling(f, w7)
    if want("fp8_allreduce"):
        out["fp8_allreduce_sum_8ranks_mlp7b_dW"] = secondary_dequant_sum(f, w7, flush)
    if want("cublaslt"):
        out["context_cublaslt_fp8_mlp7b"] = cublaslt_context(f, w7, flush)
    del flush
    if want("drift"):
        out["drift_range_counts"] = drift_range_report(f)
    return out


def secondary_mlp70b(f, args, pk):
    """The 70B-shaped layer step (device time only)."""
    w = wl.WORKLOADS["mlp70b"]
    sub = argparse.Namespace(**{**vars(args), "steps": max(10, min(args.steps, 30)),
                                "warmup": 3, "no_e2e": True})
    r = run_layer_bench(f, w, sub, 1, pk, "measured")
    return {"value": r["value"], "unit": "TFLOPS", "ms_per_step": r["ms_per_step"],
            "gemm_frac": r["roofline"]["frac"], "gemm_tflops": r["roofline"]["achieved"],
            "cast_gbs": r["cast_roofline"]["achieved"]}


def secondary_cast_sweep(f):
    """Standalone amax and cast+transpose GB/s on the 2^24 / 2^26 / 2^28 sweep
    tensors (23 launches of each per size, the first 3 untimed)."""
    sweep = {}
    for n in (24, 26, 28):
        x = wl.sweep_tensor(n, device="cuda")
        rows, cols = x.shape
        o8 = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        o8t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
        am = torch.empty(1, device="cuda")
        sc = torch.ones(1, device="cuda")
        tm = EventTimer()
        for i in range(23):
            tm.time("amax", lambda: f.fp8_amax(x, am))
            tm.time("cast", lambda: f.fp8_quantize_transpose(x, sc, 0, o8, o8t, am))
        torch.cuda.synchronize()
        tm.pairs = {k: v[3:] for k, v in tm.pairs.items()}
        ne = rows * cols
        sweep[f"2^{n}"] = {"amax_gbs": 2 * ne / (tm.mean_ms("amax") / 1e3) / 1e9,
                           "cast_transpose_gbs": 4 * ne / (tm.mean_ms("cast") / 1e3) / 1e9}
        del x, o8, o8t
    return sweep


def secondary_layernorm_cast(f, w7, flush, pk):
    """LayerNorm + cast of the 7B layer's X against the plain cast of the same
    tensor: with the transposed copy, without it, and the transposed copy
    alone (the two-kernel path: row statistics, then the cast).  Then the row
    statistics alone (2 B/element algorithmic), on X and on 16 copies of X
    stacked (1 GiB), where the fixed cost of a launch no longer counts."""
    X = wl.layer_x(w7, 0, "cuda")
    g = torch.ones(w7.K, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(w7.K, dtype=torch.bfloat16, device="cuda")
    o8 = torch.empty((w7.M, w7.K), dtype=torch.uint8, device="cuda")
    o8t = torch.empty((w7.K, w7.M), dtype=torch.uint8, device="cuda")
    mean = torch.empty(w7.M, device="cuda")
    rstd = torch.empty(w7.M, device="cuda")
    sc = torch.ones(1, device="cuda")
    tm = EventTimer()
    for i in range(23):
        flush()
        tm.time("ln_cast", lambda: f.fp8_layernorm_quantize_transpose(X, g, b, 1e-5, sc, 0, mean,
                                                                      rstd, o8, o8t))
        flush()
        tm.time("cast", lambda: f.fp8_quantize_transpose(X, sc, 0, o8, o8t))
        flush()
        tm.time("ln_cast_rows", lambda: f.fp8_layernorm_quantize_transpose(
            X, g, b, 1e-5, sc, 0, mean, rstd, o8, None))
        flush()
        tm.time("ln_cast_t_only", lambda: f.fp8_layernorm_quantize_transpose(
            X, g, b, 1e-5, sc, 0, mean, rstd, None, o8t))
    big = X.repeat(16, 1)
    mean_b = torch.empty(big.shape[0], device="cuda")
    rstd_b = torch.empty(big.shape[0], device="cuda")
    for i in range(23):
        flush()
        tm.time("ln_stats", lambda: f.fp8_layernorm_stats(X, g, b, 1e-5, mean, rstd))
        flush()
        tm.time("ln_stats_1g", lambda: f.fp8_layernorm_stats(big, g, b, 1e-5, mean_b, rstd_b))
    torch.cuda.synchronize()
    del big
    tm.pairs = {k: v[3:] for k, v in tm.pairs.items()}
    ne = w7.M * w7.K
    stats = {}
    for k, n in (("ln_stats", ne), ("ln_stats_1g", 16 * ne)):
        us = tm.mean_ms(k) * 1e3
        gbs = 2 * n / us / 1e3
        stats[k] = {"us": us, "gbs": gbs, "frac": gbs / pk["hbm_gbs"], "elements": n}
    return {"ln_stats": stats["ln_stats"], "ln_stats_16x": stats["ln_stats_1g"],
            "ln_cast_us": tm.mean_ms("ln_cast") * 1e3, "cast_us": tm.mean_ms("cast") * 1e3,
            "ln_cast_gbs": 4 * ne / (tm.mean_ms("ln_cast") / 1e3) / 1e9,
            "ln_cast_rows_us": tm.mean_ms("ln_cast_rows") * 1e3,
            "ln_cast_rows_gbs": 3 * ne / (tm.mean_ms("ln_cast_rows") / 1e3) / 1e9,
            "ln_cast_t_only_us": tm.mean_ms("ln_cast_t_only") * 1e3,
            "note": "ln_cast: the codes and their transposed copy (one pass over X, then a byte "
                    "transpose of the codes), 4 B/element algorithmic; ln_cast_rows: the codes "
                    "only (one kernel, one read of X), 3 B/element; ln_cast_t_only: the "
                    "transposed copy only (row statistics, then the cast kernel); ln_stats: "
                    "the row statistics alone on X and on 16 copies of X (2 B/element), frac "
                    "of measured HBM; L2 flushed before each launch"}


def secondary_adam(f, w7, flush):
    """One decoupled-precision Adam step over the 7B layer's weight (45 M params)."""
    tm = EventTimer()
    st = f.Fp8AdamState(wl.layer_weight(w7, "cuda"))
    grad = wl.layer_weight(w7, "cuda")
    wout = torch.empty_like(grad)
    hp = f.AdamHyper(lr=1e-4, weight_decay=0.1)
    for i in range(23):
        flush()
        tm.time("adam", lambda: st.step(grad, wout, hp))
    torch.cuda.synchronize()
    tm.pairs["adam"] = tm.pairs["adam"][3:]
    nw = w7.N * w7.K
    return {
        "us": tm.mean_ms("adam") * 1e3,
        "gbs_algorithmic": 14 * nw / (tm.mean_ms("adam") / 1e3) / 1e9,
        "note": "14 B/param algorithmic (grad 2 + m1 1 + m2 2 + w16 2 read, the same written "
                "plus 2 B BF16 weights minus the grad); the kernel reads the inputs twice "
                "(amax pass, then the update pass) for just-in-time state scales"}


def secondary_jit_scaling(f, w7):
    """Just-in-time (current) scaling: the 7B layer step with X, W and dY
    scaled from their own amax (an amax pass before each cast)."""
    lj = f.Fp8Linear(wl.layer_weight(w7, "cuda"), w7.M,
                     f.Recipe(margin=w7.margin, history_len=w7.history_len, hybrid=w7.hybrid,
                              current=True))
    xs7 = [wl.layer_x(w7, k, "cuda") for k in (0, 1)]
    dys7 = [wl.layer_dy(w7, k, "cuda") for k in (0, 1)]
    for i in range(3):
        lj.step(xs7[i % 2], dys7[i % 2])
    torch.cuda.synchronize()
    nj = 30
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for i in range(nj):
        lj.step(xs7[i % 2], dys7[i % 2])
    s1.record()
    torch.cuda.synchronize()
    msj = s0.elapsed_time(s1) / nj
    return {"ms_per_step": msj, "value": 6 * w7.M * w7.N * w7.K / (msj / 1e3) / 1e12,
            "unit": "TFLOPS", "note": "X, W and dY scaled just in time from their own amax"}


def secondary_dequant_sum(f, w7, flush):
    """The device part of the FP8 gradient all-reduce: decode and sum 8 ranks'
    FP8 codes of the 7B dW (shared scale) into BF16; 8 B read + 2 B written
    per element for 8 ranks.  The codes are 8 ranks' gradient-shaped dW
    (N(0, sigma_r) BF16, sigma_r = 1e-3 * (1 + r / 10)) cast with their
    shared scale, the minimum of the ranks' own scales, as fp8_allreduce
    does; a second row times uniformly random finite codes, whose sums span
    the most binades (the kernel's slowest case)."""
    nr, nd = 8, w7.N * w7.K
    g = torch.Generator(device="cuda").manual_seed(7)
    grads, scales = [], []
    for r in range(nr):
        x = (torch.randn((w7.N, w7.K), generator=g, device="cuda") * (1e-3 * (1 + 0.1 * r))) \
            .to(torch.bfloat16)
        am, h = torch.empty(1, device="cuda"), torch.zeros((1, 1), device="cuda")
        s1, si = torch.ones(1, device="cuda"), torch.ones(1, device="cuda")
        f.fp8_amax(x, am)
        f.fp8_scale_update(h, am, s1, si, f.E5M2, 0)
        grads.append(x)
        scales.append(s1)
    sg = torch.min(torch.cat(scales)).reshape(1)
    parts = torch.empty((nr, nd), dtype=torch.uint8, device="cuda")
    for r in range(nr):
        f.fp8_quantize_transpose(grads[r], sg, f.E5M2, out=parts[r].view(w7.N, w7.K))
    del grads
    uniform = torch.randint(0, 0x7B, (nr, nd), dtype=torch.uint8, device="cuda")
    dsum = torch.empty(nd, dtype=torch.bfloat16, device="cuda")
    res = {}
    for name, (codes, sc) in {"gradient": (parts, sg),
                              "uniform_codes": (uniform, torch.full((1,), 64.0, device="cuda"))}.items():
        tm = EventTimer()
        for i in range(23):
            flush()
            tm.time("dequant_sum", lambda: f.fp8_dequant_sum(codes, f.E5M2, sc, dsum))
        torch.cuda.synchronize()
        tm.pairs["dequant_sum"] = tm.pairs["dequant_sum"][3:]
        us = tm.mean_ms("dequant_sum") * 1e3
        res[name] = {"us": us, "gbs_algorithmic": (nr + 2) * nd / (us / 1e6) / 1e9}
    res["note"] = ("exact decode + sum of 8 ranks' E5M2 codes -> BF16 (rounded once); "
                   "L2 flushed before each; 10 B/element algorithmic")
    del parts, uniform, dsum
    return res


def range_counts(x: torch.Tensor, codes: torch.Tensor, s: torch.Tensor, fmax: float):
    """How a cast under scale ``s`` treated one tensor: ``saturated`` = elements
    with |fl32(x * s)| above the format's largest finite value (clipped to it),
    ``underflow`` = non-zero elements whose FP8 code is +-0.  ``x`` BF16,
    ``codes`` the cast's FP8 bytes, ``s`` a one-element fp32 tensor; any device.
    A diagnostic of the recipe, not part of the layer."""
    v = x.float() * s
    sat = int((v.abs() > fmax).sum())
    under = int(((x != 0) & ((codes & 0x7F) == 0)).sum())
    return sat, under


def drift_range_report(f, steps: int = 130):
    """Per-step saturation / underflow counts of the drifting-scale workload
    (M = K = N = 4096, history 512, margin 0) under delayed scaling, in the
    HYBRID and the E4M3-everywhere arms.  X and dY are drawn on the device
    with the workload's recipe (a CUDA generator, so the bytes differ from the
    host-drawn ones the parity tests use).  The x1000 spike at step 50 is cast
    with the scale of the steps before it, so it saturates; at step 51 the
    history holds the spike and the ordinary X loses its small values."""
    w = wl.WORKLOADS["drift"]
    n_el = w.M * w.K
    out = {}
    for hybrid in (True, False):
        lin = f.Fp8Linear(wl.layer_weight(w, "cuda"), w.M,
                          f.Recipe(margin=w.margin, history_len=w.history_len, hybrid=hybrid))
        fmax_dy = 57344.0 if hybrid else 448.0
        per = []
        for t in range(steps):
            X, dY = wl.layer_x(w, t, "cuda"), wl.layer_dy(w, t, "cuda")
            sx, sdy = lin.meta.scale[0:1].clone(), lin.meta.scale[3:4].clone()
            lin.step(X, dY)
            xs, xu = range_counts(X, lin.X8, sx, 448.0)
            ds, du = range_counts(dY, lin.dY8, sdy, fmax_dy)
            per.append((t, xs, xu, ds, du, float(sx.item())))
        torch.cuda.synchronize()
        notable = {str(t): {"scale_X": sc, "X_saturated": xs, "X_underflow": xu,
                            "dY_saturated": ds, "dY_underflow": du}
                   for t, xs, xu, ds, du, sc in per if t in (0, 1, 49, 50, 51, 75, 76, 100)}
        out["hybrid" if hybrid else "e4m3_everywhere"] = {
            "steps": steps, "elements_per_tensor": n_el, "at_step": notable,
            "X_saturated_total": sum(p[1] for p in per),
            "X_underflow_total": sum(p[2] for p in per),
            "dY_saturated_total": sum(p[3] for p in per),
            "dY_underflow_total": sum(p[4] for p in per)}
        del lin
    return out


def cublaslt_context(f, w, flush):
    """Context only (never on the product path): the vendor library's FP8
    GEMM (torch._scaled_mm -> cuBLASLt) on the layer's own FP8 operands,
    interleaved with this library's GEMM, L2 flushed before each launch,
    median of 15.  cuBLASLt computes no output amax."""
    try:
        lin = f.Fp8Linear(wl.layer_weight(w, "cuda"), w.M,
                          f.Recipe(margin=w.margin, history_len=w.history_len, hybrid=w.hybrid))
        X, dY = wl.layer_x(w, 0, "cuda"), wl.layer_dy(w, 0, "cuda")
        for _ in range(3):
            lin.step(X, dY)
        torch.cuda.synchronize()
        m, E4, E5 = lin.meta, f.E4M3, f.E5M2
        fg = E5 if w.hybrid else E4
        t8 = {E4: torch.float8_e4m3fn, E5: torch.float8_e5m2}
        one = torch.ones((), device="cuda")
        cases = {
            "fprop": ((lin.X8, E4, lin.W8, E4, 0, 1, lin.Y)),
            "dgrad": ((lin.dY8, fg, lin.W8t, E4, 3, 1, lin.dX)),
            "wgrad": ((lin.dY8t, fg, lin.X8t, E4, 3, 0, lin.dW)),
        }
        res = {}
        for name, (A, fa, B, fb, ia, ib, D) in cases.items():
            ours = lambda: f.fp8_gemm_tn(A, fa, B, fb, m.scale_inv[ia:ia + 1],
                                         m.scale_inv[ib:ib + 1], D)
            lib = lambda: torch._scaled_mm(A.view(t8[fa]), B.view(t8[fb]).t(), scale_a=one,
                                           scale_b=one, out_dtype=torch.bfloat16)
            lib()
            to, tl = [], []
            for _ in range(15):
                for fn, acc in ((ours, to), (lib, tl)):
                    flush()
                    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    s.record()
                    fn()
                    e.record()
                    torch.cuda.synchronize()
                    acc.append(s.elapsed_time(e))
            fl = 2 * w.M * w.N * w.K
            mo, ml = statistics.median(to), statistics.median(tl)
            res[name] = {"ours_us": mo * 1e3, "cublaslt_us": ml * 1e3,
                         "ours_tflops": fl / (mo / 1e3) / 1e12,
                         "cublaslt_tflops": fl / (ml / 1e3) / 1e12}
        return res
    except Exception as ex:   # the context row is optional
        return {"unavailable": str(ex)[:200]}


def main():
    args = parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import __graft_entry__
    # one rank (re)builds the in-tree library if it is stale; the others wait
    if rank == 0:
        __graft_entry__._build_module().build()
    barrier(world)
    import fp8_mixed_precision_amax_gb300 as f
    pk, peak_kind = peaks()
    w = wl.WORKLOADS[args.workload]
    r = run_layer_bench(f, w, args, world, pk, peak_kind,
                        sustained_s=args.sustained_seconds if world == 1 else 0.0,
                        e2e=not args.no_e2e)
    line = {
        "metric": METRIC, "value": r["value"], "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8 e4m3/e5m2 operands, f32 accumulate, bf16 out",
        "data": "synthetic (seeded fp8_workloads, resident in HBM)",
        "config": workload_config(w, world),
        "launch": r["launch"], "ms_per_step_eager": r["ms_per_step_eager"],
        "ms_per_step_graph": r["ms_per_step_graph"],
        "roofline": r["roofline"], "cast_roofline": r["cast_roofline"], "clocks": r["clocks"],
        "gpu_launches": r["gpu_launches"], "breakdown_ms": r["breakdown_ms"],
        "peaks_source": peak_kind,
    }
    if "sustained" in r:
        line["sustained"] = r["sustained"]
    if world == 1 and not args.no_extras:
        line["sweep_2e28"] = sweep_line(f, pk)
        if w.name != "mlp7b":
            sub = argparse.Namespace(**{**vars(args), "steps": max(args.steps, 20)})
            r7 = run_layer_bench(f, wl.WORKLOADS["mlp7b"], sub, 1, pk, peak_kind, e2e=False)
            line["mlp7b"] = {"value": r7["value"], "unit": "TFLOPS",
                             "ms_per_step": r7["ms_per_step"], "steps": sub.steps,
                             "config": workload_config(wl.WORKLOADS["mlp7b"])["workload"],
                             "roofline": r7["roofline"], "cast_roofline": r7["cast_roofline"],
                             "clocks": r7["clocks"]}
    if "e2e" in r:
        line["e2e"] = r["e2e"]
    if args.secondary and rank == 0:
        line["secondary"] = run_secondary(f, args, pk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
