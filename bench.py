"""Throughput benchmark of the fused attention path on GB300.

One step = one training-style pass of the whole hot path over one batch:
fa_fwd (causal) followed by fa_bwd (causal, atomic dQ) on the largest
forward + backward workload, B=2, Hq=Hkv=16, S=8192, D=128, bf16 (synthetic
N(0,1) inputs).  FLOPs per step follow the measurement convention:
4*B*Hq*Sq*Sk*D forward, halved for causal, plus 2.5x that for the backward
pass.  The same line also reports, under ``extra``, the training-scale step
(B=4, H=16, S=2048, causal) measured the same way, and the non-causal D=128
forward at S = 8k, 16k and 32k (16k tokens per batch).

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  torchrun --nproc-per-node N bench.py --gpus N ...   (one rank per GPU)
  python bench.py --only fwd:S:D:causal --steps K --warmup W
  python bench.py --only bwd:S:D:causal[:det] --steps K --warmup W
      (one forward or backward shape alone, for a profiler capture)

With N > 1 every rank runs its own batch of the same workload (independent
units, no collective on the data path); the timing is the max over ranks and
``value`` counts the FLOPs of all ranks ("weak" scaling).

``--impl reference`` times the fp64 CPU oracle as it stands, on a bounded
sample of the same workload, on this host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "attention fwd/bwd TFLOPs/s (BF16, 1×GB300) and % of tensor-core peak"
UNIT = "TFLOP/s"
WORKLOAD = synth.BWD  # B=2, Hq=Hkv=16, S=8192, D=128, causal: the headline step
SECONDARY = synth.TRAIN  # B=4, Hq=Hkv=16, S=2048, D=128, causal
# the forward target: non-causal, D=128, S >= 8k (16k tokens per batch)
LONG_FWD = [(8192, 128, False), (16384, 128, False), (32768, 128, False)]
# the head-dimension-64 forward at S = 8k (its ring-of-score-buffers kernel)
D64_FWD = [(8192, 64, False), (8192, 64, True)]
NOMINAL_DENSE_BF16_TFLOPS = 2250.0
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------- helpers

def step_flops(w: synth.Workload) -> float:
    return w.flops(backward=False) + w.flops(backward=True)


def config_dict(w: synth.Workload) -> dict:
    return {"workload": f"attention fwd+bwd, {'causal' if w.causal else 'non-causal'}, B={w.B} "
                        f"Hq={w.Hq} Hkv={w.Hkv} S={w.Sq} D={w.D} bf16",
            "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
            "causal": w.causal, "dq_mode": "atomic",
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write)"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured (MEASURED_PEAKS.json)"
    return dict(FALLBACK_PEAKS), "fallback (no MEASURED_PEAKS.json)"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_blackwell_tiled_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of ``kernel`` on ``workload`` recorded by an ncu
    capture (profiles/traffic.json, keyed "kernel@workload"), or None when
    absent or taken on different kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}@{workload}")
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = sorted(float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit())
        mx = max((float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in self.samples for n, v in zip(names, s[5:9])
                          if v.lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(self.samples)}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank float across the process group (identity when world == 1)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle

_ORACLE_INPUTS: dict = {}

def cpu_oracle_sample(w: synth.Workload, budget_s: float = 12.0, max_heads: int | None = None):
    """Time the fp64 oracle (forward + backward of whole kv heads) on a bounded
    sample of the workload.  Returns (TFLOP/s in the FLOP convention, cores,
    sample description, seconds)."""
    import numpy as np
    import oracle

    key = (w, "f64")
    if key not in _ORACLE_INPUTS:  # widen to fp64 once, outside the timed region
        _ORACLE_INPUTS.clear()
        _ORACLE_INPUTS[key] = [t.double().numpy() for t in synth.make_inputs(w, with_do=True)]
    q, k, v, do = _ORACLE_INPUTS[key]
    cores = oracle.max_threads()
    n_units = w.B * w.Hkv
    per_unit_flops = step_flops(w) / n_units
    done, t0 = 0, time.perf_counter()
    cap = n_units if max_heads is None else min(n_units, max_heads)
    while done < cap:
        oracle.bwd(q, k, v, do, w.causal, w.softmax_scale, units=[done])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    value = per_unit_flops * done / dt / 1e12
    sample = (f"fp64 oracle forward+backward of {done} of {n_units} kv heads "
              f"(B*Hkv units) of the workload, {dt:.1f} s; FLOPs counted by the same convention")
    return value, cores, sample, dt


# ----------------------------------------------------------------------------- GPU arm

def time_step(fa, w, dev, tensors, steps, warmup, flush, world, stream):
    """Time W + K fwd+bwd steps (atomic dQ) on workload ``w``, then the forward
    kernel and the backward main kernel alone (events around each on the
    launching stream) and the deterministic backward's main kernel.  Returns a
    dict of per-step / per-kernel times in ms and the launches of the timed
    steps."""
    import torch
    qd, kd, vd, dod, o, lse, dq, dk, dv, ws = tensors
    scale = w.softmax_scale

    def step(time_kernels=None):
        launches = 0
        if time_kernels is not None:
            fa.set_timing_events(*time_kernels[0])
        fa.fwd(qd, kd, vd, causal=w.causal, scale=scale, out=o, lse=lse)
        launches += fa.last_launch_count()
        if time_kernels is not None:
            fa.set_timing_events(*time_kernels[1])
        fa.bwd(qd, kd, vd, o, dod, lse, causal=w.causal, scale=scale, workspace=ws, dq=dq, dk=dk,
               dv=dv)
        launches += fa.last_launch_count()
        return launches

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    assert fa.fwd_status() == fa.FA_OK and fa.bwd_status(ws) == fa.FA_OK

    # Timed region: whole steps bracketed by events, nothing recorded between
    # the kernels (an event there would serialise their programmatic overlap).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    launches = 0
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for i in range(steps):
            flush.zero_()  # L2 flush outside the timed interval
            e = ev[i]
            e[0].record(stream)
            launches += step()
            e[1].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world, dev)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    # Per-kernel breakdown (the roofline's launch duration): a separate run with
    # events around the forward kernel and the backward main kernel.
    n_k = min(steps, 200)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_k)]
    for i in range(n_k):
        flush.zero_()
        e = kev[i]
        step(time_kernels=((e[0], e[1]), (e[2], e[3])))
    torch.cuda.synchronize(dev)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in kev]
    bwd_main_ms = [e[2].elapsed_time(e[3]) for e in kev]
    # the deterministic backward (semaphore-ordered dQ adds), main kernel only
    ws_det = torch.empty(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True),
                         dtype=torch.uint8, device=dev)
    det = []
    for i in range(min(steps, 50) + 3):
        flush.zero_()
        e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        fa.set_timing_events(*e)
        fa.bwd(qd, kd, vd, o, dod, lse, causal=w.causal, scale=scale, workspace=ws_det, dq=dq,
               dk=dk, dv=dv, deterministic=True)
        if i >= 3:
            det.append(e)
    torch.cuda.synchronize(dev)
    assert fa.bwd_status(ws_det) == fa.FA_OK
    det_ms = [a.elapsed_time(b) for a, b in det]
    del ws_det
    # the CTA-pair main kernel (2-CTA MMA, dQ reduced over 256 keys), where it applies
    pair = []
    if w.D == 128:
        prev = fa.set_bwd_kernel(fa.BWD_KERNEL_PAIR)
        try:
            for i in range(min(steps, 50) + 3):
                flush.zero_()
                e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                fa.set_timing_events(*e)
                fa.bwd(qd, kd, vd, o, dod, lse, causal=w.causal, scale=scale, workspace=ws,
                       dq=dq, dk=dk, dv=dv)
                if i >= 3:
                    pair.append(e)
            torch.cuda.synchronize(dev)
        finally:
            fa.set_bwd_kernel(prev)
        assert fa.bwd_status(ws) == fa.FA_OK
    pair_ms = [a.elapsed_time(b) for a, b in pair]
    return {"step_ms": step_ms, "launches": launches, "clocks": clk.summary(),
            "fwd_ms": sum(fwd_ms) / len(fwd_ms), "bwd_main_ms": sum(bwd_main_ms) / len(bwd_main_ms),
            "det_ms": sum(det_ms) / len(det_ms),
            "pair_ms": sum(pair_ms) / len(pair_ms) if pair_ms else None}


def kernel_rates(w, t, peak):
    """TFLOP/s and fractions of peak of a workload's kernels from time_step()."""
    fwd_f, bwd_f = w.flops(False), w.flops(True)
    step_ms = sum(t["step_ms"]) / len(t["step_ms"])
    fwd_tf = fwd_f / (t["fwd_ms"] * 1e-3) / 1e12
    bwd_tf = bwd_f / (t["bwd_main_ms"] * 1e-3) / 1e12
    det_tf = bwd_f / (t["det_ms"] * 1e-3) / 1e12
    return {"step_tflops": round(step_flops(w) / (step_ms * 1e-3) / 1e12, 1),
            "ms_per_step": round(step_ms, 4),
            "fwd_tflops": round(fwd_tf, 1), "fwd_ms": round(t["fwd_ms"], 4),
            "fwd_frac_of_peak": round(fwd_tf / peak, 4),
            "bwd_main_tflops": round(bwd_tf, 1), "bwd_main_ms": round(t["bwd_main_ms"], 4),
            "bwd_main_frac_of_peak": round(bwd_tf / peak, 4),
            "bwd_main_det_tflops": round(det_tf, 1), "bwd_main_det_ms": round(t["det_ms"], 4),
            "det_over_atomic": round(t["bwd_main_ms"] / t["det_ms"], 3),
            "bwd_main_pair_tflops": (round(bwd_f / (t["pair_ms"] * 1e-3) / 1e12, 1)
                                     if t.get("pair_ms") else None),
            "fwd_frac_of_nominal": round(fwd_tf / NOMINAL_DENSE_BF16_TFLOPS, 4),
            "bwd_main_frac_of_nominal": round(bwd_tf / NOMINAL_DENSE_BF16_TFLOPS, 4)}


def alloc_step(fa, w, dev, rank):
    """Seeded inputs of workload ``w`` (rank r draws its own batch) on the device,
    with the outputs and the backward workspace of one step."""
    import torch
    w = w.with_(seed=w.seed + 1000 * rank)
    q, k, v, do = synth.make_inputs(w, with_do=True)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D), dtype=torch.uint8,
                     device=dev)
    return (q, k, v, do), (qd, kd, vd, dod, o, lse, dq, dk, dv, ws)


def run_ours(args):
    import torch
    import exact_attention_blackwell_tiled_gb300 as fa

    rank, local, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if args.only:
        return run_only(fa, args, dev)
    w = WORKLOAD
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    host, tensors = alloc_step(fa, w, dev, rank)
    q, k, v, do = host
    qd, kd, vd, dod, o, lse, dq, dk, dv, ws = tensors
    scale = w.softmax_scale
    t = time_step(fa, w, dev, tensors, args.steps, args.warmup, flush, world, stream)
    total_ms_local = sum(t["step_ms"])
    total_ms = max_over_ranks(total_ms_local, world, dev)
    ms_per_step = total_ms / args.steps
    flops = step_flops(w)
    value = flops * world * args.steps / (total_ms * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    rates = kernel_rates(w, t, peak)
    if t["bwd_main_ms"] >= t["fwd_ms"]:
        dom, dom_ms, dom_flops = "bwd_main<128>", t["bwd_main_ms"], w.flops(True)
    else:
        dom, dom_ms, dom_flops = "fwd_kernel<128>", t["fwd_ms"], w.flops(False)
    dom_tf = dom_flops / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(dom_tf, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(dom_tf / peak, 4), "traffic": profiled_traffic(dom, w.name),
                "kernel": dom, "flops_per_launch": dom_flops,
                "peak_source": f"bf16_tflops burst, {peak_src}"}
    clocks = t["clocks"]

    # End to end through the public API: every step copies its inputs from
    # pinned host memory, runs fwd + bwd and copies the gradients back.  As in a
    # data-loading pipeline, the copies run on their own streams with
    # double-buffered device tensors, so step i+1's upload and step i-1's
    # download overlap step i's compute; all of them lie inside the timed region.
    e2e = None
    if rank == 0 or world > 1:
        hq, hk, hv, hdo = (x.pin_memory() for x in (q, k, v, do))
        out_h = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (q, k, v)]
        ins = [[torch.empty_like(x) for x in (qd, kd, vd, dod)] for _ in range(2)]
        outs = [[torch.empty_like(x) for x in (qd, kd, vd)] for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        n_e2e = max(3, min(args.steps, 50))
        torch.cuda.synchronize(dev)
        t_e0 = torch.cuda.Event(enable_timing=True)
        t_e1 = torch.cuda.Event(enable_timing=True)

        def upload(i):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[b])  # step i-2 has finished reading slot b
                for dst, src in zip(ins[b], (hq, hk, hv, hdo)):
                    dst.copy_(src, non_blocking=True)
                ev_in[b].record(s_in)

        def run(n_steps):
            upload(0)
            for it in range(n_steps):
                b = it % 2
                if it + 1 < n_steps:
                    upload(it + 1)
                stream.wait_event(ev_in[b])
                if it >= 2:
                    stream.wait_event(ev_out[b])  # step i-2's gradients have left slot b
                xq, xk, xv, xdo = ins[b]
                fa.fwd(xq, xk, xv, causal=w.causal, scale=scale, out=o, lse=lse)
                fa.bwd(xq, xk, xv, o, xdo, lse, causal=w.causal, scale=scale, workspace=ws,
                       dq=outs[b][0], dk=outs[b][1], dv=outs[b][2])
                ev_done[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[b])
                    for hdst, dsrc in zip(out_h, outs[b]):
                        hdst.copy_(dsrc, non_blocking=True)
                    ev_out[b].record(s_out)
            stream.wait_event(ev_out[(n_steps - 1) % 2])

        run(2)  # warm-up
        torch.cuda.synchronize(dev)
        # timed: the pipeline restarts after t_e0, so every step's upload,
        # compute and download lies between the two events (fill and drain
        # included)
        t_e0.record(stream)
        s_in.wait_event(t_e0)
        run(n_e2e)
        t_e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(t_e0.elapsed_time(t_e1) / n_e2e, world, dev)
        h2d = sum(x.numel() * x.element_size() for x in (q, k, v, do))
        d2h = sum(x.numel() * x.element_size() for x in out_h)
        e2e = {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 4),
               "overlap": "upload of step i+1 and download of step i-1 overlap step i"}
        del ins, outs, hq, hk, hv, hdo, out_h

    assert fa.fwd_status() == fa.FA_OK and fa.bwd_status(ws) == fa.FA_OK
    del host, tensors, qd, kd, vd, dod, o, lse, dq, dk, dv, ws

    extra = dict(rates)
    extra["peak_tflops"] = peak
    # the vendor's dense bf16 figure for one GB300 (2.25 PFLOP/s without
    # sparsity), the like-for-like denominator of a "% of theoretical peak"
    extra["nominal_dense_bf16_tflops"] = NOMINAL_DENSE_BF16_TFLOPS
    # the training-scale step (B=4, H=16, S=2048, causal), measured the same way
    if not args.no_train_step:
        w2 = SECONDARY
        _, tensors2 = alloc_step(fa, w2, dev, rank)
        t2 = time_step(fa, w2, dev, tensors2, args.steps, args.warmup, flush, world, stream)
        r2 = kernel_rates(w2, t2, peak)
        r2["workload"] = config_dict(w2)["workload"]
        r2["traffic_bwd_main"] = profiled_traffic("bwd_main<128>", w2.name)
        extra["train_step"] = r2
        del tensors2
    # the forward target: non-causal D=128 at S >= 8k (16k tokens per batch)
    if rank == 0 and not args.no_long_fwd:
        extra["fwd_noncausal_long"] = fwd_sweep(fa, dev, peak, shapes=LONG_FWD)
        extra["fwd_d64"] = fwd_sweep(fa, dev, peak, shapes=D64_FWD)
    if args.sweep and rank == 0:
        extra["fwd_sweep"] = fwd_sweep(fa, dev, peak)
    if args.mod_sweep and rank == 0:
        extra["mod_sweep"] = mod_sweep(fa, dev, peak)
    if args.split_sweep and rank == 0:
        extra["split_sweep"] = split_sweep(fa, dev, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, cores, sample, _ = cpu_oracle_sample(w, budget_s=args.cpu_budget)
        cpu = {"value": v_cpu, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 inputs of the workload's shape)",
            "config": config_dict(w), "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": t["launches"], "clocks": clocks, "extra": extra}
    print(json.dumps(line), flush=True)


def run_only(fa, args, dev):
    """One kernel call shape alone, W + K times, nothing else -- the command a
    profiler capture of that kernel runs:
      --only fwd:S:D:causal             the forward on the sweep workload of that S, D
      --only bwd:S:D:causal[:det|:pair] the backward on it: atomic dQ, deterministic dQ,
                                        or atomic on the CTA-pair kernel
      --only-batch B                    that shape with batch B instead
    """
    import torch
    parts = args.only.split(":")
    kind, S, D, c = parts[:4]
    mode = parts[4] if len(parts) > 4 else ""
    if kind not in ("fwd", "bwd") or mode not in ("", "det", "pair"):
        raise SystemExit(f"--only: unknown kind or mode {args.only!r}")
    det = mode == "det"
    if mode == "pair":
        fa.set_bwd_kernel(fa.BWD_KERNEL_PAIR)
    w = synth.sweep(int(S), int(D), c in ("1", "c", "causal", "true"))
    if args.only_batch:
        w = w.with_(B=args.only_batch)
    gen = torch.Generator(device=dev).manual_seed(w.seed)
    q, k, v, do = (torch.randn(w.B, w.Hq, w.Sq, w.D, device=dev, generator=gen).to(torch.bfloat16)
                   for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    fa.fwd(q, k, v, causal=w.causal, out=o, lse=lse)
    ws = grads = None
    if kind == "bwd":
        ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, det),
                         dtype=torch.uint8, device=dev)
        grads = [torch.empty_like(q) for _ in range(3)]
    ev = []
    for i in range(args.warmup + args.steps):
        e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        fa.set_timing_events(*e)
        if kind == "fwd":
            fa.fwd(q, k, v, causal=w.causal, out=o, lse=lse)
        else:
            fa.bwd(q, k, v, o, do, lse, causal=w.causal, workspace=ws, dq=grads[0], dk=grads[1],
                   dv=grads[2], deterministic=det)
        if i >= args.warmup:
            ev.append(e)
    torch.cuda.synchronize(dev)
    assert fa.fwd_status() == fa.FA_OK
    if ws is not None:
        assert fa.bwd_status(ws) == fa.FA_OK
    ms = sorted(a.elapsed_time(b) for a, b in ev)[len(ev) // 2]
    flops = w.flops(backward=(kind == "bwd"))
    print(json.dumps({"only": args.only, "workload": w.name, "B": w.B, "H": w.Hq, "S": w.Sq,
                      "D": w.D, "causal": w.causal, "deterministic": det,
                      "bwd_kernel": "pair" if mode == "pair" else "default", "ms": round(ms, 4),
                      "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}), flush=True)


def fwd_sweep(fa, dev, peak, iters=10, shapes=None):
    """Forward-only TFLOP/s over the sequence-length sweep (16k tokens per batch),
    or over ``shapes`` [(S, D, causal), ...] of it."""
    import torch
    out = []
    if shapes is None:
        shapes = [(S, D, c) for S in synth.SWEEP_S for D in (64, 128) for c in (False, True)]
    for S, D, causal in shapes:
        w = synth.sweep(S, D, causal)
        q, k, v = (torch.randn(w.B, w.Hq, S, D, device=dev, dtype=torch.bfloat16)
                   for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, S), dtype=torch.float32, device=dev)
        for _ in range(3):
            fa.fwd(q, k, v, causal=causal, out=o, lse=lse)
        torch.cuda.synchronize(dev)
        t = []
        for _ in range(iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            fa.set_timing_events(e0, e1)
            fa.fwd(q, k, v, causal=causal, out=o, lse=lse)
            t.append((e0, e1))
        torch.cuda.synchronize(dev)
        ms = sorted(a.elapsed_time(b) for a, b in t)[len(t) // 2]
        tf = w.flops() / (ms * 1e-3) / 1e12
        out.append({"S": S, "D": D, "B": w.B, "causal": causal, "ms": round(ms, 4),
                    "tflops": round(tf, 1), "frac": round(tf / peak, 4)})
        del q, k, v, o, lse
    return out


def visible_pairs(Sq: int, Sk: int, wl: int, wr: int) -> int:
    """(query, key) pairs a window (wl, wr) leaves visible; negative = unbounded."""
    import numpy as np
    i = np.arange(Sq, dtype=np.int64)
    lo = np.maximum(0, i - wl) if wl >= 0 else np.zeros_like(i)
    hi = np.minimum(Sk - 1, i + wr) if wr >= 0 else np.full_like(i, Sk - 1)
    return int(np.maximum(0, hi - lo + 1).sum())


# padded batch: keys per batch element as fractions of S, repeated over B
PAD_FRACS = (1.0, 0.75, 0.5, 0.25)

# B, H, S, D, window_left, window_right, bias, padded
MOD_SWEEP = [
    (1, 16, 16384, 128, -1, 0, False, False),     # causal (the plain kernels)
    (1, 16, 16384, 128, -1, 0, True, False),      # causal with the relative-position bias
    (1, 16, 16384, 128, 1023, 0, False, False),   # causal local window of 1024 keys
    (1, 16, 16384, 128, 4095, 0, False, False),   # causal local window of 4096 keys
    (1, 16, 16384, 128, 512, 512, True, False),   # two-sided window of 1025 keys with the bias
    (4, 16, 2048, 128, 255, 0, False, False),     # the train shape with a 256-key local window
    (8, 16, 4096, 128, -1, -1, False, True),      # padded batch, keys S, 3S/4, S/2, S/4
    (8, 16, 4096, 128, -1, 0, False, True),       # the same, causal
]


def mod_sweep(fa, dev, peak, iters=10):
    """Forward and backward-main TFLOP/s with a sliding window, the
    relative-position bias and / or the key padding mask; FLOPs counted over the
    visible (query, key) pairs."""
    import torch
    out = []
    for B, H, S, D, wl, wr, bias, padded in MOD_SWEEP:
        gen = torch.Generator(device=dev).manual_seed(9)
        q, k, v, do = (torch.randn(B, H, S, D, device=dev, generator=gen).to(torch.bfloat16)
                       for _ in range(4))
        slopes = (torch.tensor([0.5 ** (1 + h % 8) for h in range(H)], device=dev)
                  if bias else None)
        counts = [int(S * PAD_FRACS[b % len(PAD_FRACS)]) for b in range(B)] if padded else None
        kw = dict(window=(wl, wr), alibi_slopes=slopes,
                  seqlens_k=None if counts is None else torch.tensor(counts, dtype=torch.int32,
                                                                      device=dev))
        ws = torch.empty(fa.bwd_workspace_bytes(B, H, H, S, S, D), dtype=torch.uint8, device=dev)
        o, lse = fa.fwd(q, k, v, **kw)
        grads = [torch.empty_like(q) for _ in range(3)]

        def run(which, e=None):
            if e is not None:
                fa.set_timing_events(*e)
            if which == "fwd":
                fa.fwd(q, k, v, out=o, lse=lse, **kw)
            else:
                fa.bwd(q, k, v, o, do, lse, workspace=ws, dq=grads[0], dk=grads[1], dv=grads[2],
                       **kw)

        ms = {}
        for which in ("fwd", "bwd"):
            for _ in range(3):
                run(which)
            torch.cuda.synchronize(dev)
            t = []
            for _ in range(iters):
                e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                run(which, e)
                t.append(e)
            torch.cuda.synchronize(dev)
            ms[which] = sorted(a.elapsed_time(b) for a, b in t)[len(t) // 2]
        assert fa.fwd_status() == fa.FA_OK and fa.bwd_status(ws) == fa.FA_OK
        f_fwd = 4.0 * H * D * sum(visible_pairs(S, S if counts is None else counts[b], wl, wr)
                                  for b in range(B))
        tf_f = f_fwd / (ms["fwd"] * 1e-3) / 1e12
        tf_b = 2.5 * f_fwd / (ms["bwd"] * 1e-3) / 1e12
        out.append({"B": B, "H": H, "S": S, "D": D, "window": [wl, wr], "bias": bias,
                    "key_counts": counts,
                    "fwd_ms": round(ms["fwd"], 4), "fwd_tflops": round(tf_f, 1),
                    "fwd_frac": round(tf_f / peak, 4), "bwd_main_ms": round(ms["bwd"], 4),
                    "bwd_main_tflops": round(tf_b, 1), "bwd_main_frac": round(tf_b / peak, 4)})
        del q, k, v, do, o, lse, ws, grads
    return out


# B, H, Sq, Sk, D, window_right (-1: none; Sk - Sq: bottom-right causal)
SPLIT_SWEEP = [
    (1, 16, 1024, 32768, 128, 32768 - 1024),   # chunked prefill at the end of a 32k context
    (1, 16, 1024, 32768, 64, 32768 - 1024),
    (2, 16, 128, 16384, 128, -1),              # 128-query block against 16k keys
    (1, 8, 512, 131072, 128, 131072 - 512),    # 512 queries at the end of a 128k context
    (1, 4, 4096, 65536, 128, -1),              # few heads, long context
]


def split_sweep(fa, dev, peak, iters=10):
    """Forward TFLOP/s of the split-KV path (split kernel + merge, timed together)
    against the unsplit kernel, where the unsplit units are fewer than the SMs."""
    import torch
    out = []
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    hbm_peak = float(load_peaks()[0]["hbm_gbs"])
    for B, H, Sq, Sk, D, wr in SPLIT_SWEEP:
        gen = torch.Generator(device=dev).manual_seed(10)
        q = torch.randn(B, H, Sq, D, device=dev, generator=gen).to(torch.bfloat16)
        k, v = (torch.randn(B, H, Sk, D, device=dev, generator=gen).to(torch.bfloat16)
                for _ in range(2))
        o = torch.empty_like(q)
        lse = torch.empty(B, H, Sq, device=dev)
        n_auto = fa.fwd_split_count(B, H, Sq, Sk, sms)
        counts = sorted({1, max(1, n_auto // 2), n_auto, 2 * n_auto})
        ws = torch.empty(max(fa.fwd_split_workspace_bytes(B, H, Sq, Sk, D, n) for n in counts)
                         + 1, dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev)
        f = 4.0 * B * H * D * visible_pairs(Sq, Sk, -1, wr)
        row = {"B": B, "H": H, "Sq": Sq, "Sk": Sk, "D": D, "window_right": wr, "n_auto": n_auto}
        for n in counts:
            def run():
                fa.fwd(q, k, v, out=o, lse=lse, window=(-1, wr), n_splits=n,
                       split_workspace=ws)
            for _ in range(3):
                run()
            torch.cuda.synchronize(dev)
            t = []
            for _ in range(iters):
                e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                e[0].record(stream)
                run()
                e[1].record(stream)
                t.append(e)
            torch.cuda.synchronize(dev)
            ms = sorted(a.elapsed_time(b) for a, b in t)[len(t) // 2]
            tf = f / (ms * 1e-3) / 1e12
            row[f"n{n}"] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                            "frac": round(tf / peak, 4)}
        assert fa.fwd_status() == fa.FA_OK
        # the merge alone, on the automatic count's parts: HBM-bound
        if n_auto > 1:
            rows = B * H * Sq
            parts_o = torch.randn(n_auto, rows, D, device=dev)
            parts_l = torch.randn(n_auto, rows, device=dev)
            for _ in range(3):
                fa.lse_merge(parts_o, parts_l, out=o.view(rows, D), lse=lse.view(rows))
            flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
            t = []
            for _ in range(iters):
                flush.zero_()  # the parts would otherwise sit in L2
                e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                e[0].record(stream)
                fa.lse_merge(parts_o, parts_l, out=o.view(rows, D), lse=lse.view(rows))
                e[1].record(stream)
                t.append(e)
            torch.cuda.synchronize(dev)
            ms = sorted(a.elapsed_time(b) for a, b in t)[len(t) // 2]
            nbytes = rows * (n_auto * (4 * D + 4) + 2 * D + 4)
            gbs = nbytes / (ms * 1e-3) / 1e9
            row["merge"] = {"ms": round(ms, 4), "bytes": nbytes, "gbs": round(gbs, 1),
                            "frac_hbm": round(gbs / hbm_peak, 4)}
            del parts_o, parts_l, flush
        out.append(row)
        del q, k, v, o, lse, ws
    return out


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return  # the CPU oracle runs once, on rank 0
    w = WORKLOAD
    steps, per_step = [], []
    budget = max(2.0, args.cpu_budget / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        v, cores, sample, dt = cpu_oracle_sample(w, budget_s=budget, max_heads=1)
        if i >= args.warmup:
            steps.append(v)
            per_step.append(dt)
    value = sum(steps) / len(steps)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1000 * sum(per_step) / len(per_step), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 inputs of the workload's shape)",
            "config": config_dict(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--sweep", action="store_true", help="also time the forward S/D sweep")
    ap.add_argument("--split-sweep", action="store_true",
                    help="also time the split-KV forward against the unsplit kernel")
    ap.add_argument("--mod-sweep", action="store_true",
                    help="also time sliding-window / relative-position-bias attention")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of CPU oracle work for the baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-train-step", action="store_true",
                    help="skip the training-scale step reported under extra")
    ap.add_argument("--no-long-fwd", action="store_true",
                    help="skip the non-causal S >= 8k D=128 and the S = 8k D=64 forwards reported under extra")
    ap.add_argument("--only", default=None,
                    help="fwd:S:D:causal or bwd:S:D:causal[:det] -- time one kernel call "
                         "shape alone and exit")
    ap.add_argument("--only-batch", type=int, default=0,
                    help="with --only: the batch size instead of the sweep's (e.g. 4 at S=2048 "
                         "for the training-scale shape B4 H16 S2048)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
