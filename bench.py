#!/usr/bin/env python
"""Throughput of exact tiled attention on GB300, printed as one JSON line.

A step is one pass of the whole hot path over one batch of synthetic input:
the forward (fa_fwd) and, where the library has it, the backward by
recomputation (fa_bwd) on the same batch, on the long-sequence,
large-logit workload (B=2, H=16, N=8192, d=128, bf16, Q and K drawn x8).
``value`` is TFLOP/s under the attention flop convention: 4*B*H*N^2*d for the
forward plus 2.5x that for the backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU as an
independent replica (heads are independent problems: no data-path
collective); the slowest rank's time sets the step time and rank 0 prints.
``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload (rank 0 only).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
REF_ROWS = 512  # query rows per reference-arm step
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3, help="workload index (configs.WORKLOADS)")
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d[,window[,qk_mult]]: a bf16 problem of another shape instead of a workload "
                         "(for measuring other head dimensions; not a bench line of record)")
    ap.add_argument("--no-bwd", action="store_true", help="forward only")
    ap.add_argument("--dtype", choices=["bf16", "f32"], default="bf16", help="dtype of a --shape problem")
    ap.add_argument("--f32-path", choices=["simt", "3xtf32"], default="simt",
                    help="float32 forward: exact CUDA-core kernel, or the tensor-core 3xTF32 split (d <= 128, "
                         "forward only)")
    ap.add_argument("--schedule", choices=["query-major", "key-major"], default="query-major",
                    help="forward loop order; key-major (outer loop over key tiles, O in device memory between "
                         "steps) is a comparison schedule and runs forward only")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-kernel timing of the other bf16 workloads (2, 4, 5) in the default line")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# ncu traffic figure (only while the kernel source is unchanged since capture)
# ---------------------------------------------------------------------------
def kernel_source_hash(name: str) -> str:
    path = os.path.join(ROOT, "exact_tiled_attention_02_gb300", "csrc", name)
    h = hashlib.sha256()
    for p in (path, os.path.join(ROOT, "exact_tiled_attention_02_gb300", "csrc", "sm103.cuh")):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(summary: str, source: str):
    """Per-launch DRAM bytes recorded in a profiles/ summary, if the summary's
    source hash matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        text = open(path).read()
    except OSError:
        return None
    want = kernel_source_hash(source)
    meta = {}
    for ln in text.splitlines():
        if ln.startswith("bench-key:"):
            for kv in ln[len("bench-key:"):].split():
                k, _, v = kv.partition("=")
                meta[k] = v
    if meta.get("source_sha") != want:
        return None
    try:
        return float(meta["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(w, q, k, v, do, with_bwd, budget_s: float, max_heads=None, rows=None):
    """Times the float64 oracle head by head until ``budget_s`` is spent;
    returns (flops done, seconds, heads).  With ``rows`` (unmasked workloads
    only) each head contributes just its first ``rows`` query rows against all
    keys: the forward of those rows and their share of the backward (their dQ
    rows and their contributions to dK and dV), i.e. rows/N of the head's
    flops."""
    import numpy as np

    import oracle

    n_rows = w.N if rows is None else min(rows, w.N)
    if n_rows < w.N and w.window > 0:
        raise ValueError("row samples are only defined for unmasked workloads")
    flops_head_f = w.fwd_flops() / (w.B * w.H) * n_rows / w.N
    done_f, t_total, heads = 0.0, 0.0, 0
    order = [(b, h) for b in range(w.B) for h in range(w.H)]
    for b, h in order:
        if max_heads is not None and heads >= max_heads:
            break
        qh = q[b, h, :n_rows].float().numpy().astype(np.float64)
        kh = k[b, h].float().numpy().astype(np.float64)
        vh = v[b, h].float().numpy().astype(np.float64)
        t0 = time.perf_counter()
        oracle.dense_forward(qh, kh, vh, w.scale, w.window)
        if with_bwd:
            oracle.dense_backward(qh, kh, vh, do[b, h, :n_rows].float().numpy().astype(np.float64), w.scale,
                                  w.window)
        t_total += time.perf_counter() - t0
        done_f += flops_head_f * (3.5 if with_bwd else 1.0)
        heads += 1
        if t_total >= budget_s:
            break
    return done_f, t_total, heads


def data_desc(w):
    return "synthetic (seeded standard normals" + (f", Q,K x{w.qk_mult:g}" if w.qk_mult != 1.0 else "") + ")"


def l2_note(w, qd):
    total = 4 * qd.numel() * qd.element_size()
    if total > L2_BYTES:
        return f"inputs larger than L2 (Q,K,V,O {total / 1e6:.0f} MB > 129 MB); no flush"
    return f"inputs smaller than L2 ({total / 1e6:.2f} MB); no flush (latency-bound case)"


def dist_max(x: float, pg=None, device=None) -> float:
    """Maximum of ``x`` over all ranks (the slowest rank sets the step time);
    ``x`` itself when there is no process group."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank processes its own full workload (heads
    are independent problems), so the job does world x the work of one rank
    in the slowest rank's time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------------------
def main():
    args = parse_args()
    import torch

    from exact_tiled_attention_02_gb300 import configs, inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = configs.WORKLOADS[args.workload] if args.shape is None else configs.custom_workload(args.shape, args.dtype)

    if args.impl == "reference":
        if rank != 0:
            return 0
        run_reference(args, w, world)
        return 0

    from exact_tiled_attention_02_gb300 import binding as fa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    key_major = args.schedule == "key-major"
    tf32x3 = w.dtype == "f32" and args.f32_path == "3xtf32"
    with_bwd = not args.no_bwd and not key_major and not tf32x3
    q, k, v, do = inputs.workload_inputs(w, with_do=True)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    fwd_fn = fa.fa_fwd
    if key_major:
        km_ws = torch.empty(fa.fa_fwd_key_major_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)

        def fwd_fn(q_, k_, v_, **kw):
            return fa.fa_fwd_key_major(q_, k_, v_, workspace=km_ws, **kw)
    if tf32x3:
        tc_ws = torch.empty(fa.fa_fwd_f32_3xtf32_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)

        def fwd_fn(q_, k_, v_, **kw):
            return fa.fa_fwd_f32_3xtf32(q_, k_, v_, workspace=tc_ws, **kw)
    od = torch.empty_like(qd)
    lsed = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    dqd, dkd, dvd = (torch.empty_like(qd) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)

    # The library has no backward for bf16 d = 256 only; such a problem is
    # timed forward only and its metric says so.  For every other head
    # dimension a refusal is an error, never a silent forward-only line.
    if with_bwd and w.dtype == "bf16" and w.d == 256:
        with_bwd = False
    if with_bwd:
        fa.fa_bwd(qd, kd, vd, *fa.fa_fwd(qd, kd, vd, scale=w.scale, window=w.window), dod, scale=w.scale,
                  window=w.window, dq=dqd, dk=dkd, dv=dvd, workspace=ws)
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        fwd_fn(qd, kd, vd, scale=w.scale, window=w.window, o=od, lse=lsed)
        if evs is not None:
            evs[1].record(stream)
        if with_bwd:
            fa.fa_bwd(qd, kd, vd, od, lsed, dod, scale=w.scale, window=w.window, dq=dqd, dk=dkd, dv=dvd,
                      workspace=ws)
            if evs is not None:
                evs[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device())
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    sampler.start()
    start.record(stream)
    for i in range(K):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if pg is not None:
        pg.barrier()
    total_ms = start.elapsed_time(end)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) if with_bwd else None
    total_ms = dist_max(total_ms, pg, dev)
    assert fa.fa_last_device_status() == fa.FA_OK, "a device-side wait timed out during the bench"

    ms_per_step = total_ms / K
    flops_fwd = w.fwd_flops()
    flops_bwd = w.bwd_flops() if with_bwd else 0.0
    flops_step = flops_fwd + flops_bwd
    value = weak_scaling_value(flops_step, world, ms_per_step)

    peaks, peak_src = load_peaks()
    peak, bound, peak_note = peaks["bf16_tflops"], "tensor", f"{peak_src} bf16 dense (burst)"
    if tf32x3:
        # three tf32 products per float32 product; tf32 at the nominal tf32/bf16 ratio of the measured bf16 peak
        peak = peaks["bf16_tflops"] * (1.1 / 2.25) / 3.0
        peak_note = f"{peak_src} bf16 dense (burst) x 1.1/2.25 (nominal tf32/bf16) / 3 (3xTF32 products)"
    elif w.dtype == "f32":
        # CUDA-core fp32 FMA: SMs x 128 lanes x 2 flops x 2.07 GHz (the maximum SM clock)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak, bound = sms * 128 * 2 * 2.07e9 / 1e12, "alu"
        peak_note = f"fp32 FMA: {sms} SMs x 128 lanes x 2 flops x 2.07 GHz"
    kernels = {"fwd": {"ms": fwd_ms, "tflops": flops_fwd / (fwd_ms * 1e-3) / 1e12}}
    kernels["fwd"]["frac"] = kernels["fwd"]["tflops"] / peak
    if with_bwd:
        kernels["bwd"] = {"ms": bwd_ms, "tflops": flops_bwd / (bwd_ms * 1e-3) / 1e12}
        kernels["bwd"]["frac"] = kernels["bwd"]["tflops"] / peak
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    win_kernel = w.dtype == "bf16" and w.d != 256 and 0 < w.window <= 257  # radius <= 128
    kname = {"fwd": "fwd_keymajor_sm103" if key_major else
             ("fwd_f32_tc128_sm103" if w.d > 64 else "fwd_f32_tc_sm103") if tf32x3 else
             "fwd_f32_simt" if w.dtype == "f32" else "fwd_bf16_d256_sm103" if w.d == 256 else
             "fwd_bf16_win_sm103" if win_kernel else "fwd_bf16_sm103",
             "bwd": "bwd_f32_simt" if w.dtype == "f32" else "bwd_bf16_d64_sm103" if w.d == 64 else
             "bwd_bf16_sm103"}[dom]
    traffic = ncu_traffic(f"{kname}_{w.name}.md", kname + ".cu")
    roofline = {"bound": bound, "kernel": dom, "achieved": round(kernels[dom]["tflops"], 2),
                "peak": round(peak, 2), "unit": "TFLOP/s", "frac": round(kernels[dom]["frac"], 4),
                "traffic": traffic, "peak_source": peak_note}

    workloads = None
    default_line = args.shape is None and args.workload == 3 and not key_major and not args.no_bwd
    if default_line and not args.no_workloads:
        workloads = time_workloads(fa, (2, 4, 5), K, peaks, dev)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(fa, w, q, k, v, do, with_bwd, dev, K, pg, fwd_fn)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, secs, heads = oracle_sample(w, q, k, v, do, with_bwd, budget_s=10.0)
        cpu = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{heads} of {w.B * w.H} heads, float64 numpy oracle "
                         f"({'forward + backward' if with_bwd else 'forward'}), {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": "attention TFLOP/s (fwd 4*B*H*N^2*d" + (" + bwd 2.5x" if with_bwd else "") + ")",
            "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": data_desc(w),
            "config": {"workload": w.name + (" + bwd on the same batch" if with_bwd else ""), "B": w.B, "H": w.H,
                       "N": w.N, "d": w.d, "window": w.window, "qk_mult": w.qk_mult,
                       "schedule": args.schedule,
                       "f32_path": args.f32_path if w.dtype == "f32" else None,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "sms": torch.cuda.get_device_properties(dev).multi_processor_count,
                       "l2": l2_note(w, qd)},
            "kernels": {n: {kk: round(vv, 4) for kk, vv in d.items()} for n, d in kernels.items()},
            "roofline": roofline,
            "workloads": workloads,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": K * ((-(-w.N // 128) + 1) if key_major else (4 if w.d <= 64 else 3) if tf32x3 else
                                 (1 + (3 if with_bwd else 0))),
            "clocks": clocks,
        }
        print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()
    return 0


def algorithmic_bytes(w, with_bwd: bool):
    """HBM bytes the forward (and backward) must move at the least: the
    forward reads Q, K, V and writes O and lse; the backward reads Q, K, V, O,
    dO and lse and writes dQ, dK, dV."""
    elt = 2 if w.dtype == "bf16" else 4
    t = w.B * w.H * w.N * w.d * elt
    rows = w.B * w.H * w.N * 4
    fwd = 4 * t + rows
    bwd = 8 * t + rows if with_bwd else 0
    return fwd, bwd


def time_workloads(fa, indices, steps, peaks, dev):
    """Per-kernel times of other workloads of record, each on its own seeded
    inputs, with CUDA events around each launch on the launching stream:
    forward, then backward on the same batch.  Inputs smaller than L2 get an
    L2 flush (a write of twice L2's size) before every step, outside the
    timed launches.  Returns {workload name: {...}}."""
    import torch

    from exact_tiled_attention_02_gb300 import configs, inputs

    out = {}
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    for idx in indices:
        w = configs.WORKLOADS[idx]
        q, k, v, do = (t.to(dev) for t in inputs.workload_inputs(w, with_do=True))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)
        small = 4 * q.numel() * q.element_size() <= L2_BYTES

        def one(evs=None):
            if small:
                flush.fill_(1)
            if evs:
                evs[0].record(stream)
            fa.fa_fwd(q, k, v, scale=w.scale, window=w.window, o=o, lse=lse)
            if evs:
                evs[1].record(stream)
            fa.fa_bwd(q, k, v, o, lse, do, scale=w.scale, window=w.window, dq=dq, dk=dk, dv=dv, workspace=ws)
            if evs:
                evs[2].record(stream)

        for _ in range(3):
            one()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            one(evs[i])
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK, f"a device-side wait timed out in workload {idx}"
        fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
        bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
        fb, bb = algorithmic_bytes(w, True)
        rec = {}
        for name, ms, fl, by in (("fwd", fwd_ms, w.fwd_flops(), fb), ("bwd", bwd_ms, w.bwd_flops(), bb)):
            tf = fl / (ms * 1e-3) / 1e12
            r = {"ms": round(ms, 4), "tflops": round(tf, 2), "frac": round(tf / peaks["bf16_tflops"], 4)}
            if w.window > 0:
                gbs = by / (ms * 1e-3) / 1e9
                r.update({"hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)})
            rec[name] = r
        rec["config"] = {"B": w.B, "H": w.H, "N": w.N, "d": w.d, "window": w.window, "qk_mult": w.qk_mult,
                         "l2": "flushed before every step" if small else "inputs larger than L2; no flush"}
        out[w.name] = rec
        del q, k, v, do, o, lse, dq, dk, dv, ws
    del flush
    torch.cuda.empty_cache()
    return out


def run_e2e(fa, w, q, k, v, do, with_bwd, dev, steps, pg, fwd_fn=None):
    """Same metric through the public API with pinned host buffers: every step
    copies its inputs host->device, runs the pass(es) and copies its results
    device->host, and all of it lies inside the timed region.  As a training
    loop's data loader would, the copies run on their own streams, overlapped
    with the compute of the neighbouring steps: step i+1's inputs go up while
    step i computes, and step i-1's results come down meanwhile (two device
    buffer sets; events order every reuse).  The timed region starts before
    step 0's upload and ends after the last step's download, and spans the
    same number of steps as the kernel timing, so the one upload and one
    download that nothing overlaps are spread over as many steps."""
    import torch

    fwd = fwd_fn or fa.fa_fwd
    hin = [t.pin_memory() for t in ((q, k, v, do) if with_bwd else (q, k, v))]
    hout = [torch.empty_like(q).pin_memory(), torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()]
    if with_bwd:
        hout += [torch.empty_like(q).pin_memory() for _ in range(3)]
    din = [[torch.empty_like(t, device=dev) for t in hin] for _ in range(2)]
    dout = [[torch.empty_like(t, device=dev) for t in hout] for _ in range(2)]
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)
    compute = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free, out_ready, out_free = ([ev(), ev()] for _ in range(4))
    started = [False, False]

    def upload(i):
        s = i % 2
        with torch.cuda.stream(up):
            if started[s]:
                up.wait_event(in_free[s])
            for d, h in zip(din[s], hin):
                d.copy_(h, non_blocking=True)
            in_ready[s].record(up)

    def run(i):
        s = i % 2
        compute.wait_event(in_ready[s])
        if started[s]:
            compute.wait_event(out_free[s])
        x = din[s]
        o, l = dout[s][0], dout[s][1]
        fwd(x[0], x[1], x[2], scale=w.scale, window=w.window, o=o, lse=l)
        if with_bwd:
            fa.fa_bwd(x[0], x[1], x[2], o, l, x[3], scale=w.scale, window=w.window, dq=dout[s][2], dk=dout[s][3],
                      dv=dout[s][4], workspace=ws)
        in_free[s].record(compute)
        out_ready[s].record(compute)
        started[s] = True

    def download(i):
        s = i % 2
        with torch.cuda.stream(down):
            down.wait_event(out_ready[s])
            for h, d in zip(hout, dout[s]):
                h.copy_(d, non_blocking=True)
            out_free[s].record(down)

    def loop(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            run(i)
            download(i)

    loop(3)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(compute)
    up.wait_stream(compute)  # the first upload starts after the start event
    loop(steps)
    compute.wait_stream(down)  # the end event follows the last download
    b.record(compute)
    torch.cuda.synchronize()
    ms = dist_max(a.elapsed_time(b) / steps, pg, dev)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    flops = w.fwd_flops() + (w.bwd_flops() if with_bwd else 0.0)
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    return {"value": round(weak_scaling_value(flops, world, ms), 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "overlap": "copies on their own streams"}


def run_reference(args, w, world):
    """The oracle as it stands, timed on the host cores.  Each step is a
    bounded sample of the same workload: the first REF_ROWS query rows of head
    (0, 0) against all of its keys (forward, and backward share), so that the
    whole --steps/--warmup run stays within a few minutes."""
    from exact_tiled_attention_02_gb300 import inputs

    q, k, v, do = inputs.workload_inputs(w, with_do=True)
    with_bwd = not args.no_bwd
    rows = REF_ROWS if w.window <= 0 else None
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, do, with_bwd, budget_s=0.0, max_heads=1, rows=rows)
    fl_tot, t_tot = 0.0, 0.0
    for _ in range(args.steps):
        fl, secs, _ = oracle_sample(w, q, k, v, do, with_bwd, budget_s=0.0, max_heads=1, rows=rows)
        fl_tot += fl
        t_tot += secs
    value = fl_tot / t_tot / 1e12
    cores = cpu_cores()
    sample = (f"first {rows} query rows of head (0,0) against all {w.N} keys per step" if rows else
              "head (0,0) per step") + ", float64 numpy oracle" + (" (forward + backward)" if with_bwd else "")
    line = {
        "metric": "attention TFLOP/s (fwd 4*B*H*N^2*d" + (" + bwd 2.5x" if with_bwd else "") + ")",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": data_desc(w), "impl": "reference",
        "config": {"workload": w.name + (" + bwd on the same batch" if with_bwd else ""), "B": w.B, "H": w.H,
                   "N": w.N, "d": w.d, "window": w.window, "qk_mult": w.qk_mult},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    sys.exit(main())
