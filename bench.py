"""Benchmark: exact attention forward + split-KV decode on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * fa_fwd on the prefill workload [B=16, S=8192, Hq=Hkv=32, D=128], bf16, non-causal
    (the shape of the pages' largest benchmark column, page
    "ampere_flash_attention_from_scratch", "Performance Test");
  * fa_decode_splitkv on the decode workload (B=8, Hq=32, Hkv=8, D=128, per-sequence
    KV lengths U[1024, 32768], Smax=32768, default split count).
The headline value is the forward's algorithmic TFLOP/s (4*B*Hq*Sq*Sk*D per step) over
the whole step time; the decode's HBM GB/s is reported in the "decode" object.  Inputs
are resident in HBM before the timed region and larger than L2 (4 GiB for the forward,
1 GiB of KV cache for decode).  Each kernel is timed with CUDA events on the stream it is
launched on.  `e2e` repeats the step through the public API from pinned host buffers,
every step's host<->device copies included, pipelined so that one step's compute overlaps
the neighbouring steps' copies.  `cpu_baseline` times the CPU oracle on a bounded sample
of the same workload on the host's cores.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 run under torch.distributed.run: each rank runs the same per-GPU workload on
its own GPU (independent replicas, weak scaling, no data-path collective); timing takes
the maximum over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16) and % of GB300 tensor peak; decode HBM GB/s"
# The pages' own number for this workload (official FlashAttention-2 on an RTX 3080, fp16,
# [16, 8192, 32, 128]: 292.02 ms), restated in this benchmark's 4*B*H*S^2*D count.
PAGES_TFLOPS_16_8192 = 4.0 * 16 * 32 * 8192 * 8192 * 128 / 292.02e-3 / 1e12
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", action="store_true",
                    help="instead of the step, time each widened entry point (window, varlen, "
                         "paged and multi-token decode) and print one JSON line per row")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers ----

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity for a single process)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_20_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when absent or
    taken on kernel sources that have changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- workloads ----

def make_workloads(device):
    import torch

    from exact_tiled_attention_20_gb300 import inputs

    wf = inputs.PREFILL_LONG[0]
    wd = inputs.DECODE
    q, k, v = inputs.fwd_inputs(wf)
    dq, dk, dv, lens = inputs.decode_inputs(wd)
    host = dict(q=q, k=k, v=v, dq=dq, dk=dk, dv=dv, lens=lens)
    dev = {n: t.to(device) for n, t in host.items()}
    dev["o"] = torch.empty_like(dev["q"])
    dev["lse"] = torch.empty((wf.B, wf.Hq, wf.Sq), dtype=torch.float32, device=device)
    dev["do"] = torch.empty_like(dev["dq"])
    dev["dlse"] = torch.empty((wd.B, wd.Hq), dtype=torch.float32, device=device)
    return wf, wd, host, dev


def decode_bytes(wd, lens) -> float:
    """Algorithmic HBM bytes of one decode: valid K/V rows, Q, O and LSE."""
    kv = sum(int(n) for n in lens) * wd.Hkv * wd.D * 2 * 2
    return float(kv + wd.B * wd.Hq * wd.D * 2 * 2 + wd.B * wd.Hq * 4)


# --------------------------------------------------------------- native arm ----

def run_native(args, rank, local_rank, world):
    import torch

    import exact_tiled_attention_20_gb300 as fa
    from exact_tiled_attention_20_gb300 import build

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    build.build_library()
    fa.load()
    wf, wd, host, d = make_workloads(device)
    stream = torch.cuda.current_stream()
    ns = fa.fa_decode_default_splits(wd.B, wd.Hkv, wd.Smax)
    ws = torch.empty(fa.fa_decode_workspace_bytes(wd.B, wd.Hq, wd.D, ns), dtype=torch.uint8,
                     device=device)

    def step():
        fa.fa_fwd(d["q"], d["k"], d["v"], causal=wf.causal, scale=wf.scale, out=d["o"],
                  lse=d["lse"], stream=stream)
        fa.fa_decode_splitkv(d["dq"], d["dk"], d["dv"], d["lens"], scale=wd.scale,
                             num_splits=ns, workspace=ws, out=d["do"], lse=d["dlse"],
                             stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.fa_last_device_status() != 0:
        raise RuntimeError("device status reported a kernel timeout during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        fa.fa_fwd(d["q"], d["k"], d["v"], causal=wf.causal, scale=wf.scale, out=d["o"],
                  lse=d["lse"], stream=stream)
        ev[i][1].record(stream)
        fa.fa_decode_splitkv(d["dq"], d["dk"], d["dv"], d["lens"], scale=wd.scale,
                             num_splits=ns, workspace=ws, out=d["do"], lse=d["dlse"],
                             stream=stream)
        ev[i][2].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    if fa.fa_last_device_status() != 0:
        raise RuntimeError("device status reported a kernel timeout in the timed region")

    total_ms = max_over_ranks(t0.elapsed_time(t1), world, device)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    dec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    fwd_ms = max_over_ranks(fwd_ms, world, device)
    dec_ms = max_over_ranks(dec_ms, world, device)
    ms_per_step = total_ms / K
    fwd_flops = wf.flops()
    value = world * fwd_flops / (ms_per_step * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    fwd_tflops = fwd_flops / (fwd_ms * 1e-3) / 1e12
    peak_t = float(peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"])
    dbytes = decode_bytes(wd, host["lens"].tolist())
    dec_gbs = dbytes / (dec_ms * 1e-3) / 1e9
    peak_h = float(peaks["hbm_gbs"])
    fwd_traffic = ncu_traffic("fa_fwd_kernel")
    dec_traffic = ncu_traffic("fa_decode_split_kernel")

    # ---- end to end through the public API, host buffers, copies inside the timed region
    # Every step copies its inputs from pinned host memory, runs the step and reads its
    # results back.  Steps are pipelined over two buffer sets on three streams (inputs in,
    # compute, results out), so step i's compute overlaps step i+1's upload and step i-1's
    # download; the timed region runs from the first upload to the last download.  (Spreading
    # the uploads over several streams measured no faster: the host link is the limit.)
    e2e = None
    if args.e2e_steps > 0:
        pin = {n: t.pin_memory() for n, t in host.items()}
        bufs = [d]
        d2 = {n: torch.empty_like(t) for n, t in d.items()}
        bufs.append(d2)
        outs = [dict(o=torch.empty_like(pin["q"]).pin_memory(),
                     lse=torch.empty(tuple(d["lse"].shape), dtype=torch.float32).pin_memory(),
                     do=torch.empty_like(pin["dq"]).pin_memory(),
                     dlse=torch.empty(tuple(d["dlse"].shape), dtype=torch.float32).pin_memory())
                for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
        s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
        ws2 = [ws, torch.empty_like(ws)]
        in_ready = [torch.cuda.Event() for _ in range(2)]
        cmp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            b = i % 2
            db, ob = bufs[b], outs[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(cmp_done[b])  # step i-2 has finished reading buffer b
                for n in ("q", "k", "v", "dq", "dk", "dv", "lens"):
                    db[n].copy_(pin[n], non_blocking=True)
                in_ready[b].record(s_in)
            s_cmp.wait_event(in_ready[b])
            if i >= 2:
                s_cmp.wait_event(out_done[b])  # step i-2's results have left buffer b
            fa.fa_fwd(db["q"], db["k"], db["v"], causal=wf.causal, scale=wf.scale, out=db["o"],
                      lse=db["lse"], stream=s_cmp)
            fa.fa_decode_splitkv(db["dq"], db["dk"], db["dv"], db["lens"], scale=wd.scale,
                                 num_splits=ns, workspace=ws2[b], out=db["do"], lse=db["dlse"],
                                 stream=s_cmp)
            cmp_done[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[b])
                for n in ("o", "lse", "do", "dlse"):
                    ob[n].copy_(db[n], non_blocking=True)
                out_done[b].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        for i in range(args.e2e_steps):
            e2e_step(i)
        a1.record(s_out)
        torch.cuda.synchronize()
        if fa.fa_last_device_status() != 0:
            raise RuntimeError("device status reported a kernel timeout in the end-to-end run")
        e_ms = max_over_ranks(a0.elapsed_time(a1) / args.e2e_steps, world, device)
        e2e = {"value": round(world * fwd_flops / (e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(e_ms, 3), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps,
               "pipelined": "2 buffer sets, upload / compute / download streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wf, host)

    if rank != 0:
        return
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(value / (world * PAGES_TFLOPS_16_8192), 2),
        "vs_baseline_ref": ("official FlashAttention-2 on an RTX 3080, fp16, [16,8192,32,128], "
                            f"{PAGES_TFLOPS_16_8192:.1f} TFLOP/s in this count (other hardware: context)"),
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": ("fa_fwd prefill [B=16,S=8192,Hq=Hkv=32,D=128] non-causal + "
                         f"fa_decode_splitkv [B=8,Hq=32,Hkv=8,D=128,kv_len~U[1024,32768],"
                         f"Smax=32768,num_splits={ns}]"),
            "global_batch": wf.B * world,
            "seq_len": wf.Sq,
            "parallelism": "replicas" if world == 1 else f"replicas{world}",
            "l2": "inputs larger than L2 (fwd 4 GiB, decode KV 1 GiB)",
        },
        "pct_of_tensor_peak": round(100.0 * fwd_tflops / peak_t, 1),
        "roofline": {
            "kernel": "fa_fwd_kernel",
            "bound": "tensor",
            "achieved": round(fwd_tflops, 1),
            "peak": peak_t,
            "peak_source": f"{peak_src} bf16 sustained (kernel timed inside a long step)",
            "unit": "TFLOP/s",
            "frac": round(fwd_tflops / peak_t, 4),
            "frac_of_burst": round(fwd_tflops / float(peaks["bf16_tflops"]), 4),
            "traffic": fwd_traffic,
            "ms_per_launch": round(fwd_ms, 4),
        },
        "decode": {
            "value": round(dec_gbs, 1),
            "unit": "GB/s",
            "ms_per_launch": round(dec_ms, 4),
            "algorithmic_bytes": int(dbytes),
            "roofline": {
                "kernel": "fa_decode_split_kernel + fa_decode_combine_kernel",
                "bound": "hbm",
                "achieved": round(dec_gbs, 1),
                "peak": peak_h,
                "peak_source": f"{peak_src} copy bandwidth",
                "unit": "GB/s",
                "frac": round(dec_gbs / peak_h, 4),
                "traffic": dec_traffic,
            },
        },
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------- CPU baseline ----

def _sample_rows(wf, n_rows, seed=7):
    import numpy as np

    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, wf.B, n_rows), rng.integers(0, wf.Hq, n_rows),
                     rng.integers(0, wf.Sq, n_rows)], axis=1)
    return rows.astype(np.int64)


def _row_flops(wf, rows) -> float:
    if not wf.causal:
        return 4.0 * wf.Sk * wf.D * len(rows)
    return float(sum(4.0 * min(wf.Sk, int(i) + wf.Sk - wf.Sq + 1) * wf.D for i in rows[:, 2]))


def cpu_baseline(wf, host, target_s: float = 8.0):
    """The oracle (fp64, as it stands) on a bounded random sample of output rows of the
    forward workload, on all host cores; reported in the same unit as the GPU number."""
    import oracle

    cores = os.cpu_count() or 1
    probe = _sample_rows(wf, cores, seed=3)
    t = time.perf_counter()
    oracle.fwd(host["q"], host["k"], host["v"], scale=wf.scale, causal=wf.causal, rows=probe,
               nthreads=cores)
    per_batch = max(time.perf_counter() - t, 1e-3)
    n = max(cores, int(cores * target_s / per_batch))
    rows = _sample_rows(wf, n)
    t = time.perf_counter()
    oracle.fwd(host["q"], host["k"], host["v"], scale=wf.scale, causal=wf.causal, rows=rows,
               nthreads=cores)
    dt = time.perf_counter() - t
    return {"value": round(_row_flops(wf, rows) / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": cores, "kind": "oracle",
            "sample": (f"{n} random output rows (all {wf.Sk} keys each) of the fa_fwd workload, "
                       f"fp64, {dt:.1f} s wall")}


# ----------------------------------------------------------- reference arm ----

def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded sample of output rows
    of the same forward workload, timed on the host cores."""
    if rank != 0:
        return
    import numpy as np  # noqa: F401

    import oracle
    from exact_tiled_attention_20_gb300 import inputs

    wf = inputs.PREFILL_LONG[0]
    q, k, v = inputs.fwd_inputs(wf)
    cores = os.cpu_count() or 1
    n = 2 * cores
    for i in range(args.warmup):
        oracle.fwd(q, k, v, scale=wf.scale, causal=wf.causal, rows=_sample_rows(wf, cores, 100 + i),
                   nthreads=cores)
    flops = 0.0
    t = time.perf_counter()
    for i in range(args.steps):
        rows = _sample_rows(wf, n, 1000 + i)
        oracle.fwd(q, k, v, scale=wf.scale, causal=wf.causal, rows=rows, nthreads=cores)
        flops += _row_flops(wf, rows)
    dt = time.perf_counter() - t
    value = flops / dt / 1e12
    sample = f"{n} random output rows per step of the fa_fwd workload, fp64"
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / max(args.steps, 1) * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "fa_fwd prefill [B=16,S=8192,Hq=Hkv=32,D=128] non-causal (row sample)",
                   "global_batch": wf.B, "seq_len": wf.Sq, "parallelism": "host threads"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------- widened rows ----

def _time_ms(fn, reps=10, warmup=3):
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_rows(args):
    """One JSON line per widened entry point, each with its roofline.  Forward variants
    count the visible (query, key) pairs: 4 * D * pairs * Hq FLOPs; decode variants count
    the valid K/V bytes plus Q, O and LSE."""
    import numpy as np
    import torch

    import exact_tiled_attention_20_gb300 as fa
    from exact_tiled_attention_20_gb300 import build, inputs

    build.build_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, src = load_peaks()
    peak_t = float(peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"])
    peak_h = float(peaks["hbm_gbs"])

    def emit(row, workload, ms, achieved, unit, bound, extra=None):
        peak = peak_t if bound == "tensor" else peak_h
        d = {"row": row, "workload": workload, "ms": round(ms, 4), "value": round(achieved, 1),
             "unit": unit, "roofline": {"bound": bound, "achieved": round(achieved, 1), "peak": peak,
                                        "peak_source": f"{src}", "frac": round(achieved / peak, 4)}}
        if extra:
            d.update(extra)
        print(json.dumps(d), flush=True)
        if fa.fa_last_device_status() != 0:
            raise RuntimeError(f"device status after {row}")

    # sliding window: [16, 8192, 32, 128] causal, window of 1024 keys
    w = inputs.PREFILL_LONG[0]
    q, k, v = (t.to(dev) for t in inputs.fwd_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), device=dev)
    win = 1023
    ms = _time_ms(lambda: fa.fa_fwd(q, k, v, causal=True, window=(win, 0), out=o, lse=lse))
    pairs = sum(min(i + 1, win + 1) for i in range(w.Sq))
    flops = 4.0 * w.D * pairs * w.Hq * w.B
    emit("sliding_window", "fa_fwd_window [16,8192,32,128] causal, window (1023, 0)", ms,
         flops / ms / 1e9, "TFLOP/s", "tensor")
    # variable length: 16 sequences of U[256, 8192] rows, causal, packed
    rng = np.random.default_rng(1005)
    lens = [int(x) for x in rng.integers(256, 8193, 16)]
    tq = sum(lens)
    qv, kv_, vv = q.view(-1, w.Hq, w.D)[:tq], k.view(-1, w.Hkv, w.D)[:tq], v.view(-1, w.Hkv, w.D)[:tq]
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
    ov = torch.empty_like(qv)
    lv = torch.empty((w.Hq, tq), device=dev)
    ms = _time_ms(lambda: fa.fa_fwd_varlen(qv, kv_, vv, cu, cu, causal=True, out=ov, lse=lv))
    pairs = sum(n * (n + 1) // 2 for n in lens)
    emit("varlen", f"fa_fwd_varlen 16 sequences U[256,8192] (total {tq}), Hq=Hkv=32, D=128, causal",
         ms, 4.0 * w.D * pairs * w.Hq / ms / 1e9, "TFLOP/s", "tensor")
    del q, k, v, o, lse, qv, kv_, vv, ov, lv
    torch.cuda.empty_cache()
    # decode variants on the decode workload
    wd = inputs.DECODE
    dq, dk, dv, dl = inputs.decode_inputs(wd)
    nbytes = decode_bytes(wd, dl.tolist())
    page = 256
    mp = wd.Smax // page
    perm = torch.randperm(wd.B * mp, generator=torch.Generator().manual_seed(7))
    table = perm.view(wd.B, mp).to(torch.int32)
    kp = torch.empty((wd.B * mp, page, wd.Hkv, wd.D), dtype=dk.dtype)
    vp = torch.empty_like(kp)
    kp[perm] = dk.view(wd.B * mp, page, wd.Hkv, wd.D)
    vp[perm] = dv.view(wd.B * mp, page, wd.Hkv, wd.D)
    dqd, kpd, vpd, tbd, dld = (t.to(dev) for t in (dq, kp, vp, table, dl))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flushed(fn):
        def run():
            flush.sum()  # read 256 MiB to evict the cache from L2 (clean lines)
            fn()
        return run
    base = _time_ms(flushed(lambda: None))
    ms = _time_ms(flushed(lambda: fa.fa_decode_splitkv_paged(dqd, kpd, vpd, tbd, dld))) - base
    emit("paged_decode", "fa_decode_splitkv_paged, decode workload in 256-key pages (random page order)",
         ms, nbytes / ms / 1e6, "GB/s", "hbm")
    del kpd, vpd
    dkd, dvd = dk.to(dev), dv.to(dev)
    ms = _time_ms(flushed(lambda: fa.fa_decode_splitkv(dqd, dkd, dvd, dld))) - base
    emit("decode", "fa_decode_splitkv, decode workload (L2 flushed by a 256 MiB read between calls)",
         ms, nbytes / ms / 1e6, "GB/s", "hbm")
    q4 = torch.randn((wd.B, 4, wd.Hq, wd.D), device=dev).to(torch.bfloat16)
    nb4 = nbytes + 3 * wd.B * wd.Hq * wd.D * 2 * 2
    ms = _time_ms(flushed(lambda: fa.fa_decode_splitkv_multi(q4, dkd, dvd, dld, causal=True))) - base
    emit("multi_token_decode", "fa_decode_splitkv_multi, decode workload with 4 causal tokens",
         ms, nb4 / ms / 1e6, "GB/s", "hbm")


def main(argv=None):
    args = parse_args(argv)
    rank, local_rank, world = dist_env()
    if args.rows:
        if rank == 0:
            run_rows(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_native(args, rank, local_rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
