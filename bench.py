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
of the forward workload and on the whole decode workload, on the host's cores.

`configs` then measures every workload on its own: each prefill shape of the pages'
table, both causal settings of the long one, the grouped-query head-dim sweep, tiny,
decode, and the widened rows (sliding window, variable length, paged and multi-token
decode).  Each entry carries its median CUDA-event time (L2 flushed before every launch
by writing one buffer larger than L2 and reading another), the algorithmic rate, the
fraction of the measured peak, and the oracle run on a sample of that workload's outputs
on the host cores: its time and rate, and max|dO| / max|dLSE| of the GPU output there.

The roofline peak of each figure is chosen from the clock record of its own timed
region: the measured burst bf16 peak while the SM clock stays at its maximum and the
power cap is not engaged for most samples, the sustained (power-capped) peak otherwise.
Both fractions are printed, and `peak_kind` names the one `frac` uses.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-configs]
python bench.py --case KIND ARGS...   (one kernel on its own, e.g. under ncu; see CASES)
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
# Dense bf16 tensor-core rate of one SM per clock: one 128x256x16 MMA per 128 cycles
# (a 128x128x16 MMA measured 67 cycles in isolation against 64 at this rate).  Used only
# for the secondary "fraction of the clock-scaled nominal peak".
NOMINAL_BF16_FLOP_PER_CLK_SM = 8192
O_TOL, LSE_TOL = 1e-2, 1e-3

CASES = """\
  --case fwd B S Hq Hkv D causal [iters]
  --case fwd_window B S Hq Hkv D left right [iters]
  --case fwd_varlen_workload [iters]          16 causal sequences U[256, 8192], Hq=Hkv=32, D=128
  --case decode B Hq Hkv D Smax [iters]       lengths U[Smax/32, Smax]
  --case decode_workload [iters] [D]          the decode workload (its lengths at head dim D,
                                              default 128), default split count
  --case decode_paged_workload [iters]        the same in 256-key pages, random page order
"""


def parse_args(argv=None):
    ap = argparse.ArgumentParser(epilog=CASES, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload measurements (the `configs` array)")
    ap.add_argument("--configs-only", action="store_true",
                    help="run only the per-workload measurements and print them as the line")
    ap.add_argument("--config-reps", type=int, default=20)
    ap.add_argument("--oracle-budget-s", type=float, default=1.5,
                    help="host seconds of oracle work per workload for its parity sample")
    ap.add_argument("--case", nargs=argparse.REMAINDER,
                    help="run one kernel a few times on device-resident inputs and print its "
                         "mean time per call (see the list below)")
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


def choose_tensor_peak(peaks, src, clocks):
    """(peak TFLOP/s, kind) for a kernel whose timed region left the clock record
    ``clocks``: the burst figure while the SM clock held its maximum and the power cap
    was engaged for fewer than half of the samples under load, the sustained one
    otherwise (and when there is no record)."""
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained") or burst)
    if clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        at_max = clocks["sm_mhz"] >= 0.97 * clocks["sm_max_mhz"]
        capped = clocks.get("power_cap_frac", 0.0) >= 0.5
        if at_max and not capped:
            return burst, f"{src} bf16 burst (SM clock at its maximum, power cap not engaged)"
    return sustained, f"{src} bf16 sustained (power-capped or lowered SM clock, or no clock record)"


def tensor_roofline(achieved, peaks, src, clocks, num_sms=152):
    """Roofline object of a tensor-bound figure (TFLOP/s)."""
    peak, kind = choose_tensor_peak(peaks, src, clocks)
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained") or burst)
    r = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "peak_kind": kind,
         "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
         "frac_of_burst": round(achieved / burst, 4), "frac_of_sustained": round(achieved / sustained, 4)}
    if clocks and clocks.get("sm_mhz"):
        nominal = num_sms * NOMINAL_BF16_FLOP_PER_CLK_SM * clocks["sm_mhz"] * 1e6 / 1e12
        r["clock_nominal"] = {"peak": round(nominal, 1), "frac": round(achieved / nominal, 4),
                              "basis": f"{num_sms} SMs x {NOMINAL_BF16_FLOP_PER_CLK_SM} dense bf16 "
                                       "FLOP/clk/SM x median SM MHz under load"}
    return r


# Sources a kernel's traffic depends on: its own files, the shared PTX layer and the ABI
# (which encodes the tensor maps and picks the launch shape).
KERNEL_SOURCES = {
    "fa_fwd_kernel": ("fa_fwd",),
    "fa_decode_split_kernel": ("fa_decode",),
}
SHARED_SOURCES = ("fa_ptx.cuh", "fa_internal.h", "fa_api.cu")


def kernel_source_files(kernel: str):
    csrc = os.path.join(ROOT, "exact_tiled_attention_20_gb300", "csrc")
    prefixes = KERNEL_SOURCES.get(kernel, ("",))
    return [n for n in sorted(os.listdir(csrc)) if n in SHARED_SOURCES or n.startswith(prefixes)]


def _code_only(text: str) -> str:
    """C/CUDA source with comments removed and whitespace collapsed (string literals, such
    as inline PTX, are kept), so that the hash follows the code and not its comments."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_20_gb300", "csrc")
    for name in kernel_source_files(kernel):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
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
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("bytes_per_launch")


def parse_clock_csv(lines, load_watts=300.0):
    """Summary of nvidia-smi samples (index, sm MHz, max sm MHz, power W, active mask,
    hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap).  Clocks and the
    power-cap share are taken over the samples under load (power above ``load_watts``),
    or over all samples when none is; a throttle reason is listed if any sample shows it."""
    rows, reasons = [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    smax = None
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm, mx = float(parts[1]), float(parts[2])
        except ValueError:
            continue
        try:
            pw = float(parts[3])
        except ValueError:
            pw = 0.0
        smax = mx
        act = [v.lower().startswith("active") for v in parts[5:9]]
        for n, a in zip(names, act):
            if a:
                reasons.add(n)
        rows.append((sm, pw, act[3]))
    if not rows:
        return None
    loaded = [r for r in rows if r[1] >= load_watts] or rows
    return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": smax,
            "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
            "power_cap_frac": round(sum(1 for r in loaded if r[2]) / len(loaded), 3),
            "power_w_max": max(r[1] for r in rows)}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while a timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, tag: str = ""):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_bench_clocks_{os.getpid()}{tag}.csv")

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
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return parse_clock_csv(lines)


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


def decode_bytes(wd, lens, sq: int = 1) -> float:
    """Algorithmic HBM bytes of one decode: valid K/V rows, Q, O and LSE (Sq tokens)."""
    kv = sum(int(n) for n in lens) * wd.Hkv * wd.D * 2 * 2
    return float(kv + sq * (wd.B * wd.Hq * wd.D * 2 * 2 + wd.B * wd.Hq * 4))


# --------------------------------------------------------------- native arm ----

def run_native(args, rank, local_rank, world):
    import torch

    import exact_tiled_attention_20_gb300 as fa
    from exact_tiled_attention_20_gb300 import build

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    build.build_library()
    fa.load()
    num_sms = torch.cuda.get_device_properties(device).multi_processor_count
    peaks, peak_src = load_peaks()
    if args.configs_only:
        if rank == 0:
            res = sweep_configs(args, fa, device, peaks, peak_src, num_sms)
            print(json.dumps({"metric": METRIC, "configs": res["configs"],
                              "configs_clocks": res["clocks"]}), flush=True)
        return
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

    fwd_tflops = fwd_flops / (fwd_ms * 1e-3) / 1e12
    roof = tensor_roofline(fwd_tflops, peaks, peak_src, clocks, num_sms)
    dbytes = decode_bytes(wd, host["lens"].tolist())
    dec_gbs = dbytes / (dec_ms * 1e-3) / 1e9
    peak_h = float(peaks["hbm_gbs"])
    fwd_traffic = ncu_traffic("fa_fwd_kernel")
    dec_traffic = ncu_traffic("fa_decode_split_kernel")

    # Host time of one decode call through the public API (argument checks, cached tensor
    # maps, two launches), measured over back-to-back calls that only enqueue work.
    n_host = 200
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    for _ in range(n_host):
        fa.fa_decode_splitkv(d["dq"], d["dk"], d["dv"], d["lens"], scale=wd.scale,
                             num_splits=ns, workspace=ws, out=d["do"], lse=d["dlse"],
                             stream=stream)
    decode_host_us = (time.perf_counter() - h0) / n_host * 1e6
    torch.cuda.synchronize()

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
        del bufs, d2, pin, outs, ws2
    del d
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wf, wd, host, dbytes)
    del host

    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        configs = sweep_configs(args, fa, device, peaks, peak_src, num_sms)

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
        "pct_of_tensor_peak": round(100.0 * roof["frac"], 1),
        "roofline": dict(kernel="fa_fwd_kernel", **roof, traffic=fwd_traffic,
                         ms_per_launch=round(fwd_ms, 4)),
        "decode": {
            "value": round(dec_gbs, 1),
            "unit": "GB/s",
            "ms_per_launch": round(dec_ms, 4),
            "algorithmic_bytes": int(dbytes),
            "host_us_per_call": round(decode_host_us, 2),
            "roofline": {
                "kernel": "fa_decode_split_kernel + fa_decode_combine_kernel",
                "bound": "hbm",
                "achieved": round(dec_gbs, 1),
                "peak": peak_h,
                "peak_kind": f"{peak_src} copy bandwidth",
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
    if configs is not None:
        out["configs"] = configs["configs"]
        out["configs_clocks"] = configs["clocks"]
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------- CPU baseline ----

def _sample_rows(wf, n_rows, seed=7):
    import numpy as np

    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, wf.B, n_rows), rng.integers(0, wf.Hq, n_rows),
                     rng.integers(0, wf.Sq, n_rows)], axis=1)
    return rows.astype(np.int64)


def visible_keys(i, Sq, Sk, causal, window=(-1, -1)):
    """Number of keys query i sees: bottom-right causal, optional sliding window."""
    off = Sk - Sq
    hi = Sk - 1
    if causal:
        hi = min(hi, i + off)
    if window[1] >= 0:
        hi = min(hi, i + off + window[1])
    lo = 0 if window[0] < 0 else max(0, i + off - window[0])
    return max(0, hi - lo + 1)


def _row_flops(wf, rows, window=(-1, -1)) -> float:
    """Two GEMMs' FLOPs of the given (b, h, i) rows, counting the keys each row sees."""
    if not wf.causal and window == (-1, -1):
        return 4.0 * wf.Sk * wf.D * len(rows)
    return float(sum(4.0 * wf.D * visible_keys(int(i), wf.Sq, wf.Sk, wf.causal, window)
                     for i in rows[:, 2]))


def cpu_baseline(wf, wd, host, dbytes, target_s: float = 8.0):
    """The oracle (fp64, as it stands) on a bounded random sample of output rows of the
    forward workload, and on the whole decode workload, on all host cores; reported in the
    units of the GPU numbers."""
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
    t = time.perf_counter()
    oracle.decode(host["dq"], host["dk"], host["dv"], host["lens"].numpy(), scale=wd.scale,
                  nthreads=cores)
    ddt = time.perf_counter() - t
    return {"value": round(_row_flops(wf, rows) / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": cores, "kind": "oracle",
            "sample": (f"{n} random output rows (all {wf.Sk} keys each) of the fa_fwd workload, "
                       f"fp64, {dt:.1f} s wall"),
            "decode": {"value": round(dbytes / ddt / 1e9, 4), "unit": "GB/s", "cores": cores,
                       "kind": "oracle", "seconds": round(ddt, 3),
                       "sample": "the whole decode workload (every sequence and head), fp64"}}


# ------------------------------------------------------ per-workload sweep ----

class L2Flush:
    """Writes one buffer larger than L2, then reads another, so that the next launch
    starts with none of its data in L2 and no dirty lines left to write back."""

    def __init__(self, device, mib=256):
        import torch

        n = (mib << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.zeros(n, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.fill_(1.0)
        self.r.sum()


def time_launches(fn, reps, warmup, flush):
    """Median, min and max CUDA-event time (ms) of ``fn`` over ``reps`` launches, each
    after an L2 flush that stays outside its event pair."""
    import torch

    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for e0, e1 in ev:
        flush()
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    ms = sorted(e0.elapsed_time(e1) for e0, e1 in ev)
    return statistics.median(ms), ms[0], ms[-1]


def _parity(o_gpu, lse_gpu, o_ref, lse_ref):
    import numpy as np

    o_gpu = np.asarray(o_gpu, dtype=np.float64).reshape(o_ref.shape)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64).reshape(lse_ref.shape)
    fin = np.isfinite(lse_ref)
    same_inf = bool(np.array_equal(fin, np.isfinite(lse_gpu)))
    do = float(np.abs(o_gpu - o_ref).max()) if o_ref.size else 0.0
    dl = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    return {"max_abs_dO": do, "max_abs_dLSE": dl,
            "pass": bool(do <= O_TOL and dl <= LSE_TOL and same_inf),
            "tolerance": {"O": O_TOL, "LSE": LSE_TOL}}


def _fwd_sample_rows(w, budget_flops, window=(-1, -1), seed=11):
    """Rows (b, h, i) the oracle checks for a forward workload: every row when the
    whole output fits the budget, else every row of head (B - 1, Hq - 1) plus random rows
    up to the budget."""
    import numpy as np

    per_row = 4.0 * w.D * (w.Sk if not w.causal and window == (-1, -1) else max(1, w.Sk // 2))
    total = per_row * w.B * w.Hq * w.Sq
    if total <= budget_flops:
        bb, hh, ii = np.meshgrid(np.arange(w.B), np.arange(w.Hq), np.arange(w.Sq), indexing="ij")
        return np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1).astype(np.int64), "all rows"
    head = np.stack([np.full(w.Sq, w.B - 1), np.full(w.Sq, w.Hq - 1), np.arange(w.Sq)], axis=1)
    n_rand = int(max(0.0, budget_flops - per_row * w.Sq) / per_row)
    n_rand = min(max(n_rand, 32), 4096)
    rng = np.random.default_rng(seed)
    rnd = np.stack([rng.integers(0, w.B, n_rand), rng.integers(0, w.Hq, n_rand),
                    rng.integers(0, w.Sq, n_rand)], axis=1)
    return (np.concatenate([head, rnd]).astype(np.int64),
            f"every row of head (b={w.B - 1}, h={w.Hq - 1}) + {n_rand} random rows")


def sweep_configs(args, fa, device, peaks, peak_src, num_sms):
    """Every workload on its own, with its roofline fraction and the oracle beside it."""
    import numpy as np
    import torch

    import oracle
    from exact_tiled_attention_20_gb300 import inputs

    cores = os.cpu_count() or 1
    flush = L2Flush(device)
    peak_h = float(peaks["hbm_gbs"])
    reps, warm = args.config_reps, 5
    # oracle throughput on this host, to size each parity sample to the time budget
    w0 = inputs.PREFILL_MID[0]
    q0, k0, v0 = inputs.make_qkv(1, 256, 1024, 4, 4, 128, seed=1)
    t = time.perf_counter()
    oracle.fwd(q0, k0, v0, scale=0.1, rows=np.array([[0, h, i] for h in range(4) for i in range(256)]),
               nthreads=cores)
    rate = 4.0 * 1024 * 128 * 1024 / max(time.perf_counter() - t, 1e-4)
    budget = rate * args.oracle_budget_s
    del q0, k0, v0, w0
    out = []
    sampler = ClockSampler(device.index or 0, tag="_sweep")
    sampler.start()

    def fwd_entry(name, entry, w, qkv, window=(-1, -1), shape=None):
        qh, kh, vh = qkv
        qd, kd, vd = qh.to(device), kh.to(device), vh.to(device)
        od = torch.empty_like(qd)
        ld = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=device)
        win = None if window == (-1, -1) else window
        call = lambda: fa.fa_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, out=od, lse=ld,  # noqa: E731
                                 window=win)
        med, lo, hi = time_launches(call, reps, warm, flush)
        if window == (-1, -1):
            flops = w.flops()
        else:
            flops = 4.0 * w.D * w.B * w.Hq * sum(visible_keys(i, w.Sq, w.Sk, w.causal, window)
                                                  for i in range(w.Sq))
        call()
        torch.cuda.synchronize()
        rows, how = _fwd_sample_rows(w, budget, window)
        t0 = time.perf_counter()
        o_ref, lse_ref = oracle.fwd(qh, kh, vh, scale=w.scale, causal=w.causal, rows=rows,
                                    nthreads=cores, window=window)
        odt = time.perf_counter() - t0
        b, h, i = (torch.as_tensor(rows[:, c], device=device) for c in range(3))
        par = _parity(od[b, i, h].float().cpu().numpy(), ld[b, h, i].cpu().numpy(), o_ref, lse_ref)
        rf = _row_flops(w, rows, window)
        achieved = flops / (med * 1e-3) / 1e12
        e = {"name": name, "entry": entry,
             "shape": shape or f"[{w.B},{w.Sq},{w.Hq},{w.D}] Hkv={w.Hkv} "
                               f"{'causal' if w.causal else 'non-causal'}",
             "ms": round(med, 4), "ms_min": round(lo, 4), "ms_max": round(hi, 4), "reps": reps,
             "flops": flops, "value": round(achieved, 1), "unit": "TFLOP/s",
             "oracle": {"seconds": round(odt, 3), "value": round(rf / odt / 1e12, 6),
                        "unit": "TFLOP/s", "cores": cores, "sample": f"{len(rows)} rows: {how}"},
             "parity": dict(par, rows=int(len(rows)))}
        del qd, kd, vd, od, ld
        return e, achieved

    # -- forward workloads of the pages' table, the long shape both ways, the GQA sweep
    fwd_list = ([("tiny", w) for w in inputs.TINY] + [("prefill_mid", w) for w in inputs.PREFILL_MID]
                + [("prefill_long", w) for w in inputs.PREFILL_LONG]
                + [("gqa_sweep", w) for w in inputs.GQA_SWEEP])
    cache = {}
    for group, w in fwd_list:
        key = (w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D, w.amp, w.seed)
        if key not in cache:
            cache.clear()
            cache[key] = inputs.fwd_inputs(w)
        name = f"{w.name}{'_causal' if w.causal else ''}"
        e, ach = fwd_entry(name, "fa_fwd", w, cache[key])
        e["group"] = group
        out.append((e, "tensor", ach))
        torch.cuda.empty_cache()

    # -- sliding window on the long causal shape (reuses its inputs)
    wl = inputs.PREFILL_LONG[1]
    key = (wl.B, wl.Sq, wl.Sk, wl.Hq, wl.Hkv, wl.D, wl.amp, wl.seed)
    if key not in cache:
        cache.clear()
        cache[key] = inputs.fwd_inputs(wl)
    qh, kh, vh = cache[key]
    win = (inputs.WINDOW_LEFT, 0)
    e, ach = fwd_entry("sliding_window", "fa_fwd_window", wl, (qh, kh, vh), window=win,
                       shape=f"[16,8192,32,128] causal, window ({win[0]}, {win[1]})")
    e["group"] = "widened"
    e["flops_note"] = "visible (query, key) pairs x 4 x D x Hq x B"
    out.append((e, "tensor", ach))

    # -- variable-length batch: 16 causal sequences packed from the long shape's rows
    lens = inputs.varlen_lengths()
    tq = sum(lens)
    qv, kv_, vv = (t.reshape(-1, t.shape[2], t.shape[3])[:tq] for t in (qh, kh, vh))
    cu_h = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    qd, kd, vd, cud = qv.to(device), kv_.to(device), vv.to(device), cu_h.to(device)
    od = torch.empty_like(qd)
    ld = torch.empty((wl.Hq, tq), dtype=torch.float32, device=device)
    call = lambda: fa.fa_fwd_varlen(qd, kd, vd, cud, cud, causal=True, out=od, lse=ld)  # noqa: E731
    med, lo, hi = time_launches(call, reps, warm, flush)
    pairs = sum(n * (n + 1) // 2 for n in lens)
    flops = 4.0 * wl.D * pairs * wl.Hq
    call()
    torch.cuda.synchronize()
    # parity sample: every row of the last head of the shortest and of the longest sequence
    pick = sorted({int(np.argmin(lens)), int(np.argmax(lens))})
    o_g, l_g, o_r, l_r, nrows, rf, odt = [], [], [], [], 0, 0.0, 0.0
    for bsel in pick:
        a0, a1 = int(cu_h[bsel]), int(cu_h[bsel + 1])
        n = a1 - a0
        rows = np.stack([np.zeros(n), np.full(n, wl.Hq - 1), np.arange(n)], axis=1).astype(np.int64)
        t0 = time.perf_counter()
        orf, lrf = oracle.fwd(qv[None, a0:a1], kv_[None, a0:a1], vv[None, a0:a1], scale=wl.scale,
                              causal=True, rows=rows, nthreads=cores)
        odt += time.perf_counter() - t0
        o_g.append(od[a0:a1, wl.Hq - 1].float().cpu().numpy())
        l_g.append(ld[wl.Hq - 1, a0:a1].cpu().numpy())
        o_r.append(orf)
        l_r.append(lrf)
        nrows += n
        rf += 4.0 * wl.D * n * (n + 1) / 2
    par = _parity(np.concatenate(o_g), np.concatenate(l_g), np.concatenate(o_r), np.concatenate(l_r))
    ach = flops / (med * 1e-3) / 1e12
    out.append(({"name": "varlen", "group": "widened", "entry": "fa_fwd_varlen",
                 "shape": f"16 causal sequences U[256,8192] (total {tq} rows), Hq=Hkv=32, D=128",
                 "ms": round(med, 4), "ms_min": round(lo, 4), "ms_max": round(hi, 4), "reps": reps,
                 "flops": flops, "flops_note": "visible (query, key) pairs x 4 x D x Hq",
                 "value": round(ach, 1), "unit": "TFLOP/s",
                 "oracle": {"seconds": round(odt, 3), "value": round(rf / odt / 1e12, 6),
                            "unit": "TFLOP/s", "cores": cores,
                            "sample": f"{nrows} rows: every row of head {wl.Hq - 1} of sequences {pick}"},
                 "parity": dict(par, rows=nrows)}, "tensor", ach))
    del qd, kd, vd, cud, od, ld, qv, kv_, vv, qh, kh, vh
    cache.clear()
    torch.cuda.empty_cache()

    # -- decode workloads: contiguous, paged, several tokens; every output checked
    wd = inputs.DECODE
    dq, dk, dv, dl = inputs.decode_inputs(wd)
    lens_l = dl.tolist()
    nbytes = decode_bytes(wd, lens_l)
    ns = fa.fa_decode_default_splits(wd.B, wd.Hkv, wd.Smax)

    def dec_entry(name, entry, call, o_dev, l_dev, oracle_call, nb, shape, bytes_note=None):
        med, lo, hi = time_launches(call, reps, warm, flush)
        call()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        o_ref, lse_ref = oracle_call()
        odt = time.perf_counter() - t0
        par = _parity(o_dev.float().cpu().numpy(), l_dev.cpu().numpy(), o_ref, lse_ref)
        gbs = nb / (med * 1e-3) / 1e9
        e = {"name": name, "group": "decode" if entry == "fa_decode_splitkv" else "widened",
             "entry": entry, "shape": shape, "ms": round(med, 4), "ms_min": round(lo, 4),
             "ms_max": round(hi, 4), "reps": reps, "algorithmic_bytes": int(nb),
             "value": round(gbs, 1), "unit": "GB/s",
             "oracle": {"seconds": round(odt, 3), "value": round(nb / odt / 1e9, 4), "unit": "GB/s",
                        "cores": cores, "sample": "every output (whole workload)"},
             "parity": dict(par, rows=int(o_ref.size // o_ref.shape[-1]))}
        if bytes_note:
            e["bytes_note"] = bytes_note
        return e, gbs

    q_d, k_d, v_d, l_d = (t.to(device) for t in (dq, dk, dv, dl))
    ws = torch.empty(fa.fa_decode_workspace_bytes(wd.B * 4, wd.Hq, wd.D, ns), dtype=torch.uint8,
                     device=device)
    o_d = torch.empty_like(q_d)
    lse_d = torch.empty((wd.B, wd.Hq), dtype=torch.float32, device=device)
    e, gbs = dec_entry(
        "decode", "fa_decode_splitkv",
        lambda: fa.fa_decode_splitkv(q_d, k_d, v_d, l_d, scale=wd.scale, num_splits=ns, workspace=ws,
                                     out=o_d, lse=lse_d),
        o_d, lse_d, lambda: oracle.decode(dq, dk, dv, lens_l, scale=wd.scale, nthreads=cores), nbytes,
        f"B=8, Hq=32, Hkv=8, D=128, kv_len~U[1024,32768] (sum {sum(lens_l)}), Smax=32768, "
        f"num_splits={ns}")
    out.append((e, "hbm", gbs))
    q4 = inputs.decode_multi_queries(wd, sq=4)
    q4_d = q4.to(device)
    o4 = torch.empty_like(q4_d)
    l4 = torch.empty((wd.B, wd.Hq, 4), dtype=torch.float32, device=device)
    e, gbs = dec_entry(
        "multi_token_decode", "fa_decode_splitkv_multi",
        lambda: fa.fa_decode_splitkv_multi(q4_d, k_d, v_d, l_d, causal=True, scale=wd.scale,
                                           num_splits=ns, workspace=ws, out=o4, lse=l4),
        o4, l4, lambda: oracle.decode_multi(q4, dk, dv, lens_l, scale=wd.scale, causal=True,
                                            nthreads=cores),
        decode_bytes(wd, lens_l, sq=4), "decode workload with 4 causal query tokens per sequence")
    out.append((e, "hbm", gbs))
    del k_d, v_d, q4_d, o4, l4
    torch.cuda.empty_cache()
    kp, vp, table = inputs.paged_layout(dk, dv, page=256)
    kp_d, vp_d, tb_d = kp.to(device), vp.to(device), table.to(device)
    e, gbs = dec_entry(
        "paged_decode", "fa_decode_splitkv_paged",
        lambda: fa.fa_decode_splitkv_paged(q_d, kp_d, vp_d, tb_d, l_d, scale=wd.scale, num_splits=ns,
                                           workspace=ws, out=o_d, lse=lse_d),
        o_d, lse_d, lambda: oracle.decode_paged(dq, kp, vp, table, lens_l, scale=wd.scale,
                                                nthreads=cores), nbytes,
        "decode workload in 256-key pages of a pool, pages in a seeded random order")
    out.append((e, "hbm", gbs))
    del kp_d, vp_d, tb_d, kp, vp, q_d, l_d, o_d, lse_d, ws
    torch.cuda.empty_cache()

    # -- the decode workload's shape and lengths at the other head dims
    for wdd in inputs.DECODE_D_SWEEP:
        dq, dk, dv, dl = inputs.decode_inputs(wdd)
        lens_l = dl.tolist()
        ns = fa.fa_decode_default_splits(wdd.B, wdd.Hkv, wdd.Smax)
        q_d, k_d, v_d, l_d = (t.to(device) for t in (dq, dk, dv, dl))
        ws = torch.empty(fa.fa_decode_workspace_bytes(wdd.B, wdd.Hq, wdd.D, ns), dtype=torch.uint8,
                         device=device)
        o_d = torch.empty_like(q_d)
        lse_d = torch.empty((wdd.B, wdd.Hq), dtype=torch.float32, device=device)
        e, gbs = dec_entry(
            f"decode_d{wdd.D}", "fa_decode_splitkv",
            lambda: fa.fa_decode_splitkv(q_d, k_d, v_d, l_d, scale=wdd.scale, num_splits=ns,
                                         workspace=ws, out=o_d, lse=lse_d),
            o_d, lse_d, lambda: oracle.decode(dq, dk, dv, lens_l, scale=wdd.scale, nthreads=cores),
            decode_bytes(wdd, lens_l),
            f"B=8, Hq=32, Hkv=8, D={wdd.D}, the decode workload's lengths, Smax=32768, "
            f"num_splits={ns}")
        out.append((e, "hbm", gbs))
        del q_d, k_d, v_d, l_d, ws, o_d, lse_d, dq, dk, dv
        torch.cuda.empty_cache()

    clocks = sampler.stop()
    if fa.fa_last_device_status() != 0:
        raise RuntimeError("device status reported a kernel timeout during the per-workload runs")
    entries = []
    for e, bound, ach in out:
        if bound == "tensor":
            e["roofline"] = tensor_roofline(ach, peaks, peak_src, clocks, num_sms)
        else:
            e["roofline"] = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak_h,
                             "peak_kind": f"{peak_src} copy bandwidth", "unit": "GB/s",
                             "frac": round(ach / peak_h, 4)}
        entries.append(e)
    return {"configs": entries, "clocks": clocks}


# ----------------------------------------------------------- reference arm ----

def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded sample of output rows
    of the same forward workload, timed on the host cores."""
    if rank != 0:
        return
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


# ------------------------------------------------------------ single case ----

def run_case(argv):
    """One kernel a few times on device-resident inputs (values drawn on the device from a
    fixed seed; they do not matter for profiling); prints the mean time per call."""
    import numpy as np
    import torch

    import exact_tiled_attention_20_gb300 as fa
    from exact_tiled_attention_20_gb300 import build, inputs

    if not argv:
        raise SystemExit("bench.py --case needs a kind:\n" + CASES)
    build.build_library()
    fa.load()
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(0)

    def rnd(*shape):
        return torch.randn(*shape, device=dev, generator=g, dtype=torch.bfloat16)

    kind, rest = argv[0], argv[1:]
    if kind in ("fwd", "fwd_window"):
        n = 6 if kind == "fwd" else 7
        vals = [int(x) for x in rest[:n]]
        iters = int(rest[n]) if len(rest) > n else 3
        B, S, Hq, Hkv, D = vals[:5]
        q, k, v = rnd(B, S, Hq, D), rnd(B, S, Hkv, D), rnd(B, S, Hkv, D)
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, S, device=dev, dtype=torch.float32)
        if kind == "fwd":
            call = lambda: fa.fa_fwd(q, k, v, causal=bool(vals[5]), out=o, lse=lse)  # noqa: E731
        else:
            call = lambda: fa.fa_fwd(q, k, v, window=(vals[5], vals[6]), out=o, lse=lse)  # noqa: E731
    elif kind == "fwd_varlen_workload":
        iters = int(rest[0]) if rest else 3
        lens = inputs.varlen_lengths()
        tq = sum(lens)
        q, k, v = rnd(tq, 32, 128), rnd(tq, 32, 128), rnd(tq, 32, 128)
        cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(32, tq, device=dev, dtype=torch.float32)
        call = lambda: fa.fa_fwd_varlen(q, k, v, cu, cu, causal=True, out=o, lse=lse)  # noqa: E731
    elif kind == "decode":
        B, Hq, Hkv, D, Smax = (int(x) for x in rest[:5])
        iters = int(rest[5]) if len(rest) > 5 else 3
        q, kc, vc = rnd(B, 1, Hq, D), rnd(B, Smax, Hkv, D), rnd(B, Smax, Hkv, D)
        lens = torch.randint(Smax // 32, Smax + 1, (B,), device=dev, generator=g, dtype=torch.int32)
        ns = fa.fa_decode_default_splits(B, Hkv, Smax)
        ws = torch.empty(fa.fa_decode_workspace_bytes(B, Hq, D, ns), dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        call = lambda: fa.fa_decode_splitkv(q, kc, vc, lens, num_splits=ns, workspace=ws, out=o)  # noqa: E731
    elif kind in ("decode_workload", "decode_paged_workload"):
        iters = int(rest[0]) if rest else 3
        d = int(rest[1]) if kind == "decode_workload" and len(rest) > 1 else inputs.DECODE.D
        w = next((x for x in [inputs.DECODE] + inputs.DECODE_D_SWEEP if x.D == d), None)
        if w is None:
            raise SystemExit(f"no decode workload at head dim {d}")
        qh, kh, vh, lh = inputs.decode_inputs(w)
        ns = fa.fa_decode_default_splits(w.B, w.Hkv, w.Smax)
        ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.Hq, w.D, ns), dtype=torch.uint8, device=dev)
        q, lens = qh.to(dev), lh.to(dev)
        o = torch.empty_like(q)
        if kind == "decode_workload":
            kc, vc = kh.to(dev), vh.to(dev)
            call = lambda: fa.fa_decode_splitkv(q, kc, vc, lens, num_splits=ns, workspace=ws, out=o)  # noqa: E731
        else:
            kp, vp, table = (t.to(dev) for t in inputs.paged_layout(kh, vh, page=256))
            call = lambda: fa.fa_decode_splitkv_paged(q, kp, vp, table, lens, num_splits=ns,  # noqa: E731
                                                      workspace=ws, out=o)
    else:
        raise SystemExit(f"unknown case {kind!r}; kinds:\n" + CASES)
    call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        call()
    e1.record()
    torch.cuda.synchronize()
    st = fa.fa_last_device_status()
    print(f"{kind} {' '.join(rest)}: {e0.elapsed_time(e1) / iters:.4f} ms/call, status {st}")
    if st != 0:
        raise SystemExit(1)


def main(argv=None):
    args = parse_args(argv)
    rank, local_rank, world = dist_env()
    if args.case is not None:
        if rank == 0:
            run_case(args.case)
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
