"""Runs one forward or decode case a few times -- a small, self-contained driver for
profiling a single kernel (e.g. under ncu) on inputs resident on the GPU.

  python -m exact_tiled_attention_20_gb300.run_case fwd B S Hq Hkv D causal [iters]
  python -m exact_tiled_attention_20_gb300.run_case fwd_window B S Hq Hkv D left right [iters]
  python -m exact_tiled_attention_20_gb300.run_case fwd_varlen_workload [iters]
  python -m exact_tiled_attention_20_gb300.run_case decode B Hq Hkv D Smax [iters]
  python -m exact_tiled_attention_20_gb300.run_case decode_workload [iters]
  python -m exact_tiled_attention_20_gb300.run_case decode_paged_workload [iters]

Inputs are drawn on the device from a fixed seed (values do not matter for profiling);
the script prints the mean time per call from CUDA events.
"""
from __future__ import annotations

import sys

import torch

from . import _lib as fa
from . import build


def main(argv):
    build.build_library()
    fa.load()
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev).manual_seed(0)
    kind = argv[0]
    if kind == "fwd":
        B, S, Hq, Hkv, D, causal = (int(x) for x in argv[1:7])
        iters = int(argv[7]) if len(argv) > 7 else 3
        q = torch.randn(B, S, Hq, D, device=dev, generator=g, dtype=torch.bfloat16)
        k = torch.randn(B, S, Hkv, D, device=dev, generator=g, dtype=torch.bfloat16)
        v = torch.randn(B, S, Hkv, D, device=dev, generator=g, dtype=torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, S, device=dev, dtype=torch.float32)
        call = lambda: fa.fa_fwd(q, k, v, causal=bool(causal), out=o, lse=lse)  # noqa: E731
    elif kind == "fwd_window":
        B, S, Hq, Hkv, D, left, right = (int(x) for x in argv[1:8])
        iters = int(argv[8]) if len(argv) > 8 else 3
        q = torch.randn(B, S, Hq, D, device=dev, generator=g, dtype=torch.bfloat16)
        k = torch.randn(B, S, Hkv, D, device=dev, generator=g, dtype=torch.bfloat16)
        v = torch.randn(B, S, Hkv, D, device=dev, generator=g, dtype=torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, S, device=dev, dtype=torch.float32)
        call = lambda: fa.fa_fwd(q, k, v, window=(left, right), out=o, lse=lse)  # noqa: E731
    elif kind == "fwd_varlen_workload":
        # 16 causal sequences of U[256, 8192] rows (seed 1005), Hq = Hkv = 32, D = 128, packed
        import numpy as np

        iters = int(argv[1]) if len(argv) > 1 else 3
        lens = [int(x) for x in np.random.default_rng(1005).integers(256, 8193, 16)]
        tq = sum(lens)
        q = torch.randn(tq, 32, 128, device=dev, generator=g, dtype=torch.bfloat16)
        k = torch.randn(tq, 32, 128, device=dev, generator=g, dtype=torch.bfloat16)
        v = torch.randn(tq, 32, 128, device=dev, generator=g, dtype=torch.bfloat16)
        cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(32, tq, device=dev, dtype=torch.float32)
        call = lambda: fa.fa_fwd_varlen(q, k, v, cu, cu, causal=True, out=o, lse=lse)  # noqa: E731
    elif kind == "decode":
        B, Hq, Hkv, D, Smax = (int(x) for x in argv[1:6])
        iters = int(argv[6]) if len(argv) > 6 else 3
        q = torch.randn(B, 1, Hq, D, device=dev, generator=g, dtype=torch.bfloat16)
        kc = torch.randn(B, Smax, Hkv, D, device=dev, generator=g, dtype=torch.bfloat16)
        vc = torch.randn(B, Smax, Hkv, D, device=dev, generator=g, dtype=torch.bfloat16)
        lens = torch.randint(Smax // 32, Smax + 1, (B,), device=dev, generator=g, dtype=torch.int32)
        ns = fa.fa_decode_default_splits(B, Hkv, Smax)
        ws = torch.empty(fa.fa_decode_workspace_bytes(B, Hq, D, ns), dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        call = lambda: fa.fa_decode_splitkv(q, kc, vc, lens, num_splits=ns, workspace=ws, out=o)  # noqa: E731
    elif kind == "decode_workload":
        # the benchmark's decode workload, same seeded inputs and default split count
        from . import inputs

        w = inputs.DECODE
        iters = int(argv[1]) if len(argv) > 1 else 3
        q, kc, vc, lens = (t.to(dev) for t in inputs.decode_inputs(w))
        ns = fa.fa_decode_default_splits(w.B, w.Hkv, w.Smax)
        ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.Hq, w.D, ns), dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        call = lambda: fa.fa_decode_splitkv(q, kc, vc, lens, num_splits=ns, workspace=ws, out=o)  # noqa: E731
    elif kind == "decode_paged_workload":
        # the same workload in 256-key pages of a pool, the pages in a seeded random order
        from . import inputs

        w = inputs.DECODE
        iters = int(argv[1]) if len(argv) > 1 else 3
        q, kc, vc, lens = inputs.decode_inputs(w)
        page = 256
        mp = w.Smax // page
        perm = torch.randperm(w.B * mp, generator=torch.Generator().manual_seed(7))
        table = perm.view(w.B, mp).to(torch.int32)
        kp = torch.empty((w.B * mp, page, w.Hkv, w.D), dtype=kc.dtype)
        vp = torch.empty_like(kp)
        kp[perm] = kc.view(w.B * mp, page, w.Hkv, w.D)
        vp[perm] = vc.view(w.B * mp, page, w.Hkv, w.D)
        q, kp, vp, table, lens = (t.to(dev) for t in (q, kp, vp, table, lens))
        o = torch.empty_like(q)
        call = lambda: fa.fa_decode_splitkv_paged(q, kp, vp, table, lens, out=o)  # noqa: E731
    else:
        raise SystemExit(__doc__)
    call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        call()
    e1.record()
    torch.cuda.synchronize()
    st = fa.fa_last_device_status()
    print(f"{kind} {' '.join(argv[1:])}: {e0.elapsed_time(e1) / iters:.4f} ms/call, status {st}")
    if st != 0:
        raise SystemExit(1)


if __name__ == "__main__":
    main(sys.argv[1:])
