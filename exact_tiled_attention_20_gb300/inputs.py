"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no attention arithmetic: it draws Q/K/V (and per-sequence KV lengths)
from a seeded CPU generator, so that the CUDA path and the oracle read the very same
16-bit values.  Recipe, fixed for every workload:

* ``g = torch.Generator("cpu").manual_seed(seed)``;
* decode workloads first draw ``kv_lens = torch.randint(lo, hi + 1, (B,), generator=g)``;
* then Q, K, V in that order, each ``torch.randn(shape, generator=g, dtype=float32)``,
  multiplied by the workload's ``amp`` (1.0, or 0.5 for the grouped-query sweep), and
  rounded once to bf16/fp16.

The named workloads carry the shapes of the pages' benchmarks ([batch, seq_len,
num_heads, head_dim] = [16, 1k..8k, 32, 128], page "ampere_flash_attention_from_scratch",
section "Performance Test") and of the decode setting the pages describe (one query
token over long per-sequence KV caches, page "flash-attention-v100", "Changelog",
"2.2: Optimize for inference").  No dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math

import torch

_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass(frozen=True)
class FwdWorkload:
    name: str
    B: int
    Sq: int
    Sk: int
    Hq: int
    Hkv: int
    D: int
    causal: bool
    amp: float = 1.0
    dtype: str = "bf16"
    seed: int = 1000

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def flops(self) -> float:
        """Two GEMMs, 4*B*Hq*Sq*Sk*D, halved when causal."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.D
        return f / 2 if self.causal else f


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    Smax: int
    len_lo: int
    len_hi: int
    amp: float = 1.0
    dtype: str = "bf16"
    seed: int = 1004

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The workloads: a tiny case the oracle finishes at once, the prefill shapes of the
# pages' benchmark table, a grouped-query head-dim sweep and single-token decode.
TINY = [FwdWorkload("tiny", 1, 128, 128, 2, 2, 64, c, seed=1000) for c in (False, True)]
PREFILL_MID = [FwdWorkload(f"prefill_mid_s{s}", 16, s, s, 32, 32, 128, False, seed=1001)
               for s in (1024, 2048, 4096)]
PREFILL_LONG = [FwdWorkload("prefill_long_s8192", 16, 8192, 8192, 32, 32, 128, c, seed=1002)
                for c in (False, True)]
GQA_SWEEP = [FwdWorkload(f"gqa_d{d}", 4, 4096, 4096, 32, 8, d, True, amp=0.5, seed=1003)
             for d in (64, 96, 128, 256)]
DECODE = DecodeWorkload("decode_splitkv", 8, 32, 8, 128, 32768, 1024, 32768, seed=1004)
# The decode workload at the other head dims (same seed, so the same KV lengths).
DECODE_D_SWEEP = [DecodeWorkload(f"decode_splitkv_d{d}", 8, 32, 8, d, 32768, 1024, 32768, seed=1004)
                  for d in (64, 96, 256)]


def fwd_inputs(w: FwdWorkload):
    """(q, k, v) CPU tensors in the workload's dtype: q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D]."""
    return make_qkv(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D, seed=w.seed, amp=w.amp, dtype=w.dtype)


def make_qkv(B, Sq, Sk, Hq, Hkv, D, seed, amp=1.0, dtype="bf16"):
    g = torch.Generator("cpu").manual_seed(int(seed))
    dt = _DTYPES[dtype]
    q = (torch.randn((B, Sq, Hq, D), generator=g, dtype=torch.float32) * amp).to(dt)
    k = (torch.randn((B, Sk, Hkv, D), generator=g, dtype=torch.float32) * amp).to(dt)
    v = (torch.randn((B, Sk, Hkv, D), generator=g, dtype=torch.float32) * amp).to(dt)
    return q, k, v


def decode_inputs(w: DecodeWorkload):
    """(q [B,1,Hq,D], k_cache, v_cache [B,Smax,Hkv,D], kv_lens int32 [B]) on the CPU."""
    return make_decode(w.B, w.Hq, w.Hkv, w.D, w.Smax, w.len_lo, w.len_hi, seed=w.seed,
                       amp=w.amp, dtype=w.dtype)


def make_decode(B, Hq, Hkv, D, Smax, len_lo, len_hi, seed, amp=1.0, dtype="bf16"):
    g = torch.Generator("cpu").manual_seed(int(seed))
    dt = _DTYPES[dtype]
    lens = torch.randint(len_lo, len_hi + 1, (B,), generator=g).to(torch.int32)
    q = (torch.randn((B, 1, Hq, D), generator=g, dtype=torch.float32) * amp).to(dt)
    k = (torch.randn((B, Smax, Hkv, D), generator=g, dtype=torch.float32) * amp).to(dt)
    v = (torch.randn((B, Smax, Hkv, D), generator=g, dtype=torch.float32) * amp).to(dt)
    return q, k, v, lens


# Inputs of the widened rows, measured beside the workloads above.
WINDOW_LEFT = 1023  # sliding window: each query sees itself and the 1023 keys before it


def varlen_lengths(n=16, lo=256, hi=8192, seed=1005):
    """Sequence lengths of the variable-length batch: n draws from U[lo, hi] (numpy
    generator ``default_rng(seed)``), packed in draw order."""
    import numpy as np

    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, n)]


def decode_multi_queries(w: DecodeWorkload, sq=4, seed=12):
    """Query tokens [B, sq, Hq, D] for decoding several tokens over the cache of ``w``:
    ``randn`` from ``Generator("cpu").manual_seed(seed)``, rounded to the workload dtype."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    return (torch.randn((w.B, sq, w.Hq, w.D), generator=g, dtype=torch.float32) * w.amp).to(
        _DTYPES[w.dtype])


def paged_layout(k_cache, v_cache, page=256, seed=7):
    """The same cache stored as a pool of ``page``-key pages in a seeded random order:
    returns (k_pages, v_pages [B * Smax / page, page, Hkv, D], block_table int32
    [B, Smax / page]) with page block_table[b][i] holding keys [i * page, (i + 1) * page)
    of sequence b."""
    B, smax, hkv, d = k_cache.shape
    mp = smax // page
    perm = torch.randperm(B * mp, generator=torch.Generator("cpu").manual_seed(int(seed)))
    kp = torch.empty((B * mp, page, hkv, d), dtype=k_cache.dtype)
    vp = torch.empty_like(kp)
    kp[perm] = k_cache.reshape(B * mp, page, hkv, d)
    vp[perm] = v_cache.reshape(B * mp, page, hkv, d)
    return kp, vp, perm.view(B, mp).to(torch.int32)
