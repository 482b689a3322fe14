"""Low-precision CPU baseline -- TEST INFRASTRUCTURE ONLY.

The pages' test criterion (page "flash-attention-v100", section "Tests") compares the
error of the fast kernel with that of a plain PyTorch implementation: the fast kernel's
maximum error must be at most twice the plain one's.  This module is
that baseline, restated plainly with PyTorch CPU ops: scores accumulated in fp32 from
the stored 16-bit inputs, an fp32 softmax, the probabilities rounded to the input dtype
before the second product, fp32 accumulation, and one rounding of the output to the
input dtype.  Both errors are measured against the fp64 oracle.  Small sizes only.
"""
from __future__ import annotations

import torch


def fwd(q, k, v, scale: float, causal: bool = False):
    """q [B, Sq, Hq, D], k/v [B, Sk, Hkv, D] in bf16/fp16 -> o [B, Sq, Hq, D] (input dtype)."""
    dt = q.dtype
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    qf = q.float().permute(0, 2, 1, 3)                                   # [B, Hq, Sq, D]
    kf = k.float().permute(0, 2, 1, 3).repeat_interleave(g, dim=1)       # [B, Hq, Sk, D]
    vf = v.float().permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    s = torch.matmul(qf, kf.transpose(-1, -2)) * scale                  # fp32 scores
    if causal:
        i = torch.arange(Sq).view(Sq, 1)
        j = torch.arange(Sk).view(1, Sk)
        s = s.masked_fill(j > i + (Sk - Sq), float("-inf"))
    p = torch.softmax(s, dim=-1)
    p = torch.nan_to_num(p, nan=0.0)                                     # all-masked rows -> 0
    o = torch.matmul(p.to(dt).float(), vf)                              # P rounded, fp32 acc
    return o.permute(0, 2, 1, 3).contiguous().to(dt)
