"""GPU parity of fa_fwd against the CPU oracle (fp64).

Bars (the tolerances the attention forward is held to): max|dO| <= 1e-2 and
max|dLSE| <= 1e-3 for N(0,1) bf16 inputs, element by element.  Secondary (page
"flash-attention-v100", section "Tests"): the kernel's max error is at most twice the
max error of a plain low-precision CPU baseline (oracle/lowp.py) on the same inputs.
Shapes span several 128-row/128-key tiles and ragged tails; the edge cases are Sq != Sk
with bottom-right causal alignment (including fully masked rows), a single query or key,
grouped-query heads and every supported head dim.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import lowp
from exact_tiled_attention_20_gb300 import inputs

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_20_gb300 as fa_mod
    from exact_tiled_attention_20_gb300 import build

    build.build_library()
    fa_mod.load()
    return fa_mod


def _run(fa, q, k, v, causal, scale=None):
    dev = torch.device("cuda:0")
    o, lse = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    return o.cpu(), lse.cpu()


def _compare(o, lse, o_ref, lse_ref, base=None):
    o = o.float().numpy()
    lse = lse.numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse)), "LSE -inf pattern differs"
    assert np.all(lse[~fin] == -np.inf)
    do = np.abs(o - o_ref).max() if o.size else 0.0
    dl = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert do <= O_TOL, f"max|dO| = {do:.3e}"
    assert dl <= LSE_TOL, f"max|dLSE| = {dl:.3e}"
    if base is not None:
        berr = np.abs(base.float().numpy() - o_ref).max()
        assert do <= 2 * berr + 1e-6, f"max|dO| {do:.3e} > 2x baseline error {berr:.3e}"
    return do, dl


CASES = [
    # (B, Sq, Sk, Hq, Hkv, D)
    (1, 128, 128, 2, 2, 64),       # the tiny workload
    (2, 300, 300, 4, 2, 128),      # ragged tails over 2+ query blocks, GQA 2
    (1, 513, 513, 2, 1, 64),       # MQA, one key beyond 4 tiles
    (1, 257, 257, 4, 4, 96),
    (1, 200, 333, 2, 2, 256),
    (2, 64, 700, 4, 4, 128),       # Sq < Sk
]


@pytest.mark.parametrize("shape", CASES)
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_matches_oracle(fa, shape, causal):
    B, Sq, Sk, Hq, Hkv, D = shape
    q, k, v = inputs.make_qkv(B, Sq, Sk, Hq, Hkv, D, seed=11 + Sq + D)
    o, lse = _run(fa, q, k, v, causal)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=1 / math.sqrt(D), causal=causal)
    base = lowp.fwd(q, k, v, 1 / math.sqrt(D), causal) if B * Sq * Sk <= 3e5 else None
    _compare(o, lse, o_ref, lse_ref, base)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("sq,sk", [(520, 200), (300, 1), (1, 300), (1, 1), (129, 2)])
def test_fwd_causal_bottom_right_edges(fa, sq, sk, D):
    """Sq > Sk leaves the first Sq - Sk rows with no visible key: O = 0, LSE = -inf.  At
    D = 64 the masked scores go through the FMA-pipe mask, where a row whose scores in a
    block are all masked must still count as having no maximum there."""
    q, k, v = inputs.make_qkv(1, sq, sk, 2, 1, D, seed=3 + sq + sk)
    o, lse = _run(fa, q, k, v, True)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=1 / math.sqrt(D), causal=True)
    _compare(o, lse, o_ref, lse_ref)
    if sq > sk:
        assert torch.all(o[:, : sq - sk] == 0)


@pytest.mark.parametrize("sq,sk", [(2700, 2700), (2700, 3000)])
def test_fwd_causal_paired_walk(fa, sq, sk):
    """Causal batches walk query blocks qb and nqb-1-qb of a head back to back when that
    balances the CTAs better.  This shape (16 heads, 11 query blocks of 256 rows each, the
    last one ragged) takes the paired walk with an odd block count, where the middle
    block has no partner; every row is checked."""
    q, k, v = inputs.make_qkv(2, sq, sk, 8, 2, 128, seed=sq + sk)
    o, lse = _run(fa, q, k, v, True)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=1 / math.sqrt(128), causal=True)
    _compare(o, lse, o_ref, lse_ref)


def test_fwd_fp16(fa):
    q, k, v = inputs.make_qkv(1, 260, 260, 4, 2, 128, seed=21, dtype="fp16")
    for causal in (False, True):
        o, lse = _run(fa, q, k, v, causal)
        o_ref, lse_ref = oracle.fwd(q, k, v, scale=1 / math.sqrt(128), causal=causal)
        _compare(o, lse, o_ref, lse_ref)


def test_fwd_closed_forms(fa):
    """Q = 0 gives the mean of the visible V rows and LSE = ln(count); V = 1 gives 1."""
    B, S, H, D = 1, 384, 2, 128
    _, k, v = inputs.make_qkv(B, S, S, H, H, D, seed=5)
    q = torch.zeros((B, S, H, D), dtype=torch.bfloat16)
    o, lse = _run(fa, q, k, v, True)
    counts = torch.arange(1, S + 1, dtype=torch.float64)
    mean = torch.cumsum(v.double(), dim=1) / counts.view(1, S, 1, 1)
    assert (o.double() - mean).abs().max().item() <= O_TOL
    assert (lse.double() - counts.log().view(1, 1, S)).abs().max().item() <= LSE_TOL
    ones = torch.ones_like(v)
    q2, _, _ = inputs.make_qkv(B, S, S, H, H, D, seed=6)
    o, _ = _run(fa, q2, k, ones, False)
    assert (o.float() - 1).abs().max().item() <= 4e-3


def test_fwd_one_hot_selection(fa):
    """K rows e_j, q_i = e_pi(i) with a large scale: O_i = V_pi(i) (bf16-exact rows)."""
    S, D = 64, 64
    perm = torch.randperm(S, generator=torch.Generator().manual_seed(2))
    k = torch.eye(S, dtype=torch.bfloat16).view(1, S, 1, D)
    q = torch.eye(S, dtype=torch.bfloat16)[perm].view(1, S, 1, D)
    _, _, v = inputs.make_qkv(1, S, S, 1, 1, D, seed=9)
    o, lse = _run(fa, q, k, v, False, scale=100.0)
    assert torch.equal(o[0, :, 0], v[0, perm, 0])
    assert (lse[0, 0] - 100.0).abs().max().item() <= LSE_TOL


def test_fwd_is_deterministic(fa):
    q, k, v = inputs.make_qkv(2, 384, 384, 4, 2, 128, seed=33)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = fa.fa_fwd(qd, kd, vd, causal=True)
    o2, l2 = fa.fa_fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_output_guard_bands(fa):
    """Writes stay inside O and LSE: sentinel pages around them are untouched."""
    B, S, H, D = 1, 200, 2, 128
    q, k, v = inputs.make_qkv(B, S, S, H, H, D, seed=44)
    dev = torch.device("cuda:0")
    pad = 4096
    o_buf = torch.full((pad + B * S * H * D + pad,), 7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((pad + B * H * S + pad,), 7.0, dtype=torch.float32, device=dev)
    o = o_buf[pad:pad + B * S * H * D].view(B, S, H, D)
    lse = l_buf[pad:pad + B * H * S].view(B, H, S)
    fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(l_buf[:pad] == 7.0) and torch.all(l_buf[-pad:] == 7.0)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=1 / math.sqrt(D), causal=True)
    _compare(o.cpu(), lse.cpu(), o_ref, lse_ref)
