"""GPU parity of fa_fwd_window (sliding-window local attention) against the oracle.

Window semantics: page "flash-attention-v100", flash_attn_func window_size, and
"Changelog", "2.3: Local (i.e., sliding window) attention".  Element-by-element
against the fp64 oracle with max|dO| <= 1e-2, max|dLSE| <= 1e-3, over windows on both
or one side, combined with the causal flag, Sq != Sk (bottom-right aligned), every head
dim, and windows that leave rows with no visible key.  Special windows must reproduce
fa_fwd bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
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


def _check(o, lse, o_ref, lse_ref):
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse)), "LSE -inf pattern differs"
    do = np.abs(o - o_ref).max()
    dl = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert do <= O_TOL, f"max|dO| = {do:.3e}"
    assert dl <= LSE_TOL, f"max|dLSE| = {dl:.3e}"


CASES = [
    # (B, Sq, Sk, Hq, Hkv, D, left, right, causal)
    (1, 600, 600, 2, 1, 128, 100, 100, False),
    (1, 600, 600, 2, 2, 128, 130, 0, True),
    (2, 300, 300, 4, 2, 64, 0, 257, False),
    (1, 700, 700, 2, 1, 128, 255, -1, False),
    (1, 700, 700, 2, 1, 128, -1, 17, False),
    (1, 257, 257, 2, 2, 96, 64, 64, True),
    (1, 300, 333, 2, 1, 256, 40, 10, False),
    (1, 200, 900, 2, 2, 128, 300, 0, True),     # Sq < Sk: window near the bottom-right
    (1, 500, 120, 2, 1, 128, 30, 5, False),     # Sq > Sk: leading rows see no key
    (1, 400, 400, 2, 1, 128, 0, 0, False),      # one key per row
    # fixed-length windows skip a Q sub-tile's blocks outside its window:
    (2, 1030, 1030, 2, 2, 128, 127, 0, True),   # short window: most blocks dead for one sub-tile
    (1, 1100, 1100, 2, 1, 96, 200, 0, False),   # D = 96, several tiles
    (1, 300, 300, 2, 1, 128, 50, 0, False),     # last tile's second sub-tile lies past Sq
    # D = 64 (general kernel, FMA-pipe mask with two bounds):
    (1, 500, 120, 2, 1, 64, 30, 5, False),      # Sq > Sk: leading rows see no key
    (1, 600, 600, 2, 2, 64, 130, 0, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "_".join(map(str, c)))
def test_window_matches_oracle(fa, case):
    B, Sq, Sk, Hq, Hkv, D, left, right, causal = case
    q, k, v = inputs.make_qkv(B, Sq, Sk, Hq, Hkv, D, seed=300 + Sq + left)
    dev = torch.device("cuda:0")
    o, lse = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, window=(left, right))
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=1 / math.sqrt(D), causal=causal,
                                window=(left, right))
    _check(o.cpu(), lse.cpu(), o_ref, lse_ref)


@pytest.mark.parametrize("D", [96, 128])
def test_window_fp16(fa, D):
    """fp16 inputs through the fixed-length window kernel (the skipping instantiation)."""
    q, k, v = inputs.make_qkv(1, 700, 700, 2, 1, D, seed=420 + D, dtype="fp16")
    dev = torch.device("cuda:0")
    o, lse = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, window=(200, 0))
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=1 / math.sqrt(D), causal=True, window=(200, 0))
    _check(o.cpu(), lse.cpu(), o_ref, lse_ref)


def test_special_windows_reproduce_fa_fwd_bitwise(fa):
    q, k, v = (t.to("cuda:0") for t in inputs.make_qkv(2, 520, 520, 4, 2, 128, seed=410))
    o_full, l_full = fa.fa_fwd(q, k, v)
    o_c, l_c = fa.fa_fwd(q, k, v, causal=True)
    for win, causal, ref in (((-1, -1), False, (o_full, l_full)), ((10**6, 10**6), False, (o_full, l_full)),
                             ((-1, 0), False, (o_c, l_c)), ((-1, -1), True, (o_c, l_c))):
        o, l = fa.fa_fwd(q, k, v, causal=causal, window=win)
        torch.cuda.synchronize()
        assert torch.equal(o, ref[0]) and torch.equal(l, ref[1]), (win, causal)


def test_window_rejects_bad_bounds(fa):
    q, k, v = (t.to("cuda:0") for t in inputs.make_qkv(1, 64, 64, 1, 1, 64, seed=411))
    with pytest.raises(fa.FaError):
        fa.fa_fwd(q, k, v, window=(-2, 5))


def test_window_full_size_local_attention(fa):
    """[16, 8192, 32, 128] causal with a 1024-key window, launched as a user would;
    sampled rows against the oracle, every row finite."""
    w = inputs.PREFILL_LONG[0]
    q, k, v = inputs.fwd_inputs(w)
    dev = torch.device("cuda:0")
    o, lse = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, window=(1023, 0))
    torch.cuda.synchronize()
    assert torch.isfinite(o).all().item() and torch.isfinite(lse).all().item()
    rng = np.random.default_rng(5)
    rows = np.stack([rng.integers(0, w.B, 96), rng.integers(0, w.Hq, 96), rng.integers(0, w.Sq, 96)], 1)
    rows = np.concatenate([rows, [[0, 0, 0], [0, 0, 1023], [0, 0, 1024], [15, 31, 8191]]]).astype(np.int64)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=w.scale, causal=True, rows=rows, window=(1023, 0))
    b, h, i = (torch.as_tensor(rows[:, c], device=dev) for c in range(3))
    assert np.abs(o[b, i, h].float().cpu().numpy() - o_ref).max() <= O_TOL
    assert np.abs(lse[b, h, i].cpu().numpy() - lse_ref).max() <= LSE_TOL
