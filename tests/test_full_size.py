"""Full-size forward workloads on the GPU, checked against the oracle.

Each workload runs at its full size through fa_fwd, exactly as the benchmark launches
it (same inputs recipe, default scale, persistent grid).  The oracle computes whole
heads -- every row of (b, h) = (0, 0), (B - 1, Hq - 1) and two seeded random heads --
plus rows on both sides of the 128-row tile boundaries of a middle head and random rows
anywhere; at S <= 1024 every row of every head.  Those rows must match within max|dO| <= 1e-2 and max|dLSE| <= 1e-3.  Every
output row is also checked for properties that hold at any size:
  * O and LSE are finite;
  * each output is a convex combination of the visible V rows, so
    min_j V[j, d] <= O[i, d] <= max_j V[j, d] (up to bf16 rounding of O);
  * LSE is at least the largest scaled score of its row; this is checked on the
    sampled rows, where the scores are available.
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

WORKLOADS = inputs.PREFILL_MID + inputs.PREFILL_LONG + inputs.GQA_SWEEP


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_20_gb300 as fa_mod
    from exact_tiled_attention_20_gb300 import build

    build.build_library()
    fa_mod.load()
    return fa_mod


_cache = {}


def _inputs(w):
    key = (w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D, w.amp, w.seed)
    if key not in _cache:
        _cache.clear()
        _cache[key] = inputs.fwd_inputs(w)
    return _cache[key]


def _heads(w, seed=0):
    """(0, 0), (B - 1, Hq - 1) and two seeded random (b, h) pairs, all distinct."""
    rng = np.random.default_rng(seed + w.seed)
    heads = [(0, 0), (w.B - 1, w.Hq - 1)]
    while len(heads) < 4:
        bh = (int(rng.integers(w.B)), int(rng.integers(w.Hq)))
        if bh not in heads:
            heads.append(bh)
    return heads


FULL_CHECK_MAX_S = 1024  # at and below this length every row of every head is checked


def _sample_rows(w, n_random=160, seed=0):
    if w.Sq <= FULL_CHECK_MAX_S:
        bb, hh, ii = np.meshgrid(np.arange(w.B), np.arange(w.Hq), np.arange(w.Sq), indexing="ij")
        return np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1).astype(np.int64)
    rng = np.random.default_rng(seed)
    rows = set()
    for b, h in _heads(w, seed):
        rows.update((b, h, i) for i in range(w.Sq))
    b, h = w.B // 2, w.Hq // 3
    for i in (0, 1, 127, 128, 129, 255, 256, w.Sq // 2, w.Sq - 129, w.Sq - 128, w.Sq - 2, w.Sq - 1):
        if 0 <= i < w.Sq:
            rows.add((b, h, i))
    for _ in range(n_random):
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.Hq)), int(rng.integers(w.Sq))))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: f"{w.name}{'_causal' if w.causal else ''}")
def test_full_size_workload(fa, w):
    q, k, v = _inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = fa.fa_fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0

    # properties of every output row (on the device, then reduced)
    assert torch.isfinite(o).all().item()
    assert torch.isfinite(lse).all().item()
    g = w.Hq // w.Hkv
    if not w.causal:
        vmin = vd.float().amin(dim=1).repeat_interleave(g, dim=1)  # [B, Hq, D]
        vmax = vd.float().amax(dim=1).repeat_interleave(g, dim=1)
        of = o.float()
        lo, hi = vmin.unsqueeze(1), vmax.unsqueeze(1)
        assert (of >= lo - 1e-2 - 4e-3 * lo.abs()).all().item()
        assert (of <= hi + 1e-2 + 4e-3 * hi.abs()).all().item()
    else:
        # prefix extrema of V along the keys bound each causal row (Sq == Sk here)
        vf = vd.float()
        pmin = torch.cummin(vf, dim=1).values.repeat_interleave(g, dim=2)
        pmax = torch.cummax(vf, dim=1).values.repeat_interleave(g, dim=2)
        of = o.float()
        assert (of >= pmin - 1e-2 - 4e-3 * pmin.abs()).all().item()
        assert (of <= pmax + 1e-2 + 4e-3 * pmax.abs()).all().item()
        del pmin, pmax, vf
    del of

    # sampled rows against the oracle
    rows = _sample_rows(w)
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=w.scale, causal=w.causal, rows=rows)
    b, h, i = (torch.as_tensor(rows[:, c], device=dev) for c in range(3))
    o_s = o[b, i, h].float().cpu().numpy()
    lse_s = lse[b, h, i].cpu().numpy()
    do = np.abs(o_s - o_ref).max()
    dl = np.abs(lse_s - lse_ref).max()
    heads = _heads(w)
    print(f"{w.name}: {len(rows)} rows checked, whole heads {heads}, "
          f"max|dO| = {do:.3e}, max|dLSE| = {dl:.3e}")
    assert len(rows) >= 4 * w.Sq
    assert do <= O_TOL, f"max|dO| = {do:.3e} over {len(rows)} rows"
    assert dl <= LSE_TOL, f"max|dLSE| = {dl:.3e} over {len(rows)} rows"
    # LSE >= max scaled score of the row
    hk = rows[:, 1] // g
    for n in range(0, len(rows), max(37, len(rows) // 400)):
        bb, hh, ii = rows[n]
        kk = k[bb, :, hk[n]].double().numpy()
        s = w.scale * (kk @ q[bb, ii, hh].double().numpy())
        if w.causal:
            s = s[: ii + w.Sk - w.Sq + 1]
        assert lse_s[n] >= s.max() - LSE_TOL
