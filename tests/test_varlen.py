"""GPU parity of fa_fwd_varlen (variable-length batches packed along the rows).

Semantics: page "flash-attention-v100", "Changelog", "2.0" (flash_attn_varlen_func):
every sequence is an independent attention problem over its own rows; the causal mask
is aligned to each sequence's own bottom-right corner.  Checked element by element
against the fp64 oracle with max|dO| <= 1e-2, max|dLSE| <= 1e-3 over length mixes that
include empty sequences, single rows, tile-boundary lengths and Sq != Sk per sequence;
with windows, grouped-query heads and every head dim; and bit for bit against fa_fwd
when all lengths are equal.
"""
import math

import numpy as np
import pytest
import torch

import oracle

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


def _packed(lens_q, lens_k, Hq, Hkv, D, seed, amp=1.0):
    g = torch.Generator().manual_seed(seed)
    tq, tk = sum(lens_q), sum(lens_k)
    q = (torch.randn((tq, Hq, D), generator=g) * amp).to(torch.bfloat16)
    k = (torch.randn((tk, Hkv, D), generator=g) * amp).to(torch.bfloat16)
    v = (torch.randn((tk, Hkv, D), generator=g) * amp).to(torch.bfloat16)
    cq = torch.tensor([0] + list(np.cumsum(lens_q)), dtype=torch.int32)
    ck = torch.tensor([0] + list(np.cumsum(lens_k)), dtype=torch.int32)
    return q, k, v, cq, ck


CASES = [
    # (lens_q, lens_k, Hq, Hkv, D, causal, window)
    ([300, 1, 0, 257, 128, 513], [300, 1, 5, 257, 128, 513], 4, 2, 128, False, (-1, -1)),
    ([300, 1, 0, 257, 128, 513], [300, 1, 5, 257, 128, 513], 4, 2, 128, True, (-1, -1)),
    ([100, 700, 33], [400, 200, 33], 2, 1, 128, True, (-1, -1)),      # Sq != Sk per sequence
    ([200, 260], [0, 260], 2, 2, 64, False, (-1, -1)),                # a sequence with no keys
    ([511, 64], [511, 64], 2, 1, 96, True, (50, 0)),
    ([384, 129], [384, 129], 2, 2, 256, False, (20, 30)),
    ([300, 0, 90], [40, 7, 300], 2, 1, 64, True, (-1, -1)),          # rows with no visible key
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"D{c[4]}_c{int(c[5])}_w{c[6][0]}")
def test_varlen_matches_oracle(fa, case):
    lens_q, lens_k, Hq, Hkv, D, causal, window = case
    q, k, v, cq, ck = _packed(lens_q, lens_k, Hq, Hkv, D, seed=sum(lens_q) + D)
    dev = torch.device("cuda:0")
    o, lse = fa.fa_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev),
                              causal=causal, window=window)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    o_ref, lse_ref = oracle.fwd_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=1 / math.sqrt(D),
                                       causal=causal, window=window)
    of, lf = o.float().cpu().numpy(), lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lf)), "LSE -inf pattern differs"
    assert np.abs(of - o_ref).max() <= O_TOL
    if fin.any():
        assert np.abs(lf[fin] - lse_ref[fin]).max() <= LSE_TOL


def test_varlen_output_guard_bands(fa):
    """Writes stay inside the packed O and LSE: sentinel pages around them are untouched,
    with an empty sequence, a single row and a ragged tail in the batch."""
    lens_q, lens_k, Hq, Hkv, D = [130, 0, 1, 257], [130, 7, 1, 300], 4, 2, 128
    q, k, v, cq, ck = _packed(lens_q, lens_k, Hq, Hkv, D, seed=515)
    dev = torch.device("cuda:0")
    tq = sum(lens_q)
    pad = 4096
    o_buf = torch.full((pad + tq * Hq * D + pad,), 7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((pad + Hq * tq + pad,), 7.0, dtype=torch.float32, device=dev)
    o = o_buf[pad:pad + tq * Hq * D].view(tq, Hq, D)
    lse = l_buf[pad:pad + Hq * tq].view(Hq, tq)
    fa.fa_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), causal=True,
                     out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(l_buf[:pad] == 7.0) and torch.all(l_buf[-pad:] == 7.0)
    o_ref, lse_ref = oracle.fwd_varlen(q, k, v, cq.numpy(), ck.numpy(), scale=1 / math.sqrt(D),
                                       causal=True, window=(-1, -1))
    fin = np.isfinite(lse_ref)
    lf = lse.cpu().numpy()
    assert np.array_equal(fin, np.isfinite(lf))
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= O_TOL
    assert np.abs(lf[fin] - lse_ref[fin]).max() <= LSE_TOL


def test_varlen_equal_lengths_reproduce_fa_fwd_bitwise(fa):
    B, S, Hq, Hkv, D = 3, 333, 4, 2, 128
    g = torch.Generator().manual_seed(9)
    q = torch.randn((B, S, Hq, D), generator=g).to(torch.bfloat16).cuda()
    k = torch.randn((B, S, Hkv, D), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((B, S, Hkv, D), generator=g).to(torch.bfloat16).cuda()
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32).cuda()
    for causal in (False, True):
        o, l = fa.fa_fwd(q, k, v, causal=causal)
        ov, lv = fa.fa_fwd_varlen(q.view(B * S, Hq, D), k.view(B * S, Hkv, D), v.view(B * S, Hkv, D),
                                  cu, cu, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(ov.view(B, S, Hq, D), o)
        assert torch.equal(lv.view(Hq, B, S).permute(1, 0, 2), l)


def test_varlen_large_mixed_batch(fa):
    """A length mix resembling packed prefill: 24 sequences of 1..4096 rows, causal,
    grouped-query heads; sampled rows against the oracle, every row finite."""
    rng = np.random.default_rng(3)
    lens = [int(x) for x in rng.integers(1, 4097, 24)]
    q, k, v, cq, ck = _packed(lens, lens, 32, 8, 128, seed=77)
    dev = torch.device("cuda:0")
    o, lse = fa.fa_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all().item() and torch.isfinite(lse).all().item()
    for b in (0, 5, 23):
        s0, s1 = int(cq[b]), int(cq[b + 1])
        rows = sorted(set([0, s1 - s0 - 1, (s1 - s0) // 2]))
        ob, lb = oracle.fwd(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], scale=1 / math.sqrt(128),
                            causal=True, rows=[(0, h, i) for h in (0, 31) for i in rows])
        got = torch.stack([o[s0 + i, h] for h in (0, 31) for i in rows]).float().cpu().numpy()
        gl = np.array([lse[h, s0 + i].item() for h in (0, 31) for i in rows])
        assert np.abs(got - ob).max() <= O_TOL
        assert np.abs(gl - lb).max() <= LSE_TOL
