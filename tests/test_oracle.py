"""Pins for the CPU oracle (no GPU).

The oracle is the correctness authority for the CUDA path, so it is pinned here to
things other than itself: the worked examples printed in the pages (tests/golden/),
closed forms, invariants, library routines (scipy's softmax / logsumexp, numpy's tril)
on the textbook definition, and the log-sum-exp partition identity.  A plausible slip
(a dropped term, a wrong sign or index, a transposed operand, a top-left instead of
bottom-right causal mask, h % Hkv instead of h / g) fails at least one of these.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle

RNG = np.random.default_rng(1234)


def _rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


def _scipy_attention(q, k, v, scale, causal):
    """Textbook attention with scipy's softmax/logsumexp; mask from numpy.tril."""
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    g = Hq // Hkv
    o = np.zeros((B, Sq, Hq, D))
    lse = np.zeros((B, Hq, Sq))
    keep = np.tril(np.ones((Sq, Sk), bool), k=Sk - Sq) if causal else np.ones((Sq, Sk), bool)
    for b in range(B):
        for h in range(Hq):
            s = scale * (q[b, :, h, :] @ k[b, :, h // g, :].T)
            s = np.where(keep, s, -np.inf)
            for i in range(Sq):
                if not keep[i].any():
                    lse[b, h, i] = -np.inf
                    continue
                p = scipy.special.softmax(s[i])
                o[b, i, h] = p @ v[b, :, h // g, :]
                lse[b, h, i] = scipy.special.logsumexp(s[i])
    return o, lse


# --------------------------------------------------------------- page examples ----

@pytest.mark.parametrize("sq,sk,name", [(2, 5, "causal_mask_sq2_sk5.txt"),
                                        (5, 2, "causal_mask_sq5_sk2.txt")])
def test_causal_mask_matches_pages_examples(sq, sk, name, golden):
    """With Q = 0 every visible key weighs 1/|J_i|; V = one-hot rows reveal the mask."""
    D = 8
    q = np.zeros((1, sq, 1, D))
    k = _rand(1, sk, 1, D)
    v = np.zeros((1, sk, 1, D))
    for j in range(sk):
        v[0, j, 0, j] = 1.0
    o, lse = oracle.fwd(q, k, v, scale=0.7, causal=True)
    mask = (o[0, :, 0, :sk] > 0).astype(int)
    assert mask.tolist() == golden(name)
    for i in range(sq):
        n = mask[i].sum()
        if n == 0:  # fully masked row: zero output, log-sum-exp -inf
            assert np.all(o[0, i, 0] == 0.0)
            assert lse[0, 0, i] == -np.inf
        else:
            assert np.allclose(o[0, i, 0, :sk][mask[i] == 1], 1.0 / n, atol=1e-15)
            assert lse[0, 0, i] == pytest.approx(math.log(n), abs=1e-14)


def test_gqa_head_map_matches_pages_example(golden):
    """6 Q heads over 2 K/V heads: V of K/V head hk is the constant hk + 1."""
    B, S, D = 2, 7, 16
    q = _rand(B, S, 6, D)
    k = _rand(B, S, 2, D)
    v = np.zeros((B, S, 2, D))
    v[:, :, 0, :] = 1.0
    v[:, :, 1, :] = 2.0
    o, _ = oracle.fwd(q, k, v, scale=0.3, causal=False)
    head_map = [int(round(o[0, 0, h, 0])) - 1 for h in range(6)]
    assert [head_map] == golden("gqa_heads_6_over_2.txt")
    for h in range(6):
        assert np.allclose(o[:, :, h, :], head_map[h] + 1.0, atol=1e-14)


# ---------------------------------------------------------------- closed forms ----

@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_v_and_log_count(causal):
    B, Sq, Sk, H, D = 2, 9, 9, 3, 5
    q = np.zeros((B, Sq, H, D))
    k = _rand(B, Sk, H, D)
    v = _rand(B, Sk, H, D)
    o, lse = oracle.fwd(q, k, v, scale=1.3, causal=causal)
    for i in range(Sq):
        n = i + 1 if causal else Sk
        assert np.allclose(o[:, i], v[:, :n].mean(axis=1), atol=1e-14)
        assert np.allclose(lse[:, :, i], math.log(n), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_v_gives_ones(causal):
    """Rows of P sum to one."""
    q, k = _rand(1, 11, 2, 8), _rand(1, 13, 2, 8)
    v = np.ones((1, 13, 2, 8))
    o, _ = oracle.fwd(q, k, v, scale=0.9, causal=causal)
    assert np.allclose(o, 1.0, atol=1e-14)


def test_one_hot_keys_with_large_scale_select_rows():
    """K rows e_j, q_i = e_pi(i), scale 100: softmax is one-hot up to e^-100."""
    D = Sk = 64
    Sq = 40
    perm = RNG.permutation(Sk)[:Sq]
    k = np.eye(Sk)[None, :, None, :]
    q = np.eye(Sk)[perm][None, :, None, :]
    v = _rand(1, Sk, 1, D)
    o, lse = oracle.fwd(q, k, v, scale=100.0, causal=False)
    assert np.allclose(o[0, :, 0], v[0, perm, 0], atol=1e-12)
    assert np.allclose(lse[0, 0], 100.0, atol=1e-12)


def test_single_key_returns_that_value():
    q, k, v = _rand(2, 3, 2, 6), _rand(2, 1, 2, 6), _rand(2, 1, 2, 6)
    o, lse = oracle.fwd(q, k, v, scale=0.5, causal=False)
    for i in range(3):
        assert np.allclose(o[:, i], v[:, 0], atol=1e-15)
    s = 0.5 * np.einsum("bihd,bhd->bhi", q, k[:, 0])
    assert np.allclose(lse, s, atol=1e-14)


# ---------------------------------------------------------- library reference ----

@pytest.mark.parametrize("shape", [(1, 5, 5, 1, 1, 4), (2, 7, 12, 4, 2, 8),
                                   (1, 12, 7, 3, 1, 16), (2, 33, 33, 2, 2, 32),
                                   (1, 1, 17, 6, 3, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_scipy_softmax_definition(shape, causal):
    B, Sq, Sk, Hq, Hkv, D = shape
    q, k, v = _rand(B, Sq, Hq, D), _rand(B, Sk, Hkv, D), _rand(B, Sk, Hkv, D)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.fwd(q, k, v, scale=scale, causal=causal)
    o_ref, lse_ref = _scipy_attention(q, k, v, scale, causal)
    assert np.allclose(o, o_ref, atol=1e-12, rtol=0)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.allclose(lse[fin], lse_ref[fin], atol=1e-12, rtol=0)


def test_selected_rows_match_full_evaluation():
    q, k, v = _rand(2, 9, 4, 8), _rand(2, 11, 2, 8), _rand(2, 11, 2, 8)
    o, lse = oracle.fwd(q, k, v, scale=0.4, causal=True)
    rows = [(1, 3, 8), (0, 0, 0), (1, 2, 4)]
    o_r, lse_r = oracle.fwd(q, k, v, scale=0.4, causal=True, rows=rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(o_r[n], o[b, i, h])
        assert lse_r[n] == lse[b, h, i]


@pytest.mark.parametrize("tdt", [torch.bfloat16, torch.float16])
def test_16bit_inputs_decode_exactly(tdt):
    """The oracle's bf16/fp16 decoders agree with torch's own widening to fp64."""
    g = torch.Generator().manual_seed(5)
    q = (torch.randn(1, 6, 2, 8, generator=g) * 3).to(tdt)
    k = (torch.randn(1, 6, 2, 8, generator=g) * 3).to(tdt)
    v = (torch.randn(1, 6, 2, 8, generator=g) * 3).to(tdt)
    # include subnormal / tiny and large magnitudes in V
    v[0, 0, 0, :4] = torch.tensor([1e-6, -3e-5, 6e4 if tdt == torch.float16 else 1e30, -0.0])
    o16, l16 = oracle.fwd(q, k, v, scale=0.2, causal=True)
    o64, l64 = oracle.fwd(q.double(), k.double(), v.double(), scale=0.2, causal=True)
    assert np.array_equal(o16, o64)
    assert np.array_equal(l16, l64)


# -------------------------------------------------------------------- invariants ----

def test_lse_bounds():
    q, k, v = _rand(1, 10, 2, 8), _rand(1, 10, 2, 8), _rand(1, 10, 2, 8)
    o, lse = oracle.fwd(q, k, v, scale=0.8, causal=True)
    for h in range(2):
        s = 0.8 * q[0, :, h] @ k[0, :, h].T
        for i in range(10):
            m = s[i, : i + 1].max()
            assert m <= lse[0, h, i] <= m + math.log(i + 1) + 1e-12


def test_noncausal_invariant_to_joint_key_permutation():
    q, k, v = _rand(2, 6, 2, 8), _rand(2, 9, 1, 8), _rand(2, 9, 1, 8)
    perm = RNG.permutation(9)
    o1, l1 = oracle.fwd(q, k, v, scale=0.6)
    o2, l2 = oracle.fwd(q, k[:, perm], v[:, perm], scale=0.6)
    assert np.allclose(o1, o2, atol=1e-13)
    assert np.allclose(l1, l2, atol=1e-13)


def test_affine_in_v():
    q, k, v = _rand(1, 6, 2, 8), _rand(1, 8, 2, 8), _rand(1, 8, 2, 8)
    o1, _ = oracle.fwd(q, k, v, scale=0.6, causal=True)
    o2, _ = oracle.fwd(q, k, 2.5 * v - 1.0, scale=0.6, causal=True)
    assert np.allclose(o2, 2.5 * o1 - 1.0, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv_heads():
    q, k, v = _rand(2, 5, 6, 8), _rand(2, 7, 2, 8), _rand(2, 7, 2, 8)
    o1, l1 = oracle.fwd(q, k, v, scale=0.5, causal=True)
    o2, l2 = oracle.fwd(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2), scale=0.5,
                        causal=True)
    assert np.allclose(o1, o2, atol=1e-14)
    assert np.allclose(l1, l2, atol=1e-14)


def test_causal_first_row_equals_first_value():
    q, k, v = _rand(1, 8, 1, 4), _rand(1, 8, 1, 4), _rand(1, 8, 1, 4)
    o, _ = oracle.fwd(q, k, v, scale=1.0, causal=True)
    assert np.allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15)


# -------------------------------------------------------- decode, split, merge ----

def _decode_case(B=3, Hq=8, Hkv=2, D=16, Smax=40, seed=3):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, 1, Hq, D))
    kc = rng.standard_normal((B, Smax, Hkv, D))
    vc = rng.standard_normal((B, Smax, Hkv, D))
    lens = np.array([Smax, 1, 23][:B], np.int32)
    return q, kc, vc, lens


def test_decode_equals_forward_over_valid_prefix():
    q, kc, vc, lens = _decode_case()
    o, lse = oracle.decode(q, kc, vc, lens, scale=0.25)
    for b, n in enumerate(lens):
        of, lf = oracle.fwd(q[b:b + 1], kc[b:b + 1, :n], vc[b:b + 1, :n], scale=0.25)
        assert np.allclose(o[b], of[0, 0], atol=1e-14)
        assert np.allclose(lse[b], lf[0, :, 0], atol=1e-14)


def test_decode_matches_scipy():
    q, kc, vc, lens = _decode_case()
    o, lse = oracle.decode(q, kc, vc, lens, scale=0.25)
    for b, n in enumerate(lens):
        for h in range(8):
            s = 0.25 * kc[b, :n, h // 4] @ q[b, 0, h]
            assert np.allclose(o[b, h], scipy.special.softmax(s) @ vc[b, :n, h // 4],
                               atol=1e-12)
            assert lse[b, h] == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)


def test_decode_empty_cache_gives_zero_and_minus_inf():
    q, kc, vc, _ = _decode_case()
    o, lse = oracle.decode(q, kc, vc, np.array([0, 5, 0], np.int32), scale=0.25)
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    assert np.all(lse[0] == -np.inf) and np.all(lse[2] == -np.inf)
    assert np.all(np.isfinite(lse[1]))


@pytest.mark.parametrize("cuts", [[0, 40], [0, 13, 40], [0, 1, 2, 3, 39, 40],
                                  [0, 16, 16, 32, 40], [0, 0, 40, 40]])
def test_partials_merge_to_the_full_result(cuts):
    """Any partition of the keys, empty parts included, merges back exactly."""
    q, kc, vc, _ = _decode_case()
    o_full, l_full = oracle.decode(q, kc, vc, np.array([40, 40, 40], np.int32), scale=0.3)
    for b in range(3):
        for h in (0, 5):
            parts = [oracle.partial(q, kc, vc, b, h, cuts[s], cuts[s + 1], 0.3)
                     for s in range(len(cuts) - 1)]
            o, lse = oracle.combine(np.stack([p[0] for p in parts]), [p[1] for p in parts])
            assert np.allclose(o, o_full[b, h], atol=1e-13)
            assert lse == pytest.approx(l_full[b, h], abs=1e-13)


def test_combine_closed_forms():
    o_a, o_b = _rand(8), _rand(8)
    o, lse = oracle.combine(np.stack([o_a, o_b]), [1.5, 1.5])       # equal weights
    assert np.allclose(o, 0.5 * (o_a + o_b), atol=1e-15)
    assert lse == pytest.approx(1.5 + math.log(2.0), abs=1e-15)
    o, lse = oracle.combine(np.stack([o_a, o_b]), [-np.inf, 0.25])  # empty part weighs 0
    assert np.allclose(o, o_b, atol=1e-15) and lse == pytest.approx(0.25, abs=1e-15)
    o, lse = oracle.combine(np.stack([o_a, o_b]), [-np.inf, -np.inf])
    assert np.all(o == 0) and lse == -np.inf
    o, lse = oracle.combine(np.stack([o_a, o_b]), [0.0, math.log(3.0)])  # weights 1/4, 3/4
    assert np.allclose(o, 0.25 * o_a + 0.75 * o_b, atol=1e-15)
    assert lse == pytest.approx(math.log(4.0), abs=1e-15)


def test_bad_arguments_are_rejected():
    q, k, v = _rand(1, 4, 3, 8), _rand(1, 4, 2, 8), _rand(1, 4, 2, 8)
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v, scale=1.0)                 # 3 Q heads over 2 K/V heads
    q, kc, vc, _ = _decode_case()
    with pytest.raises(ValueError):
        oracle.decode(q, kc, vc, np.array([41, 1, 1], np.int32), scale=1.0)  # > Smax


# ---------------------------------------------------------- sliding window ----

def _band_keep(Sq, Sk, left, right, causal):
    """Visible-key mask of a sliding window from numpy's triu/tril (bottom-right aligned)."""
    keep = np.ones((Sq, Sk), bool)
    off = Sk - Sq
    if right >= 0:
        keep &= np.tril(np.ones((Sq, Sk), bool), k=off + right)
    if causal:
        keep &= np.tril(np.ones((Sq, Sk), bool), k=off)
    if left >= 0:
        keep &= np.triu(np.ones((Sq, Sk), bool), k=off - left)
    return keep


@pytest.mark.parametrize("sq,sk,left,right,causal", [
    (9, 9, 2, 1, False), (9, 9, 3, -1, True), (5, 12, 0, 0, False), (12, 5, 1, 2, False),
    (12, 5, 4, 0, True), (7, 7, -1, 2, False), (6, 20, 3, 3, True)])
def test_window_matches_band_mask(sq, sk, left, right, causal):
    """Q = 0 gives the mean over exactly the visible keys: the band mask is recovered."""
    D = max(sk, 4)
    q = np.zeros((1, sq, 1, D))
    k = _rand(1, sk, 1, D)
    v = np.zeros((1, sk, 1, D))
    for j in range(sk):
        v[0, j, 0, j] = 1.0
    o, lse = oracle.fwd(q, k, v, scale=0.5, causal=causal, window=(left, right))
    keep = _band_keep(sq, sk, left, right, causal)
    assert np.array_equal(o[0, :, 0, :sk] > 0, keep)
    for i in range(sq):
        n = keep[i].sum()
        if n == 0:
            assert lse[0, 0, i] == -np.inf and np.all(o[0, i] == 0)
        else:
            assert lse[0, 0, i] == pytest.approx(math.log(n), abs=1e-14)


def test_window_special_cases_reduce_to_full_and_causal():
    q, k, v = _rand(2, 11, 2, 8), _rand(2, 11, 1, 8), _rand(2, 11, 1, 8)
    full = oracle.fwd(q, k, v, scale=0.6)
    causal = oracle.fwd(q, k, v, scale=0.6, causal=True)
    for a, b in ((oracle.fwd(q, k, v, scale=0.6, window=(-1, -1)), full),
                 (oracle.fwd(q, k, v, scale=0.6, window=(100, 100)), full),
                 (oracle.fwd(q, k, v, scale=0.6, window=(-1, 0)), causal),
                 (oracle.fwd(q, k, v, scale=0.6, causal=True, window=(100, 5)), causal)):
        assert np.allclose(a[0], b[0], atol=1e-14) and np.allclose(a[1], b[1], atol=1e-14)


def test_window_matches_scipy_with_band_mask():
    B, Sq, Sk, Hq, Hkv, D = 1, 10, 13, 2, 1, 8
    q, k, v = _rand(B, Sq, Hq, D), _rand(B, Sk, Hkv, D), _rand(B, Sk, Hkv, D)
    left, right = 3, 2
    o, lse = oracle.fwd(q, k, v, scale=0.4, window=(left, right))
    keep = _band_keep(Sq, Sk, left, right, False)
    for h in range(Hq):
        s = 0.4 * q[0, :, h] @ k[0, :, 0].T
        for i in range(Sq):
            p = scipy.special.softmax(s[i][keep[i]])
            assert np.allclose(o[0, i, h], p @ v[0, keep[i], 0], atol=1e-12)
            assert lse[0, h, i] == pytest.approx(scipy.special.logsumexp(s[i][keep[i]]), abs=1e-12)


# ---------------------------------------------------------------- paged cache ----

def _paged_case(B=3, Hq=4, Hkv=2, D=8, page=4, max_pages=5, seed=11):
    rng = np.random.default_rng(seed)
    smax = page * max_pages
    q = rng.standard_normal((B, 1, Hq, D))
    kc = rng.standard_normal((B, smax, Hkv, D))
    vc = rng.standard_normal((B, smax, Hkv, D))
    lens = np.array([smax, 7, 0][:B], np.int32)
    return q, kc, vc, lens


def test_paged_identity_table_equals_contiguous_decode():
    q, kc, vc, lens = _paged_case()
    B, smax, Hkv, D = kc.shape
    page, max_pages = 4, 5
    k_pages = kc.reshape(B * max_pages, page, Hkv, D)
    v_pages = vc.reshape(B * max_pages, page, Hkv, D)
    table = np.arange(B * max_pages, dtype=np.int32).reshape(B, max_pages)
    o1, l1 = oracle.decode_paged(q, k_pages, v_pages, table, lens, scale=0.4)
    o2, l2 = oracle.decode(q, kc, vc, lens, scale=0.4)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_permuted_pages_equal_contiguous_decode():
    """Pages scattered through the pool by a random permutation (and spare pages that
    no sequence uses) give the same result as the contiguous cache."""
    q, kc, vc, lens = _paged_case()
    B, smax, Hkv, D = kc.shape
    page, max_pages = 4, 5
    n_pool = B * max_pages + 3
    perm = RNG.permutation(n_pool)[: B * max_pages]
    k_pages = RNG.standard_normal((n_pool, page, Hkv, D))
    v_pages = RNG.standard_normal((n_pool, page, Hkv, D))
    table = np.zeros((B, max_pages), np.int32)
    for b in range(B):
        for t in range(max_pages):
            pg = perm[b * max_pages + t]
            table[b, t] = pg
            k_pages[pg] = kc[b, t * page:(t + 1) * page]
            v_pages[pg] = vc[b, t * page:(t + 1) * page]
    o1, l1 = oracle.decode_paged(q, k_pages, v_pages, table, lens, scale=0.4)
    o2, l2 = oracle.decode(q, kc, vc, lens, scale=0.4)
    assert np.allclose(o1, o2, atol=1e-15) and np.array_equal(np.isfinite(l1), np.isfinite(l2))
    fin = np.isfinite(l2)
    assert np.allclose(l1[fin], l2[fin], atol=1e-15)


def test_paged_rejects_out_of_pool_pages():
    q, kc, vc, lens = _paged_case()
    B, smax, Hkv, D = kc.shape
    k_pages = kc.reshape(B * 5, 4, Hkv, D)
    table = np.arange(B * 5, dtype=np.int32).reshape(B, 5)
    table[0, 1] = 99
    with pytest.raises(ValueError):
        oracle.decode_paged(q, k_pages, k_pages, table, lens, scale=0.4)


# ------------------------------------------------------------- varlen batches ----

def test_varlen_with_equal_lengths_equals_batched():
    q, k, v = _rand(3, 7, 4, 8), _rand(3, 9, 2, 8), _rand(3, 9, 2, 8)
    o_b, l_b = oracle.fwd(q, k, v, scale=0.5, causal=True)
    o_v, l_v = oracle.fwd_varlen(q.reshape(21, 4, 8), k.reshape(27, 2, 8), v.reshape(27, 2, 8),
                                 [0, 7, 14, 21], [0, 9, 18, 27], scale=0.5, causal=True)
    assert np.array_equal(o_v.reshape(3, 7, 4, 8), o_b)
    assert np.array_equal(l_v.reshape(4, 3, 7).transpose(1, 0, 2), l_b)


def test_varlen_sequences_are_independent_and_empty_ones_are_zero():
    q, k, v = _rand(10, 2, 8), _rand(12, 1, 8), _rand(12, 1, 8)
    cq, ck = [0, 4, 4, 10], [0, 5, 9, 9]  # sequence 1 has no queries, sequence 2 no keys
    o, lse = oracle.fwd_varlen(q, k, v, cq, ck, scale=0.7)
    o0, l0 = oracle.fwd(q[None, 0:4], k[None, 0:5], v[None, 0:5], scale=0.7)
    assert np.array_equal(o[0:4], o0[0]) and np.array_equal(lse[:, 0:4], l0[0])
    assert np.all(o[4:10] == 0) and np.all(lse[:, 4:10] == -np.inf)
    k2 = k.copy()
    k2[5:] += 3.0  # other sequences' keys do not touch sequence 0
    o2, _ = oracle.fwd_varlen(q, k2, v, cq, ck, scale=0.7)
    assert np.array_equal(o2[0:4], o[0:4])


def test_decode_multi_reduces_to_single_token_decode():
    q, kc, vc, lens = _decode_case()
    o1, l1 = oracle.decode(q, kc, vc, lens, scale=0.3)
    o2, l2 = oracle.decode_multi(q, kc, vc, lens, scale=0.3, causal=True)
    assert np.array_equal(o2[:, 0], o1) and np.array_equal(l2[:, :, 0], l1)


def test_decode_multi_causal_rows_see_growing_prefixes():
    """Query s of sequence b sees keys [0, len - Sq + s]: with Q = 0 its output is the
    mean of exactly those V rows."""
    rng = np.random.default_rng(4)
    B, Sq, Hq, Hkv, D, smax = 2, 3, 2, 1, 8, 10
    q = np.zeros((B, Sq, Hq, D))
    kc, vc = rng.standard_normal((B, smax, Hkv, D)), rng.standard_normal((B, smax, Hkv, D))
    lens = [7, 2]
    o, lse = oracle.decode_multi(q, kc, vc, lens, scale=1.0, causal=True)
    for b in range(B):
        for s in range(Sq):
            n = lens[b] - Sq + s + 1
            if n <= 0:
                assert np.all(o[b, s] == 0) and np.all(lse[b, :, s] == -np.inf)
            else:
                assert np.allclose(o[b, s, 0], vc[b, :n, 0].mean(0), atol=1e-14)
                assert lse[b, 0, s] == pytest.approx(math.log(n), abs=1e-14)
