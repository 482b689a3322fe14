"""GPU parity of fa_decode_splitkv_paged (split-KV decode over a paged KV cache).

Paging semantics: page "flash-attention-v100", flash_attn_with_kvcache block_table,
and "Changelog", "2.5: Paged KV cache".  Checked element by element against the fp64
oracle (oracle.decode_paged) with max|dO| <= 1e-2, max|dLSE| <= 1e-3, with pages
scattered through a larger pool, page sizes 128/256/512, empty and single-key
sequences, and against the contiguous kernel on the same data (identical chunking, so
identical bits).
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


def _scatter(kc, vc, page, extra_pages, seed):
    """Cut a contiguous [B, Smax, Hkv, D] cache into pages scattered through a pool."""
    B, smax, Hkv, D = kc.shape
    mp = smax // page
    n_pool = B * mp + extra_pages
    perm = np.random.default_rng(seed).permutation(n_pool)[: B * mp]
    g = torch.Generator().manual_seed(seed)
    k_pages = torch.randn((n_pool, page, Hkv, D), generator=g).to(kc.dtype)
    v_pages = torch.randn((n_pool, page, Hkv, D), generator=g).to(kc.dtype)
    table = torch.zeros((B, mp), dtype=torch.int32)
    for b in range(B):
        for t in range(mp):
            pg = int(perm[b * mp + t])
            table[b, t] = pg
            k_pages[pg] = kc[b, t * page:(t + 1) * page]
            v_pages[pg] = vc[b, t * page:(t + 1) * page]
    return k_pages, v_pages, table


@pytest.mark.parametrize("page,ns,D", [(128, 3, 128), (256, 5, 128), (512, 2, 128), (256, 16, 128),
                                       (128, 3, 64), (256, 5, 96), (128, 4, 256), (512, 7, 256)])
def test_paged_matches_oracle_and_contiguous(fa, page, ns, D):
    B, Hq, Hkv, smax = 4, 16, 4, 2048
    q, kc, vc, _ = inputs.make_decode(B, Hq, Hkv, D, smax, 1, smax, seed=500 + page)
    lens = torch.tensor([smax, 1, 0, 1234], dtype=torch.int32)
    k_pages, v_pages, table = _scatter(kc, vc, page, extra_pages=7, seed=page)
    dev = torch.device("cuda:0")
    o, lse = fa.fa_decode_splitkv_paged(q.to(dev), k_pages.to(dev), v_pages.to(dev), table.to(dev),
                                        lens.to(dev), num_splits=ns)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    o_ref, lse_ref = oracle.decode_paged(q, k_pages, v_pages, table.numpy(), lens.numpy(),
                                         scale=1 / math.sqrt(D))
    of = o.float().cpu().numpy()[:, 0]
    lf = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lf))
    assert np.abs(of - o_ref).max() <= O_TOL
    assert np.abs(lf[fin] - lse_ref[fin]).max() <= LSE_TOL
    # the contiguous kernel on the gathered cache chunks identically: same bits
    oc, lc = fa.fa_decode_splitkv(q.to(dev), kc.to(dev), vc.to(dev), lens.to(dev), num_splits=ns)
    torch.cuda.synchronize()
    assert torch.equal(o, oc) and torch.equal(lse, lc)


def test_paged_full_size_decode(fa):
    """The decode workload (B=8, Hq=32, Hkv=8, D=128, lengths U[1024, 32768]) stored in
    256-key pages scattered through the pool; every output against the oracle."""
    w = inputs.DECODE
    q, kc, vc, lens = inputs.decode_inputs(w)
    k_pages, v_pages, table = _scatter(kc, vc, 256, extra_pages=16, seed=1)
    dev = torch.device("cuda:0")
    o, lse = fa.fa_decode_splitkv_paged(q.to(dev), k_pages.to(dev), v_pages.to(dev), table.to(dev),
                                        lens.to(dev))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(q, kc, vc, lens, scale=w.scale)
    assert np.abs(o.float().cpu().numpy()[:, 0] - o_ref).max() <= O_TOL
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_TOL


def test_paged_rejects_bad_page_size(fa):
    dev = torch.device("cuda:0")
    q, kc, vc, lens = (t.to(dev) for t in inputs.make_decode(1, 4, 1, 128, 200, 1, 200, seed=3))
    k_pages = kc.view(2, 100, 1, 128)
    table = torch.zeros((1, 2), dtype=torch.int32, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fa_decode_splitkv_paged(q, k_pages, k_pages, table, lens)
    assert e.value.status == 2  # FA_ERR_UNSUPPORTED: page size not a multiple of 128
