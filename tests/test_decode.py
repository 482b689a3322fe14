"""GPU parity of fa_decode_splitkv (split-KV single-token decode) against the CPU oracle.

Bars: max|dO| <= 1e-2, max|dLSE| <= 1e-3 against the fp64 definition (oracle.decode),
element by element.  The per-piece partials in the workspace are checked against the
oracle's attention over each piece's key range (oracle.partial), and the merged output
against the full definition, for several split counts, zero-length caches, group sizes
1..16, fp16, and the full-size decode workload (every output).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_plan import pieces as _pieces
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


def _dev(*ts):
    return [t.to("cuda:0") for t in ts]


def _check(o, lse, o_ref, lse_ref):
    o = o.float().cpu().numpy().reshape(o_ref.shape)
    lse = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.all(lse[~fin] == -np.inf)
    do = np.abs(o - o_ref).max()
    dl = np.abs(lse[fin] - lse_ref[fin]).max() if fin.any() else 0.0
    assert do <= O_TOL, f"max|dO| = {do:.3e}"
    assert dl <= LSE_TOL, f"max|dLSE| = {dl:.3e}"
    return do, dl


HEAD_DIMS = [64, 96, 128, 256]


@pytest.mark.parametrize("D,ns", [(d, n) for d in HEAD_DIMS for n in (1, 3, 16)]
                         + [(128, 2), (128, 7)])
def test_decode_matches_oracle(fa, D, ns):
    q, kc, vc, _ = inputs.make_decode(3, 8, 2, D, 700, 1, 700, seed=50 + ns + D)
    lens = torch.tensor([700, 1, 333], dtype=torch.int32)
    o, lse = fa.fa_decode_splitkv(*_dev(q, kc, vc, lens), num_splits=ns)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    o_ref, lse_ref = oracle.decode(q, kc, vc, lens, scale=1 / math.sqrt(D))
    _check(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("D,ns,Hkv", [(128, 2, 2), (128, 4, 2), (128, 64, 2), (64, 5, 2), (96, 3, 2),
                                      (256, 4, 2), (256, 64, 2), (64, 5, 8), (96, 3, 4),
                                      (128, 7, 16), (128, 4, 3), (96, 3, 6)])
def test_decode_partials_match_oracle_pieces(fa, D, ns, Hkv):
    """The workspace holds, per (b, head, piece), the piece's own attention and LSE; kv heads
    in groups of 2, 4 and 8 (Hkv = 16: two groups per sequence), and none (Hkv = 3)."""
    B, Smax = 3, 3000
    Hq = 8 if 8 % Hkv == 0 else 2 * Hkv
    q, kc, vc, _ = inputs.make_decode(B, Hq, Hkv, D, Smax, 1, Smax, seed=61 + ns)
    lens = torch.tensor([3000, 250, 1300], dtype=torch.int32)
    nbytes = fa.fa_decode_workspace_bytes(B, Hq, D, ns)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda:0")
    fa.fa_decode_splitkv(*_dev(q, kc, vc, lens), num_splits=ns, workspace=ws)
    torch.cuda.synchronize()
    rows = B * Hq * ns
    o_bytes = (rows * D * 4 + 255) // 256 * 256
    o_part = ws[: rows * D * 4].view(torch.float32).view(B, Hq, ns, D).cpu().numpy()
    l_part = ws[o_bytes: o_bytes + rows * 4].view(torch.float32).view(B, Hq, ns).cpu().numpy()
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    pieces = _pieces(lens.tolist(), Hkv, ns, grid)
    scale = 1 / math.sqrt(D)
    g = Hq // Hkv
    checked = 0
    for b in range(B):
        for h in range(Hq):
            for slot, j0, j1 in pieces[(b, h // g)]:
                assert slot < ns
                o_ref, l_ref = oracle.partial(q, kc, vc, b, h, j0, j1, scale)
                assert np.abs(o_part[b, h, slot] - o_ref).max() <= O_TOL
                assert abs(l_part[b, h, slot] - l_ref) <= LSE_TOL
                checked += 1
    assert checked >= B * Hq


def test_decode_empty_and_single_key_sequences(fa):
    q, kc, vc, _ = inputs.make_decode(4, 4, 4, 128, 300, 1, 300, seed=62)
    lens = torch.tensor([0, 1, 0, 300], dtype=torch.int32)
    o, lse = fa.fa_decode_splitkv(*_dev(q, kc, vc, lens), num_splits=3)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(q, kc, vc, lens, scale=1 / math.sqrt(128))
    _check(o, lse, o_ref, lse_ref)
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)


def test_decode_all_empty(fa):
    q, kc, vc, _ = inputs.make_decode(2, 4, 2, 128, 256, 1, 256, seed=63)
    lens = torch.zeros(2, dtype=torch.int32)
    o, lse = fa.fa_decode_splitkv(*_dev(q, kc, vc, lens), num_splits=2)
    torch.cuda.synchronize()
    assert torch.all(o == 0)
    assert torch.all(lse == float("-inf"))


@pytest.mark.parametrize("g,D,Hkv", [(1, 128, 2), (2, 128, 2), (3, 128, 2), (4, 128, 2), (8, 128, 2),
                                     (16, 128, 2), (16, 64, 2), (16, 256, 2), (3, 96, 2),
                                     (2, 96, 3), (1, 96, 1), (2, 64, 8), (4, 96, 4), (1, 128, 16),
                                     (2, 96, 6), (4, 256, 8)])
def test_decode_group_sizes(fa, g, D, Hkv):
    """GQA group sizes 1..16, with kv heads planned in groups of 2, 4 and 8 where Hkv
    allows and one by one where it is odd."""
    q, kc, vc, lens = inputs.make_decode(2, g * Hkv, Hkv, D, 520, 1, 520, seed=70 + g)
    o, lse = fa.fa_decode_splitkv(*_dev(q, kc, vc, lens), num_splits=5)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(q, kc, vc, lens, scale=1 / math.sqrt(D))
    _check(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("D", HEAD_DIMS)
def test_decode_fp16(fa, D):
    q, kc, vc, lens = inputs.make_decode(3, 8, 2, D, 640, 1, 640, seed=80, dtype="fp16")
    o, lse = fa.fa_decode_splitkv(*_dev(q, kc, vc, lens), num_splits=4)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.decode(q, kc, vc, lens, scale=1 / math.sqrt(D))
    _check(o, lse, o_ref, lse_ref)


def test_decode_independent_of_splits_and_deterministic(fa):
    q, kc, vc, lens = _dev(*inputs.make_decode(4, 16, 4, 128, 2000, 100, 2000, seed=81))
    outs = []
    for ns in (1, 2, 5, 16, 64):
        o, lse = fa.fa_decode_splitkv(q, kc, vc, lens, num_splits=ns)
        o2, lse2 = fa.fa_decode_splitkv(q, kc, vc, lens, num_splits=ns)
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
        outs.append((o.float(), lse))
    for o, lse in outs[1:]:
        assert (o - outs[0][0]).abs().max().item() <= O_TOL
        assert (lse - outs[0][1]).abs().max().item() <= LSE_TOL


def test_decode_one_split_equals_forward(fa):
    """Decode of sequence b equals the forward pass with Sq = 1 over its valid prefix."""
    q, kc, vc, lens = inputs.make_decode(2, 8, 2, 128, 400, 50, 400, seed=82)
    o, lse = fa.fa_decode_splitkv(*_dev(q, kc, vc, lens), num_splits=1)
    torch.cuda.synchronize()
    for b in range(2):
        n = int(lens[b])
        of, lf = fa.fa_fwd(*_dev(q[b:b + 1], kc[b:b + 1, :n].contiguous(), vc[b:b + 1, :n].contiguous()))
        torch.cuda.synchronize()
        assert (of[0, 0].float() - o[b, 0].float()).abs().max().item() <= O_TOL
        assert (lf[0, :, 0] - lse[b]).abs().max().item() <= LSE_TOL


@pytest.mark.parametrize("w", [inputs.DECODE] + inputs.DECODE_D_SWEEP, ids=lambda w: w.name)
def test_decode_full_size_workload(fa, w):
    """The decode workload at full size (B=8, Hq=32, Hkv=8, Smax=32768, lengths
    U[1024, 32768]; D = 128, and the same lengths and shape at D = 64, 96 and 256) with the
    default split count, launched as the benchmark launches it; every output row checked
    against the oracle."""
    q, kc, vc, lens = inputs.decode_inputs(w)
    o, lse = fa.fa_decode_splitkv(*_dev(q, kc, vc, lens))
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    o_ref, lse_ref = oracle.decode(q, kc, vc, lens, scale=w.scale)
    _check(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("D", HEAD_DIMS)
def test_decode_output_and_workspace_guard_bands(fa, D):
    """Writes stay inside O, LSE and the workspace: sentinel pages around each are
    untouched, including with an empty sequence and a length one past a tile."""
    B, Hq, Hkv, Smax, ns = 3, 8, 2, 900, 4
    q, kc, vc, _ = inputs.make_decode(B, Hq, Hkv, D, Smax, 1, Smax, seed=91)
    lens = torch.tensor([900, 0, 129], dtype=torch.int32)
    dev = torch.device("cuda:0")
    pad = 4096
    n_o, n_l = B * Hq * D, B * Hq
    nbytes = fa.fa_decode_workspace_bytes(B, Hq, D, ns)
    o_buf = torch.full((pad + n_o + pad,), 7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((pad + n_l + pad,), 7.0, dtype=torch.float32, device=dev)
    w_buf = torch.full((pad + nbytes + pad,), 0xA5, dtype=torch.uint8, device=dev)
    o = o_buf[pad:pad + n_o].view(B, 1, Hq, D)
    lse = l_buf[pad:pad + n_l].view(B, Hq)
    fa.fa_decode_splitkv(*_dev(q, kc, vc, lens), num_splits=ns, workspace=w_buf[pad:pad + nbytes],
                         out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(l_buf[:pad] == 7.0) and torch.all(l_buf[-pad:] == 7.0)
    assert torch.all(w_buf[:pad] == 0xA5) and torch.all(w_buf[-pad:] == 0xA5)
    o_ref, lse_ref = oracle.decode(q, kc, vc, lens, scale=1 / math.sqrt(D))
    _check(o, lse, o_ref, lse_ref)


def test_decode_rejects_bad_arguments(fa):
    q, kc, vc, lens = _dev(*inputs.make_decode(2, 8, 2, 128, 256, 1, 256, seed=83))
    with pytest.raises(fa.FaError) as e:
        fa.fa_decode_splitkv(q, kc, vc, lens, num_splits=4,
                             workspace=torch.empty(16, dtype=torch.uint8, device="cuda:0"))
    assert e.value.status == 3  # FA_ERR_WORKSPACE
    with pytest.raises(fa.FaError) as e:
        fa.fa_decode_splitkv(q[:, :, :7].contiguous(), kc, vc, lens)  # 7 heads over 2
    assert e.value.status == 1  # FA_ERR_INVALID_ARG
