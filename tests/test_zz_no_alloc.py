"""fa_decode_splitkv_noalloc: the decode entry point for callers that cannot allocate
device memory (a plugin inside a host runtime that owns all device allocations, or a
serving loop that must never call cudaMalloc).  It keeps its scratch in a fixed array in
the library's device image.  Called here through the C ABI; its output must match the
regular fa_decode_splitkv (which takes a caller-allocated workspace) and the CPU oracle's
decode (the fp64 definition) within the decode tolerances, on two calls in a row (the
second reuses the scratch the first left behind).

This file is collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_20_gb300 import inputs

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3
SCRATCH_BYTES = 8 << 20  # FA_DECODE_NOALLOC_SCRATCH_BYTES in include/fa.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_20_gb300 import build

    raw = ctypes.CDLL(build.build_library())
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    raw.fa_decode_splitkv_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, I, P]
    raw.fa_decode_splitkv_noalloc.restype = I
    raw.fa_decode_workspace_bytes.argtypes = [I, I, I, I]
    raw.fa_decode_workspace_bytes.restype = ctypes.c_size_t
    return raw


def _noalloc(lib, q, kc, vc, lens, o, lse, ns):
    B, _, Hq, D = q.shape
    Smax, Hkv = kc.shape[1], kc.shape[2]
    return lib.fa_decode_splitkv_noalloc(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), lens.data_ptr(), o.data_ptr(), lse.data_ptr(),
        B, Hq, Hkv, D, Smax, 1.0 / math.sqrt(D), ns, 0,
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_decode_matches_workspace_decode_twice(lib):
    import exact_tiled_attention_20_gb300 as fa

    dev = torch.device("cuda:0")
    cases = [(inputs.make_decode(4, 32, 8, 128, 4096, 100, 4096, seed=91), 0),
             (inputs.make_decode(3, 16, 2, 128, 2500, 1, 2500, seed=92), 7),
             (inputs.make_decode(3, 16, 4, 96, 2000, 1, 2000, seed=94), 5),   # kv heads in fours
             (inputs.make_decode(2, 8, 2, 64, 3000, 1, 3000, seed=95), 0)]    # 256-key steps, pairs
    for (qh, kh, vh, lh), ns in cases:
        o_def, lse_def = oracle.decode(qh, kh, vh, lh, scale=1.0 / math.sqrt(qh.shape[-1]))
        q, kc, vc, lens = (t.to(dev) for t in (qh, kh, vh, lh))
        o_ref, lse_ref = fa.fa_decode_splitkv(q, kc, vc, lens, num_splits=ns)
        for _ in range(2):
            o = torch.full_like(q, float("nan"))
            lse = torch.full((q.shape[0], q.shape[2]), float("nan"), dtype=torch.float32, device=dev)
            assert _noalloc(lib, q, kc, vc, lens, o, lse, ns) == 0
            torch.cuda.synchronize()
            assert (o.float() - o_ref.float()).abs().max().item() <= O_TOL
            assert (lse - lse_ref).abs().max().item() <= LSE_TOL
            o_np = o.float().cpu().numpy()[:, 0]
            assert np.abs(o_np - o_def).max() <= O_TOL
            assert np.abs(lse.cpu().numpy() - lse_def).max() <= LSE_TOL


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    dev = torch.device("cuda:0")
    q, kc, vc, lens = (t.to(dev) for t in inputs.make_decode(2, 8, 2, 128, 4096, 1, 4096, seed=93))
    o = torch.empty_like(q)
    lse = torch.empty((2, 8), dtype=torch.float32, device=dev)
    # a split count whose partials need more than the scratch holds
    ns = 2048
    assert lib.fa_decode_workspace_bytes(2, 8, 128, ns) > SCRATCH_BYTES
    assert _noalloc(lib, q, kc, vc, lens, o, lse, ns) == 3  # FA_ERR_WORKSPACE
