"""Failure detection on the GPU without a fault: a barrier wait that nothing completes runs
out, and the host reads the timeout.

fa_selftest_bounded_wait runs the same bounded wait that every kernel's barrier waits go
through.  One warp waits on a phase that never completes. After the wait limit (2 s) it
records FA_ERR_TIMEOUT in the device status word and raises the CTA's abort flag. A second
warp, waiting on its own such barrier, must leave on that flag before its own limit. The
context must stay usable afterwards: a forward call that follows still matches the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_20_gb300 import inputs

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_TIMEOUT = 0, 5


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_20_gb300 as fa_mod
    from exact_tiled_attention_20_gb300 import build

    build.build_library()
    fa_mod.load()
    return fa_mod


def test_wait_runs_out_and_is_reported(fa):
    dev = torch.device("cuda:0")
    assert fa.fa_last_device_status() == FA_OK  # nothing pending before the test
    result = torch.zeros(4, dtype=torch.int32, device=dev)
    assert fa.fa_selftest_bounded_wait(result) == FA_OK
    torch.cuda.synchronize()
    gave_up, left_on_flag, waited_ms = result.cpu().tolist()[:3]
    assert gave_up == 1, "the wait on a phase nothing completes did not give up"
    assert left_on_flag == 1, "the second warp did not leave on the CTA abort flag"
    assert 1900 <= waited_ms <= 10000, f"waited {waited_ms} ms against a 2 s limit"
    assert fa.fa_last_device_status() == FA_ERR_TIMEOUT
    assert fa.fa_last_device_status() == FA_OK  # reading the status cleared it

    # The context is still usable: a small forward matches the fp64 oracle.
    q, k, v = inputs.make_qkv(1, 200, 200, 2, 1, 64, seed=4242)
    o, lse = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.fwd(q, k, v, scale=1 / math.sqrt(64), causal=True)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= 1e-2
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3
