"""The C ABI on the host (no GPU): the library loads, exports every entry point that
include/fa.h declares, and validates its arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_20_gb300 import build

    path = build.build_library()
    import exact_tiled_attention_20_gb300 as fa

    return fa.load(), path


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    return re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", src)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"fa_fwd", "fa_decode_splitkv", "fa_decode_workspace_bytes",
            "fa_decode_default_splits", "fa_status_string", "fa_last_device_status"} <= names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib[1])
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in include/fa.h but not exported"


def test_status_strings(lib):
    L = lib[0]
    for code in range(6):
        assert L.fa_status_string(code).startswith(b"FA_")
    assert L.fa_status_string(99) == b"unknown fa_status"


def test_workspace_bytes(lib):
    L = lib[0]
    rows = 8 * 32 * 16
    expect = (rows * 128 * 4 + 255) // 256 * 256 + (rows * 4 + 255) // 256 * 256
    assert L.fa_decode_workspace_bytes(8, 32, 128, 16) == expect
    assert L.fa_decode_workspace_bytes(0, 32, 128, 16) == 0
    assert L.fa_decode_workspace_bytes(8, 32, 128, 0) == 0


def test_default_splits_policy(lib):
    L = lib[0]
    # 8 items per SM over B*Hkv groups, chunks of at least 256 keys, at least 1
    assert L.fa_decode_default_splits(8, 8, 32768, 152) == 19
    assert L.fa_decode_default_splits(8, 8, 1000, 152) == 4
    assert L.fa_decode_default_splits(1, 1, 100, 152) == 1
    assert L.fa_decode_default_splits(256, 8, 32768, 152) == 1
    assert L.fa_decode_default_splits(0, 8, 32768, 152) == -1


FAKE = 1 << 20  # a 16-byte-aligned non-null address; validation rejects before any use


@pytest.mark.parametrize("args,code", [
    # (q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, scale, causal, dtype) -> status
    ((0, FAKE, FAKE, FAKE, None, 1, 8, 8, 2, 2, 64, 0.1, 0, 0), 1),          # null q
    ((FAKE + 8, FAKE, FAKE, FAKE, None, 1, 8, 8, 2, 2, 64, 0.1, 0, 0), 1),   # misaligned q
    ((FAKE, FAKE, FAKE, FAKE, FAKE + 2, 1, 8, 8, 2, 2, 64, 0.1, 0, 0), 1),   # misaligned lse
    ((FAKE, FAKE, FAKE, FAKE, None, 0, 8, 8, 2, 2, 64, 0.1, 0, 0), 1),       # B = 0
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 8, 8, 3, 2, 64, 0.1, 0, 0), 1),       # Hq % Hkv
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 8, 8, 2, 2, 64, float("nan"), 0, 0), 1),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 8, 8, 2, 2, 80, 0.1, 0, 0), 2),       # head dim 80
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 8, 8, 2, 2, 64, 0.1, 0, 7), 2),       # dtype
])
def test_fwd_argument_validation(lib, args, code):
    assert lib[0].fa_fwd(*args, None) == code


def test_decode_argument_validation(lib):
    L = lib[0]
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 256, 0.1, 4, FAKE, 1 << 30, 0, None]
    assert L.fa_decode_splitkv(*base[:3], None, *base[4:]) == 1          # null kv_lens
    bad = list(base); bad[7] = 7                                         # 7 heads over 2
    assert L.fa_decode_splitkv(*bad) == 1
    bad = list(base); bad[9] = 80                                        # head dim 80
    assert L.fa_decode_splitkv(*bad) == 2
    bad = list(base); bad[9] = 512                                       # head dim 512
    assert L.fa_decode_splitkv(*bad) == 2
    bad = list(base); bad[7] = 64; bad[8] = 2                            # group of 32 > 16
    assert L.fa_decode_splitkv(*bad) == 2
    bad = list(base); bad[6] = 1024; bad[7] = 256; bad[8] = 256; bad[10] = 1 << 20
    assert L.fa_decode_splitkv(*bad) == 2                                # 2^31 tiles over all pairs


def test_selftest_argument_validation(lib):
    L = lib[0]
    L.fa_selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert L.fa_selftest_bounded_wait(None, None) == 1       # null result
    assert L.fa_selftest_bounded_wait(FAKE + 4, None) == 1   # misaligned result


def test_valid_call_without_a_device_fails_loudly(lib):
    """With arguments that pass validation but no usable GPU, the call reports
    FA_ERR_CUDA; there is no CPU fallback."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib[0].fa_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 8, 2, 2, 64, 0.1, 0, 0, None) == 4


def test_binding_rejects_cpu_tensors():
    import torch

    import exact_tiled_attention_20_gb300 as fa

    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fa.fa_fwd(q, q, q)


def test_noalloc_decode_validates_like_the_workspace_decode(lib):
    """fa_decode_splitkv_noalloc runs the same argument checks as fa_decode_splitkv before
    it looks at its scratch: an invalid or unsupported call gets the same status."""
    raw = ctypes.CDLL(lib[1])
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    raw.fa_decode_splitkv_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, I, P]
    raw.fa_decode_splitkv_noalloc.restype = I
    L = lib[0]
    # (q, k, v, kv_lens, o, lse, B, Hq, Hkv, D, Smax, scale, num_splits)
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 256, 0.1, 4]
    cases = []
    bad = list(base); bad[0] = None; cases.append((bad, 1))             # null q
    bad = list(base); bad[3] = None; cases.append((bad, 1))             # null kv_lens
    bad = list(base); bad[9] = 80; cases.append((bad, 2))               # head dim 80
    bad = list(base); bad[7] = 3; cases.append((bad, 1))                # 8 heads over 3
    bad = list(base); bad[7] = 64; bad[8] = 2; cases.append((bad, 2))   # group of 32 > 16
    # an unsupported size whose partials would also overflow the scratch
    bad = list(base); bad[9] = 4096; bad[12] = 4096; cases.append((bad, 2))
    for args, code in cases:
        assert raw.fa_decode_splitkv_noalloc(*args, 0, None) == code, args
        ws = [FAKE, 1 << 30, 0, None]
        assert L.fa_decode_splitkv(*args, *ws) == code, args
