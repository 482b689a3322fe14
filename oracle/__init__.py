"""CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product path (``exact_tiled_attention_20_gb300``) never does:
it has no CPU fallback and fails loudly when its CUDA library is missing.

The arithmetic lives in ``fa_oracle.c`` (fp64, materialised scores, two-pass softmax);
this module only builds it with the host C compiler and marshals arrays.  It follows
the pages as cited in that file's header:

* ``fwd``      -- flash_attn_func semantics (page "flash-attention-v100", "How to use
  FlashAttention"), bottom-right causal mask ("Changelog", "2.1: Change behavior of
  causal flag"), grouped-query head map (same docstring, 6 Q heads over 2 KV heads).
* ``decode``   -- one query token over a KV cache with per-sequence lengths
  (flash_attn_with_kvcache, cache_seqlens).
* ``partial``  -- attention over a key sub-range, one Flash-Decoding split
  (page "flash attention-2 github", steps 1-2).
* ``combine``  -- the log-sum-exp merge of partials (same snippet, step 3; the formula
  is the exact identity over a partition of the key set).
* ``decode_paged`` -- decode over a paged KV cache addressed through a block table
  (flash_attn_with_kvcache block_table; "Changelog", "2.5: Paged KV cache").
* ``decode_multi`` -- several query tokens per sequence over a KV cache, bottom-right
  causal (flash_attn_with_kvcache with seqlen_q > 1).
* ``fwd_varlen`` -- variable-length batches: independent sequences packed along rows
  (flash_attn_varlen_func; "Changelog", "2.0").
* ``fwd(..., window=(left, right))`` -- sliding-window local attention (page
  "flash-attention-v100", flash_attn_func window_size; "Changelog", "2.3").

Parity pins: every function is pinned in ``tests/test_oracle.py`` against closed forms,
the pages' worked mask examples, library routines and brute force (see that file).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

BF16, FP16, F32, F64 = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into liboracle.so with the host C compiler (portable C11)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lpthread", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # FA_ORACLE_LIB points the pins at a deliberately broken copy of the oracle
            # (tests/test_oracle_mutations.py); normally the library built here is used.
            path = os.environ.get("FA_ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            L, D_, P, I = ctypes.c_long, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.fa_oracle_fwd.argtypes = [P, P, P, I, L, L, L, L, L, L, D_, I, L, L, P, L, P, P, I]
            lib.fa_oracle_fwd.restype = I
            lib.fa_oracle_partial.argtypes = [P, P, P, I, L, L, L, L, L, L, L, L, L, D_, P, P]
            lib.fa_oracle_partial.restype = I
            lib.fa_oracle_decode.argtypes = [P, P, P, I, P, L, L, L, L, L, D_, P, P, I]
            lib.fa_oracle_decode.restype = I
            lib.fa_oracle_combine.argtypes = [P, P, L, L, P, P]
            lib.fa_oracle_combine.restype = I
            lib.fa_oracle_decode_paged.argtypes = [P, P, P, I, P, P, L, L, L, L, L, L, L, D_, P,
                                                   P, I]
            lib.fa_oracle_decode_paged.restype = I
            _lib = lib
    return _lib


def _as_input(x):
    """Return (contiguous numpy array, dtype code) holding the exact stored values.

    bf16/fp16 torch tensors are passed as their raw 16-bit patterns (widened exactly
    inside the oracle); float32/float64 arrays are passed as they are.
    """
    try:
        import torch  # plumbing only: reading the stored bits of a CPU tensor

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float16:
                return x.view(torch.int16).numpy().view(np.uint16), FP16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            if x.dtype == torch.float64:
                return x.numpy(), F64
            raise TypeError(f"unsupported tensor dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    raise TypeError(f"unsupported array dtype {a.dtype}; pass torch bf16/fp16 or float32/64")


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def fwd(q, k, v, scale: float, causal: bool = False, rows=None, nthreads=None,
        window=(-1, -1)):
    """Exact attention forward, fp64.

    q: [B, Sq, Hq, D], k/v: [B, Sk, Hkv, D] (same dtype).  ``window=(left, right)``
    restricts query i to keys i+Sk-Sq-left .. i+Sk-Sq+right (-1: unbounded).
    Returns ``(o, lse)``:
    with ``rows=None`` o is [B, Sq, Hq, D] and lse is [B, Hq, Sq]; with ``rows`` an
    (n, 3) integer array of (b, h, i) it returns o [n, D] and lse [n].
    """
    qa, dt = _as_input(q)
    ka, dk = _as_input(k)
    va, dv = _as_input(v)
    if not (dt == dk == dv):
        raise TypeError("q, k, v must share one dtype")
    B, Sq, Hq, D = qa.shape
    Bk, Sk, Hkv, Dk = ka.shape
    if va.shape != ka.shape or Bk != B or Dk != D:
        raise ValueError("shape mismatch")
    if rows is None:
        o = np.zeros((B, Sq, Hq, D), np.float64)
        lse = np.zeros((B, Hq, Sq), np.float64)
        rp, nr = None, 0
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        o = np.zeros((r.shape[0], D), np.float64)
        lse = np.zeros((r.shape[0],), np.float64)
        rp, nr = _ptr(r), r.shape[0]
    wl, wr = (int(window[0]), int(window[1]))
    rc = _load().fa_oracle_fwd(_ptr(qa), _ptr(ka), _ptr(va), dt, B, Sq, Sk, Hq, Hkv, D,
                               float(scale), int(bool(causal)), wl, wr, rp, nr, _ptr(o),
                               _ptr(lse), _threads(nthreads))
    if rc:
        raise ValueError(f"fa_oracle_fwd failed with code {rc}")
    return o, lse


def decode(q, k_cache, v_cache, kv_lens, scale: float, nthreads=None):
    """Single-token attention over a KV cache.

    q: [B, Hq, D] (or [B, 1, Hq, D]); k_cache/v_cache: [B, Smax, Hkv, D];
    kv_lens: B integers.  Returns o [B, Hq, D], lse [B, Hq] in fp64.
    """
    qa, dt = _as_input(q)
    ka, _ = _as_input(k_cache)
    va, _ = _as_input(v_cache)
    if qa.ndim == 4:
        qa = qa.reshape(qa.shape[0], qa.shape[2], qa.shape[3])
    B, Hq, D = qa.shape
    _, Smax, Hkv, _ = ka.shape
    lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32).reshape(-1))
    o = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = _load().fa_oracle_decode(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(lens), B, Hq, Hkv, D,
                                  Smax, float(scale), _ptr(o), _ptr(lse), _threads(nthreads))
    if rc:
        raise ValueError(f"fa_oracle_decode failed with code {rc}")
    return o, lse


def partial(q, k_cache, v_cache, b: int, h: int, j0: int, j1: int, scale: float):
    """Attention of query (b, h) over cache keys [j0, j1): one split's (o [D], lse)."""
    qa, dt = _as_input(q)
    ka, _ = _as_input(k_cache)
    va, _ = _as_input(v_cache)
    if qa.ndim == 4:
        qa = qa.reshape(qa.shape[0], qa.shape[2], qa.shape[3])
    B, Hq, D = qa.shape
    _, Smax, Hkv, _ = ka.shape
    o = np.zeros((D,), np.float64)
    lse = np.zeros((1,), np.float64)
    rc = _load().fa_oracle_partial(_ptr(qa), _ptr(ka), _ptr(va), dt, B, Hq, Hkv, D, Smax, b, h,
                                   j0, j1, float(scale), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"fa_oracle_partial failed with code {rc}")
    return o, float(lse[0])


def combine(o_parts, lse_parts):
    """Log-sum-exp merge of n partials: o_parts [n, D], lse_parts [n] -> (o [D], lse)."""
    op = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    lp = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64).reshape(-1))
    n, D = op.shape
    o = np.zeros((D,), np.float64)
    lse = np.zeros((1,), np.float64)
    rc = _load().fa_oracle_combine(_ptr(op), _ptr(lp), n, D, _ptr(o), _ptr(lse))
    if rc:
        raise ValueError(f"fa_oracle_combine failed with code {rc}")
    return o, float(lse[0])


def decode_paged(q, k_pages, v_pages, block_table, kv_lens, scale: float, nthreads=None):
    """Decode over a paged cache: k_pages/v_pages [num_pages, page_size, Hkv, D];
    block_table [B, max_pages] ints; kv_lens [B].  Returns o [B, Hq, D], lse [B, Hq]."""
    qa, dt = _as_input(q)
    ka, _ = _as_input(k_pages)
    va, _ = _as_input(v_pages)
    if qa.ndim == 4:
        qa = qa.reshape(qa.shape[0], qa.shape[2], qa.shape[3])
    B, Hq, D = qa.shape
    num_pages, page_size, Hkv, _ = ka.shape
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32).reshape(-1))
    o = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = _load().fa_oracle_decode_paged(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(bt), _ptr(lens), B,
                                        Hq, Hkv, D, num_pages, page_size, bt.shape[1],
                                        float(scale), _ptr(o), _ptr(lse), _threads(nthreads))
    if rc:
        raise ValueError(f"fa_oracle_decode_paged failed with code {rc}")
    return o, lse


def fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool = False,
               window=(-1, -1), nthreads=None):
    """Variable-length batch (flash_attn_varlen_func; page "flash-attention-v100",
    "Changelog", "2.0"): sequence b is the independent attention problem over query rows
    cu_q[b]:cu_q[b+1] and key rows cu_k[b]:cu_k[b+1] of packed [total, H, D] tensors.
    Returns o [total_q, Hq, D] and lse [Hq, total_q], fp64."""
    cq = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    ck = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    total_q, Hq, D = q.shape
    o = np.zeros((total_q, Hq, D), np.float64)
    lse = np.full((Hq, total_q), -np.inf)
    for b in range(len(cq) - 1):
        sq, sk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
        if sq <= 0:
            continue
        if sk <= 0:
            continue  # no keys: zero output, -inf log-sum-exp
        ob, lb = fwd(q[None, cq[b]:cq[b + 1]], k[None, ck[b]:ck[b + 1]], v[None, ck[b]:ck[b + 1]],
                     scale=scale, causal=causal, window=window, nthreads=nthreads)
        o[cq[b]:cq[b + 1]] = ob[0]
        lse[:, cq[b]:cq[b + 1]] = lb[0]
    return o, lse


def decode_multi(q, k_cache, v_cache, kv_lens, scale: float, causal: bool = True, nthreads=None):
    """Several query tokens per sequence over a KV cache (flash_attn_with_kvcache with
    seqlen_q > 1; page "flash-attention-v100", "How to use FlashAttention"): the Sq
    queries of sequence b attend to cache keys [0, kv_lens[b]), and with ``causal`` the
    mask is aligned to the bottom-right corner, so query s sees keys
    j <= kv_lens[b] - Sq + s.  q [B, Sq, Hq, D]; returns o [B, Sq, Hq, D] and
    lse [B, Hq, Sq] in fp64."""
    B, Sq, Hq, D = q.shape
    lens = [int(x) for x in np.asarray(kv_lens).reshape(-1)]
    o = np.zeros((B, Sq, Hq, D), np.float64)
    lse = np.full((B, Hq, Sq), -np.inf)
    for b in range(B):
        if lens[b] <= 0:
            continue
        ob, lb = fwd(q[b:b + 1], k_cache[b:b + 1, :lens[b]], v_cache[b:b + 1, :lens[b]], scale=scale,
                     causal=causal, nthreads=nthreads)
        o[b] = ob[0]
        lse[b] = lb[0]
    return o, lse
