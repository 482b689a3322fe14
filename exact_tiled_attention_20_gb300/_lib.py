"""ctypes binding of libfa.so -- argument marshalling only.

Every name here mirrors an entry point of include/fa.h.  Tensors are PyTorch CUDA tensors
(PyTorch provides device memory and streams); all arithmetic runs in the library's CUDA
kernels.  There is no CPU fallback: if libfa.so is missing or a call fails, an exception
is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_WORKSPACE, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(6)
FA_BF16, FA_FP16 = 0, 1

_DTYPE = {torch.bfloat16: FA_BF16, torch.float16: FA_FP16}

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {fa_status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load():
    """Loads libfa.so (raising if it has not been built) and declares the signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, P]
        lib.fa_fwd.restype = I
        lib.fa_fwd_window.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, I, P]
        lib.fa_fwd_window.restype = I
        lib.fa_decode_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_decode_workspace_bytes.restype = SZ
        lib.fa_decode_default_splits.argtypes = [I, I, I, I]
        lib.fa_decode_default_splits.restype = I
        lib.fa_decode_splitkv.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, P, SZ, I, P]
        lib.fa_decode_splitkv.restype = I
        lib.fa_status_string.argtypes = [I]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_last_device_status.argtypes = []
        lib.fa_last_device_status.restype = I
        lib.fa_selftest_bounded_wait.argtypes = [P, P]
        lib.fa_selftest_bounded_wait.restype = I
        _lib = lib
        return lib


def _check_cuda(name, t, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def fa_status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_last_device_status() -> int:
    """Reads and clears the device status word (synchronises the device)."""
    return int(load().fa_last_device_status())


def fa_selftest_bounded_wait(result, stream=None) -> int:
    """Enqueues the bounded-wait self-test (see include/fa.h); result is a CUDA int32
    tensor of 3 elements.  Returns the launch status."""
    _check_cuda("result", result, torch.int32)
    if result.numel() < 3:
        raise ValueError("result needs 3 elements")
    return int(load().fa_selftest_bounded_wait(ctypes.c_void_p(result.data_ptr()),
                                               ctypes.c_void_p(_stream_handle(stream))))


def fa_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
           return_lse: bool = True, stream=None, window=None):
    """Exact attention forward through fa_fwd (or fa_fwd_window when ``window=(left,
    right)`` is given; -1 = unbounded side).  q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D].

    Returns (o, lse): o like q, lse fp32 [B, Hq, Sq] (None if return_lse is False and no
    lse buffer was given).  scale defaults to 1/sqrt(D).
    """
    if q.dtype not in _DTYPE:
        raise TypeError("q/k/v must be bf16 or fp16")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda("out", out, q.dtype)
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError("out must have q's shape")
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_cuda("lse", lse, torch.float32)
        if tuple(lse.shape) != (B, Hq, Sq):
            raise ValueError("lse must be [B, Hq, Sq]")
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        lp = lse.data_ptr() if lse is not None else None
        if window is None:
            st = load().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lp, B, Sq,
                               Sk, Hq, Hkv, D, sc, int(bool(causal)), _DTYPE[q.dtype],
                               _stream_handle(stream))
        else:
            st = load().fa_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lp,
                                      B, Sq, Sk, Hq, Hkv, D, sc, int(bool(causal)), int(window[0]),
                                      int(window[1]), _DTYPE[q.dtype], _stream_handle(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_window" if window is not None else "fa_fwd")
    return out, lse


def fa_decode_workspace_bytes(B: int, Hq: int, D: int, num_splits: int) -> int:
    return int(load().fa_decode_workspace_bytes(B, Hq, D, num_splits))


def fa_decode_default_splits(B: int, Hkv: int, max_kv_len: int, num_sms: int = 0) -> int:
    return int(load().fa_decode_default_splits(B, Hkv, max_kv_len, num_sms))


def fa_decode_splitkv(q, k_cache, v_cache, kv_lens, scale: float | None = None,
                      num_splits: int = 0, workspace=None, out=None, lse=None,
                      return_lse: bool = True, stream=None):
    """Split-KV decode through fa_decode_splitkv.

    q [B,1,Hq,D]; k_cache/v_cache [B,Smax,Hkv,D]; kv_lens int32 [B] on the device.
    workspace: a CUDA uint8 tensor of at least fa_decode_workspace_bytes(...) bytes, or
    None to allocate one with PyTorch.  Returns (o [B,1,Hq,D], lse [B,Hq]).
    """
    if q.dtype not in _DTYPE:
        raise TypeError("q/k_cache/v_cache must be bf16 or fp16")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("kv_lens", kv_lens, torch.int32)
    if q.dim() == 3:
        q = q.unsqueeze(1)
    B, one, Hq, D = q.shape
    if one != 1:
        raise ValueError("decode takes one query token per sequence: q [B, 1, Hq, D]")
    Bk, Smax, Hkv, Dk = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or Bk != B or Dk != D:
        raise ValueError("cache shape mismatch")
    if kv_lens.numel() != B:
        raise ValueError("kv_lens must hold B lengths")
    lib = load()
    with torch.cuda.device(q.device):
        ns = int(num_splits) if num_splits and num_splits > 0 else \
            lib.fa_decode_default_splits(B, Hkv, Smax, 0)
        if ns <= 0:
            raise FaError(FA_ERR_CUDA, "fa_decode_default_splits")
        ns = min(ns, Smax)
        need = lib.fa_decode_workspace_bytes(B, Hq, D, ns)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        _check_cuda("workspace", workspace)
        ws_bytes = workspace.numel() * workspace.element_size()
        if out is None:
            out = torch.empty_like(q)
        _check_cuda("out", out, q.dtype)
        if lse is None and return_lse:
            lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
        if lse is not None:
            _check_cuda("lse", lse, torch.float32)
        sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
        st = lib.fa_decode_splitkv(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   kv_lens.data_ptr(), out.data_ptr(),
                                   lse.data_ptr() if lse is not None else None, B, Hq, Hkv, D,
                                   Smax, sc, ns, workspace.data_ptr(), ws_bytes, _DTYPE[q.dtype],
                                   _stream_handle(stream))
    if st != FA_OK:
        raise FaError(st, "fa_decode_splitkv")
    return out, lse


_noalloc_declared = False


def fa_decode_splitkv_noalloc(q, k_cache, v_cache, kv_lens, scale: float | None = None,
                              num_splits: int = 0, out=None, lse=None, stream=None):
    """fa_decode_splitkv_noalloc: split-KV decode without a caller workspace, for callers
    that cannot allocate device memory (the partials go to a fixed scratch array inside
    the library; see include/fa.h for its size limit and sharing rules).  Output tensors
    must be given or are created here with PyTorch."""
    global _noalloc_declared
    lib = load()
    if not _noalloc_declared:
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_decode_splitkv_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, I, P]
        lib.fa_decode_splitkv_noalloc.restype = I
        _noalloc_declared = True
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("kv_lens", kv_lens, torch.int32)
    B, _, Hq, D = q.shape
    _, Smax, Hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        st = lib.fa_decode_splitkv_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           kv_lens.data_ptr(), out.data_ptr(), lse.data_ptr(), B,
                                           Hq, Hkv, D, Smax, sc, int(num_splits), _DTYPE[q.dtype],
                                           _stream_handle(stream))
    if st != FA_OK:
        raise FaError(st, "fa_decode_splitkv_noalloc")
    return out, lse


_paged_declared = False


def fa_decode_splitkv_paged(q, k_pages, v_pages, block_table, kv_lens, scale: float | None = None,
                            num_splits: int = 0, workspace=None, out=None, lse=None, stream=None):
    """Split-KV decode over a paged cache through fa_decode_splitkv_paged.

    q [B,1,Hq,D]; k_pages/v_pages [num_pages, page_size, Hkv, D]; block_table int32
    [B, max_pages_per_seq] and kv_lens int32 [B] on the device.  Returns (o, lse)."""
    global _paged_declared
    lib = load()
    if not _paged_declared:
        P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_decode_splitkv_paged.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P,
                                                SZ, I, P]
        lib.fa_decode_splitkv_paged.restype = I
        _paged_declared = True
    if q.dtype not in _DTYPE:
        raise TypeError("q/k_pages/v_pages must be bf16 or fp16")
    for name, t in (("q", q), ("k_pages", k_pages), ("v_pages", v_pages)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("block_table", block_table, torch.int32)
    _check_cuda("kv_lens", kv_lens, torch.int32)
    B, _, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    max_pages = block_table.shape[1]
    with torch.cuda.device(q.device):
        ns = int(num_splits) if num_splits and num_splits > 0 else \
            lib.fa_decode_default_splits(B, Hkv, page_size * max_pages, 0)
        if ns <= 0:
            raise FaError(FA_ERR_CUDA, "fa_decode_default_splits")
        ns = min(ns, page_size * max_pages)
        if workspace is None:
            workspace = torch.empty(lib.fa_decode_workspace_bytes(B, Hq, D, ns), dtype=torch.uint8,
                                    device=q.device)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
        sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
        st = lib.fa_decode_splitkv_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                         block_table.data_ptr(), kv_lens.data_ptr(), out.data_ptr(),
                                         lse.data_ptr(), B, Hq, Hkv, D, num_pages, page_size,
                                         max_pages, sc, ns, workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(),
                                         _DTYPE[q.dtype], _stream_handle(stream))
    if st != FA_OK:
        raise FaError(st, "fa_decode_splitkv_paged")
    return out, lse


_varlen_declared = False


def fa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool = False,
                  scale: float | None = None, window=(-1, -1), out=None, lse=None, stream=None):
    """Variable-length batch through fa_fwd_varlen: q [total_q, Hq, D], k/v [total_k, Hkv, D],
    cu_seqlens_q/k int32 [B+1] on the device.  Returns (o [total_q, Hq, D], lse [Hq, total_q])."""
    global _varlen_declared
    lib = load()
    if not _varlen_declared:
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.fa_fwd_varlen.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, I, P]
        lib.fa_fwd_varlen.restype = I
        _varlen_declared = True
    if q.dtype not in _DTYPE:
        raise TypeError("q/k/v must be bf16 or fp16")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _check_cuda("cu_seqlens_k", cu_seqlens_k, torch.int32)
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have B + 1 entries")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B,
                               total_q, total_k, Hq, Hkv, D, sc, int(bool(causal)), int(window[0]),
                               int(window[1]), _DTYPE[q.dtype], _stream_handle(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen")
    return out, lse


_multi_declared = False


def fa_decode_splitkv_multi(q, k_cache, v_cache, kv_lens, causal: bool = True,
                            scale: float | None = None, num_splits: int = 0, workspace=None,
                            out=None, lse=None, stream=None):
    """Several query tokens per sequence through fa_decode_splitkv_multi.
    q [B, Sq, Hq, D]; returns (o [B, Sq, Hq, D], lse [B, Hq, Sq])."""
    global _multi_declared
    lib = load()
    if not _multi_declared:
        P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_decode_splitkv_multi.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, SZ,
                                                I, P]
        lib.fa_decode_splitkv_multi.restype = I
        _multi_declared = True
    if q.dtype not in _DTYPE:
        raise TypeError("q/k_cache/v_cache must be bf16 or fp16")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _check_cuda(name, t, q.dtype)
    _check_cuda("kv_lens", kv_lens, torch.int32)
    B, Sq, Hq, D = q.shape
    _, Smax, Hkv, _ = k_cache.shape
    with torch.cuda.device(q.device):
        ns = int(num_splits) if num_splits and num_splits > 0 else \
            lib.fa_decode_default_splits(B, Hkv, Smax, 0)
        ns = min(ns, Smax)
        if workspace is None:
            workspace = torch.empty(lib.fa_decode_workspace_bytes(B * Sq, Hq, D, ns),
                                    dtype=torch.uint8, device=q.device)
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
        sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
        st = lib.fa_decode_splitkv_multi(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                         kv_lens.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Sq,
                                         Hq, Hkv, D, Smax, sc, int(bool(causal)), ns,
                                         workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(),
                                         _DTYPE[q.dtype], _stream_handle(stream))
    if st != FA_OK:
        raise FaError(st, "fa_decode_splitkv_multi")
    return out, lse
