"""Exact tiled attention for NVIDIA GB300 (sm_103a).

The product is the C library ``libfa.so`` declared in ``include/fa.h``; this package is
its thin Python binding (``_lib``), the in-tree build (``build``) and the seeded input
generators (``inputs``).  The binding's names mirror the C entry points:

* ``fa_fwd`` -- exact attention forward with per-row log-sum-exp;
* ``fa_fwd(..., window=(left, right))`` -- sliding-window local attention (fa_fwd_window);
* ``fa_fwd_varlen`` -- variable-length batches packed along the rows (cu_seqlens);
* ``fa_decode_splitkv`` -- split-KV (Flash-Decoding) single-token decode;
* ``fa_decode_splitkv_multi`` -- the same with several query tokens per sequence;
* ``fa_decode_splitkv_paged`` -- the same over a paged KV cache with a block table;
* ``fa_decode_splitkv_noalloc`` -- decode with library-owned scratch (no workspace);
* ``fa_decode_workspace_bytes``, ``fa_decode_default_splits``, ``fa_status_string``,
  ``fa_last_device_status``, ``fa_selftest_bounded_wait`` (the bounded-wait self-test).

Importing the package does not load the library; the first call does, and raises if
``libfa.so`` has not been built.
"""
from ._lib import (FA_BF16, FA_FP16, FaError, fa_decode_default_splits, fa_decode_splitkv,
                   fa_decode_splitkv_multi, fa_decode_splitkv_noalloc, fa_decode_splitkv_paged, fa_decode_workspace_bytes,
                   fa_fwd, fa_fwd_varlen, fa_last_device_status, fa_selftest_bounded_wait,
                   fa_status_string, library_path, load)

__all__ = [
    "FA_BF16", "FA_FP16", "FaError", "fa_fwd", "fa_fwd_varlen", "fa_decode_splitkv", "fa_decode_splitkv_paged",
    "fa_decode_splitkv_noalloc", "fa_decode_splitkv_multi", "fa_decode_workspace_bytes", "fa_decode_default_splits",
    "fa_status_string", "fa_last_device_status", "fa_selftest_bounded_wait", "library_path", "load",
]
