// fa_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Arguments of one forward call after validation.
struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    int B, Sq, Sk, Hq, Hkv, D;
    float scale;
    int causal;
    int window_left, window_right;  // -1: unbounded
    const int32_t* cu_q;            // variable-length batch: null for [B, S, H, D]
    const int32_t* cu_k;
    int total_q, total_k;
    bool bf16;
    int num_sms;
    int* dev_status;
};

// Arguments of one split-KV decode call after validation.
struct DecodeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* kv_lens;
    void* o;
    float* lse;
    int B, Hq, Hkv, D, Smax;
    float scale;
    int num_splits;
    float* o_part;    // [B, Hq, num_splits, D]
    float* lse_part;  // [B, Hq, num_splits]
    int sq, causal;              // query tokens per sequence (1 = plain decode)
    const int32_t* block_table;  // null for a contiguous cache
    int num_pages, page_size, max_pages;  // paged pool (Smax = page_size * max_pages)
    bool bf16;
    int num_sms;
    int* dev_status;
};

// Encodes a 4-D tiled TMA map over a [dim3][dim2][dim1][dim0] row-major 16-bit tensor
// with a (64, 1, box_rows, 1) box and 128-byte swizzling.  Returns false on failure.
bool encode_tmap_4d(CUtensorMap* map, const void* base, bool bf16, uint64_t dim0, uint64_t dim1,
                    uint64_t dim2, uint64_t dim3, uint32_t box_rows);

// Same with an explicit (64, box1, box2, 1) box.
bool encode_tmap_4d_box(CUtensorMap* map, const void* base, bool bf16, uint64_t dim0,
                        uint64_t dim1, uint64_t dim2, uint64_t dim3, uint32_t box1,
                        uint32_t box2);

// Per-head-dim forward launchers (one translation unit each, compiled in parallel).
fa_status launch_fwd_d64(const FwdArgs& a, cudaStream_t s);
fa_status launch_fwd_d96(const FwdArgs& a, cudaStream_t s);
fa_status launch_fwd_d128(const FwdArgs& a, cudaStream_t s);
fa_status launch_fwd_d256(const FwdArgs& a, cudaStream_t s);

fa_status launch_decode(const DecodeArgs& a, cudaStream_t s);
fa_status launch_decode_d64(const DecodeArgs& a, cudaStream_t s);
fa_status launch_decode_d96(const DecodeArgs& a, cudaStream_t s);
fa_status launch_decode_d128(const DecodeArgs& a, cudaStream_t s);
fa_status launch_decode_d256(const DecodeArgs& a, cudaStream_t s);

// Argument checks shared by every decode entry point (pointers, alignment, sizes, dtype,
// head dim, group size); FA_OK or the status the entry point returns.  Host only.
fa_status decode_check_args(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* kv_lens, const void* o, const float* lse, int B, int Sq,
                            int Hq, int Hkv, int D, int Smax, float scale, fa_dtype dtype);

// Sets the dynamic shared-memory limit of `func` once per device.
bool ensure_smem_attr(const void* func, int bytes, int* done_flags);

}  // namespace fa
