// fa_api.cu -- the C ABI: argument validation, TMA tensor-map encoding, dispatch, and the
// self-test of the bounded barrier wait.
//
// Nothing here allocates device memory.  Every call validates its arguments before it
// enqueues anything, launches on the caller's stream and returns without synchronising.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

// Sticky device status word written by kernels whose bounded waits give up.  Host code
// never dereferences the symbol: it resolves the device address per device.
__device__ int g_fa_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct DeviceInfo {
    int num_sms = 0;
    int* status = nullptr;  // device address of g_fa_device_status
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

bool device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.num_sms == 0) {
        int sms = 0;
        void* st = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0)
            return false;
        if (cudaGetSymbolAddress(&st, g_fa_device_status) != cudaSuccess) return false;
        d.status = static_cast<int*>(st);
        d.num_sms = sms;
    }
    *out = d;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bool encode_tmap_4d(CUtensorMap* map, const void* base, bool bf16, uint64_t dim0, uint64_t dim1,
                    uint64_t dim2, uint64_t dim3, uint32_t box_rows) {
    return encode_tmap_4d_box(map, base, bf16, dim0, dim1, dim2, dim3, 1, box_rows);
}

namespace {

// Encoded maps are a pure function of their arguments (address, dtype, extents, box), so
// the last maps encoded are kept and reused: a caller that runs the same shapes on the
// same buffers every step, such as an iterative decode loop, pays for the encoding once.
struct TmapKey {
    const void* base;
    uint64_t dims[4];
    uint32_t box1, box2;
    int bf16;
    bool operator==(const TmapKey& o) const {
        return base == o.base && dims[0] == o.dims[0] && dims[1] == o.dims[1] &&
               dims[2] == o.dims[2] && dims[3] == o.dims[3] && box1 == o.box1 && box2 == o.box2 &&
               bf16 == o.bf16;
    }
};

struct TmapEntry {
    bool used = false;
    TmapKey key;
    CUtensorMap map;
};

constexpr int kTmapCacheSlots = 256;  // direct-mapped
TmapEntry g_tmap_cache[kTmapCacheSlots];
std::mutex g_tmap_mu;

uint32_t tmap_slot(const TmapKey& k) {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    for (int i = 0; i < 4; ++i) h = (h ^ k.dims[i]) * 0x100000001B3ull;
    h = (h ^ ((uint64_t)k.box1 << 32 | k.box2)) * 0x100000001B3ull;
    h ^= (uint64_t)k.bf16;
    return (uint32_t)(h >> 40) % kTmapCacheSlots;
}

}  // namespace

bool encode_tmap_4d_box(CUtensorMap* map, const void* base, bool bf16, uint64_t dim0,
                        uint64_t dim1, uint64_t dim2, uint64_t dim3, uint32_t box1,
                        uint32_t box2) {
    const TmapKey key{base, {dim0, dim1, dim2, dim3}, box1, box2, bf16 ? 1 : 0};
    const uint32_t slot = tmap_slot(key);
    {
        std::lock_guard<std::mutex> lk(g_tmap_mu);
        const TmapEntry& e = g_tmap_cache[slot];
        if (e.used && e.key == key) {
            *map = e.map;
            return true;
        }
    }
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {dim0, dim1, dim2, dim3};
    const cuuint64_t strides[3] = {dim0 * 2, dim0 * dim1 * 2, dim0 * dim1 * dim2 * 2};
    const cuuint32_t box[4] = {64, box1, box2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    TmapEntry& e = g_tmap_cache[slot];
    e.used = true;
    e.key = key;
    e.map = *map;
    return true;
}

bool ensure_smem_attr(const void* func, int bytes, int* done_flags) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (__atomic_load_n(&done_flags[dev], __ATOMIC_ACQUIRE)) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return false;
    __atomic_store_n(&done_flags[dev], 1, __ATOMIC_RELEASE);
    return true;
}

// Self-test of the bounded wait that every kernel's barrier waits go through.  Warp 0
// waits on a barrier phase that nothing completes until the wait limit passes; it then
// records the timeout and raises the CTA abort flag.  Warp 1 starts its own such wait half
// a second later and must leave on that flag, before its own limit.  Lane 0 of each warp
// writes: result[0] = warp 0 gave up, result[1] = warp 1 left on the flag, result[2] =
// warp 0's wait in ms.
__global__ void __launch_bounds__(64, 1) selftest_bounded_wait_kernel(int* result, int* status) {
    __shared__ uint64_t bars[2];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtx wc{&abort_flag, status};
    if (warp == 1) {  // a bounded delay, so that warp 0's limit passes first
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < kWaitLimitNs / 4) {
        }
    }
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait(smem_u32(&bars[warp]), 0, wc);
    const uint64_t waited = globaltimer_ns() - t0;
    if (lane == 0) {
        if (warp == 0) {
            result[0] = ok ? 0 : 1;
            result[2] = (int)(waited / 1000000ull);
        } else {
            result[1] = (!ok && waited < kWaitLimitNs) ? 1 : 0;
        }
    }
}

fa_status decode_check_args(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* kv_lens, const void* o, const float* lse, int B, int Sq,
                            int Hq, int Hkv, int D, int Smax, float scale, fa_dtype dtype) {
    if (!q || !k_cache || !v_cache || !kv_lens || !o) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(kv_lens) & 3u))
        return FA_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Smax <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_UNSUPPORTED;
    if (D != 64 && D != 96 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
    if (Sq <= 0) return FA_ERR_INVALID_ARG;
    if ((Hq / Hkv) * Sq > 16 || B > 1024) return FA_ERR_UNSUPPORTED;
    if ((long long)B * Smax > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    // The kernels count 128-key tiles over all (sequence, kv head) pairs in 32 bits.
    if ((long long)B * ((Smax + 127) / 128) * Hkv > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Sq, int Sk, int Hq, int Hkv, int D, float scale, int causal,
                        int window_left, int window_right, fa_dtype dtype, fa_stream_t stream) {
    if (!q || !k || !v || !o) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
    if (B <= 0 || Sq <= 0 || Sk <= 0 || Hq <= 0 || Hkv <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_UNSUPPORTED;
    if (D != 64 && D != 96 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
    // TMA coordinates are 32-bit signed; the batch and sequence extents must fit.
    if ((long long)B * Sq > 0x7fffffffLL || (long long)B * Sk > 0x7fffffffLL)
        return FA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(&di)) return FA_ERR_CUDA;
    FwdArgs a{q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, scale, causal, window_left, window_right,
              nullptr, nullptr, 0, 0, dtype == FA_BF16, di.num_sms, di.status};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (D) {
        case 64: return launch_fwd_d64(a, s);
        case 96: return launch_fwd_d96(a, s);
        case 128: return launch_fwd_d128(a, s);
        default: return launch_fwd_d256(a, s);
    }
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B,
                        int total_q, int total_k, int Hq, int Hkv, int D, float scale, int causal,
                        int window_left, int window_right, fa_dtype dtype, fa_stream_t stream) {
    if (!q || !k || !v || !o || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
        return FA_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
    if (B <= 0 || total_q <= 0 || total_k <= 0 || Hq <= 0 || Hkv <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_UNSUPPORTED;
    if (D != 64 && D != 96 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
    if (B > 1024) return FA_ERR_UNSUPPORTED;
    if ((long long)total_q * Hq > 0x7fffffffLL || (long long)total_k * Hkv > 0x7fffffffLL)
        return FA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(&di)) return FA_ERR_CUDA;
    FwdArgs a{q, k, v, o, lse, B, 0, 0, Hq, Hkv, D, scale, causal, window_left, window_right,
              cu_seqlens_q, cu_seqlens_k, total_q, total_k, dtype == FA_BF16, di.num_sms,
              di.status};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (D) {
        case 64: return launch_fwd_d64(a, s);
        case 96: return launch_fwd_d96(a, s);
        case 128: return launch_fwd_d128(a, s);
        default: return launch_fwd_d256(a, s);
    }
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq,
                 int Sk, int Hq, int Hkv, int D, float scale, int causal, fa_dtype dtype,
                 fa_stream_t stream) {
    return fa_fwd_window(q, k, v, o, lse, B, Sq, Sk, Hq, Hkv, D, scale, causal, -1, -1, dtype,
                         stream);
}

size_t fa_decode_workspace_bytes(int B, int Hq, int D, int num_splits) {
    if (B <= 0 || Hq <= 0 || D <= 0 || num_splits <= 0) return 0;
    const size_t rows = (size_t)B * Hq * num_splits;
    const size_t o_bytes = (rows * D * sizeof(float) + 255) & ~size_t(255);
    const size_t l_bytes = (rows * sizeof(float) + 255) & ~size_t(255);
    return o_bytes + l_bytes;
}

int fa_decode_default_splits(int B, int Hkv, int max_kv_len, int num_sms) {
    if (B <= 0 || Hkv <= 0 || max_kv_len <= 0) return -1;
    if (num_sms <= 0) {
        DeviceInfo di;
        if (!device_info(&di)) return -1;
        num_sms = di.num_sms;
    }
    // Allow about eight pieces per SM over the (sequence, kv head) pairs, and no more than
    // one piece per 256 keys of the longest sequence.
    const long long groups = (long long)B * Hkv;
    long long ns = (8LL * num_sms + groups - 1) / groups;
    const long long max_by_len = ((long long)max_kv_len + 255) / 256;
    if (ns > max_by_len) ns = max_by_len;
    if (ns > 1024) ns = 1024;
    if (ns < 1) ns = 1;
    return (int)ns;
}

namespace {

// Shared validation and dispatch of the contiguous and paged decode entry points.
fa_status decode_common(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_table, const int32_t* kv_lens, void* o, float* lse,
                        int B, int Sq, int Hq, int Hkv, int D, int Smax, int num_pages,
                        int page_size, int max_pages, float scale, int causal, int num_splits,
                        void* workspace, size_t workspace_bytes, fa_dtype dtype,
                        fa_stream_t stream) {
    const fa_status chk = decode_check_args(q, k_cache, v_cache, kv_lens, o, lse, B, Sq, Hq, Hkv,
                                            D, Smax, scale, dtype);
    if (chk != FA_OK) return chk;
    DeviceInfo di;
    if (!device_info(&di)) return FA_ERR_CUDA;
    if (num_splits <= 0) num_splits = fa_decode_default_splits(B, Hkv, Smax, di.num_sms);
    if (num_splits > Smax) num_splits = Smax;
    const size_t need = fa_decode_workspace_bytes(B * Sq, Hq, D, num_splits);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FA_ERR_WORKSPACE;
    const size_t rows = (size_t)B * Sq * Hq * num_splits;
    float* o_part = static_cast<float*>(workspace);
    float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                               ((rows * D * sizeof(float) + 255) & ~size_t(255)));
    DecodeArgs a{q, k_cache, v_cache, kv_lens, o, lse, B, Hq, Hkv, D, Smax, scale, num_splits,
                 o_part, lse_part, Sq, causal, block_table, num_pages, page_size, max_pages,
                 dtype == FA_BF16, di.num_sms, di.status};
    return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

fa_status fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* kv_lens, void* o, float* lse, int B, int Hq, int Hkv,
                            int D, int Smax, float scale, int num_splits, void* workspace,
                            size_t workspace_bytes, fa_dtype dtype, fa_stream_t stream) {
    return decode_common(q, k_cache, v_cache, nullptr, kv_lens, o, lse, B, 1, Hq, Hkv, D, Smax, 0,
                         0, 0, scale, 0, num_splits, workspace, workspace_bytes, dtype, stream);
}

fa_status fa_decode_splitkv_multi(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* kv_lens, void* o, float* lse, int B, int Sq, int Hq,
                                  int Hkv, int D, int Smax, float scale, int causal, int num_splits,
                                  void* workspace, size_t workspace_bytes, fa_dtype dtype,
                                  fa_stream_t stream) {
    return decode_common(q, k_cache, v_cache, nullptr, kv_lens, o, lse, B, Sq, Hq, Hkv, D, Smax, 0,
                         0, 0, scale, causal, num_splits, workspace, workspace_bytes, dtype,
                         stream);
}

fa_status fa_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                                  const int32_t* block_table, const int32_t* kv_lens, void* o,
                                  float* lse, int B, int Hq, int Hkv, int D, int num_pages,
                                  int page_size, int max_pages_per_seq, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  fa_dtype dtype, fa_stream_t stream) {
    if (!block_table || (reinterpret_cast<uintptr_t>(block_table) & 3u)) return FA_ERR_INVALID_ARG;
    if (num_pages <= 0 || max_pages_per_seq <= 0 || page_size <= 0) return FA_ERR_INVALID_ARG;
    if (page_size % 128 != 0) return FA_ERR_UNSUPPORTED;
    const long long smax = (long long)page_size * max_pages_per_seq;
    if (smax > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    return decode_common(q, k_pages, v_pages, block_table, kv_lens, o, lse, B, 1, Hq, Hkv, D,
                         (int)smax, num_pages, page_size, max_pages_per_seq, scale, 0, num_splits,
                         workspace, workspace_bytes, dtype, stream);
}

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dim, dtype or size";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: decode workspace missing or too small";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA call failed";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel gave up on a bounded wait";
        default: return "unknown fa_status";
    }
}

fa_status fa_selftest_bounded_wait(int* result, fa_stream_t stream) {
    if (!result || !aligned16(result)) return FA_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di)) return FA_ERR_CUDA;
    selftest_bounded_wait_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(result, di.status);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_last_device_status(void) {
    DeviceInfo di;
    if (!device_info(&di)) return FA_ERR_CUDA;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemcpy(&v, di.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(di.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return v == 0 ? FA_OK : (fa_status)v;
}

}  // extern "C"
