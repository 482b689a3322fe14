// fa_decode_noalloc.cu -- split-KV decode with library-owned scratch, for callers that
// cannot allocate device memory.
//
// fa_decode_splitkv needs a workspace for its per-piece partial results, which the caller
// normally allocates.  Some callers cannot: a plugin running inside a host runtime that
// owns every device allocation, or a latency-critical serving loop that must never call
// cudaMalloc (which may synchronise the device).  For them this file keeps the workspace
// in a fixed-size array in device global memory that is part of the library image, so
// the call itself allocates nothing.
//
// Cost: every GPU that loads this library holds kNoAllocScratchBytes (8 MiB) for this
// array until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = FA_DECODE_NOALLOC_SCRATCH_BYTES;  // 8 MiB
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the symbol, not a
// device address: the address is looked up per device below.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// One-time set-up per device, done by the first call with that device current.
bool scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return false;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return true;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* kv_lens, void* o, float* lse, int B, int Hq,
                                    int Hkv, int D, int Smax, float scale, int num_splits,
                                    fa_dtype dtype, fa_stream_t stream) {
    // The same argument checks as fa_decode_splitkv come first, so an invalid or
    // unsupported call returns the same status from either entry point.
    const fa_status chk = fa::decode_check_args(q, k_cache, v_cache, kv_lens, o, lse, B, 1, Hq,
                                                Hkv, D, Smax, scale, dtype);
    if (chk != FA_OK) return chk;
    int ns = num_splits;
    if (ns <= 0) ns = fa_decode_default_splits(B, Hkv, Smax, 0);
    if (ns <= 0) return FA_ERR_CUDA;
    if (ns > Smax) ns = Smax;
    const size_t need = fa_decode_workspace_bytes(B, Hq, D, ns);
    if (need == 0 || need > fa::kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (!fa::scratch_address(&scratch)) return FA_ERR_CUDA;
    return fa_decode_splitkv(q, k_cache, v_cache, kv_lens, o, lse, B, Hq, Hkv, D, Smax, scale,
                             ns, scratch, fa::kNoAllocScratchBytes, dtype, stream);
}

}  // extern "C"
