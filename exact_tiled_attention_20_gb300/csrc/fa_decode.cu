// fa_decode.cu -- head-dim dispatch of the split-KV decode (kernels in fa_decode.cuh, one
// instantiation per head dim in fa_decode_d{64,96,128,256}.cu, compiled in parallel).
#include "fa_internal.h"

namespace fa {

fa_status launch_decode(const DecodeArgs& a, cudaStream_t s) {
    switch (a.D) {
        case 64: return launch_decode_d64(a, s);
        case 96: return launch_decode_d96(a, s);
        case 128: return launch_decode_d128(a, s);
        case 256: return launch_decode_d256(a, s);
        default: return FA_ERR_UNSUPPORTED;
    }
}

}  // namespace fa
