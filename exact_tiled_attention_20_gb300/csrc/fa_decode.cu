// fa_decode.cu -- placeholder until the split-KV kernels land.
#include "fa_internal.h"

namespace fa {

fa_status launch_decode(const DecodeArgs&, cudaStream_t) { return FA_ERR_UNSUPPORTED; }

}  // namespace fa
