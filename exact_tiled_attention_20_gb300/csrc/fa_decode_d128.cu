// fa_decode_d128.cu -- split-KV decode instantiation for head dim 128:
// one 128-key MMA tile per split-plan tile, two column atoms per row, 3-stage ring.
#include "fa_decode.cuh"

namespace fa {

fa_status launch_decode_d128(const DecodeArgs& a, cudaStream_t s) { return launch_decode_d<128>(a, s); }

}  // namespace fa
