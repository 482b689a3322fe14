// fa_decode_d64.cu -- split-KV decode instantiation for head dim 64:
// one 128-key MMA tile per split-plan tile, one 64-column atom per row, 6-stage ring.
#include "fa_decode.cuh"

namespace fa {

fa_status launch_decode_d64(const DecodeArgs& a, cudaStream_t s) { return launch_decode_d<64>(a, s); }

}  // namespace fa
