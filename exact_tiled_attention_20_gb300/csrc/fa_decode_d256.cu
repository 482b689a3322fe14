// fa_decode_d256.cu -- split-KV decode instantiation for head dim 256:
// two 64-key MMA tiles per split-plan tile, O^T in two 128-row blocks, 3-stage ring.
#include "fa_decode.cuh"

namespace fa {

fa_status launch_decode_d256(const DecodeArgs& a, cudaStream_t s) { return launch_decode_d<256>(a, s); }

}  // namespace fa
