// fa_decode_d96.cu -- split-KV decode instantiation for head dim 96:
// one 128-key MMA tile per split-plan tile, two column atoms (the second zero-filled past 96), 3-stage ring.
#include "fa_decode.cuh"

namespace fa {

fa_status launch_decode_d96(const DecodeArgs& a, cudaStream_t s) { return launch_decode_d<96>(a, s); }

}  // namespace fa
