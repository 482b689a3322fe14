// fa_fwd_d256.cu -- forward kernel instantiation for head dim 256.
// Tile: 1 x 128 query rows per CTA, 64 keys per K/V tile, 2-stage K/V ring.
#include "fa_fwd.cuh"

namespace fa {

fa_status launch_fwd_d256(const FwdArgs& a, cudaStream_t s) {
    return launch_fwd_cfg<FwdConfig<256, 64, 1, 2>>(a, s);
}

}  // namespace fa
