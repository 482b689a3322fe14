// fa_fwd_d64.cu -- forward kernel instantiation for head dim 64.
// Tile: 2 x 128 query rows per CTA, 128 keys per K/V tile, 3-stage K/V ring.
#include "fa_fwd.cuh"

namespace fa {

fa_status launch_fwd_d64(const FwdArgs& a, cudaStream_t s) {
    return launch_fwd_cfg<FwdConfig<64, 128, 2, 3>>(a, s);
}

}  // namespace fa
