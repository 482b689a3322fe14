// fa_fwd_d128.cu -- forward kernel instantiation for head dim 128.
// Tile: 2 x 128 query rows per CTA, 128 keys per K/V tile, 2-stage K/V ring.
#include "fa_fwd.cuh"

namespace fa {

fa_status launch_fwd_d128(const FwdArgs& a, cudaStream_t s) {
    return launch_fwd_cfg<FwdConfig<128, 128, 2, 2>>(a, s);
}

}  // namespace fa
