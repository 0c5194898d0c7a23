// Forward kernel instances for fp32 storage.
#include "fwd_kernels.cuh"

namespace rrn {

cudaError_t launch_fwd_f32(const FwdArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_fwd<float>(a, l, stream);
}

int occupancy_fwd_f32(bool fused, const Launch &l) { return occupancy_fwd_t<float>(fused, l); }

}  // namespace rrn
