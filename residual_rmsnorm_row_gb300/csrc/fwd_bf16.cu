// Forward kernel instances for bf16 storage.
#include "fwd_kernels.cuh"

namespace rrn {

cudaError_t launch_fwd_bf16(const FwdArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_fwd<__nv_bfloat16>(a, l, stream);
}

int occupancy_fwd_bf16(bool fused, const Launch &l) { return occupancy_fwd_t<__nv_bfloat16>(fused, l); }

}  // namespace rrn
