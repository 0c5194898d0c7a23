// Backward kernel instances for bf16 and fp32 storage.
#include "bwd_kernels.cuh"

namespace rrn {

cudaError_t launch_bwd_bf16(const BwdArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_bwd<__nv_bfloat16>(a, l, stream);
}
cudaError_t launch_bwd_f32(const BwdArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_bwd<float>(a, l, stream);
}
int occupancy_bwd_bf16(bool add_grad, const Launch &l) {
    return occupancy_bwd_t<__nv_bfloat16>(add_grad, l);
}
int occupancy_bwd_f32(bool add_grad, const Launch &l) { return occupancy_bwd_t<float>(add_grad, l); }

}  // namespace rrn
