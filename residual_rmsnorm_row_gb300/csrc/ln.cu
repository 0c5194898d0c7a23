// LayerNorm kernel instances for bf16 and fp32 storage.
#include "ln_kernels.cuh"

namespace rrn {

cudaError_t launch_ln_fwd_bf16(const LnFwdArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_ln_fwd<__nv_bfloat16>(a, l, stream);
}
cudaError_t launch_ln_fwd_f32(const LnFwdArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_ln_fwd<float>(a, l, stream);
}
cudaError_t launch_ln_bwd_bf16(const LnBwdArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_ln_bwd<__nv_bfloat16>(a, l, stream);
}
cudaError_t launch_ln_bwd_f32(const LnBwdArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_ln_bwd<float>(a, l, stream);
}
int occupancy_ln_bf16(bool bwd, bool flag, const Launch &l) {
    return occupancy_ln_t<__nv_bfloat16>(bwd, flag, l);
}
int occupancy_ln_f32(bool bwd, bool flag, const Launch &l) { return occupancy_ln_t<float>(bwd, flag, l); }

}  // namespace rrn
