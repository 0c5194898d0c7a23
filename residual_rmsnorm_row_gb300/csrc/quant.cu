// RMSNorm -> fp8 e4m3 kernel instances for bf16 and fp32 storage.
#include "quant_kernels.cuh"

namespace rrn {

cudaError_t launch_quant_bf16(const QuantArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_quant<__nv_bfloat16>(a, l, stream);
}
cudaError_t launch_quant_f32(const QuantArgs &a, const Launch &l, cudaStream_t stream) {
    return launch_quant<float>(a, l, stream);
}
int occupancy_quant_bf16(bool fused, const Launch &l) { return occupancy_quant_t<__nv_bfloat16>(fused, l); }
int occupancy_quant_f32(bool fused, const Launch &l) { return occupancy_quant_t<float>(fused, l); }

}  // namespace rrn
