// ln_f32.cu -- LayerNorm forward and backward kernels for fp32.
#include "bwd_kernels.cuh"
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_ln_fwd_f32(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return ln_launch_t<float>(plan_id, fused, p, grid, stream);
}
int launch_ln_bwd_f32(int plan_id, bool fused, const BwdParams &p, int grid, int smem, void *stream) {
    return ln_bwd_launch_t<float>(plan_id, fused, p, grid, smem, stream);
}
const void *ln_bwd_kernel_ptr_f32(int plan_id, bool fused) { return ln_bwd_ptr_t<float>(plan_id, fused); }
int launch_ln_fwd_staged_f32(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_fwd_launch_t<float, float, true>(plan_id, fused, p, grid, smem, stream);
}
const void *ln_fwd_staged_kernel_ptr_f32(int plan_id, bool fused) { return staged_fwd_ptr_t<float, float, true>(plan_id, fused); }
}  // namespace rmsn
