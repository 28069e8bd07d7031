// ln_f16w32.cu -- LayerNorm forward and backward kernels for fp16 activations
// with fp32 gamma and beta.
#include "bwd_kernels.cuh"
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_ln_fwd_f16w32(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return ln_launch_t<__half, float>(plan_id, fused, p, grid, stream);
}
int launch_ln_bwd_f16w32(int plan_id, bool fused, const BwdParams &p, int grid, int smem, void *stream) {
    return ln_bwd_launch_t<__half, float>(plan_id, fused, p, grid, smem, stream);
}
const void *ln_bwd_kernel_ptr_f16w32(int plan_id, bool fused) { return ln_bwd_ptr_t<__half, float>(plan_id, fused); }
int launch_ln_fwd_staged_f16w32(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_fwd_launch_t<__half, float, true>(plan_id, fused, p, grid, smem, stream);
}
const void *ln_fwd_staged_kernel_ptr_f16w32(int plan_id, bool fused) {
    return staged_fwd_ptr_t<__half, float, true>(plan_id, fused);
}
}  // namespace rmsn
