// fwd_bf16w32.cu -- forward kernels for bf16 activations with an fp32 weight.
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_fwd_bf16w32(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return launch_t<__nv_bfloat16, float>(plan_id, fused, p, grid, stream);
}
const void *fwd_kernel_ptr_bf16w32(int plan_id, bool fused) { return ptr_t<__nv_bfloat16, float>(plan_id, fused); }
int launch_fwd_staged_bf16w32(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_fwd_launch_t<__nv_bfloat16, float, false>(plan_id, fused, p, grid, smem, stream);
}
const void *fwd_staged_kernel_ptr_bf16w32(int plan_id, bool fused) {
    return staged_fwd_ptr_t<__nv_bfloat16, float, false>(plan_id, fused);
}
}  // namespace rmsn
