// fwd8_bf16w32.cu -- forward kernels with E4M3 output for bf16 activations with an
// fp32 weight.
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_fwd8_bf16w32(int plan_id, bool fused, int mode, const FwdParams &p, int grid, void *stream) {
    return launch_q<__nv_bfloat16, float>(plan_id, fused, mode, p, grid, stream);
}
int launch_fwd8_staged_bf16w32(int plan_id, bool fused, int mode, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_launch_q<__nv_bfloat16, float>(plan_id, fused, mode, p, grid, smem, stream);
}
const void *fwd8_staged_kernel_ptr_bf16w32(int plan_id, bool fused, int mode) {
    return staged_ptr_q<__nv_bfloat16, float>(plan_id, fused, mode);
}
}  // namespace rmsn
