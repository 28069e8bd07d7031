// fwd_f16.cu -- forward kernels for fp16.
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_fwd_f16(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return launch_t<__half, __half>(plan_id, fused, p, grid, stream);
}
const void *fwd_kernel_ptr_f16(int plan_id, bool fused) { return ptr_t<__half, __half>(plan_id, fused); }
int launch_fwd_staged_f16(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_fwd_launch_t<__half, __half, false>(plan_id, fused, p, grid, smem, stream);
}
const void *fwd_staged_kernel_ptr_f16(int plan_id, bool fused) {
    return staged_fwd_ptr_t<__half, __half, false>(plan_id, fused);
}
}  // namespace rmsn
