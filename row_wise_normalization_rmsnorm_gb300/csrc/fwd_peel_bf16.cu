// fwd_peel_bf16.cu -- RMSNorm and LayerNorm forward kernels for bf16 rows at a
// common offset past a 16-byte boundary (the default vectorised plans,
// compiled with the row's wrapped chunk 0).
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_fwd_peel_bf16(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return launch_t<__nv_bfloat16, __nv_bfloat16, QOUT_NONE, true>(plan_id, fused, p, grid, stream);
}
int launch_fwd_staged_peel_bf16(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_fwd_launch_t<__nv_bfloat16, __nv_bfloat16, false, QOUT_NONE, true>(plan_id, fused, p, grid, smem, stream);
}
const void *fwd_staged_kernel_ptr_peel_bf16(int plan_id, bool fused) {
    return staged_fwd_ptr_t<__nv_bfloat16, __nv_bfloat16, false, QOUT_NONE, true>(plan_id, fused);
}
int launch_ln_fwd_peel_bf16(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return ln_launch_t<__nv_bfloat16, __nv_bfloat16, true>(plan_id, fused, p, grid, stream);
}
int launch_ln_fwd_staged_peel_bf16(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_fwd_launch_t<__nv_bfloat16, __nv_bfloat16, true, QOUT_NONE, true>(plan_id, fused, p, grid, smem, stream);
}
const void *ln_fwd_staged_kernel_ptr_peel_bf16(int plan_id, bool fused) {
    return staged_fwd_ptr_t<__nv_bfloat16, __nv_bfloat16, true, QOUT_NONE, true>(plan_id, fused);
}
}  // namespace rmsn
