// fwd_peel_f16.cu -- RMSNorm and LayerNorm forward kernels for fp16 rows at a
// common offset past a 16-byte boundary (the default vectorised plans,
// compiled with the row's wrapped chunk 0).
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_fwd_peel_f16(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return launch_t<__half, __half, QOUT_NONE, true>(plan_id, fused, p, grid, stream);
}
int launch_fwd_staged_peel_f16(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_fwd_launch_t<__half, __half, false, QOUT_NONE, true>(plan_id, fused, p, grid, smem, stream);
}
const void *fwd_staged_kernel_ptr_peel_f16(int plan_id, bool fused) {
    return staged_fwd_ptr_t<__half, __half, false, QOUT_NONE, true>(plan_id, fused);
}
int launch_ln_fwd_peel_f16(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return ln_launch_t<__half, __half, true>(plan_id, fused, p, grid, stream);
}
int launch_ln_fwd_staged_peel_f16(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    return staged_fwd_launch_t<__half, __half, true, QOUT_NONE, true>(plan_id, fused, p, grid, smem, stream);
}
const void *ln_fwd_staged_kernel_ptr_peel_f16(int plan_id, bool fused) {
    return staged_fwd_ptr_t<__half, __half, true, QOUT_NONE, true>(plan_id, fused);
}
}  // namespace rmsn
