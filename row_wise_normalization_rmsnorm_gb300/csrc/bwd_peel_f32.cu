// bwd_peel_f32.cu -- RMSNorm and LayerNorm backward main kernels for fp32
// rows at a common offset past a 16-byte boundary (the default vectorised
// plans, compiled with the row's wrapped chunk 0).
#include "bwd_kernels.cuh"

namespace rmsn {
int launch_bwd_main_peel_f32(int plan_id, bool fused, bool packed, const BwdParams &p, int grid, int smem,
                            void *stream) {
    return bwd_launch_t<float, float, true>(plan_id, fused, packed, p, grid, smem, stream);
}
const void *bwd_main_kernel_ptr_peel_f32(int plan_id, bool fused, bool packed) {
    return bwd_ptr_t<float, float, true>(plan_id, fused, packed);
}
int launch_ln_bwd_peel_f32(int plan_id, bool fused, const BwdParams &p, int grid, int smem, void *stream) {
    return ln_bwd_launch_t<float, float, true>(plan_id, fused, p, grid, smem, stream);
}
const void *ln_bwd_kernel_ptr_peel_f32(int plan_id, bool fused) { return ln_bwd_ptr_t<float, float, true>(plan_id, fused); }
}  // namespace rmsn
