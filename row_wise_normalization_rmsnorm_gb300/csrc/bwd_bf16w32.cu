// bwd_bf16w32.cu -- backward kernels for bf16 activations with an fp32 weight.
#include "bwd_kernels.cuh"

namespace rmsn {
int launch_bwd_main_bf16w32(int plan_id, bool fused, bool packed, const BwdParams &p, int grid, int smem,
                         void *stream) {
    return bwd_launch_t<__nv_bfloat16, float>(plan_id, fused, packed, p, grid, smem, stream);
}
const void *bwd_main_kernel_ptr_bf16w32(int plan_id, bool fused, bool packed) {
    return bwd_ptr_t<__nv_bfloat16, float>(plan_id, fused, packed);
}
}  // namespace rmsn
