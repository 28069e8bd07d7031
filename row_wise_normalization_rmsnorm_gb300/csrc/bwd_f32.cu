// bwd_f32.cu -- backward kernels for fp32.
#include "bwd_kernels.cuh"

namespace rmsn {
int launch_bwd_main_f32(int plan_id, bool fused, bool packed, const BwdParams &p, int grid, int smem,
                         void *stream) {
    return bwd_launch_t<float, float>(plan_id, fused, packed, p, grid, smem, stream);
}
const void *bwd_main_kernel_ptr_f32(int plan_id, bool fused, bool packed) {
    return bwd_ptr_t<float, float>(plan_id, fused, packed);
}
int launch_dw_finalize_f32(const float *ws, int parts, int ncols, void *out0, void *out1, int split, int peel,
                           void *stream, bool serial, int sms) {
    return finalize_launch_t<float>(ws, parts, ncols, out0, out1, split, peel, stream, serial, sms);
}
}  // namespace rmsn
