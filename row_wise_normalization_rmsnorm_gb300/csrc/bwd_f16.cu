// bwd_f16.cu -- backward kernels for fp16.
#include "bwd_kernels.cuh"

namespace rmsn {
int launch_bwd_main_f16(int plan_id, bool fused, bool packed, const BwdParams &p, int grid, int smem,
                         void *stream) {
    return bwd_launch_t<__half, __half>(plan_id, fused, packed, p, grid, smem, stream);
}
const void *bwd_main_kernel_ptr_f16(int plan_id, bool fused, bool packed) {
    return bwd_ptr_t<__half, __half>(plan_id, fused, packed);
}
int launch_dw_finalize_f16(const float *ws, int parts, int ncols, void *out0, void *out1, int split, int peel,
                           void *stream, bool serial, int sms) {
    return finalize_launch_t<__half>(ws, parts, ncols, out0, out1, split, peel, stream, serial, sms);
}
}  // namespace rmsn
