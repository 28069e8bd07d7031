// fwd_f32.cu -- f32 instantiations of the forward kernels.
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_fwd_f32(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return launch_t<float>(plan_id, fused, p, grid, stream);
}
const void *fwd_kernel_ptr_f32(int plan_id, bool fused) { return ptr_t<float>(plan_id, fused); }
}  // namespace rmsn
