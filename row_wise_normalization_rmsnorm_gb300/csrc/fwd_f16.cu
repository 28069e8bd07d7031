// fwd_f16.cu -- f16 instantiations of the forward kernels.
#include "fwd_kernels.cuh"

namespace rmsn {
int launch_fwd_f16(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    return launch_t<__half>(plan_id, fused, p, grid, stream);
}
const void *fwd_kernel_ptr_f16(int plan_id, bool fused) { return ptr_t<__half>(plan_id, fused); }
}  // namespace rmsn
