// noalloc.cu -- rmsnorm_bwd_noalloc: the plain backward for callers that
// cannot allocate device memory at call time.
//
// Who needs this: code that may not call cudaMalloc (or cudaMallocAsync)
// when it runs, for example an inference or training engine that reserves
// all device memory at start-up and forbids later allocation, or a plug-in
// whose host framework owns the allocator and hands the op no workspace.
// rmsnorm_bwd needs a workspace for its per-CTA dW partial rows; this entry
// point takes it from a fixed array compiled into the library instead of
// from the caller or an allocator.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library's kernels are loaded holds RMSNORM_NOALLOC_SCRATCH_BYTES of it
// until the process exits. Host code must not pass the array's name to a
// kernel: on the host that name is a stand-in object, not a device
// address. The device address is looked up once per device with
// cudaGetSymbolAddress, on that device's first call, and kept for the life
// of the process (a cudaDeviceReset would leave it stale).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/rmsnorm.h"

namespace rmsn {
void set_last_cuda_error(int e);  // defined in api.cu
}

static __device__ __align__(256) float
    g_rmsnorm_noalloc_scratch[RMSNORM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch[kMaxDevices];

// Device address of the scratch array on the current device (looked up on
// the first call per device).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mutex);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_rmsnorm_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" rmsnorm_status_t rmsnorm_bwd_noalloc(const void *dy, const void *x, const void *w,
                                                const float *rstd, void *dx, void *dw, int64_t M,
                                                int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                                                rmsnorm_stream_t stream) {
    // Every storage type rmsnorm_bwd takes is served; its own checks decide
    // the arguments. Only the size is this entry point's to check (below).
    if (N < 1 || N > RMSNORM_MAX_N || M < 0) return RMSNORM_ERR_INVALID_ARG;
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        rmsn::set_last_cuda_error((int)e);
        return RMSNORM_ERR_CUDA;
    }
    // The scratch goes in as a caller workspace of the full array size, so
    // rmsnorm_bwd never reaches its stream-ordered allocation. Its own size
    // check refuses, with RMSNORM_ERR_WORKSPACE and before any launch, a
    // call whose partial rows would not fit.
    return rmsnorm_bwd(dy, x, w, rstd, dx, dw, scratch, (size_t)RMSNORM_NOALLOC_SCRATCH_BYTES, M, N, dt, eps,
                       offset, stream);
}
