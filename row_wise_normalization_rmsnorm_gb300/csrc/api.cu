// api.cu -- the C ABI of librmsnorm_gb300.so (declared in include/rmsnorm.h):
// argument checks, plan selection from the specialisation table, the
// backward's workspace, and the launches on the caller's stream.
//
// The host path does no per-call marshalling: plain pointers and scalars go
// straight into a by-value kernel parameter block, the stream is the
// caller's, and the only cached state is per-device SM counts and
// occupancies (Liger-Kernel PR #1388, section 1: the direct-call launch;
// ROCm/FlyDSL PR #855, "Hot-cache launch path" and "Runtime configuration
// and ownership": raw caller stream, SM count cached per device, workspace
// owned per call).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <initializer_list>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>

#include "../../include/rmsnorm.h"
#include "plans.h"

namespace rmsn {

struct PlanDesc {
    int id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax;
};

static const PlanDesc kPlans[] = {
#define RMSN_DESC(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) {id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax},
    RMSNORM_PLAN_TABLE(RMSN_DESC)
#undef RMSN_DESC
};
static const int kNumPlans = (int)(sizeof(kPlans) / sizeof(kPlans[0]));

static const PlanDesc *find_plan(int id) {
    for (int i = 0; i < kNumPlans; ++i)
        if (kPlans[i].id == id) return &kPlans[i];
    return nullptr;
}

// The dtype argument: the activations' storage type, optionally OR'ed with
// RMSNORM_WEIGHT_F32 (w and dW in fp32). Kernel variants are indexed by
// "kind": 0 fp32, 1 bf16, 2 fp16 (weight in the same type), 3 bf16 and
// 4 fp16 activations with an fp32 weight. fp32 | RMSNORM_WEIGHT_F32 is fp32.
constexpr int kNumKinds = 5;
static bool valid_dtype(int dt) {
    const int base = dt & ~RMSNORM_WEIGHT_F32;
    return base == RMSNORM_F32 || base == RMSNORM_BF16 || base == RMSNORM_F16;
}
static int base_dtype(int dt) { return dt & ~RMSNORM_WEIGHT_F32; }
static int kind_of(int dt) {
    const int base = base_dtype(dt);
    if (base == RMSNORM_F32 || !(dt & RMSNORM_WEIGHT_F32)) return base;
    return base == RMSNORM_BF16 ? 3 : 4;
}
static bool mixed_kind(int kind) { return kind >= 3; }
// Bytes per activation element and per weight element.
static int elem_size(int dt) { return base_dtype(dt) == RMSNORM_F32 ? 4 : 2; }
static int weight_size(int dt) { return (base_dtype(dt) == RMSNORM_F32 || (dt & RMSNORM_WEIGHT_F32)) ? 4 : 2; }

static int dtype_bit(int dt) {
    const int base = base_dtype(dt);
    return base == RMSNORM_BF16 ? DT_BF16 : (base == RMSNORM_F16 ? DT_F16 : DT_F32);
}

// Default plan for (op, dtype, chunks per row): a row-in-registers
// (vector) or staged plan; nullptr when none covers C.
static bool row_path(int path) { return path == PATH_VECTOR || staged_path(path); }

static const PlanDesc *default_vector_plan(int op, int dt, int64_t C) {
    for (int i = 0; i < kNumPlans; ++i) {
        const PlanDesc &d = kPlans[i];
        if (d.op == op && row_path(d.path) && d.cmin > 0 && (d.dtm & dtype_bit(dt)) && C >= d.cmin && C <= d.cmax)
            return &d;
    }
    return nullptr;
}

static const PlanDesc *generic_plan(int op) {
    for (int i = 0; i < kNumPlans; ++i)
        if (kPlans[i].op == op && kPlans[i].path == PATH_GENERIC) return &kPlans[i];
    return nullptr;
}

// Rows a streamed kernel's stage holds: x and dy (and dres) for the
// backward, x (and residual) for the forward.
static int stream_arrays(const PlanDesc &d, bool fused) {
    return d.op == OP_BWD ? (fused ? 3 : 2) : (fused ? 2 : 1);
}

// A streamed generic kernel's shared memory: `depth` stages of row covers.
static int64_t stream_smem_at(const PlanDesc &d, int64_t N, int es, bool fused, int depth) {
    return (int64_t)depth * stream_arrays(d, fused) * stream_slot_bytes(N, es);
}

static int cta_threads(const PlanDesc &d) { return d.path == PATH_GENERIC ? 256 : d.tpr * d.teams; }

// Largest dynamic shared memory a plan may ask for: the 227 KB a CTA may
// opt into on sm_103a, less room for the kernels' static arrays.
constexpr int kMaxDynamicSmem = 226 * 1024;

// Stages a streamed generic kernel takes: the plan's depth, or fewer (at
// least two) where the covers would not fit; 0: none fits.
static int stream_depth(const PlanDesc &d, int64_t N, int es, bool fused) {
    for (int k = d.depth; k >= 2; --k)
        if (stream_smem_at(d, N, es, fused, k) <= kMaxDynamicSmem) return k;
    return 0;
}

// Whether a streamed generic plan takes rows of N elements.
static bool stream_fits(const PlanDesc &d, int64_t N, int es) {
    return N <= (int64_t)d.tpr * d.v && stream_depth(d, N, es, true) >= 2;
}

// The plan for rows no vectorised plan takes: the streamed plan whose
// range holds N (where its stages fit; for the forward only where the
// caller takes it: the RMSNorm forward with output in the activations'
// type), else the one-CTA-a-row kernel.
static const PlanDesc *fallback_plan(int op, int64_t N, int es, bool stream_ok) {
    const int sop = op == RMSNORM_OP_FWD ? OP_FWD_STAGED : op;
    if (stream_ok && (op == RMSNORM_OP_BWD || op == RMSNORM_OP_FWD)) {
        for (int i = 0; i < kNumPlans; ++i) {
            const PlanDesc &d = kPlans[i];
            if (d.op == sop && d.path == PATH_STREAM && d.cmin > 0 && N >= d.cmin && N <= d.cmax &&
                stream_fits(d, N, es))
                return &d;
        }
    }
    return generic_plan(op);
}
// Longest row (bytes) the generic LayerNorm forward keeps in shared memory
// between its three passes: eight 256-thread CTAs an SM still fit. (The
// RMSNorm forward, two passes, measured slower with the cache.)
constexpr int64_t kGenericRowCache = 24 * 1024;

// Largest row cache (x and dy slots) the generic LayerNorm backward takes,
// and what an SM's shared memory must hold for it: every CTA that the
// registers let reside (the grid is sized by that count), each with the
// driver's 1 KB reserve and the kernel's static arrays beside its cache.
// (The RMSNorm generic backward measured slower with the same cache: 86 ->
// 88 us on misaligned bf16 4096x7168, its re-reads being L1 hits already;
// it re-reads global memory.)
constexpr int64_t kGenericBwdRowCache = 40 * 1024;
constexpr int64_t kSmemPerSM = 228 * 1024;
constexpr int64_t kSmemPerCtaOverhead = 1024 + 256;

// Whether a generic LayerNorm backward keeps the row in shared memory: only
// where it updates partial rows (then each row is read three times) and the
// cache lowers no SM's resident CTA count.
static int generic_bwd_cache(int path, int64_t N, int es, bool partials, int cps) {
    if (path != PATH_GENERIC || !partials) return 0;
    const int64_t b = 2 * generic_bwd_cache_slot(N, es);
    if (b > kGenericBwdRowCache || cps * (b + kSmemPerCtaOverhead) > kSmemPerSM) return 0;
    return 1;
}

// A staged plan's shared memory: `depth` stages of x and dy (and dres for
// the fused variant) rows of C chunks, or of one CTA's slice (a cs-th,
// rounded up to whole chunks) of a row shared by a cluster, each row buffer
// one slot longer for rows at a common offset (peel > 0: aligned chunk C,
// which wraps chunk 0); the LayerNorm's re-read schedule also keeps (its
// slice of) gamma there.
static int64_t staged_smem_at(const PlanDesc &d, int64_t C, int peel, bool fused, int depth) {
    const int64_t row = ((C + d.cs - 1) / d.cs + (peel > 0 ? 1 : 0)) * 16;
    const int64_t gamma = d.path == PATH_RESTAGED && d.op == OP_LN_BWD ? row : 0;
    // a stage holds x and dy (and dres) rows; the staged forward's x (and residual)
    const int rows = d.op == OP_FWD_STAGED ? (fused ? 2 : 1) : (fused ? 3 : 2);
    return (int64_t)depth * rows * row + gamma;
}

// Stages a call takes: the plan's depth, or fewer (at least two) where the
// rows (three a stage for the fused variant) would not fit; 0: none fits.
static int staged_depth(const PlanDesc &d, int64_t C, int peel, bool fused) {
    for (int k = d.depth; k >= 2; --k)
        if (staged_smem_at(d, C, peel, fused, k) <= kMaxDynamicSmem) return k;
    return 0;
}

// Shared memory at the stages a call takes (above the limit when none fits).
static int64_t staged_smem_bytes(const PlanDesc &d, int64_t C, int peel, bool fused) {
    const int k = staged_depth(d, C, peel, fused);
    return staged_smem_at(d, C, peel, fused, k > 0 ? k : 2);
}

static int nominal_ctas_per_sm(const PlanDesc &d) {
    // the streamed kernels' register budget (their launch bounds)
    if (d.path == PATH_STREAM) return d.tpr >= 512 ? 1 : 512 / d.tpr;
    const int t = cta_threads(d);
    int c = 2048 / t;
    return c < 1 ? 1 : c;
}

// Partial rows per backward unit: dW (RMSNorm) or dgamma and dbeta (LayerNorm).
static int partial_rows(int op) { return op == OP_LN_BWD ? 2 : 1; }

static int bwd_smem_bytes(const PlanDesc &d, int64_t N) {
    if (d.path != PATH_VECTOR || d.teams <= 1) return 0;
    return (int)((d.teams - 1) * partial_rows(d.op) * N * 4);
}

// Chunks one plan can hold per row.
static int64_t plan_capacity(const PlanDesc &d) { return (int64_t)d.tpr * d.v * d.cs; }

// Pure selection: no CUDA calls. `peel` is the call's row layout
// (row_layout: 0 aligned, > 0 rows at a common offset, < 0 generic only).
// max_parts is the largest useful number of backward dW partial rows:
// resident CTAs (or, for cluster plans, resident clusters) on the device;
// ctas_per_sm is reported only.
static rmsnorm_status_t select_plan(int op, int64_t M, int64_t N, int dt, int peel, int64_t max_parts,
                                    int ctas_per_sm, int force_plan, int force_ctas, rmsnorm_plan_t *out,
                                    bool stream_ok = true) {
    if (!out) return RMSNORM_ERR_INVALID_ARG;
    if (op != RMSNORM_OP_FWD && op != RMSNORM_OP_BWD && op != RMSNORM_OP_LN_BWD) return RMSNORM_ERR_INVALID_ARG;
    if (!valid_dtype(dt)) return RMSNORM_ERR_INVALID_ARG;
    if (N < 1 || N > RMSNORM_MAX_N || M < 0 || M > 0x7fffffffLL) return RMSNORM_ERR_INVALID_ARG;
    if (max_parts < 1) return RMSNORM_ERR_INVALID_ARG;
    const int s = elem_size(dt);
    const bool vec_ok = peel >= 0 && (N * s) % 16 == 0 && peel < 16 / s;
    const int64_t C = vec_ok ? N * s / 16 : 0;  // 16-byte chunks a row holds

    const PlanDesc *d = nullptr;
    if (force_plan >= 0) {
        d = find_plan(force_plan);
        // a forward may take a staged forward plan
        const bool staged_fwd = d && op == RMSNORM_OP_FWD && d->op == OP_FWD_STAGED;
        if (!d || (d->op != op && !staged_fwd)) return RMSNORM_ERR_UNSUPPORTED;
        if (d->path == PATH_VECTOR && (!vec_ok || C > plan_capacity(*d))) return RMSNORM_ERR_UNSUPPORTED;
        // staged plans: aligned rows that fit
        if (staged_path(d->path) && (!vec_ok || C > plan_capacity(*d))) return RMSNORM_ERR_UNSUPPORTED;
        // a streamed generic kernel: rows of any layout that it holds, for a
        // caller that takes it
        if (d->path == PATH_STREAM && (!stream_ok || !stream_fits(*d, N, s))) return RMSNORM_ERR_UNSUPPORTED;
        // with an fp32 weight only the default plans (and the generic one) are compiled
        if (mixed_kind(kind_of(dt)) && row_path(d->path) && d->cmin == 0) return RMSNORM_ERR_UNSUPPORTED;
        // so are the kernels for rows at a common offset
        if (peel > 0 && row_path(d->path) && d->cmin == 0) return RMSNORM_ERR_UNSUPPORTED;
    } else {
        d = vec_ok ? default_vector_plan(op, dt, C) : nullptr;
        // a staged forward plan that covers the row is preferred
        if (op == RMSNORM_OP_FWD && vec_ok) {
            const PlanDesc *sd = default_vector_plan(OP_FWD_STAGED, dt, C);
            if (sd) d = sd;
        }
        if (!d) d = fallback_plan(op, N, s, stream_ok);
    }
    if (!d) return RMSNORM_ERR_UNSUPPORTED;

    std::memset(out, 0, sizeof(*out));
    // the ABI names one staged path and one generic path
    out->path = staged_path(d->path) ? PATH_STAGED : (generic_path(d->path) ? PATH_GENERIC : d->path);
    out->peel = (!generic_path(d->path) && peel > 0) ? peel : 0;
    out->plan_id = d->id;
    out->threads_per_row = d->path == PATH_GENERIC ? 256 : d->tpr;
    out->chunks_per_thread = generic_path(d->path) ? 0 : d->v;  // generic kernels hold no chunks
    out->rows_per_cta = d->path == PATH_GENERIC ? 1 : d->teams;
    out->cta_threads = cta_threads(*d);
    out->packed = generic_path(d->path) ? 0 : 1;
    out->cluster_size = d->cs;
    const int64_t units = (M + out->rows_per_cta - 1) / out->rows_per_cta;  // CTAs (or clusters) with rows
    const bool staged_fwd = d->op == OP_FWD_STAGED;
    if (op == RMSNORM_OP_FWD && !staged_fwd) {
        out->ctas = (int32_t)(units * d->cs);
        return RMSNORM_SUCCESS;
    }
    int64_t P = max_parts;
    if (force_ctas > 0) P = force_ctas;
    if (P > units) P = units;
    out->ws_rows = (int32_t)P;
    out->ctas = (int32_t)(P * d->cs);
    out->ctas_per_sm = ctas_per_sm;
    out->smem_bytes = bwd_smem_bytes(*d, N);
    // dynamic shared memory stays below 48 KB with room for the kernels'
    // static arrays (a few KB at most)
    if (staged_path(d->path)) {
        // the plain variant's stages; the fused one is checked by the backward
        const int64_t sm = staged_smem_bytes(*d, C, out->peel, false);
        if (sm > kMaxDynamicSmem) return RMSNORM_ERR_UNSUPPORTED;
        out->smem_bytes = (int32_t)sm;
    }
    if (d->path == PATH_STREAM)  // the plain variant's stages; the fused one is set by the call
        out->smem_bytes = (int32_t)stream_smem_at(*d, N, s, false, stream_depth(*d, N, s, false));
    else if (!staged_path(d->path) && out->smem_bytes > 44 * 1024)
        return RMSNORM_ERR_UNSUPPORTED;
    const int64_t bytes = staged_fwd ? 0 : P * partial_rows(op) * N * 4;  // the forward has no partial rows
    out->workspace_bytes = (bytes + 255) / 256 * 256;
    return RMSNORM_SUCCESS;
}

// A staged kernel takes more than 48 KB of dynamic shared memory, which
// needs an opt-in per kernel and device. It is given once, for the most a
// CTA of this kernel may take (the device's opt-in limit less the kernel's
// static shared memory), so later launches make no extra runtime call. A
// failed call's error is cleared so that it cannot surface at a later launch.
int allow_staged_smem(const void *k) {
    constexpr int kSlots = 1024;  // staged kernels a process may use (more: opted in at every launch)
    static std::mutex mu;
    static const void *kern[kSlots];
    static uint64_t devs[kSlots];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    std::lock_guard<std::mutex> lk(mu);
    int i = 0;
    for (; i < kSlots && kern[i] != nullptr && kern[i] != k; ++i) {
    }
    if (dev >= 0 && dev < 64 && i < kSlots && kern[i] == k && (devs[i] >> dev & 1u)) return 0;
    int optin = 0;
    cudaFuncAttributes fa;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return (int)e;
    }
    if (dev >= 0 && dev < 64 && i < kSlots) {
        kern[i] = k;
        devs[i] |= 1ull << dev;
    }
    return 0;
}

// ------------------------------------------------------ device queries --

static thread_local int g_last_cuda_error = 0;

static rmsnorm_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return RMSNORM_ERR_CUDA;
}

void set_last_cuda_error(int e) { g_last_cuda_error = e; }

// Device status word: a kernel whose bounded wait gave up writes a non-zero
// code here (rmsnorm_device_status reads it). One per device; its address
// is looked up once per device.
static __device__ int g_rmsnorm_device_status;
static std::mutex g_status_mutex;
static int *g_status_ptr[64];

static cudaError_t status_word(int dev, int **out) {
    std::lock_guard<std::mutex> lk(g_status_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_rmsnorm_device_status);
        if (e != cudaSuccess) return e;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    *out = g_status_ptr[dev];
    return cudaSuccess;
}

constexpr int kMaxDevices = 64;
static std::atomic<int> g_sm_count[kMaxDevices];

static cudaError_t device_sms(int *dev_out, int *sms_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int sms = g_sm_count[dev].load(std::memory_order_relaxed);
    if (sms <= 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    *dev_out = dev;
    *sms_out = sms;
    return cudaSuccess;
}

// The kernels of a call's type pair. `peel`: the instantiation for rows at a
// common offset, which exists for the default vectorised plans of the types
// whose weight is the activations' type (NULL elsewhere).
static const void *bwd_kernel(int plan_id, int dt, bool fused, bool packed, bool peel = false) {
    if (peel) {
        switch (kind_of(dt)) {
        case 0: return bwd_main_kernel_ptr_peel_f32(plan_id, fused, packed);
        case 1: return bwd_main_kernel_ptr_peel_bf16(plan_id, fused, packed);
        case 2: return bwd_main_kernel_ptr_peel_f16(plan_id, fused, packed);
        default: return nullptr;
        }
    }
    switch (kind_of(dt)) {
    case 1: return bwd_main_kernel_ptr_bf16(plan_id, fused, packed);
    case 2: return bwd_main_kernel_ptr_f16(plan_id, fused, packed);
    case 3: return bwd_main_kernel_ptr_bf16w32(plan_id, fused, packed);
    case 4: return bwd_main_kernel_ptr_f16w32(plan_id, fused, packed);
    default: return bwd_main_kernel_ptr_f32(plan_id, fused, packed);
    }
}

static const void *ln_bwd_kernel(int plan_id, int dt, bool fused, bool peel = false) {
    if (peel) {
        switch (kind_of(dt)) {
        case 0: return ln_bwd_kernel_ptr_peel_f32(plan_id, fused);
        case 1: return ln_bwd_kernel_ptr_peel_bf16(plan_id, fused);
        case 2: return ln_bwd_kernel_ptr_peel_f16(plan_id, fused);
        default: return nullptr;
        }
    }
    switch (kind_of(dt)) {
    case 1: return ln_bwd_kernel_ptr_bf16(plan_id, fused);
    case 2: return ln_bwd_kernel_ptr_f16(plan_id, fused);
    case 3: return ln_bwd_kernel_ptr_bf16w32(plan_id, fused);
    case 4: return ln_bwd_kernel_ptr_f16w32(plan_id, fused);
    default: return ln_bwd_kernel_ptr_f32(plan_id, fused);
    }
}

static const void *fwd_staged_kernel(int plan_id, int dt, bool fused, bool ln, bool peel = false) {
    if (peel) {
        switch (kind_of(dt)) {
        case 0:
            return ln ? ln_fwd_staged_kernel_ptr_peel_f32(plan_id, fused) : fwd_staged_kernel_ptr_peel_f32(plan_id, fused);
        case 1:
            return ln ? ln_fwd_staged_kernel_ptr_peel_bf16(plan_id, fused)
                      : fwd_staged_kernel_ptr_peel_bf16(plan_id, fused);
        case 2:
            return ln ? ln_fwd_staged_kernel_ptr_peel_f16(plan_id, fused) : fwd_staged_kernel_ptr_peel_f16(plan_id, fused);
        default: return nullptr;
        }
    }
    if (ln) {
        switch (kind_of(dt)) {
        case 1: return ln_fwd_staged_kernel_ptr_bf16(plan_id, fused);
        case 2: return ln_fwd_staged_kernel_ptr_f16(plan_id, fused);
        case 3: return ln_fwd_staged_kernel_ptr_bf16w32(plan_id, fused);
        case 4: return ln_fwd_staged_kernel_ptr_f16w32(plan_id, fused);
        default: return ln_fwd_staged_kernel_ptr_f32(plan_id, fused);
        }
    }
    switch (kind_of(dt)) {
    case 1: return fwd_staged_kernel_ptr_bf16(plan_id, fused);
    case 2: return fwd_staged_kernel_ptr_f16(plan_id, fused);
    case 3: return fwd_staged_kernel_ptr_bf16w32(plan_id, fused);
    case 4: return fwd_staged_kernel_ptr_f16w32(plan_id, fused);
    default: return fwd_staged_kernel_ptr_f32(plan_id, fused);
    }
}

static const void *fwd8_staged_kernel(int plan_id, int dt, bool fused, int mode) {
    switch (kind_of(dt)) {
    case 1: return fwd8_staged_kernel_ptr_bf16(plan_id, fused, mode);
    case 2: return fwd8_staged_kernel_ptr_f16(plan_id, fused, mode);
    case 3: return fwd8_staged_kernel_ptr_bf16w32(plan_id, fused, mode);
    case 4: return fwd8_staged_kernel_ptr_f16w32(plan_id, fused, mode);
    default: return fwd8_staged_kernel_ptr_f32(plan_id, fused, mode);
    }
}

// The E4M3 forward of the call's type pair (stages > 0: a staged plan).
static int launch_fwd8_dt(int dt, int plan_id, bool fused, int mode, const FwdParams &p, int grid, int stages,
                          int smem, void *stream) {
    switch (kind_of(dt)) {
    case 1: return stages > 0 ? launch_fwd8_staged_bf16(plan_id, fused, mode, p, grid, smem, stream)
                              : launch_fwd8_bf16(plan_id, fused, mode, p, grid, stream);
    case 2: return stages > 0 ? launch_fwd8_staged_f16(plan_id, fused, mode, p, grid, smem, stream)
                              : launch_fwd8_f16(plan_id, fused, mode, p, grid, stream);
    case 3: return stages > 0 ? launch_fwd8_staged_bf16w32(plan_id, fused, mode, p, grid, smem, stream)
                              : launch_fwd8_bf16w32(plan_id, fused, mode, p, grid, stream);
    case 4: return stages > 0 ? launch_fwd8_staged_f16w32(plan_id, fused, mode, p, grid, smem, stream)
                              : launch_fwd8_f16w32(plan_id, fused, mode, p, grid, stream);
    default: return stages > 0 ? launch_fwd8_staged_f32(plan_id, fused, mode, p, grid, smem, stream)
                               : launch_fwd8_f32(plan_id, fused, mode, p, grid, stream);
    }
}

// Launches by type pair; rows at a common offset (p.peel > 0) take the
// PEEL instantiations.
static int launch_fwd_staged_dt(int dt, bool ln, int plan_id, bool fused, const FwdParams &p, int grid, int smem,
                                void *stream) {
    if (p.peel > 0) {
        switch (kind_of(dt)) {
        case 0: return ln ? launch_ln_fwd_staged_peel_f32(plan_id, fused, p, grid, smem, stream)
                          : launch_fwd_staged_peel_f32(plan_id, fused, p, grid, smem, stream);
        case 1: return ln ? launch_ln_fwd_staged_peel_bf16(plan_id, fused, p, grid, smem, stream)
                          : launch_fwd_staged_peel_bf16(plan_id, fused, p, grid, smem, stream);
        case 2: return ln ? launch_ln_fwd_staged_peel_f16(plan_id, fused, p, grid, smem, stream)
                          : launch_fwd_staged_peel_f16(plan_id, fused, p, grid, smem, stream);
        default: return (int)cudaErrorInvalidValue;
        }
    }
    if (ln) {
        switch (kind_of(dt)) {
        case 1: return launch_ln_fwd_staged_bf16(plan_id, fused, p, grid, smem, stream);
        case 2: return launch_ln_fwd_staged_f16(plan_id, fused, p, grid, smem, stream);
        case 3: return launch_ln_fwd_staged_bf16w32(plan_id, fused, p, grid, smem, stream);
        case 4: return launch_ln_fwd_staged_f16w32(plan_id, fused, p, grid, smem, stream);
        default: return launch_ln_fwd_staged_f32(plan_id, fused, p, grid, smem, stream);
        }
    }
    switch (kind_of(dt)) {
    case 1: return launch_fwd_staged_bf16(plan_id, fused, p, grid, smem, stream);
    case 2: return launch_fwd_staged_f16(plan_id, fused, p, grid, smem, stream);
    case 3: return launch_fwd_staged_bf16w32(plan_id, fused, p, grid, smem, stream);
    case 4: return launch_fwd_staged_f16w32(plan_id, fused, p, grid, smem, stream);
    default: return launch_fwd_staged_f32(plan_id, fused, p, grid, smem, stream);
    }
}

static int launch_fwd_dt(int dt, int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    if (p.peel > 0) {
        switch (kind_of(dt)) {
        case 0: return launch_fwd_peel_f32(plan_id, fused, p, grid, stream);
        case 1: return launch_fwd_peel_bf16(plan_id, fused, p, grid, stream);
        case 2: return launch_fwd_peel_f16(plan_id, fused, p, grid, stream);
        default: return (int)cudaErrorInvalidValue;
        }
    }
    switch (kind_of(dt)) {
    case 1: return launch_fwd_bf16(plan_id, fused, p, grid, stream);
    case 2: return launch_fwd_f16(plan_id, fused, p, grid, stream);
    case 3: return launch_fwd_bf16w32(plan_id, fused, p, grid, stream);
    case 4: return launch_fwd_f16w32(plan_id, fused, p, grid, stream);
    default: return launch_fwd_f32(plan_id, fused, p, grid, stream);
    }
}

static int launch_bwd_dt(int dt, int plan_id, bool fused, bool packed, const BwdParams &p, int grid, int smem,
                         void *stream) {
    if (p.peel > 0) {
        switch (kind_of(dt)) {
        case 0: return launch_bwd_main_peel_f32(plan_id, fused, packed, p, grid, smem, stream);
        case 1: return launch_bwd_main_peel_bf16(plan_id, fused, packed, p, grid, smem, stream);
        case 2: return launch_bwd_main_peel_f16(plan_id, fused, packed, p, grid, smem, stream);
        default: return (int)cudaErrorInvalidValue;
        }
    }
    switch (kind_of(dt)) {
    case 1: return launch_bwd_main_bf16(plan_id, fused, packed, p, grid, smem, stream);
    case 2: return launch_bwd_main_f16(plan_id, fused, packed, p, grid, smem, stream);
    case 3: return launch_bwd_main_bf16w32(plan_id, fused, packed, p, grid, smem, stream);
    case 4: return launch_bwd_main_f16w32(plan_id, fused, packed, p, grid, smem, stream);
    default: return launch_bwd_main_f32(plan_id, fused, packed, p, grid, smem, stream);
    }
}

// dW is written in the weight's storage type.
static int launch_finalize_dt(int dt, const float *ws, int parts, int ncols, void *out0, void *out1, int split,
                              int peel, void *stream, bool serial, int sms) {
    switch (kind_of(dt)) {
    case 1: return launch_dw_finalize_bf16(ws, parts, ncols, out0, out1, split, peel, stream, serial, sms);
    case 2: return launch_dw_finalize_f16(ws, parts, ncols, out0, out1, split, peel, stream, serial, sms);
    default: return launch_dw_finalize_f32(ws, parts, ncols, out0, out1, split, peel, stream, serial, sms);
    }
}

// Largest number of backward dW partial rows worth launching for a plan:
// resident CTAs on the device (resident clusters for a cluster plan), the
// minimum over its packed and scalar variants, and its instantiations for
// aligned rows and rows at a common offset, for the given fusion mode, so
// that all of them use the same count (and dW the same summation order,
// and the workspace the same size whatever the rows' offset).
// Cached per device, kernel kind, plan and mode.
static std::mutex g_occ_mutex;
static int g_parts_cache[kMaxDevices][kNumKinds][2][kMaxPlanId];
static int g_cps_cache[kMaxDevices][kNumKinds][2][kMaxPlanId];

static cudaError_t bwd_max_parts(int dev, int sms, int dt, const PlanDesc &d, int64_t N, bool fused,
                                 int *parts_out, int *cps_out) {
    const int slot = d.id;
    if (slot < 0 || slot >= kMaxPlanId) return cudaErrorInvalidValue;
    const int dti = kind_of(dt);
    const int fi = fused ? 1 : 0;
    {
        std::lock_guard<std::mutex> lk(g_occ_mutex);
        if (g_parts_cache[dev][dti][fi][slot] > 0) {
            *parts_out = g_parts_cache[dev][dti][fi][slot];
            *cps_out = g_cps_cache[dev][dti][fi][slot];
            return cudaSuccess;
        }
    }
    const int threads = cta_threads(d);
    const int E = 16 / elem_size(dt);
    // The dynamic shared memory of the team combine depends on N; occupancy
    // is taken for the largest N the plan serves (the conservative value).
    const int64_t nmax = !generic_path(d.path) ? plan_capacity(d) * E : N;
    // (a staged plan's rows may need less than its capacity: the occupancy
    // query is capped at the largest shared memory a CTA may take)
    const int smem = staged_path(d.path)
                         ? (int)std::min<int64_t>(staged_smem_bytes(d, plan_capacity(d), 1, fused), kMaxDynamicSmem)
                     : d.path == PATH_STREAM
                         ? (int)std::min<int64_t>(stream_smem_at(d, (int64_t)d.tpr * d.v, elem_size(dt), fused, d.depth),
                                                  kMaxDynamicSmem)
                         : bwd_smem_bytes(d, nmax);
    int best = 1 << 30;
    // rows at a common offset: default vectorised plans, weight in the activations' type
    const bool has_peel = row_path(d.path) && d.cmin > 0 && !mixed_kind(kind_of(dt));
    for (int var = 0; var < 4; ++var) {
        const int pk = var & 1;
        const bool pe = var >= 2;
        if (pe && !has_peel) continue;
        // the LayerNorm and generic kernels have one variant; a staged plan
        // has the scalar one only where staged_scalar_variant says so
        if ((generic_path(d.path) || d.op == OP_LN_BWD) && pk == 1) continue;
        if (staged_path(d.path) && pk == 0 && !staged_scalar_variant(kind_of(dt), d.cmin)) continue;
        const void *k =
            d.op == OP_LN_BWD ? ln_bwd_kernel(d.id, dt, fused, pe) : bwd_kernel(d.id, dt, fused, pk != 0, pe);
        if (!k) return cudaErrorInvalidDeviceFunction;
        if (staged_path(d.path) || d.path == PATH_STREAM) {  // more than 48 KB of dynamic shared memory needs an opt-in
            cudaError_t e = (cudaError_t)allow_staged_smem(k);
            if (e != cudaSuccess) return e;
        }
        int n = 0;
        cudaError_t e;
        if (d.cs > 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(d.cs * sms));
            cfg.blockDim = dim3((unsigned)threads);
            cfg.dynamicSmemBytes = (size_t)smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)d.cs;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
        } else {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem);
            n *= sms;
        }
        if (e != cudaSuccess) return e;
        if (n < best) best = n;
    }
    // A kernel that cannot be resident at all (its shared memory or
    // registers exceed an SM) must not run as one serial CTA: refuse it.
    if (best < 1) return cudaErrorInvalidConfiguration;
    const int cps = (int)(((int64_t)best * d.cs + sms - 1) / sms);
    std::lock_guard<std::mutex> lk(g_occ_mutex);
    g_parts_cache[dev][dti][fi][slot] = best;
    g_cps_cache[dev][dti][fi][slot] = cps;
    *parts_out = best;
    *cps_out = cps;
    return cudaSuccess;
}

// ----------------------------------------------------- argument checks --

static bool aligned_to(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// How a call's row arrays (and its weight, when given) sit in memory:
//   0   every one 16-byte aligned: the vectorised kernels;
//   k   every one k elements past a 16-byte boundary (one common offset),
//       rows of whole 16-byte chunks, the weight in the activations' type:
//       the vectorised kernels, each row spanning one chunk more, the two
//       edge chunks split with the neighbouring rows;
//  -1   anything else: the generic kernels.
// Rows of whole chunks keep every row at the first row's offset.
static int row_layout(int dt, int64_t N, std::initializer_list<const void *> rows, const void *w) {
    const int s = elem_size(dt);
    if ((N * s) % 16 != 0) return -1;
    const uintptr_t a = (uintptr_t)*rows.begin() & 15u;
    for (const void *p : rows)
        if (((uintptr_t)p & 15u) != a) return -1;
    if (w && ((uintptr_t)w & 15u) != a) return -1;
    if (a == 0) return 0;
    if (mixed_kind(kind_of(dt))) return -1;  // an fp32 weight: aligned rows only
    return (int)(a / (uintptr_t)s);
}

// A row pointer as the vectorised kernels take it: moved back to the
// 16-byte boundary below the rows' common offset.
static const void *to_chunk_base(const void *p, int peel, int es) {
    return (p && peel > 0) ? static_cast<const char *>(p) - (ptrdiff_t)peel * es : p;
}
static void *to_chunk_base(void *p, int peel, int es) {
    return (p && peel > 0) ? static_cast<char *>(p) - (ptrdiff_t)peel * es : p;
}

static bool finite_scalar(float v) { return std::isfinite(v); }

// Resident units (CTAs, or clusters) of a staged forward plan on the
// device, taken at the plan's largest rows (the conservative value) and
// cached per device, type, fusion mode, RMSNorm/LayerNorm, output mode and
// row layout (`peel`: the instantiation for rows at a common offset, whose
// row buffers are one slot longer). The forward keeps no partial rows, so
// the two layouts may differ in their unit count.
static std::map<uint64_t, int> g_sfwd_parts;

static cudaError_t staged_fwd_parts(int dev, int sms, int dt, const PlanDesc &d, bool fused, bool ln, int qmode,
                                    bool peel, int *parts_out) {
    if (d.id < 0 || d.id >= kMaxPlanId || qmode < 0 || qmode > QOUT_F16) return cudaErrorInvalidValue;
    if (peel && (qmode != QOUT_NONE || d.path == PATH_STREAM)) return cudaErrorInvalidValue;
    const uint64_t key =
        (((((((uint64_t)dev * kNumKinds + kind_of(dt)) * 2 + (fused ? 1 : 0)) * 2 + (ln ? 1 : 0)) * 2 + (peel ? 1 : 0)) *
              (QOUT_F16 + 1) +
          (uint64_t)qmode) *
         kMaxPlanId) +
        (uint64_t)d.id;
    {
        std::lock_guard<std::mutex> lk(g_occ_mutex);
        auto it = g_sfwd_parts.find(key);
        if (it != g_sfwd_parts.end()) {
            *parts_out = it->second;
            return cudaSuccess;
        }
    }
    const void *k = qmode != QOUT_NONE ? fwd8_staged_kernel(d.id, dt, fused, qmode)
                                       : fwd_staged_kernel(d.id, dt, fused, ln, peel);
    if (!k) return cudaErrorInvalidDeviceFunction;
    cudaError_t e = (cudaError_t)allow_staged_smem(k);
    if (e != cudaSuccess) return e;
    const int64_t sm = d.path == PATH_STREAM ? stream_smem_at(d, (int64_t)d.tpr * d.v, elem_size(dt), fused, d.depth)
                                             : staged_smem_bytes(d, plan_capacity(d), peel ? 1 : 0, fused);
    const int smem = (int)std::min<int64_t>(sm, kMaxDynamicSmem);
    int n = 0;
    if (d.cs > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(d.cs * sms));
        cfg.blockDim = dim3((unsigned)d.tpr);
        cfg.dynamicSmemBytes = (size_t)smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)d.cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, d.tpr, smem);
        n *= sms;
    }
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;  // not resident at all: refuse
    std::lock_guard<std::mutex> lk(g_occ_mutex);
    g_sfwd_parts[key] = n;
    *parts_out = n;
    return cudaSuccess;
}

// A forward on a staged plan: the grid becomes the resident units walking
// the rows, and the stages in use, the shared memory and the status word
// are set. Other plans are left as they are.
static rmsnorm_status_t prepare_staged_fwd(int64_t M, int64_t N, int dt, int peel, bool fused, bool ln,
                                           int qmode, int force_plan, rmsnorm_plan_t *plan, int *stages,
                                           int **status) {
    *stages = 0;
    *status = nullptr;
    const PlanDesc *d = find_plan(plan->plan_id);
    if (!d || d->op != OP_FWD_STAGED) return RMSNORM_SUCCESS;
    const bool stream = d->path == PATH_STREAM;
    // the streamed generic forward serves the RMSNorm forward in the activations' type
    if (stream && (ln || qmode != QOUT_NONE)) return RMSNORM_ERR_UNSUPPORTED;
    const int es = elem_size(dt);
    const int64_t C = N * es / 16;
    const int pk = peel > 0 ? peel : 0;
    const int depth = stream ? stream_depth(*d, N, es, fused) : staged_depth(*d, C, pk, fused);
    if (depth == 0) return RMSNORM_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    cudaError_t e = device_sms(&dev, &sms);
    if (e != cudaSuccess) return cuda_fail(e);
    int parts = 1;
    e = staged_fwd_parts(dev, sms, dt, *d, fused, ln, qmode, pk > 0, &parts);
    if (e != cudaSuccess) return cuda_fail(e);
    rmsnorm_status_t st = select_plan(RMSNORM_OP_FWD, M, N, dt, peel, parts, 0, force_plan, 0, plan, stream);
    if (st != RMSNORM_SUCCESS) return st;
    plan->smem_bytes = (int32_t)(stream ? stream_smem_at(*d, N, es, fused, depth) : staged_smem_bytes(*d, C, pk, fused));
    e = status_word(dev, status);
    if (e != cudaSuccess) return cuda_fail(e);
    *stages = depth;
    return RMSNORM_SUCCESS;
}

static std::atomic<int> g_table_ok{-1};

int self_check_impl() {
    int bad = 0;
    for (int op = 0; op < 3; ++op) {
        for (int dt = 0; dt < 3; ++dt) {  // the activations' type decides the defaults
            int64_t expect = 1;
            for (int i = 0; i < kNumPlans; ++i) {
                const PlanDesc &d = kPlans[i];
                if (d.op != op || !row_path(d.path) || d.cmin == 0 || !(d.dtm & dtype_bit(dt))) continue;
                // ranges of a dtype's default plans must tile [1, max] in table order
                if (d.cmin != expect || d.cmax < d.cmin) ++bad;
                expect = d.cmax + 1;
                // the plan must hold every chunk of the largest row it serves
                if (plan_capacity(d) < d.cmax) ++bad;
                // both ends of its range must select it again
                if (default_vector_plan(op, dt, d.cmin) != &d || default_vector_plan(op, dt, d.cmax) != &d) ++bad;
            }
        }
        if (!generic_plan(op)) ++bad;
    }
    // streamed defaults, backward and forward: ranges of N tiling [1, max] in table order
    for (int op : {(int)OP_BWD, (int)OP_FWD_STAGED}) {
        int64_t expect = 1;
        for (int i = 0; i < kNumPlans; ++i) {
            const PlanDesc &d = kPlans[i];
            if (d.op != op || d.path != PATH_STREAM || d.cmin == 0) continue;
            if (d.cmin != expect || d.cmax < d.cmin) ++bad;
            expect = d.cmax + 1;
        }
    }
    // staged forward defaults: contiguous ranges (they need not start at 1),
    // each selecting its entry and held by it
    for (int dt = 0; dt < 3; ++dt) {
        int64_t expect = -1;
        for (int i = 0; i < kNumPlans; ++i) {
            const PlanDesc &d = kPlans[i];
            if (d.op != OP_FWD_STAGED || d.path == PATH_STREAM || d.cmin == 0 || !(d.dtm & dtype_bit(dt))) continue;
            if ((expect >= 0 && d.cmin != expect) || d.cmax < d.cmin || plan_capacity(d) < d.cmax) ++bad;
            expect = d.cmax + 1;
            if (default_vector_plan(OP_FWD_STAGED, dt, d.cmin) != &d ||
                default_vector_plan(OP_FWD_STAGED, dt, d.cmax) != &d)
                ++bad;
        }
    }
    for (int i = 0; i < kNumPlans; ++i) {
        const PlanDesc &d = kPlans[i];
        if (find_plan(d.id) != &d) ++bad;  // ids unique
        if (d.op == OP_FWD_STAGED && d.path != PATH_RESTAGED && d.path != PATH_STREAM) ++bad;
        if (d.path == PATH_VECTOR) {
            const bool pow2 = d.tpr > 0 && (d.tpr & (d.tpr - 1)) == 0;
            if (!pow2 || d.tpr * d.teams > kMaxCtaThreads || d.tpr * d.teams < 32 || d.v < 1) ++bad;
            // a cluster row has one team per CTA, of whole warps, and at most 8 CTAs
            if (d.cs < 1 || d.cs > 8 || (d.cs > 1 && (d.teams != 1 || d.tpr < 32))) ++bad;
        }
        if (staged_path(d.path)) {
            // one team per CTA of whole warps, at least two stages, backward
            // only; a cluster (2, 4 or 8 CTAs) only on the re-read schedule
            if (d.op == OP_FWD || (d.op == OP_FWD_STAGED && d.path != PATH_RESTAGED) ||
                !staged_plan(d.path, d.teams, d.cs) || d.depth < 2 || d.tpr % 32 != 0 || d.tpr < 64 ||
                d.tpr > kMaxCtaThreads || d.v < 1)
                ++bad;
        }
        // a streamed generic kernel: a backward or a forward of whole warps
        // with 2..8 stages that holds the longest row of its range
        if (d.path == PATH_STREAM && ((d.op != OP_BWD && d.op != OP_FWD_STAGED) || d.tpr % 32 != 0 || d.tpr < 64 || d.tpr > kMaxCtaThreads ||
                                      d.v < 1 || d.depth < 2 || d.depth > 8 || d.teams != 1 ||
                                      d.cs != 1 || (int64_t)d.tpr * d.v < d.cmax))
            ++bad;
        if (d.dtm < 1 || d.dtm > DT_ANY) ++bad;
        if (d.id < 0 || d.id >= kMaxPlanId) ++bad;
    }
    return bad;
}

static bool table_ok() {
    int s = g_table_ok.load(std::memory_order_relaxed);
    if (s < 0) {
        s = self_check_impl() == 0 ? 1 : 0;
        g_table_ok.store(s, std::memory_order_relaxed);
    }
    return s == 1;
}

// Run the table check when the library is loaded.
static const bool g_loaded_check = [] {
    if (!table_ok()) std::fprintf(stderr, "librmsnorm_gb300: plan table self-check failed\n");
    return true;
}();

// ------------------------------------------------- generic-kernel note --
// Optional one-time note on stderr when a call falls to the generic kernels
// (the counterpart of the fallback warning the TransformerEngine tuning page
// prints the first time no tuned kernel serves a config, "[ROCm] RMSNorm
// tuning", Description). Off by default; rmsnorm_set_generic_note switches
// it. One note per kind of call (forward, backward, LayerNorm forward and
// backward) until the switch is set again.
static std::atomic<int> g_note_on{0};
static std::atomic<unsigned> g_noted{0};
enum : unsigned { NOTE_FWD = 1, NOTE_BWD = 2, NOTE_LN_FWD = 4, NOTE_LN_BWD = 8 };

static const char *dtype_name(int dt) {
    switch (dt) {
    case RMSNORM_F32: return "fp32";
    case RMSNORM_BF16: return "bf16";
    case RMSNORM_F16: return "fp16";
    case RMSNORM_BF16_W32: return "bf16, fp32 weight";
    case RMSNORM_F16_W32: return "fp16, fp32 weight";
    default: return "?";
    }
}

static void note_generic(unsigned kind, int64_t N, int dt) {
    if (!g_note_on.load(std::memory_order_relaxed)) return;
    if (g_noted.fetch_or(kind, std::memory_order_relaxed) & kind) return;
    const char *op = kind == NOTE_FWD ? "rmsnorm forward"
                     : kind == NOTE_BWD ? "rmsnorm backward"
                     : kind == NOTE_LN_FWD ? "layernorm forward" : "layernorm backward";
    const bool whole = (N * elem_size(dt)) % 16 == 0;
    std::fprintf(stderr,
                 "librmsnorm_gb300: %s, N=%lld, %s: falling back to the generic kernel (%s); "
                 "later such calls are not reported\n",
                 op, (long long)N, dtype_name(dt),
                 whole ? "the arrays are not all 16-byte aligned at one common offset"
                       : "a row is not a whole number of 16-byte chunks");
}

// --------------------------------------------------------------- forward --

// Quantised output of the forward (E4M3); qmode QOUT_NONE is the plain
// forward and ignores the other three.
struct QuantOut {
    int qmode;
    const float *scale;
    float *scale_inv;
    float *amax;
};

static rmsnorm_status_t fwd_impl(const void *x, const void *residual, const void *w, void *y,
                                 void *residual_out, float *rstd, int64_t M, int64_t N, int dt_arg, float eps,
                                 float offset, cudaStream_t stream, int force_plan, rmsnorm_plan_t *used,
                                 const QuantOut &q_arg = QuantOut{QOUT_NONE, nullptr, nullptr, nullptr}) {
    if (!table_ok()) return RMSNORM_ERR_UNSUPPORTED;
    // fp32 activations with y in bf16 or fp16 (RMSNORM_OUT_BF16 / _F16): the
    // kernels' narrow output modes, on the E4M3 forward's launch path
    int dt = dt_arg;
    QuantOut q = q_arg;
    const int om = dt & (RMSNORM_OUT_BF16 | RMSNORM_OUT_F16);
    if (om != 0) {
        dt &= ~(RMSNORM_OUT_BF16 | RMSNORM_OUT_F16);
        if (om == (RMSNORM_OUT_BF16 | RMSNORM_OUT_F16) || base_dtype(dt) != RMSNORM_F32)
            return RMSNORM_ERR_INVALID_ARG;
        if (q.qmode != QOUT_NONE) return RMSNORM_ERR_UNSUPPORTED;  // E4M3 is an output type of its own
        q = QuantOut{om == RMSNORM_OUT_BF16 ? QOUT_BF16 : QOUT_F16, nullptr, nullptr, nullptr};
    }
    if (!valid_dtype(dt)) return RMSNORM_ERR_INVALID_ARG;
    if (N < 1 || N > RMSNORM_MAX_N || M < 0 || M > 0x7fffffffLL) return RMSNORM_ERR_INVALID_ARG;
    if (!finite_scalar(eps) || !finite_scalar(offset) || eps < 0.f) return RMSNORM_ERR_INVALID_ARG;
    // quant: y in another type than x (E4M3, or the narrow outputs)
    const bool quant = q.qmode != QOUT_NONE;
    if (fp8_out(q.qmode)) {
        if (q.qmode == QOUT_FP8_TENSOR && (!q.scale || !aligned_to(q.scale, 4))) return RMSNORM_ERR_INVALID_ARG;
        if (q.qmode == QOUT_FP8_ROW && (q.scale || (M > 0 && !q.scale_inv))) return RMSNORM_ERR_INVALID_ARG;
        if ((q.scale_inv && !aligned_to(q.scale_inv, 4)) || (q.amax && !aligned_to(q.amax, 4)))
            return RMSNORM_ERR_INVALID_ARG;
    }
    // The max over this call's rows starts from 0 (also the empty max).
    auto clear_amax = [&]() -> cudaError_t {
        return (quant && q.amax) ? cudaMemsetAsync(q.amax, 0, sizeof(float), stream) : cudaSuccess;
    };
    // An empty batch reads and writes nothing; its (empty) tensors may be NULL.
    if (M == 0) {
        cudaError_t e = clear_amax();
        return e == cudaSuccess ? RMSNORM_SUCCESS : cuda_fail(e);
    }
    const bool fused = residual != nullptr || residual_out != nullptr;
    if (fused && (!residual || !residual_out)) return RMSNORM_ERR_INVALID_ARG;
    if (!x || !y || !rstd) return RMSNORM_ERR_INVALID_ARG;  // w NULL: non-affine
    const uintptr_t s = (uintptr_t)elem_size(dt);
    const uintptr_t ws_ = (uintptr_t)weight_size(dt);
    const uintptr_t ys = fp8_out(q.qmode) ? 1 : (narrow_out(q.qmode) ? 2 : s);
    if (!aligned_to(x, s) || (w && !aligned_to(w, ws_)) || !aligned_to(y, ys) || !aligned_to(rstd, 4))
        return RMSNORM_ERR_INVALID_ARG;
    if (fused && (!aligned_to(residual, s) || !aligned_to(residual_out, s))) return RMSNORM_ERR_INVALID_ARG;

    int peel = fused ? row_layout(dt, N, {x, y, residual, residual_out}, w) : row_layout(dt, N, {x, y}, w);
    if (quant) {
        // E4M3 or narrow output: 16-byte aligned rows only
        const int in = fused ? row_layout(dt, N, {x, residual, residual_out}, w) : row_layout(dt, N, {x}, w);
        peel = (in == 0 && aligned_to(y, 16)) ? 0 : -1;
    }

    rmsnorm_plan_t plan;
    rmsnorm_status_t st = select_plan(RMSNORM_OP_FWD, M, N, dt, peel, 1, 0, force_plan, 0, &plan, !quant);
    if (st != RMSNORM_SUCCESS) return st;
    // the E4M3 and narrow-output kernels are compiled for the default plans and the generic one
    if (quant && force_plan >= 0 && plan.path != PATH_GENERIC && find_plan(plan.plan_id)->cmin == 0)
        return RMSNORM_ERR_UNSUPPORTED;
    if (plan.path == PATH_GENERIC && force_plan < 0) note_generic(NOTE_FWD, N, dt);
    int stages = 0;
    int *status = nullptr;
    st = prepare_staged_fwd(M, N, dt, peel, fused, false, q.qmode, force_plan, &plan, &stages, &status);
    if (st != RMSNORM_SUCCESS) return st;

    // rows at a common offset: every row pointer moved back to the 16-byte
    // boundary below it (plan.peel is 0 for aligned rows and the generic kernels)
    const int pl = plan.peel;
    const int es = (int)s;
    FwdParams p;
    p.x = to_chunk_base(x, pl, es);
    p.residual = to_chunk_base(residual, pl, es);
    p.w = to_chunk_base(w, pl, es);
    p.y = to_chunk_base(y, pl, es);
    p.residual_out = to_chunk_base(residual_out, pl, es);
    p.peel = pl;
    p.rstd = rstd;
    p.M = M;
    p.N = (int)N;
    p.eps = eps;
    p.offset = offset;
    p.qscale = q.scale;
    p.qscale_inv = q.scale_inv;
    p.qamax = reinterpret_cast<unsigned int *>(q.amax);
    p.beta = nullptr;
    p.mean = nullptr;
    p.stages = stages;
    p.status = status;
    int le;
    if (quant) {
        cudaError_t e = clear_amax();
        if (e != cudaSuccess) return cuda_fail(e);
        le = launch_fwd8_dt(dt, plan.plan_id, fused, q.qmode, p, plan.ctas, stages, plan.smem_bytes, stream);
    } else if (stages > 0) {
        le = launch_fwd_staged_dt(dt, false, plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream);
    } else {
        le = launch_fwd_dt(dt, plan.plan_id, fused, p, plan.ctas, stream);
    }
    if (le != 0) return cuda_fail((cudaError_t)le);
    if (used) *used = plan;
    return RMSNORM_SUCCESS;
}

// -------------------------------------------------------------- backward --

// The plan a backward call (op RMSNORM_OP_BWD or RMSNORM_OP_LN_BWD) runs on
// the current device: the row layout of its arrays, the table entry, the
// CTA count from the device's occupancy, and a staged plan's shared memory.
// The entry points and the exact workspace query share it.
struct BwdCall {
    rmsnorm_plan_t plan;
    const PlanDesc *d;
    int dev, sms, cps;
};

static rmsnorm_status_t plan_bwd_call(int op, const void *dy, const void *dres, const void *x, const void *w,
                                      const void *dx, int64_t M, int64_t N, int dt, bool fused, int force_plan,
                                      int force_ctas, BwdCall *c) {
    const int peel = dres ? row_layout(dt, N, {dy, x, dx, dres}, w) : row_layout(dt, N, {dy, x, dx}, w);
    cudaError_t e = device_sms(&c->dev, &c->sms);
    if (e != cudaSuccess) return cuda_fail(e);
    rmsnorm_status_t st = select_plan(op, M, N, dt, peel, 1, 0, force_plan, force_ctas, &c->plan);
    if (st != RMSNORM_SUCCESS) return st;
    c->d = find_plan(c->plan.plan_id);
    const int64_t C = N * elem_size(dt) / 16;
    if (staged_path(c->d->path) && staged_smem_bytes(*c->d, C, c->plan.peel, fused) > kMaxDynamicSmem)
        return RMSNORM_ERR_UNSUPPORTED;
    int parts = 1;
    c->cps = 1;
    e = bwd_max_parts(c->dev, c->sms, dt, *c->d, N, fused, &parts, &c->cps);
    if (e != cudaSuccess) return cuda_fail(e);
    st = select_plan(op, M, N, dt, peel, parts, c->cps, force_plan, force_ctas, &c->plan);
    if (st != RMSNORM_SUCCESS) return st;
    // the stages this call's rows take (the fused variant holds three rows a stage)
    if (c->plan.path == PATH_STAGED) c->plan.smem_bytes = (int32_t)staged_smem_bytes(*c->d, C, c->plan.peel, fused);
    if (c->d->path == PATH_STREAM) {
        const int es = elem_size(dt);
        c->plan.smem_bytes = (int32_t)stream_smem_at(*c->d, N, es, fused, stream_depth(*c->d, N, es, fused));
    }
    return RMSNORM_SUCCESS;
}

static rmsnorm_status_t bwd_impl(const void *dy, const void *dres, const void *x, const void *w,
                                 const float *rstd, void *dx, void *dw, void *workspace, size_t ws_bytes,
                                 int64_t M, int64_t N, int dt, float eps, float offset, cudaStream_t stream,
                                 bool fused, int force_plan, int force_ctas, int force_packed,
                                 void *event_after_main, rmsnorm_plan_t *used) {
    if (!table_ok()) return RMSNORM_ERR_UNSUPPORTED;
    if (!valid_dtype(dt)) return RMSNORM_ERR_INVALID_ARG;
    if (N < 1 || N > RMSNORM_MAX_N || M < 0 || M > 0x7fffffffLL) return RMSNORM_ERR_INVALID_ARG;
    if (!finite_scalar(eps) || !finite_scalar(offset) || eps < 0.f) return RMSNORM_ERR_INVALID_ARG;
    if (force_packed < -1 || force_packed > 1) return RMSNORM_ERR_INVALID_ARG;
    if (!fused) dres = nullptr;
    const uintptr_t s = (uintptr_t)elem_size(dt);
    const uintptr_t wsz = (uintptr_t)weight_size(dt);
    // Non-affine (w NULL): there is no dW, so dw must be NULL as well.
    if ((w == nullptr) != (dw == nullptr)) return RMSNORM_ERR_INVALID_ARG;
    const bool affine = w != nullptr;
    if (M == 0) {
        // dw is the empty sum; the empty [0, N] tensors may be NULL
        if (!affine) return RMSNORM_SUCCESS;
        if (!aligned_to(dw, wsz)) return RMSNORM_ERR_INVALID_ARG;
        cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)N * wsz, stream);
        if (e != cudaSuccess) return cuda_fail(e);
        return RMSNORM_SUCCESS;
    }
    if (!dy || !x || !rstd || !dx) return RMSNORM_ERR_INVALID_ARG;
    if (!aligned_to(dy, s) || !aligned_to(x, s) || (affine && (!aligned_to(w, wsz) || !aligned_to(dw, wsz))) ||
        !aligned_to(dx, s) || !aligned_to(rstd, 4) || (dres && !aligned_to(dres, s)))
        return RMSNORM_ERR_INVALID_ARG;
    if (workspace && !aligned_to(workspace, 16)) return RMSNORM_ERR_WORKSPACE;

    BwdCall call;
    rmsnorm_status_t st = plan_bwd_call(RMSNORM_OP_BWD, dy, dres, x, w, dx, M, N, dt, fused, force_plan,
                                        force_ctas, &call);
    if (st != RMSNORM_SUCCESS) return st;
    rmsnorm_plan_t &plan = call.plan;
    const PlanDesc *d = call.d;
    cudaError_t e;
    if (plan.path == PATH_GENERIC && force_plan < 0) note_generic(NOTE_BWD, N, dt);
    bool packed = plan.packed != 0;
    if (force_packed == 0) packed = false;
    if (force_packed == 1 && plan.path == PATH_VECTOR) packed = true;
    if (plan.path == PATH_STAGED) {
        // packed unless the scalar variant is asked for and compiled
        packed = force_packed != 0;
        if (!packed && !staged_scalar_variant(kind_of(dt), d->cmin)) return RMSNORM_ERR_UNSUPPORTED;
    }
    plan.packed = packed ? 1 : 0;

    float *ws = static_cast<float *>(workspace);
    bool owned = false;
    if (!affine) {
        ws = nullptr;  // non-affine: no dW partials, no workspace
    } else if (ws) {
        if (ws_bytes < (size_t)plan.workspace_bytes) return RMSNORM_ERR_WORKSPACE;
    } else {
        void *tmp = nullptr;
        e = cudaMallocAsync(&tmp, (size_t)plan.workspace_bytes, stream);
        if (e != cudaSuccess) return cuda_fail(e);
        ws = static_cast<float *>(tmp);
        owned = true;
    }

    int *status = nullptr;
    e = status_word(call.dev, &status);
    if (e != cudaSuccess) {
        if (owned) cudaFreeAsync(ws, stream);
        return cuda_fail(e);
    }

    // rows at a common offset: every row pointer moved back to the 16-byte
    // boundary below it (the partial rows come out rotated by pl columns)
    const int pl = plan.peel;
    const int es = (int)s;
    BwdParams p;
    p.status = status;
    p.dy = to_chunk_base(dy, pl, es);
    p.x = to_chunk_base(x, pl, es);
    p.w = to_chunk_base(w, pl, es);
    p.rstd = rstd;
    p.dres = to_chunk_base(dres, pl, es);
    p.dx = to_chunk_base(dx, pl, es);
    p.ws = ws;
    p.mean = nullptr;
    p.M = M;
    p.N = (int)N;
    p.offset = offset;
    p.peel = pl;
    p.stages = staged_path(d->path)       ? staged_depth(*d, N * es / 16, pl, fused)
               : d->path == PATH_STREAM ? stream_depth(*d, N, es, fused)
                                        : 0;
    int le = launch_bwd_dt(dt, plan.plan_id, fused, packed, p, plan.ctas, plan.smem_bytes, stream);
    if (le == 0 && event_after_main) le = (int)cudaEventRecord(static_cast<cudaEvent_t>(event_after_main), stream);
    if (le == 0 && affine)
        le = launch_finalize_dt(dt, ws, plan.ws_rows, (int)N, dw, nullptr, (int)N, pl, stream,
                                event_after_main != nullptr, call.sms);
    if (owned) {
        cudaError_t fe = cudaFreeAsync(ws, stream);
        if (le == 0 && fe != cudaSuccess) le = (int)fe;
    }
    if (le != 0) return cuda_fail((cudaError_t)le);
    if (used) *used = plan;
    return RMSNORM_SUCCESS;
}

// Bytes of workspace a backward (op RMSNORM_OP_BWD or RMSNORM_OP_LN_BWD)
// needs on the current device: the largest need over the row layouts
// (aligned, at a common offset, generic) and the plain and fused variants,
// so one size serves every call.
static size_t bwd_workspace_bytes(int op, int64_t M, int64_t N, int dt) {
    if (M <= 0 || N < 1 || N > RMSNORM_MAX_N || !valid_dtype(dt)) return 0;
    if (M > 0x7fffffffLL || !table_ok()) return 0;
    int dev = 0, sms = 0;
    if (device_sms(&dev, &sms) != cudaSuccess) return 0;
    size_t best = 0;
    // (every common offset gives the same plan: rows one chunk longer)
    for (int layout = -1; layout <= 1; ++layout) {
        for (int fused = 0; fused < 2; ++fused) {
            rmsnorm_plan_t plan;
            if (select_plan(op, M, N, dt, layout, 1, 0, -1, 0, &plan) != RMSNORM_SUCCESS)
                return 0;
            int parts = 1, cps = 1;
            if (bwd_max_parts(dev, sms, dt, *find_plan(plan.plan_id), N, fused != 0, &parts, &cps) !=
                cudaSuccess)
                return 0;
            if (select_plan(op, M, N, dt, layout, parts, cps, -1, 0, &plan) != RMSNORM_SUCCESS)
                return 0;
            if ((size_t)plan.workspace_bytes > best) best = (size_t)plan.workspace_bytes;
        }
    }
    return best;
}

// Bytes of workspace one RMSNorm backward call with these arrays needs on
// the current device (the plan the call itself selects); 0 without dW.
static size_t call_workspace_bytes(const void *dy, const void *dres, const void *x, const void *w, const void *dx,
                                   int64_t M, int64_t N, int dt, bool fused) {
    if (!w || !dy || !x || !dx || M <= 0 || M > 0x7fffffffLL || N < 1 || N > RMSNORM_MAX_N) return 0;
    if (!valid_dtype(dt) || !table_ok()) return 0;
    BwdCall call;
    if (plan_bwd_call(RMSNORM_OP_BWD, dy, fused ? dres : nullptr, x, w, dx, M, N, dt, fused, -1, 0, &call) !=
        RMSNORM_SUCCESS)
        return 0;
    return (size_t)call.plan.workspace_bytes;
}

// ------------------------------------------------------------- LayerNorm --

static rmsnorm_status_t ln_fwd_impl(const void *x, const void *residual, const void *gamma, const void *beta,
                                    void *y, void *residual_out, float *mean, float *rstd, int64_t M, int64_t N,
                                    int dt, float eps, float offset, cudaStream_t stream, int force_plan,
                                    rmsnorm_plan_t *used) {
    if (!table_ok()) return RMSNORM_ERR_UNSUPPORTED;
    if (!valid_dtype(dt)) return RMSNORM_ERR_INVALID_ARG;
    if (N < 1 || N > RMSNORM_MAX_N || M < 0 || M > 0x7fffffffLL) return RMSNORM_ERR_INVALID_ARG;
    if (!finite_scalar(eps) || !finite_scalar(offset) || eps < 0.f) return RMSNORM_ERR_INVALID_ARG;
    if (M == 0) return RMSNORM_SUCCESS;
    const bool fused = residual != nullptr || residual_out != nullptr;
    if (fused && (!residual || !residual_out)) return RMSNORM_ERR_INVALID_ARG;
    if (!x || !y || !mean || !rstd) return RMSNORM_ERR_INVALID_ARG;
    const uintptr_t s = (uintptr_t)elem_size(dt);
    const uintptr_t wsz = (uintptr_t)weight_size(dt);  // gamma and beta: the activations' type or fp32
    if (!aligned_to(x, s) || !aligned_to(y, s) || (gamma && !aligned_to(gamma, wsz)) ||
        (beta && !aligned_to(beta, wsz)) || !aligned_to(mean, 4) || !aligned_to(rstd, 4))
        return RMSNORM_ERR_INVALID_ARG;
    if (fused && (!aligned_to(residual, s) || !aligned_to(residual_out, s))) return RMSNORM_ERR_INVALID_ARG;
    // gamma and beta must share the rows' offset (beta as a second "row")
    int peel = fused ? row_layout(dt, N, {x, y, residual, residual_out}, gamma)
                     : row_layout(dt, N, {x, y}, gamma);
    if (peel >= 0 && beta && row_layout(dt, N, {x, beta}, nullptr) != peel) peel = -1;

    rmsnorm_plan_t plan;
    rmsnorm_status_t st = select_plan(RMSNORM_OP_FWD, M, N, dt, peel, 1, 0, force_plan, 0, &plan, false);
    if (st != RMSNORM_SUCCESS) return st;
    // the LayerNorm forward is compiled for the default plans and the generic one
    if (plan.path == PATH_VECTOR && find_plan(plan.plan_id)->cmin == 0) return RMSNORM_ERR_UNSUPPORTED;
    if (plan.path == PATH_GENERIC && force_plan < 0) note_generic(NOTE_LN_FWD, N, dt);
    int stages = 0;
    int *status = nullptr;
    st = prepare_staged_fwd(M, N, dt, peel, fused, true, QOUT_NONE, force_plan, &plan, &stages, &status);
    if (st != RMSNORM_SUCCESS) return st;

    const int pl = plan.peel;  // rows at a common offset: pointers moved back to the 16-byte boundary
    FwdParams p;
    std::memset(&p, 0, sizeof p);
    p.x = to_chunk_base(x, pl, (int)s);
    p.residual = to_chunk_base(residual, pl, (int)s);
    p.w = to_chunk_base(gamma, pl, (int)s);
    p.beta = to_chunk_base(beta, pl, (int)s);
    p.y = to_chunk_base(y, pl, (int)s);
    p.residual_out = to_chunk_base(residual_out, pl, (int)s);
    p.peel = pl;
    p.rstd = rstd;
    p.mean = mean;
    p.M = M;
    p.N = (int)N;
    p.eps = eps;
    p.offset = offset;
    p.stages = stages;
    p.status = status;
    p.cache_row = plan.path == PATH_GENERIC && N * (int64_t)s <= kGenericRowCache ? 1 : 0;
    int le;
    if (stages > 0) {
        le = launch_fwd_staged_dt(dt, true, plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream);
    } else if (p.peel > 0) {
        switch (kind_of(dt)) {
        case 0: le = launch_ln_fwd_peel_f32(plan.plan_id, fused, p, plan.ctas, stream); break;
        case 1: le = launch_ln_fwd_peel_bf16(plan.plan_id, fused, p, plan.ctas, stream); break;
        case 2: le = launch_ln_fwd_peel_f16(plan.plan_id, fused, p, plan.ctas, stream); break;
        default: le = (int)cudaErrorInvalidValue; break;
        }
    } else {
        switch (kind_of(dt)) {
        case 1: le = launch_ln_fwd_bf16(plan.plan_id, fused, p, plan.ctas, stream); break;
        case 2: le = launch_ln_fwd_f16(plan.plan_id, fused, p, plan.ctas, stream); break;
        case 3: le = launch_ln_fwd_bf16w32(plan.plan_id, fused, p, plan.ctas, stream); break;
        case 4: le = launch_ln_fwd_f16w32(plan.plan_id, fused, p, plan.ctas, stream); break;
        default: le = launch_ln_fwd_f32(plan.plan_id, fused, p, plan.ctas, stream); break;
        }
    }
    if (le != 0) return cuda_fail((cudaError_t)le);
    if (used) *used = plan;
    return RMSNORM_SUCCESS;
}

static rmsnorm_status_t ln_bwd_impl(const void *dy, const void *dres, const void *x, const void *gamma,
                                    const float *mean, const float *rstd, void *dx, void *dgamma, void *dbeta,
                                    void *workspace, size_t ws_bytes, int64_t M, int64_t N, int dt, float eps,
                                    float offset, cudaStream_t stream, int force_plan, int force_ctas,
                                    rmsnorm_plan_t *used) {
    if (!table_ok()) return RMSNORM_ERR_UNSUPPORTED;
    if (!valid_dtype(dt)) return RMSNORM_ERR_INVALID_ARG;
    if (N < 1 || N > RMSNORM_MAX_N || M < 0 || M > 0x7fffffffLL) return RMSNORM_ERR_INVALID_ARG;
    if (!finite_scalar(eps) || !finite_scalar(offset) || eps < 0.f) return RMSNORM_ERR_INVALID_ARG;
    const uintptr_t s = (uintptr_t)elem_size(dt);
    const uintptr_t wsz = (uintptr_t)weight_size(dt);  // gamma, dgamma, dbeta: the activations' type or fp32
    // dgamma needs gamma; without gamma the weight factor is 1 and there is no dgamma
    if (dgamma && !gamma) return RMSNORM_ERR_INVALID_ARG;
    if ((gamma && !aligned_to(gamma, wsz)) || (dgamma && !aligned_to(dgamma, wsz)) || (dbeta && !aligned_to(dbeta, wsz)))
        return RMSNORM_ERR_INVALID_ARG;
    const bool want = dgamma != nullptr || dbeta != nullptr;
    if (M == 0) {  // the parameter gradients are the empty sums
        cudaError_t e = cudaSuccess;
        if (dgamma) e = cudaMemsetAsync(dgamma, 0, (size_t)N * wsz, stream);
        if (e == cudaSuccess && dbeta) e = cudaMemsetAsync(dbeta, 0, (size_t)N * wsz, stream);
        return e == cudaSuccess ? RMSNORM_SUCCESS : cuda_fail(e);
    }
    if (!dy || !x || !mean || !rstd || !dx) return RMSNORM_ERR_INVALID_ARG;
    if (!aligned_to(dy, s) || !aligned_to(x, s) || !aligned_to(dx, s) || !aligned_to(mean, 4) ||
        !aligned_to(rstd, 4) || (dres && !aligned_to(dres, s)))
        return RMSNORM_ERR_INVALID_ARG;
    if (workspace && !aligned_to(workspace, 16)) return RMSNORM_ERR_WORKSPACE;
    const bool fused = dres != nullptr;

    BwdCall call;
    rmsnorm_status_t st = plan_bwd_call(RMSNORM_OP_LN_BWD, dy, dres, x, gamma, dx, M, N, dt, fused, force_plan,
                                        force_ctas, &call);
    if (st != RMSNORM_SUCCESS) return st;
    rmsnorm_plan_t &plan = call.plan;
    cudaError_t e;
    if (plan.path == PATH_GENERIC && force_plan < 0) note_generic(NOTE_LN_BWD, N, dt);

    float *ws = static_cast<float *>(workspace);
    bool owned = false;
    if (!want) {
        ws = nullptr;  // no parameter gradients: no partial rows, no finalizer
    } else if (ws) {
        if (ws_bytes < (size_t)plan.workspace_bytes) return RMSNORM_ERR_WORKSPACE;
    } else {
        void *tmp = nullptr;
        e = cudaMallocAsync(&tmp, (size_t)plan.workspace_bytes, stream);
        if (e != cudaSuccess) return cuda_fail(e);
        ws = static_cast<float *>(tmp);
        owned = true;
    }
    int *status = nullptr;
    e = status_word(call.dev, &status);
    if (e != cudaSuccess) {
        if (owned) cudaFreeAsync(ws, stream);
        return cuda_fail(e);
    }

    // rows at a common offset: pointers moved back to the 16-byte boundary
    // (the partial rows come out rotated by pl columns)
    const int pl = plan.peel;
    const int es = (int)s;
    BwdParams p;
    std::memset(&p, 0, sizeof p);
    p.status = status;
    p.dy = to_chunk_base(dy, pl, es);
    p.x = to_chunk_base(x, pl, es);
    p.w = to_chunk_base(gamma, pl, es);
    p.rstd = rstd;
    p.mean = mean;
    p.dres = to_chunk_base(dres, pl, es);
    p.dx = to_chunk_base(dx, pl, es);
    p.ws = ws;
    p.M = M;
    p.N = (int)N;
    p.offset = offset;
    p.peel = pl;
    const PlanDesc *pd = call.d;
    p.stages = staged_path(pd->path) ? staged_depth(*pd, N * es / 16, pl, fused) : 0;
    p.cache_row = generic_bwd_cache(pd->path, N, (int)s, ws != nullptr, call.cps);
    if (p.cache_row) plan.smem_bytes = (int32_t)(2 * generic_bwd_cache_slot(N, (int)s));
    int le;
    if (pl > 0) {
        switch (kind_of(dt)) {
        case 0: le = launch_ln_bwd_peel_f32(plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream); break;
        case 1: le = launch_ln_bwd_peel_bf16(plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream); break;
        case 2: le = launch_ln_bwd_peel_f16(plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream); break;
        default: le = (int)cudaErrorInvalidValue; break;
        }
    } else {
        switch (kind_of(dt)) {
        case 1: le = launch_ln_bwd_bf16(plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream); break;
        case 2: le = launch_ln_bwd_f16(plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream); break;
        case 3: le = launch_ln_bwd_bf16w32(plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream); break;
        case 4: le = launch_ln_bwd_f16w32(plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream); break;
        default: le = launch_ln_bwd_f32(plan.plan_id, fused, p, plan.ctas, plan.smem_bytes, stream); break;
        }
    }
    // one finalizer over the [units, 2N] partial rows: dgamma | dbeta (a
    // NULL output's half is not written)
    if (le == 0 && want)
        le = launch_finalize_dt(dt, ws, plan.ws_rows, (int)(2 * N), dgamma, dbeta, (int)N, pl, stream, false,
                                call.sms);
    if (owned) {
        cudaError_t fe = cudaFreeAsync(ws, stream);
        if (le == 0 && fe != cudaSuccess) le = (int)fe;
    }
    if (le != 0) return cuda_fail((cudaError_t)le);
    plan.packed = plan.path == PATH_VECTOR ? 1 : 0;
    if (used) *used = plan;
    return RMSNORM_SUCCESS;
}

}  // namespace rmsn

using namespace rmsn;

extern "C" {

rmsnorm_status_t rmsnorm_fwd(const void *x, const void *w, void *y, float *rstd, int64_t M, int64_t N,
                             rmsnorm_dtype_t dt, float eps, float offset, rmsnorm_stream_t stream) {
    return fwd_impl(x, nullptr, w, y, nullptr, rstd, M, N, dt, eps, offset, (cudaStream_t)stream, -1, nullptr);
}

rmsnorm_status_t rmsnorm_add_fwd(const void *x, const void *residual, const void *w, void *y,
                                 void *residual_out, float *rstd, int64_t M, int64_t N, rmsnorm_dtype_t dt,
                                 float eps, float offset, rmsnorm_stream_t stream) {
    if (!residual || !residual_out) return RMSNORM_ERR_INVALID_ARG;
    return fwd_impl(x, residual, w, y, residual_out, rstd, M, N, dt, eps, offset, (cudaStream_t)stream, -1,
                    nullptr);
}

rmsnorm_status_t rmsnorm_fwd_fp8(const void *x, const void *residual, const void *w, void *y, void *residual_out,
                                 float *rstd, rmsnorm_fp8_scaling_t scaling, const float *scale, float *scale_inv,
                                 float *amax, int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                                 rmsnorm_stream_t stream) {
    int mode;
    if (scaling == RMSNORM_FP8_TENSOR) mode = QOUT_FP8_TENSOR;
    else if (scaling == RMSNORM_FP8_ROW) mode = QOUT_FP8_ROW;
    else return RMSNORM_ERR_INVALID_ARG;
    return fwd_impl(x, residual, w, y, residual_out, rstd, M, N, dt, eps, offset, (cudaStream_t)stream, -1,
                    nullptr, QuantOut{mode, scale, scale_inv, amax});
}

rmsnorm_status_t rmsnorm_fwd_fp8_ex(const void *x, const void *residual, const void *w, void *y,
                                    void *residual_out, float *rstd, rmsnorm_fp8_scaling_t scaling,
                                    const float *scale, float *scale_inv, float *amax, int64_t M, int64_t N,
                                    rmsnorm_dtype_t dt, float eps, float offset, rmsnorm_stream_t stream,
                                    int force_plan, rmsnorm_plan_t *plan_used) {
    int mode;
    if (scaling == RMSNORM_FP8_TENSOR) mode = QOUT_FP8_TENSOR;
    else if (scaling == RMSNORM_FP8_ROW) mode = QOUT_FP8_ROW;
    else return RMSNORM_ERR_INVALID_ARG;
    return fwd_impl(x, residual, w, y, residual_out, rstd, M, N, dt, eps, offset, (cudaStream_t)stream,
                    force_plan, plan_used, QuantOut{mode, scale, scale_inv, amax});
}

rmsnorm_status_t rmsnorm_fwd_ex(const void *x, const void *residual, const void *w, void *y,
                                void *residual_out, float *rstd, int64_t M, int64_t N, rmsnorm_dtype_t dt,
                                float eps, float offset, rmsnorm_stream_t stream, int force_plan,
                                rmsnorm_plan_t *plan_used) {
    return fwd_impl(x, residual, w, y, residual_out, rstd, M, N, dt, eps, offset, (cudaStream_t)stream,
                    force_plan, plan_used);
}

rmsnorm_status_t rmsnorm_bwd(const void *dy, const void *x, const void *w, const float *rstd, void *dx,
                             void *dw, void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
                             rmsnorm_dtype_t dt, float eps, float offset, rmsnorm_stream_t stream) {
    return bwd_impl(dy, nullptr, x, w, rstd, dx, dw, workspace, workspace_bytes, M, N, dt, eps, offset,
                    (cudaStream_t)stream, false, -1, 0, -1, nullptr, nullptr);
}

rmsnorm_status_t rmsnorm_add_bwd(const void *dy, const void *dresidual_out, const void *h, const void *w,
                                 const float *rstd, void *dx, void *dw, void *workspace, size_t workspace_bytes,
                                 int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                                 rmsnorm_stream_t stream) {
    return bwd_impl(dy, dresidual_out, h, w, rstd, dx, dw, workspace, workspace_bytes, M, N, dt, eps, offset,
                    (cudaStream_t)stream, true, -1, 0, -1, nullptr, nullptr);
}

rmsnorm_status_t rmsnorm_bwd_ex(const void *dy, const void *dresidual_out, const void *x, const void *w,
                                const float *rstd, void *dx, void *dw, void *workspace, size_t workspace_bytes,
                                int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                                rmsnorm_stream_t stream, int fused, int force_plan, int force_ctas,
                                int force_packed, void *event_after_main, rmsnorm_plan_t *plan_used) {
    return bwd_impl(dy, dresidual_out, x, w, rstd, dx, dw, workspace, workspace_bytes, M, N, dt, eps, offset,
                    (cudaStream_t)stream, fused != 0, force_plan, force_ctas, force_packed, event_after_main,
                    plan_used);
}

size_t rmsnorm_bwd_workspace_bytes(int64_t M, int64_t N, rmsnorm_dtype_t dt) {
    return bwd_workspace_bytes(RMSNORM_OP_BWD, M, N, dt);
}

size_t rmsnorm_bwd_call_workspace_bytes(const void *dy, const void *dresidual_out, const void *x, const void *w,
                                        const void *dx, int64_t M, int64_t N, rmsnorm_dtype_t dt, int fused) {
    return call_workspace_bytes(dy, dresidual_out, x, w, dx, M, N, dt, fused != 0);
}

rmsnorm_status_t layernorm_fwd(const void *x, const void *residual, const void *gamma, const void *beta, void *y,
                               void *residual_out, float *mean, float *rstd, int64_t M, int64_t N,
                               rmsnorm_dtype_t dt, float eps, float offset, rmsnorm_stream_t stream) {
    return ln_fwd_impl(x, residual, gamma, beta, y, residual_out, mean, rstd, M, N, dt, eps, offset,
                       (cudaStream_t)stream, -1, nullptr);
}

rmsnorm_status_t layernorm_fwd_ex(const void *x, const void *residual, const void *gamma, const void *beta,
                                  void *y, void *residual_out, float *mean, float *rstd, int64_t M, int64_t N,
                                  rmsnorm_dtype_t dt, float eps, float offset, rmsnorm_stream_t stream,
                                  int force_plan, rmsnorm_plan_t *plan_used) {
    return ln_fwd_impl(x, residual, gamma, beta, y, residual_out, mean, rstd, M, N, dt, eps, offset,
                       (cudaStream_t)stream, force_plan, plan_used);
}

rmsnorm_status_t layernorm_bwd(const void *dy, const void *dresidual_out, const void *x, const void *gamma,
                               const float *mean, const float *rstd, void *dx, void *dgamma, void *dbeta,
                               void *workspace, size_t workspace_bytes, int64_t M, int64_t N, rmsnorm_dtype_t dt,
                               float eps, float offset, rmsnorm_stream_t stream) {
    return ln_bwd_impl(dy, dresidual_out, x, gamma, mean, rstd, dx, dgamma, dbeta, workspace, workspace_bytes, M,
                       N, dt, eps, offset, (cudaStream_t)stream, -1, 0, nullptr);
}

rmsnorm_status_t layernorm_bwd_ex(const void *dy, const void *dresidual_out, const void *x, const void *gamma,
                                  const float *mean, const float *rstd, void *dx, void *dgamma, void *dbeta,
                                  void *workspace, size_t workspace_bytes, int64_t M, int64_t N,
                                  rmsnorm_dtype_t dt, float eps, float offset, rmsnorm_stream_t stream,
                                  int force_plan, int force_ctas, rmsnorm_plan_t *plan_used) {
    return ln_bwd_impl(dy, dresidual_out, x, gamma, mean, rstd, dx, dgamma, dbeta, workspace, workspace_bytes, M,
                       N, dt, eps, offset, (cudaStream_t)stream, force_plan, force_ctas, plan_used);
}

size_t layernorm_bwd_workspace_bytes(int64_t M, int64_t N, rmsnorm_dtype_t dt) {
    return bwd_workspace_bytes(RMSNORM_OP_LN_BWD, M, N, dt);
}

rmsnorm_status_t rmsnorm_plan_query(int op, int64_t M, int64_t N, rmsnorm_dtype_t dt, int aligned, int num_sms,
                                    int ctas_per_sm, int force_plan, int force_ctas, rmsnorm_plan_t *out) {
    if (!table_ok()) return RMSNORM_ERR_UNSUPPORTED;
    if (num_sms < 1 || aligned < 0) return RMSNORM_ERR_INVALID_ARG;
    // aligned: 0 generic, 1 aligned rows, 1 + k rows at a common offset of k elements
    const int layout = aligned == 0 ? -1 : aligned - 1;
    // Without a device the resident-CTA count is the caller's (or the plan's
    // nominal 2048 threads per SM); a cluster plan packs cluster-size CTAs.
    int cps = ctas_per_sm;
    int cs = 1;
    if (force_plan >= 0) {
        const PlanDesc *fd = find_plan(force_plan);
        if (fd) {
            if (cps <= 0) cps = nominal_ctas_per_sm(*fd);
            cs = fd->cs;
        }
    } else {
        rmsnorm_plan_t probe;
        rmsnorm_status_t st = select_plan(op, M, N, dt, layout, 1, 0, -1, 0, &probe);
        if (st != RMSNORM_SUCCESS) return st;
        const PlanDesc *pd = find_plan(probe.plan_id);
        if (cps <= 0) cps = nominal_ctas_per_sm(*pd);
        cs = pd->cs;
    }
    if (cps <= 0) cps = 1;
    int64_t parts = (int64_t)cps * num_sms / cs;
    if (parts < 1) parts = 1;
    return select_plan(op, M, N, dt, layout, parts, cps, force_plan, force_ctas, out);
}

int rmsnorm_plan_count(void) { return kNumPlans; }

int rmsnorm_plan_id_at(int index) { return (index >= 0 && index < kNumPlans) ? kPlans[index].id : -1; }

const char *rmsnorm_status_string(rmsnorm_status_t status) {
    switch (status) {
    case RMSNORM_SUCCESS: return "success";
    case RMSNORM_ERR_INVALID_ARG: return "invalid argument";
    case RMSNORM_ERR_UNSUPPORTED: return "unsupported plan or configuration";
    case RMSNORM_ERR_WORKSPACE: return "workspace too small or misaligned";
    case RMSNORM_ERR_CUDA: return "CUDA error (see rmsnorm_last_cuda_error)";
    default: return "unknown status";
    }
}

int rmsnorm_last_cuda_error(void) { return g_last_cuda_error; }

int rmsnorm_self_check(void) { return self_check_impl(); }

void rmsnorm_set_generic_note(int enabled) {
    g_noted.store(0, std::memory_order_relaxed);
    g_note_on.store(enabled ? 1 : 0, std::memory_order_relaxed);
}

int rmsnorm_device_status(int clear) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    int *w = nullptr;
    if (status_word(dev, &w) != cudaSuccess) return -1;
    int v = 0;
    if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
    if (clear && v != 0) {
        const int zero = 0;
        if (cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return -1;
    }
    return v;
}

}  // extern "C"
