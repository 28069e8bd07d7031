/*
 * rmsnorm.h -- C ABI of librmsnorm_gb300.so: RMSNorm forward and backward
 * over a row-major [M, N] activation matrix on one GB300 GPU (sm_103a).
 *
 * Operation (llama mode: every step in fp32, each output rounded once, to
 * nearest-even, when it is stored):
 *
 *   forward   rstd_i = 1 / sqrt( (1/N) sum_j h_ij^2 + eps )
 *             y_ij   = h_ij * rstd_i * (offset + w_j)
 *             with h = x (plain) or h = R(x + residual) (fused residual add)
 *   backward  xhat = h * rstd,  g = dy * (offset + w),
 *             c_i  = (1/N) sum_j g_ij xhat_ij
 *             dx   = rstd * (g - xhat * c)  [+ dresidual_out, fused variant]
 *             dw_j = sum_i dy_ij xhat_ij
 *
 * Sources: Liger-Kernel PR #1388 "perf(cutedsl): add Blackwell fast path to
 * RMSNorm" (Summary; section 1 for eps/offset as runtime fp32 scalars and a
 * launch path without per-call marshalling; section 2 for the fused
 * backward that produces dX and dW) and ROCm/FlyDSL PR #855 "[Perf]
 * Optimize RMSNorm backward with staged reduction and vec8 I/O"
 * (Implementation: a persistent main kernel writing one fp32 dweight
 * partial per program, a finalizer that reduces the [num_programs, N]
 * workspace and writes dweight in the parameter dtype, the fused-add
 * specialisation with dx == dresidual; Runtime configuration and
 * ownership: per-call workspace of num_programs * N * 4 bytes, launch on
 * the caller's stream).
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers on the calling thread's current
 *     CUDA device. The caller owns every buffer; the library keeps no
 *     pointer after the call returns.
 *   - Matrices are contiguous row-major [M, N] (row stride N elements).
 *     w, dw are [N]; rstd is [M] fp32.
 *   - x, residual, y, dy, dx, residual_out, dresidual_out share the
 *     activations' storage type `dt`; w and dw have the same type, or fp32
 *     when `dt` carries RMSNORM_WEIGHT_F32. Pointers must be aligned to
 *     their element size. With N * sizeof(activation) % 16 == 0, the
 *     vectorised kernels serve every call whose pointers are all 16-byte
 *     aligned, and also every call whose row arrays (and the weight, in the
 *     activations' type) all sit at one common offset past a 16-byte
 *     boundary (e.g. each one element past an aligned allocation): a row's
 *     head and tail, which share 16-byte blocks with the neighbouring rows,
 *     are read as whole aligned blocks (never past the 16 bytes that hold
 *     one of the row's elements), joined into one chunk, and written back
 *     element by element; no element outside the arrays is ever written.
 *     Anything else takes the generic kernels. The generic backward for
 *     rows of up to 8192 elements likewise reads each row of x, dy (and
 *     dresidual_out) as the whole 16-byte blocks that hold its elements,
 *     wherever each array starts, and writes dx element by element. With
 *     an fp32 weight only the default plans are compiled (forcing an
 *     alternative plan id returns UNSUPPORTED) and only aligned rows are
 *     vectorised. Rows at a common offset run kernels of their own
 *     (compiled for the default plans only, so that aligned rows pay
 *     nothing for the wrapped chunk): forcing an alternative plan id on
 *     them returns UNSUPPORTED as well.
 *   - Every call is asynchronous on `stream` (NULL = legacy default
 *     stream). The library never synchronises and never copies between
 *     host and device.
 *   - eps >= 0 and offset are runtime values; they never change the kernel
 *     chosen. M is runtime; the kernel depends on (dt, N, alignment) and the
 *     backward's CTA count on M and the device's SM count.
 *   - Errors are returned as status codes; nothing aborts or throws.
 *     M == 0 is a successful call that launches no kernel (the backward
 *     then sets dw to zero, the empty sum, with one cudaMemsetAsync).
 *     INVALID_ARG: N < 1, N > RMSNORM_MAX_N, M < 0, M > 2^31 - 1, a
 *     required pointer NULL or not element-aligned, eps < 0, eps or offset
 *     not finite, an unknown dtype. WORKSPACE: a non-NULL workspace smaller
 *     than rmsnorm_bwd_workspace_bytes() or not 16-byte aligned.
 *     CUDA: a CUDA call failed; rmsnorm_last_cuda_error() returns its code.
 *   - Aliasing: y may equal x; dx may equal dy; in the fused variants
 *     residual_out may equal residual and dx may equal dresidual_out. No
 *     other pair of buffers may overlap.
 */
#ifndef RMSNORM_GB300_H
#define RMSNORM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *rmsnorm_stream_t; /* same type as cudaStream_t */

typedef enum {
    RMSNORM_F32 = 0,  /* IEEE binary32 storage */
    RMSNORM_BF16 = 1, /* bfloat16 storage, fp32 compute */
    RMSNORM_F16 = 2,  /* IEEE binary16 storage, fp32 compute */
    /* Flag OR'ed into the activations' type: w and dw are stored in fp32
     * (an fp32 master weight beside 16-bit activations). fp32 | flag is the
     * same as fp32. */
    RMSNORM_WEIGHT_F32 = 0x100,
    RMSNORM_BF16_W32 = 0x101, /* bf16 activations, fp32 w and dw */
    RMSNORM_F16_W32 = 0x102,  /* fp16 activations, fp32 w and dw */
    /* Forward only (rmsnorm_fwd, rmsnorm_add_fwd, rmsnorm_fwd_ex): OR'ed
     * into RMSNORM_F32, y is stored in bf16 or fp16 (the key's otype apart
     * from its itype), rounded once from the fp32 result; residual_out
     * stays fp32. Vectorised where x, y (and the residual buffers) are
     * 16-byte aligned and N % 4 == 0, generic otherwise. Other entry
     * points return INVALID_ARG for these flags. */
    RMSNORM_OUT_BF16 = 0x200,
    RMSNORM_OUT_F16 = 0x400
} rmsnorm_dtype_t;

typedef enum {
    RMSNORM_SUCCESS = 0,
    RMSNORM_ERR_INVALID_ARG = 1,
    RMSNORM_ERR_UNSUPPORTED = 2,
    RMSNORM_ERR_WORKSPACE = 3,
    RMSNORM_ERR_CUDA = 4
} rmsnorm_status_t;

#define RMSNORM_MAX_N 65536

/*
 * Forward. Reads x [M,N] and w [N]; writes y [M,N] and rstd [M] (fp32).
 * Liger-Kernel PR #1388, Summary and section 1 (vector forward with a
 * CTA-level reduction; eps and offset runtime scalars).
 * w == NULL: non-affine RMSNorm, y = x * rstd (the weight factor is 1 and
 * offset is unused; Liger-Kernel PR #1388, Validation: affine and
 * non-affine launches).
 */
rmsnorm_status_t rmsnorm_fwd(const void *x, const void *w, void *y, float *rstd,
                             int64_t M, int64_t N, rmsnorm_dtype_t dt,
                             float eps, float offset, rmsnorm_stream_t stream);

/*
 * Backward. Reads dy, x [M,N], w [N] and the forward's rstd [M]; writes
 * dx [M,N] and dw [N]. rstd is read, not recomputed, so eps is only
 * validated (kept for symmetry with the forward). Two kernels run on
 * `stream`: a persistent main kernel that writes dx and one fp32 dw
 * partial row per CTA into the workspace, then a finalizer that sums the
 * partial rows in a fixed order and writes dw in the storage type
 * (FlyDSL PR #855, Implementation).
 * workspace: NULL, or device memory of at least
 * rmsnorm_bwd_workspace_bytes(M, N, dt) bytes, 16-byte aligned, not used
 * by any other call in flight. Its contents on entry do not matter (every
 * byte read is first written by this call). With NULL the library takes
 * stream-ordered memory (cudaMallocAsync/cudaFreeAsync on `stream`).
 * w == NULL: non-affine backward (g = dy); dw must then be NULL too (there
 * is no weight gradient), no workspace is used and only the main kernel runs.
 */
rmsnorm_status_t rmsnorm_bwd(const void *dy, const void *x, const void *w, const float *rstd,
                             void *dx, void *dw, void *workspace, size_t workspace_bytes,
                             int64_t M, int64_t N, rmsnorm_dtype_t dt,
                             float eps, float offset, rmsnorm_stream_t stream);

/*
 * Fused residual add + forward. h = R(x + residual) is rounded to the
 * storage type, written to residual_out [M,N] and normalised into y
 * (FlyDSL PR #855, Implementation: fused-add RMSNorm as a specialisation
 * of the same kernels). residual_out may equal residual. w may be NULL
 * (non-affine), as in rmsnorm_fwd.
 */
rmsnorm_status_t rmsnorm_add_fwd(const void *x, const void *residual, const void *w,
                                 void *y, void *residual_out, float *rstd,
                                 int64_t M, int64_t N, rmsnorm_dtype_t dt,
                                 float eps, float offset, rmsnorm_stream_t stream);

/*
 * Fused residual add backward. h is the forward's residual_out. dx [M,N]
 * receives rstd * (g - xhat * c) + dresidual_out, the gradient of both x
 * and residual (one buffer serves as dx and dresidual, FlyDSL PR #855,
 * Implementation). dresidual_out may be NULL (treated as zero) or equal dx.
 * Workspace and non-affine (w, dw NULL) rules as in rmsnorm_bwd.
 */
rmsnorm_status_t rmsnorm_add_bwd(const void *dy, const void *dresidual_out, const void *h,
                                 const void *w, const float *rstd, void *dx, void *dw,
                                 void *workspace, size_t workspace_bytes,
                                 int64_t M, int64_t N, rmsnorm_dtype_t dt,
                                 float eps, float offset, rmsnorm_stream_t stream);

/* Scaling of the E4M3 output of rmsnorm_fwd_fp8. */
typedef enum {
    RMSNORM_FP8_TENSOR = 0, /* one given scale for the whole tensor */
    RMSNORM_FP8_ROW = 1     /* each row scaled by 448 / max_j |y_ij| */
} rmsnorm_fp8_scaling_t;

/*
 * Forward with an fp8 E4M3 output, the quantised output of a norm that
 * feeds an fp8 GEMM (the TransformerEngine tuning page, "[ROCm] RMSNorm
 * tuning", Description and review: the norm kernel key's output type
 * kFloat8E4M3, beside the input, weight and compute types).
 * y [M,N] holds one E4M3 byte per element: y_ij = E4M3(y'_ij * s), where y'
 * is the fp32 forward value (as rmsnorm_fwd computes it, not rounded to the
 * input type), the product is rounded to fp32, and E4M3() rounds to
 * nearest-even, saturating to +-448. rstd [M] as in rmsnorm_fwd.
 *   RMSNORM_FP8_TENSOR: s = *scale (a device pointer to one fp32, required);
 *     scale_inv (optional, one fp32) receives 1/s.
 *   RMSNORM_FP8_ROW: scale must be NULL; a_i = max_j |y'_ij| (fp32),
 *     s_i = 448 / a_i (1 when a_i == 0); scale_inv [M] (required) receives
 *     a_i / 448 (1 when a_i == 0), so y'_ij ~ decode(y_ij) * scale_inv_i.
 *   amax (optional, one fp32, either scaling) receives max_ij |y'_ij| over
 *     this call (set to 0 first, then combined with an atomic maximum; 0
 *     when M == 0).
 * residual / residual_out: both NULL (plain) or both set (fused add, as in
 * rmsnorm_add_fwd). w may be NULL (non-affine). dt is fp32, bf16 or fp16
 * with the weight in the same type, or RMSNORM_BF16_W32 / RMSNORM_F16_W32
 * (an fp32 weight beside 16-bit activations: the key's wtype apart from its
 * itype). y needs no alignment beyond 1 byte; 16-byte alignment of x, w, y
 * (and the residual buffers) with N * sizeof(elem) % 16 == 0 selects the
 * vectorised kernels. With M == 0 nothing but amax is written. All
 * pointers are device pointers; argument errors as for rmsnorm_fwd.
 */
rmsnorm_status_t rmsnorm_fwd_fp8(const void *x, const void *residual, const void *w, void *y,
                                 void *residual_out, float *rstd, rmsnorm_fp8_scaling_t scaling,
                                 const float *scale, float *scale_inv, float *amax,
                                 int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                                 rmsnorm_stream_t stream);

/*
 * LayerNorm, the sibling norm the TransformerEngine tuning page registers
 * tuned kernels for beside RMSNorm ("[ROCm] RMSNorm tuning", Description:
 * matching tuned configs for LayerNorm), on the same kernels' geometry:
 *
 *   forward   mean_i = (1/N) sum_j h_ij
 *             rstd_i = 1 / sqrt( (1/N) sum_j (h_ij - mean_i)^2 + eps )
 *             y_ij   = (h_ij - mean_i) * rstd_i * (offset + gamma_j) + beta_j
 *   backward  xhat = (h - mean) * rstd,  g = dy * (offset + gamma),
 *             dx   = rstd * (g - mean_j(g) - xhat * mean_j(g xhat)) [+ dresidual_out]
 *             dgamma_j = sum_i dy_ij xhat_ij,  dbeta_j = sum_i dy_ij
 *
 * Every step in fp32, each output rounded once (as for RMSNorm); the
 * variance is the biased one, computed from the row held in registers in
 * two passes (sum, then squared deviations from the mean).
 * gamma == NULL: factor 1 (offset unused); beta == NULL: no bias.
 * gamma, beta, dgamma, dbeta have the activations' storage type, or fp32
 * beside bf16 / fp16 activations (RMSNORM_BF16_W32, RMSNORM_F16_W32; then
 * only rows on 16-byte boundaries are vectorised and a forced alternative
 * plan returns UNSUPPORTED, as for RMSNorm). mean and rstd [M] are fp32.
 * residual / residual_out: both NULL, or both set for the fused add
 * (h = R(x + residual), stored to residual_out, as in rmsnorm_add_fwd).
 * Pointers, alignment, errors and aliasing as for the RMSNorm calls.
 */
rmsnorm_status_t layernorm_fwd(const void *x, const void *residual, const void *gamma, const void *beta,
                               void *y, void *residual_out, float *mean, float *rstd,
                               int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                               rmsnorm_stream_t stream);

/*
 * LayerNorm backward. Reads dy, x (h of the fused forward) [M,N], gamma
 * [N] and the forward's mean and rstd; writes dx [M,N] (plus
 * dresidual_out when that is non-NULL: the fused add's gradient of both x
 * and residual) and, when non-NULL, dgamma [N] and dbeta [N]. dgamma
 * requires gamma. Persistent main kernel with fp32 partial rows
 * [units, 2N] (dgamma | dbeta) in the workspace, then one finalizer that
 * sums them in a fixed order (as rmsnorm_bwd). workspace: NULL (stream-
 * ordered allocation) or at least layernorm_bwd_workspace_bytes(M, N, dt)
 * bytes, 16-byte aligned. With dgamma and dbeta both NULL no workspace is
 * used and only the main kernel runs. M == 0 sets dgamma and dbeta to 0.
 */
rmsnorm_status_t layernorm_bwd(const void *dy, const void *dresidual_out, const void *x,
                               const void *gamma, const float *mean, const float *rstd,
                               void *dx, void *dgamma, void *dbeta,
                               void *workspace, size_t workspace_bytes,
                               int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                               rmsnorm_stream_t stream);

/* Workspace bytes layernorm_bwd needs for (M, N, dt) on the current device
 * (2 * units * N * 4, rounded up to 256; 0 without a device). */
size_t layernorm_bwd_workspace_bytes(int64_t M, int64_t N, rmsnorm_dtype_t dt);

/*
 * Backward without any allocation, for callers that cannot allocate device
 * memory when they call (an engine that reserves all device memory at
 * start-up and forbids later allocation, a plug-in host that passes its ops
 * no workspace). The pages have no counterpart to this entry point.
 * Same arguments and results as rmsnorm_bwd (every storage type, the
 * fp32-weight ones included; w and dw NULL for the non-affine backward),
 * but the dW partial rows live in a fixed array inside the library,
 * RMSNORM_NOALLOC_SCRATCH_BYTES per GPU, held from the time the library's
 * kernels load on that GPU until the process exits. Returns
 * RMSNORM_ERR_WORKSPACE, launching nothing, when the workspace this call
 * needs (at most rmsnorm_bwd_workspace_bytes(M, N, dt)) exceeds that size.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * The address is kept for the life of the process: do not use the library
 * across a cudaDeviceReset.
 * Every call on a device uses the same array and leaves its partial rows
 * there; nothing needs clearing, because each call writes every partial it
 * reads. Calls that can overlap on the GPU (other streams, other threads)
 * race on the array: serialise them.
 */
rmsnorm_status_t rmsnorm_bwd_noalloc(const void *dy, const void *x, const void *w,
                                     const float *rstd, void *dx, void *dw,
                                     int64_t M, int64_t N, rmsnorm_dtype_t dt,
                                     float eps, float offset, rmsnorm_stream_t stream);

#define RMSNORM_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */

/*
 * Bytes of workspace the backward needs for (M, N, dt) on the current
 * device, whatever the call's pointers and fusion: the largest need over
 * the row layouts (aligned, at a common offset, generic) and the plain and
 * fused variants, so one allocation of this size serves every call. A
 * call's own need is (dW partial rows) * (row columns) * 4 rounded up to
 * 256 (FlyDSL PR #855, Runtime configuration and ownership: one fp32
 * partial row per program), where the partial rows are the persistent CTAs
 * (or clusters) and the row columns N; rmsnorm_bwd_call_workspace_bytes
 * gives it exactly.
 * Returns 0 for M == 0 and for invalid arguments or when no CUDA device is
 * usable.
 */
size_t rmsnorm_bwd_workspace_bytes(int64_t M, int64_t N, rmsnorm_dtype_t dt);

/*
 * Exact workspace need of one rmsnorm_bwd call (fused == 0) or
 * rmsnorm_add_bwd call (fused != 0) with these arrays on the current
 * device: the plan that call selects. dresidual_out is used only when
 * fused (may be NULL). Returns 0 for the non-affine backward (w == NULL,
 * no workspace), M == 0, invalid arguments or no usable device.
 */
size_t rmsnorm_bwd_call_workspace_bytes(const void *dy, const void *dresidual_out, const void *x,
                                        const void *w, const void *dx, int64_t M, int64_t N,
                                        rmsnorm_dtype_t dt, int fused);

/* ------------------------------------------------------------------------
 * Plans: which kernel runs. Exposed for tests and benchmarks (the analogue
 * of the A/B toggles of Liger-Kernel PR #1388, "Behavior when the fast path
 * does not apply", and of the tuned-kernel registry of
 * ROCm/TransformerEngine PR #583, Description).
 * --------------------------------------------------------------------- */

typedef enum {
    RMSNORM_PATH_VECTOR = 0,   /* 128-bit loads, row held in registers       */
    RMSNORM_PATH_STAGED = 1,   /* row staged in shared memory by bulk copies */
                               /* (held in registers or re-read, by plan)    */
    RMSNORM_PATH_GENERIC = 2   /* any N and alignment: element head and tail */
                               /* around 16-byte chunks, or (backward, rows  */
                               /* up to 8192 elements) rows streamed into    */
                               /* shared memory as whole 16-byte blocks      */
} rmsnorm_path_t;

typedef struct {
    int32_t path;               /* rmsnorm_path_t                               */
    int32_t plan_id;            /* index into the library's plan table          */
    int32_t threads_per_row;
    int32_t chunks_per_thread;  /* 16-byte chunks a thread holds per row (0:
                                   the generic kernels)                         */
    int32_t rows_per_cta;       /* rows a CTA works on concurrently             */
    int32_t cta_threads;
    int32_t packed;             /* 1: packed f32x2 arithmetic                   */
    int32_t ctas;               /* grid size in CTAs                            */
    int32_t ctas_per_sm;        /* backward: resident CTAs per SM used for `ctas`
                                   (0 where the library queried the device)     */
    int32_t smem_bytes;         /* dynamic shared memory per CTA: a call's plan
                                   counts it as launched (a generic LayerNorm
                                   backward's row cache included); the host-only
                                   query leaves that cache out               */
    int32_t cluster_size;       /* CTAs of a thread-block cluster sharing a row (1: none) */
    int32_t ws_rows;            /* persistent grids (the backward and a staged
                                   forward): units walking the rows, CTAs or
                                   clusters; backward: dW partial rows          */
    int64_t workspace_bytes;    /* backward only                                */
    int32_t peel;               /* rows at a common offset: elements of the
                                   16-byte block holding a row's first element
                                   that precede it (the vectorised kernels join
                                   the row's head and tail into one chunk); 0 for
                                   aligned rows and the generic kernels         */
    int32_t reserved;
} rmsnorm_plan_t;

#define RMSNORM_OP_FWD 0
#define RMSNORM_OP_BWD 1
#define RMSNORM_OP_LN_BWD 2 /* LayerNorm backward (its forward uses RMSNORM_OP_FWD plans) */

/*
 * Host-only plan query: no CUDA call, usable without a GPU. `aligned` gives
 * the row layout: 1 every pointer 16-byte aligned; 1 + k every row array
 * (and the weight) k elements past a 16-byte boundary; 0 anything else
 * (the generic kernels). `num_sms` is the device's SM
 * count and `ctas_per_sm` the resident backward CTAs per SM (<= 0: the
 * plan's nominal value). force_plan < 0 picks the default plan; otherwise
 * the plan with that id (UNSUPPORTED if it cannot serve N/dt/alignment).
 * force_ctas > 0 sets the backward's CTA count (capped by the rows
 * available).
 */
rmsnorm_status_t rmsnorm_plan_query(int op, int64_t M, int64_t N, rmsnorm_dtype_t dt,
                                    int aligned, int num_sms, int ctas_per_sm,
                                    int force_plan, int force_ctas, rmsnorm_plan_t *out);

/* Number of entries in the plan table. */
int rmsnorm_plan_count(void);

/* Plan id of table entry `index` (0 <= index < rmsnorm_plan_count()), or -1. */
int rmsnorm_plan_id_at(int index);

/*
 * rmsnorm_fwd_fp8 with a forced plan (force_plan < 0: default; the E4M3
 * kernels exist for the default plans and the generic one, other ids give
 * UNSUPPORTED). Reports the plan that ran in *plan_used (may be NULL).
 */
rmsnorm_status_t rmsnorm_fwd_fp8_ex(const void *x, const void *residual, const void *w, void *y,
                                    void *residual_out, float *rstd, rmsnorm_fp8_scaling_t scaling,
                                    const float *scale, float *scale_inv, float *amax,
                                    int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                                    rmsnorm_stream_t stream, int force_plan, rmsnorm_plan_t *plan_used);

/*
 * LayerNorm with a forced plan (force_plan < 0: default; the forward takes
 * RMSNORM_OP_FWD plan ids, the default ones and the generic one; the
 * backward RMSNORM_OP_LN_BWD ids) and, for the backward, a forced CTA
 * count (force_ctas > 0). Report the plan that ran in *plan_used.
 */
rmsnorm_status_t layernorm_fwd_ex(const void *x, const void *residual, const void *gamma,
                                  const void *beta, void *y, void *residual_out, float *mean, float *rstd,
                                  int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                                  rmsnorm_stream_t stream, int force_plan, rmsnorm_plan_t *plan_used);
rmsnorm_status_t layernorm_bwd_ex(const void *dy, const void *dresidual_out, const void *x,
                                  const void *gamma, const float *mean, const float *rstd,
                                  void *dx, void *dgamma, void *dbeta,
                                  void *workspace, size_t workspace_bytes,
                                  int64_t M, int64_t N, rmsnorm_dtype_t dt, float eps, float offset,
                                  rmsnorm_stream_t stream, int force_plan, int force_ctas,
                                  rmsnorm_plan_t *plan_used);

/*
 * Forward with a forced plan (force_plan < 0: default). residual and
 * residual_out NULL: plain forward; both non-NULL: fused add. Reports the
 * plan that ran in *plan_used (may be NULL).
 */
rmsnorm_status_t rmsnorm_fwd_ex(const void *x, const void *residual, const void *w,
                                void *y, void *residual_out, float *rstd,
                                int64_t M, int64_t N, rmsnorm_dtype_t dt,
                                float eps, float offset, rmsnorm_stream_t stream,
                                int force_plan, rmsnorm_plan_t *plan_used);

/*
 * Backward with a forced plan and CTA count (negative / zero: default),
 * plain when `fused` is 0 (dresidual_out ignored), fused otherwise.
 * force_packed: -1 default, 0 scalar fp32 arithmetic, 1 packed f32x2; both
 * use the same even/odd accumulator pairing, so they agree bit for bit. The
 * staged plans run packed by default; their scalar variant is compiled for
 * the default plans of fp32 and bf16 (weight in the activations' type) and
 * forcing it elsewhere returns UNSUPPORTED.
 * event_after_main: if non-NULL, a cudaEvent_t recorded on `stream` between
 * the main kernel and the finalizer (for timing the two separately).
 */
rmsnorm_status_t rmsnorm_bwd_ex(const void *dy, const void *dresidual_out, const void *x,
                                const void *w, const float *rstd, void *dx, void *dw,
                                void *workspace, size_t workspace_bytes,
                                int64_t M, int64_t N, rmsnorm_dtype_t dt,
                                float eps, float offset, rmsnorm_stream_t stream,
                                int fused, int force_plan, int force_ctas, int force_packed,
                                void *event_after_main, rmsnorm_plan_t *plan_used);

/*
 * Device status word of the current device, for diagnostics: 0 normally;
 * 1 if a backward kernel gave up one of its bounded waits: a cluster row's
 * wait for a peer's partial sum, or a staged kernel's wait for a row's bulk
 * copy into shared memory (that call's outputs are then incomplete).
 * Synchronises the device; clear != 0 resets the word. Returns -1 if the
 * device cannot be queried.
 */
int rmsnorm_device_status(int clear);

/*
 * Optional one-time note on stderr when a call falls to the generic kernels
 * (rows that are not whole 16-byte chunks, or arrays not 16-byte aligned at
 * one common offset), which run well below the vectorised kernels' speed:
 * the counterpart of the fallback warning printed the first time no tuned
 * kernel serves a config (TransformerEngine tuning page, "[ROCm] RMSNorm
 * tuning", Description). Off by default. enabled != 0 switches it on and
 * re-arms it: the next fallback of each kind of call (RMSNorm forward and
 * backward, LayerNorm forward and backward) prints one line; later ones of
 * that kind print nothing. Calls that force a plan are not reported.
 * Thread-safe; no CUDA call.
 */
void rmsnorm_set_generic_note(int enabled);

/* Static description of a status code. */
const char *rmsnorm_status_string(rmsnorm_status_t status);

/* cudaError_t of the last call on this thread that returned RMSNORM_ERR_CUDA. */
int rmsnorm_last_cuda_error(void);

/*
 * Consistency check of the plan table, run once when the library loads and
 * callable again: every (dtype, N-class) a table entry is registered for
 * must select that entry, and its geometry must cover the class (the
 * analogue of the key round-trip check of ROCm/TransformerEngine PR #583).
 * Returns 0 when consistent, else the number of inconsistent entries.
 */
int rmsnorm_self_check(void);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H */
