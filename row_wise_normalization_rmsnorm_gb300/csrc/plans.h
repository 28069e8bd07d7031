// plans.h -- the specialisation table shared by the host selector and the
// kernel instantiations, and the parameter blocks the kernels receive.
//
// A plan fixes the geometry of one kernel: how many threads share a row
// (a "team"), how many 16-byte chunks of the row each thread holds, and how
// many teams a CTA runs side by side. Plans are keyed by the row length in
// 16-byte chunks, C = N * sizeof(elem) / 16, so one table serves bf16 and
// fp32 (a bf16 row of 8192 and an fp32 row of 4096 are both 1024 chunks).
// The geometry depends only on (dtype, N, alignment), never on M: a row's
// in-CTA reduction order, and with it y, rstd and dx, is the same whatever
// the batch size (ROCm/FlyDSL PR #855, "Runtime configuration and
// ownership": M is a runtime argument of one compiled kernel).
#pragma once

#include <stdint.h>

namespace rmsn {

// OP_FWD plans serve the RMSNorm and the LayerNorm forward; OP_LN_BWD
// plans the LayerNorm backward, whose rows carry two sums and two parameter
// gradients (more registers per chunk than the RMSNorm backward).
// OP_FWD_STAGED plans are forward plans that stream rows through shared
// memory; where one covers a row it is preferred to the OP_FWD plan.
enum PlanOp { OP_FWD = 0, OP_BWD = 1, OP_LN_BWD = 2, OP_FWD_STAGED = 3 };
// PATH_STAGED and PATH_RESTAGED stream rows into shared memory; the first
// copies a row's chunks into registers for both passes, the second reads
// them from the stage in each pass (fewer registers, the stage stays busy
// for the whole row). The C ABI reports both as the staged path.
// PATH_STREAM is a generic (any N, any alignment) backward that streams each
// row's 16-byte covers into shared memory; the C ABI reports it as the
// generic path.
enum PlanPath { PATH_VECTOR = 0, PATH_STAGED = 1, PATH_GENERIC = 2, PATH_RESTAGED = 3, PATH_STREAM = 4 };
constexpr bool generic_path(int path) { return path == PATH_GENERIC || path == PATH_STREAM; }
constexpr bool staged_path(int path) { return path == PATH_STAGED || path == PATH_RESTAGED; }
// The staged kernels run one row team a CTA; a row may be shared by a
// cluster of CTAs only on the re-read schedule.
constexpr bool staged_plan(int path, int teams, int cs) {
    return teams == 1 && ((path == PATH_STAGED && cs == 1) || (path == PATH_RESTAGED && (cs == 1 || cs == 2 || cs == 4 || cs == 8)));
}
// The staged backward is compiled with packed f32x2 arithmetic and, for the
// default plans of fp32 and bf16 (weight in the activations' type: kernel
// kinds 0 and 1), also with per-lane fp32 arithmetic in the same pairing,
// for A/B measurements of the packed math; the two agree bit for bit.
constexpr bool staged_scalar_variant(int kind, int cmin) { return (kind == 0 || kind == 1) && cmin > 0; }

// Storage types a default plan applies to (bit 0: fp32, bit 1: bf16,
// bit 2: fp16; DT_16 = both 2-byte types).
enum PlanDtypes { DT_F32 = 1, DT_BF16 = 2, DT_F16 = 4, DT_16 = 6, DT_ANY = 7 };

// X(id, op, path, threads_per_row, chunks_per_thread, teams_per_cta, depth, cluster, dtypes, cmin, cmax)
// [cmin, cmax] is the range of C for which the plan is the default for the
// storage types in `dtypes`; 0, 0 marks an alternative that runs only when
// forced (tuning and A/B tests).
// depth (backward only): rows whose x/dy loads are in flight while the
// current row is computed (a register ring of depth + 1 rows); for staged
// plans the most shared-memory stages rows are streamed into (a call takes
// as many of them as fit its rows, at least two).
// cluster: CTAs of a thread-block cluster that share one row; each holds
// threads_per_row * chunks_per_thread chunks of it in registers and the row
// sums meet in distributed shared memory (1: no cluster).
// Generic plans are chosen by the row layout, not by C: PATH_GENERIC uses
// a 256-thread CTA per row; a PATH_STREAM plan (backward) persistent CTAs
// that each stream `depth` rows ahead, for rows of cmin .. cmax elements
// (there chunks_per_thread counts the elements a thread owns, and
// threads_per_row * chunks_per_thread >= cmax); past the last PATH_STREAM
// range, PATH_GENERIC.
#define RMSNORM_PLAN_TABLE(X) \
    /* forward, row in registers */ \
    X( 0, OP_FWD, PATH_VECTOR ,    8, 1, 32, 0, 1, DT_ANY,     1,     8) \
    X( 1, OP_FWD, PATH_VECTOR ,   16, 1, 16, 0, 1, DT_ANY,     9,    16) \
    X( 2, OP_FWD, PATH_VECTOR ,   32, 1,  8, 0, 1, DT_ANY,    17,    32) \
    X( 3, OP_FWD, PATH_VECTOR ,   32, 2,  8, 0, 1, DT_ANY,    33,    64) \
    X( 4, OP_FWD, PATH_VECTOR ,   32, 4,  8, 0, 1, DT_ANY,    65,   128) \
    X( 5, OP_FWD, PATH_VECTOR ,   64, 4,  4, 0, 1, DT_ANY,   129,   256) \
    X( 6, OP_FWD, PATH_VECTOR ,  128, 4,  2, 0, 1, DT_ANY,   257,   512) \
    X( 7, OP_FWD, PATH_VECTOR ,  256, 4,  1, 0, 1, DT_ANY,   513,  1024) \
    X( 8, OP_FWD, PATH_VECTOR ,  512, 4,  1, 0, 1, DT_ANY,  1025,  2048) \
    X(17, OP_FWD, PATH_VECTOR ,  512, 4,  1, 0, 2, DT_ANY,  2049,  4096) \
    X(18, OP_FWD, PATH_VECTOR ,  512, 4,  1, 0, 4, DT_ANY,  4097,  8192) \
    X(19, OP_FWD, PATH_VECTOR ,  512, 4,  1, 0, 8, DT_ANY,  8193, 16384) \
    X( 9, OP_FWD, PATH_VECTOR , 1024, 4,  1, 0, 1, DT_ANY,     0,     0) \
    X(10, OP_FWD, PATH_VECTOR ,  128, 8,  2, 0, 1, DT_ANY,     0,     0) \
    X(11, OP_FWD, PATH_VECTOR ,  512, 2,  1, 0, 1, DT_ANY,     0,     0) \
    X(12, OP_FWD, PATH_VECTOR , 1024, 1,  1, 0, 1, DT_ANY,     0,     0) \
    X(13, OP_FWD, PATH_VECTOR ,  256, 2,  2, 0, 1, DT_ANY,     0,     0) \
    X(14, OP_FWD, PATH_VECTOR ,   64, 8,  4, 0, 1, DT_ANY,     0,     0) \
    X(15, OP_FWD, PATH_VECTOR ,   16, 2, 16, 0, 1, DT_ANY,     0,     0) \
    /* forward rows wider than 2048 chunks, streamed through two \
       shared-memory stages by a persistent grid of 2- or 4-CTA clusters \
       (two stages leave room for 2-3 CTAs an SM); rows above 8192 chunks \
       keep the register cluster plans */ \
    X(141, OP_FWD_STAGED, PATH_RESTAGED, 512, 3, 1, 2, 2, DT_ANY, 2049,  3072) \
    X(139, OP_FWD_STAGED, PATH_RESTAGED, 512, 4, 1, 2, 2, DT_ANY, 3073,  4096) \
    X(145, OP_FWD_STAGED, PATH_RESTAGED, 512, 3, 1, 2, 4, DT_ANY, 4097,  6144) \
    X(143, OP_FWD_STAGED, PATH_RESTAGED, 512, 4, 1, 2, 4, DT_ANY, 6145,  8192) \
    X(138, OP_FWD_STAGED, PATH_RESTAGED, 512, 4, 1, 4, 1, DT_ANY,    0,     0) \
    /* forward rows no vectorised plan takes (any alignment): streamed \
       generic plans, rows in [cmin, cmax] elements */ \
    X(104, OP_FWD_STAGED, PATH_STREAM,   64,  4, 1, 6, 1, DT_ANY,     1,   256) \
    X(105, OP_FWD_STAGED, PATH_STREAM,   64, 16, 1, 4, 1, DT_ANY,   257,  1024) \
    X(106, OP_FWD_STAGED, PATH_STREAM,  128, 16, 1, 4, 1, DT_ANY,  1025,  2048) \
    X(107, OP_FWD_STAGED, PATH_STREAM,  256, 16, 1, 4, 1, DT_ANY,  2049,  4096) \
    X(108, OP_FWD_STAGED, PATH_STREAM,  512, 16, 1, 4, 1, DT_ANY,  4097,  8192) \
    X(109, OP_FWD_STAGED, PATH_STREAM, 1024, 16, 1, 4, 1, DT_ANY,  8193, 16384) \
    /* forward, any N and alignment */ \
    X(16, OP_FWD, PATH_GENERIC,  256, 0,  1, 0, 1, DT_ANY,     0,     0) \
    /* backward main kernel, persistent: rows in registers (vector) or \
       streamed into `depth` shared-memory stages by bulk copies (staged; \
       re-read from the stage in both passes from 1025 chunks on, where \
       holding four chunks a thread in registers spills; rows wider than \
       2048 chunks shared by a cluster of 2 or 4 staged CTAs) */ \
    X(20, OP_BWD, PATH_VECTOR ,    8, 1, 32, 1, 1, DT_ANY,     1,     8) \
    X(21, OP_BWD, PATH_VECTOR ,   16, 1, 16, 1, 1, DT_ANY,     9,    16) \
    X(22, OP_BWD, PATH_VECTOR ,   32, 1,  8, 1, 1, DT_ANY,    17,    32) \
    X(23, OP_BWD, PATH_VECTOR ,   32, 2,  8, 1, 1, DT_ANY,    33,    64) \
    X(24, OP_BWD, PATH_VECTOR ,   64, 2,  4, 1, 1, DT_ANY,    65,   128) \
    X(25, OP_BWD, PATH_VECTOR ,  128, 2,  2, 1, 1, DT_ANY,   129,   256) \
    X(95, OP_BWD, PATH_STAGED ,  256, 2,  1, 4, 1, DT_ANY,   257,   512) \
    X(88, OP_BWD, PATH_STAGED ,  512, 2,  1, 4, 1, DT_ANY,   513,  1024) \
    X(121, OP_BWD, PATH_RESTAGED, 512, 3, 1, 3, 1, DT_ANY,  1025,  1536) \
    X(118, OP_BWD, PATH_RESTAGED, 512, 4, 1, 2, 1, DT_ANY,  1537,  2048) \
    X(127, OP_BWD, PATH_RESTAGED, 512, 3, 1, 3, 2, DT_ANY,  2049,  3072) \
    X(123, OP_BWD, PATH_RESTAGED, 512, 4, 1, 2, 2, DT_ANY,  3073,  4096) \
    X(128, OP_BWD, PATH_RESTAGED, 512, 3, 1, 3, 4, DT_ANY,  4097,  6144) \
    X(124, OP_BWD, PATH_RESTAGED, 512, 4, 1, 2, 4, DT_ANY,  6145,  8192) \
    X(46, OP_BWD, PATH_VECTOR ,  512, 2,  1, 1, 4, DT_ANY,     0,     0) \
    X(47, OP_BWD, PATH_VECTOR ,  512, 2,  1, 1, 8, DT_ANY,     0,     0) \
    X(26, OP_BWD, PATH_VECTOR ,  256, 2,  2, 1, 1, DT_ANY,     0,     0) \
    X(96, OP_BWD, PATH_STAGED ,  512, 3,  1, 3, 1, DT_ANY,     0,     0) \
    X(97, OP_BWD, PATH_STAGED ,  512, 4,  1, 2, 1, DT_ANY,     0,     0) \
    X(45, OP_BWD, PATH_VECTOR ,  512, 2,  1, 1, 2, DT_ANY,     0,     0) \
    X(38, OP_BWD, PATH_VECTOR ,  256, 2,  2, 2, 1, DT_ANY,     0,     0) \
    X(27, OP_BWD, PATH_VECTOR ,  512, 2,  1, 1, 1, DT_ANY,     0,     0) \
    X(34, OP_BWD, PATH_VECTOR ,  512, 2,  1, 2, 1, DT_ANY,     0,     0) \
    X(42, OP_BWD, PATH_VECTOR ,  512, 3,  1, 1, 1, DT_ANY,     0,     0) \
    X(32, OP_BWD, PATH_VECTOR ,  256, 1,  2, 2, 1, DT_ANY,     0,     0) \
    X(33, OP_BWD, PATH_VECTOR ,   16, 2, 16, 1, 1, DT_ANY,     0,     0) \
    X(35, OP_BWD, PATH_VECTOR ,  512, 2,  1, 0, 1, DT_ANY,     0,     0) \
    X(40, OP_BWD, PATH_VECTOR ,  128, 2,  2, 2, 1, DT_ANY,     0,     0) \
    X(41, OP_BWD, PATH_VECTOR ,  128, 2,  4, 1, 1, DT_ANY,     0,     0) \
    X(44, OP_BWD, PATH_VECTOR ,  512, 3,  1, 2, 1, DT_ANY,     0,     0) \
    X(48, OP_BWD, PATH_VECTOR ,  512, 3,  1, 1, 2, DT_ANY,     0,     0) \
    X(49, OP_BWD, PATH_VECTOR ,  512, 2,  1, 2, 2, DT_ANY,     0,     0) \
    X(50, OP_BWD, PATH_VECTOR ,  256, 2,  1, 1, 2, DT_ANY,     0,     0) \
    X(51, OP_BWD, PATH_VECTOR ,  512, 1,  1, 1, 2, DT_ANY,     0,     0) \
    X(52, OP_BWD, PATH_VECTOR ,  128, 2,  1, 1, 2, DT_ANY,     0,     0) \
    X(53, OP_BWD, PATH_VECTOR ,  256, 1,  1, 1, 2, DT_ANY,     0,     0) \
    X(54, OP_BWD, PATH_VECTOR ,  256, 2,  1, 1, 4, DT_ANY,     0,     0) \
    X(55, OP_BWD, PATH_VECTOR ,  128, 2,  1, 1, 4, DT_ANY,     0,     0) \
    X(89, OP_BWD, PATH_STAGED ,  512, 2,  1, 3, 1, DT_ANY,     0,     0) \
    X(90, OP_BWD, PATH_STAGED ,  256, 4,  1, 4, 1, DT_ANY,     0,     0) \
    X(91, OP_BWD, PATH_STAGED ,  512, 1,  1, 6, 1, DT_ANY,     0,     0) \
    X(92, OP_BWD, PATH_STAGED ,  256, 2,  1, 6, 1, DT_ANY,     0,     0) \
    X(93, OP_BWD, PATH_STAGED ,  256, 1,  1, 8, 1, DT_ANY,     0,     0) \
    X(94, OP_BWD, PATH_STAGED ,  128, 2,  1, 8, 1, DT_ANY,     0,     0) \
    X(98, OP_BWD, PATH_STAGED ,  512, 3,  1, 2, 1, DT_ANY,     0,     0) \
    X(119, OP_BWD, PATH_RESTAGED, 512, 4, 1, 3, 1, DT_ANY,     0,     0) \
    X(131, OP_BWD, PATH_RESTAGED, 512, 4, 1, 3, 2, DT_ANY,     0,     0) \
    /* backward main kernel, any N and alignment */ \
    X(36, OP_BWD, PATH_GENERIC,  256, 0,  1, 0, 1, DT_ANY,     0,     0) \
    /* ... streamed (rows in [cmin, cmax] elements; the smaller CTAs of \
       shorter rows keep more rows in flight an SM) */ \
    X(58, OP_BWD, PATH_STREAM ,   64,  4, 1, 6, 1, DT_ANY,     1,   256) \
    X(57, OP_BWD, PATH_STREAM ,   64, 16, 1, 4, 1, DT_ANY,   257,  1024) \
    X(56, OP_BWD, PATH_STREAM ,  128, 16, 1, 4, 1, DT_ANY,  1025,  2048) \
    X(43, OP_BWD, PATH_STREAM ,  256, 16, 1, 3, 1, DT_ANY,  2049,  4096) \
    X(37, OP_BWD, PATH_STREAM ,  512, 16, 1, 8, 1, DT_ANY,  4097,  8192) \
    /* LayerNorm backward main kernel, persistent, row in registers (two \
       chunks a thread where the row allows) or staged; from 1025 chunks of \
       a 2-byte type on the re-read schedule with gamma in shared memory */ \
    X(60, OP_LN_BWD, PATH_VECTOR,    8, 1, 32, 1, 1, DT_ANY,     1,     8) \
    X(61, OP_LN_BWD, PATH_VECTOR,   16, 1, 16, 1, 1, DT_ANY,     9,    16) \
    X(62, OP_LN_BWD, PATH_VECTOR,   32, 1,  8, 1, 1, DT_ANY,    17,    32) \
    X(63, OP_LN_BWD, PATH_VECTOR,   64, 1,  4, 1, 1, DT_ANY,    33,    64) \
    X(64, OP_LN_BWD, PATH_VECTOR,  128, 1,  2, 1, 1, DT_ANY,    65,   128) \
    X(103, OP_LN_BWD, PATH_STAGED, 128, 2,  1, 6, 1, DT_ANY,   129,   256) \
    X(100, OP_LN_BWD, PATH_STAGED, 256, 2,  1, 4, 1, DT_ANY,   257,   512) \
    X(112, OP_LN_BWD, PATH_STAGED, 256, 4,  1, 4, 1, DT_ANY,   513,  1024) \
    X(101, OP_LN_BWD, PATH_STAGED, 512, 3,  1, 3, 1, DT_F32,  1025,  1536) \
    X(122, OP_LN_BWD, PATH_RESTAGED, 512, 3, 1, 2, 1, DT_16,  1025,  1536) \
    X(116, OP_LN_BWD, PATH_RESTAGED, 512, 4, 1, 2, 1, DT_ANY,  1537,  2048) \
    X(129, OP_LN_BWD, PATH_RESTAGED, 512, 3, 1, 3, 2, DT_ANY, 2049,  3072) \
    X(125, OP_LN_BWD, PATH_RESTAGED, 512, 4, 1, 2, 2, DT_ANY, 3073,  4096) \
    X(130, OP_LN_BWD, PATH_RESTAGED, 512, 3, 1, 3, 4, DT_ANY, 4097,  6144) \
    X(126, OP_LN_BWD, PATH_RESTAGED, 512, 4, 1, 2, 4, DT_ANY, 6145,  8192) \
    X(87, OP_LN_BWD, PATH_VECTOR,  512, 2,  1, 1, 4, DT_ANY,     0,     0) \
    X(70, OP_LN_BWD, PATH_VECTOR,  512, 2,  1, 1, 8, DT_ANY,     0,     0) \
    X(81, OP_LN_BWD, PATH_VECTOR,  128, 2,  2, 1, 1, DT_ANY,     0,     0) \
    X(86, OP_LN_BWD, PATH_VECTOR,  512, 2,  1, 1, 2, DT_ANY,     0,     0) \
    X(82, OP_LN_BWD, PATH_VECTOR,  256, 2,  1, 1, 1, DT_ANY,     0,     0) \
    X(65, OP_LN_BWD, PATH_VECTOR,  256, 1,  1, 1, 1, DT_ANY,     0,     0) \
    X(66, OP_LN_BWD, PATH_VECTOR,  512, 1,  1, 1, 1, DT_ANY,     0,     0) \
    X(67, OP_LN_BWD, PATH_VECTOR,  512, 1,  1, 1, 2, DT_ANY,     0,     0) \
    X(68, OP_LN_BWD, PATH_VECTOR,  512, 1,  1, 1, 4, DT_ANY,     0,     0) \
    X(69, OP_LN_BWD, PATH_VECTOR,  512, 1,  1, 1, 8, DT_ANY,     0,     0) \
    X(71, OP_LN_BWD, PATH_VECTOR,  512, 1,  1, 2, 1, DT_ANY,     0,     0) \
    X(73, OP_LN_BWD, PATH_VECTOR,  512, 1,  1, 2, 2, DT_ANY,     0,     0) \
    X(74, OP_LN_BWD, PATH_VECTOR,  256, 1,  1, 1, 4, DT_ANY,     0,     0) \
    X(77, OP_LN_BWD, PATH_VECTOR,  256, 2,  1, 1, 2, DT_ANY,     0,     0) \
    X(79, OP_LN_BWD, PATH_VECTOR,  256, 1,  2, 1, 1, DT_ANY,     0,     0) \
    X(83, OP_LN_BWD, PATH_VECTOR,  256, 2,  2, 1, 1, DT_ANY,     0,     0) \
    X(99, OP_LN_BWD, PATH_STAGED,  512, 2,  1, 4, 1, DT_ANY,     0,     0) \
    X(102, OP_LN_BWD, PATH_STAGED, 512, 4,  1, 2, 1, DT_ANY,     0,     0) \
    X(76, OP_LN_BWD, PATH_VECTOR,  512, 2,  1, 1, 1, DT_ANY,     0,     0) \
    X(113, OP_LN_BWD, PATH_STAGED, 512, 2,  1, 3, 1, DT_ANY,     0,     0) \
    X(114, OP_LN_BWD, PATH_STAGED, 512, 2,  1, 6, 1, DT_ANY,     0,     0) \
    X(115, OP_LN_BWD, PATH_RESTAGED, 512, 4, 1, 3, 1, DT_ANY,    0,     0) \
    X(117, OP_LN_BWD, PATH_RESTAGED, 512, 3, 1, 3, 1, DT_ANY,    0,     0) \
    X(120, OP_LN_BWD, PATH_RESTAGED, 512, 2, 1, 4, 1, DT_ANY,    0,     0) \
    X(72, OP_LN_BWD, PATH_GENERIC,  256, 0,  1, 0, 1, DT_ANY,     0,     0)

// Largest CTA any plan uses.
constexpr int kMaxCtaThreads = 1024;
// Plan ids are below this bound (host caches are indexed by id).
constexpr int kMaxPlanId = 160;

struct FwdParams {
    const void *x;
    const void *residual;    // NULL: plain forward
    const void *w;
    void *y;
    void *residual_out;      // fused only
    float *rstd;
    int64_t M;
    int N;
    float eps;
    float offset;
    // E4M3 output (y holds one byte per element): the given per-tensor
    // scale, the reported 1/scale (one value, or one per row) and the
    // tensor's max |y| as fp32 bits (atomic max; NULL: not reported).
    const float *qscale;
    float *qscale_inv;
    unsigned int *qamax;
    // LayerNorm: the bias (NULL: none) and the per-row mean output
    const void *beta;
    float *mean;
    // staged forward: stages in use (0: the plan's depth) and the device
    // status word a bounded wait that gives up writes
    int stages = 0;
    int *status = nullptr;
    // generic LayerNorm forward: the row's h is kept in dynamic shared
    // memory between the passes (N elements + 16 bytes) instead of re-read
    // from L1/L2
    int cache_row = 0;
    // vectorised kernels: every row array starts `peel` elements past a
    // 16-byte boundary and the host passed each pointer moved back by that
    // many elements to the boundary; chunk 0 of a row is then wrapped
    // (wrap_chunk in common.cuh). 0: rows start on 16-byte boundaries.
    int peel = 0;
};

// Output of the forward: the activations' type, or E4M3 with a per-tensor
// scale, or E4M3 with a per-row scale from the row's own max |y|, or (fp32
// activations) bf16 or fp16: y rounded once from fp32 to the narrower type.
enum { QOUT_NONE = 0, QOUT_FP8_TENSOR = 1, QOUT_FP8_ROW = 2, QOUT_BF16 = 3, QOUT_F16 = 4 };
constexpr bool narrow_out(int q) { return q == QOUT_BF16 || q == QOUT_F16; }
constexpr bool fp8_out(int q) { return q == QOUT_FP8_TENSOR || q == QOUT_FP8_ROW; }

struct BwdParams {
    const void *dy;
    const void *x;           // h for the fused variant
    const void *w;
    const float *rstd;
    const void *dres;        // fused only, may be NULL
    void *dx;
    float *ws;               // [units, N] fp32 partial rows of dw (LayerNorm: [units, 2N], dgamma | dbeta)
    int *status;             // device word: set non-zero if a bounded wait gave up
    int64_t M;
    int N;
    float offset;
    const float *mean;       // LayerNorm: the forward's per-row mean
    int stages = 0;          // staged kernels: stages in use (2 .. the plan's depth; 0: the depth)
    int cache_row = 0;       // generic LayerNorm kernel: keep the row's x and dy in shared memory
    int peel = 0;            // vectorised kernels: rows at a common offset (as FwdParams::peel); a
                             // workspace partial row then holds parameter column (i - peel) mod N
                             // in its column i
};

// The generic LayerNorm backward's row cache: x and dy of the current row, each in
// a slot of this many bytes, placed at x's address mod 16 so that the
// row's 16-byte chunks stay aligned.
constexpr int64_t generic_bwd_cache_slot(int64_t N, int es) { return (N * es + 31) / 16 * 16; }

// The streamed generic backward's stage slot for one array's row: its
// 16-byte cover at the worst offset (15 bytes past a boundary).
constexpr int64_t stream_slot_bytes(int64_t N, int es) { return (N * es + 30) / 16 * 16; }

// Codes written to the status word: a bounded wait (a cluster row's peer
// partial, or a staged row's bulk copy) gave up.
constexpr int kStatusWaitTimeout = 1;
// Polls of an mbarrier before a wait gives up (at most seconds).
constexpr uint32_t kWaitLimit = 1u << 22;

// Launchers, defined in the per-type translation units that instantiate
// the kernels (suffix: activations' type, "w32" = fp32 weight). They return
// the launch's cudaError_t.
#define RMSN_DECLARE_LAUNCHERS(suf)                                                                       \
    int launch_fwd_##suf(int plan_id, bool fused, const FwdParams &p, int grid, void *stream);           \
    const void *fwd_kernel_ptr_##suf(int plan_id, bool fused);                                           \
    int launch_bwd_main_##suf(int plan_id, bool fused, bool packed, const BwdParams &p, int grid, int smem, \
                              void *stream);                                                           \
    const void *bwd_main_kernel_ptr_##suf(int plan_id, bool fused, bool packed);                          \
    int launch_fwd_staged_##suf(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream); \
    const void *fwd_staged_kernel_ptr_##suf(int plan_id, bool fused);
RMSN_DECLARE_LAUNCHERS(f32)
RMSN_DECLARE_LAUNCHERS(bf16)
RMSN_DECLARE_LAUNCHERS(f16)
RMSN_DECLARE_LAUNCHERS(bf16w32)
RMSN_DECLARE_LAUNCHERS(f16w32)
#undef RMSN_DECLARE_LAUNCHERS

// Rows at a common offset (FwdParams / BwdParams peel > 0): the default
// vectorised plans of RMSNorm and LayerNorm, forward and backward, compiled
// with the row's wrapped chunk 0 (PEEL), for the types whose weight (gamma,
// beta) is in the activations' type. The launchers above serve aligned rows.
#define RMSN_DECLARE_PEEL(suf)                                                                                  \
    int launch_fwd_peel_##suf(int plan_id, bool fused, const FwdParams &p, int grid, void *stream);            \
    int launch_fwd_staged_peel_##suf(int plan_id, bool fused, const FwdParams &p, int grid, int smem,           \
                                     void *stream);                                                             \
    const void *fwd_staged_kernel_ptr_peel_##suf(int plan_id, bool fused);                                     \
    int launch_ln_fwd_peel_##suf(int plan_id, bool fused, const FwdParams &p, int grid, void *stream);         \
    int launch_ln_fwd_staged_peel_##suf(int plan_id, bool fused, const FwdParams &p, int grid, int smem,        \
                                        void *stream);                                                          \
    const void *ln_fwd_staged_kernel_ptr_peel_##suf(int plan_id, bool fused);                                  \
    int launch_bwd_main_peel_##suf(int plan_id, bool fused, bool packed, const BwdParams &p, int grid, int smem, \
                                   void *stream);                                                               \
    const void *bwd_main_kernel_ptr_peel_##suf(int plan_id, bool fused, bool packed);                           \
    int launch_ln_bwd_peel_##suf(int plan_id, bool fused, const BwdParams &p, int grid, int smem, void *stream); \
    const void *ln_bwd_kernel_ptr_peel_##suf(int plan_id, bool fused);
RMSN_DECLARE_PEEL(f32)
RMSN_DECLARE_PEEL(bf16)
RMSN_DECLARE_PEEL(f16)
#undef RMSN_DECLARE_PEEL

// Forward with E4M3 output (mode QOUT_FP8_TENSOR or QOUT_FP8_ROW), for
// fp32, bf16 and fp16 activations with the weight in the same type, and
// for bf16 and fp16 activations with an fp32 weight ("w32"); on the
// register plans and the generic one, and on the staged forward plans
// (OP_FWD_STAGED defaults).
#define RMSN_DECLARE_FWD8(suf)                                                                            \
    int launch_fwd8_##suf(int plan_id, bool fused, int mode, const FwdParams &p, int grid, void *stream); \
    int launch_fwd8_staged_##suf(int plan_id, bool fused, int mode, const FwdParams &p, int grid, int smem, \
                                 void *stream);                                                           \
    const void *fwd8_staged_kernel_ptr_##suf(int plan_id, bool fused, int mode);
RMSN_DECLARE_FWD8(f32)
RMSN_DECLARE_FWD8(bf16)
RMSN_DECLARE_FWD8(f16)
RMSN_DECLARE_FWD8(bf16w32)
RMSN_DECLARE_FWD8(f16w32)
#undef RMSN_DECLARE_FWD8

// Opt a staged kernel into its largest dynamic shared memory on the current
// device (once per kernel and device); returns a cudaError_t.
int allow_staged_smem(const void *kernel);

// Parameter-gradient finalizers, by the parameters' storage type: column
// c < split of the [parts, ncols] workspace goes to out0[c], the others to
// out1[c - split] (out1 may be NULL: those columns are not written).
// Within each half (of split columns) the workspace column c holds
// parameter column (c - peel) mod split (peel > 0: rows at a common offset).
// sms: the device's SM count (it picks the finalizer's variant).
int launch_dw_finalize_f32(const float *ws, int parts, int ncols, void *out0, void *out1, int split, int peel,
                           void *stream, bool serial, int sms);
int launch_dw_finalize_bf16(const float *ws, int parts, int ncols, void *out0, void *out1, int split, int peel,
                            void *stream, bool serial, int sms);
int launch_dw_finalize_f16(const float *ws, int parts, int ncols, void *out0, void *out1, int split, int peel,
                           void *stream, bool serial, int sms);

// LayerNorm forward and backward main kernels (gamma and beta in the
// activations' type, or fp32 beside 16-bit activations: "w32"; the default
// plans and the generic one).
#define RMSN_DECLARE_LN(suf)                                                                               \
    int launch_ln_fwd_##suf(int plan_id, bool fused, const FwdParams &p, int grid, void *stream);         \
    int launch_ln_bwd_##suf(int plan_id, bool fused, const BwdParams &p, int grid, int smem, void *stream); \
    const void *ln_bwd_kernel_ptr_##suf(int plan_id, bool fused);                                        \
    int launch_ln_fwd_staged_##suf(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream); \
    const void *ln_fwd_staged_kernel_ptr_##suf(int plan_id, bool fused);
RMSN_DECLARE_LN(f32)
RMSN_DECLARE_LN(bf16)
RMSN_DECLARE_LN(f16)
RMSN_DECLARE_LN(bf16w32)
RMSN_DECLARE_LN(f16w32)
#undef RMSN_DECLARE_LN

}  // namespace rmsn
