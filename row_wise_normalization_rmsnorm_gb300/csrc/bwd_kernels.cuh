// bwd_kernels.cuh -- RMSNorm and LayerNorm backward kernels (plain and fused
// residual add): the register kernel, the staged (bulk-copy) kernel, the
// generic kernel and the parameter-gradient finalizer.
//
// Two launches, no global atomics and no inter-CTA waits (the kernel
// boundary is the only grid-wide barrier), after ROCm/FlyDSL PR #855
// (Implementation, "Hybrid atomic / two-stage backward"):
//
//  1. Main kernel, persistent: P CTAs walk the rows in a grid-stride loop.
//     A team of TPR threads owns a row; each thread holds V 16-byte chunks
//     of x and dy in registers across both passes over the row, and its
//     slice of (offset + w) for the whole run (loaded once per CTA):
//       pass 1  dot = sum_j g_j xhat_j       (g = dy (offset + w), xhat = x rstd)
//       pass 2  dx_j = rstd (g_j - xhat_j dot / N) [+ dres_j], stored directly
//               acc_j += dy_j xhat_j           (fp32, in registers)
//     At the end the CTA's teams are added in team order and the CTA writes
//     one fp32 partial row ws[cta, 0..N).
//  2. Finalizer: dw_j = R( sum_{p=0..P-1} ws[p, j] ) in a fixed order,
//     written in the parameter dtype.
//
// Arithmetic is done on fp32 pairs (even, odd column). With PACKED the pair
// ops are single f32x2 instructions (Liger-Kernel PR #1388, section 2:
// packed math where the wide-row backward is issue-bound); without it they
// are two fp32 intrinsics per pair. The association is the same, so the two
// variants produce identical bits.
//
// The LayerNorm backward runs on the same machinery (LN = true): the row
// carries the forward's mean as well as rstd, pass 1 reduces the pair
// (sum g, sum g (x - mean)), pass 2 writes
// dx = rstd (g - mean(g) - xhat mean(g xhat)), and each unit keeps two
// partial rows, dgamma = sum dy xhat and dbeta = sum dy, written as one
// [units, 2N] workspace row that one finalizer launch reduces.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "plans.h"

namespace rmsn {

// x, dy (and dres) chunks of one row, and its rstd, into registers. Rows
// past M are clamped to the last row (their results are masked later), so
// every thread of the CTA keeps taking part in the reductions. Rows at a
// common offset (p.peel) read their chunk 0 wrapped (ld_row_chunk).
template <typename T, int TPR, int V, bool LN, bool PEEL>
__device__ __forceinline__ void bwd_load_row(const BwdParams &p, int64_t row, int C, int cbase, int t,
                                             bool has_dres, uint4 (&x)[V], uint4 (&d)[V], uint4 (&r)[V],
                                             float &rs, float &mu) {
    const int64_t rr = row < p.M ? row : p.M - 1;
    const int64_t base = rr * C;
    const uint4 *x4 = reinterpret_cast<const uint4 *>(p.x) + base;
    const uint4 *d4 = reinterpret_cast<const uint4 *>(p.dy) + base;
    const uint4 *r4 = reinterpret_cast<const uint4 *>(p.dres) + base;
    const int peel = peel_of<PEEL>(p);
    const bool e0 = peel != 0 && cbase + t == 0;  // slot 0 is the row's wrapped chunk
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = cbase + v * TPR + t;
        const bool in = c < C;
        const bool edge = v == 0 && e0;
        x[v] = in ? ld_row_chunk<T>(x4, c, C, peel, edge) : make_uint4(0, 0, 0, 0);
        d[v] = in ? ld_row_chunk<T>(d4, c, C, peel, edge) : make_uint4(0, 0, 0, 0);
        r[v] = (has_dres && in) ? ld_row_chunk<T>(r4, c, C, peel, edge) : make_uint4(0, 0, 0, 0);
    }
    rs = p.rstd[rr];
    if constexpr (LN) mu = p.mean[rr];
}

// Persistent main kernel. Rows are software-pipelined through a register
// ring of D + 1 slots: while row k is reduced and written, the loads of rows
// k+1 .. k+D are already in flight, so the SM keeps memory requests
// outstanding across the reduction barrier and the stores. Each row's x and
// dy stay in registers across both passes.
// CS > 1: the CTAs of a cluster share each row (CTA rank r holds chunks
// [r TPR V, (r+1) TPR V)); the row sum meets in distributed shared memory
// and the cluster, not the CTA, owns one dW partial row.
template <typename T, typename TW, int TPR, int V, int TEAMS, int D, int CS, bool PACKED, bool FUSED, bool LN,
          bool PEEL>
__device__ __forceinline__ void bwd_vector_body(const BwdParams &p) {
    static_assert(CS == 1 || TEAMS == 1, "a cluster row uses one team per CTA");
    using Pk = Pair<PACKED>;
    using RT = typename std::conditional<LN, float2, float>::type;  // what a row reduces
    constexpr int E = Elem<T>::E;
    constexpr int NP = Elem<T>::NP;
    constexpr int W = TPR > 32 ? TPR / 32 : 1;
    constexpr int B = D + 1;              // ring slots
    constexpr int BR = FUSED ? B : 1;     // dres slots
    constexpr int NACC = LN ? 2 : 1;      // partial rows per unit
    __shared__ RT red[2][TEAMS][W * CS];              // row partials, double-buffered
    __shared__ __align__(8) uint64_t rbar[2][1];      // cluster rows: arrival of the peers' partials
    extern __shared__ float4 comb_smem[];      // (TEAMS - 1) * NACC * N floats
    pdl_wait();  // the kernel before it has completed (the forward's rstd, say)

    const int team = threadIdx.x / TPR;
    const int t = threadIdx.x % TPR;
    const int N = p.N;
    const int C = N / E;
    uint4 *dx4 = reinterpret_cast<uint4 *>(p.dx);
    const bool has_dres = FUSED && p.dres != nullptr;
    uint32_t rank = 0;
    if constexpr (CS > 1) rank = cluster_ctarank();
    const int cbase = (int)rank * TPR * V;  // first chunk of this CTA's slice
    const int peel = peel_of<PEEL>(p);
    const bool e0 = peel != 0 && cbase + t == 0;  // slot 0 is the row's wrapped chunk

    // (offset + w) for this thread's columns: loaded once per CTA. Without
    // a weight (non-affine) the factor is 1 and there is no dW.
    const bool has_w = p.w != nullptr;
    // partial rows wanted: RMSNorm with a weight; LayerNorm when the host
    // passes a workspace (dgamma and/or dbeta requested)
    const bool want_acc = LN ? p.ws != nullptr : has_w;
    const float2 o2 = make_float2(p.offset, p.offset);
    // The LayerNorm backward on 2-byte types keeps gamma as loaded (4
    // registers a chunk instead of 8) and forms offset + gamma when used:
    // the same fp32 add, so the same bits, and room for two chunks a thread.
    // The fp16 RMSNorm backward does the same (its fused variant otherwise
    // spills); for bf16 RMSNorm holding the fp32 factors measured faster.
    constexpr bool RAWW = std::is_same<T, TW>::value && Elem<T>::E == 8 &&
                          (LN || std::is_same<T, __half>::value);
    float2 wp[RAWW ? 1 : V][NP], acc[V][NP];
    uint4 wraw[RAWW ? V : 1];
    float2 accb[LN ? V : 1][NP];  // LayerNorm: sum dy (dbeta)
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = cbase + v * TPR + t;
        if constexpr (RAWW) {
            wraw[v] = (has_w && c < C) ? ld_w_raw<T>(p.w, c, C, peel, peel != 0 && c == 0) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < NP; ++k) {
                acc[v][k] = make_float2(0.f, 0.f);
                accb[v][k] = make_float2(0.f, 0.f);
            }
            continue;
        }
        float2 wv[NP];
        if (has_w && c < C) {
            load_w_chunk_row<T, TW>(p.w, c, C, peel, peel != 0 && c == 0, wv);
        } else {
#pragma unroll
            for (int k = 0; k < NP; ++k) wv[k] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            wp[v][k] = has_w ? Pk::add(o2, wv[k]) : make_float2(1.f, 1.f);
            acc[v][k] = make_float2(0.f, 0.f);
            if constexpr (LN) accb[v][k] = make_float2(0.f, 0.f);
        }
    }
    // the weight factors (offset + w) of chunk v
    auto wfac = [&](int v, float2 (&f)[NP]) {
        if constexpr (RAWW) {
            unpack<T>(wraw[v], f);
#pragma unroll
            for (int k = 0; k < NP; ++k) f[k] = has_w ? Pk::add(o2, f[k]) : make_float2(1.f, 1.f);
        } else {
#pragma unroll
            for (int k = 0; k < NP; ++k) f[k] = wp[v][k];
        }
    };

    // Every team of the CTA runs the same number of iterations (that of
    // team 0, which has the lowest first row) so the CTA-wide barrier in the
    // reduction is reached by all threads; rows past M are masked.
    // With clusters the unit is the cluster: cluster q takes rows q, q + Q, ...
    const int64_t unit = CS > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t units = CS > 1 ? (int64_t)cluster_count_x() : (int64_t)gridDim.x;
    const int64_t G = units * TEAMS;
    const int64_t first = unit * TEAMS + team;
    const int64_t iters = (p.M - unit * TEAMS + G - 1) / G;

    uint4 xb[B][V], db[B][V], rb[BR][V];
    float rs[B], mus[B];

    constexpr uint32_t kSlotBytes = CS * W * sizeof(RT);  // one row's partials from the whole cluster
    bool failed = false;

    auto process = [&](uint4 (&xv)[V], uint4 (&dv)[V], uint4 (&rv)[V], float r, float mu, int64_t k) {
        const int64_t row = first + k * G;
        const bool valid = row < p.M;
        const float2 r2 = make_float2(r, r);
        const float2 nmu2 = make_float2(-mu, -mu);  // LayerNorm: x - mean as x + (-mean)
        // the row's xhat for this pair of columns
        auto xhat = [&](float2 xf) { return LN ? Pk::mul(Pk::add(xf, nmu2), r2) : Pk::mul(xf, r2); };
        // pass 1: sum of g * x (g = dy (offset + w)); LayerNorm: the pair
        // (sum g, sum g (x - mean)). Even and odd columns accumulate in
        // separate lanes and are folded before the reduction.
        float2 dot = make_float2(0.f, 0.f), gsum = make_float2(0.f, 0.f);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float2 xf[NP], df[NP], wf[NP];
            unpack<T>(xv[v], xf);
            unpack<T>(dv[v], df);
            wfac(v, wf);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 g = Pk::mul(df[q], wf[q]);
                if constexpr (LN) {
                    dot = Pk::fma(g, Pk::add(xf[q], nmu2), dot);
                    gsum = Pk::add(gsum, g);
                } else {
                    dot = Pk::fma(g, xf[q], dot);
                }
            }
        }
        RT part;
        if constexpr (LN) part = make_float2(__fadd_rn(gsum.x, gsum.y), __fadd_rn(dot.x, dot.y));
        else part = __fadd_rn(dot.x, dot.y);
        RT s;
        if constexpr (CS > 1) {
            // Split-phase row sum across the cluster. Row k uses slot buffer
            // b = k & 1, whose barrier phase for it has parity (k >> 1) & 1.
            // Each warp sends its sum to its slot in every CTA of the
            // cluster with st.async, counted in bytes on the receiver's
            // barrier. A CTA reuses buffer b (row k + 2) only after every
            // warp of the row has sent its row k + 1 partial, which each
            // warp does after reading buffer b for row k.
            const int b = (int)(k & 1);
            RT wsum = part;
            if constexpr (LN) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) wsum = add2(wsum, shfl_xor2(wsum, o));
            } else {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) wsum = __fadd_rn(wsum, __shfl_xor_sync(0xffffffffu, wsum, o));
            }
            if ((t & 31) == 0) {
#pragma unroll
                for (int c = 0; c < CS; ++c) {
                    if constexpr (LN)
                        st_async_cluster2(&red[b][0][rank * W + (t >> 5)], &rbar[b][0], (uint32_t)c, wsum);
                    else
                        st_async_cluster(&red[b][0][rank * W + (t >> 5)], &rbar[b][0], (uint32_t)c, wsum);
                }
            }
            // while the partials travel: the parameter partials, which do
            // not need the row sums
            if (valid && want_acc) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    float2 xf[NP], df[NP];
                    unpack<T>(xv[v], xf);
                    unpack<T>(dv[v], df);
#pragma unroll
                    for (int q = 0; q < NP; ++q) {
                        acc[v][q] = Pk::fma(df[q], xhat(xf[q]), acc[v][q]);
                        if constexpr (LN) accb[v][q] = Pk::add(accb[v][q], df[q]);
                    }
                }
            }
            if (!mbar_wait(&rbar[b][0], (uint32_t)((k >> 1) & 1), kWaitLimit)) failed = true;
            if constexpr (LN) s = sum_slots2<CS * W>(&red[b][0][0], t & 31);
            else s = sum_slots<CS * W>(&red[b][0][0], t & 31);
            // re-arm this buffer for row k + 2 (its phase for row k is done)
            if (t == 0) mbar_arrive_expect_tx(&rbar[b][0], kSlotBytes);
        } else {
            if constexpr (LN) s = team_allreduce2<TPR>(part, &red[k & 1][team][0], t);
            else s = team_allreduce<TPR>(part, &red[k & 1][team][0], t);
        }
        // c = (1/N) sum g xhat = rstd * (sum g x) / N  (LayerNorm: sum g (x - mean));
        // LayerNorm also subtracts mean(g) = (sum g) / N
        float cm, nmg = 0.f;
        if constexpr (LN) {
            cm = -__fdiv_rn(__fmul_rn(s.y, r), (float)N);
            nmg = -__fdiv_rn(s.x, (float)N);
        } else {
            cm = -__fdiv_rn(__fmul_rn(s, r), (float)N);
        }
        const float2 nc2 = make_float2(cm, cm);
        const float2 nmg2 = make_float2(nmg, nmg);
        // pass 2: dx = rstd (g - xhat c) [+ dres], stored directly; dW partial
        const int64_t base = (valid ? row : p.M - 1) * C;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = cbase + v * TPR + t;
            float2 xf[NP], df[NP], out[NP];
            unpack<T>(xv[v], xf);
            unpack<T>(dv[v], df);
            float2 wf[NP];
            wfac(v, wf);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 xh = xhat(xf[q]);
                float2 g = Pk::mul(df[q], wf[q]);
                if constexpr (LN) g = Pk::add(g, nmg2);
                out[q] = Pk::mul(Pk::fma(xh, nc2, g), r2);
                if (CS == 1 && valid && want_acc) {
                    acc[v][q] = Pk::fma(df[q], xh, acc[v][q]);
                    if constexpr (LN) accb[v][q] = Pk::add(accb[v][q], df[q]);
                }
            }
            if (has_dres) {
                float2 rf[NP];
                unpack<T>(rv[v], rf);
#pragma unroll
                for (int q = 0; q < NP; ++q) out[q] = Pk::add(out[q], rf[q]);
            }
            if (valid && c < C) st_row_chunk<T>(dx4 + base, c, C, peel, v == 0 && e0, pack<T>(out));
        }
    };

    if constexpr (CS > 1) {
        if (t == 0) {
            // one arrival (the re-arm) plus the row's bytes
            mbar_init(&rbar[0][0], 1);
            mbar_init(&rbar[1][0], 1);
            mbar_arrive_expect_tx(&rbar[0][0], kSlotBytes);  // rows 0 and 1
            mbar_arrive_expect_tx(&rbar[1][0], kSlotBytes);
            mbar_init_fence();
        }
    }

    // prologue: rows 0 .. D-1 into slots 0 .. D-1
#pragma unroll
    for (int s = 0; s < D; ++s)
        if (s < iters)
            bwd_load_row<T, TPR, V, LN, PEEL>(p, first + s * G, C, cbase, t, has_dres, xb[s], db[s],
                                        rb[FUSED ? s : 0], rs[s], mus[s]);
    // every CTA of the cluster runs, with its barriers initialised, before
    // any peer stores into its shared memory
    if constexpr (CS > 1) cluster_sync();

    for (int64_t k0 = 0; k0 < iters; k0 += B) {
#pragma unroll
        for (int s = 0; s < B; ++s) {
            const int64_t k = k0 + s;
            if (k < iters) {
                // slot (s + D) % B held row k - 1, already done: refill it with row k + D
                const int sn = (s + D) % B;
                if (k + D < iters)
                    bwd_load_row<T, TPR, V, LN, PEEL>(p, first + (k + D) * G, C, cbase, t, has_dres, xb[sn], db[sn],
                                                rb[FUSED ? sn : 0], rs[sn], mus[sn]);
                process(xb[s], db[s], rb[FUSED ? s : 0], rs[s], mus[s], k);
                if (failed) break;
            }
        }
        if (failed) break;
    }
    if (failed) {
        // A peer's partial never arrived: record it and stop taking rows
        // (this call's outputs are incomplete). The host reads the word
        // with rmsnorm_device_status().
        if (p.status) *p.status = kStatusWaitTimeout;
    }

    // The finalizer may start launching now; it waits for this grid to
    // finish (pdl_wait) before it reads the workspace.
    pdl_trigger();

    if (!want_acc) return;  // no parameter partials (non-affine)

    // Combine the CTA's teams in team order, then write the unit's partial
    // row(s) ws[unit, :] (a cluster's CTAs each write their slice of it).
    // LayerNorm rows hold dgamma in [0, N) and dbeta in [N, 2N).
    float *wsrow = p.ws + unit * (int64_t)(NACC * N);
    if constexpr (TEAMS > 1) {
        float *comb = reinterpret_cast<float *>(comb_smem);
        if (team > 0) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int c = v * TPR + t;
                if (c < C) {
                    float *d = comb + (int64_t)(team - 1) * NACC * N + c * E;
#pragma unroll
                    for (int q = 0; q < NP; ++q) {
                        d[2 * q] = acc[v][q].x;
                        d[2 * q + 1] = acc[v][q].y;
                        if constexpr (LN) {
                            d[N + 2 * q] = accb[v][q].x;
                            d[N + 2 * q + 1] = accb[v][q].y;
                        }
                    }
                }
            }
        }
        __syncthreads();
        if (team != 0) return;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * TPR + t;
            if (c < C) {
                for (int tm = 1; tm < TEAMS; ++tm) {
                    const float *s2 = comb + (int64_t)(tm - 1) * NACC * N + c * E;
#pragma unroll
                    for (int q = 0; q < NP; ++q) {
                        acc[v][q] = Pk::add(acc[v][q], make_float2(s2[2 * q], s2[2 * q + 1]));
                        if constexpr (LN)
                            accb[v][q] = Pk::add(accb[v][q], make_float2(s2[N + 2 * q], s2[N + 2 * q + 1]));
                    }
                }
            }
        }
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = cbase + v * TPR + t;
        if (c < C) {
            float4 *d = reinterpret_cast<float4 *>(wsrow + c * E);
#pragma unroll
            for (int q = 0; q < NP / 2; ++q)
                d[q] = make_float4(acc[v][2 * q].x, acc[v][2 * q].y, acc[v][2 * q + 1].x, acc[v][2 * q + 1].y);
            if constexpr (LN) {
                float4 *db4 = reinterpret_cast<float4 *>(wsrow + N + c * E);
#pragma unroll
                for (int q = 0; q < NP / 2; ++q)
                    db4[q] = make_float4(accb[v][2 * q].x, accb[v][2 * q].y, accb[v][2 * q + 1].x,
                                         accb[v][2 * q + 1].y);
            }
        }
    }
}

template <typename T, typename TW, int TPR, int V, int TEAMS, int D, int CS, bool PACKED, bool FUSED,
          bool PEEL = false>
__global__ void __launch_bounds__(TPR *TEAMS) rmsnorm_bwd_vector(const BwdParams p) {
    bwd_vector_body<T, TW, TPR, V, TEAMS, D, CS, PACKED, FUSED, false, PEEL>(p);
}

template <typename T, typename TW, int TPR, int V, int TEAMS, int D, int CS, bool FUSED, bool PEEL = false>
__global__ void __launch_bounds__(TPR *TEAMS) layernorm_bwd_vector(const BwdParams p) {
    bwd_vector_body<T, TW, TPR, V, TEAMS, D, CS, true, FUSED, true, PEEL>(p);
}

// Staged persistent main kernel (bulk-copy pipeline). Each row's x and dy
// (and dres) stream from HBM into one of S shared-memory stages with
// cp.async.bulk, counted in bytes on the stage's mbarrier; the row team
// copies the stage into registers and runs the same two passes as the
// register kernel. The row reduction's barrier also proves that every warp
// has copied the stage out, so right after it thread 0 refills the stage
// with row k + S: S rows stay in flight whatever the register budget, no
// producer warp is needed (an extra warp would cut the registers a thread
// may use), and a row's loads never stall a consumer between its passes.
// Every wait is bounded: a wait that gives up records the status word and
// the kernel carries on (its outputs are then incomplete), so every thread
// still reaches every barrier and the kernel always ends.
//
// HOLD = false is the re-read schedule, for plans whose registers cannot
// hold a row's chunks across the reduction next to the parameter-gradient
// accumulators (the LayerNorm backward keeps two of them): both passes read
// the chunks from the stage, so the stage stays busy until the second pass
// ends. Each warp then counts itself done on the stage's counter and the
// last one to arrive refills the stage; no thread waits for the others. The
// arithmetic, and so every output bit, is that of HOLD = true.
template <typename T, typename TW, int TPR, int V, int S, int CS, bool FUSED, bool LN, bool HOLD, bool PACKED,
          bool PEEL>
__device__ __forceinline__ void staged_body(const BwdParams &p) {
    static_assert(CS == 1 || !HOLD, "cluster rows use the re-read schedule (no CTA barrier orders their refills)");
    using Pk = Pair<PACKED>;
    using RT = typename std::conditional<LN, float2, float>::type;  // what a row reduces
    constexpr int NACC = LN ? 2 : 1;     // partial rows per CTA
    constexpr int E = Elem<T>::E;
    constexpr int NP = Elem<T>::NP;
    constexpr int W = TPR / 32;          // warps of the row team
    constexpr int NB = FUSED ? 3 : 2;    // rows a stage holds: x, dy (, dres)
    static_assert(TPR % 32 == 0 && TPR >= 64, "whole warps");
    __shared__ RT red[2][CS * W];
    __shared__ __align__(8) uint64_t full[S];
    __shared__ __align__(8) uint64_t rbar[2];  // cluster rows: arrival of the peers' partials
    __shared__ unsigned done[HOLD ? 1 : S];  // re-read: warps through the stage's row
    extern __shared__ float4 stage_smem[];  // ns * NB * Cb chunks of 16 bytes (+ Cb for gamma)
    pdl_wait();  // before any read of the rows (the bulk copies included)
    // The LayerNorm re-read schedule keeps gamma in shared memory after the
    // stages rather than in registers (its two accumulators fill them); an
    // fp32 gamma beside 16-bit activations is read from global memory (L1)
    // where it is used instead.
    constexpr bool WSM = LN && !HOLD && std::is_same<T, TW>::value;
    constexpr bool GG = LN && !HOLD && !std::is_same<T, TW>::value;

    const int N = p.N;
    const int C = N / E;
    const int tid = threadIdx.x;
    // CS > 1: the CTAs of a cluster share each row in equal slices; CTA
    // rank r streams and owns chunks [r Cst, (r+1) Cst) of it (Cs of them,
    // fewer in the last slices, maybe none), the row sums meet in
    // distributed shared memory and the cluster is the unit that walks the
    // rows and owns a parameter-gradient partial row
    uint32_t rank = 0;
    if constexpr (CS > 1) rank = cluster_ctarank();
    const int Cst = (C + CS - 1) / CS;  // chunks of a CTA's slice (at most TPR V)
    const int cbase = (int)rank * Cst;
    const int Cs = C - cbase <= 0 ? 0 : (C - cbase < Cst ? C - cbase : Cst);
    // rows at a common offset: the CTA holding chunk 0 also stages aligned
    // chunk C (after its slice) to wrap chunk 0; a stage's row buffers are
    // one slot longer
    const int peel = peel_of<PEEL>(p);
    const bool wrap = peel != 0 && cbase == 0;
    const int Cb = Cst + (peel != 0 ? 1 : 0);  // slots of a stage's row buffer
    // chunk cl = v TPR + t of this CTA's slice from a staged row buffer;
    // only slot v = 0 of thread 0 can be the wrapped chunk (e0). The held
    // schedule reads a stage once: that thread merges the two parts as it
    // loads. The re-read schedule reads it twice: that thread wraps the
    // stage's chunk 0 in place once a row (wrap_staged) before reading it.
    const bool e0 = wrap && tid == 0;
    auto staged = [&](const uint4 *buf, int v, int cl) {
        if constexpr (HOLD)
            return v == 0 && e0 ? wrap_chunk<T>(lds128(buf), lds128(buf + Cst), peel) : lds128(buf + cl);
        else
            return lds128(buf + cl);
    };
    const int64_t unit = CS > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t G = CS > 1 ? (int64_t)cluster_count_x() : (int64_t)gridDim.x;
    const int64_t iters = unit < p.M ? (p.M - unit + G - 1) / G : 0;
    const bool has_dres = FUSED && p.dres != nullptr;
    const uint32_t row_bytes = (uint32_t)Cs * 16u;
    const int ns = p.stages >= 2 && p.stages < S ? p.stages : S;  // stages in use
    uint4 *stages = reinterpret_cast<uint4 *>(stage_smem);
    const uint4 *x4 = reinterpret_cast<const uint4 *>(p.x);
    const uint4 *d4 = reinterpret_cast<const uint4 *>(p.dy);
    const uint4 *r4 = reinterpret_cast<const uint4 *>(p.dres);
    // thread 0: stream row k into stage s (a CTA holding the whole row
    // stages aligned chunks 0 .. C of a row at a common offset in one copy)
    auto issue = [&](int64_t k, int s) {
        const int64_t row0 = (unit + k * G) * C;
        const int64_t off = row0 + cbase;
        uint4 *dst = stages + (size_t)s * NB * Cb;
        const uint32_t extra = wrap ? 16u : 0u;
        mbar_arrive_expect_tx(&full[s], (row_bytes + extra) * (has_dres ? 3u : 2u));
        if (row_bytes == 0) return;  // an empty slice: the arrival alone completes the phase
        auto copy = [&](uint4 *to, const uint4 *from) {
            if (CS == 1 || !wrap) {
                bulk_g2s(to, from + off, row_bytes + extra, &full[s]);
            } else {
                bulk_g2s(to, from + off, row_bytes, &full[s]);
                bulk_g2s(to + Cst, from + row0 + C, 16u, &full[s]);
            }
        };
        copy(dst, x4);
        copy(dst + Cb, d4);
        if (has_dres) copy(dst + 2 * Cb, r4);
    };
    uint4 *wsm = stages + (size_t)ns * NB * Cb;
    if constexpr (WSM) {
        if (p.w != nullptr)
            for (int c = tid; c < Cs; c += TPR) wsm[c] = ld_w_raw<T>(p.w, cbase + c, C, peel, wrap && c == 0);
    }
    constexpr uint32_t kSlotBytes = CS * W * sizeof(RT);  // one row's partials from the whole cluster
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        if constexpr (!HOLD) {
#pragma unroll
            for (int s = 0; s < S; ++s) done[s] = 0;
        }
        if constexpr (CS > 1) {
            // one arrival (the re-arm) plus the row's bytes; rows 0 and 1 armed here
            mbar_init(&rbar[0], 1);
            mbar_init(&rbar[1], 1);
            mbar_arrive_expect_tx(&rbar[0], kSlotBytes);
            mbar_arrive_expect_tx(&rbar[1], kSlotBytes);
        }
        mbar_init_fence();
        for (int s = 0; s < ns && s < iters; ++s) issue(s, s);
    }
    __syncthreads();
    // every CTA of the cluster runs, with its barriers initialised, before
    // any peer stores into its shared memory
    if constexpr (CS > 1) cluster_sync();

    const int t = tid;
    const int lane = t & 31;
    uint4 *dx4 = reinterpret_cast<uint4 *>(p.dx);
    const bool has_w = p.w != nullptr;
    // partial rows wanted: RMSNorm with a weight; LayerNorm when the host
    // passes a workspace (dgamma and/or dbeta requested)
    const bool want_acc = LN ? p.ws != nullptr : has_w;
    const float2 o2 = make_float2(p.offset, p.offset);
    // (offset + w) for this thread's chunks, in fp32; with three or more
    // chunks of a 2-byte type, w is held as loaded instead (one uint4 a
    // chunk) and offset + w formed when used (the same fp32 add each time),
    // which keeps the thread within its registers
    constexpr bool RAW = V >= 3 && E == 8 && std::is_same<T, TW>::value && !WSM;
    uint4 wraw[RAW ? V : 1];
    float2 wp[RAW || WSM || GG ? 1 : V][NP], acc[V][NP];
    float2 accb[LN ? V : 1][NP];  // LayerNorm: sum dy (dbeta)
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int cl = v * TPR + t;  // chunk of this CTA's slice; cbase + cl in the row
        if constexpr (WSM || GG) {
        } else if constexpr (RAW) {
            wraw[v] = (has_w && cl < Cs) ? ld_w_raw<T>(p.w, cbase + cl, C, peel, v == 0 && e0) : make_uint4(0, 0, 0, 0);
        } else {
            float2 wv[NP];
            if (has_w && cl < Cs) {
                load_w_chunk_row<T, TW>(p.w, cbase + cl, C, peel, v == 0 && e0, wv);
            } else {
#pragma unroll
                for (int q = 0; q < NP; ++q) wv[q] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < NP; ++q) wp[v][q] = has_w ? Pk::add(o2, wv[q]) : make_float2(1.f, 1.f);
        }
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            acc[v][q] = make_float2(0.f, 0.f);
            if constexpr (LN) accb[v][q] = make_float2(0.f, 0.f);
        }
    }
    auto wfac = [&](int v, float2 (&f)[NP]) {
        if constexpr (GG) {
            const int cl = v * TPR + t;
            if (has_w && cl < Cs) {
                load_w_chunk_row<T, TW>(p.w, cbase + cl, C, peel, v == 0 && e0, f);
            } else {
#pragma unroll
                for (int q = 0; q < NP; ++q) f[q] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < NP; ++q) f[q] = has_w ? Pk::add(o2, f[q]) : make_float2(1.f, 1.f);
        } else if constexpr (WSM || RAW) {
            const int cl = v * TPR + t;
            if constexpr (WSM)
                unpack<T>(has_w && cl < Cs ? lds128(wsm + cl) : make_uint4(0, 0, 0, 0), f);
            else
                unpack<T>(wraw[v], f);
#pragma unroll
            for (int q = 0; q < NP; ++q) f[q] = has_w ? Pk::add(o2, f[q]) : make_float2(1.f, 1.f);
        } else {
#pragma unroll
            for (int q = 0; q < NP; ++q) f[q] = wp[v][q];
        }
    };

    bool failed = false;
    int s = 0;          // stage of row k (k mod ns)
    uint32_t ph = 0;    // parity of k / S
    // the row statistics are loaded one row ahead, like the rows themselves
    float r_next = iters > 0 ? p.rstd[unit] : 0.f;
    float mu_next = (LN && iters > 0) ? p.mean[unit] : 0.f;
    for (int64_t k = 0; k < iters; ++k) {
        const int64_t row = unit + k * G;
        const float r = r_next;
        const float mu = mu_next;
        if (k + 1 < iters) {
            r_next = p.rstd[row + G];
            if constexpr (LN) mu_next = p.mean[row + G];
        }
        if (!mbar_wait(&full[s], ph, kWaitLimit)) failed = true;
        const int sk = s;  // this row's stage
        const uint4 *src = stages + (size_t)s * NB * Cb;
        if (!HOLD && e0) wrap_staged<T>(stages + (size_t)s * NB * Cb, Cb, has_dres ? 3 : 2, Cst, peel);
        // HOLD: the row's chunks, read once and kept for both passes
        uint4 xv[HOLD ? V : 1], dv[HOLD ? V : 1], rv[FUSED && HOLD ? V : 1];
        if constexpr (HOLD) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int cl = v * TPR + t;
                const bool in = cl < Cs;
                xv[v] = in ? staged(src, v, cl) : make_uint4(0, 0, 0, 0);
                dv[v] = in ? staged(src + Cb, v, cl) : make_uint4(0, 0, 0, 0);
                if constexpr (FUSED) rv[v] = (in && has_dres) ? staged(src + 2 * Cb, v, cl) : make_uint4(0, 0, 0, 0);
            }
        }
        // chunk v of the stage's x (b = 0), dy (1) or dres (2) row
        auto chunk = [&](int b, int v) {
            const int cl = v * TPR + t;
            return cl < Cs ? staged(src + b * Cb, v, cl) : make_uint4(0, 0, 0, 0);
        };

        const float2 r2 = make_float2(r, r);
        const float2 nmu2 = make_float2(-mu, -mu);  // LayerNorm: x - mean as x + (-mean)
        float2 dot = make_float2(0.f, 0.f), gsum = make_float2(0.f, 0.f);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float2 xf[NP], df[NP], wf[NP];
            unpack<T>(HOLD ? xv[HOLD ? v : 0] : chunk(0, v), xf);
            unpack<T>(HOLD ? dv[HOLD ? v : 0] : chunk(1, v), df);
            wfac(v, wf);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 g = Pk::mul(df[q], wf[q]);
                if constexpr (LN) {
                    dot = Pk::fma(g, Pk::add(xf[q], nmu2), dot);
                    gsum = Pk::add(gsum, g);
                } else {
                    dot = Pk::fma(g, xf[q], dot);
                }
            }
        }
        RT part;
        if constexpr (LN) {
            part = make_float2(__fadd_rn(gsum.x, gsum.y), __fadd_rn(dot.x, dot.y));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part = add2(part, shfl_xor2(part, o));
        } else {
            part = __fadd_rn(dot.x, dot.y);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, o));
        }
        RT *slots = &red[k & 1][0];
        if constexpr (CS > 1) {
            // Row k's warp sums go to slot buffer b = k & 1 of every CTA of
            // the cluster (st.async, counted in bytes on the receiver's
            // barrier, whose phase for row k has parity (k >> 1) & 1). A
            // buffer is written again (row k + 2) only after every warp of
            // the cluster sent its row k + 1 sum, which each warp does after
            // reading the buffer for row k.
            const int b = (int)(k & 1);
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < CS; ++c) {
                    if constexpr (LN)
                        st_async_cluster2(&red[b][rank * W + (t >> 5)], &rbar[b], (uint32_t)c, part);
                    else
                        st_async_cluster(&red[b][rank * W + (t >> 5)], &rbar[b], (uint32_t)c, part);
                }
            }
            if (!mbar_wait(&rbar[b], (uint32_t)((k >> 1) & 1), kWaitLimit)) failed = true;
        } else {
            if (lane == 0) slots[t >> 5] = part;
            __syncthreads();
            // every warp has copied stage s into registers: refill it with row k + ns
            if (HOLD && tid == 0 && k + ns < iters) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(k + ns, s);
            }
        }
        if (++s == ns) {
            s = 0;
            ph ^= 1u;
        }
        // c = rstd (sum g x) / N (LayerNorm: sum g (x - mean)); LayerNorm
        // also subtracts mean(g) = (sum g) / N
        float cm, nmg = 0.f;
        if constexpr (LN) {
            const float2 sum = sum_slots2<CS * W>(slots, lane);
            cm = -__fdiv_rn(__fmul_rn(sum.y, r), (float)N);
            nmg = -__fdiv_rn(sum.x, (float)N);
        } else {
            const float sum = sum_slots<CS * W>(slots, lane);
            cm = -__fdiv_rn(__fmul_rn(sum, r), (float)N);
        }
        // re-arm the slot buffer's barrier for row k + 2 (its phase for row k is done)
        if (CS > 1 && t == 0) mbar_arrive_expect_tx(&rbar[k & 1], kSlotBytes);
        const float2 nc2 = make_float2(cm, cm);
        const float2 nmg2 = make_float2(nmg, nmg);
        const int64_t base = row * C;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int cl = v * TPR + t;
            float2 xf[NP], df[NP], out[NP], wf[NP];
            unpack<T>(HOLD ? xv[HOLD ? v : 0] : chunk(0, v), xf);
            unpack<T>(HOLD ? dv[HOLD ? v : 0] : chunk(1, v), df);
            wfac(v, wf);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float2 xh = LN ? Pk::mul(Pk::add(xf[q], nmu2), r2) : Pk::mul(xf[q], r2);
                float2 g = Pk::mul(df[q], wf[q]);
                if constexpr (LN) g = Pk::add(g, nmg2);
                out[q] = Pk::mul(Pk::fma(xh, nc2, g), r2);
                if (want_acc) {
                    acc[v][q] = Pk::fma(df[q], xh, acc[v][q]);
                    if constexpr (LN) accb[v][q] = Pk::add(accb[v][q], df[q]);
                }
            }
            if constexpr (FUSED) {
                if (has_dres) {
                    float2 rf[NP];
                    unpack<T>(HOLD ? rv[HOLD ? v : 0] : chunk(2, v), rf);
#pragma unroll
                    for (int q = 0; q < NP; ++q) out[q] = Pk::add(out[q], rf[q]);
                }
            }
            if (cl < Cs) st_row_chunk<T>(dx4 + base, cbase + cl, C, peel, v == 0 && e0, pack<T>(out));
        }
        if constexpr (!HOLD) {
            // re-read: the warp is through stage sk; the last warp to say so
            // refills it with row k + ns (the fences order every warp's reads
            // of the stage before the bulk copies that overwrite it)
            __syncwarp();
            if (lane == 0 && k + ns < iters) {
                __threadfence_block();
                if (atomicAdd(&done[sk], 1u) == (unsigned)(W - 1)) {
                    __threadfence_block();
                    done[sk] = 0;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(k + ns, sk);
                }
            }
        }
    }
    if (failed && p.status) *p.status = kStatusWaitTimeout;
    // no CTA leaves while a peer may still store into its shared memory
    if constexpr (CS > 1) cluster_sync();

    // The finalizer may start launching now; it waits for this grid to
    // finish (pdl_wait) before it reads the workspace.
    pdl_trigger();
    if (!want_acc) return;
    // the unit's partial row(s): dW, or LayerNorm's dgamma | dbeta (a
    // cluster CTA writes the columns of its slice)
    float *wsrow = p.ws + unit * (int64_t)(NACC * N);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int cl = v * TPR + t;
        if (cl < Cs) {
            const int c = cbase + cl;
            float4 *d = reinterpret_cast<float4 *>(wsrow + c * E);
#pragma unroll
            for (int q = 0; q < NP / 2; ++q)
                d[q] = make_float4(acc[v][2 * q].x, acc[v][2 * q].y, acc[v][2 * q + 1].x, acc[v][2 * q + 1].y);
            if constexpr (LN) {
                float4 *db4 = reinterpret_cast<float4 *>(wsrow + N + c * E);
#pragma unroll
                for (int q = 0; q < NP / 2; ++q)
                    db4[q] = make_float4(accb[v][2 * q].x, accb[v][2 * q].y, accb[v][2 * q + 1].x,
                                         accb[v][2 * q + 1].y);
            }
        }
    }
}

template <typename T, typename TW, int TPR, int V, int S, int CS, bool FUSED, bool HOLD, bool PACKED = true,
          bool PEEL = false>
__global__ void __launch_bounds__(TPR, 1) rmsnorm_bwd_staged(const BwdParams p) {
    staged_body<T, TW, TPR, V, S, CS, FUSED, false, HOLD, PACKED, PEEL>(p);
}

template <typename T, typename TW, int TPR, int V, int S, int CS, bool FUSED, bool HOLD, bool PEEL = false>
__global__ void __launch_bounds__(TPR, 1) layernorm_bwd_staged(const BwdParams p) {
    staged_body<T, TW, TPR, V, S, CS, FUSED, true, HOLD, true, PEEL>(p);
}

// Generic main kernel: one 256-thread CTA per row at a time, any N and
// alignment, each row read twice (the second read is served by L1/L2). The
// CTA's dW partial row lives in the workspace itself: the thread that
// handles column j writes ws[cta, j] on the CTA's first row and updates it
// on later rows; the row reduction's barrier orders those updates, so no
// atomics are needed. Rows split by x's address into an element-wise head,
// 16-byte chunks and an element-wise tail; dy, dx and dres take 16-byte
// accesses where they share x's address mod 16. The workspace is updated
// one column a thread (coalesced) in a loop of its own.
template <typename T, typename TW, bool FUSED>
__global__ void __launch_bounds__(256) rmsnorm_bwd_generic(const BwdParams p) {
    __shared__ float red[32];
    pdl_wait();
    constexpr int NP = Elem<T>::NP;
    const int N = p.N;
    const TW *w = reinterpret_cast<const TW *>(p.w);
    float *wsrow = p.ws + (int64_t)blockIdx.x * N;
    const bool has_dres = FUSED && p.dres != nullptr;
    const uint32_t a16 = addr_mod16(p.x);
    const bool vdy = addr_mod16(p.dy) == a16, vdx = addr_mod16(p.dx) == a16;
    const bool vdr = has_dres && addr_mod16(p.dres) == a16;
    bool first = true;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const T *x = reinterpret_cast<const T *>(p.x) + row * N;
        const T *dy = reinterpret_cast<const T *>(p.dy) + row * N;
        const T *dr = reinterpret_cast<const T *>(p.dres) + row * N;
        T *dx = reinterpret_cast<T *>(p.dx) + row * N;
        const float r = p.rstd[row];
        const RowSplit sp = row_split(x, N, true);
        // the chunk at column j0: dy, x and the weight factors
        auto chunk = [&](int64_t j0, float2 (&dv)[NP], float2 (&xv)[NP], float2 (&wf)[NP]) {
            load_chunk_at(dy, j0, vdy, dv);
            load_chunk_at(x, j0, true, xv);
            if (w) {
                w_chunk_at<T, TW>(w, (int)j0, wf);
#pragma unroll
                for (int q = 0; q < NP; ++q) wf[q] = make_float2(__fadd_rn(p.offset, wf[q].x), __fadd_rn(p.offset, wf[q].y));
            }
        };
        float dot = 0.f;
        auto dot_elem = [&](int j) {
            const float dyj = load_elem(dy, j);
            const float g = w ? __fmul_rn(dyj, __fadd_rn(p.offset, load_w(w, j))) : dyj;
            dot = __fmaf_rn(g, __fmul_rn(load_elem(x, j), r), dot);
        };
        for (int j = threadIdx.x; j < sp.head; j += blockDim.x) dot_elem(j);
        for (int c = threadIdx.x; c < sp.nb; c += blockDim.x) {
            float2 dv[NP], xv[NP], wf[NP];
            chunk(sp.head + (int64_t)c * Elem<T>::E, dv, xv, wf);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float gx = w ? __fmul_rn(dv[q].x, wf[q].x) : dv[q].x;
                const float gy = w ? __fmul_rn(dv[q].y, wf[q].y) : dv[q].y;
                dot = __fmaf_rn(gx, __fmul_rn(xv[q].x, r), dot);
                dot = __fmaf_rn(gy, __fmul_rn(xv[q].y, r), dot);
            }
        }
        for (int j = sp.tail0 + threadIdx.x; j < N; j += blockDim.x) dot_elem(j);
        // the dW partial, one column a thread (coalesced; the reads are L1
        // hits), before the reduction's barrier: dx may overwrite dy later
        if (w) {
            for (int j = threadIdx.x; j < N; j += blockDim.x) {
                const float dyj = load_elem(dy, j), xh = __fmul_rn(load_elem(x, j), r);
                wsrow[j] = first ? __fmul_rn(dyj, xh) : __fmaf_rn(dyj, xh, wsrow[j]);
            }
        }
        const float cm = -__fdiv_rn(cta_allreduce(dot, red), (float)N);
        // dx of column j from xhat_j and g_j
        auto out_elem = [&](float xh, float g, float drj) {
            float d = __fmul_rn(__fmaf_rn(xh, cm, g), r);
            if (has_dres) d = __fadd_rn(d, drj);
            return d;
        };
        auto dx_elem = [&](int j) {
            const float dyj = load_elem(dy, j);
            const float xh = __fmul_rn(load_elem(x, j), r);
            const float g = w ? __fmul_rn(dyj, __fadd_rn(p.offset, load_w(w, j))) : dyj;
            store_elem(dx, j, out_elem(xh, g, has_dres ? load_elem(dr, j) : 0.f));
        };
        for (int j = threadIdx.x; j < sp.head; j += blockDim.x) dx_elem(j);
        for (int c = threadIdx.x; c < sp.nb; c += blockDim.x) {
            const int64_t j0 = sp.head + (int64_t)c * Elem<T>::E;
            float2 dv[NP], xv[NP], wf[NP], rv[NP];
            chunk(j0, dv, xv, wf);
            if (has_dres) load_chunk_at(dr, j0, vdr, rv);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float xhx = __fmul_rn(xv[q].x, r), xhy = __fmul_rn(xv[q].y, r);
                const float gx = w ? __fmul_rn(dv[q].x, wf[q].x) : dv[q].x;
                const float gy = w ? __fmul_rn(dv[q].y, wf[q].y) : dv[q].y;
                xv[q] = make_float2(out_elem(xhx, gx, has_dres ? rv[q].x : 0.f), out_elem(xhy, gy, has_dres ? rv[q].y : 0.f));
            }
            store_chunk_at(dx, j0, vdx, xv);
        }
        for (int j = sp.tail0 + threadIdx.x; j < N; j += blockDim.x) dx_elem(j);
        first = false;
    }
    pdl_trigger();  // this CTA's rows done (the finalizer waits for the whole grid)
}

// Streamed generic main kernel: persistent CTAs, rows of any alignment and
// of at most TPR * K elements. Row k of a CTA streams into stage k mod ns
// by bulk copies of the 16-byte covers (cover16) of its x and dy (and dres)
// rows, each array's row at its own offset within its first block, so the
// arrays need not share an address mod 16 and N need not fill whole
// blocks. The row's rstd travels with it (a 4-byte asynchronous copy into
// the stage, counted as the stage barrier's second arrival), so no global
// load sits on a row's critical path. Thread t owns columns t + i TPR
// (i < K) of every row: its share of the dW partial row stays in registers
// for the whole kernel and is written to the workspace once. Each thread
// reads its elements of the stage into registers before the row
// reduction's barrier; right after the barrier thread 0 refills the stage
// with row k + ns, as the staged kernels do. dx is stored element by
// element: a row's first and last 16-byte blocks may hold a neighbouring
// row, which another CTA writes. The arithmetic is the staged kernels' in
// per-lane fp32: g = dy (offset + w), c = rstd (sum g x) / N,
// dx = (xhat (-c) + g) rstd (+ dres), dW += dy xhat. Every wait is bounded:
// one that gives up records the status word, waits (again bounded) for the
// stages' last copies and lets the kernel end.
template <typename T, typename TW, int TPR, int K, int SMAX, bool FUSED>
__global__ void __launch_bounds__(TPR, TPR >= 512 ? 1 : 512 / TPR) rmsnorm_bwd_stream(const BwdParams p) {
    static_assert(TPR % 32 == 0 && TPR >= 64 && TPR <= 1024, "whole warps");
    constexpr int W = TPR / 32;
    constexpr int NB = FUSED ? 3 : 2;  // arrays a stage holds: x, dy (, dres)
    __shared__ float red[2][W];
    __shared__ __align__(8) uint64_t full[SMAX];
    __shared__ float rs_ring[SMAX];         // the stage's row rstd
    extern __shared__ float4 stage_smem[];  // ns * NB slots of stream_slot_bytes(N, sizeof(T))
    pdl_wait();  // before any read of the rows (the bulk copies included)
    const int N = p.N;
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int ns = p.stages;  // 2 .. SMAX, chosen by the host to fit
    const int64_t G = gridDim.x;
    const int64_t unit = blockIdx.x;
    const int64_t iters = unit < p.M ? (p.M - unit + G - 1) / G : 0;
    const bool has_dres = FUSED && p.dres != nullptr;
    const bool has_w = p.w != nullptr;
    const uint32_t rb = (uint32_t)N * (uint32_t)sizeof(T);  // bytes of a row
    const uint32_t slot = (uint32_t)stream_slot_bytes(N, (int)sizeof(T));
    char *const stages = reinterpret_cast<char *>(stage_smem);
    const char *gx = static_cast<const char *>(p.x);
    const char *gd = static_cast<const char *>(p.dy);
    const char *gr = static_cast<const char *>(p.dres);
    // thread 0: the covers of row k's arrays, and its rstd, into stage s
    auto issue = [&](int64_t k, int s) {
        const int64_t row = unit + k * G;
        const int64_t off = row * (int64_t)rb;
        const Cover cx = cover16(gx + off, rb);
        const Cover cd = cover16(gd + off, rb);
        const Cover cr = has_dres ? cover16(gr + off, rb) : Cover{nullptr, 0u, 0u};
        char *dst = stages + (size_t)s * NB * slot;
        mbar_arrive_expect_tx(&full[s], cx.bytes + cd.bytes + cr.bytes);
        bulk_g2s(dst, cx.src, cx.bytes, &full[s]);
        bulk_g2s(dst + slot, cd.src, cd.bytes, &full[s]);
        if (has_dres) bulk_g2s(dst + 2 * slot, cr.src, cr.bytes, &full[s]);
        cp_async4(&rs_ring[s], p.rstd + row);
        cp_async_arrive_noinc(&full[s]);
    };
    // (offset + w) of this thread's columns, and its dW partials
    const TW *w = static_cast<const TW *>(p.w);
    float wf[K], acc[K];
#pragma unroll
    for (int i = 0; i < K; ++i) {
        const int j = t + i * TPR;
        wf[i] = (has_w && j < N) ? __fadd_rn(p.offset, load_w(w, j)) : 1.f;
        acc[i] = 0.f;
    }
    if (t == 0) {
        // two arrivals a phase: the copies' announcement and the rstd copy's
        for (int s = 0; s < ns; ++s) mbar_init(&full[s], 2);
        mbar_init_fence();
        for (int s = 0; s < ns && s < iters; ++s) issue(s, s);
    }
    __syncthreads();

    bool failed = false;
    int s = 0;        // stage of row k (k mod ns)
    uint32_t ph = 0;  // parity of k / ns
    for (int64_t k = 0; k < iters; ++k) {
        const int64_t row = unit + k * G;
        if (!mbar_wait(&full[s], ph, kWaitLimit)) failed = true;
        const float r = rs_ring[s];  // read before the barrier that frees the stage
        // element 0 of the row's arrays in the stage
        const int64_t off = row * (int64_t)rb;
        const char *sb = stages + (size_t)s * NB * slot;
        const T *xs = reinterpret_cast<const T *>(sb + addr_mod16(gx + off));
        const T *ds = reinterpret_cast<const T *>(sb + slot + addr_mod16(gd + off));
        const T *rs = reinterpret_cast<const T *>(sb + 2 * slot + (has_dres ? addr_mod16(gr + off) : 0u));
        float xv[K], dv[K], rv[FUSED ? K : 1];
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int j = t + i * TPR;
            const bool in = j < N;
            xv[i] = in ? load_elem(xs, j) : 0.f;
            dv[i] = in ? load_elem(ds, j) : 0.f;
            if constexpr (FUSED) rv[i] = (in && has_dres) ? load_elem(rs, j) : 0.f;
            dot = __fmaf_rn(__fmul_rn(dv[i], wf[i]), xv[i], dot);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, o));
        float *slots = red[k & 1];
        if (lane == 0) slots[t >> 5] = dot;
        __syncthreads();
        // every thread has its elements of stage s: refill it with row k + ns
        if (t == 0 && k + ns < iters) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(k + ns, s);
        }
        if (++s == ns) {
            s = 0;
            ph ^= 1u;
        }
        const float cm = -__fdiv_rn(__fmul_rn(sum_slots<W>(slots, lane), r), (float)N);
        T *dx = static_cast<T *>(p.dx) + row * (int64_t)N;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int j = t + i * TPR;
            if (j < N) {
                const float xh = __fmul_rn(xv[i], r);
                float d = __fmul_rn(__fmaf_rn(xh, cm, __fmul_rn(dv[i], wf[i])), r);
                if constexpr (FUSED) {
                    if (has_dres) d = __fadd_rn(d, rv[i]);
                }
                store_elem(dx, j, d);
                acc[i] = __fmaf_rn(dv[i], xh, acc[i]);
            }
        }
    }
    if (failed) {
        // the last copy into each stage has landed (or its wait gives up
        // again) before the CTA ends
        for (int s2 = 0; s2 < ns && s2 < iters; ++s2) {
            const int64_t kl = s2 + (iters - 1 - s2) / ns * ns;
            mbar_wait(&full[s2], (uint32_t)((kl / ns) & 1), kWaitLimit);
        }
        if (p.status) *p.status = kStatusWaitTimeout;
    }
    if (t == 0) cp_async_wait_all();
    pdl_trigger();  // the finalizer waits for the whole grid before it reads
    if (!has_w) return;
    float *wsrow = p.ws + unit * (int64_t)N;
#pragma unroll
    for (int i = 0; i < K; ++i) {
        const int j = t + i * TPR;
        if (j < N) wsrow[j] = acc[i];
    }
}

// Generic LayerNorm backward, the same scheme: per row the pair (sum g,
// sum g (x - mean)), then dx; the partial row ws[cta, 0..2N) holds dgamma
// and dbeta, updated one column a thread. Each row is read three times
// (the sums, the dgamma and dbeta update, dx). Where the host gave a row
// cache, the first read keeps x and dy in shared memory (at x's address
// mod 16, so chunks stay aligned) and the other two read them there, the
// update after the reduction's barrier; otherwise they re-read global
// memory (L1/L2) and the update comes before the barrier, since dx may
// overwrite dy. Both variants are held to the registers of five CTAs an
// SM, the residency the grid is sized for.
template <typename T, typename TW, bool FUSED, bool CACHE>
__global__ void __launch_bounds__(256, 5) layernorm_bwd_generic(const BwdParams p) {
    __shared__ float2 red[32];
    extern __shared__ uint4 gen_smem[];
    pdl_wait();
    constexpr int E = Elem<T>::E;
    constexpr int NP = Elem<T>::NP;
    const int N = p.N;
    const TW *w = reinterpret_cast<const TW *>(p.w);
    float *wsrow = p.ws ? p.ws + (int64_t)blockIdx.x * 2 * N : nullptr;
    const bool has_dres = FUSED && p.dres != nullptr;
    const uint32_t a16 = addr_mod16(p.x);
    const bool vdy = addr_mod16(p.dy) == a16, vdx = addr_mod16(p.dx) == a16;
    const bool vdr = has_dres && addr_mod16(p.dres) == a16;
    constexpr bool cache = CACHE;
    const int64_t slot = generic_bwd_cache_slot(N, (int)sizeof(T));
    bool first = true;
    for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x) {
        const T *x = reinterpret_cast<const T *>(p.x) + row * N;
        const T *dy = reinterpret_cast<const T *>(p.dy) + row * N;
        const T *dr = reinterpret_cast<const T *>(p.dres) + row * N;
        T *dx = reinterpret_cast<T *>(p.dx) + row * N;
        const float r = p.rstd[row];
        const float nmu = -p.mean[row];
        const RowSplit sp = row_split(x, N, true);
        T *xs = reinterpret_cast<T *>(reinterpret_cast<char *>(gen_smem) + addr_mod16(x));
        T *ds = reinterpret_cast<T *>(reinterpret_cast<char *>(gen_smem) + slot + addr_mod16(x));
        const T *xr = cache ? static_cast<const T *>(xs) : x;
        const T *dyr = cache ? static_cast<const T *>(ds) : dy;
        const bool vdyr = cache || vdy;
        auto gof = [&](float dyj, float wj) { return w ? __fmul_rn(dyj, __fadd_rn(p.offset, wj)) : dyj; };
        float2 part = make_float2(0.f, 0.f);
        auto sums = [&](float g, float xj) {
            part.x = __fadd_rn(part.x, g);
            part.y = __fmaf_rn(g, __fadd_rn(xj, nmu), part.y);
        };
        row_visit<E>(
            sp, N,
            [&](int j) {
                const float dyj = load_elem(dy, j), xj = load_elem(x, j);
                if (cache) {
                    store_elem(xs, j, xj);
                    store_elem(ds, j, dyj);
                }
                sums(gof(dyj, w ? load_w(w, j) : 0.f), xj);
            },
            [&](int j0) {
                float2 dv[NP], xv[NP], wv[NP];
                load_chunk_at(dy, j0, vdy, dv);
                load_chunk_at(x, j0, true, xv);
                if (w) w_chunk_at<T, TW>(w, j0, wv);
                if (cache) {
                    store_chunk_at(xs, j0, true, xv);
                    store_chunk_at(ds, j0, true, dv);
                }
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                    sums(gof(dv[q].x, w ? wv[q].x : 0.f), xv[q].x);
                    sums(gof(dv[q].y, w ? wv[q].y : 0.f), xv[q].y);
                }
            });
        // the dgamma and dbeta partials, one column a thread (coalesced)
        auto param_update = [&]() {
            for (int j = threadIdx.x; j < N; j += blockDim.x) {
                const float dyj = load_elem(dyr, j), xh = __fmul_rn(__fadd_rn(load_elem(xr, j), nmu), r);
                wsrow[j] = first ? __fmul_rn(dyj, xh) : __fmaf_rn(dyj, xh, wsrow[j]);
                wsrow[N + j] = first ? dyj : __fadd_rn(wsrow[N + j], dyj);
            }
        };
        if (wsrow && !cache) param_update();
        const float2 s = cta_allreduce2(part, red);
        if (wsrow && cache) param_update();
        const float cm = -__fdiv_rn(__fmul_rn(s.y, r), (float)N);
        const float nmg = -__fdiv_rn(s.x, (float)N);
        // dx of a column
        auto out = [&](float dyj, float xj, float wj, float drj) {
            const float xh = __fmul_rn(__fadd_rn(xj, nmu), r);
            float d = __fmul_rn(__fmaf_rn(xh, cm, __fadd_rn(gof(dyj, wj), nmg)), r);
            if (has_dres) d = __fadd_rn(d, drj);
            return d;
        };
        row_visit<E>(
            sp, N,
            [&](int j) {
                store_elem(dx, j, out(load_elem(dyr, j), load_elem(xr, j), w ? load_w(w, j) : 0.f,
                                      has_dres ? load_elem(dr, j) : 0.f));
            },
            [&](int j0) {
                float2 dv[NP], xv[NP], wv[NP], rv[NP];
                load_chunk_at(dyr, j0, vdyr, dv);
                load_chunk_at(xr, j0, true, xv);
                if (w) w_chunk_at<T, TW>(w, j0, wv);
                if (has_dres) load_chunk_at(dr, j0, vdr, rv);
#pragma unroll
                for (int q = 0; q < NP; ++q)
                    xv[q] = make_float2(out(dv[q].x, xv[q].x, w ? wv[q].x : 0.f, has_dres ? rv[q].x : 0.f),
                                        out(dv[q].y, xv[q].y, w ? wv[q].y : 0.f, has_dres ? rv[q].y : 0.f));
                store_chunk_at(dx, j0, vdx, xv);
            });
        // the next row's first pass overwrites the cache
        if (cache) __syncthreads();
        first = false;
    }
    pdl_trigger();
}

// Dynamic shared memory of a generic backward launch: the two row-cache
// slots where the host asked for the cache (at most 40 KB), else none.
template <typename T>
static int generic_bwd_smem(const BwdParams &p) {
    return p.cache_row ? (int)(2 * generic_bwd_cache_slot(p.N, (int)sizeof(T))) : 0;
}

// Finalizer. When launched as a programmatic dependent of the main kernel
// it starts early and waits here until the main grid has completed and its
// workspace writes are visible; otherwise the wait returns at once.
__device__ __forceinline__ void wait_for_main_grid() { pdl_wait(); }

// Vector finalizer (N % 4 == 0): a CTA owns 32 columns as 8 float4 lanes and
// splits the P partial rows into 32 groups; group q sums rows
// [q P / 32, (q+1) P / 32) in order, then each column adds the 32 group sums
// in order. A few float4 loads per thread keep the L2 round trips short.
// Columns c < split go to out0, the rest to out1 (a NULL output's columns
// are not written); within its half, workspace column c is parameter
// column (c - peel) mod split (rows at a common offset wrap their first
// chunk, peel > 0); N is the workspace's row length.
template <typename T>
__device__ __forceinline__ void store_param(T *out0, T *out1, int split, int peel, int c, float v) {
    T *out = c < split ? out0 : out1;
    int oc = (c < split ? c : c - split) - peel;
    if (oc < 0) oc += split;
    if (out) store_elem(out, oc, v);
}

// KB > 0: a group of at most KB partial rows issues all its loads before
// its adds (one round trip to L2 instead of one a row), at the price of KB
// float4 registers a thread (84 registers at KB = 16: three CTAs an SM);
// KB = 0: one row at a time (32 registers: eight CTAs an SM). The host takes
// the batched kernel where its grid fits one wave of it. Both add the rows
// in the same order, so they give the same bits.
template <typename T, int LANES = 8, int RG = 32, int KB = 16>
__global__ void __launch_bounds__(LANES *RG) rmsnorm_dw_finalize4(const float *ws, int parts, int N, T *dw, T *dw1,
                                                                  int split, int peel) {
    constexpr int COLS = 4 * LANES;       // columns per CTA
    __shared__ float part[RG][COLS + 1];
    wait_for_main_grid();
    pdl_trigger();
    const int lane = threadIdx.x % LANES;  // float4 column within the CTA's columns
    const int rg = threadIdx.x / LANES;    // row group
    const int col = blockIdx.x * COLS + lane * 4;
    const int p0 = (int)((int64_t)parts * rg / RG);
    const int p1 = (int)((int64_t)parts * (rg + 1) / RG);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < N) {
        const float4 *src = reinterpret_cast<const float4 *>(ws + col);
        const int64_t stride = N / 4;
        auto add = [&](const float4 &v) {
            s.x = __fadd_rn(s.x, v.x);
            s.y = __fadd_rn(s.y, v.y);
            s.z = __fadd_rn(s.z, v.z);
            s.w = __fadd_rn(s.w, v.w);
        };
        // up to KB rows a group (P <= RG * KB): every load in flight at
        // once, one round trip to L2, then the adds in row order
        if (KB > 0 && p1 - p0 <= KB) {
            float4 v[KB > 0 ? KB : 1];
#pragma unroll
            for (int i = 0; i < KB; ++i)
                if (p0 + i < p1) v[i] = src[(int64_t)(p0 + i) * stride];
#pragma unroll
            for (int i = 0; i < KB; ++i)
                if (p0 + i < p1) add(v[i]);
        } else {
#pragma unroll 4
            for (int q = p0; q < p1; ++q) add(src[(int64_t)q * stride]);
        }
    }
    part[rg][lane * 4 + 0] = s.x;
    part[rg][lane * 4 + 1] = s.y;
    part[rg][lane * 4 + 2] = s.z;
    part[rg][lane * 4 + 3] = s.w;
    __syncthreads();
    if (threadIdx.x < COLS) {
        const int c = blockIdx.x * COLS + threadIdx.x;
        if (c < N) {
            float tot = part[0][threadIdx.x];
#pragma unroll
            for (int g = 1; g < RG; ++g) tot = __fadd_rn(tot, part[g][threadIdx.x]);
            store_param(dw, dw1, split, peel, c, tot);
        }
    }
}

// Scalar finalizer for any N: 32 columns per CTA, 8 groups of partial rows,
// same fixed order rules.
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_dw_finalize(const float *ws, int parts, int N, T *dw, T *dw1,
                                                           int split, int peel) {
    constexpr int RG = 8;
    __shared__ float part[RG][32];
    wait_for_main_grid();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int rg = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + lane;
    const int p0 = (int)((int64_t)parts * rg / RG);
    const int p1 = (int)((int64_t)parts * (rg + 1) / RG);
    float s = 0.f;
    if (col < N) {
        const float *src = ws + col;
#pragma unroll 8
        for (int q = p0; q < p1; ++q) s = __fadd_rn(s, src[(int64_t)q * N]);
    }
    part[rg][lane] = s;
    __syncthreads();
    if (rg == 0 && col < N) {
        float tot = part[0][lane];
#pragma unroll
        for (int g = 1; g < RG; ++g) tot = __fadd_rn(tot, part[g][lane]);
        store_param(dw, dw1, split, peel, col, tot);
    }
}

// ------------------------------------------------------------- dispatch --


template <typename T, typename TW, int TPR, int V, int TEAMS, int D, int CS, bool PACKED, bool PEEL>
static int bwd_launch_vec(bool fused, const BwdParams &p, int grid, int smem, cudaStream_t s) {
    LaunchCfg lc((unsigned)grid, TPR * TEAMS, (size_t)smem, s, CS > 1 ? CS : 0);
    return fused
               ? (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, PACKED, true, PEEL>, p)
               : (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, PACKED, false, PEEL>, p);
}

// A weight type other than the activations' is compiled for the default
// plans (and the generic one) only; alternatives are for tuning. The PEEL
// instantiations (rows at a common offset, weight in the activations'
// type) exist for the default vectorised plans only.
template <typename T, typename TW, int PATH, int CMIN, bool PEEL = false>
constexpr bool bwd_instantiated() {
    if constexpr (PEEL)
        return std::is_same<T, TW>::value && CMIN > 0 && !generic_path(PATH);
    else
        return std::is_same<T, TW>::value || generic_path(PATH) || CMIN > 0;
}

// Streamed generic kernel: launched as a cluster of one CTA (its bulk
// copies name a shared::cluster destination) with the stages' dynamic
// shared memory.
template <typename T, typename TW, int TPR, int K, int SMAX>
static int bwd_launch_stream(bool fused, const BwdParams &p, int grid, int smem, cudaStream_t s) {
    const void *k = fused ? (const void *)rmsnorm_bwd_stream<T, TW, TPR, K, SMAX, true>
                          : (const void *)rmsnorm_bwd_stream<T, TW, TPR, K, SMAX, false>;
    const int e = allow_staged_smem(k);
    if (e != 0) return e;
    LaunchCfg lc((unsigned)grid, TPR, (size_t)smem, s, 1);
    return fused ? (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_bwd_stream<T, TW, TPR, K, SMAX, true>, p)
                 : (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_bwd_stream<T, TW, TPR, K, SMAX, false>, p);
}

// Staged kernel: launched as a cluster of CS CTAs (of one where a CTA
// holds the whole row; its bulk copies name a shared::cluster destination)
// with the stages' dynamic shared memory.
template <typename T, typename TW, int TPR, int V, int S, int CS, bool HOLD, bool PACKED, bool PEEL>
static int bwd_launch_staged(bool fused, const BwdParams &p, int grid, int smem, cudaStream_t s) {
    const void *k = fused ? (const void *)rmsnorm_bwd_staged<T, TW, TPR, V, S, CS, true, HOLD, PACKED, PEEL>
                          : (const void *)rmsnorm_bwd_staged<T, TW, TPR, V, S, CS, false, HOLD, PACKED, PEEL>;
    const int e = allow_staged_smem(k);
    if (e != 0) return e;
    // a cluster of CS CTAs (of one where a CTA holds the whole row: its bulk
    // copies name a shared::cluster destination)
    LaunchCfg lc((unsigned)grid, TPR, (size_t)smem, s, CS);
    return fused
               ? (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_bwd_staged<T, TW, TPR, V, S, CS, true, HOLD, PACKED, PEEL>, p)
               : (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_bwd_staged<T, TW, TPR, V, S, CS, false, HOLD, PACKED, PEEL>, p);
}

// Kernel kind of an (activation, weight) type pair, as the host numbers it:
// 0 fp32, 1 bf16, 2 fp16, 3 bf16 with an fp32 weight, 4 fp16 with one.
template <typename T, typename TW>
constexpr int kernel_kind() {
    return std::is_same<T, float>::value ? 0
           : std::is_same<T, TW>::value   ? (std::is_same<T, __nv_bfloat16>::value ? 1 : 2)
                                          : (std::is_same<T, __nv_bfloat16>::value ? 3 : 4);
}

template <typename T, typename TW, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int D, int CS, int CMIN>
static int bwd_launch_entry(bool fused, bool packed, const BwdParams &p, int grid, int smem, cudaStream_t s) {
    if constexpr (OP != OP_BWD || !bwd_instantiated<T, TW, PATH, CMIN, PEEL>()) {
        return (int)cudaErrorInvalidValue;
    } else if constexpr (PATH == PATH_GENERIC) {
        LaunchCfg lc((unsigned)grid, 256, 0, s);
        return fused ? (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_bwd_generic<T, TW, true>, p)
                     : (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_bwd_generic<T, TW, false>, p);
    } else if constexpr (PATH == PATH_STREAM) {
        return bwd_launch_stream<T, TW, TPR, V, D>(fused, p, grid, smem, s);
    } else if constexpr (PATH == PATH_VECTOR) {
        return packed ? bwd_launch_vec<T, TW, TPR, V, TEAMS, D, CS, true, PEEL>(fused, p, grid, smem, s)
                      : bwd_launch_vec<T, TW, TPR, V, TEAMS, D, CS, false, PEEL>(fused, p, grid, smem, s);
    } else if constexpr (staged_plan(PATH, TEAMS, CS)) {
        if constexpr (staged_scalar_variant(kernel_kind<T, TW>(), CMIN)) {
            if (!packed)
                return bwd_launch_staged<T, TW, TPR, V, D, CS, PATH == PATH_STAGED, false, PEEL>(fused, p, grid, smem,
                                                                                                 s);
        } else if (!packed) {
            return (int)cudaErrorInvalidValue;
        }
        return bwd_launch_staged<T, TW, TPR, V, D, CS, PATH == PATH_STAGED, true, PEEL>(fused, p, grid, smem, s);
    } else {
        return (int)cudaErrorInvalidValue;
    }
}

template <typename T, typename TW, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int D, int CS, int CMIN>
static const void *bwd_ptr_entry(bool fused, bool packed) {
    if constexpr (OP != OP_BWD || !bwd_instantiated<T, TW, PATH, CMIN, PEEL>()) {
        return nullptr;
    } else if constexpr (PATH == PATH_GENERIC) {
        return fused ? (const void *)rmsnorm_bwd_generic<T, TW, true> : (const void *)rmsnorm_bwd_generic<T, TW, false>;
    } else if constexpr (PATH == PATH_STREAM) {
        return fused ? (const void *)rmsnorm_bwd_stream<T, TW, TPR, V, D, true>
                     : (const void *)rmsnorm_bwd_stream<T, TW, TPR, V, D, false>;
    } else if constexpr (PATH == PATH_VECTOR) {
        if (packed)
            return fused ? (const void *)rmsnorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, true, true, PEEL>
                         : (const void *)rmsnorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, true, false, PEEL>;
        return fused ? (const void *)rmsnorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, false, true, PEEL>
                     : (const void *)rmsnorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, false, false, PEEL>;
    } else if constexpr (staged_plan(PATH, TEAMS, CS)) {
        constexpr bool HOLD = PATH == PATH_STAGED;
        // the scalar variant where it is compiled (nullptr where it is not)
        if constexpr (staged_scalar_variant(kernel_kind<T, TW>(), CMIN)) {
            if (!packed)
                return fused ? (const void *)rmsnorm_bwd_staged<T, TW, TPR, V, D, CS, true, HOLD, false, PEEL>
                             : (const void *)rmsnorm_bwd_staged<T, TW, TPR, V, D, CS, false, HOLD, false, PEEL>;
        } else if (!packed) {
            return nullptr;
        }
        return fused ? (const void *)rmsnorm_bwd_staged<T, TW, TPR, V, D, CS, true, HOLD, true, PEEL>
                     : (const void *)rmsnorm_bwd_staged<T, TW, TPR, V, D, CS, false, HOLD, true, PEEL>;
    } else {
        return nullptr;
    }
}

template <typename T, typename TW, bool PEEL = false>
static int bwd_launch_t(int plan_id, bool fused, bool packed, const BwdParams &p, int grid, int smem,
                        void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (plan_id) {
#define RMSN_BWD_CASE(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id:                                                                    \
        return bwd_launch_entry<T, TW, PEEL, op, path, tpr, v, teams, depth, cs, cmin>(fused, packed, p, grid, smem, s);
        RMSNORM_PLAN_TABLE(RMSN_BWD_CASE)
#undef RMSN_BWD_CASE
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <typename T, typename TW, bool PEEL = false>
static const void *bwd_ptr_t(int plan_id, bool fused, bool packed) {
    switch (plan_id) {
#define RMSN_BWD_PTR(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id: return bwd_ptr_entry<T, TW, PEEL, op, path, tpr, v, teams, depth, cs, cmin>(fused, packed);
        RMSNORM_PLAN_TABLE(RMSN_BWD_PTR)
#undef RMSN_BWD_PTR
    default:
        return nullptr;
    }
}

// The finalizer is launched as a programmatic dependent of the main kernel
// (its launch overlaps the main kernel's tail) unless `serial` asks for a
// plain launch (when the caller records an event between the two). `sms`:
// the device's SM count, which picks the batched vector finalizer where its
// grid fits one wave (three of its CTAs an SM).
template <typename T>
static int finalize_launch_t(const float *ws, int parts, int N, void *dw, void *dw1, int split, int peel,
                             void *stream, bool serial, int sms) {
    constexpr int kLanes = 8, kGroups = 32;  // vector finalizer: 4 * kLanes columns a CTA
    constexpr int kBatchPerSm = 3;           // resident CTAs an SM of the batched finalizer
    // float4 columns need every group of 4 on one side of the split
    const bool vec = N % 4 == 0 && split % 4 == 0;
    const int vgrid = (N + 4 * kLanes - 1) / (4 * kLanes);
    const bool batch = vgrid <= kBatchPerSm * sms;
    LaunchCfg lc(vec ? (unsigned)((N + 4 * kLanes - 1) / (4 * kLanes)) : (unsigned)((N + 31) / 32),
                 vec ? kLanes * kGroups : 256, 0, static_cast<cudaStream_t>(stream), 0, !serial);
    T *out = static_cast<T *>(dw);
    T *out1 = static_cast<T *>(dw1);
    cudaError_t e = !vec    ? cudaLaunchKernelEx(&lc.cfg, rmsnorm_dw_finalize<T>, ws, parts, N, out, out1, split, peel)
                    : batch ? cudaLaunchKernelEx(&lc.cfg, rmsnorm_dw_finalize4<T, kLanes, kGroups, 16>, ws, parts, N,
                                                 out, out1, split, peel)
                            : cudaLaunchKernelEx(&lc.cfg, rmsnorm_dw_finalize4<T, kLanes, kGroups, 0>, ws, parts, N,
                                                 out, out1, split, peel);
    return (int)e;
}

// ------------------------------------------------- LayerNorm dispatch --

template <typename T, typename TW, int TPR, int V, int TEAMS, int D, int CS, bool PEEL>
static int ln_bwd_launch_vec(bool fused, const BwdParams &p, int grid, int smem, cudaStream_t s) {
    LaunchCfg lc((unsigned)grid, TPR * TEAMS, (size_t)smem, s, CS > 1 ? CS : 0);
    return fused ? (int)cudaLaunchKernelEx(&lc.cfg, layernorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, true, PEEL>, p)
                 : (int)cudaLaunchKernelEx(&lc.cfg, layernorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, false, PEEL>, p);
}

template <typename T, typename TW, int TPR, int V, int S, int CS, bool HOLD, bool PEEL>
static int ln_bwd_launch_staged(bool fused, const BwdParams &p, int grid, int smem, cudaStream_t s) {
    const void *k = fused ? (const void *)layernorm_bwd_staged<T, TW, TPR, V, S, CS, true, HOLD, PEEL>
                          : (const void *)layernorm_bwd_staged<T, TW, TPR, V, S, CS, false, HOLD, PEEL>;
    const int e = allow_staged_smem(k);
    if (e != 0) return e;
    LaunchCfg lc((unsigned)grid, TPR, (size_t)smem, s, CS);
    return fused ? (int)cudaLaunchKernelEx(&lc.cfg, layernorm_bwd_staged<T, TW, TPR, V, S, CS, true, HOLD, PEEL>, p)
                 : (int)cudaLaunchKernelEx(&lc.cfg, layernorm_bwd_staged<T, TW, TPR, V, S, CS, false, HOLD, PEEL>, p);
}

// An fp32 gamma beside 16-bit activations is compiled for the default
// plans and the generic one only; the PEEL instantiations for the default
// vectorised plans with gamma in the activations' type.
template <typename T, typename TW, int PATH, int CMIN, bool PEEL>
constexpr bool ln_bwd_instantiated() {
    if constexpr (PEEL)
        return std::is_same<T, TW>::value && CMIN > 0 && !generic_path(PATH);
    else
        return std::is_same<T, TW>::value || PATH == PATH_GENERIC || CMIN > 0;
}

template <typename T, typename TW, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int D, int CS, int CMIN>
static int ln_bwd_launch_entry(bool fused, const BwdParams &p, int grid, int smem, cudaStream_t s) {
    if constexpr (OP != OP_LN_BWD || !ln_bwd_instantiated<T, TW, PATH, CMIN, PEEL>()) {
        return (int)cudaErrorInvalidValue;
    } else if constexpr (PATH == PATH_GENERIC) {
        const int gs = generic_bwd_smem<T>(p);
        LaunchCfg lc((unsigned)grid, 256, (size_t)gs, s);
        if (fused)
            return gs ? (int)cudaLaunchKernelEx(&lc.cfg, layernorm_bwd_generic<T, TW, true, true>, p)
                      : (int)cudaLaunchKernelEx(&lc.cfg, layernorm_bwd_generic<T, TW, true, false>, p);
        return gs ? (int)cudaLaunchKernelEx(&lc.cfg, layernorm_bwd_generic<T, TW, false, true>, p)
                  : (int)cudaLaunchKernelEx(&lc.cfg, layernorm_bwd_generic<T, TW, false, false>, p);
    } else if constexpr (PATH == PATH_VECTOR) {
        return ln_bwd_launch_vec<T, TW, TPR, V, TEAMS, D, CS, PEEL>(fused, p, grid, smem, s);
    } else if constexpr (staged_plan(PATH, TEAMS, CS)) {
        return ln_bwd_launch_staged<T, TW, TPR, V, D, CS, PATH == PATH_STAGED, PEEL>(fused, p, grid, smem, s);
    } else {
        return (int)cudaErrorInvalidValue;
    }
}

template <typename T, typename TW, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int D, int CS, int CMIN>
static const void *ln_bwd_ptr_entry(bool fused) {
    if constexpr (OP != OP_LN_BWD || !ln_bwd_instantiated<T, TW, PATH, CMIN, PEEL>()) {
        return nullptr;
    } else if constexpr (PATH == PATH_GENERIC) {
        return fused ? (const void *)layernorm_bwd_generic<T, TW, true, false>
                     : (const void *)layernorm_bwd_generic<T, TW, false, false>;
    } else if constexpr (PATH == PATH_VECTOR) {
        return fused ? (const void *)layernorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, true, PEEL>
                     : (const void *)layernorm_bwd_vector<T, TW, TPR, V, TEAMS, D, CS, false, PEEL>;
    } else if constexpr (staged_plan(PATH, TEAMS, CS)) {
        return fused ? (const void *)layernorm_bwd_staged<T, TW, TPR, V, D, CS, true, PATH == PATH_STAGED, PEEL>
                     : (const void *)layernorm_bwd_staged<T, TW, TPR, V, D, CS, false, PATH == PATH_STAGED, PEEL>;
    } else {
        return nullptr;
    }
}

// (TW: gamma's type, the activations' or fp32)
template <typename T, typename TW = T, bool PEEL = false>
static int ln_bwd_launch_t(int plan_id, bool fused, const BwdParams &p, int grid, int smem, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (plan_id) {
#define RMSN_LN_BWD_CASE(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id:                                                                       \
        return ln_bwd_launch_entry<T, TW, PEEL, op, path, tpr, v, teams, depth, cs, cmin>(fused, p, grid, smem, s);
        RMSNORM_PLAN_TABLE(RMSN_LN_BWD_CASE)
#undef RMSN_LN_BWD_CASE
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <typename T, typename TW = T, bool PEEL = false>
static const void *ln_bwd_ptr_t(int plan_id, bool fused) {
    switch (plan_id) {
#define RMSN_LN_BWD_PTR(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id: return ln_bwd_ptr_entry<T, TW, PEEL, op, path, tpr, v, teams, depth, cs, cmin>(fused);
        RMSNORM_PLAN_TABLE(RMSN_LN_BWD_PTR)
#undef RMSN_LN_BWD_PTR
    default:
        return nullptr;
    }
}

}  // namespace rmsn
