// fwd_kernels.cuh -- RMSNorm forward kernels (plain and fused residual add,
// bf16/fp16/fp32 or E4M3 output) and the LayerNorm forward.
//
// Vector kernel: a team of TPR threads owns one row; each thread loads V
// 16-byte chunks of it (chunk c = v * TPR + t, so a warp's loads are
// contiguous), keeps them in registers, reduces the sum of squares (warp
// butterfly, then shared memory across the team's warps), and writes
// y = x * rstd * (offset + w) from the same registers, rounded once.
// This is the row-in-registers forward with vector loads and a CTA-level
// reduction of Liger-Kernel PR #1388 (Summary; "_launch_fwd_vector"), with
// the warps per row chosen by N as in the tuned per-hidden-size kernels of
// ROCm/TransformerEngine PR #583 (Description).
//
// Rows wider than 2048 chunks are shared by a thread-block cluster: the
// staged kernel streams each CTA's slice through shared-memory stages on a
// persistent grid of clusters (rows of up to 8192 chunks, every output
// type), the register kernel holds the slices of wider rows.
//
// Generic kernel: one 256-thread CTA per row, the row read twice (the
// second read hits L1/L2), split into an element-wise head, 16-byte chunks
// and an element-wise tail. Serves any N and any element-aligned pointers
// (Liger-Kernel PR #1388, "Behavior when the fast path does not apply":
// irregular or unaligned shapes take scalar paths).
#pragma once

#include "common.cuh"
#include "plans.h"

namespace rmsn {

// Register budget of the vector forward: its CTAs hold a row (or a team's
// rows) in registers only between the loads and the stores, so the number
// of rows in flight per SM, and with it the bandwidth of a short call, is
// the number of resident CTAs. Left to itself the compiler gives the
// four-chunk plans 69-72 registers a thread: three 256-thread CTAs an SM
// (one of 512 threads). The bound below asks for the registers of
// RMSNORM_FWD_OCC 256-thread CTAs an SM: at 5, 48 registers (a few bytes
// of spill in the four-chunk plans) and two 512-thread CTAs an SM.
// Measured on bf16 rows, sustained calls: 4096x7168 27.3 -> 23.0 us,
// 16384x8192 93.5 -> 82.6 us, 4096x16384 71.0 -> 47.9 us (4 a little
// slower at 4096x7168, 24.5 us; the same elsewhere).
#ifndef RMSNORM_FWD_OCC
#define RMSNORM_FWD_OCC 5
#endif
template <int THREADS>
constexpr int fwd_min_blocks() {
    return THREADS >= 1024 || RMSNORM_FWD_OCC * 256 / THREADS < 1 ? 1 : RMSNORM_FWD_OCC * 256 / THREADS;
}

// A chunk of fp32 y (four values) stored in the narrower output type of Q
// (bf16 or fp16, rounded to nearest even): 8 bytes at chunk index i of y.
template <int Q>
__device__ __forceinline__ void st_narrow_chunk(void *y, int64_t i, const float2 (&a)[2]) {
    const uint2 u = Q == QOUT_BF16 ? make_uint2(f2_to_bf16x2(a[0]), f2_to_bf16x2(a[1]))
                                   : make_uint2(f2_to_f16x2(a[0]), f2_to_f16x2(a[1]));
    reinterpret_cast<uint2 *>(y)[i] = u;
}

// The row's chunks into registers; with FUSED, h = R(x + residual) is
// formed in place and stored to residual_out. Chunks past the row are zero.
// Rows are C chunks apart. Rows at a common offset (p.peel) wrap chunk 0:
// its thread (t = 0 of the slice holding chunk 0, always chunk slot v = 0)
// loads the second aligned block beside its other loads and merges the two
// once every load is in flight, so no warp waits on a load before issuing
// the rest.
template <typename T, int TPR, int V, bool FUSED, bool PEEL>
__device__ __forceinline__ void fwd_load_row(const FwdParams &p, int64_t base, int C, int cbase, int t, int cend,
                                             bool valid, uint4 (&xv)[V]) {
    using Pk = Pair<true>;
    constexpr int NP = Elem<T>::NP;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const int peel = peel_of<PEEL>(p);
    const bool wrap0 = peel != 0 && cbase + t == 0;
    const uint4 *x4 = reinterpret_cast<const uint4 *>(p.x) + base;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = cbase + v * TPR + t;
        xv[v] = c < cend ? ld_stream(x4 + c) : zero;
    }
    const uint4 xt = wrap0 ? ld_stream(x4 + C) : zero;
    if constexpr (!FUSED) {
        if (wrap0) xv[0] = wrap_chunk<T>(xv[0], xt, peel);
    } else {
        // h = R(x + residual). For bf16 inputs the fp32 sum is exact unless
        // the exponents differ by more than 15, and then both it and the
        // exact sum round to the larger operand: one rounding to bf16 gives
        // the correctly rounded sum. For fp32 the add is the rounding.
        uint4 rv[V];
        const uint4 *r4 = reinterpret_cast<const uint4 *>(p.residual) + base;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = cbase + v * TPR + t;
            rv[v] = c < cend ? ld_stream(r4 + c) : zero;
        }
        const uint4 rt = wrap0 ? ld_stream(r4 + C) : zero;
        if (wrap0) {
            xv[0] = wrap_chunk<T>(xv[0], xt, peel);
            rv[0] = wrap_chunk<T>(rv[0], rt, peel);
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float2 a[NP], b[NP];
            unpack<T>(xv[v], a);
            unpack<T>(rv[v], b);
#pragma unroll
            for (int k = 0; k < NP; ++k) a[k] = Pk::add(a[k], b[k]);
            xv[v] = pack<T>(a);
            const int c = cbase + v * TPR + t;
            if (valid && c < cend)
                st_row_chunk<T>(reinterpret_cast<uint4 *>(p.residual_out) + base, c, C, peel, v == 0 && wrap0, xv[v]);
        }
    }
}

// CS > 1: the CTAs of a cluster share one row; CTA rank r holds chunks
// [r TPR V, (r+1) TPR V) and the sum of squares meets in distributed shared
// memory (wide rows whose chunks exceed one CTA's registers).
//
// Q selects the output: QOUT_NONE stores y in T; the E4M3 modes store
// E4M3(y * s), one byte per element, with s the given per-tensor scale or
// 448 / max|y| of the row (a second, max-combining row reduction); the
// narrow modes (fp32 activations) store y in bf16 or fp16, 8 bytes a chunk.
template <typename T, typename TW, int TPR, int V, int TEAMS, int CS, bool FUSED, int Q = QOUT_NONE, bool PEEL = false>
__global__ void __launch_bounds__(TPR *TEAMS, !fp8_out(Q) ? fwd_min_blocks<TPR * TEAMS>()
                                                          : (1280 / (TPR * TEAMS) > 0 ? 1280 / (TPR * TEAMS) : 1))
    rmsnorm_fwd_vector(const FwdParams p) {
    static_assert(CS == 1 || TEAMS == 1, "a cluster row uses one team per CTA");
    static_assert(!narrow_out(Q) || std::is_same<T, float>::value, "a narrower output for fp32 activations");
    using Pk = Pair<true>;
    constexpr int NP = Elem<T>::NP;
    constexpr int W = TPR > 32 ? TPR / 32 : 1;
    __shared__ float red[TEAMS][W * CS];
    __shared__ float redm[fp8_out(Q) ? TEAMS : 1][W * CS];  // the max reduction's slots
    // the kernel before it has completed; the next may launch once every
    // CTA of this one has started (no CTA of this grid is then waiting)
    pdl_wait();
    pdl_trigger();

    const int team = threadIdx.x / TPR;
    const int t = threadIdx.x % TPR;
    uint32_t rank = 0;
    int64_t row;
    if constexpr (CS > 1) {
        rank = cluster_ctarank();
        row = cluster_id_x();
    } else {
        row = (int64_t)blockIdx.x * TEAMS + team;
    }
    const bool valid = row < p.M;
    const int64_t rr = valid ? row : p.M - 1;  // keep every thread in the reductions
    const int C = p.N / Elem<T>::E;
    const int64_t base = rr * C;
    // a cluster row: equal slices of ceil(C / CS) chunks, the last shorter
    const int cslice = (C + CS - 1) / CS;
    const int cbase = (int)rank * cslice;  // first chunk of this CTA's slice
    const int cend = cbase + cslice < C ? cbase + cslice : C;

    uint4 xv[V];
    fwd_load_row<T, TPR, V, FUSED, PEEL>(p, base, C, cbase, t, cend, valid, xv);

    float2 ss = make_float2(0.f, 0.f);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        float2 a[NP];
        unpack<T>(xv[v], a);
#pragma unroll
        for (int k = 0; k < NP; ++k) ss = Pk::fma(a[k], a[k], ss);
    }
    float s;
    if constexpr (CS > 1) {
        cluster_sync();  // every CTA of the cluster runs before any distributed-shared store
        s = cluster_allreduce<TPR, CS>(__fadd_rn(ss.x, ss.y), &red[0][0], t, rank);
    } else {
        s = team_allreduce<TPR>(__fadd_rn(ss.x, ss.y), &red[team][0], t);
    }
    const float rstd = rsqrtf(__fadd_rn(__fdiv_rn(s, (float)p.N), p.eps));
    if (valid && t == 0 && rank == 0) p.rstd[row] = rstd;

    const float2 r2 = make_float2(rstd, rstd);
    const float2 o2 = make_float2(p.offset, p.offset);
    const bool has_w = p.w != nullptr;  // no weight: non-affine, factor 1
    if constexpr (!fp8_out(Q)) {
        if (!valid) return;
        // slot 0 of this thread is the row's wrapped chunk (the weight
        // shares the rows' offset)
        const int peel = peel_of<PEEL>(p);
        const bool e0 = peel != 0 && cbase + t == 0;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = cbase + v * TPR + t;
            if (c < cend) {
                float2 a[NP];
                unpack<T>(xv[v], a);
                if (has_w) {
                    float2 wv[NP];
                    load_w_chunk_row<T, TW>(p.w, c, C, peel, v == 0 && e0, wv);
#pragma unroll
                    for (int k = 0; k < NP; ++k) a[k] = Pk::mul(Pk::mul(a[k], r2), Pk::add(o2, wv[k]));
                } else {
#pragma unroll
                    for (int k = 0; k < NP; ++k) a[k] = Pk::mul(a[k], r2);
                }
                if constexpr (narrow_out(Q))
                    st_narrow_chunk<Q>(p.y, base + c, a);  // (rows on 16-byte boundaries: no peel)
                else
                    st_row_chunk<T>(reinterpret_cast<uint4 *>(p.y) + base, c, C, peel, v == 0 && e0, pack<T>(a));
            }
        }
    } else {
        // y' = (h (offset + w)) rstd in fp32, kept in registers until the
        // scale is known. Rounding a product with rstd > 0 is monotone, so
        // the row's max |y'| is exactly rstd max_j |h_j (offset + w_j)|: the
        // form every E4M3 kernel takes it in (here after the products, in
        // the staged and generic kernels in their first pass)
        float2 yv[V][NP];
        float m = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = cbase + v * TPR + t;
            unpack<T>(xv[v], yv[v]);  // zero chunks beyond the row give y = 0
            float2 wv[NP];
            if (has_w && c < cend) {
                load_w_chunk<T, TW>(p.w, c, wv);
            } else {
#pragma unroll
                for (int k = 0; k < NP; ++k) wv[k] = make_float2(1.f - p.offset, 1.f - p.offset);
            }
#pragma unroll
            for (int k = 0; k < NP; ++k) {
                const float2 hg = has_w ? Pk::mul(yv[v][k], Pk::add(o2, wv[k])) : yv[v][k];
                m = fmaxf(m, fmaxf(fabsf(hg.x), fabsf(hg.y)));
                yv[v][k] = Pk::mul(hg, r2);
            }
        }
        float mrow = 0.f;
        if (Q == QOUT_FP8_ROW || p.qamax != nullptr) {  // uniform over the grid
            if constexpr (CS > 1) {
                mrow = cluster_allreduce<TPR, CS, OpMax>(m, &redm[0][0], t, rank);
            } else {
                mrow = team_allreduce<TPR, OpMax>(m, &redm[team][0], t);
            }
        }
        // (fmaxf drops a NaN product: a zero row with eps = 0 reports 0)
        const float amax = fmaxf(0.f, __fmul_rn(rstd, mrow));
        if (!valid) return;
        float sc;
        if constexpr (Q == QOUT_FP8_ROW) {
            sc = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
            if (t == 0 && rank == 0) p.qscale_inv[row] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        } else {
            sc = __ldg(p.qscale);
            if (row == 0 && t == 0 && rank == 0 && p.qscale_inv) p.qscale_inv[0] = __fdiv_rn(1.f, sc);
        }
        if (p.qamax != nullptr && t == 0 && rank == 0) atomicMax(p.qamax, __float_as_uint(amax));
        const float2 s2 = make_float2(sc, sc);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = cbase + v * TPR + t;
            if (c < cend) {
                float2 q[NP];
#pragma unroll
                for (int k = 0; k < NP; ++k) q[k] = Pk::mul(yv[v][k], s2);
                if constexpr (NP == 4) {
                    __stcs(reinterpret_cast<uint2 *>(p.y) + base + c, make_uint2(e4m3x4(q[0], q[1]), e4m3x4(q[2], q[3])));
                } else {
                    __stcs(reinterpret_cast<unsigned int *>(p.y) + base + c, e4m3x4(q[0], q[1]));
                }
            }
        }
    }
}

// Generic forward: one 256-thread CTA per row, any N and alignment; the
// output pass reads the row again (from L1/L2). Rows are split into an
// element-wise head, 16-byte chunks and an element-wise tail.
template <typename T, typename TW, bool FUSED, int Q = QOUT_NONE>
__global__ void __launch_bounds__(256) rmsnorm_fwd_generic(const FwdParams p) {
    __shared__ float red[32];
    __shared__ float2 red2[fp8_out(Q) ? 32 : 1];  // E4M3: (sum of squares, max) slots
    pdl_wait();
    pdl_trigger();
    constexpr int NP = Elem<T>::NP;
    const int64_t row = blockIdx.x;
    const int N = p.N;
    const T *x = reinterpret_cast<const T *>(p.x) + row * N;
    const T *res = reinterpret_cast<const T *>(p.residual) + row * N;
    T *hout = reinterpret_cast<T *>(p.residual_out) + row * N;
    const TW *w = reinterpret_cast<const TW *>(p.w);
    T *y = reinterpret_cast<T *>(p.y) + row * N;

    // the row splits by x's address (the E4M3 output, one byte an element,
    // stays element by element); the other arrays take 16-byte accesses
    // where they share x's address mod 16
    const uint32_t a16 = addr_mod16(p.x);
    const bool vy = addr_mod16(p.y) == a16;
    const bool vr = FUSED && addr_mod16(p.residual) == a16;
    const bool vh = FUSED && addr_mod16(p.residual_out) == a16;
    const RowSplit sp = row_split(x, N, Q == QOUT_NONE);  // (other outputs: element by element)

    float ss = 0.f;
    // E4M3: max |h (offset + w)|, whose product with rstd is the row's max |y|
    float m = 0.f;
    auto hg_max = [&](float h, int j) {
        if constexpr (fp8_out(Q)) m = fmaxf(m, fabsf(w ? __fmul_rn(h, __fadd_rn(p.offset, load_w(w, j))) : h));
    };
    auto h_elem = [&](int j) {
        float h = load_elem(x, j);
        if constexpr (FUSED) {
            h = round_to(__fadd_rn(h, load_elem(res, j)), x);
            store_elem(hout, j, h);
        }
        return h;
    };
    for (int j = threadIdx.x; j < sp.head; j += blockDim.x) {
        const float h = h_elem(j);
        ss = __fmaf_rn(h, h, ss);
        hg_max(h, j);
    }
    for (int c = threadIdx.x; c < sp.nb; c += blockDim.x) {
        const int64_t j0 = sp.head + (int64_t)c * Elem<T>::E;
        float2 h[NP];
        load_chunk_at(x, j0, true, h);
        if constexpr (FUSED) {
            float2 r[NP];
            load_chunk_at(res, j0, vr, r);
#pragma unroll
            for (int q = 0; q < NP; ++q) h[q] = make_float2(__fadd_rn(h[q].x, r[q].x), __fadd_rn(h[q].y, r[q].y));
            unpack<T>(pack<T>(h), h);  // the stored (rounded) sum is what is normalised
            store_chunk_at(hout, j0, vh, h);
        }
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            ss = __fmaf_rn(h[q].x, h[q].x, ss);
            ss = __fmaf_rn(h[q].y, h[q].y, ss);
        }
        if constexpr (fp8_out(Q)) {
            float2 g[NP];
            if (w) w_chunk_at<T, TW>(w, (int)j0, g);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float gx = w ? __fmul_rn(h[q].x, __fadd_rn(p.offset, g[q].x)) : h[q].x;
                const float gy = w ? __fmul_rn(h[q].y, __fadd_rn(p.offset, g[q].y)) : h[q].y;
                m = fmaxf(m, fmaxf(fabsf(gx), fabsf(gy)));
            }
        }
    }
    for (int j = sp.tail0 + threadIdx.x; j < N; j += blockDim.x) {
        const float h = h_elem(j);
        ss = __fmaf_rn(h, h, ss);
        hg_max(h, j);
    }
    float s, mrow = 0.f;
    if constexpr (fp8_out(Q)) {
        const float2 r = cta_allreduce2<SumMax>(make_float2(ss, m), red2);
        s = r.x;
        mrow = r.y;
    } else {
        s = cta_allreduce(ss, red);
    }
    const float rstd = rsqrtf(__fadd_rn(__fdiv_rn(s, (float)N), p.eps));
    if (threadIdx.x == 0) p.rstd[row] = rstd;
    // The same thread wrote hout[j] above, so it reads its own value.
    auto y_at = [&](int j) {
        const float h = FUSED ? load_elem(static_cast<const T *>(hout), j) : load_elem(x, j);
        if constexpr (fp8_out(Q)) {  // E4M3: y' = (h (offset + w)) rstd, whose max is rstd max |h (offset + w)|
            return __fmul_rn(w ? __fmul_rn(h, __fadd_rn(p.offset, load_w(w, j))) : h, rstd);
        } else {
            const float hr = __fmul_rn(h, rstd);
            return w ? __fmul_rn(hr, __fadd_rn(p.offset, load_w(w, j))) : hr;
        }
    };
    if constexpr (narrow_out(Q)) {
        using TO = typename std::conditional<Q == QOUT_BF16, __nv_bfloat16, __half>::type;
        TO *yo = reinterpret_cast<TO *>(p.y) + row * N;
        for (int j = threadIdx.x; j < N; j += blockDim.x) store_elem(yo, j, y_at(j));
    } else if constexpr (Q == QOUT_NONE) {
        for (int j = threadIdx.x; j < sp.head; j += blockDim.x) store_elem(y, j, y_at(j));
        for (int c = threadIdx.x; c < sp.nb; c += blockDim.x) {
            const int64_t j0 = sp.head + (int64_t)c * Elem<T>::E;
            float2 h[NP];
            load_chunk_at(FUSED ? static_cast<const T *>(hout) : x, j0, FUSED ? vh : true, h);
            if (w) {
                float2 wv[NP];
                w_chunk_at<T, TW>(w, (int)j0, wv);
#pragma unroll
                for (int q = 0; q < NP; ++q)
                    h[q] = make_float2(__fmul_rn(__fmul_rn(h[q].x, rstd), __fadd_rn(p.offset, wv[q].x)),
                                       __fmul_rn(__fmul_rn(h[q].y, rstd), __fadd_rn(p.offset, wv[q].y)));
            } else {
#pragma unroll
                for (int q = 0; q < NP; ++q) h[q] = make_float2(__fmul_rn(h[q].x, rstd), __fmul_rn(h[q].y, rstd));
            }
            store_chunk_at(y, j0, vy, h);
        }
        for (int j = sp.tail0 + threadIdx.x; j < N; j += blockDim.x) store_elem(y, j, y_at(j));
    } else {
        // (fmaxf drops a NaN product: a zero row with eps = 0 reports 0)
        const float amax = fmaxf(0.f, __fmul_rn(rstd, mrow));
        float sc;
        if constexpr (Q == QOUT_FP8_ROW) {
            sc = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
            if (threadIdx.x == 0) p.qscale_inv[row] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        } else {
            sc = __ldg(p.qscale);
            if (row == 0 && threadIdx.x == 0 && p.qscale_inv) p.qscale_inv[0] = __fdiv_rn(1.f, sc);
        }
        if (p.qamax != nullptr && threadIdx.x == 0) atomicMax(p.qamax, __float_as_uint(amax));
        uint8_t *yq = reinterpret_cast<uint8_t *>(p.y) + row * N;
        for (int j = threadIdx.x; j < N; j += blockDim.x) yq[j] = e4m3x1(__fmul_rn(y_at(j), sc));
    }
}

// LayerNorm forward on the RMSNorm forward's geometry: the row stays in
// registers through two row reductions, the sum (for the mean) and then the
// sum of squared deviations from it (a two-pass variance, which loses
// nothing to cancellation when the mean is large), then
// y = (h - mean) rstd (offset + gamma) + beta, rounded once.
// (held to the register forward's budget, as the RMSNorm one)
template <typename T, typename TW, int TPR, int V, int TEAMS, int CS, bool FUSED, bool PEEL = false>
__global__ void __launch_bounds__(TPR *TEAMS, fwd_min_blocks<TPR * TEAMS>())
    layernorm_fwd_vector(const FwdParams p) {
    static_assert(CS == 1 || TEAMS == 1, "a cluster row uses one team per CTA");
    using Pk = Pair<true>;
    constexpr int NP = Elem<T>::NP;
    constexpr int W = TPR > 32 ? TPR / 32 : 1;
    __shared__ float red[TEAMS][W * CS], red2[TEAMS][W * CS];
    pdl_wait();
    pdl_trigger();

    const int team = threadIdx.x / TPR;
    const int t = threadIdx.x % TPR;
    uint32_t rank = 0;
    int64_t row;
    if constexpr (CS > 1) {
        rank = cluster_ctarank();
        row = cluster_id_x();
    } else {
        row = (int64_t)blockIdx.x * TEAMS + team;
    }
    const bool valid = row < p.M;
    const int64_t rr = valid ? row : p.M - 1;
    const int C = p.N / Elem<T>::E;
    const int64_t base = rr * C;
    const int cslice = (C + CS - 1) / CS;  // a cluster row: equal slices
    const int cbase = (int)rank * cslice;
    const int cend = cbase + cslice < C ? cbase + cslice : C;

    uint4 xv[V];
    fwd_load_row<T, TPR, V, FUSED, PEEL>(p, base, C, cbase, t, cend, valid, xv);

    float2 sm = make_float2(0.f, 0.f);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        float2 a[NP];
        unpack<T>(xv[v], a);  // chunks past the slice are zero
#pragma unroll
        for (int k = 0; k < NP; ++k) sm = Pk::add(sm, a[k]);
    }
    float s;
    if constexpr (CS > 1) {
        cluster_sync();  // every CTA of the cluster runs before any distributed-shared store
        s = cluster_allreduce<TPR, CS>(__fadd_rn(sm.x, sm.y), &red[0][0], t, rank);
    } else {
        s = team_allreduce<TPR>(__fadd_rn(sm.x, sm.y), &red[team][0], t);
    }
    const float mu = __fdiv_rn(s, (float)p.N);
    const float2 nmu2 = make_float2(-mu, -mu);
    float2 sq = make_float2(0.f, 0.f);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = cbase + v * TPR + t;
        if (c < cend) {
            float2 a[NP];
            unpack<T>(xv[v], a);
#pragma unroll
            for (int k = 0; k < NP; ++k) {
                const float2 d = Pk::add(a[k], nmu2);
                sq = Pk::fma(d, d, sq);
            }
        }
    }
    if constexpr (CS > 1) {
        s = cluster_allreduce<TPR, CS>(__fadd_rn(sq.x, sq.y), &red2[0][0], t, rank);
    } else {
        s = team_allreduce<TPR>(__fadd_rn(sq.x, sq.y), &red2[team][0], t);
    }
    const float rstd = rsqrtf(__fadd_rn(__fdiv_rn(s, (float)p.N), p.eps));
    if (!valid) return;
    if (t == 0 && rank == 0) {
        p.rstd[row] = rstd;
        p.mean[row] = mu;
    }
    const float2 r2 = make_float2(rstd, rstd);
    const float2 o2 = make_float2(p.offset, p.offset);
    const int peel = peel_of<PEEL>(p);
    const bool e0 = peel != 0 && cbase + t == 0;  // slot 0 is the row's wrapped chunk
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = cbase + v * TPR + t;
        if (c < cend) {
            float2 a[NP], gv[NP], bv[NP];
            unpack<T>(xv[v], a);
            if (p.w) {
                load_w_chunk_row<T, TW>(p.w, c, C, peel, v == 0 && e0, gv);
#pragma unroll
                for (int k = 0; k < NP; ++k) gv[k] = Pk::add(o2, gv[k]);
            } else {
#pragma unroll
                for (int k = 0; k < NP; ++k) gv[k] = make_float2(1.f, 1.f);
            }
            if (p.beta) {
                load_w_chunk_row<T, TW>(p.beta, c, C, peel, v == 0 && e0, bv);
            } else {
#pragma unroll
                for (int k = 0; k < NP; ++k) bv[k] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < NP; ++k) a[k] = Pk::fma(Pk::mul(Pk::add(a[k], nmu2), r2), gv[k], bv[k]);
            st_row_chunk<T>(reinterpret_cast<uint4 *>(p.y) + base, c, C, peel, v == 0 && e0, pack<T>(a));
        }
    }
}

// Generic LayerNorm forward: one 256-thread CTA per row, three passes over
// the row (the later ones served by L1/L2), split like the RMSNorm one.
template <typename T, typename TW, bool FUSED>
__global__ void __launch_bounds__(256) layernorm_fwd_generic(const FwdParams p) {
    __shared__ float red[32];
    extern __shared__ uint4 gen_smem[];
    pdl_wait();
    pdl_trigger();
    constexpr int E = Elem<T>::E;
    constexpr int NP = Elem<T>::NP;
    const int64_t row = blockIdx.x;
    const int N = p.N;
    const T *x = reinterpret_cast<const T *>(p.x) + row * N;
    const T *res = reinterpret_cast<const T *>(p.residual) + row * N;
    T *hout = reinterpret_cast<T *>(p.residual_out) + row * N;
    const TW *g = reinterpret_cast<const TW *>(p.w);
    const TW *b = reinterpret_cast<const TW *>(p.beta);
    T *y = reinterpret_cast<T *>(p.y) + row * N;
    const uint32_t a16 = addr_mod16(p.x);
    const bool vy = addr_mod16(p.y) == a16;
    const bool vr = FUSED && addr_mod16(p.residual) == a16;
    const bool vh = FUSED && addr_mod16(p.residual_out) == a16;
    const RowSplit sp = row_split(x, N, true);
    // h is re-read by the thread that wrote it: from the shared-memory row
    // cache (16-byte chunks aligned as in x) where the host gave one, else
    // from residual_out or x
    const bool cache = p.cache_row != 0;
    T *hs = reinterpret_cast<T *>(reinterpret_cast<char *>(gen_smem) + addr_mod16(x));
    const T *hsrc = cache ? static_cast<const T *>(hs) : (FUSED ? static_cast<const T *>(hout) : x);
    auto h_at = [&](int j) { return load_elem(hsrc, j); };
    auto h_chunk = [&](int j0, float2 (&h)[NP]) { load_chunk_at(hsrc, j0, cache || !FUSED || vh, h); };

    float sm = 0.f;
    row_visit<E>(
        sp, N,
        [&](int j) {
            float h = load_elem(x, j);
            if constexpr (FUSED) {
                h = round_to(__fadd_rn(h, load_elem(res, j)), x);
                store_elem(hout, j, h);
            }
            if (cache) store_elem(hs, j, h);
            sm = __fadd_rn(sm, h);
        },
        [&](int j0) {
            float2 h[NP];
            load_chunk_at(x, j0, true, h);
            if constexpr (FUSED) {
                float2 r[NP];
                load_chunk_at(res, j0, vr, r);
#pragma unroll
                for (int q = 0; q < NP; ++q) h[q] = make_float2(__fadd_rn(h[q].x, r[q].x), __fadd_rn(h[q].y, r[q].y));
                unpack<T>(pack<T>(h), h);
                store_chunk_at(hout, j0, vh, h);
            }
            if (cache) store_chunk_at(hs, j0, true, h);
#pragma unroll
            for (int q = 0; q < NP; ++q) sm = __fadd_rn(__fadd_rn(sm, h[q].x), h[q].y);
        });
    const float mu = __fdiv_rn(cta_allreduce(sm, red), (float)N);
    float sq = 0.f;
    row_visit<E>(
        sp, N,
        [&](int j) {
            const float d = __fadd_rn(h_at(j), -mu);
            sq = __fmaf_rn(d, d, sq);
        },
        [&](int j0) {
            float2 h[NP];
            h_chunk(j0, h);
#pragma unroll
            for (int q = 0; q < NP; ++q) {
                const float d0 = __fadd_rn(h[q].x, -mu), d1 = __fadd_rn(h[q].y, -mu);
                sq = __fmaf_rn(d1, d1, __fmaf_rn(d0, d0, sq));
            }
        });
    const float rstd = rsqrtf(__fadd_rn(__fdiv_rn(cta_allreduce(sq, red), (float)N), p.eps));
    if (threadIdx.x == 0) {
        p.rstd[row] = rstd;
        p.mean[row] = mu;
    }
    auto y_of = [&](float h, float gj, float bj) {
        const float xh = __fmul_rn(__fadd_rn(h, -mu), rstd);
        return __fmaf_rn(xh, g ? __fadd_rn(p.offset, gj) : 1.f, bj);
    };
    row_visit<E>(
        sp, N,
        [&](int j) { store_elem(y, j, y_of(h_at(j), g ? load_w(g, j) : 0.f, b ? load_w(b, j) : 0.f)); },
        [&](int j0) {
            float2 h[NP], gv[NP], bv[NP];
            h_chunk(j0, h);
            if (g) w_chunk_at<T, TW>(g, j0, gv);
            if (b) w_chunk_at<T, TW>(b, j0, bv);
#pragma unroll
            for (int q = 0; q < NP; ++q)
                h[q] = make_float2(y_of(h[q].x, g ? gv[q].x : 0.f, b ? bv[q].x : 0.f),
                                   y_of(h[q].y, g ? gv[q].y : 0.f, b ? bv[q].y : 0.f));
            store_chunk_at(y, j0, vy, h);
        });
}

// Staged persistent forward, for rows that one CTA's registers serve badly
// (wider than 2048 chunks: one row per short-lived cluster keeps too few
// loads in flight). A unit (a CTA, or a cluster whose CTAs take equal
// slices of each row) walks rows unit, unit + G, ...; each row's x (and
// residual) slice streams by cp.async.bulk into one of the stages, counted
// in bytes on the stage's mbarrier. Pass 1 forms h (fused: R(x + r), stored
// to residual_out) and the row sum of squares (LayerNorm: the sum, then in
// a pass of its own the squared deviations; E4M3: beside the sum of squares
// the max of |h (offset + w)|, the pair meeting in one reduction); pass 2
// reads the stage again and writes y. The last warp through a stage refills it, as in the
// backward's re-read schedule. A thread's chunks, their order and the
// reduction tree are the register forward's, so y and rstd are the same
// bits. Every wait is bounded; one that gives up writes the status word and
// the kernel carries on.
template <typename T, typename TW, int TPR, int V, int S, int CS, bool FUSED, bool LN, int Q, bool PEEL>
__device__ __forceinline__ void staged_fwd_body(const FwdParams &p) {
    static_assert(Q == QOUT_NONE || !LN, "E4M3 output: RMSNorm only");
    using Pk = Pair<true>;
    constexpr int E = Elem<T>::E;
    constexpr int NP = Elem<T>::NP;
    constexpr int W = TPR / 32;
    constexpr int NB = FUSED ? 2 : 1;  // rows a stage holds: x (, residual)
    static_assert(TPR % 32 == 0 && TPR >= 64, "whole warps");
    __shared__ float red[2][CS * W];
    __shared__ __align__(8) uint64_t full[S];
    __shared__ __align__(8) uint64_t rbar[2];  // cluster rows: arrival of the peers' sums
    // E4M3: one reduction a row of (sum of squares, max), its own slots and barriers
    constexpr bool PAIR = fp8_out(Q);
    __shared__ float2 red2[PAIR ? 2 : 1][PAIR ? CS * W : 1];
    __shared__ __align__(8) uint64_t rbar2[PAIR ? 2 : 1];
    __shared__ unsigned done[S];               // warps through the stage's row
    extern __shared__ float4 fstage_smem[];    // ns * NB * Cb chunks of 16 bytes
    pdl_wait();  // before any read of the rows (the bulk copies included)

    const int N = p.N;
    const int C = N / E;
    const int t = threadIdx.x;
    const int lane = t & 31;
    uint32_t rank = 0;
    if constexpr (CS > 1) rank = cluster_ctarank();
    const int Cst = (C + CS - 1) / CS;  // this CTA's slice: chunks [cbase, cbase + Cs)
    const int cbase = (int)rank * Cst;
    const int Cs = C - cbase <= 0 ? 0 : (C - cbase < Cst ? C - cbase : Cst);
    // rows at a common offset: the CTA holding chunk 0 also stages aligned
    // chunk C (after its slice) to wrap chunk 0; row buffers are one slot longer
    const int peel = peel_of<PEEL>(p);
    const bool wrap = peel != 0 && cbase == 0;
    const int Cb = Cst + (peel != 0 ? 1 : 0);
    // (only slot v = 0 of thread 0 can be the wrapped chunk: e0, which
    // that thread wraps in place once a row before reading it)
    const bool e0 = wrap && threadIdx.x == 0;
    auto staged = [&](const uint4 *buf, int /*v*/, int cl) { return lds128(buf + cl); };
    const int64_t unit = CS > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t G = CS > 1 ? (int64_t)cluster_count_x() : (int64_t)gridDim.x;
    const int64_t iters = unit < p.M ? (p.M - unit + G - 1) / G : 0;
    const int ns = p.stages >= 2 && p.stages < S ? p.stages : S;
    const uint32_t row_bytes = (uint32_t)Cs * 16u;
    uint4 *stages = reinterpret_cast<uint4 *>(fstage_smem);
    const uint4 *x4 = reinterpret_cast<const uint4 *>(p.x);
    const uint4 *r4 = reinterpret_cast<const uint4 *>(p.residual);
    auto issue = [&](int64_t k, int s) {
        const int64_t row0 = (unit + k * G) * C;
        const int64_t off = row0 + cbase;
        uint4 *dst = stages + (size_t)s * NB * Cb;
        const uint32_t extra = wrap ? 16u : 0u;
        mbar_arrive_expect_tx(&full[s], (row_bytes + extra) * NB);
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
        if constexpr (FUSED) copy(dst + Cb, r4);
    };
    constexpr uint32_t kSlotBytes = CS * W * sizeof(float);
    constexpr uint32_t kSlotBytes2 = CS * W * sizeof(float2);
    if (t == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            done[s] = 0;
        }
        if constexpr (CS > 1) {
            mbar_init(&rbar[0], 1);
            mbar_init(&rbar[1], 1);
            mbar_arrive_expect_tx(&rbar[0], kSlotBytes);
            mbar_arrive_expect_tx(&rbar[1], kSlotBytes);
            if constexpr (PAIR) {
                mbar_init(&rbar2[0], 1);
                mbar_init(&rbar2[1], 1);
                mbar_arrive_expect_tx(&rbar2[0], kSlotBytes2);
                mbar_arrive_expect_tx(&rbar2[1], kSlotBytes2);
            }
        }
        mbar_init_fence();
        for (int s = 0; s < ns && s < iters; ++s) issue(s, s);
    }
    __syncthreads();
    if constexpr (CS > 1) cluster_sync();

    bool failed = false;
    // Row sum across the unit. Reduction q uses slot buffer q & 1; a cluster
    // sends each warp's sum to every CTA (st.async, counted in bytes on the
    // receiver's barrier, phase parity (q >> 1) & 1) and re-arms the barrier
    // after reading; a buffer is written again (q + 2) only after every warp
    // sent its q + 1 sum, which it does after reading the buffer for q.
    uint32_t q = 0;
    // combines with Op (OpAdd: a row sum)
    auto rowred = [&](auto op, float v) {
        using Op = decltype(op);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = Op::f(v, __shfl_xor_sync(0xffffffffu, v, o));
        const int b = (int)(q & 1);
        float sum;
        if constexpr (CS > 1) {
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < CS; ++c) st_async_cluster(&red[b][rank * W + (t >> 5)], &rbar[b], (uint32_t)c, v);
            }
            if (!mbar_wait(&rbar[b], (q >> 1) & 1u, kWaitLimit)) failed = true;
            sum = sum_slots<CS * W, Op>(&red[b][0], lane);
            if (t == 0) mbar_arrive_expect_tx(&rbar[b], kSlotBytes);
        } else {
            if (lane == 0) red[b][t >> 5] = v;
            __syncthreads();
            sum = sum_slots<W, Op>(&red[b][0], lane);
        }
        ++q;
        return sum;
    };
    auto rowsum = [&](float v) { return rowred(OpAdd{}, v); };
    // the E4M3 row's (sum of squares, max) in one reduction, with the same
    // buffer and barrier rules on its own slots (q2: its reduction count)
    uint32_t q2 = 0;
    auto rowred2 = [&](float2 v) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = SumMax::f(v, shfl_xor2(v, o));
        const int b = (int)(q2 & 1);
        float2 r;
        if constexpr (CS > 1) {
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < CS; ++c)
                    st_async_cluster2(&red2[b][rank * W + (t >> 5)], &rbar2[b], (uint32_t)c, v);
            }
            if (!mbar_wait(&rbar2[b], (q2 >> 1) & 1u, kWaitLimit)) failed = true;
            r = sum_slots2<CS * W, SumMax>(&red2[b][0], lane);
            if (t == 0) mbar_arrive_expect_tx(&rbar2[b], kSlotBytes2);
        } else {
            if (lane == 0) red2[b][t >> 5] = v;
            __syncthreads();
            r = sum_slots2<W, SumMax>(&red2[b][0], lane);
        }
        ++q2;
        return r;
    };

    const float2 o2 = make_float2(p.offset, p.offset);
    int s = 0;
    uint32_t ph = 0;
    for (int64_t k = 0; k < iters; ++k) {
        const int64_t row = unit + k * G;
        if (!mbar_wait(&full[s], ph, kWaitLimit)) failed = true;
        const int sk = s;
        const uint4 *src = stages + (size_t)s * NB * Cb;
        if (e0) wrap_staged<T>(stages + (size_t)s * NB * Cb, Cb, NB, Cst, peel);
        const int64_t base = row * C + cbase;
        const int64_t rowbase = row * C;
        // h of chunk v of the slice (fused: R(x + r), stored once in pass 1)
        auto hchunk = [&](int v, float2 (&h)[NP], bool store) {
            const int cl = v * TPR + t;
            if (cl < Cs) {
                unpack<T>(staged(src, v, cl), h);
                if constexpr (FUSED) {
                    float2 rr[NP];
                    unpack<T>(staged(src + Cb, v, cl), rr);
#pragma unroll
                    for (int j = 0; j < NP; ++j) h[j] = Pk::add(h[j], rr[j]);
                    const uint4 hp = pack<T>(h);
                    if (store)
                        st_row_chunk<T>(reinterpret_cast<uint4 *>(p.residual_out) + rowbase, cbase + cl, C, peel,
                                        v == 0 && e0, hp);
                    unpack<T>(hp, h);
                }
            } else {
#pragma unroll
                for (int j = 0; j < NP; ++j) h[j] = make_float2(0.f, 0.f);
            }
        };
        float2 acc = make_float2(0.f, 0.f);
        float mh = 0.f;  // E4M3: max |h (offset + w)| of this thread's elements
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float2 h[NP];
            hchunk(v, h, true);
#pragma unroll
            for (int j = 0; j < NP; ++j) acc = LN ? Pk::add(acc, h[j]) : Pk::fma(h[j], h[j], acc);
            if constexpr (PAIR) {
                const int cl = v * TPR + t;
                float2 g[NP];
                if (p.w && cl < Cs) {
                    load_w_chunk_row<T, TW>(p.w, cbase + cl, C, peel, v == 0 && e0, g);
#pragma unroll
                    for (int j = 0; j < NP; ++j) g[j] = Pk::mul(h[j], Pk::add(o2, g[j]));
                } else {
#pragma unroll
                    for (int j = 0; j < NP; ++j) g[j] = h[j];  // factor 1 (zero past the slice)
                }
#pragma unroll
                for (int j = 0; j < NP; ++j) mh = fmaxf(mh, fmaxf(fabsf(g[j].x), fabsf(g[j].y)));
            }
        }
        float rstd, mu = 0.f, mrow = 0.f;
        if constexpr (PAIR) {
            const float2 r = rowred2(make_float2(__fadd_rn(acc.x, acc.y), mh));
            rstd = rsqrtf(__fadd_rn(__fdiv_rn(r.x, (float)N), p.eps));
            mrow = r.y;
        } else if constexpr (LN) {
            mu = __fdiv_rn(rowsum(__fadd_rn(acc.x, acc.y)), (float)N);
            const float2 nmu2 = make_float2(-mu, -mu);
            float2 sq = make_float2(0.f, 0.f);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if (v * TPR + t < Cs) {
                    float2 h[NP];
                    hchunk(v, h, false);
#pragma unroll
                    for (int j = 0; j < NP; ++j) {
                        const float2 d = Pk::add(h[j], nmu2);
                        sq = Pk::fma(d, d, sq);
                    }
                }
            }
            rstd = rsqrtf(__fadd_rn(__fdiv_rn(rowsum(__fadd_rn(sq.x, sq.y)), (float)N), p.eps));
        } else {
            rstd = rsqrtf(__fadd_rn(__fdiv_rn(rowsum(__fadd_rn(acc.x, acc.y)), (float)N), p.eps));
        }
        if (t == 0 && rank == 0) {
            p.rstd[row] = rstd;
            if constexpr (LN) p.mean[row] = mu;
        }
        const float2 r2 = make_float2(rstd, rstd);
        const float2 nmu2 = make_float2(-mu, -mu);
        // y of chunk v of the slice (RMSNorm: x rstd (offset + w))
        auto ychunk = [&](int v, float2 (&a)[NP]) {
            const int c = cbase + v * TPR + t;
            hchunk(v, a, false);
            if constexpr (LN) {
                float2 gv[NP], bv[NP];
                if (p.w) {
                    load_w_chunk_row<T, TW>(p.w, c, C, peel, v == 0 && e0, gv);
#pragma unroll
                    for (int j = 0; j < NP; ++j) gv[j] = Pk::add(o2, gv[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < NP; ++j) gv[j] = make_float2(1.f, 1.f);
                }
                if (p.beta) {
                    load_w_chunk_row<T, TW>(p.beta, c, C, peel, v == 0 && e0, bv);
                } else {
#pragma unroll
                    for (int j = 0; j < NP; ++j) bv[j] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < NP; ++j) a[j] = Pk::fma(Pk::mul(Pk::add(a[j], nmu2), r2), gv[j], bv[j]);
            } else if (p.w) {
                float2 wv[NP];
                load_w_chunk_row<T, TW>(p.w, c, C, peel, v == 0 && e0, wv);
#pragma unroll
                for (int j = 0; j < NP; ++j)  // (E4M3: y' = (h (offset + w)) rstd, as the first pass's max)
                    a[j] = PAIR ? Pk::mul(Pk::mul(a[j], Pk::add(o2, wv[j])), r2)
                                : Pk::mul(Pk::mul(a[j], r2), Pk::add(o2, wv[j]));
            } else {
#pragma unroll
                for (int j = 0; j < NP; ++j) a[j] = Pk::mul(a[j], r2);
            }
        };
        if constexpr (!fp8_out(Q)) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int cl = v * TPR + t;
                if (cl < Cs) {
                    float2 a[NP];
                    ychunk(v, a);
                    if constexpr (narrow_out(Q))
                        st_narrow_chunk<Q>(p.y, rowbase + cbase + cl, a);  // (no peel)
                    else
                        st_row_chunk<T>(reinterpret_cast<uint4 *>(p.y) + rowbase, cbase + cl, C, peel, v == 0 && e0,
                                        pack<T>(a));
                }
            }
        } else {
            // E4M3: the row's max |y| = rstd max |h (offset + w)| from the
            // first pass's reduction, then the codes from one more pass
            const float amax = fmaxf(0.f, __fmul_rn(rstd, mrow));
            float sc;
            if constexpr (Q == QOUT_FP8_ROW) {
                sc = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
                if (t == 0 && rank == 0) p.qscale_inv[row] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
            } else {
                sc = __ldg(p.qscale);
                if (row == 0 && t == 0 && rank == 0 && p.qscale_inv) p.qscale_inv[0] = __fdiv_rn(1.f, sc);
            }
            if (p.qamax != nullptr && t == 0 && rank == 0) atomicMax(p.qamax, __float_as_uint(amax));
            const float2 s2 = make_float2(sc, sc);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int cl = v * TPR + t;
                if (cl < Cs) {
                    float2 a[NP];
                    ychunk(v, a);
#pragma unroll
                    for (int j = 0; j < NP; ++j) a[j] = Pk::mul(a[j], s2);
                    if constexpr (NP == 4) {
                        __stcs(reinterpret_cast<uint2 *>(p.y) + base + cl, make_uint2(e4m3x4(a[0], a[1]), e4m3x4(a[2], a[3])));
                    } else {
                        __stcs(reinterpret_cast<unsigned int *>(p.y) + base + cl, e4m3x4(a[0], a[1]));
                    }
                }
            }
        }
        // the warp is through stage sk; the last warp to say so refills it
        // with row k + ns (the fences order every warp's reads of the stage
        // before the bulk copies that overwrite it)
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
        if (++s == ns) {
            s = 0;
            ph ^= 1u;
        }
    }
    if (failed && p.status) *p.status = kStatusWaitTimeout;
    pdl_trigger();  // every row done: the next kernel may launch
    // no CTA leaves while a peer may still store into its shared memory
    if constexpr (CS > 1) cluster_sync();
}

template <typename T, typename TW, int TPR, int V, int S, int CS, bool FUSED, int Q = QOUT_NONE, bool PEEL = false>
__global__ void __launch_bounds__(TPR, 1) rmsnorm_fwd_staged(const FwdParams p) {
    staged_fwd_body<T, TW, TPR, V, S, CS, FUSED, false, Q, PEEL>(p);
}

template <typename T, typename TW, int TPR, int V, int S, int CS, bool FUSED, bool PEEL = false>
__global__ void __launch_bounds__(TPR, 1) layernorm_fwd_staged(const FwdParams p) {
    staged_fwd_body<T, TW, TPR, V, S, CS, FUSED, true, QOUT_NONE, PEEL>(p);
}

// Streamed generic forward: persistent CTAs, rows of any alignment and of
// at most TPR * K elements, the forward counterpart of the streamed generic
// backward. Row k of a CTA streams into stage k mod ns by bulk copies of
// the 16-byte covers (cover16) of its x (and residual) rows, each at its
// own offset within its first block. Thread t owns columns t + i TPR
// (i < K) of every row, with (offset + w) for them held in registers; it
// reads its elements of the stage before the row reduction's barrier, after
// which thread 0 refills the stage with row k + ns. h = x (fused: the sum
// x + residual rounded to the storage type, which is also stored),
// rstd = 1 / sqrt(sum h^2 / N + eps), y = (h rstd) (offset + w), each
// stored element by element (a row's edge blocks may hold a neighbouring
// row, which another CTA writes). Every wait is bounded: one that gives up
// records the status word, waits (again bounded) for the stages' last
// copies and lets the kernel end.
template <typename T, typename TW, int TPR, int K, int SMAX, bool FUSED>
__global__ void __launch_bounds__(TPR, TPR >= 512 ? 1 : 512 / TPR) rmsnorm_fwd_stream(const FwdParams p) {
    static_assert(TPR % 32 == 0 && TPR >= 64 && TPR <= 1024, "whole warps");
    constexpr int W = TPR / 32;
    constexpr int NB = FUSED ? 2 : 1;  // arrays a stage holds: x (, residual)
    __shared__ float red[2][W];
    __shared__ __align__(8) uint64_t full[SMAX];
    extern __shared__ float4 sstage_smem[];  // ns * NB slots of stream_slot_bytes(N, sizeof(T))
    pdl_wait();  // before any read of the rows (the bulk copies included)
    const int N = p.N;
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int ns = p.stages;  // 2 .. SMAX, chosen by the host to fit
    const int64_t G = gridDim.x;
    const int64_t unit = blockIdx.x;
    const int64_t iters = unit < p.M ? (p.M - unit + G - 1) / G : 0;
    const uint32_t rb = (uint32_t)N * (uint32_t)sizeof(T);  // bytes of a row
    const uint32_t slot = (uint32_t)stream_slot_bytes(N, (int)sizeof(T));
    char *const stages = reinterpret_cast<char *>(sstage_smem);
    const char *gx = static_cast<const char *>(p.x);
    const char *gr = static_cast<const char *>(p.residual);
    // thread 0: the covers of row k's arrays into stage s
    auto issue = [&](int64_t k, int s) {
        const int64_t off = (unit + k * G) * (int64_t)rb;
        const Cover cx = cover16(gx + off, rb);
        const Cover cr = FUSED ? cover16(gr + off, rb) : Cover{nullptr, 0u, 0u};
        char *dst = stages + (size_t)s * NB * slot;
        mbar_arrive_expect_tx(&full[s], cx.bytes + cr.bytes);
        bulk_g2s(dst, cx.src, cx.bytes, &full[s]);
        if constexpr (FUSED) bulk_g2s(dst + slot, cr.src, cr.bytes, &full[s]);
    };
    const TW *w = static_cast<const TW *>(p.w);
    const bool has_w = w != nullptr;
    float wf[K];
#pragma unroll
    for (int i = 0; i < K; ++i) {
        const int j = t + i * TPR;
        wf[i] = (has_w && j < N) ? __fadd_rn(p.offset, load_w(w, j)) : 1.f;
    }
    if (t == 0) {
        for (int s = 0; s < ns; ++s) mbar_init(&full[s], 1);
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
        const int64_t off = row * (int64_t)rb;
        const char *sb = stages + (size_t)s * NB * slot;
        const T *xs = reinterpret_cast<const T *>(sb + addr_mod16(gx + off));
        const T *rs = reinterpret_cast<const T *>(sb + slot + (FUSED ? addr_mod16(gr + off) : 0u));
        T *hout = static_cast<T *>(p.residual_out) + row * (int64_t)N;
        float hv[K];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int j = t + i * TPR;
            hv[i] = 0.f;
            if (j < N) {
                hv[i] = load_elem(xs, j);
                if constexpr (FUSED) {
                    hv[i] = round_to(__fadd_rn(hv[i], load_elem(rs, j)), xs);
                    store_elem(hout, j, hv[i]);
                }
            }
            ss = __fmaf_rn(hv[i], hv[i], ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        float *slots = red[k & 1];
        if (lane == 0) slots[t >> 5] = ss;
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
        const float rstd = rsqrtf(__fadd_rn(__fdiv_rn(sum_slots<W>(slots, lane), (float)N), p.eps));
        if (t == 0) p.rstd[row] = rstd;
        T *y = static_cast<T *>(p.y) + row * (int64_t)N;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int j = t + i * TPR;
            if (j < N) store_elem(y, j, __fmul_rn(__fmul_rn(hv[i], rstd), wf[i]));
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
    pdl_trigger();  // every row done: the next kernel may launch
}

// Launch of a staged forward kernel: a cluster of CS CTAs (of one where a
// CTA holds the whole row; its bulk copies name a shared::cluster
// destination) with the stages' dynamic shared memory.
static int launch_fwd_staged_kernel(const void *k, int cs, int threads, const FwdParams &p, int grid, int smem,
                                    void *stream) {
    const int e = allow_staged_smem(k);
    if (e != 0) return e;
    LaunchCfg lc((unsigned)grid, (unsigned)threads, (size_t)smem, static_cast<cudaStream_t>(stream), (unsigned)cs);
    void *args[] = {const_cast<FwdParams *>(&p)};
    return (int)cudaLaunchKernelExC(&lc.cfg, k, args);
}

// ------------------------------------------------------------- dispatch --

template <typename T, typename TW, int TPR, int V, int TEAMS, int CS, int Q, bool PEEL>
static int launch_vec(bool fused, const FwdParams &p, int grid, void *stream) {
    LaunchCfg lc((unsigned)grid, TPR * TEAMS, 0, static_cast<cudaStream_t>(stream), CS > 1 ? CS : 0);
    return fused ? (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_fwd_vector<T, TW, TPR, V, TEAMS, CS, true, Q, PEEL>, p)
                 : (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_fwd_vector<T, TW, TPR, V, TEAMS, CS, false, Q, PEEL>, p);
}

template <typename T, typename TW, int TPR, int V, int TEAMS, int CS, bool PEEL>
static const void *ptr_vec(bool fused) {
    return fused ? (const void *)rmsnorm_fwd_vector<T, TW, TPR, V, TEAMS, CS, true, QOUT_NONE, PEEL>
                 : (const void *)rmsnorm_fwd_vector<T, TW, TPR, V, TEAMS, CS, false, QOUT_NONE, PEEL>;
}

// The generic LayerNorm forward's row cache: N elements and 16 bytes of
// alignment slack (set by the host only for rows of up to 24 KB).
template <typename T>
static int gen_cache_bytes(const FwdParams &p) {
    return p.cache_row ? p.N * (int)sizeof(T) + 16 : 0;
}

template <typename T, typename TW, int Q>
static int launch_gen(bool fused, const FwdParams &p, int grid, void *stream) {
    LaunchCfg lc((unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream));
    return fused ? (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_fwd_generic<T, TW, true, Q>, p)
                 : (int)cudaLaunchKernelEx(&lc.cfg, rmsnorm_fwd_generic<T, TW, false, Q>, p);
}

template <typename T, typename TW>
static const void *ptr_gen(bool fused) {
    return fused ? (const void *)rmsnorm_fwd_generic<T, TW, true> : (const void *)rmsnorm_fwd_generic<T, TW, false>;
}

// A weight type other than the activations', and the E4M3 outputs, are
// compiled for the default plans (and the generic one) only; alternatives
// are for tuning. The PEEL instantiations (rows at a common offset, which
// take neither) exist for the default vectorised plans only.
template <typename T, typename TW, int PATH, int CMIN, int Q, bool PEEL = false>
constexpr bool instantiated() {
    if constexpr (PEEL)
        return std::is_same<T, TW>::value && Q == QOUT_NONE && CMIN > 0 && !generic_path(PATH);
    else
        return (std::is_same<T, TW>::value && Q == QOUT_NONE) || PATH == PATH_GENERIC || CMIN > 0;
}

// One switch case per table entry; `if constexpr` keeps kernels of other
// ops, paths, weight types and outputs from being instantiated here.
template <typename T, typename TW, int Q, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int CS, int CMIN>
static int launch_entry(bool fused, const FwdParams &p, int grid, void *stream) {
    if constexpr (OP != OP_FWD || !instantiated<T, TW, PATH, CMIN, Q, PEEL>()) return (int)cudaErrorInvalidValue;
    else if constexpr (PATH == PATH_GENERIC) return launch_gen<T, TW, Q>(fused, p, grid, stream);
    else if constexpr (PATH == PATH_VECTOR) return launch_vec<T, TW, TPR, V, TEAMS, CS, Q, PEEL>(fused, p, grid, stream);
    else return (int)cudaErrorInvalidValue;
}

template <typename T, typename TW, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int CS, int CMIN>
static const void *ptr_entry(bool fused) {
    if constexpr (OP != OP_FWD || !instantiated<T, TW, PATH, CMIN, QOUT_NONE, PEEL>()) return nullptr;
    else if constexpr (PATH == PATH_GENERIC) return ptr_gen<T, TW>(fused);
    else if constexpr (PATH == PATH_VECTOR) return ptr_vec<T, TW, TPR, V, TEAMS, CS, PEEL>(fused);
    else return nullptr;
}

template <typename T, typename TW, int Q = QOUT_NONE, bool PEEL = false>
static int launch_t(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    switch (plan_id) {
#define RMSN_FWD_CASE(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id: return launch_entry<T, TW, Q, PEEL, op, path, tpr, v, teams, cs, cmin>(fused, p, grid, stream);
        RMSNORM_PLAN_TABLE(RMSN_FWD_CASE)
#undef RMSN_FWD_CASE
    default:
        return (int)cudaErrorInvalidValue;
    }
}

template <typename T, typename TW, bool PEEL = false>
static const void *ptr_t(int plan_id, bool fused) {
    switch (plan_id) {
#define RMSN_FWD_PTR(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id: return ptr_entry<T, TW, PEEL, op, path, tpr, v, teams, cs, cmin>(fused);
        RMSNORM_PLAN_TABLE(RMSN_FWD_PTR)
#undef RMSN_FWD_PTR
    default:
        return nullptr;
    }
}

// Staged forward plans (OP_FWD_STAGED): one entry per table row; kernels of
// other ops are not instantiated, and a weight type other than the
// activations' only for the default plans.
template <typename T, typename TW, bool LN, int Q, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int D,
          int CS, int CMIN>
static const void *staged_fwd_ptr_entry(bool fused) {
    if constexpr (OP == OP_FWD_STAGED && PATH == PATH_STREAM) {
        // the streamed generic forward: RMSNorm, output in the activations' type
        if constexpr (LN || Q != QOUT_NONE || PEEL) {
            return nullptr;
        } else {
            return fused ? (const void *)rmsnorm_fwd_stream<T, TW, TPR, V, D, true>
                         : (const void *)rmsnorm_fwd_stream<T, TW, TPR, V, D, false>;
        }
    } else if constexpr (OP != OP_FWD_STAGED || PATH != PATH_RESTAGED || !staged_plan(PATH, TEAMS, CS) ||
                         !instantiated<T, TW, PATH, CMIN, Q, PEEL>() || (LN && Q != QOUT_NONE)) {
        return nullptr;
    } else if constexpr (LN) {
        return fused ? (const void *)layernorm_fwd_staged<T, TW, TPR, V, D, CS, true, PEEL>
                     : (const void *)layernorm_fwd_staged<T, TW, TPR, V, D, CS, false, PEEL>;
    } else {
        return fused ? (const void *)rmsnorm_fwd_staged<T, TW, TPR, V, D, CS, true, Q, PEEL>
                     : (const void *)rmsnorm_fwd_staged<T, TW, TPR, V, D, CS, false, Q, PEEL>;
    }
}

template <typename T, typename TW, bool LN, int Q, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int D,
          int CS, int CMIN>
static int staged_fwd_launch_entry(bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    const void *k = staged_fwd_ptr_entry<T, TW, LN, Q, PEEL, OP, PATH, TPR, V, TEAMS, D, CS, CMIN>(fused);
    if (!k) return (int)cudaErrorInvalidValue;
    return launch_fwd_staged_kernel(k, CS, TPR, p, grid, smem, stream);
}

template <typename T, typename TW, bool LN, int Q = QOUT_NONE, bool PEEL = false>
static const void *staged_fwd_ptr_t(int plan_id, bool fused) {
    switch (plan_id) {
#define RMSN_SFWD_PTR(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id: return staged_fwd_ptr_entry<T, TW, LN, Q, PEEL, op, path, tpr, v, teams, depth, cs, cmin>(fused);
        RMSNORM_PLAN_TABLE(RMSN_SFWD_PTR)
#undef RMSN_SFWD_PTR
    default:
        return nullptr;
    }
}

template <typename T, typename TW, bool LN, int Q = QOUT_NONE, bool PEEL = false>
static int staged_fwd_launch_t(int plan_id, bool fused, const FwdParams &p, int grid, int smem, void *stream) {
    switch (plan_id) {
#define RMSN_SFWD_CASE(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id:                                                                    \
        return staged_fwd_launch_entry<T, TW, LN, Q, PEEL, op, path, tpr, v, teams, depth, cs, cmin>(fused, p, grid, \
                                                                                                  smem, stream);
        RMSNORM_PLAN_TABLE(RMSN_SFWD_CASE)
#undef RMSN_SFWD_CASE
    default:
        return (int)cudaErrorInvalidValue;
    }
}

// E4M3 output of the staged forward: the mode picks the instantiation
// (TW: the weight's type, the activations' or fp32).
template <typename T, typename TW = T>
static int staged_launch_q(int plan_id, bool fused, int mode, const FwdParams &p, int grid, int smem, void *stream) {
    if (mode == QOUT_FP8_TENSOR) return staged_fwd_launch_t<T, TW, false, QOUT_FP8_TENSOR>(plan_id, fused, p, grid, smem, stream);
    if (mode == QOUT_FP8_ROW) return staged_fwd_launch_t<T, TW, false, QOUT_FP8_ROW>(plan_id, fused, p, grid, smem, stream);
    if constexpr (std::is_same<T, float>::value) {
        if (mode == QOUT_BF16) return staged_fwd_launch_t<T, TW, false, QOUT_BF16>(plan_id, fused, p, grid, smem, stream);
        if (mode == QOUT_F16) return staged_fwd_launch_t<T, TW, false, QOUT_F16>(plan_id, fused, p, grid, smem, stream);
    }
    return (int)cudaErrorInvalidValue;
}
template <typename T, typename TW = T>
static const void *staged_ptr_q(int plan_id, bool fused, int mode) {
    if (mode == QOUT_FP8_TENSOR) return staged_fwd_ptr_t<T, TW, false, QOUT_FP8_TENSOR>(plan_id, fused);
    if (mode == QOUT_FP8_ROW) return staged_fwd_ptr_t<T, TW, false, QOUT_FP8_ROW>(plan_id, fused);
    if constexpr (std::is_same<T, float>::value) {
        if (mode == QOUT_BF16) return staged_fwd_ptr_t<T, TW, false, QOUT_BF16>(plan_id, fused);
        if (mode == QOUT_F16) return staged_fwd_ptr_t<T, TW, false, QOUT_F16>(plan_id, fused);
    }
    return nullptr;
}

// E4M3 (and, for fp32 activations, bf16 or fp16) output: the mode picks
// the instantiation.
template <typename T, typename TW = T>
static int launch_q(int plan_id, bool fused, int mode, const FwdParams &p, int grid, void *stream) {
    if (mode == QOUT_FP8_TENSOR) return launch_t<T, TW, QOUT_FP8_TENSOR>(plan_id, fused, p, grid, stream);
    if (mode == QOUT_FP8_ROW) return launch_t<T, TW, QOUT_FP8_ROW>(plan_id, fused, p, grid, stream);
    if constexpr (std::is_same<T, float>::value) {
        if (mode == QOUT_BF16) return launch_t<T, TW, QOUT_BF16>(plan_id, fused, p, grid, stream);
        if (mode == QOUT_F16) return launch_t<T, TW, QOUT_F16>(plan_id, fused, p, grid, stream);
    }
    return (int)cudaErrorInvalidValue;
}

// LayerNorm forward: the forward plans' geometry, default plans and the
// generic one.
template <typename T, typename TW, bool PEEL, int OP, int PATH, int TPR, int V, int TEAMS, int CS, int CMIN>
static int ln_launch_entry(bool fused, const FwdParams &p, int grid, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if constexpr (OP != OP_FWD || !(PATH == PATH_GENERIC || CMIN > 0) ||
                  (PEEL && !instantiated<T, TW, PATH, CMIN, QOUT_NONE, true>())) {
        return (int)cudaErrorInvalidValue;
    } else if constexpr (PATH == PATH_GENERIC) {
        LaunchCfg lc((unsigned)grid, 256, (size_t)gen_cache_bytes<T>(p), s);
        return fused ? (int)cudaLaunchKernelEx(&lc.cfg, layernorm_fwd_generic<T, TW, true>, p)
                     : (int)cudaLaunchKernelEx(&lc.cfg, layernorm_fwd_generic<T, TW, false>, p);
    } else {
        LaunchCfg lc((unsigned)grid, TPR * TEAMS, 0, s, CS > 1 ? CS : 0);
        return fused ? (int)cudaLaunchKernelEx(&lc.cfg, layernorm_fwd_vector<T, TW, TPR, V, TEAMS, CS, true, PEEL>, p)
                     : (int)cudaLaunchKernelEx(&lc.cfg, layernorm_fwd_vector<T, TW, TPR, V, TEAMS, CS, false, PEEL>, p);
    }
}

// (TW: gamma's and beta's type, the activations' or fp32)
template <typename T, typename TW = T, bool PEEL = false>
static int ln_launch_t(int plan_id, bool fused, const FwdParams &p, int grid, void *stream) {
    switch (plan_id) {
#define RMSN_LN_FWD_CASE(id, op, path, tpr, v, teams, depth, cs, dtm, cmin, cmax) \
    case id: return ln_launch_entry<T, TW, PEEL, op, path, tpr, v, teams, cs, cmin>(fused, p, grid, stream);
        RMSNORM_PLAN_TABLE(RMSN_LN_FWD_CASE)
#undef RMSN_LN_FWD_CASE
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace rmsn
