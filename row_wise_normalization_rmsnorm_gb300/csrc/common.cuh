// common.cuh -- device helpers shared by the kernels: 16-byte chunk access,
// bf16/fp16/fp32 pair conversion, packed f32x2 arithmetic, team (sub-warp,
// warp, multi-warp) and cluster all-reduces, mbarrier waits, bulk copies
// into shared memory and E4M3 conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace rmsn {

// Elements per 16-byte chunk and per register pair.
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int E = 4;   // elements per chunk
    static constexpr int NP = 2;  // float2 pairs per chunk
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int E = 8;
    static constexpr int NP = 4;
};
template <> struct Elem<__half> {
    static constexpr int E = 8;
    static constexpr int NP = 4;
};

// ------------------------------------------------- launch and ordering --
// Every kernel is launched on the caller's stream as a programmatic
// dependent of the kernel before it (cudaLaunchAttributeProgrammatic-
// StreamSerialization). When that kernel is one of ours and has signalled
// its dependents (pdl_trigger), this one's CTAs are launched while it
// drains; each of our kernels calls pdl_wait before it touches global
// memory, which returns once the kernel before it has completed and its
// writes are visible (at once when there is none, or when it was not
// launched this way). Every CTA waits, so a kernel completes only after the
// one before it: the ordering stays transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Programmatic dependent launches on (1) or off (0, every kernel waits for
// the one before it as a plain stream launch does), for A/B measurements.
#ifndef RMSNORM_PDL
#define RMSNORM_PDL 1
#endif

// Launch configuration: grid, block, dynamic shared memory, stream, the
// cluster size (0: no cluster attribute; 1: clusters of one CTA, for the
// kernels whose bulk copies name a shared::cluster destination) and the
// programmatic dependency (on unless `pdl` is false). Used in place (its
// attribute array is referenced by the configuration), never copied.
struct LaunchCfg {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    LaunchCfg(unsigned grid, unsigned block, size_t smem, cudaStream_t s, unsigned cs = 0, bool pdl = true) {
        cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(block);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        unsigned n = 0;
        if (cs > 0) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = cs;
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        if (pdl && RMSNORM_PDL) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        cfg.attrs = attr;
        cfg.numAttrs = n;
    }
    LaunchCfg(const LaunchCfg &) = delete;
    LaunchCfg &operator=(const LaunchCfg &) = delete;
};

// ----------------------------------------------------------- 16-byte I/O --
// Row data is read once: ld.global.cs (streaming, evict-first). The weight
// is shared by every row: the read-only path. Writes are plain stores.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }
__device__ __forceinline__ uint4 ld_keep(const uint4 *p) { return __ldg(p); }
__device__ __forceinline__ void st_chunk(uint4 *p, const uint4 &v) { *p = v; }

// ------------------------------------------------- chunk <-> fp32 pairs --
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t u) {
    // bf16 is the upper half of a binary32: widening is a shift / mask.
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf16x2(float2 v) {
    __nv_bfloat162 b = __float22bfloat162_rn(v);  // round to nearest even
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ float2 f16x2_to_f2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);  // exact widening
}
__device__ __forceinline__ uint32_t f2_to_f16x2(float2 v) {
    __half2 h = __float22half2_rn(v);  // round to nearest even
    return *reinterpret_cast<uint32_t *>(&h);
}

template <typename T> __device__ __forceinline__ void unpack(const uint4 &c, float2 (&p)[Elem<T>::NP]);
template <> __device__ __forceinline__ void unpack<__half>(const uint4 &c, float2 (&p)[4]) {
    p[0] = f16x2_to_f2(c.x);
    p[1] = f16x2_to_f2(c.y);
    p[2] = f16x2_to_f2(c.z);
    p[3] = f16x2_to_f2(c.w);
}
template <> __device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4 &c, float2 (&p)[4]) {
    p[0] = bf16x2_to_f2(c.x);
    p[1] = bf16x2_to_f2(c.y);
    p[2] = bf16x2_to_f2(c.z);
    p[3] = bf16x2_to_f2(c.w);
}
template <> __device__ __forceinline__ void unpack<float>(const uint4 &c, float2 (&p)[2]) {
    p[0] = make_float2(__uint_as_float(c.x), __uint_as_float(c.y));
    p[1] = make_float2(__uint_as_float(c.z), __uint_as_float(c.w));
}

template <typename T> __device__ __forceinline__ uint4 pack(const float2 (&p)[Elem<T>::NP]);
template <> __device__ __forceinline__ uint4 pack<__half>(const float2 (&p)[4]) {
    return make_uint4(f2_to_f16x2(p[0]), f2_to_f16x2(p[1]), f2_to_f16x2(p[2]), f2_to_f16x2(p[3]));
}
template <> __device__ __forceinline__ uint4 pack<__nv_bfloat16>(const float2 (&p)[4]) {
    return make_uint4(f2_to_bf16x2(p[0]), f2_to_bf16x2(p[1]), f2_to_bf16x2(p[2]), f2_to_bf16x2(p[3]));
}
template <> __device__ __forceinline__ uint4 pack<float>(const float2 (&p)[2]) {
    return make_uint4(__float_as_uint(p[0].x), __float_as_uint(p[0].y), __float_as_uint(p[1].x),
                      __float_as_uint(p[1].y));
}

// Weight values for activation chunk c (chunk = 16 bytes of activations).
// The weight is stored either in the activations' type (one 16-byte load)
// or in fp32 next to 2-byte activations (two 16-byte loads); the pairs come
// out in the chunk's (even, odd) column order either way.
template <typename T, typename TW>
__device__ __forceinline__ void load_w_chunk(const void *w, int c, float2 (&wv)[Elem<T>::NP]) {
    if constexpr (std::is_same<T, TW>::value) {
        unpack<T>(ld_keep(reinterpret_cast<const uint4 *>(w) + c), wv);
    } else {
        static_assert(std::is_same<TW, float>::value && Elem<T>::E == 8, "fp32 weight with 2-byte activations");
        const uint4 *w4 = reinterpret_cast<const uint4 *>(w) + 2 * c;
        float2 a[2], b[2];
        unpack<float>(ld_keep(w4), a);
        unpack<float>(ld_keep(w4 + 1), b);
        wv[0] = a[0];
        wv[1] = a[1];
        wv[2] = b[0];
        wv[3] = b[1];
    }
}

// Scalar element access for the generic kernels.
__device__ __forceinline__ float load_elem(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ float load_elem(const __half *p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ float load_w(const float *p, int64_t i) { return __ldg(p + i); }
__device__ __forceinline__ float load_w(const __half *p, int64_t i) { return __half2float(__ldg(p + i)); }
__device__ __forceinline__ float load_w(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(__ldg(p + i));
}
__device__ __forceinline__ void store_elem(float *p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_elem(__half *p, int64_t i, float v) { p[i] = __float2half_rn(v); }
__device__ __forceinline__ void store_elem(__nv_bfloat16 *p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}
// Value a store of v would hold (round to the storage type).
__device__ __forceinline__ float round_to(float v, const float *) { return v; }
__device__ __forceinline__ float round_to(float v, const __half *) { return __half2float(__float2half_rn(v)); }
__device__ __forceinline__ float round_to(float v, const __nv_bfloat16 *) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

// ----------------------------------------------- rows at a common offset --
// When every array of a call starts `peel` elements past a 16-byte boundary
// (0 < peel < E) and rows are whole 16-byte chunks long (C of them), the
// host moves each pointer back by `peel` elements, to the boundary. Row r
// then covers C + 1 aligned chunks from (base + r C): its first `E - peel`
// elements are the last ones of aligned chunk 0 and its last `peel` ones
// the first ones of aligned chunk C. The kernels keep C chunks per row,
// exactly as for aligned rows: chunks 1 .. C-1 are aligned chunks 1 .. C-1,
// and chunk 0 is "wrapped": elements l < peel come from aligned chunk C
// (columns N - peel + l), elements l >= peel from aligned chunk 0 (columns
// l - peel). Each of those two reads stays inside the aligned 16 bytes that
// hold one of the row's elements; their stores write the row's own
// elements one by one. A thread's wrapped chunk therefore holds columns
// (16-byte lane l) -> (l - peel) mod N, and so does a partial row written
// from it: the finalizer rotates columns back.

// Keep the row's elements of aligned chunk 0 (`first`: l >= peel) or of
// aligned chunk C (l < peel); the others become zero bits.
template <typename T>
__device__ __forceinline__ uint4 keep_part(uint4 v, bool first, int peel) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int l0 = 2 * k, l1 = 2 * k + 1;  // low half-word: element 2k
            const bool k0 = first ? l0 >= peel : l0 < peel;
            const bool k1 = first ? l1 >= peel : l1 < peel;
            w[k] &= (k0 ? 0x0000ffffu : 0u) | (k1 ? 0xffff0000u : 0u);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const bool keep = first ? k >= peel : k < peel;
            w[k] = keep ? w[k] : 0u;
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The wrapped chunk from aligned chunks 0 (`head`) and C (`tail`).
template <typename T>
__device__ __forceinline__ uint4 wrap_chunk(uint4 head, uint4 tail, int peel) {
    const uint4 a = keep_part<T>(head, true, peel), b = keep_part<T>(tail, false, peel);
    return make_uint4(a.x | b.x, a.y | b.y, a.z | b.z, a.w | b.w);
}

// Store the row's elements of `v` into aligned chunk 0 (`first`) or C.
template <typename T>
__device__ __forceinline__ void store_part(uint4 *p, uint4 v, bool first, int peel) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (sizeof(T) == 2) {
        uint16_t *q = reinterpret_cast<uint16_t *>(p);
#pragma unroll
        for (int l = 0; l < 8; ++l)
            if (first ? l >= peel : l < peel) q[l] = (uint16_t)(w[l >> 1] >> (16 * (l & 1)));
    } else {
        uint32_t *q = reinterpret_cast<uint32_t *>(p);
#pragma unroll
        for (int l = 0; l < 4; ++l)
            if (first ? l >= peel : l < peel) q[l] = w[l];
    }
}

// The rows' common offset as a vectorised kernel sees it. Each such kernel
// is compiled twice: PEEL = false serves aligned rows, and there the offset
// is the constant 0, so every wrapped-chunk test, load, merge and store
// below folds away and the kernel is the plain aligned one (registers and
// instructions included); PEEL = true reads it from the parameters.
template <bool PEEL, typename Params>
__device__ __forceinline__ int peel_of(const Params &p) {
    return PEEL ? p.peel : 0;
}

// The helpers below take `edge`: the chunk is the row's wrapped chunk 0
// (peel != 0 and c == 0). Kernels pass it as `v == 0 && e0`, v the
// compile-time slot of the chunk among a thread's and e0 whether the
// thread's slot 0 is chunk 0 of a peeled row, so that the test folds away
// for every other slot.

// The wrapped chunk's two loads and its element stores are kept out of
// line: only the one thread holding a peeled row's chunk 0 calls them, and
// inlined the compiler would predicate them into every thread's chunk 0.
template <typename T>
__device__ __noinline__ uint4 ld_wrapped(const uint4 *row, int C, int peel) {
    return wrap_chunk<T>(ld_stream(row), ld_stream(row + C), peel);
}
template <typename T>
__device__ __noinline__ void st_wrapped(uint4 *row, int C, int peel, uint4 v) {
    store_part<T>(row, v, true, peel);
    store_part<T>(row + C, v, false, peel);
}

// Chunk c of the row starting at `row` (C chunks a row): a streaming load,
// or for the wrapped chunk two loads merged.
template <typename T>
__device__ __forceinline__ uint4 ld_row_chunk(const uint4 *row, int c, int C, int peel, bool edge) {
    if (edge) return ld_wrapped<T>(row, C, peel);
    return ld_stream(row + c);
}

// Store chunk c of the row starting at `row`: whole, or the wrapped chunk's
// two parts element by element.
template <typename T>
__device__ __forceinline__ void st_row_chunk(uint4 *row, int c, int C, int peel, bool edge, const uint4 &v) {
    if (edge)
        st_wrapped<T>(row, C, peel, v);
    else
        row[c] = v;
}

// load_w_chunk for chunk c of a row of C chunks (the weight vector shares
// the rows' offset: its chunk 0 is wrapped as well). Rows at a common
// offset take the weight in the activations' type; the fp32-weight kernels
// always see peel == 0.
template <typename T, typename TW>
__device__ __forceinline__ void load_w_chunk_row(const void *w, int c, int C, int peel, bool edge,
                                                 float2 (&wv)[Elem<T>::NP]) {
    if constexpr (std::is_same<T, TW>::value) {
        const uint4 *w4 = reinterpret_cast<const uint4 *>(w);
        unpack<T>(edge ? wrap_chunk<T>(ld_keep(w4), ld_keep(w4 + C), peel) : ld_keep(w4 + c), wv);
    } else {
        load_w_chunk<T, TW>(w, c, wv);
    }
}
// The raw 16 bytes of the weight's chunk c (weight in the activations' type).
template <typename T>
__device__ __forceinline__ uint4 ld_w_raw(const void *w, int c, int C, int peel, bool edge) {
    const uint4 *w4 = reinterpret_cast<const uint4 *>(w);
    return edge ? wrap_chunk<T>(ld_keep(w4), ld_keep(w4 + C), peel) : ld_keep(w4 + c);
}

// --------------------------------------------------- peeled generic rows --
// The generic kernels take rows of any length and alignment. A row is split
// by the address of its x (or h) row: `head` elements up to the first
// 16-byte boundary, `nb` whole 16-byte chunks, then a tail from element
// `tail0`; each thread visits its share in that order, so the row's
// arithmetic depends on that address and N alone. Each other array of the
// row is moved a chunk at a time with one 16-byte access where it shares
// x's address mod 16, and element by element otherwise (the same values).
__device__ __forceinline__ uint32_t addr_mod16(const void *p) {
    return (uint32_t)reinterpret_cast<uintptr_t>(p) & 15u;
}

struct RowSplit {
    int head, nb, tail0;
};

template <typename T>
__device__ __forceinline__ RowSplit row_split(const T *row, int N, bool peel) {
    RowSplit r{N, 0, N};
    if (peel) {
        const int h = (int)(((16u - addr_mod16(row)) & 15u) / sizeof(T));
        r.head = h < N ? h : N;
        r.nb = (N - r.head) / Elem<T>::E;
        r.tail0 = r.head + r.nb * Elem<T>::E;
    }
    return r;
}

// Chunk of a row at column j0 as fp32 pairs, and back (round to nearest
// even, as the element stores do).
template <typename T>
__device__ __forceinline__ void load_chunk_at(const T *p, int64_t j0, bool vec, float2 (&v)[Elem<T>::NP]) {
    if (vec) {
        unpack<T>(*reinterpret_cast<const uint4 *>(p + j0), v);
    } else {
#pragma unroll
        for (int q = 0; q < Elem<T>::NP; ++q) v[q] = make_float2(load_elem(p, j0 + 2 * q), load_elem(p, j0 + 2 * q + 1));
    }
}
template <typename T>
__device__ __forceinline__ void store_chunk_at(T *p, int64_t j0, bool vec, const float2 (&v)[Elem<T>::NP]) {
    if (vec) {
        *reinterpret_cast<uint4 *>(p + j0) = pack<T>(v);
    } else {
#pragma unroll
        for (int q = 0; q < Elem<T>::NP; ++q) {
            store_elem(p, j0 + 2 * q, v[q].x);
            store_elem(p, j0 + 2 * q + 1, v[q].y);
        }
    }
}

// This thread's share of a split row, in a fixed order: the head's columns
// one by one, the 16-byte chunks (by first column), then the tail's columns.
template <int E, typename FE, typename FC>
__device__ __forceinline__ void row_visit(const RowSplit &sp, int N, FE &&elem, FC &&chunk) {
    for (int j = threadIdx.x; j < sp.head; j += blockDim.x) elem(j);
    for (int c = threadIdx.x; c < sp.nb; c += blockDim.x) chunk(sp.head + c * E);
    for (int j = sp.tail0 + threadIdx.x; j < N; j += blockDim.x) elem(j);
}

// The weight values of the chunk starting at column j0: one or two 16-byte
// loads when w + j0 is 16-byte aligned, else element loads.
template <typename T, typename TW>
__device__ __forceinline__ void w_chunk_at(const TW *w, int j0, float2 (&wv)[Elem<T>::NP]) {
    if (addr_mod16(w + j0) == 0) {
        load_w_chunk<T, TW>(w + j0, 0, wv);
    } else {
#pragma unroll
        for (int q = 0; q < Elem<T>::NP; ++q) wv[q] = make_float2(load_w(w, j0 + 2 * q), load_w(w, j0 + 2 * q + 1));
    }
}

// ------------------------------------------------------- pair arithmetic --
// Two implementations with identical IEEE results lane by lane: packed
// f32x2 instructions (one instruction for two fp32 lanes on data-centre
// Blackwell, Liger-Kernel PR #1388 section 2) and per-lane fp32 intrinsics
// that the compiler may not contract. The kernels use one even/odd pairing
// for both, so the packed and scalar variants agree bit for bit.
template <bool PACKED> struct Pair;

template <> struct Pair<true> {
    static __device__ __forceinline__ float2 fma(float2 a, float2 b, float2 c) {
        float2 d;
        asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
            "mov.b64 ra, {%2, %3};\n\t"
            "mov.b64 rb, {%4, %5};\n\t"
            "mov.b64 rc, {%6, %7};\n\t"
            "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
            "mov.b64 {%0, %1}, rd;\n\t}"
            : "=f"(d.x), "=f"(d.y)
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
        return d;
    }
    static __device__ __forceinline__ float2 mul(float2 a, float2 b) {
        float2 d;
        asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
            "mov.b64 ra, {%2, %3};\n\t"
            "mov.b64 rb, {%4, %5};\n\t"
            "mul.rn.f32x2 rd, ra, rb;\n\t"
            "mov.b64 {%0, %1}, rd;\n\t}"
            : "=f"(d.x), "=f"(d.y)
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
        return d;
    }
    static __device__ __forceinline__ float2 add(float2 a, float2 b) {
        float2 d;
        asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
            "mov.b64 ra, {%2, %3};\n\t"
            "mov.b64 rb, {%4, %5};\n\t"
            "add.rn.f32x2 rd, ra, rb;\n\t"
            "mov.b64 {%0, %1}, rd;\n\t}"
            : "=f"(d.x), "=f"(d.y)
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
        return d;
    }
};

template <> struct Pair<false> {
    static __device__ __forceinline__ float2 fma(float2 a, float2 b, float2 c) {
        return make_float2(__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y));
    }
    static __device__ __forceinline__ float2 mul(float2 a, float2 b) {
        return make_float2(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y));
    }
    static __device__ __forceinline__ float2 add(float2 a, float2 b) {
        return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
    }
};

// --------------------------------------------------------- team reduce --
// The combining operation of a reduction: fp32 addition (row sums) or the
// maximum (a row's largest magnitude, for a quantised output's scale).
struct OpAdd {
    static __device__ __forceinline__ float f(float a, float b) { return __fadd_rn(a, b); }
};
struct OpMax {
    static __device__ __forceinline__ float f(float a, float b) { return fmaxf(a, b); }
};

// Combination of the S slots red[0..S) (S a power of two), computed by
// every warp: lane i starts from red[i mod S] (S <= 32) or from
// red[i] + red[i+32] + ... (S > 32), then a butterfly over min(S, 32)
// lanes. Every lane of every warp ends with the same bits (same values,
// same association).
template <int S, class Op = OpAdd>
__device__ __forceinline__ float sum_slots(const float *red, int lane) {
    static_assert((S & (S - 1)) == 0, "slot count must be a power of two");
    float s;
    if constexpr (S <= 32) {
        s = red[lane & (S - 1)];
    } else {
        s = red[lane];
#pragma unroll
        for (int j = 1; j < S / 32; ++j) s = Op::f(s, red[lane + 32 * j]);
    }
    constexpr int WIDTH = S < 32 ? S : 32;
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) s = Op::f(s, __shfl_xor_sync(0xffffffffu, s, o));
    return s;
}

// All-reduce of one float over a team of TPR consecutive threads
// (TPR a power of two). Within a warp: xor butterfly; every lane ends with
// the same bits because fp32 addition is commutative. Across the warps of
// a team: lane 0 of each warp writes `red[warp]`, a CTA barrier, then every
// warp combines the W slots with a second butterfly (sum_slots). The
// barrier is CTA-wide, so every thread of the CTA must call this the same
// number of times.
template <int TPR, class Op = OpAdd>
__device__ __forceinline__ float team_allreduce(float v, float *red, int t) {
    constexpr int WIDTH = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) v = Op::f(v, __shfl_xor_sync(0xffffffffu, v, o));
    if constexpr (TPR > 32) {
        constexpr int W = TPR / 32;
        if ((t & 31) == 0) red[t >> 5] = v;
        __syncthreads();
        v = sum_slots<W, Op>(red, t & 31);
    }
    return v;
}

// CTA-wide sum for the generic kernels (blockDim.x a multiple of 32, at most
// 1024). Same ordering rules as team_allreduce; `red` holds 32 floats.
template <class Op = OpAdd>
__device__ __forceinline__ float cta_allreduce(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = Op::f(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int W = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = red[0];
    for (int i = 1; i < W; ++i) s = Op::f(s, red[i]);
    __syncthreads();  // red is reused by the next call
    return s;
}

// ------------------------------------------------------------- clusters --
// A row can be shared by the CTAs of a thread-block cluster: each CTA keeps
// its slice in registers and the per-warp partial sums are exchanged
// through distributed shared memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Barrier over every thread of every CTA in the cluster. Writes made to
// (distributed) shared memory before it are visible to all after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store v at the address of `local` (a shared variable of this CTA) in the
// shared memory of cluster CTA `cta`.
__device__ __forceinline__ void st_cluster(float *local, uint32_t cta, float v) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(cta));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(r), "f"(v) : "memory");
}

// ------------------------------------------------------------ mbarriers --
// Used by the backward's cluster rows: partial sums travel to the peers'
// shared memory with st.async, whose completion is counted in bytes on an
// mbarrier of the receiving CTA. The asynchronous store carries its own
// release, so, unlike a cluster barrier, the sender never has to wait for
// its earlier global stores (the previous row's dx) to become visible.
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival that also announces `bytes` of incoming asynchronous data.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// True once the phase with the given parity has completed; acquire at
// cluster scope, so data delivered by the peers' st.async is visible.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Bounded wait: gives up after `limit` polls (each poll may suspend the
// thread for a short, hardware-chosen time) and reports false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// 16-byte load from this CTA's shared memory, addressed in the shared
// window (so it never takes the generic load path).
__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// 16-byte store into this CTA's shared memory (shared-window address).
__device__ __forceinline__ void sts128(void *p, const uint4 &v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// A stage's rows' chunk 0 wrapped in place (rows at a common offset, for
// the kernels that read a stage more than once): each of the `nb` row
// buffers (`stride` slots apart) holds aligned chunks 0 .. Cst of its
// slice, and its slot 0 becomes the wrapped chunk from slots 0 and Cst.
// Called once a row by the thread that alone reads slot 0 (thread 0 of the
// CTA holding chunk 0), after the stage's copies landed and before it reads
// the slot. The proxy fence orders the writes before the bulk copy that
// later refills the stage, whichever thread issues it.
template <typename T>
__device__ __noinline__ void wrap_staged(uint4 *buf, int stride, int nb, int Cst, int peel) {
    for (int b = 0; b < nb; ++b) {
        uint4 *r = buf + b * stride;
        sts128(r, wrap_chunk<T>(lds128(r), lds128(r + Cst), peel));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk copy (the TMA engine's 1-D form) of `bytes` from global memory into
// this CTA's shared memory, counted in bytes on `bar`. Both addresses
// 16-byte aligned, `bytes` a multiple of 16. The kernel is launched as a
// cluster (of one CTA), so the shared::cluster destination is this CTA's.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Asynchronous copy of one 4-byte word from global into this CTA's shared
// memory (both 4-byte aligned). cp_async_arrive_noinc makes `bar` receive
// one arrival once every asynchronous copy this thread has issued so far
// has landed; the arrival is one of those counted at mbar_init.
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The 16-byte cover of `bytes` bytes at address a: the whole 16-byte
// blocks that hold them, starting `off` = a mod 16 bytes before a, a
// multiple of 16 bytes long (what a bulk copy of a row at any alignment
// moves). A 16-byte block never crosses a page, so a block that holds any
// byte of an allocation can be read without a fault; the bytes of the
// cover outside [a, a + bytes) are copied and never used.
struct Cover {
    const char *src;
    uint32_t off, bytes;
};
__device__ __forceinline__ Cover cover16(const void *a, uint32_t bytes) {
    const uintptr_t u = reinterpret_cast<uintptr_t>(a);
    const uint32_t off = (uint32_t)u & 15u;
    return Cover{reinterpret_cast<const char *>(u - off), off, (off + bytes + 15u) & ~15u};
}

// Store v at the address of `local_slot` in cluster CTA `cta` and count 4
// bytes on that CTA's barrier at the address of `local_bar`.
__device__ __forceinline__ void st_async_cluster(float *local_slot, uint64_t *local_bar, uint32_t cta, float v) {
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local_slot)), "r"(cta));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(local_bar)), "r"(cta));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
                 "r"(__float_as_uint(v)), "r"(rb)
                 : "memory");
}

// All-reduce of one float over a row shared by the CS CTAs of a cluster
// (one team of TPR >= 32 threads per CTA), in two halves so that work that
// does not need the result can run while the cluster barrier completes:
//  begin: warp butterfly; lane 0 of each warp stores its warp sum into slot
//         [rank * W + warp] of every CTA of the cluster; barrier arrive.
//  end:   barrier wait; every warp combines the CS * W slots (sum_slots),
//         so every thread of the cluster obtains the same bits.
// `red` holds CS * W floats; callers alternate buffers between rows.
template <int TPR, int CS, class Op = OpAdd>
__device__ __forceinline__ void cluster_allreduce_begin(float v, float *red, int t, uint32_t rank) {
    static_assert(TPR >= 32, "cluster rows need whole warps");
    constexpr int W = TPR / 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = Op::f(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((t & 31) == 0) {
#pragma unroll
        for (int c = 0; c < CS; ++c) st_cluster(&red[rank * W + (t >> 5)], (uint32_t)c, v);
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

template <int TPR, int CS, class Op = OpAdd>
__device__ __forceinline__ float cluster_allreduce_end(const float *red, int t) {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    return sum_slots<CS *(TPR / 32), Op>(red, t & 31);
}

template <int TPR, int CS, class Op = OpAdd>
__device__ __forceinline__ float cluster_allreduce(float v, float *red, int t, uint32_t rank) {
    cluster_allreduce_begin<TPR, CS, Op>(v, red, t, rank);
    return cluster_allreduce_end<TPR, CS, Op>(red, t);
}

// ------------------------------------------------- two sums at once --
// The same reductions on a pair of values (the LayerNorm backward's sum of
// g and sum of g (x - mean); the E4M3 forward's sum of squares and row
// max), each component combined with its own op (PairOp) exactly as the
// single-value versions combine theirs, so each component has their bits.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y)); }
__device__ __forceinline__ float2 shfl_xor2(float2 v, int o) {
    return make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o));
}
template <class OA = OpAdd, class OB = OpAdd>
struct PairOp {
    static __device__ __forceinline__ float2 f(float2 a, float2 b) { return make_float2(OA::f(a.x, b.x), OB::f(a.y, b.y)); }
};
using SumMax = PairOp<OpAdd, OpMax>;  // (sum of squares, max |value|)

template <int S, class PO = PairOp<>>
__device__ __forceinline__ float2 sum_slots2(const float2 *red, int lane) {
    static_assert((S & (S - 1)) == 0, "slot count must be a power of two");
    float2 s;
    if constexpr (S <= 32) {
        s = red[lane & (S - 1)];
    } else {
        s = red[lane];
#pragma unroll
        for (int j = 1; j < S / 32; ++j) s = PO::f(s, red[lane + 32 * j]);
    }
    constexpr int WIDTH = S < 32 ? S : 32;
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) s = PO::f(s, shfl_xor2(s, o));
    return s;
}

template <int TPR, class PO = PairOp<>>
__device__ __forceinline__ float2 team_allreduce2(float2 v, float2 *red, int t) {
    constexpr int WIDTH = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) v = PO::f(v, shfl_xor2(v, o));
    if constexpr (TPR > 32) {
        constexpr int W = TPR / 32;
        if ((t & 31) == 0) red[t >> 5] = v;
        __syncthreads();
        v = sum_slots2<W, PO>(red, t & 31);
    }
    return v;
}

template <class PO = PairOp<>>
__device__ __forceinline__ float2 cta_allreduce2(float2 v, float2 *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = PO::f(v, shfl_xor2(v, o));
    const int W = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float2 s = red[0];
    for (int i = 1; i < W; ++i) s = PO::f(s, red[i]);
    __syncthreads();  // red is reused by the next call
    return s;
}

// cluster_allreduce on a pair (8-byte distributed shared-memory stores).
__device__ __forceinline__ void st_cluster2(float2 *local, uint32_t cta, float2 v) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(cta));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(r), "f"(v.x), "f"(v.y) : "memory");
}
template <int TPR, int CS, class PO = PairOp<>>
__device__ __forceinline__ float2 cluster_allreduce2(float2 v, float2 *red, int t, uint32_t rank) {
    static_assert(TPR >= 32, "cluster rows need whole warps");
    constexpr int W = TPR / 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = PO::f(v, shfl_xor2(v, o));
    if ((t & 31) == 0) {
#pragma unroll
        for (int c = 0; c < CS; ++c) st_cluster2(&red[rank * W + (t >> 5)], (uint32_t)c, v);
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    return sum_slots2<CS * W, PO>(red, t & 31);
}

// st_async_cluster for a pair: 8 bytes counted on the receiver's barrier.
__device__ __forceinline__ void st_async_cluster2(float2 *local_slot, uint64_t *local_bar, uint32_t cta, float2 v) {
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local_slot)), "r"(cta));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(local_bar)), "r"(cta));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(ra),
                 "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(rb)
                 : "memory");
}

// ------------------------------------------------------------ E4M3 out --
// Two fp32 values to two E4M3 codes (nearest-even, saturating to +-448):
// a.x in the low byte. Four values packed into 32 bits, lowest first.
__device__ __forceinline__ uint32_t e4m3x4(float2 a, float2 b) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}
__device__ __forceinline__ uint8_t e4m3x1(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

}  // namespace rmsn
