// Row kernels for RMSNorm and fused residual-add RMSNorm on sm_103a.
//
// Arithmetic (Kernscope, "Numerical contract"): every element is widened to FP32, the sum of
// squares is accumulated in FP32 (per-thread FMA chain, then a warp-shuffle tree, then a fixed-
// order sum over warps), mean = ss / fp32(H) is one IEEE division, scale is the correctly
// rounded FP32 reciprocal square root of mean + eps, and each output is ((v * scale) * w)
// rounded to nearest even into the element type. The fused kernels form s = fp32(x) + fp32(r)
// with one FP32 add, store cast(s) into the residual, and normalise the unrounded s.
//
// Memory (the op moves 2*H*e bytes per row plain, 4*H*e fused, and does ~4 flops per element,
// so HBM bandwidth bounds it; no tensor cores apply): each row is read once with 16-byte
// coalesced loads (streaming, evict-first) into registers, written once with 16-byte
// streaming stores; the weight slice a thread needs is loaded once and kept in registers for
// every row it touches; the grid is persistent. Teams either load their next row before they
// reduce the current one (prefetch) or load each row in turn with fewer registers and more
// resident warps; the launch heuristic picks per width. The staged kernel instead streams whole
// rows (or, split over a cluster, row slices) into a ring of shared-memory stages with bulk
// asynchronous copies (one issuing thread, an mbarrier per stage), so several rows per CTA are
// in flight without spending registers on them.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include "ks_internal.h"
#include "ks_ptx.cuh"

namespace ks {

// ------------------------------------------------------------------------ element traits

template <typename T>
struct Elem;

// Vectors are unpacked to FP32 pairs (element 2i, 2i + 1; unpack2/pack2), and the row kernels run
// each element step on a pair (pair_add, pair_mul, pair_fma below). kPairMath: the step is one
// packed FP32 instruction (FADD2/FMUL2/FFMA2, sm_100 and later); otherwise two scalar operations.
// Either way each element gets one IEEE round-to-nearest operation, so the two forms give the
// same bits, and the packed one takes half the floating-point instructions. Measured on GB300 for
// bf16: RMSNorm rows of 1024..8192 elements 0-1 point of the copy peak faster, LayerNorm rows of
// 768..4096 vectors 4-8 points. fp16 (whose conversions are not plain shifts) measured between 2
// points slower and 1 faster, and fp32 rows (2 pairs per vector) gained nothing, so those two
// keep scalar operations.
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    static constexpr bool kPairMath = true;
    __device__ __forceinline__ static void unpack(const uint4 &v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            memcpy(&w[i], &h, sizeof(uint32_t));
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    // as FP32 pairs (element 2i, 2i + 1) for the packed FP32 instructions
    __device__ __forceinline__ static void unpack2(const uint4 &v, float2 (&f)[4]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    }
    __device__ __forceinline__ static uint4 pack2(const float2 (&f)[4]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __float22bfloat162_rn(f[i]);
            memcpy(&w[i], &h, sizeof(uint32_t));
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ static float load1(const void *p, int64_t i) {
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    }
    __device__ __forceinline__ static void store1(void *p, int64_t i, float v) {
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    }
};

template <>
struct Elem<__half> {
    static constexpr int kPerVec = 8;
    static constexpr bool kPairMath = false;
    __device__ __forceinline__ static void unpack(const uint4 &v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], sizeof(uint32_t));
            const float2 p = __half22float2(h);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            memcpy(&w[i], &h, sizeof(uint32_t));
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ static void unpack2(const uint4 &v, float2 (&f)[4]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], sizeof(uint32_t));
            f[i] = __half22float2(h);
        }
    }
    __device__ __forceinline__ static uint4 pack2(const float2 (&f)[4]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __float22half2_rn(f[i]);
            memcpy(&w[i], &h, sizeof(uint32_t));
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ __forceinline__ static float load1(const void *p, int64_t i) {
        return __half2float(static_cast<const __half *>(p)[i]);
    }
    __device__ __forceinline__ static void store1(void *p, int64_t i, float v) {
        static_cast<__half *>(p)[i] = __float2half_rn(v);
    }
};

template <>
struct Elem<float> {
    static constexpr int kPerVec = 4;
    static constexpr bool kPairMath = false;
    __device__ __forceinline__ static void unpack(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static void unpack2(const uint4 &v, float2 (&f)[2]) {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    __device__ __forceinline__ static uint4 pack2(const float2 (&f)[2]) {
        return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                          __float_as_uint(f[1].y));
    }
    __device__ __forceinline__ static float load1(const void *p, int64_t i) {
        return static_cast<const float *>(p)[i];
    }
    __device__ __forceinline__ static void store1(void *p, int64_t i, float v) {
        static_cast<float *>(p)[i] = v;
    }
};

// ---------------------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Sum over a team: kTeam lanes of a warp (8, 16 or 32; an aligned group of lanes, so the xor
// offsets below kTeam stay inside it; shuffles only, every lane of the warp taking part) or, with
// kTeam = 0, the whole CTA. Every thread of the team returns the same value (the per-warp sums
// are added in warp order). `red` is one of two alternating 32-float slots: a warp can only
// write a slot again after passing the barrier of the row in between, which every warp reaches
// only after it has read this row's slot, so one barrier per row suffices.
template <int kTeam>
__device__ __forceinline__ float team_sum(float v, float *red) {
    if constexpr (kTeam == 8 || kTeam == 16) {
#pragma unroll
        for (int o = kTeam / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        return v;
    }
    v = warp_sum(v);
    if (kTeam == 32) return v;
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    float s = 0.0f;
    const int nw = blockDim.x >> 5;
    for (int i = 0; i < nw; ++i) s += red[i];
    return s;
}

__device__ __forceinline__ float row_scale(float ss, float h, float eps) {
    return __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, h), eps));
}

// Four independent FMA chains per thread (element e feeds chain e % 4), added pairwise at the end:
// a single chain would serialise on the FMA latency.
struct SumSq {
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    template <int N>
    __device__ __forceinline__ void add(const float (&f)[N]) {
#pragma unroll
        for (int e = 0; e < N; ++e) a[e & 3] = __fmaf_rn(f[e], f[e], a[e & 3]);
    }
    __device__ __forceinline__ float total() const {
        return __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
    }
};

// ------------------------------------------------------------- element steps on FP32 pairs

template <bool kPair>
__device__ __forceinline__ float2 pair_add(float2 a, float2 b) {
    if constexpr (kPair) return __fadd2_rn(a, b);
    else return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
}

template <bool kPair>
__device__ __forceinline__ float2 pair_mul(float2 a, float2 b) {
    if constexpr (kPair) return __fmul2_rn(a, b);
    else return make_float2(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y));
}

template <bool kPair>
__device__ __forceinline__ float2 pair_fma(float2 a, float2 b, float2 c) {
    if constexpr (kPair) return __ffma2_rn(a, b, c);
    else return make_float2(__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y));
}

// The four FMA chains of SumSq held as two pairs: element e feeds chain e % 4, which is lane
// e % 2 of pair (e / 2) % 2; the total adds the chains in the same order.
template <bool kPair>
struct PairSumSq {
    float2 a[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
    template <int P>
    __device__ __forceinline__ void add(const float2 (&f)[P]) {
#pragma unroll
        for (int i = 0; i < P; ++i) a[i & 1] = pair_fma<kPair>(f[i], f[i], a[i & 1]);
    }
    __device__ __forceinline__ float total() const {
        return __fadd_rn(__fadd_rn(a[0].x, a[0].y), __fadd_rn(a[1].x, a[1].y));
    }
};

// One vector's values: fp32(x), or for the fused op s = fp32(x) + fp32(r) (one FP32 add each).
template <typename T, bool kFused>
__device__ __forceinline__ void row_values(const uint4 &x, const uint4 &r,
                                           float2 (&s)[Elem<T>::kPerVec / 2]) {
    Elem<T>::unpack2(x, s);
    if (kFused) {
        float2 q[Elem<T>::kPerVec / 2];
        Elem<T>::unpack2(r, q);
#pragma unroll
        for (int i = 0; i < Elem<T>::kPerVec / 2; ++i) s[i] = pair_add<Elem<T>::kPairMath>(s[i], q[i]);
    }
}

// One output vector: cast((s * scale) * w), the products in that order.
template <typename T>
__device__ __forceinline__ uint4 scaled_weighted(float2 (&s)[Elem<T>::kPerVec / 2], float scale,
                                                 const uint4 &w) {
    constexpr bool kPair = Elem<T>::kPairMath;
    float2 wf[Elem<T>::kPerVec / 2];
    Elem<T>::unpack2(w, wf);
    const float2 s2 = make_float2(scale, scale);
#pragma unroll
    for (int i = 0; i < Elem<T>::kPerVec / 2; ++i) s[i] = pair_mul<kPair>(pair_mul<kPair>(s[i], s2), wf[i]);
    return Elem<T>::pack2(s);
}

// --------------------------------------------------------------- vectorised row kernel

// Register budget per thread grows with V (current + prefetched rows, weight slice); the
// launch bound keeps the compiler's register cap above it: 256 threads for warp teams, and for
// CTA teams 1024 threads at V <= 2, 512 at V = 4.
template <int V, bool kWarpTeam>
struct VecBound {
    static constexpr int value = kWarpTeam ? 256 : (V <= 2 ? 1024 : 512);
};

template <int V>
__device__ __forceinline__ void load_row(const uint4 *base, int t, int g, int64_t hv,
                                         uint4 (&v)[V]) {
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const int64_t c = t + (int64_t)k * g;
        v[k] = (c < hv) ? __ldcs(base + c) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Hides a register's value from the optimiser, so values derived from it before this point are
// not reused after it (the second pass unpacks the raw 16-bit vectors again instead of keeping
// 8 floats per vector live across the row's reduction).
__device__ __forceinline__ void opaque(uint4 &v) {
    asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
}

// One row of the vector kernel, its vectors already in registers (xc, and rc for the fused op):
// the sum of squares (the fused op also forms s and stores cast(s) into the residual), the team
// reduction through `red`, then normalise, weight, cast and store.
// One row's work for one thread of its team: vectors t, t + g, ... of the row, already loaded
// into xc (and rc). An inactive team (a sub-warp team past the last row, whose warp still takes
// part in the shuffles) computes on zeros and stores nothing.
template <typename T, int V, bool kFused, int kTeam, bool kOpaque>
__device__ __forceinline__ void vec_row(const RowArgs &a, int64_t row, int t, int g,
                                        uint4 (&xc)[V], uint4 (&rc)[V], uint4 (&wv)[V],
                                        float *red, bool active) {
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    const int64_t hv = a.hv;
    uint4 *og = static_cast<uint4 *>(a.out) + row * hv;
    uint4 *rg = kFused ? static_cast<uint4 *>(a.res) + row * hv : nullptr;

    PairSumSq<E::kPairMath> acc;
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const int64_t c = t + (int64_t)k * g;
        if (c < hv) {
            float2 f[P];
            row_values<T, kFused>(xc[k], rc[k], f);
            if (kFused && active) __stcs(rg + c, E::pack2(f));
            acc.add(f);
        }
    }
    const float ss = team_sum<kTeam>(acc.total(), red);
    const float scale = row_scale(ss, (float)a.hidden, a.eps);

    if (kOpaque) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
            opaque(xc[k]);
            if (kFused) opaque(rc[k]);
            opaque(wv[k]);
        }
    }
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const int64_t c = t + (int64_t)k * g;
        if (c < hv && active) {
            float2 f[P];
            row_values<T, kFused>(xc[k], rc[k], f);
            __stcs(og + c, scaled_weighted<T>(f, scale, wv[k]));
        }
    }
}

// One team per row: kTeam lanes of a warp (8, 16 or 32) or, with kTeam = 0, the whole CTA. Row
// r's 16-byte vector c (of hv) is handled by thread c % G of the team (G its size), as its
// (c / G)-th vector. Teams stride over rows by the number of teams in the grid. A warp of 8- or
// 16-lane teams holds several consecutive rows and runs as long as its first row does (the
// shuffles of a team's sum need every lane of the warp), its teams past the last row inactive.
// With kPrefetch a team loads its next row while it works on the current one and moves it into
// the current buffer at the end of the row. (Writing the loop body out twice for two buffers
// used in turn, with no copy, measured 2-20 points slower for bf16 on GB300 and no faster for
// fp16.) Without it, each row is loaded when its turn comes, and the raw vectors are hidden from
// the optimiser across the reduction (measured: this helps without prefetch, costs with it).
template <typename T, int V, bool kFused, int kTeam, bool kPrefetch>
__global__ void __launch_bounds__(VecBound<V, kTeam != 0>::value)
    rows_vec_kernel(const RowArgs a) {
    static_assert(kTeam == 0 || kTeam == 8 || kTeam == 16 || kTeam == 32, "team of 8, 16 or 32 lanes");
    constexpr bool kSub = kTeam == 8 || kTeam == 16;
    __shared__ float red[2][32];

    const int g = kTeam ? kTeam : (int)blockDim.x;
    const int t = kTeam ? (int)(threadIdx.x & (kTeam - 1)) : (int)threadIdx.x;
    const int teams = kTeam ? (int)(blockDim.x / kTeam) : 1;
    const int team = kTeam ? (int)(threadIdx.x / kTeam) : 0;
    const int64_t hv = a.hv;

    const uint4 *xg = static_cast<const uint4 *>(a.x);
    const uint4 *rg = static_cast<const uint4 *>(a.res);

    grid_dependency_wait();
    allow_dependents_launch();
    uint4 wv[V];
    {
        const uint4 *wg = static_cast<const uint4 *>(a.w);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            wv[k] = (c < hv) ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    int64_t row = (int64_t)blockIdx.x * teams + team;
    // the first row of this thread's warp (its own row for warp and CTA teams)
    int64_t lead = kSub ? row - (team & (32 / (kSub ? kTeam : 32) - 1)) : row;
    const int64_t stride = (int64_t)gridDim.x * teams;
    if (!kPrefetch) {
        int parity = 0;
        for (; lead < a.rows; lead += stride, row += stride) {
            const bool active = !kSub || row < a.rows;
            uint4 xc[V], rc[V];
            load_row<V>(xg + row * hv, t, g, active ? hv : 0, xc);
            if (kFused) load_row<V>(rg + row * hv, t, g, active ? hv : 0, rc);
            vec_row<T, V, kFused, kTeam, true>(a, row, t, g, xc, rc, wv, red[parity], active);
            parity ^= 1;
        }
        return;
    }

    uint4 xc[V], rc[V];
#pragma unroll
    for (int k = 0; k < V; ++k) xc[k] = rc[k] = make_uint4(0u, 0u, 0u, 0u);
    if (row < a.rows) {
        load_row<V>(xg + row * hv, t, g, hv, xc);
        if (kFused) load_row<V>(rg + row * hv, t, g, hv, rc);
    }
    int parity = 0;
    while (lead < a.rows) {
        const int64_t next = row + stride;
        uint4 xn[V], rn[V];
#pragma unroll
        for (int k = 0; k < V; ++k) xn[k] = rn[k] = make_uint4(0u, 0u, 0u, 0u);
        if (next < a.rows) {
            load_row<V>(xg + next * hv, t, g, hv, xn);
            if (kFused) load_row<V>(rg + next * hv, t, g, hv, rn);
        }
        vec_row<T, V, kFused, kTeam, false>(a, row, t, g, xc, rc, wv, red[parity],
                                            !kSub || row < a.rows);
        parity ^= 1;
        row = next;
        lead += stride;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            xc[k] = xn[k];
            rc[k] = rn[k];
        }
    }
}

// ------------------------------------------------------------------ two-pass row kernel

// One CTA per row, the row read twice from global memory with 16-byte vectors, U vectors per
// thread in flight in each loop step. The first pass forms the sum of squares (the fused op from
// s = x + r, writing nothing); the second re-reads the row and writes the outputs (the fused op
// recomputes s from the untouched inputs and writes both tensors). The second pass reads from
// L2: the launch sizes the grid so that the rows all CTAs have in flight fit in a share of it,
// so DRAM still sees each element read once and written once. Nothing but the loop bounds the
// row width: no row is held in registers, shared memory or a cluster. The first pass loads
// with the default L2 policy (the row is read again), the second with evict-first (last use).
// Asks L2 for vectors [lo, hi) of a row of x (and of the residual): threads 0.. each issue one
// bulk prefetch of at most 32 KiB.
template <bool kFused>
__device__ __forceinline__ void prefetch_slice(const uint4 *xr, const uint4 *rr, int64_t lo,
                                               int64_t hi, int t) {
    constexpr int64_t kPiece = 2048;  // vectors (32 KiB) per prefetch
    const int64_t c = lo + (int64_t)t * kPiece;
    if (c < hi) {
        const uint32_t bytes = (uint32_t)(((hi - c) < kPiece ? (hi - c) : kPiece) * 16);
        bulk_prefetch_l2(xr + c, bytes);
        if (kFused) bulk_prefetch_l2(rr + c, bytes);
    }
}

template <typename T, bool kFused, int U, int kMaxBlock>
__global__ void __launch_bounds__(kMaxBlock) rows_twopass_kernel(const RowArgs a) {
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    __shared__ float red[2][32];
    const int g = blockDim.x, t = threadIdx.x;
    const int64_t hv = a.hv;
    const int64_t chunk = (int64_t)g * U;
    const uint4 *xg = static_cast<const uint4 *>(a.x);
    uint4 *og = static_cast<uint4 *>(a.out);
    uint4 *rg = static_cast<uint4 *>(a.res);
    const uint4 *wg = static_cast<const uint4 *>(a.w);
    grid_dependency_wait();
    allow_dependents_launch();
    // With prefetch, the whole row is asked into L2 by the copy engine as it starts (see
    // rows_split_kernel).
    const bool prefetch = a.l2_prefetch != 0;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const uint4 *xr = xg + row * hv;
        uint4 *rr = kFused ? rg + row * hv : nullptr;
        if (prefetch) prefetch_slice<kFused>(xr, rr, 0, hv, t);
        PairSumSq<E::kPairMath> acc;
        for (int64_t c0 = t; c0 < hv; c0 += chunk) {
            uint4 xv[U], rv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                xv[u] = c < hv ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
                if (kFused) rv[u] = c < hv ? rr[c] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float2 f[P];
                row_values<T, kFused>(xv[u], rv[u], f);
                acc.add(f);
            }
        }
        const float ss = team_sum<0>(acc.total(), red[parity]);
        parity ^= 1;
        const float scale = row_scale(ss, (float)a.hidden, a.eps);
        uint4 *orow = og + row * hv;
        for (int64_t c0 = t; c0 < hv; c0 += chunk) {
            uint4 xv[U], rv[U], wv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                const bool in = c < hv;
                xv[u] = in ? __ldcs(xr + c) : make_uint4(0u, 0u, 0u, 0u);
                if (kFused) rv[u] = in ? __ldcs(rr + c) : make_uint4(0u, 0u, 0u, 0u);
                wv[u] = in ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                if (c < hv) {
                    float2 f[P];
                    row_values<T, kFused>(xv[u], rv[u], f);
                    if (kFused) __stcs(rr + c, E::pack2(f));
                    __stcs(orow + c, scaled_weighted<T>(f, scale, wv[u]));
                }
            }
        }
    }
}

template <typename T, bool kFused, int U>
const void *pick_twopass(int block) {
    if (block <= 256) return (const void *)rows_twopass_kernel<T, kFused, U, 256>;
    if (block <= 512) return (const void *)rows_twopass_kernel<T, kFused, U, 512>;
    return (const void *)rows_twopass_kernel<T, kFused, U, 1024>;
}

// ------------------------------------------------------- slice sums across a cluster

// A row's slice sums across a cluster of C CTAs (C <= 8) without a cluster barrier per row: each
// CTA's first C threads send the CTA's sum and a flag to every CTA of the cluster with an
// asynchronous shared-memory store that completes as 8 transaction bytes on the receiver's
// mbarrier for that row, and every CTA waits (bounded) on its own barrier for C of them. (A
// cluster barrier's arrive has release semantics: every thread would first wait for its
// earlier global stores to be acknowledged.) Rows alternate between two slots and barriers;
// slot s is used every other row, so the n-th use of a slot completes with parity n & 1. A CTA
// may send a row's sum into a slot only after every thread of it has read that slot's previous
// row, and after its peers set their barriers up (the kernels' start barrier).
struct ClusterSums {
    uint32_t part[2][8][2];  // (sum bits, flag) by sending rank
    uint64_t bar[2];
};

// Thread 0, before the kernel's start cluster barrier.
__device__ __forceinline__ void sums_init(ClusterSums &cs) {
    mbar_init(&cs.bar[0], 1);
    mbar_init(&cs.bar[1], 1);
    fence_mbar_init();
}

// Sends this CTA's sum `v` (valid in threads t < C) with `flag` for slot `slot`, and arms this
// CTA's barrier of the slot for the C sums it receives. Every thread of the CTA must have read
// the slot's previous row before this call.
__device__ __forceinline__ void sums_send(ClusterSums &cs, int slot, float v, uint32_t flag,
                                          int q, int C, int t) {
    if (t == 0) mbar_arrive_expect_tx(&cs.bar[slot], (uint32_t)C * 8u);
    if (t < C)
        st_async_v2(cluster_map(&cs.part[slot][q][0], (uint32_t)t), __float_as_uint(v), flag,
                    cluster_map(&cs.bar[slot], (uint32_t)t));
}

// Waits for slot `slot`'s use with parity `parity`; on return `sum` adds the C sums in rank order
// and the result says whether they all arrived with a zero flag.
__device__ __forceinline__ bool sums_wait(ClusterSums &cs, int slot, uint32_t parity, int C,
                                          float &sum) {
    const bool got = mbar_wait_bounded(&cs.bar[slot], parity);
    uint32_t bad = got ? 0u : 1u;
    float ss = 0.0f;
    for (int r = 0; r < C; ++r) {
        ss += __uint_as_float(cs.part[slot][r][0]);
        bad |= cs.part[slot][r][1];
    }
    sum = ss;
    return bad == 0u;
}

// ------------------------------------------------------------ split two-pass row kernel

// The two-pass scheme with each row split over a thread-block cluster of C CTAs (2..8): CTA q of
// a cluster takes the contiguous slice [q*S, min((q+1)*S, hv)) of S = ceil(hv / C) vectors of
// every row its cluster visits, forms the slice's sum of squares (default L2 policy), and writes
// the slice's outputs from a second read of it (evict-first, from L2). Between the two passes
// the slice sums meet through ClusterSums (asynchronous stores into every CTA's slot for the row,
// completing on its mbarrier), and every CTA adds the C sums in rank order, so all CTAs of a row
// agree on its scale. The first loads of the second pass are issued before the wait, so its
// latency overlaps them. The wait is bounded: after a time-out (here, or a peer's flag) the CTAs
// record KS_FAULT_WAIT_TIMEOUT and keep exchanging flags for the remaining rows without touching
// rows, so every store a peer sends is still awaited before any CTA leaves.
//
// Against one CTA per row this keeps each unit of work to a slice: a persistent grid of whole
// rows leaves SMs idle in its last wave when the rows per CTA are few (10.1 rows per CTA run as
// 11 waves), and the rows a CTA-per-row grid has in flight at once grow with the width until
// the second pass misses L2; here the rows in flight are one per cluster.
// Resident CTAs per SM the launch bound asks of the split kernel: the plain op at 2 vectors per
// step fits in 40 registers, three 512-thread CTAs (six of 256) per SM; the compiler's own
// choice took 64 and two.
template <bool kFused, int U, int kMaxBlock>
struct SplitMinBlocks {
    static constexpr int value = (!kFused && U == 2 && kMaxBlock <= 512) ? 1536 / kMaxBlock : 1;
};

template <typename T, bool kFused, int U, int kMaxBlock>
__global__ void __launch_bounds__(kMaxBlock, (SplitMinBlocks<kFused, U, kMaxBlock>::value))
    rows_split_kernel(const RowArgs a) {
    namespace cg = cooperative_groups;
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    __shared__ float red[32];
    __shared__ __align__(8) ClusterSums cs;

    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int q = (int)cluster.block_rank();
    const int g = blockDim.x, t = threadIdx.x;
    const int64_t hv = a.hv;
    const int64_t S = (hv + C - 1) / C;
    const int64_t lo = q * S;
    const int64_t hi = (lo + S < hv) ? lo + S : hv;
    const int64_t chunk = (int64_t)g * U;
    const float h = (float)a.hidden;
    const uint4 *xg = static_cast<const uint4 *>(a.x);
    uint4 *og = static_cast<uint4 *>(a.out);
    uint4 *rg = static_cast<uint4 *>(a.res);
    const uint4 *wg = static_cast<const uint4 *>(a.w);
    grid_dependency_wait();
    allow_dependents_launch();
    if (t == 0) sums_init(cs);
    // every CTA of the cluster has set its barriers up before any CTA sends to it
    cluster.barrier_arrive();
    cluster.barrier_wait();
    const int64_t nclusters = gridDim.x / C;
    // With prefetch, the whole slice of a row is asked into L2 by the copy engine as the row
    // starts, so the DRAM reads of all the first pass's steps are in flight at once.
    const bool prefetch = a.l2_prefetch != 0;
    bool fault = false;
    uint32_t j = 0;
    int64_t row = blockIdx.x / C;
    for (; row < a.rows; row += nclusters, ++j) {
        const uint4 *xr = xg + row * hv;
        uint4 *rr = kFused ? rg + row * hv : nullptr;
        if (prefetch) prefetch_slice<kFused>(xr, rr, lo, hi, t);
        PairSumSq<E::kPairMath> acc;
        for (int64_t c0 = lo + t; c0 < hi; c0 += chunk) {
            uint4 xv[U], rv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                xv[u] = c < hi ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
                if (kFused) rv[u] = c < hi ? rr[c] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float2 f[P];
                row_values<T, kFused>(xv[u], rv[u], f);
                acc.add(f);
            }
        }
        // the CTA's slice sum (warps in order); every thread has read the slot this row reuses
        // (two rows back) before this barrier
        const float wsum = warp_sum(acc.total());
        if ((t & 31) == 0) red[t >> 5] = wsum;
        __syncthreads();
        float cta = 0.0f;
        if (t < C)
            for (int i = 0; i < (g >> 5); ++i) cta += red[i];
        const int slot = (int)(j & 1u);
        sums_send(cs, slot, cta, 0u, q, C, t);
        uint4 *orow = og + row * hv;
        uint4 xv[U], rv[U], wv[U];
        int64_t c0 = lo + t;
        // the second pass's first loads do not need the scale: issue them before the wait
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = c0 + (int64_t)u * g;
            const bool in = c < hi;
            xv[u] = in ? __ldcs(xr + c) : make_uint4(0u, 0u, 0u, 0u);
            if (kFused) rv[u] = in ? __ldcs(rr + c) : make_uint4(0u, 0u, 0u, 0u);
            wv[u] = in ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        float ss = 0.0f;
        const bool good = sums_wait(cs, slot, (j >> 1) & 1u, C, ss);
        // (red is written again only after the next row's first pass, which every thread
        // reaches after this barrier)
        if (!__syncthreads_and(good)) {
            fault = true;
            break;
        }
        const float scale = row_scale(ss, h, a.eps);
        for (; c0 < hi; c0 += chunk) {
            if (c0 != lo + t) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t c = c0 + (int64_t)u * g;
                    const bool in = c < hi;
                    xv[u] = in ? __ldcs(xr + c) : make_uint4(0u, 0u, 0u, 0u);
                    if (kFused) rv[u] = in ? __ldcs(rr + c) : make_uint4(0u, 0u, 0u, 0u);
                    wv[u] = in ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                if (c < hi) {
                    float2 f[P];
                    row_values<T, kFused>(xv[u], rv[u], f);
                    if (kFused) __stcs(rr + c, E::pack2(f));
                    __stcs(orow + c, scaled_weighted<T>(f, scale, wv[u]));
                }
            }
        }
    }
    if (fault) {
        // the remaining rows' exchanges with a flag, touching no row, so that every store a peer
        // sends here is still awaited before this CTA leaves
        for (row += nclusters, ++j; row < a.rows; row += nclusters, ++j) {
            __syncthreads();  // every thread has read the slot's previous row
            float ss = 0.0f;
            sums_send(cs, (int)(j & 1u), 0.0f, 1u, q, C, t);
            (void)sums_wait(cs, (int)(j & 1u), (j >> 1) & 1u, C, ss);
        }
        if (t == 0) atomicOr(&g_fault_flags, kFaultWaitTimeout);
    }
    cluster.sync();
}

// The split two-pass scheme with two rows in flight per cluster: each CTA's one loop over its
// slice reads the *next* row (its first pass, from DRAM: the sum of squares) and re-reads the
// current row (its second pass, from L2: the outputs), so every CTA keeps DRAM reads and writes
// in flight together, where the one-row kernel alternates a read-only pass with a
// read-and-write one, all clusters in step. The next row's slice sums are sent through
// ClusterSums after the loop, and awaited after the next loop's first loads. Rows alternate
// between the two slots: row k's sums use slot k % 2, so a CTA sends row k + 1's sums only after
// every thread of it has read row k - 1's. Rows in flight are two per cluster (the grid's L2 cap
// counts them). After a time-out the CTAs keep exchanging flags without touching rows, as in the
// one-row kernel.
template <typename T, bool kFused, int U, int kMaxBlock>
__global__ void __launch_bounds__(kMaxBlock) rows_split_pipe_kernel(const RowArgs a) {
    namespace cg = cooperative_groups;
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    __shared__ float red[32];
    __shared__ __align__(8) ClusterSums cs;

    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int q = (int)cluster.block_rank();
    const int g = blockDim.x, t = threadIdx.x;
    const int64_t hv = a.hv;
    const int64_t S = (hv + C - 1) / C;
    const int64_t lo = q * S;
    const int64_t hi = (lo + S < hv) ? lo + S : hv;
    const int64_t chunk = (int64_t)g * U;
    const float h = (float)a.hidden;
    const uint4 *xg = static_cast<const uint4 *>(a.x);
    uint4 *og = static_cast<uint4 *>(a.out);
    uint4 *rg = static_cast<uint4 *>(a.res);
    const uint4 *wg = static_cast<const uint4 *>(a.w);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    grid_dependency_wait();
    allow_dependents_launch();
    if (t == 0) sums_init(cs);
    const int64_t nclusters = gridDim.x / C;
    int64_t row = blockIdx.x / C;

    // The CTA's slice sum (warps in order) sent as row k's sums (slot k % 2). The barrier also
    // orders every thread's reads of row k - 2's slot, and of `red`, before the sends.
    auto publish = [&](float v, uint32_t k, uint32_t flag) {
        const float wsum = warp_sum(v);
        if ((t & 31) == 0) red[t >> 5] = wsum;
        __syncthreads();
        float cta = 0.0f;
        if (t < C)
            for (int i = 0; i < (g >> 5); ++i) cta += red[i];
        sums_send(cs, (int)(k & 1u), cta, flag, q, C, t);
    };

    // Start: the first row's first pass alone, while the cluster's barriers are being set up;
    // every CTA has set its barriers up before any CTA sends to it.
    cluster.barrier_arrive();
    PairSumSq<E::kPairMath> acc0;
    if (row < a.rows) {
        const uint4 *xr = xg + row * hv;
        const uint4 *rr = kFused ? rg + row * hv : nullptr;
        for (int64_t c0 = lo + t; c0 < hi; c0 += chunk) {
            uint4 xv[U], rv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                xv[u] = c < hi ? xr[c] : zero;
                if (kFused) rv[u] = c < hi ? rr[c] : zero;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float2 f[P];
                row_values<T, kFused>(xv[u], rv[u], f);
                acc0.add(f);
            }
        }
    }
    cluster.barrier_wait();
    if (row < a.rows) publish(acc0.total(), 0u, 0u);

    bool fault = false;
    uint32_t j = 0;
    for (; row < a.rows; row += nclusters, ++j) {
        const int64_t nxt = row + nclusters;
        const bool more = nxt < a.rows;  // uniform over the cluster
        const uint4 *xr = xg + row * hv;
        uint4 *rr = kFused ? rg + row * hv : nullptr;
        uint4 *orow = og + row * hv;
        const uint4 *xn = xg + nxt * hv;
        const uint4 *rn = kFused ? rg + nxt * hv : nullptr;
        PairSumSq<E::kPairMath> acc;
        uint4 xv[U], rv[U], wv[U], xw[U], rw[U];
        // one step's loads: the next row's vectors (DRAM) and this row's (L2) with the weight
        auto load = [&](int64_t c0) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                const bool in = c < hi;
                xw[u] = (more && in) ? xn[c] : zero;
                if (kFused) rw[u] = (more && in) ? rn[c] : zero;
                xv[u] = in ? __ldcs(xr + c) : zero;
                if (kFused) rv[u] = in ? __ldcs(rr + c) : zero;
                wv[u] = in ? __ldg(wg + c) : zero;
            }
        };
        // one step's work: the next row's sum of squares, this row's outputs
        auto step = [&](int64_t c0, float scale) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float2 f[P];
                row_values<T, kFused>(xw[u], rw[u], f);
                acc.add(f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                if (c < hi) {
                    float2 f[P];
                    row_values<T, kFused>(xv[u], rv[u], f);
                    if (kFused) __stcs(rr + c, E::pack2(f));
                    __stcs(orow + c, scaled_weighted<T>(f, scale, wv[u]));
                }
            }
        };
        // the first step's loads need no scale: issue them before this row's wait
        int64_t c0 = lo + t;
        load(c0);
        float ss = 0.0f;
        const bool good = sums_wait(cs, (int)(j & 1u), (j >> 1) & 1u, C, ss);
        if (!__syncthreads_and(good)) {
            fault = true;
            break;
        }
        const float scale = row_scale(ss, h, a.eps);
        step(c0, scale);
        for (c0 += chunk; c0 < hi; c0 += chunk) {
            load(c0);
            step(c0, scale);
        }
        if (more) publish(acc.total(), j + 1u, 0u);
    }
    if (fault) {
        // The remaining rows' exchanges with a flag, touching no row, so that every store a peer
        // sends here is still awaited before this CTA leaves: row k + 1's sums are sent before
        // row k + 1's wait, as in the loop.
        for (row += nclusters, ++j; row < a.rows; row += nclusters, ++j) {
            publish(0.0f, j, 1u);
            float ss = 0.0f;
            (void)sums_wait(cs, (int)(j & 1u), (j >> 1) & 1u, C, ss);
        }
        if (t == 0) atomicOr(&g_fault_flags, kFaultWaitTimeout);
    }
    cluster.sync();
}

template <typename T, bool kFused, int U>
const void *pick_split(int block, bool pipelined) {
    if (pipelined) {
        if (block <= 256) return (const void *)rows_split_pipe_kernel<T, kFused, U, 256>;
        if (block <= 512) return (const void *)rows_split_pipe_kernel<T, kFused, U, 512>;
        return (const void *)rows_split_pipe_kernel<T, kFused, U, 1024>;
    }
    if (block <= 256) return (const void *)rows_split_kernel<T, kFused, U, 256>;
    if (block <= 512) return (const void *)rows_split_kernel<T, kFused, U, 512>;
    return (const void *)rows_split_kernel<T, kFused, U, 1024>;
}

// ------------------------------------------------------------------- scalar row kernel

// Any width and any alignment: one CTA per row, element loads, two passes over the row (the
// second usually hits L2). The fused op computes s twice from the untouched inputs and writes
// both outputs only in the second pass, each element by the thread that read it.
template <typename T, bool kFused>
__global__ void __launch_bounds__(1024) rows_scalar_kernel(const RowArgs a) {
    using E = Elem<T>;
    __shared__ float red[2][32];
    const int64_t H = a.hidden;
    const float h = (float)H;
    int parity = 0;
    grid_dependency_wait();
    allow_dependents_launch();
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const int64_t base = row * H;
        SumSq acc;
        int64_t j = threadIdx.x;
        for (; j + 3 * (int64_t)blockDim.x < H; j += 4 * (int64_t)blockDim.x) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t jj = j + u * (int64_t)blockDim.x;
                v[u] = E::load1(a.x, base + jj);
                if (kFused) v[u] = __fadd_rn(v[u], E::load1(a.res, base + jj));
            }
            acc.add(v);
        }
        for (; j < H; j += blockDim.x) {
            float v[1] = {E::load1(a.x, base + j)};
            if (kFused) v[0] = __fadd_rn(v[0], E::load1(a.res, base + j));
            acc.add(v);
        }
        const float ss = team_sum<0>(acc.total(), red[parity]);
        parity ^= 1;
        const float scale = row_scale(ss, h, a.eps);
        for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
            float v = E::load1(a.x, base + j);
            if (kFused) {
                v = __fadd_rn(v, E::load1(a.res, base + j));
                E::store1(a.res, base + j, v);
            }
            E::store1(a.out, base + j, __fmul_rn(__fmul_rn(v, scale), E::load1(a.w, j)));
        }
    }
}


// ------------------------------------------------------------------- staged row kernel

// One CTA per row (team = the CTA, V vectors per thread, as in the CTA-team vector kernel), but
// rows arrive through a ring of `a.stages` shared-memory stages. Thread 0 issues one bulk copy per
// row and tensor (L2 evict-first) and arms the stage's mbarrier with the byte count; every thread
// waits on the barrier, copies its vectors to registers, and computes as before. The row's
// barrier in the CTA reduction is also the point after which the stage is free, so thread 0
// refills it with the row `stages` iterations ahead right after that barrier.
//
// Shared memory: 128 bytes of barriers, then stages x (1 or 2) x hv*16 bytes.
// Every wait is bounded: on a time-out the CTA records kFaultWaitTimeout, stops at that row,
// waits (bounded) for the copies it still has in flight, and returns. (Rows too wide for one CTA
// take the staged split kernel below, which splits each row over a cluster.)
template <typename T, int V, bool kFused>
__global__ void __launch_bounds__(512) rows_bulk_kernel(const RowArgs a) {
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[2][32];

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    unsigned char *ring = smem + 128;
    const int g = blockDim.x;
    const int t = threadIdx.x;
    const int64_t hv = a.hv;
    const int64_t nv = hv;
    const int stages = a.stages;
    const uint32_t copy_bytes = (uint32_t)(nv * 16);
    const uint32_t slot_bytes = copy_bytes;  // the residual's row follows the x row
    const uint32_t stage_bytes = kFused ? 2u * slot_bytes : slot_bytes;
    const float h = (float)a.hidden;
    const int64_t first = blockIdx.x;
    const int64_t step = gridDim.x;

    const uint4 *xg = static_cast<const uint4 *>(a.x);
    uint4 *og = static_cast<uint4 *>(a.out);
    uint4 *rg = kFused ? static_cast<uint4 *>(a.res) : nullptr;

    grid_dependency_wait();
    allow_dependents_launch();
    uint4 wv[V];
    {
        const uint4 *wg = static_cast<const uint4 *>(a.w);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            wv[k] = (c < nv) ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    uint64_t policy = 0;
    if (t == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int s, int64_t row) {
        unsigned char *dst = ring + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&bars[s], kFused ? 2u * copy_bytes : copy_bytes);
        bulk_g2s(dst, xg + row * hv, copy_bytes, &bars[s], policy);
        if (kFused) bulk_g2s(dst + slot_bytes, rg + row * hv, copy_bytes, &bars[s], policy);
    };
    if (t == 0) {
        policy = l2_evict_first_policy();
        for (int s = 0; s < stages; ++s) {
            const int64_t row = first + (int64_t)s * step;
            if (row >= a.rows) break;
            issue(s, row);
        }
    }

    int s = 0;
    uint32_t phase = 0;
    int parity = 0;
    int64_t row = first;
    bool fault = false;
    for (; row < a.rows; row += step) {
        const bool ok = mbar_wait_bounded(&bars[s], phase);
        const unsigned char *sx = ring + (size_t)s * stage_bytes;
        uint4 xv[V], rv[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            const bool in = ok && c < nv;
            xv[k] = in ? ld_shared_v4(sx + c * 16) : make_uint4(0u, 0u, 0u, 0u);
            if (kFused) rv[k] = in ? ld_shared_v4(sx + slot_bytes + c * 16) : make_uint4(0u, 0u, 0u, 0u);
        }

        PairSumSq<E::kPairMath> acc;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (ok && c < nv) {
                float2 f[P];
                row_values<T, kFused>(xv[k], rv[k], f);
                if (kFused) __stcs(rg + row * hv + c, E::pack2(f));
                acc.add(f);
            }
        }
        const float wsum = warp_sum(acc.total());
        if ((t & 31) == 0) red[parity][t >> 5] = wsum;
        // The CTA barrier of this row: partial sums are visible, every thread has its stage data
        // in registers (so the stage may be refilled), and a time-out anywhere is seen by all.
        const bool bad = __syncthreads_or(!ok);
        if (bad) {
            fault = true;
            break;
        }
        if (t == 0) {
            const int64_t ahead = row + (int64_t)stages * step;
            if (ahead < a.rows) issue(s, ahead);
        }
        float ss = 0.0f;
        for (int i = 0; i < (g >> 5); ++i) ss += red[parity][i];
        parity ^= 1;
        const float scale = row_scale(ss, h, a.eps);

#pragma unroll
        for (int k = 0; k < V; ++k) {
            opaque(xv[k]);
            if (kFused) opaque(rv[k]);
            opaque(wv[k]);
        }
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (c < nv) {
                float2 f[P];
                row_values<T, kFused>(xv[k], rv[k], f);
                __stcs(og + row * hv + c, scaled_weighted<T>(f, scale, wv[k]));
            }
        }
        if (++s == stages) {
            s = 0;
            phase ^= 1u;
        }
    }
    if (fault && t == 0) {
        atomicOr(&g_fault_flags, kFaultWaitTimeout);
        // Drain what this CTA issued and did not consume: the rows from `row` up to `stages`
        // iterations ahead, stage s onwards, before the CTA's shared memory is released.
        for (int i = 0; i < stages; ++i) {
            if (row + (int64_t)i * step >= a.rows) break;
            mbar_wait_bounded(&bars[s], phase);
            if (++s == stages) {
                s = 0;
                phase ^= 1u;
            }
        }
    }
}

// ------------------------------------------------------------------ cluster row kernel

// One thread-block cluster of C CTAs per row, for few rows of wide rows, where one CTA per row
// would leave most SMs idle. CTA rank q of the cluster owns the row's 16-byte vectors
// [q*S, min(hv, (q+1)*S)), S = ceil(hv / C); its thread t owns vectors q*S + t + k*G (k < V).
// Each CTA reduces its slice (warp shuffles, then its warps in order), publishes the partial in
// its own shared memory, and after one cluster barrier every thread adds the C partials in rank
// order, read through distributed shared memory, so every CTA of the cluster computes the same
// scale. Partials alternate between two slots per row, so one cluster barrier per row suffices
// (a CTA can overwrite a slot only after the next row's barrier, which every peer reaches only
// after reading it); a last cluster barrier keeps each CTA's shared memory alive until its peers
// have read it. Clusters stride over rows. No global scratch, no spin-waits.
template <typename T, int V, bool kFused>
__global__ void __launch_bounds__(512) rows_cluster_kernel(const RowArgs a) {
    namespace cg = cooperative_groups;
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    __shared__ float red[2][32];
    __shared__ float part[2];

    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int q = (int)cluster.block_rank();
    const int g = blockDim.x;
    const int t = threadIdx.x;
    const int64_t hv = a.hv;
    const int64_t S = (hv + C - 1) / C;
    const int64_t lo = q * S;
    const int64_t hi = (lo + S < hv) ? lo + S : hv;
    const float h = (float)a.hidden;

    const uint4 *xg = static_cast<const uint4 *>(a.x);
    uint4 *og = static_cast<uint4 *>(a.out);
    uint4 *rg = static_cast<uint4 *>(a.res);

    grid_dependency_wait();
    allow_dependents_launch();
    uint4 wv[V];
    {
        const uint4 *wg = static_cast<const uint4 *>(a.w);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = lo + t + (int64_t)k * g;
            wv[k] = (c < hi) ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    const int64_t nclusters = gridDim.x / C;
    int parity = 0;
    for (int64_t row = blockIdx.x / C; row < a.rows; row += nclusters) {
        uint4 xv[V], rv[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = lo + t + (int64_t)k * g;
            xv[k] = (c < hi) ? __ldcs(xg + row * hv + c) : make_uint4(0u, 0u, 0u, 0u);
            if (kFused) rv[k] = (c < hi) ? __ldcs(rg + row * hv + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        PairSumSq<E::kPairMath> acc;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = lo + t + (int64_t)k * g;
            if (c < hi) {
                float2 f[P];
                row_values<T, kFused>(xv[k], rv[k], f);
                if (kFused) __stcs(rg + row * hv + c, E::pack2(f));
                acc.add(f);
            }
        }
        // CTA partial: warps in order, by thread 0, into this row's slot
        const float wsum = warp_sum(acc.total());
        if ((t & 31) == 0) red[parity][t >> 5] = wsum;
        __syncthreads();
        if (t == 0) {
            float cta = 0.0f;
            for (int i = 0; i < (g >> 5); ++i) cta += red[parity][i];
            part[parity] = cta;
        }
        cluster.sync();  // every CTA's partial for this row is published
        float ss = 0.0f;
        for (int r = 0; r < C; ++r) ss += *cluster.map_shared_rank(&part[parity], r);
        parity ^= 1;
        const float scale = row_scale(ss, h, a.eps);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = lo + t + (int64_t)k * g;
            if (c < hi) {
                float2 f[P];
                row_values<T, kFused>(xv[k], rv[k], f);
                __stcs(og + row * hv + c, scaled_weighted<T>(f, scale, wv[k]));
            }
        }
    }
    cluster.sync();  // peers may still be reading this CTA's partials
}

// Rows too wide for one CTA, staged through shared memory: each row split over a cluster of C
// CTAs, CTA q's slice of ceil(hv / C) vectors streamed from global memory by bulk asynchronous
// copies (one issuing thread, L2 evict-first, completing on the stage's mbarrier) into a ring of
// `stages` shared-memory stages, so up to `stages` rows per CTA are in flight and the DRAM reads
// do not wait for the SM. Every thread copies its V vectors of a stage into registers (the
// fused op forms s = x + r there and writes the residual), so the stage is free after the row's
// CTA barrier and is refilled at once with the row `stages` iterations ahead.
// The slice sums meet without a cluster barrier: each CTA sends its sum (and a time-out flag)
// to every CTA of the cluster with an asynchronous shared-memory store that completes as
// transaction bytes on the receiver's mbarrier for the row, and each CTA waits on its own
// barrier for C of them. (A cluster barrier's arrive has release semantics: every thread first
// waits for its previous row's global stores to be acknowledged, which ncu showed as the top
// stall.) Two barriers and slots alternate by row: a CTA sends row j + 2's sum only after it
// has received every peer's row j + 1 sum, which each peer sends only after reading its row j
// slots. Every wait is bounded. After a time-out (here, or a peer's flag) the CTA records
// KS_FAULT_WAIT_TIMEOUT and keeps exchanging flags for the remaining rows without touching rows
// or stages, so every store a peer sends is still awaited before any CTA leaves; then it waits
// (bounded) for its own copies in flight. Thread 0 tracks the stages with a copy in flight and
// the parity each completes with.
template <typename T, int V, bool kFused>
__global__ void __launch_bounds__(512) rows_stage_split_kernel(const RowArgs a) {
    namespace cg = cooperative_groups;
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[2][32];
    __shared__ __align__(8) uint32_t part[2][8][2];  // per row slot: (sum bits, flag) by rank
    __shared__ __align__(8) uint64_t pbar[2];          // completes when C sums have arrived

    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int q = (int)cluster.block_rank();
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    unsigned char *ring = smem + 128;
    const int g = blockDim.x, t = threadIdx.x;
    const int64_t hv = a.hv;
    const int64_t S = (hv + C - 1) / C;
    const int64_t lo = q * S;
    const int64_t nv = (lo + S < hv ? lo + S : hv) - lo;  // this CTA's vectors (>= 1)
    const int stages = a.stages;
    const uint32_t copy_bytes = (uint32_t)(nv * 16);
    const uint32_t slot_bytes = (uint32_t)(S * 16);  // the residual's slice follows the x slice
    const uint32_t stage_bytes = kFused ? 2u * slot_bytes : slot_bytes;
    const float h = (float)a.hidden;
    const int64_t first = blockIdx.x / C;
    const int64_t step = gridDim.x / C;
    const uint4 *xg = static_cast<const uint4 *>(a.x) + lo;
    uint4 *og = static_cast<uint4 *>(a.out) + lo;
    uint4 *rg = kFused ? static_cast<uint4 *>(a.res) + lo : nullptr;

    grid_dependency_wait();
    allow_dependents_launch();
    uint4 wv[V];
    {
        const uint4 *wg = static_cast<const uint4 *>(a.w) + lo;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            wv[k] = (c < nv) ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (t == 0) {
        for (int i = 0; i < stages; ++i) mbar_init(&bars[i], 1);
        mbar_init(&pbar[0], 1);
        mbar_init(&pbar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // every CTA of the cluster has started and set up its barriers before any CTA sends to it
    cluster.barrier_arrive();
    cluster.barrier_wait();

    uint64_t policy = 0;
    uint32_t pending = 0;  // thread 0: stages with a copy in flight
    uint32_t wphase = 0;   // bit i: the parity stage i's next copy completes with
    auto issue = [&](int st, int64_t r) {
        unsigned char *dst = ring + (size_t)st * stage_bytes;
        mbar_arrive_expect_tx(&bars[st], kFused ? 2u * copy_bytes : copy_bytes);
        bulk_g2s(dst, xg + r * hv, copy_bytes, &bars[st], policy);
        if (kFused) bulk_g2s(dst + slot_bytes, rg + r * hv, copy_bytes, &bars[st], policy);
        pending |= 1u << st;
    };
    if (t == 0) {
        policy = l2_evict_first_policy();
        for (int i = 0; i < stages; ++i) {
            const int64_t r = first + (int64_t)i * step;
            if (r >= a.rows) break;
            issue(i, r);
        }
    }

    int st = 0;
    uint32_t it = 0;
    bool fault = false;
    for (int64_t row = first; row < a.rows; row += step, ++it) {
        const int p = (int)(it & 1u);
        bool ok = true;
        uint4 xv[V], rv[V];
        PairSumSq<E::kPairMath> acc;
        if (!fault) {
            ok = mbar_wait_bounded(&bars[st], (wphase >> st) & 1u);
            const unsigned char *sx = ring + (size_t)st * stage_bytes;
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int64_t c = t + (int64_t)k * g;
                const bool in = ok && c < nv;
                xv[k] = in ? ld_shared_v4(sx + c * 16) : make_uint4(0u, 0u, 0u, 0u);
                if (kFused) rv[k] = in ? ld_shared_v4(sx + slot_bytes + c * 16) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int64_t c = t + (int64_t)k * g;
                if (ok && c < nv) {
                    float2 f[P];
                    row_values<T, kFused>(xv[k], rv[k], f);
                    if (kFused) __stcs(rg + row * hv + c, E::pack2(f));
                    acc.add(f);
                }
            }
        }
        const float wsum = warp_sum(acc.total());
        if ((t & 31) == 0) red[p][t >> 5] = wsum;
        // every thread has its stage data in registers: the stage is free
        const bool bad = __syncthreads_or(!ok || fault);
        if (!fault && ok) wphase ^= 1u << st;
        if (t == 0) {
            if (!fault && ok) pending &= ~(1u << st);
            const int64_t ahead = row + (int64_t)stages * step;
            if (!bad && ahead < a.rows) issue(st, ahead);
            mbar_arrive_expect_tx(&pbar[p], (uint32_t)C * 8u);
        }
        if (t < C) {
            float cta = 0.0f;
            for (int i = 0; i < (g >> 5); ++i) cta += red[p][i];
            st_async_v2(cluster_map(&part[p][q][0], (uint32_t)t), __float_as_uint(cta), bad ? 1u : 0u,
                        cluster_map(&pbar[p], (uint32_t)t));
        }
        const bool got = mbar_wait_bounded(&pbar[p], (it >> 1) & 1u);
        float ss = 0.0f;
        uint32_t any_bad = got ? 0u : 1u;
        for (int r = 0; r < C; ++r) {
            ss += __uint_as_float(part[p][r][0]);
            any_bad |= part[p][r][1];
        }
        // every thread has read this row's slots before any thread's next row (whose sends
        // into the other slot pair follow this row's barrier anyway)
        if (__syncthreads_or(any_bad != 0u) || fault) {
            fault = true;
            continue;
        }
        const float scale = row_scale(ss, h, a.eps);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            opaque(xv[k]);
            if (kFused) opaque(rv[k]);
            opaque(wv[k]);
        }
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (c < nv) {
                float2 f[P];
                row_values<T, kFused>(xv[k], rv[k], f);
                __stcs(og + row * hv + c, scaled_weighted<T>(f, scale, wv[k]));
            }
        }
        if (++st == stages) st = 0;
    }
    if (fault && t == 0) {
        atomicOr(&g_fault_flags, kFaultWaitTimeout);
        // the copies this CTA issued that have not completed, before its shared memory goes
        for (int i = 0; i < stages; ++i)
            if ((pending >> i) & 1u) mbar_wait_bounded(&bars[i], (wphase >> i) & 1u);
    }
    cluster.sync();
}

// Plain rows too wide for one CTA, kept in shared memory through both passes. As in
// rows_stage_split_kernel, each row is split over a cluster of C CTAs (here up to 16, a
// non-portable cluster size the launch opts into) and CTA q's slice streams
// into a ring of `stages` shared-memory stages by bulk asynchronous copies; here the slice is not
// copied into registers. The first pass sums its squares from the stage and the second reads it
// again from there, so a thread holds only its V weight vectors, and the loop keeps two rows in
// flight: iteration j forms row j's slice sum and sends it to the cluster, then waits for row
// j - 1's sums, writes row j - 1's outputs from its stage and hands that stage to the row
// `stages` iterations ahead (stages >= 2). The wait for one row's sums so overlaps the next
// row's first pass, where the one-row loop leaves the SM without work for a cluster round trip
// per row. With two rows in flight, a CTA may send row j's sum while a peer has yet to read its
// row j - 3 slots, so the sum slots and their mbarriers cycle over four rows: a CTA sends row j
// only after it has received every peer's row j - 2 sum, which each peer sends only after its
// threads have read their row j - 4 slots. Waits are bounded, with the fault path of
// rows_stage_split_kernel: after a time-out (here, or a peer's flag) the CTA keeps sending flags
// and waiting for the remaining rows without touching rows or stages, then waits (bounded) for
// its own copies in flight. Only the weight lives in registers, so at 4 vectors a thread the CTA
// may have up to 1024 threads: the throughput of these rows grows with the threads per SM.
template <typename T, int V>
__global__ void __launch_bounds__(V >= 8 ? 512 : 1024) rows_stage_pipe_kernel(const RowArgs a) {
    namespace cg = cooperative_groups;
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[2][32];
    __shared__ __align__(8) uint32_t part[4][16][2];  // per row slot: (sum bits, flag) by rank
    __shared__ __align__(8) uint64_t pbar[4];           // completes when C sums have arrived

    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int q = (int)cluster.block_rank();
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    unsigned char *ring = smem + 128;
    const int g = blockDim.x, t = threadIdx.x;
    const int64_t hv = a.hv;
    const int64_t S = (hv + C - 1) / C;
    const int64_t lo = q * S;
    const int64_t nv = (lo + S < hv ? lo + S : hv) - lo;  // this CTA's vectors (>= 1)
    const int stages = a.stages;
    const uint32_t copy_bytes = (uint32_t)(nv * 16);
    const uint32_t stage_bytes = (uint32_t)(S * 16);
    const float h = (float)a.hidden;
    const int64_t first = blockIdx.x / C;
    const int64_t step = gridDim.x / C;
    const int64_t n = first < a.rows ? (a.rows - 1 - first) / step + 1 : 0;  // the cluster's rows
    const uint4 *xg = static_cast<const uint4 *>(a.x) + lo;
    uint4 *og = static_cast<uint4 *>(a.out) + lo;

    grid_dependency_wait();
    allow_dependents_launch();
    uint4 wv[V];
    {
        const uint4 *wg = static_cast<const uint4 *>(a.w) + lo;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            wv[k] = (c < nv) ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (t == 0) {
        for (int i = 0; i < stages; ++i) mbar_init(&bars[i], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&pbar[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // every CTA of the cluster has started and set up its barriers before any CTA sends to it
    cluster.barrier_arrive();
    cluster.barrier_wait();

    uint64_t policy = 0;
    uint32_t pending = 0;  // thread 0: stages with a copy in flight
    uint32_t wphase = 0;   // bit i: the parity stage i's next copy completes with
    auto issue = [&](int st, int64_t r) {
        mbar_arrive_expect_tx(&bars[st], copy_bytes);
        bulk_g2s(ring + (size_t)st * stage_bytes, xg + r * hv, copy_bytes, &bars[st], policy);
        pending |= 1u << st;
    };
    if (t == 0) {
        policy = l2_evict_first_policy();
        for (int i = 0; i < stages && i < n; ++i) issue(i, first + (int64_t)i * step);
    }

    int sa = 0, sb = 0;  // the stages of the rows in the first and in the second pass
    bool fault = false;
    for (int64_t j = 0; j <= n; ++j) {
        if (j < n) {  // first pass of row j
            const int p = (int)(j & 1), sl = (int)(j & 3);
            bool ok = true;
            PairSumSq<E::kPairMath> acc;
            if (!fault) {
                ok = mbar_wait_bounded(&bars[sa], (wphase >> sa) & 1u);
                if (ok) {
                    const unsigned char *sx = ring + (size_t)sa * stage_bytes;
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        const int64_t c = t + (int64_t)k * g;
                        if (c < nv) {
                            float2 f[P];
                            const uint4 xv = ld_shared_v4(sx + c * 16);
                            row_values<T, false>(xv, xv, f);
                            acc.add(f);
                        }
                    }
                }
            }
            const float wsum = warp_sum(acc.total());
            if ((t & 31) == 0) red[p][t >> 5] = wsum;
            const bool bad = __syncthreads_or(!ok || fault);
            if (!fault && ok) wphase ^= 1u << sa;
            if (t == 0) {
                if (!fault && ok) pending &= ~(1u << sa);
                mbar_arrive_expect_tx(&pbar[sl], (uint32_t)C * 8u);
            }
            if (t < C) {
                float cta = 0.0f;
                for (int i = 0; i < (g >> 5); ++i) cta += red[p][i];
                st_async_v2(cluster_map(&part[sl][q][0], (uint32_t)t), __float_as_uint(cta),
                            bad ? 1u : 0u, cluster_map(&pbar[sl], (uint32_t)t));
            }
            fault = bad;
            if (++sa == stages) sa = 0;
        }
        if (j >= 1) {  // second pass of row j - 1
            const int64_t jb = j - 1;
            const int sl = (int)(jb & 3);
            const bool got = mbar_wait_bounded(&pbar[sl], (uint32_t)(jb >> 2) & 1u);
            float ss = 0.0f;
            uint32_t any_bad = got ? 0u : 1u;
            for (int r = 0; r < C; ++r) {
                ss += __uint_as_float(part[sl][r][0]);
                any_bad |= part[sl][r][1];
            }
            if (!fault && any_bad == 0u) {
                const int64_t row = first + jb * step;
                const float scale = row_scale(ss, h, a.eps);
                const unsigned char *sx = ring + (size_t)sb * stage_bytes;
#pragma unroll
                for (int k = 0; k < V; ++k) {
                    const int64_t c = t + (int64_t)k * g;
                    if (c < nv) {
                        float2 f[P];
                        const uint4 xv = ld_shared_v4(sx + c * 16);
                        row_values<T, false>(xv, xv, f);
                        __stcs(og + row * hv + c, scaled_weighted<T>(f, scale, wv[k]));
                    }
                }
            }
            // every thread has read the stage and this row's slots: the stage goes to the row
            // `stages` iterations ahead
            const bool bad = __syncthreads_or(fault || any_bad != 0u);
            if (t == 0 && !bad && jb + stages < n) issue(sb, first + (jb + stages) * step);
            fault = bad;
            if (++sb == stages) sb = 0;
        }
    }
    if (fault && t == 0) {
        atomicOr(&g_fault_flags, kFaultWaitTimeout);
        // the copies this CTA issued that have not completed, before its shared memory goes
        for (int i = 0; i < stages; ++i)
            if ((pending >> i) & 1u) mbar_wait_bounded(&bars[i], (wphase >> i) & 1u);
    }
    cluster.sync();
}

// ----------------------------------------------------------------------- kernel selection

// Sub-warp team kernels: 8 or 16 lanes per row, V vectors per lane.
template <typename T, int V, bool kFused>
const void *pick_team(int team, bool pf) {
    if (team == 8)
        return pf ? (const void *)rows_vec_kernel<T, V, kFused, 8, true>
                  : (const void *)rows_vec_kernel<T, V, kFused, 8, false>;
    return pf ? (const void *)rows_vec_kernel<T, V, kFused, 16, true>
              : (const void *)rows_vec_kernel<T, V, kFused, 16, false>;
}

template <typename T, bool kFused>
const void *pick_kernel(const ks_plan_t &p) {
    switch (p.kernel) {
    case KS_KERNEL_WARP_ROW: {
        const bool pf = !(p.flags & KS_PLAN_NO_PREFETCH);
        if (p.team == 8 || p.team == 16) {
            switch (p.vec_per_thread) {
            case 1: return pick_team<T, 1, kFused>(p.team, pf);
            case 2: return pick_team<T, 2, kFused>(p.team, pf);
            case 4: return pick_team<T, 4, kFused>(p.team, pf);
            default: return nullptr;
            }
        }
        switch (p.vec_per_thread) {
        case 1: return pf ? (const void *)rows_vec_kernel<T, 1, kFused, 32, true>
                          : (const void *)rows_vec_kernel<T, 1, kFused, 32, false>;
        case 2: return pf ? (const void *)rows_vec_kernel<T, 2, kFused, 32, true>
                          : (const void *)rows_vec_kernel<T, 2, kFused, 32, false>;
        case 4: return pf ? (const void *)rows_vec_kernel<T, 4, kFused, 32, true>
                          : (const void *)rows_vec_kernel<T, 4, kFused, 32, false>;
        case 6: return pf ? (const void *)rows_vec_kernel<T, 6, kFused, 32, true>
                          : (const void *)rows_vec_kernel<T, 6, kFused, 32, false>;
        case 8: return pf ? (const void *)rows_vec_kernel<T, 8, kFused, 32, true>
                          : (const void *)rows_vec_kernel<T, 8, kFused, 32, false>;
        default: return nullptr;
        }
    }
    case KS_KERNEL_CTA_ROW: {
        const bool pf = !(p.flags & KS_PLAN_NO_PREFETCH);
        switch (p.vec_per_thread) {
        case 2: return pf ? (const void *)rows_vec_kernel<T, 2, kFused, 0, true>
                          : (const void *)rows_vec_kernel<T, 2, kFused, 0, false>;
        case 4: return pf ? (const void *)rows_vec_kernel<T, 4, kFused, 0, true>
                          : (const void *)rows_vec_kernel<T, 4, kFused, 0, false>;
        default: return nullptr;
        }
    }
    case KS_KERNEL_SCALAR: return (const void *)rows_scalar_kernel<T, kFused>;
    case KS_KERNEL_TWOPASS_ROW:
        if (p.cluster >= 2) {
            switch (p.vec_per_thread) {
            case 2: return pick_split<T, kFused, 2>(p.block, p.stages == 2);
            case 4: return pick_split<T, kFused, 4>(p.block, p.stages == 2);
            default: return nullptr;
            }
        }
        switch (p.vec_per_thread) {
        case 2: return pick_twopass<T, kFused, 2>(p.block);
        case 4: return pick_twopass<T, kFused, 4>(p.block);
        default: return nullptr;
        }
    case KS_KERNEL_BULK_ROW:
        if (p.cluster >= 2 && (p.flags & KS_PLAN_SMEM_ROWS)) {
            if (kFused) return nullptr;
            if (p.vec_per_thread == 4) return (const void *)rows_stage_pipe_kernel<T, 4>;
            if (p.vec_per_thread == 8) return (const void *)rows_stage_pipe_kernel<T, 8>;
            return nullptr;
        }
        if (p.cluster >= 2) {
            if (p.vec_per_thread == 4) return (const void *)rows_stage_split_kernel<T, 4, kFused>;
            if (p.vec_per_thread == 8 && !kFused) return (const void *)rows_stage_split_kernel<T, 8, false>;
            return nullptr;
        }
        if (p.vec_per_thread != 4) return nullptr;
        return (const void *)rows_bulk_kernel<T, 4, kFused>;
    case KS_KERNEL_CLUSTER_ROW:
        switch (p.vec_per_thread) {
        case 1: return (const void *)rows_cluster_kernel<T, 1, kFused>;
        case 2: return (const void *)rows_cluster_kernel<T, 2, kFused>;
        case 4: return (const void *)rows_cluster_kernel<T, 4, kFused>;
        default: return nullptr;
        }
    default: return nullptr;
    }
}

// Dynamic shared memory of a launch (the staged kernel's barriers and ring; 0 otherwise).
inline size_t dynamic_smem(const ks_plan_t &p) {
    return p.kernel == KS_KERNEL_BULK_ROW ? (size_t)p.smem_bytes : 0;
}

template <typename T>
int blocks_per_sm_t(const ks_plan_t &p, bool fused) {
    const void *f = fused ? pick_kernel<T, true>(p) : pick_kernel<T, false>(p);
    if (!f) return -1;
    if (p.kernel == KS_KERNEL_BULK_ROW) {
        // Allow the largest ring the device takes next to the kernel's static shared memory.
        int dev = 0, optin = 0;
        cudaFuncAttributes fa;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaFuncGetAttributes(&fa, f) != cudaSuccess)
            return -1;
        const int max_dynamic = optin - (int)fa.sharedSizeBytes;
        if (p.smem_bytes > max_dynamic ||
            cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic) !=
                cudaSuccess)
            return -1;
        // clusters of more than 8 CTAs (the shared-memory rows kernel) are a non-portable size
        if (p.cluster > 8 &&
            cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return -1;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, p.block, dynamic_smem(p)) !=
        cudaSuccess)
        return -1;
    return n;
}

// Clusters of the plan's kernel that can be resident at once on the current device (0 when the
// query fails), so a persistent grid of clusters never waits for a second wave.
template <typename T>
int max_clusters_t(const ks_plan_t &p, bool fused) {
    const void *f = fused ? pick_kernel<T, true>(p) : pick_kernel<T, false>(p);
    if (!f || p.cluster < 2 || blocks_per_sm_t<T>(p, fused) < 0) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.cluster);
    cfg.blockDim = dim3((unsigned)p.block);
    cfg.dynamicSmemBytes = dynamic_smem(p);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)p.cluster;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) return 0;
    return n;
}

inline int fault_flags_t(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fault_flags, sizeof v) != cudaSuccess) return -1;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_fault_flags, &zero, sizeof zero) != cudaSuccess) return -1;
    }
    return (int)v;
}

template <typename T>
cudaError_t launch_t(const ks_plan_t &p, bool fused, const RowArgs &a, cudaStream_t s) {
    const void *f = fused ? pick_kernel<T, true>(p) : pick_kernel<T, false>(p);
    if (!f) return cudaErrorInvalidConfiguration;
    RowArgs copy = a;
    void *args[] = {&copy};
    const bool cluster = p.cluster >= 2;  // the cluster-row kernel, or the staged one split
    if (!(p.flags & KS_PLAN_PDL) && !cluster)
        return cudaLaunchKernel(f, dim3((unsigned)p.grid), dim3((unsigned)p.block), args,
                                dynamic_smem(p), s);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3((unsigned)p.block);
    cfg.dynamicSmemBytes = dynamic_smem(p);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (p.flags & KS_PLAN_PDL) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)p.cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace ks

// One translation unit per element type instantiates the launchers (parallel compilation).
#define KS_DEFINE_LAUNCHERS(SUFFIX, TYPE)                                                     \
    namespace ks {                                                                            \
    int blocks_per_sm_##SUFFIX(const ks_plan_t &p, bool fused) {                              \
        return blocks_per_sm_t<TYPE>(p, fused);                                               \
    }                                                                                         \
    int max_clusters_##SUFFIX(const ks_plan_t &p, bool fused) {                               \
        return max_clusters_t<TYPE>(p, fused);                                                \
    }                                                                                         \
    cudaError_t launch_##SUFFIX(const ks_plan_t &p, bool fused, const RowArgs &a,             \
                                cudaStream_t s) {                                             \
        return launch_t<TYPE>(p, fused, a, s);                                                \
    }                                                                                         \
    int fault_flags_##SUFFIX(bool clear) { return fault_flags_t(clear); }                     \
    }
