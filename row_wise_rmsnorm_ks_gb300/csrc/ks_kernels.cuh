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
// every row it touches; the grid is persistent and each team loads its next row before it
// reduces the current one, so a row's loads are in flight during the previous row's reduction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include "ks_internal.h"

namespace ks {

// ------------------------------------------------------------------------ element traits

template <typename T>
struct Elem;

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
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

// Sum over a team: one warp (kWarpTeam) or the whole CTA. Every thread of the team returns the
// same value (the per-warp sums are added in warp order). `red` is one of two alternating
// 32-float slots: a warp can only write a slot again after passing the barrier of the row in
// between, which every warp reaches only after it has read this row's slot, so one barrier per
// row suffices.
template <bool kWarpTeam>
__device__ __forceinline__ float team_sum(float v, float *red) {
    v = warp_sum(v);
    if (kWarpTeam) return v;
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

// One team (a warp, or the whole CTA) per row; row r's 16-byte vector c (of hv) is handled by
// thread c % G of the team, as its (c / G)-th vector. Teams stride over rows by the number of
// teams in the grid.
template <typename T, int V, bool kFused, bool kWarpTeam>
__global__ void __launch_bounds__(VecBound<V, kWarpTeam>::value)
    rows_vec_kernel(const RowArgs a) {
    using E = Elem<T>;
    constexpr int N = E::kPerVec;
    __shared__ float red[2][32];

    const int g = kWarpTeam ? 32 : (int)blockDim.x;
    const int t = kWarpTeam ? (int)(threadIdx.x & 31) : (int)threadIdx.x;
    const int teams = kWarpTeam ? (int)(blockDim.x >> 5) : 1;
    const int team = kWarpTeam ? (int)(threadIdx.x >> 5) : 0;
    const int64_t hv = a.hv;
    const float h = (float)a.hidden;

    const uint4 *xg = static_cast<const uint4 *>(a.x);
    uint4 *og = static_cast<uint4 *>(a.out);
    uint4 *rg = static_cast<uint4 *>(a.res);

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
    const int64_t stride = (int64_t)gridDim.x * teams;
    uint4 xc[V], rc[V];
    if (row < a.rows) {
        load_row<V>(xg + row * hv, t, g, hv, xc);
        if (kFused) load_row<V>(rg + row * hv, t, g, hv, rc);
    }
    int parity = 0;
    while (row < a.rows) {
        const int64_t next = row + stride;
        uint4 xn[V], rn[V];
#pragma unroll
        for (int k = 0; k < V; ++k) xn[k] = rn[k] = make_uint4(0u, 0u, 0u, 0u);
        if (next < a.rows) {
            load_row<V>(xg + next * hv, t, g, hv, xn);
            if (kFused) load_row<V>(rg + next * hv, t, g, hv, rn);
        }

        // Sum of squares; the fused op also forms s and stores cast(s) into the residual.
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (c < hv) {
                float f[N];
                E::unpack(xc[k], f);
                if (kFused) {
                    float q[N];
                    E::unpack(rc[k], q);
#pragma unroll
                    for (int e = 0; e < N; ++e) f[e] = __fadd_rn(f[e], q[e]);
                    __stcs(rg + row * hv + c, E::pack(f));
                }
#pragma unroll
                for (int e = 0; e < N; ++e) ss = __fmaf_rn(f[e], f[e], ss);
            }
        }
        ss = team_sum<kWarpTeam>(ss, red[parity]);
        parity ^= 1;
        const float scale = row_scale(ss, h, a.eps);

        // Normalise, weight, cast, store.
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (c < hv) {
                float f[N], wf[N];
                E::unpack(xc[k], f);
                if (kFused) {
                    float q[N];
                    E::unpack(rc[k], q);
#pragma unroll
                    for (int e = 0; e < N; ++e) f[e] = __fadd_rn(f[e], q[e]);
                }
                E::unpack(wv[k], wf);
#pragma unroll
                for (int e = 0; e < N; ++e) f[e] = __fmul_rn(__fmul_rn(f[e], scale), wf[e]);
                __stcs(og + row * hv + c, E::pack(f));
            }
        }

        row = next;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            xc[k] = xn[k];
            rc[k] = rn[k];
        }
    }
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
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const int64_t base = row * H;
        float ss = 0.0f;
        for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
            float v = E::load1(a.x, base + j);
            if (kFused) v = __fadd_rn(v, E::load1(a.res, base + j));
            ss = __fmaf_rn(v, v, ss);
        }
        ss = team_sum<false>(ss, red[parity]);
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

// ----------------------------------------------------------------------- kernel selection

template <typename T, bool kFused>
const void *pick_kernel(const ks_plan_t &p) {
    switch (p.kernel) {
    case KS_KERNEL_WARP_ROW:
        switch (p.vec_per_thread) {
        case 1: return (const void *)rows_vec_kernel<T, 1, kFused, true>;
        case 2: return (const void *)rows_vec_kernel<T, 2, kFused, true>;
        case 4: return (const void *)rows_vec_kernel<T, 4, kFused, true>;
        default: return nullptr;
        }
    case KS_KERNEL_CTA_ROW:
        switch (p.vec_per_thread) {
        case 2: return (const void *)rows_vec_kernel<T, 2, kFused, false>;
        case 4: return (const void *)rows_vec_kernel<T, 4, kFused, false>;
        default: return nullptr;
        }
    case KS_KERNEL_SCALAR: return (const void *)rows_scalar_kernel<T, kFused>;
    default: return nullptr;
    }
}

template <typename T>
int blocks_per_sm_t(const ks_plan_t &p, bool fused) {
    const void *f = fused ? pick_kernel<T, true>(p) : pick_kernel<T, false>(p);
    if (!f) return -1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, p.block, 0) != cudaSuccess)
        return -1;
    return n;
}

template <typename T>
cudaError_t launch_t(const ks_plan_t &p, bool fused, const RowArgs &a, cudaStream_t s) {
    const void *f = fused ? pick_kernel<T, true>(p) : pick_kernel<T, false>(p);
    if (!f) return cudaErrorInvalidConfiguration;
    RowArgs copy = a;
    void *args[] = {&copy};
    return cudaLaunchKernel(f, dim3((unsigned)p.grid), dim3((unsigned)p.block), args, 0, s);
}

}  // namespace ks

// One translation unit per element type instantiates the launchers (parallel compilation).
#define KS_DEFINE_LAUNCHERS(SUFFIX, TYPE)                                                     \
    namespace ks {                                                                            \
    int blocks_per_sm_##SUFFIX(const ks_plan_t &p, bool fused) {                              \
        return blocks_per_sm_t<TYPE>(p, fused);                                               \
    }                                                                                         \
    cudaError_t launch_##SUFFIX(const ks_plan_t &p, bool fused, const RowArgs &a,             \
                                cudaStream_t s) {                                             \
        return launch_t<TYPE>(p, fused, a, s);                                                \
    }                                                                                         \
    }
