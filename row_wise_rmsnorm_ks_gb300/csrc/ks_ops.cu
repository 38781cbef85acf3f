// The next operators of the library on sm_103a: SwiGLU (silu_and_mul), row-wise Softmax and
// LayerNorm, with their C entry points. All three are memory-bound row or element streams; they
// reuse the RMSNorm kernels' element traits, streaming loads and stores, and the two-slot CTA
// reductions.
//
// Arithmetic:
//  * SwiGLU (Kernscope, "Numerical contract / SwiGLU activation"): gate = fp32(x[:, :d]),
//    up = fp32(x[:, d:]), out = cast((gate * (1 / (1 + exp(-gate)))) * up), FP32 throughout;
//    exp is CUDA's expf for fp32 and the SFU intrinsic for 16-bit types (see exp_for), the
//    reciprocal correctly rounded (equal to the IEEE quotient).
//  * Softmax (Kernscope, "Numerical contract / Softmax"): z = fp32(x) - max(fp32(x)),
//    out = cast(exp(z) / sum(exp(z))). The contract's non-finite rules follow from IEEE
//    arithmetic: a NaN or +inf in a row makes its sum (and so every output) NaN, a row of only
//    -inf has max -inf and z = NaN, and -inf entries of a row with finite values give exp = 0. exp(z) is computed once per element and kept
//    in registers; each output is exp(z) times the correctly rounded reciprocal of the sum.
//  * LayerNorm (named on kernel-set's operator list; read as the standard definition with FP32
//    steps): mean = sum(x)/H, var = sum((x-mean)^2)/H (two reductions over the register-resident
//    row), rstd = correctly rounded rsqrt(var + eps), out = cast((((x-mean)*rstd)*w) + b); w and b
//    optional. The output pass evaluates it as fma(x, rstd, -mean*rstd), then fma(., w, b):
//    the same value with fewer roundings (within the stated tolerance of the oracle's order).
#include <cuda_runtime.h>

#include <cmath>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>
#include <utility>

#include "ks_kernels.cuh"

namespace ks {
namespace {

// ---------------------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// CTA-wide sum / max (fmaxf: NaN-ignoring); every thread returns the same value. `slot` alternates
// between two 32-float rows of `red` on every reduction: a warp writes a slot again only after
// the next reduction's barrier, which every warp passes only after reading this one.
__device__ __forceinline__ float cta_sum(float v, float (*red)[32], int &slot) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[slot][threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[slot][i];
    slot ^= 1;
    return s;
}

__device__ __forceinline__ float cta_max(float v, float (*red)[32], int &slot) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) red[slot][threadIdx.x >> 5] = v;
    __syncthreads();
    float m = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[slot][i]);
    slot ^= 1;
    return m;
}

// Reductions over a row's team: kTeam lanes of a warp (32, 16 or 8: shuffles only, no barrier, so
// the teams of a CTA work on their own rows independently; a team of 8 or 16 lanes is an aligned
// group of lanes, so xor offsets below kTeam stay inside it) or, with kTeam = 0, the whole CTA.
// Every lane of the warp must take part (full-warp shuffles).
template <int kTeam>
__device__ __forceinline__ float team_sum(float v, float (*red)[32], int &slot) {
    if constexpr (kTeam == 0) {
        return cta_sum(v, red, slot);
    } else {
#pragma unroll
        for (int o = kTeam / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        return v;
    }
}

template <int kTeam>
__device__ __forceinline__ float team_max(float v, float (*red)[32], int &slot) {
    if constexpr (kTeam == 0) {
        return cta_max(v, red, slot);
    } else {
#pragma unroll
        for (int o = kTeam / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        return v;
    }
}

// e^v. For 16-bit outputs the SFU-based intrinsic (error a few fp32 ulps, growing with |v|,
// far below half a bf16/fp16 ulp); for fp32 outputs CUDA's expf (within 2 ulp).
template <typename T>
__device__ __forceinline__ float exp_for(float v) {
    return __expf(v);
}
template <>
__device__ __forceinline__ float exp_for<float>(float v) {
    return expf(v);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTwoPowM64 = 5.421010862427522e-20f;          // 2^-64

// 2^v on the special-function unit (relative error about 2^-22; results below 2^-126 flush to
// zero, which the callers keep out of the range that matters by a power-of-two bias).
__device__ __forceinline__ float ex2_sfu(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float rcp_sfu(float v) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Softmax numerators for a pair of elements. fp32 outputs: e^z by expf, with z = v - m the
// contract's FP32 difference (as v + (-m): the same IEEE operation). 16-bit outputs:
// e^z * 2^64 = 2^(z log2(e) + 64) on the SFU; the 2^64 cancels in e / sum and keeps every exp
// above 2^-190 normal (smaller ones are below any fp32 output anyway). Two forms, chosen per row
// (a uniform branch): kFold, for rows with |m| <= kSoftmaxFoldMax, takes one FMA per element,
// v log2(e) + (64 - m log2(e)), whose folded bias is off by at most half an ulp of 64 + 370,
// 2^-16 in the exponent (1e-5 of the output, far below a 16-bit ulp); other rows first form z
// exactly as the contract does, then z log2(e) + 64 (one operation more). Folding the bias for
// any m would lose whole rows: once |m log2(e)| passes 2^31 the bias's rounding error alone
// exceeds the 64 of exponent headroom.
constexpr float kSoftmaxFoldMax = 256.0f;

template <typename T, bool kPair, bool kFold>
__device__ __forceinline__ float2 softmax_exp_pair(float2 v, float neg_m, float bias) {
    if constexpr (sizeof(T) == 4) {
        return make_float2(expf(__fadd_rn(v.x, neg_m)), expf(__fadd_rn(v.y, neg_m)));
    } else if constexpr (kFold) {
        const float2 t = pair_fma<kPair>(v, make_float2(kLog2e, kLog2e), make_float2(bias, bias));
        return make_float2(ex2_sfu(t.x), ex2_sfu(t.y));
    } else {
        const float2 z = pair_add<kPair>(v, make_float2(neg_m, neg_m));
        const float2 t = pair_fma<kPair>(z, make_float2(kLog2e, kLog2e), make_float2(64.0f, 64.0f));
        return make_float2(ex2_sfu(t.x), ex2_sfu(t.y));
    }
}

// (g * sigmoid(g)) * up with sigmoid(g) = 1 / (1 + e^-g), the products in the contract's order,
// so no intermediate is larger than the contract's own.
//  fp32 outputs: e^-g by expf, the correctly rounded reciprocal (bitwise the IEEE quotient).
//  16-bit outputs: the sigmoid on the SFU. Its flush-to-zero ex2 and rcp would lose sigmoids
//  below 2^-126 (gates in [-88.7, -87.3]), which a large `up` still carries into a 16-bit
//  output, so the reciprocal is taken of den' = (1 + e^-g) * 2^-64 = fma(2^(-g log2(e)), 2^-64,
//  2^-64), normal for every gate whose sigmoid is not 0, and scaled back by an IEEE multiply
//  (subnormal results kept): sigmoid = rcp(den') * 2^-64 <= 1. Where e^-g overflows FP32
//  (-g log2(e) >= 128, gates below about -88.72) ex2 gives inf, as the contract's exp does, so
//  den' = inf and the sigmoid is 0 exactly, 1 / (1 + inf) as in the contract; e^-g below 2^-126
//  flushes to 0, giving a sigmoid of 1, which 1 / (1 + e^-g) also rounds to. A NaN gate keeps
//  the NaN.
template <typename T>
__device__ __forceinline__ float silu_mul(float g, float up) {
    const float den = __fmaf_rn(ex2_sfu(__fmul_rn(-g, kLog2e)), kTwoPowM64, kTwoPowM64);
    const float sig = __fmul_rn(rcp_sfu(den), kTwoPowM64);
    return __fmul_rn(__fmul_rn(g, sig), up);
}
template <>
__device__ __forceinline__ float silu_mul<float>(float g, float up) {
    const float sig = __frcp_rn(__fadd_rn(1.0f, expf(-g)));
    return __fmul_rn(__fmul_rn(g, sig), up);
}

// ------------------------------------------------------------------------------- SwiGLU

// Vector paths: rows of d elements as dv = d / E 16-byte vectors in the gate half and the up half
// of each input row.
//
// Row-structured: blockIdx.y and threadIdx.y over rows, the x dimensions over a row's vectors,
// two vectors per thread per iteration with the loads issued before the math. The launch fits the
// block to the row (a multiple of 32 threads covering half the row's vectors per column of CTAs)
// and stacks narrow rows several to a CTA, so few threads sit idle.
template <typename T>
__global__ void __launch_bounds__(256) silu_mul_rows_kernel(void *out, const void *x,
                                                            int64_t rows, int64_t dv) {
    using E = Elem<T>;
    constexpr int N = E::kPerVec;
    grid_dependency_wait();
    allow_dependents_launch();
    const uint4 *xg = static_cast<const uint4 *>(x);
    uint4 *og = static_cast<uint4 *>(out);
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    const int64_t rstep = (int64_t)gridDim.y * blockDim.y;
    for (int64_t row = (int64_t)blockIdx.y * blockDim.y + threadIdx.y; row < rows; row += rstep) {
        const uint4 *gate = xg + row * 2 * dv;
        const uint4 *up = gate + dv;
        uint4 *o = og + row * dv;
        int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        for (; c + step < dv; c += 2 * step) {
            const uint4 g0 = __ldcs(gate + c), u0 = __ldcs(up + c);
            const uint4 g1 = __ldcs(gate + c + step), u1 = __ldcs(up + c + step);
            float a[N], b[N], r[N];
            E::unpack(g0, a);
            E::unpack(u0, b);
#pragma unroll
            for (int e = 0; e < N; ++e) r[e] = silu_mul<T>(a[e], b[e]);
            __stcs(o + c, E::pack(r));
            E::unpack(g1, a);
            E::unpack(u1, b);
#pragma unroll
            for (int e = 0; e < N; ++e) r[e] = silu_mul<T>(a[e], b[e]);
            __stcs(o + c + step, E::pack(r));
        }
        if (c < dv) {
            float a[N], b[N], r[N];
            E::unpack(__ldcs(gate + c), a);
            E::unpack(__ldcs(up + c), b);
#pragma unroll
            for (int e = 0; e < N; ++e) r[e] = silu_mul<T>(a[e], b[e]);
            __stcs(o + c, E::pack(r));
        }
    }
}

// Flat: the output [rows, dv] walked as one run of rows * dv vectors, grid-stride, two vectors
// per thread per iteration, so every thread has work whatever the row width (a 256-thread block
// laid across a row of 64 vectors left 7 of its 8 warps idle: bf16 d = 512 ran at 0.54 of the
// copy peak). Output vector i is input vector i + row * dv of the gate half (row = i / dv) and dv
// further on of the up half. Each thread divides once, then carries the column forward with
// either the input index (16-bit types: a stride of 2 * step vectors moves it by 2 * step +
// (2 * step / dv) * dv, and by dv more when the column wraps past the row's end, no multiply per
// vector) or the row, the index formed from it per vector (fp32). Measured on GB300 at 48..1400
// vectors: carrying the index read 0.92-0.94 of the copy peak for 16-bit types against 0.83-0.87
// carrying the row, but 0.85-0.86 for fp32 against 0.92-0.94.
template <typename T>
__global__ void __launch_bounds__(256) silu_mul_flat_kernel(void *out, const void *x, int64_t rows,
                                                           int64_t dv) {
    using E = Elem<T>;
    constexpr int N = E::kPerVec;
    grid_dependency_wait();
    allow_dependents_launch();
    const uint4 *xg = static_cast<const uint4 *>(x);
    uint4 *og = static_cast<uint4 *>(out);
    const int64_t total = rows * dv;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    constexpr bool kCarryIndex = sizeof(T) == 2;
    // row, column and gate input index of flat vectors i and i + step, and the increments of
    // 2 * step (one of the row and the index is carried, the other left to the compiler to drop)
    int64_t r0 = i / dv;
    int64_t c0 = i - r0 * dv, q0 = i + r0 * dv;
    const int64_t sr = step / dv, sc = step - sr * dv;
    const int64_t sr2 = (2 * step) / dv, sc2 = 2 * step - sr2 * dv;
    const int64_t dq = 2 * step + sr2 * dv;
    int64_t c1 = c0 + sc, r1 = r0 + sr, q1 = q0 + step + sr * dv;
    if (c1 >= dv) {
        c1 -= dv;
        ++r1;
        q1 += dv;
    }
    for (; i + step < total; i += 2 * step) {
        const uint4 *p0 = xg + (kCarryIndex ? q0 : i + r0 * dv);
        const uint4 *p1 = xg + (kCarryIndex ? q1 : i + step + r1 * dv);
        const uint4 g0 = __ldcs(p0), u0 = __ldcs(p0 + dv);
        const uint4 g1 = __ldcs(p1), u1 = __ldcs(p1 + dv);
        float a[N], b[N], r[N];
        E::unpack(g0, a);
        E::unpack(u0, b);
#pragma unroll
        for (int e = 0; e < N; ++e) r[e] = silu_mul<T>(a[e], b[e]);
        __stcs(og + i, E::pack(r));
        E::unpack(g1, a);
        E::unpack(u1, b);
#pragma unroll
        for (int e = 0; e < N; ++e) r[e] = silu_mul<T>(a[e], b[e]);
        __stcs(og + i + step, E::pack(r));
        c0 += sc2;
        c1 += sc2;
        if (kCarryIndex) {
            q0 += dq;
            q1 += dq;
        } else {
            r0 += sr2;
            r1 += sr2;
        }
        if (c0 >= dv) {
            c0 -= dv;
            if (kCarryIndex) q0 += dv; else ++r0;
        }
        if (c1 >= dv) {
            c1 -= dv;
            if (kCarryIndex) q1 += dv; else ++r1;
        }
    }
    if (i < total) {
        const uint4 *p0 = xg + (kCarryIndex ? q0 : i + r0 * dv);
        float a[N], b[N], r[N];
        E::unpack(__ldcs(p0), a);
        E::unpack(__ldcs(p0 + dv), b);
#pragma unroll
        for (int e = 0; e < N; ++e) r[e] = silu_mul<T>(a[e], b[e]);
        __stcs(og + i, E::pack(r));
    }
}

template <typename T>
__global__ void __launch_bounds__(256) silu_mul_scalar_kernel(void *out, const void *x,
                                                              int64_t rows, int64_t d) {
    using E = Elem<T>;
    grid_dependency_wait();
    allow_dependents_launch();
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) {
        for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < d; j += step) {
            const float g = E::load1(x, row * 2 * d + j);
            const float up = E::load1(x, row * 2 * d + d + j);
            E::store1(out, row * d + j, silu_mul<T>(g, up));
        }
    }
}

// ------------------------------------------------------------------------------ Softmax

// One CTA per row (or, with kTeam = 32, 16 or 8, a team of that many lanes of a warp per row, the
// teams on rows of their own; 8- and 16-lane teams put several narrow rows in one warp, so its
// lanes are not idle), V 16-byte vectors per thread held in registers; persistent over rows. With
// kPrefetch the next row's vectors are loaded before the current row's two reductions; without
// it each row is loaded when its turn comes (fewer registers, more resident warps: faster up to
// 1024 vectors per row on GB300, slower beyond). The maximum is a plain fmaxf (NaN-ignoring): a
// NaN or +inf in the row still makes the sum, and so every output, NaN, and a row of only -inf
// still gets max -inf and z = NaN, so the contract's non-finite rules hold.
template <typename T, int V, bool kPrefetch, int kTeam = 0>
__global__ void __launch_bounds__(kTeam ? 128 : 512)
    softmax_vec_kernel(void *out, const void *x, int64_t rows, int64_t hv) {
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    // packed pair instructions (bit-identical) where they measured faster on GB300: bf16 without
    // prefetch, 0.3-0.6 point of the copy peak; with prefetch they took the register count from
    // 64 to 74 and lost 7 points at 2048 vectors
    constexpr bool kPair = E::kPairMath && !kPrefetch;
    __shared__ float red[2][32];
    grid_dependency_wait();
    allow_dependents_launch();
    const uint4 *xg = static_cast<const uint4 *>(x);
    uint4 *og = static_cast<uint4 *>(out);
    const int t = kTeam ? (int)(threadIdx.x & (kTeam - 1)) : (int)threadIdx.x;
    const int g = kTeam ? kTeam : (int)blockDim.x;
    const int teams = kTeam ? (int)(blockDim.x / kTeam) : 1;
    const int64_t stride = (int64_t)gridDim.x * teams;
    int slot = 0;
    int64_t row = (int64_t)blockIdx.x * teams + (kTeam ? (int)(threadIdx.x / kTeam) : 0);
    // Every lane of a warp runs the iterations of the warp's first row, so that all of them take
    // part in the team shuffles; a team of a sub-warp whose row is past the end works on zeros
    // and stores nothing.
    int64_t lead = kTeam ? (int64_t)blockIdx.x * teams + (int)(threadIdx.x >> 5) * (32 / kTeam) : row;
    uint4 cur[V];
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const int64_t c = t + (int64_t)k * g;
        cur[k] = (kPrefetch && row < rows && c < hv) ? __ldcs(xg + row * hv + c)
                                                     : make_uint4(0u, 0u, 0u, 0u);
    }
    for (; lead < rows; lead += stride, row += stride) {
        const bool active = row < rows;
        const int64_t next = row + stride;
        uint4 nxt[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (kPrefetch)
                nxt[k] = (next < rows && c < hv) ? __ldcs(xg + next * hv + c) : make_uint4(0u, 0u, 0u, 0u);
            else
                cur[k] = (active && c < hv) ? __ldcs(xg + row * hv + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        float2 f[V][P];
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            E::unpack2(cur[k], f[k]);
            if (c < hv) {
#pragma unroll
                for (int i = 0; i < P; ++i) m = fmaxf(fmaxf(m, f[k][i].x), f[k][i].y);
            }
        }
        m = team_max<kTeam>(m, red, slot);
        // For m = +-inf or NaN, z (or the folded bias) is NaN or -inf where the formula's is,
        // which gives the contract's NaN rows and masked entries; such rows take the exact form.
        const float neg_m = -m;
        const float bias = __fmaf_rn(neg_m, kLog2e, 64.0f);
        // four running sums: element e feeds lane e % 2 of s[(e / 2) % 2]
        float2 s[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
        if (fabsf(m) <= kSoftmaxFoldMax) {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int64_t c = t + (int64_t)k * g;
                if (c < hv) {
#pragma unroll
                    for (int i = 0; i < P; ++i) {
                        f[k][i] = softmax_exp_pair<T, kPair, true>(f[k][i], neg_m, bias);
                        s[i & 1] = pair_add<kPair>(s[i & 1], f[k][i]);
                    }
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int64_t c = t + (int64_t)k * g;
                if (c < hv) {
#pragma unroll
                    for (int i = 0; i < P; ++i) {
                        f[k][i] = softmax_exp_pair<T, kPair, false>(f[k][i], neg_m, bias);
                        s[i & 1] = pair_add<kPair>(s[i & 1], f[k][i]);
                    }
                }
            }
        }
        const float sum = team_sum<kTeam>(
            __fadd_rn(__fadd_rn(s[0].x, s[0].y), __fadd_rn(s[1].x, s[1].y)), red, slot);
        // e / sum as e * (1 / sum): one correctly rounded reciprocal per row, then a product
        // per element (within 1 fp32 ulp of the quotient)
        const float inv = __frcp_rn(sum);
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (active && c < hv) {
#pragma unroll
                for (int i = 0; i < P; ++i) f[k][i] = pair_mul<kPair>(f[k][i], inv2);
                __stcs(og + row * hv + c, E::pack2(f[k]));
            }
        }
        if (kPrefetch) {
#pragma unroll
            for (int k = 0; k < V; ++k) cur[k] = nxt[k];
        }
    }
}

// Any width and alignment: one CTA per row, three passes over the row (max, sum, write); the
// second and third mostly hit L2. out may be exactly x: each element is read by the thread that
// writes it, after the row's last read by any other thread (the sum's barrier).
template <typename T>
__global__ void __launch_bounds__(1024) softmax_scalar_kernel(void *out, const void *x,
                                                              int64_t rows, int64_t H) {
    using E = Elem<T>;
    __shared__ float red[2][32];
    grid_dependency_wait();
    allow_dependents_launch();
    int slot = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t base = row * H;
        float m = -INFINITY;
        for (int64_t j = threadIdx.x; j < H; j += blockDim.x) m = fmaxf(m, E::load1(x, base + j));
        m = cta_max(m, red, slot);
        float s = 0.0f;
        for (int64_t j = threadIdx.x; j < H; j += blockDim.x)
            s = __fadd_rn(s, exp_for<T>(__fsub_rn(E::load1(x, base + j), m)));
        const float inv = __frcp_rn(cta_sum(s, red, slot));
        for (int64_t j = threadIdx.x; j < H; j += blockDim.x)
            E::store1(out, base + j,
                      __fmul_rn(exp_for<T>(__fsub_rn(E::load1(x, base + j), m)), inv));
    }
}

// ---------------------------------------------------------------------------- LayerNorm

// Which of weight and bias a LayerNorm kernel applies, fixed at compile time: a run-time test per
// element in the output pass measured 7-10 points of the copy peak slower on GB300 (the compiler
// did not hoist it out of the unrolled loop).
constexpr int kAffineWeight = 1, kAffineBias = 2;

// One CTA per row (or with kTeam = 32, 16 or 8 a team of that many lanes of a warp per row, as in
// softmax_vec_kernel), V 16-byte vectors per thread in registers, persistent over rows; the
// weight and bias slices a
// thread needs stay in registers for every row it visits, and the next row's vectors are loaded
// before the current row's two reductions. (Measured on GB300 at [32768,
// 8192] bf16: 74 % of the copy peak; weight and bias in shared memory, with or without the
// prefetch, were slower at 58-64 %.)
// LayerNorm element steps, on FP32 pairs (packed instructions where Elem::kPairMath). Four running
// sums per thread: element e of a vector feeds sum e % 4, held as lane e % 2 of pair (e / 2) % 2,
// and a row's partial sum is the pairwise total (ln_total).
template <typename T>
__device__ __forceinline__ void ln_add_sum(const uint4 &v, float2 (&s)[2]) {
    float2 f[Elem<T>::kPerVec / 2];
    Elem<T>::unpack2(v, f);
#pragma unroll
    for (int i = 0; i < Elem<T>::kPerVec / 2; ++i) s[i & 1] = pair_add<Elem<T>::kPairMath>(s[i & 1], f[i]);
}

// the squares of x - mean, summed as above (x - mean formed as x + (-mean), which is exact)
template <typename T>
__device__ __forceinline__ void ln_add_sq(const uint4 &v, float neg_mean, float2 (&q)[2]) {
    constexpr bool kPair = Elem<T>::kPairMath;
    float2 f[Elem<T>::kPerVec / 2];
    Elem<T>::unpack2(v, f);
    const float2 m = make_float2(neg_mean, neg_mean);
#pragma unroll
    for (int i = 0; i < Elem<T>::kPerVec / 2; ++i) {
        const float2 d = pair_add<kPair>(f[i], m);
        q[i & 1] = pair_fma<kPair>(d, d, q[i & 1]);
    }
}

__device__ __forceinline__ float ln_total(const float2 (&s)[2]) {
    return __fadd_rn(__fadd_rn(s[0].x, s[0].y), __fadd_rn(s[1].x, s[1].y));
}

// One output vector: (x - mean) * rstd as one FMA with shift = -mean * rstd, then the affine
// step (weight and bias, weight alone or bias alone, as kAffine says).
template <typename T, int kAffine>
__device__ __forceinline__ uint4 ln_out(const uint4 &v, const uint4 &wv, const uint4 &bv,
                                        float rstd, float shift) {
    constexpr bool kW = kAffine & kAffineWeight, kB = kAffine & kAffineBias;
    constexpr bool kPair = Elem<T>::kPairMath;
    constexpr int P = Elem<T>::kPerVec / 2;
    float2 f[P], wf[P], bf[P];
    Elem<T>::unpack2(v, f);
    if (kW) Elem<T>::unpack2(wv, wf);
    if (kB) Elem<T>::unpack2(bv, bf);
    const float2 r2 = make_float2(rstd, rstd), s2 = make_float2(shift, shift);
#pragma unroll
    for (int i = 0; i < P; ++i) {
        float2 o = pair_fma<kPair>(f[i], r2, s2);
        if (kW && kB) o = pair_fma<kPair>(o, wf[i], bf[i]);
        else if (kW) o = pair_mul<kPair>(o, wf[i]);
        else if (kB) o = pair_add<kPair>(o, bf[i]);
        f[i] = o;
    }
    return Elem<T>::pack2(f);
}

template <typename T, int V, int kAffine, int kTeam = 0>
__global__ void __launch_bounds__(kTeam ? 128 : 512) layer_norm_vec_kernel(void *out, const void *x,
                                                             const void *w, const void *b,
                                                             int64_t rows, int64_t hidden,
                                                             int64_t hv, float eps) {
    constexpr bool kW = kAffine & kAffineWeight, kB = kAffine & kAffineBias;
    __shared__ float red[2][32];
    grid_dependency_wait();
    allow_dependents_launch();
    const uint4 *xg = static_cast<const uint4 *>(x);
    uint4 *og = static_cast<uint4 *>(out);
    const int t = kTeam ? (int)(threadIdx.x & (kTeam - 1)) : (int)threadIdx.x;
    const int g = kTeam ? kTeam : (int)blockDim.x;
    const int teams = kTeam ? (int)(blockDim.x / kTeam) : 1;
    const int64_t stride = (int64_t)gridDim.x * teams;
    const float h = (float)hidden;
    // Weight and bias slices: in registers for every row a thread visits, except bf16 warp rows
    // of up to 6 vectors a lane, whose CTA keeps one copy in shared memory (every warp of the CTA
    // needs the same slices; filled once, before any warp starts its rows). That frees 8
    // registers per vector a lane holds (bf16, 4 vectors, weight and bias: 136 -> 80) and measured
    // on GB300 0.76 -> 0.94 of the copy peak at 96 vectors, 0.74 -> 0.94 at 160, 0.80 -> 0.92 at
    // 192; for bf16 at 8 vectors and for fp16 and fp32, whose rows already held more warps, it
    // measured up to 8 points slower.
    constexpr bool kSmemAffine = kTeam && std::is_same<T, __nv_bfloat16>::value && V <= 6;
    uint4 wv[V], bv[V];
    __shared__ uint4 sw[kSmemAffine && kW ? 32 * V : 1], sb[kSmemAffine && kB ? 32 * V : 1];
    if (kSmemAffine) {
        const int n = hv < 32 * V ? (int)hv : 32 * V;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            if (kW) sw[i] = __ldg(static_cast<const uint4 *>(w) + i);
            if (kB) sb[i] = __ldg(static_cast<const uint4 *>(b) + i);
        }
        __syncthreads();
    } else {
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            wv[k] = (kW && c < hv) ? __ldg(static_cast<const uint4 *>(w) + c) : make_uint4(0u, 0u, 0u, 0u);
            bv[k] = (kB && c < hv) ? __ldg(static_cast<const uint4 *>(b) + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    int slot = 0;
    int64_t row = (int64_t)blockIdx.x * teams + (kTeam ? (int)(threadIdx.x / kTeam) : 0);
    // every lane of a warp runs the iterations of the warp's first row (see softmax_vec_kernel)
    int64_t lead = kTeam ? (int64_t)blockIdx.x * teams + (int)(threadIdx.x >> 5) * (32 / kTeam) : row;
    uint4 xv[V];
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const int64_t c = t + (int64_t)k * g;
        xv[k] = (row < rows && c < hv) ? __ldcs(xg + row * hv + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    for (; lead < rows; lead += stride, row += stride) {
        const bool active = row < rows;
        const int64_t next = row + stride;
        uint4 nxt[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            nxt[k] = (next < rows && c < hv) ? __ldcs(xg + next * hv + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        float2 s2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
        for (int k = 0; k < V; ++k) ln_add_sum<T>(xv[k], s2);
        const float mean = __fdiv_rn(team_sum<kTeam>(ln_total(s2), red, slot), h);
        float2 q2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
        for (int k = 0; k < V; ++k)
            if (t + (int64_t)k * g < hv) ln_add_sq<T>(xv[k], -mean, q2);
        const float var = __fdiv_rn(team_sum<kTeam>(ln_total(q2), red, slot), h);
        const float rstd = __frsqrt_rn(__fadd_rn(var, eps));
        const float shift = -__fmul_rn(mean, rstd);
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (active && c < hv) {
                const uint4 wk = kSmemAffine ? (kW ? sw[c] : make_uint4(0u, 0u, 0u, 0u)) : wv[k];
                const uint4 bk = kSmemAffine ? (kB ? sb[c] : make_uint4(0u, 0u, 0u, 0u)) : bv[k];
                __stcs(og + row * hv + c, ln_out<T, kAffine>(xv[k], wk, bk, rstd, shift));
            }
        }
#pragma unroll
        for (int k = 0; k < V; ++k) xv[k] = nxt[k];
    }
}

// Staged LayerNorm for many rows: rows stream into a ring of `stages` shared-memory stages by
// bulk asynchronous copies (thread 0 issues one per row, L2 evict-first, completing on the
// stage's mbarrier), so several rows per CTA are in flight. Every thread copies its vectors of
// the stage into registers in the first pass; the row's first reduction barrier is therefore
// also the point after which thread 0 refills the stage with the row `stages` iterations ahead.
// (Reading the stage in all three passes instead freed registers but measured slower.) Waits
// are bounded (about 2 s); on a time-out the CTA records KS_FAULT_WAIT_TIMEOUT, drains its copies
// in flight (bounded) and returns.
// kSmemWB: the weight and bias slices live in shared memory after the ring (filled once per
// CTA) instead of in every thread's registers, 8 registers per vector a thread holds each, so
// CTAs of 288..448 threads fit twice per SM, and a CTA may have up to 1024 threads (rows of up
// to 4096 vectors, where the ring and both rows fit in shared memory).
template <typename T, int V, int kAffine, bool kSmemWB = false>
__global__ void __launch_bounds__(kSmemWB ? 1024 : 512) layer_norm_bulk_kernel(void *out, const void *x,
                                                              const void *w, const void *b,
                                                              int64_t rows, int64_t hidden,
                                                              int64_t hv, float eps, int stages) {
    constexpr bool kW = kAffine & kAffineWeight, kB = kAffine & kAffineBias;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[2][32];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    unsigned char *ring = smem + 128;
    grid_dependency_wait();
    allow_dependents_launch();
    const uint4 *xg = static_cast<const uint4 *>(x);
    uint4 *og = static_cast<uint4 *>(out);
    const int t = threadIdx.x, g = blockDim.x;
    const float h = (float)hidden;
    const uint32_t row_bytes = (uint32_t)(hv * 16);
    const int64_t step = gridDim.x;
    // with kSmemWB: [ring][weight row, if any][bias row, if any]
    unsigned char *sw = ring + (size_t)stages * row_bytes;
    unsigned char *sb = sw + (kW ? row_bytes : 0u);
    constexpr int VW = kSmemWB ? 1 : V;
    uint4 wv[VW], bv[VW];
    if (kSmemWB) {
        for (int64_t c = t; c < hv; c += g) {
            if (kW) *reinterpret_cast<uint4 *>(sw + c * 16) = __ldg(static_cast<const uint4 *>(w) + c);
            if (kB) *reinterpret_cast<uint4 *>(sb + c * 16) = __ldg(static_cast<const uint4 *>(b) + c);
        }
    } else {
#pragma unroll
        for (int k = 0; k < VW; ++k) {
            const int64_t c = t + (int64_t)k * g;
            wv[k] = (kW && c < hv) ? __ldg(static_cast<const uint4 *>(w) + c) : make_uint4(0u, 0u, 0u, 0u);
            bv[k] = (kB && c < hv) ? __ldg(static_cast<const uint4 *>(b) + c) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    uint64_t policy = 0;
    if (t == 0) {
        for (int i = 0; i < stages; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int st, int64_t r) {
        mbar_arrive_expect_tx(&bars[st], row_bytes);
        bulk_g2s(ring + (size_t)st * row_bytes, xg + r * hv, row_bytes, &bars[st], policy);
    };
    if (t == 0) {
        policy = l2_evict_first_policy();
        for (int i = 0; i < stages; ++i) {
            const int64_t r = blockIdx.x + (int64_t)i * step;
            if (r >= rows) break;
            issue(i, r);
        }
    }
    int st = 0, slot = 0;
    uint32_t phase = 0;
    bool fault = false;
    int64_t row = blockIdx.x;
    for (; row < rows; row += step) {
        const bool ok = mbar_wait_bounded(&bars[st], phase);
        const unsigned char *sx = ring + (size_t)st * row_bytes;
        uint4 xv[V];
        float2 s2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            xv[k] = (ok && c < hv) ? ld_shared_v4(sx + c * 16) : make_uint4(0u, 0u, 0u, 0u);
            ln_add_sum<T>(xv[k], s2);
        }
        // first reduction: every thread holds its vectors, so the stage is free, and a time-out
        // anywhere is seen by all
        const float part = warp_sum(ln_total(s2));
        if ((t & 31) == 0) red[slot][t >> 5] = part;
        if (__syncthreads_or(!ok)) {
            fault = true;
            break;
        }
        if (t == 0) {
            const int64_t ahead = row + (int64_t)stages * step;
            if (ahead < rows) issue(st, ahead);
        }
        float tot = 0.0f;
        for (int i = 0; i < (g >> 5); ++i) tot += red[slot][i];
        slot ^= 1;
        const float mean = __fdiv_rn(tot, h);
        float2 q2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
        for (int k = 0; k < V; ++k)
            if (t + (int64_t)k * g < hv) ln_add_sq<T>(xv[k], -mean, q2);
        const float var = __fdiv_rn(cta_sum(ln_total(q2), red, slot), h);
        const float rstd = __frsqrt_rn(__fadd_rn(var, eps));
        const float shift = -__fmul_rn(mean, rstd);
        if (!kSmemWB) {
#pragma unroll
            for (int k = 0; k < VW; ++k) {  // unpack weight and bias per row, not hoisted as floats
                opaque(wv[k]);
                opaque(bv[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t c = t + (int64_t)k * g;
            if (c < hv) {
                const uint4 wk = kSmemWB ? (kW ? ld_shared_v4(sw + c * 16) : make_uint4(0u, 0u, 0u, 0u))
                                         : wv[kSmemWB ? 0 : k];
                const uint4 bk = kSmemWB ? (kB ? ld_shared_v4(sb + c * 16) : make_uint4(0u, 0u, 0u, 0u))
                                         : bv[kSmemWB ? 0 : k];
                __stcs(og + row * hv + c, ln_out<T, kAffine>(xv[k], wk, bk, rstd, shift));
            }
        }
        if (++st == stages) {
            st = 0;
            phase ^= 1u;
        }
    }
    if (fault && t == 0) {
        atomicOr(&g_fault_flags, kFaultWaitTimeout);
        // copies still in flight: this row's stage and the ones after it
        for (int i = 0; i < stages; ++i) {
            if (row + (int64_t)i * step >= rows) break;
            mbar_wait_bounded(&bars[st], phase);
            if (++st == stages) {
                st = 0;
                phase ^= 1u;
            }
        }
    }
}

template <typename T, int kAffine>
__global__ void __launch_bounds__(1024) layer_norm_scalar_kernel(void *out, const void *x,
                                                                 const void *w, const void *b,
                                                                 int64_t rows, int64_t H,
                                                                 float eps) {
    using E = Elem<T>;
    constexpr bool kW = kAffine & kAffineWeight, kB = kAffine & kAffineBias;
    __shared__ float red[2][32];
    grid_dependency_wait();
    allow_dependents_launch();
    const float h = (float)H;
    int slot = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int64_t base = row * H;
        float s = 0.0f;
        for (int64_t j = threadIdx.x; j < H; j += blockDim.x) s = __fadd_rn(s, E::load1(x, base + j));
        const float mean = __fdiv_rn(cta_sum(s, red, slot), h);
        float q = 0.0f;
        for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
            const float d = __fsub_rn(E::load1(x, base + j), mean);
            q = __fmaf_rn(d, d, q);
        }
        const float var = __fdiv_rn(cta_sum(q, red, slot), h);
        const float rstd = __frsqrt_rn(__fadd_rn(var, eps));
        for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
            float v = __fmul_rn(__fsub_rn(E::load1(x, base + j), mean), rstd);
            if (kW) v = __fmul_rn(v, E::load1(w, j));
            if (kB) v = __fadd_rn(v, E::load1(b, j));
            E::store1(out, base + j, v);
        }
    }
}

// ----------------------------------------------------------------------- wide rows

// Rows too wide for the register kernels (more than 2048 16-byte vectors): one CTA per row, the
// row read once per pass with 16-byte vectors, U vectors per thread in flight per step; every
// pass after the first re-reads the row from L2, as the grid keeps the rows all CTAs have in
// flight inside it (wide_grid_cap), so DRAM still sees each element read once. Same arithmetic
// as the register kernels above. The first passes load with the default L2 policy, the last with
// evict-first (last use).

// Softmax, second pass: this thread's sum of the exponentials of its vectors of row xr (four
// running sums, element e of a vector feeding lane e % 2 of sum (e / 2) % 2, added in a fixed
// order at the end). The exponential's form (kFold) is a template argument, chosen once per row,
// so the loop computes one form per element.
template <typename T, int U, bool kFold>
__device__ __forceinline__ float softmax_wide_sum(const uint4 *xr, int64_t hv, int t, int g,
                                                  float neg_m, float bias) {
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    constexpr bool kPair = E::kPairMath;
    const int64_t chunk = (int64_t)g * U;
    float2 s2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
    for (int64_t c0 = t; c0 < hv; c0 += chunk) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = c0 + (int64_t)u * g;
            v[u] = c < hv ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (c0 + (int64_t)u * g < hv) {
                float2 f[P];
                E::unpack2(v[u], f);
#pragma unroll
                for (int i = 0; i < P; ++i)
                    s2[i & 1] = pair_add<kPair>(s2[i & 1], softmax_exp_pair<T, kPair, kFold>(f[i], neg_m, bias));
            }
        }
    }
    return __fadd_rn(__fadd_rn(s2[0].x, s2[0].y), __fadd_rn(s2[1].x, s2[1].y));
}

// Softmax, last pass: the outputs of row xr into orow (last use of the row: evict-first loads).
template <typename T, int U, bool kFold>
__device__ __forceinline__ void softmax_wide_out(const uint4 *xr, uint4 *orow, int64_t hv, int t,
                                                 int g, float neg_m, float bias, float inv) {
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    constexpr bool kPair = E::kPairMath;
    const int64_t chunk = (int64_t)g * U;
    const float2 inv2 = make_float2(inv, inv);
    for (int64_t c0 = t; c0 < hv; c0 += chunk) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = c0 + (int64_t)u * g;
            v[u] = c < hv ? __ldcs(xr + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = c0 + (int64_t)u * g;
            if (c < hv) {
                float2 f[P];
                E::unpack2(v[u], f);
#pragma unroll
                for (int i = 0; i < P; ++i)
                    f[i] = pair_mul<kPair>(softmax_exp_pair<T, kPair, kFold>(f[i], neg_m, bias), inv2);
                __stcs(orow + c, E::pack2(f));
            }
        }
    }
}

// Softmax: max, sum of exponentials, outputs.
template <typename T, int U>
__global__ void __launch_bounds__(1024) softmax_wide_kernel(void *out, const void *x,
                                                            int64_t rows, int64_t hv) {
    using E = Elem<T>;
    constexpr int P = E::kPerVec / 2;
    __shared__ float red[2][32];
    grid_dependency_wait();
    allow_dependents_launch();
    const uint4 *xg = static_cast<const uint4 *>(x);
    uint4 *og = static_cast<uint4 *>(out);
    const int t = threadIdx.x, g = blockDim.x;
    const int64_t chunk = (int64_t)g * U;
    int slot = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const uint4 *xr = xg + row * hv;
        float m = -INFINITY;
        for (int64_t c0 = t; c0 < hv; c0 += chunk) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                v[u] = c < hv ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (c0 + (int64_t)u * g < hv) {
                    float2 f[P];
                    E::unpack2(v[u], f);
#pragma unroll
                    for (int i = 0; i < P; ++i) m = fmaxf(fmaxf(m, f[i].x), f[i].y);
                }
            }
        }
        m = cta_max(m, red, slot);
        const float neg_m = -m;
        const float bias = __fmaf_rn(neg_m, kLog2e, 64.0f);
        const bool fold = fabsf(m) <= kSoftmaxFoldMax;  // see softmax_exp_pair; uniform per row
        const float part = fold ? softmax_wide_sum<T, U, true>(xr, hv, t, g, neg_m, bias)
                                : softmax_wide_sum<T, U, false>(xr, hv, t, g, neg_m, bias);
        const float inv = __frcp_rn(cta_sum(part, red, slot));
        uint4 *orow = og + row * hv;
        if (fold)
            softmax_wide_out<T, U, true>(xr, orow, hv, t, g, neg_m, bias, inv);
        else
            softmax_wide_out<T, U, false>(xr, orow, hv, t, g, neg_m, bias, inv);
    }
}

// LayerNorm: mean, variance, outputs.
template <typename T, int U, int kAffine>
__global__ void __launch_bounds__(512) layer_norm_wide_kernel(void *out, const void *x,
                                                               const void *w, const void *b,
                                                               int64_t rows, int64_t hidden,
                                                               int64_t hv, float eps) {
    constexpr bool kW = kAffine & kAffineWeight, kB = kAffine & kAffineBias;
    __shared__ float red[2][32];
    grid_dependency_wait();
    allow_dependents_launch();
    const uint4 *xg = static_cast<const uint4 *>(x);
    uint4 *og = static_cast<uint4 *>(out);
    const uint4 *wg = static_cast<const uint4 *>(w);
    const uint4 *bg = static_cast<const uint4 *>(b);
    const int t = threadIdx.x, g = blockDim.x;
    const int64_t chunk = (int64_t)g * U;
    const float h = (float)hidden;
    int slot = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const uint4 *xr = xg + row * hv;
        float2 s2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
        for (int64_t c0 = t; c0 < hv; c0 += chunk) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                v[u] = c < hv ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) ln_add_sum<T>(v[u], s2);
        }
        const float mean = __fdiv_rn(cta_sum(ln_total(s2), red, slot), h);
        float2 q2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
        for (int64_t c0 = t; c0 < hv; c0 += chunk) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                v[u] = c < hv ? xr[c] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (c0 + (int64_t)u * g < hv) ln_add_sq<T>(v[u], -mean, q2);
        }
        const float var = __fdiv_rn(cta_sum(ln_total(q2), red, slot), h);
        const float rstd = __frsqrt_rn(__fadd_rn(var, eps));
        const float shift = -__fmul_rn(mean, rstd);
        uint4 *orow = og + row * hv;
        for (int64_t c0 = t; c0 < hv; c0 += chunk) {
            uint4 v[U], wv[U], bv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                const bool in = c < hv;
                v[u] = in ? __ldcs(xr + c) : make_uint4(0u, 0u, 0u, 0u);
                wv[u] = (kW && in) ? __ldg(wg + c) : make_uint4(0u, 0u, 0u, 0u);
                bv[u] = (kB && in) ? __ldg(bg + c) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (int64_t)u * g;
                if (c < hv) __stcs(orow + c, ln_out<T, kAffine>(v[u], wv[u], bv[u], rstd, shift));
            }
        }
    }
}

// ------------------------------------------------------------------------ launch planning

int g_sm_count[64];
int g_l2_bytes[64];  // 0 when the query failed
std::once_flag g_sm_once[64];

// Per-device launch facts, cached: without the cache every launch would repeat the same
// occupancy query (and, for the staged LayerNorm ring, three attribute calls), host work that
// adds to small launches' latency.
std::mutex g_launch_facts_mu;
std::map<std::tuple<int, const void *, int, size_t>, int> g_occupancy;  // CTAs per SM
std::map<std::pair<int, const void *>, int> g_max_dynamic_smem;  // set on the kernel already

// CTAs of kernel f resident per SM at `block` threads and `smem` bytes of dynamic shared memory
// on the current device; 1 when the query fails (not cached then).
int cached_occupancy(const void *f, int block, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const auto key = std::make_tuple(dev, f, block, smem);
    {
        std::lock_guard<std::mutex> lock(g_launch_facts_mu);
        const auto it = g_occupancy.find(key);
        if (it != g_occupancy.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, block, smem) != cudaSuccess || n < 1)
        return 1;
    std::lock_guard<std::mutex> lock(g_launch_facts_mu);
    g_occupancy.emplace(key, n);
    return n;
}

// Lets kernel f use the largest dynamic shared memory the current device takes beside its static
// shared memory (once per device and kernel); false if `smem` does not fit or a call fails.
bool allow_dynamic_smem(const void *f, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const auto key = std::make_pair(dev, f);
    {
        std::lock_guard<std::mutex> lock(g_launch_facts_mu);
        const auto it = g_max_dynamic_smem.find(key);
        if (it != g_max_dynamic_smem.end()) return (int64_t)smem <= it->second;
    }
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, f) != cudaSuccess)
        return false;
    const int max_dynamic = optin - (int)fa.sharedSizeBytes;
    if ((int64_t)smem > max_dynamic ||
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dynamic) != cudaSuccess)
        return false;
    std::lock_guard<std::mutex> lock(g_launch_facts_mu);
    g_max_dynamic_smem.emplace(key, max_dynamic);
    return true;
}

ks_status_t sm_count(int *out) {
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
    if (dev < 0 || dev >= 64) return fail(KS_ERR_CUDA, "device ordinal %d out of range", dev);
    cudaError_t err = cudaSuccess;
    std::call_once(g_sm_once[dev], [&] {
        err = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (cudaDeviceGetAttribute(&g_l2_bytes[dev], cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
            g_l2_bytes[dev] = 0;
            (void)cudaGetLastError();
        }
    });
    if (err != cudaSuccess || g_sm_count[dev] <= 0)
        return fail(KS_ERR_CUDA, "querying the SM count failed");
    *out = g_sm_count[dev];
    return KS_SUCCESS;
}

int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up64(int64_t a, int64_t b) { return ceil_div64(a, b) * b; }

// Vectors per thread and block for a register-resident row of hv vectors: 1 vector below 64,
// 2 below 128, else 4 (measured on GB300 for Softmax and LayerNorm at 128..512 vectors: 4
// vectors per thread beat 2 by 2-12 points); the block a multiple of 32 (at most 512). 0 if the
// row does not fit.
int row_vec_plan(int64_t hv, int *block) {
    const int v = hv < 64 ? 1 : (hv < 128 ? 2 : 4);
    const int64_t b = round_up64(ceil_div64(hv, v), 32);
    if (b > 512) return 0;
    *block = (int)b;
    return v;
}

// Rows wider than the register kernels hold take the wide multi-pass kernels, 4 vectors per
// thread per step. Small CTAs keep more rows in flight per SM;
// measured on GB300 (bf16, HBM-bound rows), the best block grows with the width: Softmax 128
// threads up to 3072 vectors, 256 up to 6144, 512 beyond (0.66-0.87 of the copy peak, against
// 0.62-0.79 at a fixed 512); LayerNorm 128 up to 3072, 256 up to 12288, 512 beyond (0.52-0.86,
// against 0.38-0.62).
int wide_row_block(int64_t hv, bool layer_norm) {
    if (hv <= 3072) return 128;
    if (hv <= (layer_norm ? 12288 : 6144)) return 256;
    return 512;
}

// The L2 size of the current device as sm_count() cached it (0 when unknown).
int64_t device_l2_bytes() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    return g_l2_bytes[dev];
}

// The wide kernels re-read each row from L2: no more CTAs than keep their rows in flight within
// three quarters of it (of a GB300's 128 MiB when the size is unknown), but at least one per SM
// (as for the two-pass RMSNorm kernel).
int64_t wide_grid_cap(int64_t hv, int sms) {
    const int64_t l2 = device_l2_bytes();
    const int64_t cap = (l2 > 0 ? l2 : (128ll << 20)) / 4 * 3 / (hv * 16);
    return cap < sms ? sms : cap;
}

ks_status_t check_common(int64_t rows, int64_t width, ks_dtype_t dtype, int *e) {
    *e = elem_bytes(dtype);
    if (*e == 0) return fail(KS_ERR_UNSUPPORTED_DTYPE, "dtype code %d is not a ks_dtype_t", (int)dtype);
    if (width <= 0) return fail(KS_ERR_INVALID_ARGUMENT, "the last dimension must be > 0 (got %lld)", (long long)width);
    if (rows < 0) return fail(KS_ERR_INVALID_ARGUMENT, "rows must be >= 0 (got %lld)", (long long)rows);
    if (width > INT64_MAX / (4 * *e) || (rows > 0 && rows > INT64_MAX / (4 * width * *e)))
        return fail(KS_ERR_INVALID_ARGUMENT, "rows*width*element size overflows int64");
    return KS_SUCCESS;
}

// ------------------------------------------------------------------------ launch plans
//
// The next operators' launches are described by ks_plan_t as well (include/ks.h), so that
// ks_plan_launch reports the heuristic's choice and the *_planned entry points take an explicit
// one (the tuning hook behind bench.py --ops-bands):
//   SwiGLU     KS_KERNEL_FLAT         the flat walk over all rows' vectors (block <= 256)
//              KS_KERNEL_CTA_ROW      the row-structured kernel, its block fitted to the row with
//                                     at most `block` (32..256) threads
//              KS_KERNEL_SCALAR       element loads (any width and alignment; block <= 256)
//   Softmax,   KS_KERNEL_WARP_ROW     a warp per row, 2/4/6/8 vectors per lane, block/32 rows
//   LayerNorm                         per CTA (block 32..128)
//              KS_KERNEL_CTA_ROW      a CTA per row, 1/2/4 vectors per thread (block <= 512)
//              KS_KERNEL_BULK_ROW     LayerNorm: rows through the staged ring, 4 vectors per
//                                     thread, `stages` 2..8 rows
//              KS_KERNEL_TWOPASS_ROW  the multi-pass wide kernel, 4 vectors a step per thread
//                                     (block <= 1024 Softmax, 512 LayerNorm)
//              KS_KERNEL_SCALAR       element loads (any width and alignment; block <= 1024)
// KS_PLAN_NO_PREFETCH selects the register kernels' variant that loads each row when it comes:
// Softmax warp rows at any vector count and CTA rows at 4 vectors (LayerNorm always prefetches).
// KS_PLAN_PDL: programmatic dependent launch. A plan's grid > 0 caps the CTAs launched.

constexpr int kOpSilu = 2, kOpSoftmax = 3, kOpLayerNorm = 4;  // ks_plan_launch's op codes

ks_plan_t op_plan_of(int kernel, int v, int block, bool prefetch, int stages = 0, int team = 32) {
    ks_plan_t p;
    memset(&p, 0, sizeof p);
    p.kernel = kernel;
    p.vec_per_thread = v;
    p.block = block;
    p.team = kernel == KS_KERNEL_WARP_ROW ? team : block;
    p.flags = prefetch ? 0 : KS_PLAN_NO_PREFETCH;
    p.stages = stages;
    return p;
}

bool op_prefetch(const ks_plan_t &p) { return !(p.flags & KS_PLAN_NO_PREFETCH); }

int scalar_block(int64_t width, int max_block) {
    int b = (int)round_up64(ceil_div64(width, 8), 32);
    return b < 32 ? 32 : (b > max_block ? max_block : b);
}

// SwiGLU, from bench.py --ops-bands (widths of 16..2048 vectors, many rows, each plan timed in
// steady state and right after a kernel with a large shared-memory carveout, the worse of the
// two kept). The row-structured kernel, its CTAs fitted to the row, reads 0.92-0.94 of the copy
// peak for 16-bit rows whose width is a multiple of 32 vectors and 0.95-0.97 for fp32 rows of
// multiples of 64; at other widths it falls to 0.6-0.8, where the flat walk on 128-thread CTAs
// holds 0.85-0.89 (16-bit) and 0.94-0.95 (fp32) at every width (on 256-thread CTAs 2-4 points
// less for 16-bit).
ks_plan_t silu_plan(bool vec, int64_t dv, ks_dtype_t dtype) {
    if (!vec) return op_plan_of(KS_KERNEL_SCALAR, 0, 256, true);
    if (dv % (dtype == KS_DTYPE_F32 ? 64 : 32) == 0) return op_plan_of(KS_KERNEL_CTA_ROW, 2, 256, true);
    return op_plan_of(KS_KERNEL_FLAT, 2, 128, true);
}

// Width bands for many rows (more rows than SMs) of up to 4096 vectors: rows up to `hi` vectors
// take a team of `team` lanes per row at `v` vectors per lane (kind 'w'; 8- and 16-lane teams put
// 4 or 2 rows in a warp), a CTA per row at `v` vectors (kind 'c'), the LayerNorm staged ring of
// `v` rows per CTA (kind 'r'), the wide multi-pass kernel on `block` threads (kind 'x'), or the
// LayerNorm ring with the weight and bias in shared memory (kind 'R', plan flag
// KS_PLAN_AFFINE_SMEM), the general rule (kind 'g'); `prefetch` as the name says. The tables are
// generated, not edited:
//   python bench.py --ops-bands-record <JSON lines of bench.py --ops-bands> > record.json
//   python bench.py --ops-bands-derive record.json
// from GB300 runs of --ops-bands (8..256 and 288..4096 vectors; the record is committed as
// bands/softmax_layer_norm_bands.json beside this file, and a CPU test re-derives the tables
// from it): at each width every
// candidate is scored by the worse of two contexts (steady, and right after a kernel with a
// large shared-memory carveout) and by its worst dtype among those that share the table; the
// previous plan is kept unless another scores a point of the copy peak higher. Warp rows reduce
// with shuffles alone and fill their lanes, where a CTA per row of 33..64 threads, most of them
// idle, paid two CTA barriers per row; sub-warp teams took rows of 8..56 vectors from 0.18-0.90
// to 0.68-0.96 (e.g. Softmax bf16 16 vectors 0.42 -> 0.94, LayerNorm fp16 32 vectors 0.60 ->
// 0.94). Past 256 vectors the ring took bf16 LayerNorm rows of 257..512 vectors (0.66-0.87 ->
// 0.73-0.95) and fp32 rows at several widths (e.g. 1152 vectors 0.80 -> 0.93).
struct Band {
    int16_t hi;
    char kind;
    int8_t v;            // vectors per lane or thread; for an 'r' band, the ring's stages
    bool prefetch;
    int8_t team = 32;    // lanes per row of a 'w' band
    int16_t block = 0;   // threads per CTA of an 'x' band
};

constexpr int16_t kBandEnd = 32767;
constexpr int64_t kRingSmemLimit = 226 * 1024;  // dynamic shared memory a ring CTA may take
// BEGIN GENERATED OP BANDS
constexpr Band kSoftmax16[] = {{16, 'w', 2, true, 8}, {20, 'w', 4, false, 8}, {28, 'w', 4, true, 8}, {32, 'w', 2, true, 16}, {45, 'w', 4, false, 16}, {56, 'w', 4, true, 16}, {63, 'w', 2, true}, {112, 'w', 4, true}, {127, 'c', 4, false}, {129, 'w', 6, true}, {144, 'w', 6, false}, {169, 'w', 8, true}, {225, 'w', 8, false}, {512, 'g', 0, false}, {576, 'c', 4, true}, {640, 'g', 0, false}, {704, 'c', 4, true}, {768, 'g', 0, false}, {896, 'c', 4, true}, {1024, 'g', 0, false}, {2048, 'g', 0, true}, {2560, 'x', 4, true, 32, 128}, {6144, 'x', 4, true, 32, 256}, {8192, 'x', 4, true, 32, 512}, {kBandEnd, 'g', 0, true}};
constexpr Band kSoftmax32[] = {{8, 'w', 2, false, 8}, {12, 'w', 2, true, 8}, {20, 'w', 2, false, 16}, {28, 'w', 4, false, 8}, {32, 'w', 2, false}, {33, 'w', 4, false, 16}, {40, 'w', 2, false}, {53, 'w', 4, false, 16}, {56, 'w', 4, false}, {63, 'w', 4, true}, {64, 'g', 0, true}, {65, 'w', 4, false}, {72, 'w', 4, true}, {81, 'w', 6, false}, {96, 'w', 6, true}, {112, 'w', 8, false}, {127, 'c', 4, false}, {128, 'w', 4, false}, {129, 'w', 8, false}, {144, 'w', 8, true}, {168, 'w', 6, false}, {176, 'g', 0, false}, {177, 'c', 4, false}, {192, 'w', 6, false}, {208, 'c', 4, false}, {225, 'c', 4, true}, {256, 'w', 8, false}, {288, 'g', 0, false}, {320, 'c', 2, true}, {448, 'c', 4, true}, {512, 'c', 2, true}, {576, 'g', 0, false}, {640, 'c', 4, true}, {704, 'g', 0, false}, {768, 'c', 4, true}, {896, 'g', 0, false}, {1024, 'c', 4, true}, {1536, 'c', 4, false}, {1792, 'g', 0, true}, {2048, 'c', 4, false}, {2560, 'x', 4, true, 32, 128}, {6144, 'x', 4, true, 32, 256}, {8192, 'x', 4, true, 32, 512}, {kBandEnd, 'g', 0, true}};
constexpr Band kLayerNormBf16[] = {{16, 'w', 2, true, 8}, {28, 'w', 4, true, 8}, {32, 'w', 2, true, 16}, {52, 'w', 4, true, 16}, {53, 'w', 2, true}, {56, 'w', 4, true, 16}, {63, 'w', 2, true}, {64, 'w', 4, true, 16}, {127, 'w', 4, true}, {192, 'w', 6, true}, {256, 'w', 8, true}, {384, 'r', 2, true}, {448, 'r', 4, true}, {640, 'r', 2, true}, {704, 'R', 3, true}, {768, 'R', 2, true}, {1024, 'r', 4, true}, {1792, 'R', 2, true}, {2048, 'r', 2, true}, {2816, 'x', 4, true, 32, 128}, {3584, 'R', 2, true}, {4096, 'x', 4, true, 32, 256}, {kBandEnd, 'g', 0, true}};
constexpr Band kLayerNormF16[] = {{16, 'w', 2, true, 8}, {32, 'w', 4, true, 8}, {56, 'w', 4, true, 16}, {64, 'w', 2, true}, {128, 'w', 4, true}, {192, 'w', 6, true}, {448, 'g', 0, true}, {512, 'r', 3, true}, {576, 'c', 4, true}, {640, 'r', 6, true}, {704, 'R', 3, true}, {768, 'R', 2, true}, {896, 'c', 4, true}, {1024, 'r', 4, true}, {1280, 'R', 2, true}, {1408, 'x', 4, true, 32, 128}, {1792, 'R', 2, true}, {2048, 'c', 4, true}, {3072, 'x', 4, true, 32, 128}, {3584, 'R', 2, true}, {4096, 'x', 4, true, 32, 256}, {kBandEnd, 'g', 0, true}};
constexpr Band kLayerNormF32[] = {{16, 'w', 2, true, 8}, {32, 'w', 4, true, 8}, {52, 'w', 4, true, 16}, {53, 'w', 2, true}, {56, 'w', 4, true, 16}, {63, 'c', 2, true}, {64, 'w', 4, true, 16}, {112, 'w', 4, true}, {127, 'c', 4, true}, {169, 'w', 6, true}, {225, 'w', 8, true}, {256, 'g', 0, true}, {288, 'r', 2, true}, {320, 'c', 2, true}, {352, 'r', 6, true}, {512, 'g', 0, true}, {576, 'r', 2, true}, {640, 'c', 4, true}, {704, 'R', 4, true}, {768, 'c', 4, true}, {896, 'x', 4, true, 32, 128}, {1024, 'r', 6, true}, {1152, 'R', 3, true}, {1408, 'r', 2, true}, {1792, 'x', 4, true, 32, 128}, {3584, 'R', 2, true}, {4096, 'x', 4, true, 32, 256}, {kBandEnd, 'g', 0, true}};
// END GENERATED OP BANDS

// Applies the band of a row of hv vectors to p (the general rule's plan) when there are more rows
// than SMs; warp plans take 128-thread CTAs (4 rows each). The staged ring ('r') and the wide
// kernel ('x') were measured with many rows: on rows a register kernel can hold (at most 2048
// vectors) they apply only with at least 4 rows per SM, as the general rule's do.
void apply_band(const Band *bands, int64_t hv, int64_t rows, int sms, ks_plan_t *p) {
    if (rows <= sms) return;
    const Band *b = bands;
    while (hv > b->hi) ++b;
    const bool many = rows >= 4 * (int64_t)sms;
    const int64_t ring_block = round_up64(ceil_div64(hv, 4), 32);
    if (b->kind == 'w') {
        *p = op_plan_of(KS_KERNEL_WARP_ROW, b->v, 128, b->prefetch, 0, b->team);
    } else if (b->kind == 'c') {
        const int64_t block = round_up64(ceil_div64(hv, b->v), 32);
        if (block <= 512) *p = op_plan_of(KS_KERNEL_CTA_ROW, b->v, (int)block, b->prefetch);
    } else if (b->kind == 'r' || b->kind == 'R') {
        const int64_t affine = b->kind == 'R' ? 2 * hv * 16 : 0;  // weight and bias rows
        const int64_t max_block = b->kind == 'R' ? 1024 : 512;
        if (many && ring_block <= max_block && 128 + (int64_t)b->v * hv * 16 + affine <= kRingSmemLimit) {
            *p = op_plan_of(KS_KERNEL_BULK_ROW, 4, (int)ring_block, true, b->v);
            if (b->kind == 'R') p->flags |= KS_PLAN_AFFINE_SMEM;
        }
    } else if (b->kind == 'x') {
        if (many || hv > 2048) *p = op_plan_of(KS_KERNEL_TWOPASS_ROW, 4, b->block, true);
    }
}

// Softmax: rows of up to 512 threads x V vectors in registers (V from row_vec_plan; at 4 vectors
// no prefetch up to 1024 vectors: measured on GB300 (bf16, HBM-bound rows) 0.92-0.97 of the copy
// peak for rows of 128..1024 vectors against 0.85-0.93 with it; beyond, prefetch wins), the wide
// kernel for wider rows, the scalar kernel for rows that cannot be vectorised; many rows of at
// most 256 vectors by the bands above. `width` is in 16-byte vectors when aligned, else elements.
ks_plan_t softmax_plan(bool aligned, int64_t width, int64_t rows, int sms, ks_dtype_t dtype) {
    if (!aligned) return op_plan_of(KS_KERNEL_SCALAR, 0, scalar_block(width, 1024), true);
    int block = 0;
    const int v = row_vec_plan(width, &block);
    ks_plan_t p = v == 0 ? op_plan_of(KS_KERNEL_TWOPASS_ROW, 4, wide_row_block(width, false), true)
                         : op_plan_of(KS_KERNEL_CTA_ROW, v, block, v != 4 || width > 1024);
    apply_band(dtype == KS_DTYPE_F32 ? kSoftmax32 : kSoftmax16, width, rows, sms, &p);
    return p;
}

// Bytes of rows in each CTA's LayerNorm ring (a tuning constant, set from a GB300 measurement).
#ifndef KS_LN_RING_BYTES
#define KS_LN_RING_BYTES (64 * 1024)
#endif

// LayerNorm: register rows (V from row_vec_plan, next row always prefetched: without it the two
// reductions per row left it at 0.50-0.66 of the copy peak), the wide kernel for wider rows, the
// scalar kernel for rows that cannot be vectorised; many rows of at most 256 vectors by the bands
// above. Many rows (at least 4 per SM) wider than 512 vectors: the staged ring (KS_LN_RING_BYTES
// of rows per CTA, 2..8 stages) keeps enough bytes in flight, where the register kernel measured
// faster up to 512 vectors (0.74-0.82 of the copy peak against 0.65-0.69 for the ring). Between
// 1024 and 2048 vectors the ring's CTA (a thread per 4 vectors, ~105 registers for 16-bit types)
// leaves one CTA of 8-14 warps per SM; the wide kernel's 128-thread CTAs keep more warps resident
// and measured faster on GB300 for many rows: bf16 1280..1792 vectors 0.76-0.83 of the copy peak
// against 0.65-0.78, fp32 1024..1792 0.88-0.95 against 0.76-0.86 (at 1024 bf16 vectors the ring
// measured 0.96 against 0.81, so 16-bit rows start above it).
ks_plan_t layer_norm_plan(bool aligned, int64_t hv, int64_t hidden, int64_t rows, int sms,
                          ks_dtype_t dtype) {
    if (!aligned) return op_plan_of(KS_KERNEL_SCALAR, 0, scalar_block(hidden, 1024), true);
    int block = 0;
    const int v = row_vec_plan(hv, &block);
    ks_plan_t p = v == 0 ? op_plan_of(KS_KERNEL_TWOPASS_ROW, 4, wide_row_block(hv, true), true)
                         : op_plan_of(KS_KERNEL_CTA_ROW, v, block, true);
    if (p.kernel == KS_KERNEL_CTA_ROW && v == 4 && hv > 512 && rows >= 4 * (int64_t)sms) {
        if (hv < 2048 && hv >= (dtype == KS_DTYPE_F32 ? 1024 : 1025)) {
            p = op_plan_of(KS_KERNEL_TWOPASS_ROW, 4, 128, true);
        } else {
            const int64_t n = (KS_LN_RING_BYTES) / (hv * 16);
            p = op_plan_of(KS_KERNEL_BULK_ROW, 4, block, true, (int)(n < 2 ? 2 : (n > 8 ? 8 : n)));
        }
    }
    apply_band(dtype == KS_DTYPE_BF16 ? kLayerNormBf16
               : dtype == KS_DTYPE_F16 ? kLayerNormF16 : kLayerNormF32, hv, rows, sms, &p);
    return p;
}

// The ring's dynamic shared memory: its mbarriers, then `stages` rows of hv vectors.
size_t ln_ring_smem(int stages, int64_t hv) { return 128 + (size_t)stages * (size_t)hv * 16; }

// Checks an explicit plan for op (2 SwiGLU, 3 Softmax, 4 LayerNorm) against the call, before any
// CUDA call; `vec` tells whether the rows and pointers take 16-byte vectors, `width` is the row's
// width in 16-byte vectors when they do (for SwiGLU the output row's), `elems` in elements.
ks_status_t op_check(int op, ks_plan_t &p, bool vec, int64_t width, int64_t elems) {
    if (p.flags & ~(KS_PLAN_NO_PREFETCH | KS_PLAN_PDL | KS_PLAN_AFFINE_SMEM))
        return fail(KS_ERR_INVALID_ARGUMENT, "unknown plan flags 0x%x", (unsigned)p.flags);
    if ((p.flags & KS_PLAN_AFFINE_SMEM) && !(op == kOpLayerNorm && p.kernel == KS_KERNEL_BULK_ROW))
        return fail(KS_ERR_INVALID_ARGUMENT, "KS_PLAN_AFFINE_SMEM is for LayerNorm's staged ring");
    if (p.block < 32 || p.block % 32 != 0)
        return fail(KS_ERR_INVALID_ARGUMENT, "plan block %d is not a positive multiple of 32", p.block);
    if (p.kernel != KS_KERNEL_SCALAR && !vec)
        return fail(KS_ERR_INVALID_ARGUMENT, "vector kernel needs 16-byte rows and pointers");
    const bool pf = op_prefetch(p);
    p.cluster = 0;
    p.smem_bytes = 0;
    if (op == kOpSilu) {
        if (p.block > 256) return fail(KS_ERR_INVALID_ARGUMENT, "SwiGLU block > 256");
        if (p.kernel != KS_KERNEL_FLAT && p.kernel != KS_KERNEL_CTA_ROW && p.kernel != KS_KERNEL_SCALAR)
            return fail(KS_ERR_INVALID_ARGUMENT, "SwiGLU takes the flat, row or scalar kernel");
        p.stages = 0;
        p.team = p.block;
        return KS_SUCCESS;
    }
    const bool ln = op == kOpLayerNorm;
    if (p.kernel != KS_KERNEL_BULK_ROW) p.stages = 0;
    switch (p.kernel) {
    case KS_KERNEL_WARP_ROW:
        if (p.team == 0) p.team = 32;
        if (p.team != 32 && p.team != 16 && p.team != 8)
            return fail(KS_ERR_INVALID_ARGUMENT, "warp-row teams are 32, 16 or 8 lanes (got %d)", p.team);
        if (p.team == 32 ? (p.vec_per_thread != 2 && p.vec_per_thread != 4 &&
                            p.vec_per_thread != 6 && p.vec_per_thread != 8)
                         : (p.vec_per_thread != 2 && p.vec_per_thread != 4))
            return fail(KS_ERR_INVALID_ARGUMENT, "warp rows take 2, 4, 6 or 8 vectors per lane "
                        "(teams of 8 or 16 lanes: 2 or 4)");
        if ((int64_t)p.team * p.vec_per_thread < width || p.block > 128)
            return fail(KS_ERR_INVALID_ARGUMENT, "warp-row plan does not cover the row or block > 128");
        if (ln && !pf) return fail(KS_ERR_INVALID_ARGUMENT, "LayerNorm rows always prefetch");
        return KS_SUCCESS;
    case KS_KERNEL_CTA_ROW:
        if (p.vec_per_thread != 1 && p.vec_per_thread != 2 && p.vec_per_thread != 4)
            return fail(KS_ERR_INVALID_ARGUMENT, "CTA rows take 1, 2 or 4 vectors per thread");
        if ((int64_t)p.block * p.vec_per_thread < width || p.block > 512)
            return fail(KS_ERR_INVALID_ARGUMENT, "CTA-row plan does not cover the row or block > 512");
        if (!pf && (ln || p.vec_per_thread != 4))
            return fail(KS_ERR_INVALID_ARGUMENT, "no variant without prefetch for this plan");
        break;
    case KS_KERNEL_BULK_ROW:
        if (!ln) return fail(KS_ERR_INVALID_ARGUMENT, "the staged ring is LayerNorm's");
        if (p.vec_per_thread != 4 || (int64_t)p.block * 4 < width ||
            p.block > ((p.flags & KS_PLAN_AFFINE_SMEM) ? 1024 : 512))
            return fail(KS_ERR_INVALID_ARGUMENT, "ring plan: 4 vectors per thread covering the row, "
                        "block <= 512 (1024 with KS_PLAN_AFFINE_SMEM)");
        {
            // with the weight and bias in shared memory too (counted for both)
            const int64_t affine = (p.flags & KS_PLAN_AFFINE_SMEM) ? 2 * width * 16 : 0;
            if (p.stages < 2 || p.stages > 8 ||
                (int64_t)ln_ring_smem(p.stages, width) + affine > kRingSmemLimit)
                return fail(KS_ERR_INVALID_ARGUMENT, "ring of %d stages does not fit", p.stages);
            p.smem_bytes = (int32_t)(ln_ring_smem(p.stages, width) + affine);
        }
        break;
    case KS_KERNEL_TWOPASS_ROW:
        if (p.vec_per_thread != 4 || p.block > (ln ? 512 : 1024))
            return fail(KS_ERR_INVALID_ARGUMENT, "wide kernel: 4 vectors a step, block <= %d", ln ? 512 : 1024);
        break;
    case KS_KERNEL_SCALAR:
        if (p.block > 1024) return fail(KS_ERR_INVALID_ARGUMENT, "scalar block > 1024");
        p.vec_per_thread = 0;
        break;
    default:
        return fail(KS_ERR_INVALID_ARGUMENT, "kernel %d is not one of this operator's", p.kernel);
    }
    (void)elems;
    p.team = p.block;
    return KS_SUCCESS;
}

// A launch with programmatic dependent launch when `pdl`.
cudaError_t launch_ex(const void *f, dim3 grid, dim3 block, size_t smem, void **args,
                      cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, f, args);
}

int64_t cap_grid(int64_t grid, const ks_plan_t &p) {
    return (p.grid > 0 && grid > p.grid) ? p.grid : grid;
}

template <typename T>
cudaError_t silu_dispatch(const ks_plan_t &p, void *out, const void *x, int64_t rows, int64_t d,
                          int sms, cudaStream_t s, bool pdl) {
    int64_t nr = rows, dd = p.kernel == KS_KERNEL_SCALAR ? d : d / Elem<T>::kPerVec;
    void *args[] = {&out, const_cast<void **>(&x), &nr, &dd};
    if (p.kernel == KS_KERNEL_FLAT) {
        // a persistent grid of as many CTAs as are resident at once (fewer if the vectors run
        // out), two vectors per thread per iteration
        const void *f = (const void *)silu_mul_flat_kernel<T>;
        const int n = cached_occupancy(f, p.block, 0);
        int64_t grid = ceil_div64(rows * dd, 2 * (int64_t)p.block);
        grid = cap_grid(grid > (int64_t)sms * n ? (int64_t)sms * n : grid, p);
        return launch_ex(f, dim3((unsigned)grid), dim3(p.block), 0, args, s, pdl);
    }
    if (p.kernel == KS_KERNEL_CTA_ROW) {
        // gx CTAs across a row, each of bx threads covering two vectors a thread (bx a multiple
        // of 32, at most p.block); narrow rows stack 256 / bx rows per CTA; as many CTAs as are
        // resident at once (a CTA left for a second wave of this persistent grid would start only
        // when a first-wave one has finished all its rows)
        const void *f = (const void *)silu_mul_rows_kernel<T>;
        // the fewest CTAs across the row whose threads leave the fewest idle: 576 vectors run as
        // 3 CTAs of 96 threads (no idle thread) rather than 2 of 160 (64 idle), which measured
        // 0.93 against 0.90 of the copy peak
        int64_t gx = ceil_div64(dd, 2 * (int64_t)p.block);
        int bx = (int)round_up64(ceil_div64(dd, 2 * gx), 32);
        for (int64_t g2 = gx + 1; g2 <= 4 * gx && 2 * gx * bx > dd; ++g2) {
            const int b2 = (int)round_up64(ceil_div64(dd, 2 * g2), 32);
            if (2 * g2 * b2 < 2 * gx * bx) {
                gx = g2;
                bx = b2;
            }
        }
        int64_t by = 256 / bx;
        by = by > rows ? rows : by;
        int64_t gy = ceil_div64(rows, by);
        int64_t cap = (int64_t)sms * cached_occupancy(f, bx * (int)by, 0) / gx;
        if (p.grid > 0 && cap > p.grid / gx) cap = p.grid / gx;
        gy = gy > cap ? cap : gy;
        gy = gy < 1 ? 1 : (gy > 65535 ? 65535 : gy);
        return launch_ex(f, dim3((unsigned)gx, (unsigned)gy), dim3((unsigned)bx, (unsigned)by), 0,
                         args, s, pdl);
    }
    // scalar: enough CTAs to cover a row once; rows: fill ~8 waves of SMs
    int64_t gx = ceil_div64(d, p.block);
    gx = gx < 1 ? 1 : gx;
    int64_t gy = (int64_t)sms * 8 / gx;
    if (p.grid > 0 && gy > p.grid / gx) gy = p.grid / gx;
    gy = gy < 1 ? 1 : (gy > rows ? rows : gy);
    gy = gy > 65535 ? 65535 : gy;
    return launch_ex((const void *)silu_mul_scalar_kernel<T>, dim3((unsigned)gx, (unsigned)gy),
                     dim3(p.block), 0, args, s, pdl);
}

// Grid of a register-row launch: as many CTAs as are resident at once, no more than the rows
// need (warp plans: block / 32 rows per CTA), no more than the plan's grid when it gives one.
int64_t reg_grid(const void *f, const ks_plan_t &p, size_t smem, int64_t rows, int sms) {
    const int n = cached_occupancy(f, p.block, smem);
    const int64_t per_cta = p.kernel == KS_KERNEL_WARP_ROW ? p.block / p.team : 1;
    const int64_t need = ceil_div64(rows, per_cta);
    const int64_t grid = (int64_t)sms * n;
    return cap_grid(grid > need ? need : grid, p);
}

template <typename T>
cudaError_t softmax_dispatch(const ks_plan_t &p, void *out, const void *x, int64_t rows,
                             int64_t width, int sms, cudaStream_t s, bool pdl) {
    int64_t nr = rows, wd = width;
    void *args[] = {&out, const_cast<void **>(&x), &nr, &wd};
    const bool pf = op_prefetch(p);
    const void *f = nullptr;
    switch (p.kernel) {
    case KS_KERNEL_WARP_ROW:
        switch (p.team * 16 + p.vec_per_thread) {
        case 32 * 16 + 2: f = pf ? (const void *)softmax_vec_kernel<T, 2, true, 32>
                                 : (const void *)softmax_vec_kernel<T, 2, false, 32>; break;
        case 32 * 16 + 4: f = pf ? (const void *)softmax_vec_kernel<T, 4, true, 32>
                                 : (const void *)softmax_vec_kernel<T, 4, false, 32>; break;
        case 32 * 16 + 6: f = pf ? (const void *)softmax_vec_kernel<T, 6, true, 32>
                                 : (const void *)softmax_vec_kernel<T, 6, false, 32>; break;
        case 32 * 16 + 8: f = pf ? (const void *)softmax_vec_kernel<T, 8, true, 32>
                                 : (const void *)softmax_vec_kernel<T, 8, false, 32>; break;
        case 16 * 16 + 2: f = pf ? (const void *)softmax_vec_kernel<T, 2, true, 16>
                                 : (const void *)softmax_vec_kernel<T, 2, false, 16>; break;
        case 16 * 16 + 4: f = pf ? (const void *)softmax_vec_kernel<T, 4, true, 16>
                                 : (const void *)softmax_vec_kernel<T, 4, false, 16>; break;
        case 8 * 16 + 2: f = pf ? (const void *)softmax_vec_kernel<T, 2, true, 8>
                                : (const void *)softmax_vec_kernel<T, 2, false, 8>; break;
        case 8 * 16 + 4: f = pf ? (const void *)softmax_vec_kernel<T, 4, true, 8>
                                : (const void *)softmax_vec_kernel<T, 4, false, 8>; break;
        default: return cudaErrorInvalidConfiguration;
        }
        break;
    case KS_KERNEL_CTA_ROW:
        switch (p.vec_per_thread) {
        case 1: f = (const void *)softmax_vec_kernel<T, 1, true>; break;
        case 2: f = (const void *)softmax_vec_kernel<T, 2, true>; break;
        case 4: f = pf ? (const void *)softmax_vec_kernel<T, 4, true>
                       : (const void *)softmax_vec_kernel<T, 4, false>; break;
        default: return cudaErrorInvalidConfiguration;
        }
        break;
    case KS_KERNEL_TWOPASS_ROW: f = (const void *)softmax_wide_kernel<T, 4>; break;
    case KS_KERNEL_SCALAR: f = (const void *)softmax_scalar_kernel<T>; break;
    default: return cudaErrorInvalidConfiguration;
    }
    int64_t grid = reg_grid(f, p, 0, rows, sms);
    if (p.kernel == KS_KERNEL_TWOPASS_ROW && grid > wide_grid_cap(width, sms))
        grid = wide_grid_cap(width, sms);
    return launch_ex(f, dim3((unsigned)grid), dim3(p.block), 0, args, s, pdl);
}

// The instantiation of a LayerNorm kernel for the weight/bias combination of the call.
template <typename T, typename K>
const void *layer_norm_pick(int affine, K none, K weight, K bias, K both) {
    switch (affine) {
    case kAffineWeight: return (const void *)weight;
    case kAffineBias: return (const void *)bias;
    case kAffineWeight | kAffineBias: return (const void *)both;
    default: return (const void *)none;
    }
}

template <typename T>
cudaError_t layer_norm_dispatch(const ks_plan_t &p, void *out, const void *x, const void *w,
                                const void *b, int64_t rows, int64_t hidden, int64_t hv,
                                float eps, int sms, cudaStream_t s, bool pdl) {
    int64_t nr = rows, hd = hidden, hvv = hv;
    float ep = eps;
    int stages = p.stages;
    void *vec_args[] = {&out, const_cast<void **>(&x), const_cast<void **>(&w),
                        const_cast<void **>(&b), &nr, &hd, &hvv, &ep};
    void *sc_args[] = {&out, const_cast<void **>(&x), const_cast<void **>(&w),
                       const_cast<void **>(&b), &nr, &hd, &ep};
    void *bulk_args[] = {&out, const_cast<void **>(&x), const_cast<void **>(&w),
                         const_cast<void **>(&b), &nr, &hd, &hvv, &ep, &stages};
    void **args = vec_args;
    size_t smem = 0;
    const int affine = (w ? kAffineWeight : 0) | (b ? kAffineBias : 0);
    const void *f = nullptr;
    switch (p.kernel) {
    case KS_KERNEL_WARP_ROW:
        switch (p.team * 16 + p.vec_per_thread) {
        case 32 * 16 + 2: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 2, 0, 32>, layer_norm_vec_kernel<T, 2, 1, 32>,
                                                 layer_norm_vec_kernel<T, 2, 2, 32>, layer_norm_vec_kernel<T, 2, 3, 32>); break;
        case 32 * 16 + 4: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 4, 0, 32>, layer_norm_vec_kernel<T, 4, 1, 32>,
                                                 layer_norm_vec_kernel<T, 4, 2, 32>, layer_norm_vec_kernel<T, 4, 3, 32>); break;
        case 32 * 16 + 6: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 6, 0, 32>, layer_norm_vec_kernel<T, 6, 1, 32>,
                                                 layer_norm_vec_kernel<T, 6, 2, 32>, layer_norm_vec_kernel<T, 6, 3, 32>); break;
        case 32 * 16 + 8: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 8, 0, 32>, layer_norm_vec_kernel<T, 8, 1, 32>,
                                                 layer_norm_vec_kernel<T, 8, 2, 32>, layer_norm_vec_kernel<T, 8, 3, 32>); break;
        case 16 * 16 + 2: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 2, 0, 16>, layer_norm_vec_kernel<T, 2, 1, 16>,
                                                 layer_norm_vec_kernel<T, 2, 2, 16>, layer_norm_vec_kernel<T, 2, 3, 16>); break;
        case 16 * 16 + 4: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 4, 0, 16>, layer_norm_vec_kernel<T, 4, 1, 16>,
                                                 layer_norm_vec_kernel<T, 4, 2, 16>, layer_norm_vec_kernel<T, 4, 3, 16>); break;
        case 8 * 16 + 2: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 2, 0, 8>, layer_norm_vec_kernel<T, 2, 1, 8>,
                                                layer_norm_vec_kernel<T, 2, 2, 8>, layer_norm_vec_kernel<T, 2, 3, 8>); break;
        case 8 * 16 + 4: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 4, 0, 8>, layer_norm_vec_kernel<T, 4, 1, 8>,
                                                layer_norm_vec_kernel<T, 4, 2, 8>, layer_norm_vec_kernel<T, 4, 3, 8>); break;
        default: return cudaErrorInvalidConfiguration;
        }
        break;
    case KS_KERNEL_CTA_ROW:
        switch (p.vec_per_thread) {
        case 1: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 1, 0>, layer_norm_vec_kernel<T, 1, 1>,
                                       layer_norm_vec_kernel<T, 1, 2>, layer_norm_vec_kernel<T, 1, 3>); break;
        case 2: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 2, 0>, layer_norm_vec_kernel<T, 2, 1>,
                                       layer_norm_vec_kernel<T, 2, 2>, layer_norm_vec_kernel<T, 2, 3>); break;
        case 4: f = layer_norm_pick<T>(affine, layer_norm_vec_kernel<T, 4, 0>, layer_norm_vec_kernel<T, 4, 1>,
                                       layer_norm_vec_kernel<T, 4, 2>, layer_norm_vec_kernel<T, 4, 3>); break;
        default: return cudaErrorInvalidConfiguration;
        }
        break;
    case KS_KERNEL_TWOPASS_ROW:
        f = layer_norm_pick<T>(affine, layer_norm_wide_kernel<T, 4, 0>, layer_norm_wide_kernel<T, 4, 1>,
                               layer_norm_wide_kernel<T, 4, 2>, layer_norm_wide_kernel<T, 4, 3>);
        break;
    case KS_KERNEL_BULK_ROW:
        if (p.flags & KS_PLAN_AFFINE_SMEM) {
            f = layer_norm_pick<T>(affine, layer_norm_bulk_kernel<T, 4, 0, true>,
                                   layer_norm_bulk_kernel<T, 4, 1, true>,
                                   layer_norm_bulk_kernel<T, 4, 2, true>,
                                   layer_norm_bulk_kernel<T, 4, 3, true>);
            smem = ln_ring_smem(stages, hv) + (size_t)((w ? 1 : 0) + (b ? 1 : 0)) * (size_t)hv * 16;
        } else {
            f = layer_norm_pick<T>(affine, layer_norm_bulk_kernel<T, 4, 0>, layer_norm_bulk_kernel<T, 4, 1>,
                                   layer_norm_bulk_kernel<T, 4, 2>, layer_norm_bulk_kernel<T, 4, 3>);
            smem = ln_ring_smem(stages, hv);
        }
        args = bulk_args;
        break;
    case KS_KERNEL_SCALAR:
        f = layer_norm_pick<T>(affine, layer_norm_scalar_kernel<T, 0>, layer_norm_scalar_kernel<T, 1>,
                               layer_norm_scalar_kernel<T, 2>, layer_norm_scalar_kernel<T, 3>);
        args = sc_args;
        break;
    default: return cudaErrorInvalidConfiguration;
    }
    // allow the largest ring the device takes beside the kernel's static shared memory
    if (smem > 0 && !allow_dynamic_smem(f, smem)) return cudaErrorInvalidConfiguration;
    int64_t grid = reg_grid(f, p, smem, rows, sms);
    if (p.kernel == KS_KERNEL_TWOPASS_ROW && grid > wide_grid_cap(hv, sms)) grid = wide_grid_cap(hv, sms);
    return launch_ex(f, dim3((unsigned)grid), dim3(p.block), smem, args, s, pdl);
}

// The default plan of op (2 SwiGLU, 3 Softmax, 4 LayerNorm) for a call; for SwiGLU `hidden` is
// the output row's width d. Pure host code.
ks_plan_t op_default_plan(int op, int64_t rows, int64_t hidden, ks_dtype_t dtype, bool aligned16,
                          int sms) {
    const int e = elem_bytes(dtype);
    const bool vec = aligned16 && (hidden * e) % 16 == 0;
    const int64_t hv = vec ? hidden * e / 16 : 0;
    if (op == kOpSilu) return silu_plan(vec, hv, dtype);
    if (op == kOpSoftmax) return softmax_plan(vec, vec ? hv : hidden, rows, sms, dtype);
    return layer_norm_plan(vec, hv, hidden, rows, sms, dtype);
}

// The launch plan a call runs: `forced` checked against the call, or the default plan.
ks_status_t resolve_op_plan(int op, const ks_plan_t *forced, int64_t rows, int64_t hidden,
                            ks_dtype_t dtype, bool aligned16, int sms, ks_plan_t *p, bool *pdl) {
    if (!forced) {
        *p = op_default_plan(op, rows, hidden, dtype, aligned16, sms);
        *pdl = launch_pdl_enabled();
        return KS_SUCCESS;
    }
    *p = *forced;
    const int e = elem_bytes(dtype);
    const bool vec = aligned16 && (hidden * e) % 16 == 0;
    *pdl = (p->flags & KS_PLAN_PDL) != 0;
    return op_check(op, *p, vec, vec ? hidden * e / 16 : 0, hidden);
}

}  // namespace

ks_status_t op_plan(int op, int64_t rows, int64_t hidden, ks_dtype_t dtype, bool aligned16,
                    int sm_count, ks_plan_t *p) {
    if (rows == 0) {
        memset(p, 0, sizeof *p);
        p->kernel = KS_KERNEL_NONE;
        return KS_SUCCESS;
    }
    *p = op_default_plan(op, rows, hidden, dtype, aligned16, sm_count);
    return KS_SUCCESS;
}

int fault_flags_ops(bool clear) { return fault_flags_t(clear); }

}  // namespace ks

using namespace ks;

namespace {

ks_status_t silu_and_mul(void *out, const void *x, int64_t rows, int64_t d, ks_dtype_t dtype,
                         const ks_plan_t *forced, ks_stream_t stream) {
    int e = 0;
    ks_status_t st = check_common(rows, d, dtype, &e);
    if (st != KS_SUCCESS) return st;
    if (rows == 0) return KS_SUCCESS;
    if (!out || !x) return fail(KS_ERR_INVALID_ARGUMENT, "NULL pointer with rows > 0");
    if (misaligned(e, out, x))
        return fail(KS_ERR_INVALID_ARGUMENT, "a pointer is not aligned to the %d-byte element", e);
    if (overlaps(out, rows * d * e, x, rows * 2 * d * e))
        return fail(KS_ERR_OVERLAP, "out and x storage overlap");
    const bool al = (((uintptr_t)out | (uintptr_t)x) & 15u) == 0;
    ks_plan_t p;
    bool pdl = false;
    if (forced && (st = resolve_op_plan(kOpSilu, forced, rows, d, dtype, al, 1, &p, &pdl)) != KS_SUCCESS)
        return st;
    int sms = 0;
    if ((st = sm_count(&sms)) != KS_SUCCESS) return st;
    if (!forced) resolve_op_plan(kOpSilu, nullptr, rows, d, dtype, al, sms, &p, &pdl);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t ce;
    switch (dtype) {
    case KS_DTYPE_BF16: ce = silu_dispatch<__nv_bfloat16>(p, out, x, rows, d, sms, s, pdl); break;
    case KS_DTYPE_F16: ce = silu_dispatch<__half>(p, out, x, rows, d, sms, s, pdl); break;
    default: ce = silu_dispatch<float>(p, out, x, rows, d, sms, s, pdl); break;
    }
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "launch: %s", cudaGetErrorString(ce));
    return KS_SUCCESS;
}

ks_status_t softmax(void *out, const void *x, int64_t rows, int64_t hidden, ks_dtype_t dtype,
                    const ks_plan_t *forced, ks_stream_t stream) {
    int e = 0;
    ks_status_t st = check_common(rows, hidden, dtype, &e);
    if (st != KS_SUCCESS) return st;
    if (rows == 0) return KS_SUCCESS;
    if (!out || !x) return fail(KS_ERR_INVALID_ARGUMENT, "NULL pointer with rows > 0");
    if (misaligned(e, out, x))
        return fail(KS_ERR_INVALID_ARGUMENT, "a pointer is not aligned to the %d-byte element", e);
    const int64_t nbytes = rows * hidden * e;
    if (out != x && overlaps(out, nbytes, x, nbytes))
        return fail(KS_ERR_OVERLAP, "out partially overlaps x (only out == x is allowed)");
    const bool al = (((uintptr_t)out | (uintptr_t)x) & 15u) == 0;
    ks_plan_t p;
    bool pdl = false;
    if (forced && (st = resolve_op_plan(kOpSoftmax, forced, rows, hidden, dtype, al, 1, &p, &pdl)) != KS_SUCCESS)
        return st;
    int sms = 0;
    if ((st = sm_count(&sms)) != KS_SUCCESS) return st;
    if (!forced) resolve_op_plan(kOpSoftmax, nullptr, rows, hidden, dtype, al, sms, &p, &pdl);
    // the vector kernels take the row's width in 16-byte vectors, the scalar kernel in elements
    const bool vec = al && (hidden * e) % 16 == 0 && p.kernel != KS_KERNEL_SCALAR;
    const int64_t width = vec ? hidden * e / 16 : hidden;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t ce;
    switch (dtype) {
    case KS_DTYPE_BF16: ce = softmax_dispatch<__nv_bfloat16>(p, out, x, rows, width, sms, s, pdl); break;
    case KS_DTYPE_F16: ce = softmax_dispatch<__half>(p, out, x, rows, width, sms, s, pdl); break;
    default: ce = softmax_dispatch<float>(p, out, x, rows, width, sms, s, pdl); break;
    }
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "launch: %s", cudaGetErrorString(ce));
    return KS_SUCCESS;
}

ks_status_t layer_norm(void *out, const void *x, const void *weight, const void *bias,
                       int64_t rows, int64_t hidden, float eps, ks_dtype_t dtype,
                       const ks_plan_t *forced, ks_stream_t stream) {
    int e = 0;
    ks_status_t st = check_common(rows, hidden, dtype, &e);
    if (st != KS_SUCCESS) return st;
    if (!std::isfinite(eps) || !(eps > 0.0f))
        return fail(KS_ERR_INVALID_ARGUMENT, "eps must be finite and > 0 (got %g)", (double)eps);
    if (rows == 0) return KS_SUCCESS;
    if (!out || !x) return fail(KS_ERR_INVALID_ARGUMENT, "NULL pointer with rows > 0");
    if (misaligned(e, out, x, weight, bias))
        return fail(KS_ERR_INVALID_ARGUMENT, "a pointer is not aligned to the %d-byte element", e);
    const int64_t nbytes = rows * hidden * e, pbytes = hidden * e;
    if (out != x && overlaps(out, nbytes, x, nbytes))
        return fail(KS_ERR_OVERLAP, "out partially overlaps x (only out == x is allowed)");
    if ((weight && overlaps(out, nbytes, weight, pbytes)) || (bias && overlaps(out, nbytes, bias, pbytes)))
        return fail(KS_ERR_OVERLAP, "out overlaps weight or bias storage");
    const uintptr_t a = (uintptr_t)out | (uintptr_t)x | (uintptr_t)weight | (uintptr_t)bias;
    const bool al = (a & 15u) == 0;
    ks_plan_t p;
    bool pdl = false;
    if (forced && (st = resolve_op_plan(kOpLayerNorm, forced, rows, hidden, dtype, al, 1, &p, &pdl)) != KS_SUCCESS)
        return st;
    int sms = 0;
    if ((st = sm_count(&sms)) != KS_SUCCESS) return st;
    if (!forced) resolve_op_plan(kOpLayerNorm, nullptr, rows, hidden, dtype, al, sms, &p, &pdl);
    const int64_t hv = hidden * e / 16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t ce;
    switch (dtype) {
    case KS_DTYPE_BF16: ce = layer_norm_dispatch<__nv_bfloat16>(p, out, x, weight, bias, rows, hidden, hv, eps, sms, s, pdl); break;
    case KS_DTYPE_F16: ce = layer_norm_dispatch<__half>(p, out, x, weight, bias, rows, hidden, hv, eps, sms, s, pdl); break;
    default: ce = layer_norm_dispatch<float>(p, out, x, weight, bias, rows, hidden, hv, eps, sms, s, pdl); break;
    }
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "launch: %s", cudaGetErrorString(ce));
    return KS_SUCCESS;
}

}  // namespace

extern "C" {

ks_status_t ks_silu_and_mul(void *out, const void *x, int64_t rows, int64_t d, ks_dtype_t dtype,
                            ks_stream_t stream) {
    return silu_and_mul(out, x, rows, d, dtype, nullptr, stream);
}

ks_status_t ks_silu_and_mul_planned(void *out, const void *x, int64_t rows, int64_t d,
                                    ks_dtype_t dtype, const ks_plan_t *plan, ks_stream_t stream) {
    if (!plan) return fail(KS_ERR_INVALID_ARGUMENT, "plan is NULL");
    return silu_and_mul(out, x, rows, d, dtype, plan, stream);
}

ks_status_t ks_softmax(void *out, const void *x, int64_t rows, int64_t hidden, ks_dtype_t dtype,
                       ks_stream_t stream) {
    return softmax(out, x, rows, hidden, dtype, nullptr, stream);
}

ks_status_t ks_softmax_planned(void *out, const void *x, int64_t rows, int64_t hidden,
                               ks_dtype_t dtype, const ks_plan_t *plan, ks_stream_t stream) {
    if (!plan) return fail(KS_ERR_INVALID_ARGUMENT, "plan is NULL");
    return softmax(out, x, rows, hidden, dtype, plan, stream);
}

ks_status_t ks_layer_norm(void *out, const void *x, const void *weight, const void *bias,
                          int64_t rows, int64_t hidden, float eps, ks_dtype_t dtype,
                          ks_stream_t stream) {
    return layer_norm(out, x, weight, bias, rows, hidden, eps, dtype, nullptr, stream);
}

ks_status_t ks_layer_norm_planned(void *out, const void *x, const void *weight, const void *bias,
                                  int64_t rows, int64_t hidden, float eps, ks_dtype_t dtype,
                                  const ks_plan_t *plan, ks_stream_t stream) {
    if (!plan) return fail(KS_ERR_INVALID_ARGUMENT, "plan is NULL");
    return layer_norm(out, x, weight, bias, rows, hidden, eps, dtype, plan, stream);
}

}  // extern "C"
