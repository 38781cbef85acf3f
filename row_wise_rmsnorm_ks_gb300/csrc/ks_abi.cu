// The C ABI of libks (include/ks.h): argument checks, the launch-plan heuristic, per-device
// caches and the launch itself. Host code only; the kernels live in ks_kernels.cuh.
//
// Boundary style after kernel-set ("Operators": a status return, device pointers and a stream);
// validation rules after Kernscope ("API contract / Inputs": a non-empty last dimension,
// contiguous storage, one dtype, eps finite and positive; fused: same shape, no overlapping
// storage, in place).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "ks_internal.h"

namespace ks {
namespace {

thread_local char g_detail[256] = "";

ks_status_t fail(ks_status_t s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
    return s;
}

int elem_bytes(ks_dtype_t d) {
    switch (d) {
    case KS_DTYPE_F32: return 4;
    case KS_DTYPE_F16: return 2;
    case KS_DTYPE_BF16: return 2;
    default: return 0;
    }
}

// [a, a+na) and [b, b+nb) share a byte.
bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ---------------------------------------------------------------- per-device caches

constexpr int kMaxDevices = 64;

struct DeviceSlot {
    std::once_flag once;
    int sm_count = 0;
    cudaError_t err = cudaSuccess;
};
DeviceSlot g_devices[kMaxDevices];

std::mutex g_occ_mu;
std::unordered_map<uint64_t, int> g_occ;  // (device, dtype, fused, kernel, vec, block) -> CTAs/SM

uint64_t occ_key(int dev, ks_dtype_t d, bool fused, const ks_plan_t &p) {
    return ((uint64_t)dev << 48) | ((uint64_t)d << 44) | ((uint64_t)fused << 43) |
           ((uint64_t)p.kernel << 36) | ((uint64_t)p.vec_per_thread << 24) | (uint64_t)p.block;
}

int query_blocks_per_sm(ks_dtype_t d, const ks_plan_t &p, bool fused) {
    switch (d) {
    case KS_DTYPE_BF16: return blocks_per_sm_bf16(p, fused);
    case KS_DTYPE_F16: return blocks_per_sm_f16(p, fused);
    default: return blocks_per_sm_f32(p, fused);
    }
}

ks_status_t run(bool fused, void *out, const void *x, void *res, const void *w, int64_t rows,
                int64_t hidden, float eps, ks_dtype_t dtype, ks_stream_t stream) {
    // ---- argument checks: no CUDA call before all of them pass
    const int e = elem_bytes(dtype);
    if (e == 0) return fail(KS_ERR_UNSUPPORTED_DTYPE, "dtype code %d is not a ks_dtype_t", (int)dtype);
    if (hidden <= 0)
        return fail(KS_ERR_INVALID_ARGUMENT, "hidden must be > 0 (got %lld)", (long long)hidden);
    if (rows < 0) return fail(KS_ERR_INVALID_ARGUMENT, "rows must be >= 0 (got %lld)", (long long)rows);
    if (!std::isfinite(eps) || !(eps > 0.0f))
        return fail(KS_ERR_INVALID_ARGUMENT, "eps must be finite and > 0 (got %g)", (double)eps);
    if (hidden > INT64_MAX / e || (rows > 0 && rows > INT64_MAX / (hidden * e)))
        return fail(KS_ERR_INVALID_ARGUMENT, "rows*hidden*element size overflows int64");
    if (rows == 0) return KS_SUCCESS;  // empty input: legal, nothing to launch
    if (!out || !x || !w || (fused && !res))
        return fail(KS_ERR_INVALID_ARGUMENT, "NULL pointer with rows > 0");
    const int64_t nbytes = rows * hidden * e, wbytes = hidden * e;
    if (fused) {
        if (overlaps(x, nbytes, res, nbytes))
            return fail(KS_ERR_OVERLAP, "x and residual storage overlap");
        if (overlaps(x, nbytes, w, wbytes)) return fail(KS_ERR_OVERLAP, "x and weight storage overlap");
        if (overlaps(res, nbytes, w, wbytes))
            return fail(KS_ERR_OVERLAP, "residual and weight storage overlap");
    } else {
        if (out != x && overlaps(out, nbytes, x, nbytes))
            return fail(KS_ERR_OVERLAP, "out partially overlaps x (only out == x is allowed)");
        if (overlaps(out, nbytes, w, wbytes)) return fail(KS_ERR_OVERLAP, "out and weight storage overlap");
    }

    // ---- device facts (cached per device)
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
    if (dev < 0 || dev >= kMaxDevices) return fail(KS_ERR_CUDA, "device ordinal %d out of range", dev);
    DeviceSlot &slot = g_devices[dev];
    std::call_once(slot.once, [&] {
        slot.err = cudaDeviceGetAttribute(&slot.sm_count, cudaDevAttrMultiProcessorCount, dev);
    });
    if (slot.err != cudaSuccess)
        return fail(KS_ERR_CUDA, "querying the SM count: %s", cudaGetErrorString(slot.err));

    const uintptr_t align = (uintptr_t)out | (uintptr_t)x | (uintptr_t)w | (fused ? (uintptr_t)res : 0);
    const bool aligned16 = (align & 15u) == 0;
    ks_plan_t p;
    ks_status_t st = plan(fused ? 1 : 0, rows, hidden, e, aligned16, slot.sm_count, 0, &p);
    if (st != KS_SUCCESS) return st;

    int bps;
    {
        const uint64_t key = occ_key(dev, dtype, fused, p);
        std::lock_guard<std::mutex> lock(g_occ_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) {
            bps = it->second;
        } else {
            bps = query_blocks_per_sm(dtype, p, fused);
            if (bps > 0) g_occ.emplace(key, bps);
        }
    }
    if (bps <= 0) return fail(KS_ERR_CUDA, "kernel %d (block %d) cannot be resident", p.kernel, p.block);
    st = plan(fused ? 1 : 0, rows, hidden, e, aligned16, slot.sm_count, bps, &p);
    if (st != KS_SUCCESS) return st;

    RowArgs a;
    a.out = fused ? const_cast<void *>(x) : out;
    a.x = x;
    a.res = res;
    a.w = w;
    a.rows = rows;
    a.hidden = hidden;
    a.hv = (p.kernel == KS_KERNEL_SCALAR) ? 0 : hidden / (16 / e);
    a.eps = eps;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case KS_DTYPE_BF16: ce = launch_bf16(p, fused, a, s); break;
    case KS_DTYPE_F16: ce = launch_f16(p, fused, a, s); break;
    default: ce = launch_f32(p, fused, a, s); break;
    }
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "launch: %s", cudaGetErrorString(ce));
    return KS_SUCCESS;
}

}  // namespace

// Host heuristic (after the pages' rule of sizing the launch from the row width: Triton
// Kernels, "Kernels" table, rmsnorm row; Kernscope, "Triton CUDA backend"):
//  * rows of at most 128 16-byte vectors (bf16/fp16 H <= 1024, fp32 H <= 512): one warp per row,
//    1/2/4 vectors per lane, up to 8 rows per CTA but never fewer CTAs than SMs when the rows
//    allow it;
//  * rows of up to 2048 vectors (bf16/fp16 H <= 16384, fp32 H <= 8192): one CTA per row, 4
//    vectors per thread, the CTA as wide as the row needs (a multiple of 32 threads);
//  * anything else (H not a multiple of the vector, unaligned pointers, wider rows): the scalar
//    two-pass kernel.
// The grid is persistent: at most sm_count * blocks_per_sm CTAs.
ks_status_t plan(int op, int64_t rows, int64_t hidden, int elem, bool aligned16, int sm_count,
                 int blocks_per_sm, ks_plan_t *p) {
    if (!p) return fail(KS_ERR_INVALID_ARGUMENT, "plan pointer is NULL");
    memset(p, 0, sizeof *p);
    if (op != 0 && op != 1) return fail(KS_ERR_INVALID_ARGUMENT, "op must be 0 or 1");
    if (hidden <= 0 || rows < 0 || sm_count <= 0 || blocks_per_sm < 0 ||
        (elem != 2 && elem != 4))
        return fail(KS_ERR_INVALID_ARGUMENT, "bad plan arguments");
    if (rows == 0) {
        p->kernel = KS_KERNEL_NONE;
        return KS_SUCCESS;
    }
    const int per_vec = 16 / elem;
    const bool vec_ok = aligned16 && hidden % per_vec == 0;
    const int64_t hv = vec_ok ? hidden / per_vec : 0;
    int64_t rows_per_cta = 1;
    if (vec_ok && hv <= 128) {
        p->kernel = KS_KERNEL_WARP_ROW;
        p->vec_per_thread = hv <= 32 ? 1 : (hv <= 64 ? 2 : 4);
        p->team = 32;
        int64_t teams = ceil_div(rows, sm_count);
        teams = teams < 1 ? 1 : (teams > 8 ? 8 : teams);
        rows_per_cta = teams;
        p->block = (int32_t)(32 * teams);
    } else if (vec_ok && hv <= 2048) {
        p->kernel = KS_KERNEL_CTA_ROW;
        p->vec_per_thread = 4;
        p->block = (int32_t)round_up(ceil_div(hv, 4), 32);
        p->team = p->block;
    } else {
        p->kernel = KS_KERNEL_SCALAR;
        int64_t b = round_up(ceil_div(hidden, 8), 32);
        p->block = (int32_t)(b < 32 ? 32 : (b > 1024 ? 1024 : b));
        p->team = p->block;
    }
    const int64_t ctas = ceil_div(rows, rows_per_cta);
    const int64_t cap = (int64_t)sm_count * blocks_per_sm;
    p->grid = (blocks_per_sm > 0 && ctas > cap) ? cap : ctas;
    p->rows_per_pass = p->grid * rows_per_cta;
    return KS_SUCCESS;
}

}  // namespace ks

extern "C" {

ks_status_t ks_rms_norm(void *out, const void *x, const void *weight, int64_t rows,
                        int64_t hidden, float eps, ks_dtype_t dtype, ks_stream_t stream) {
    return ks::run(false, out, x, nullptr, weight, rows, hidden, eps, dtype, stream);
}

ks_status_t ks_fused_add_rms_norm(void *x, void *residual, const void *weight, int64_t rows,
                                  int64_t hidden, float eps, ks_dtype_t dtype,
                                  ks_stream_t stream) {
    return ks::run(true, x, x, residual, weight, rows, hidden, eps, dtype, stream);
}

const char *ks_status_string(ks_status_t status) {
    switch (status) {
    case KS_SUCCESS: return "KS_SUCCESS";
    case KS_ERR_INVALID_ARGUMENT: return "KS_ERR_INVALID_ARGUMENT";
    case KS_ERR_UNSUPPORTED_DTYPE: return "KS_ERR_UNSUPPORTED_DTYPE";
    case KS_ERR_OVERLAP: return "KS_ERR_OVERLAP";
    case KS_ERR_CUDA: return "KS_ERR_CUDA";
    default: return "KS_UNKNOWN_STATUS";
    }
}

const char *ks_last_error(void) { return ks::g_detail; }

ks_status_t ks_plan_launch(int32_t op, int64_t rows, int64_t hidden, ks_dtype_t dtype,
                           int32_t aligned16, int32_t sm_count, int32_t blocks_per_sm,
                           ks_plan_t *plan) {
    const int e = ks::elem_bytes(dtype);
    if (e == 0) return ks::fail(KS_ERR_UNSUPPORTED_DTYPE, "dtype code %d is not a ks_dtype_t", (int)dtype);
    return ks::plan(op, rows, hidden, e, aligned16 != 0, sm_count, blocks_per_sm, plan);
}

int32_t ks_version(void) { return 100; }

}  // extern "C"
