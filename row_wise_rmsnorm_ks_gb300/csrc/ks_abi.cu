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
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "ks_internal.h"

namespace ks {
namespace {
thread_local char g_detail[256] = "";
std::atomic<int32_t> g_launch_options{0};
}  // namespace

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
bool misaligned(int e, const void *a, const void *b, const void *c, const void *d) {
    const uintptr_t m = (uintptr_t)e - 1;
    return (((uintptr_t)a | (uintptr_t)b | (uintptr_t)c | (uintptr_t)d) & m) != 0;
}

bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool launch_pdl_enabled() {
    return (g_launch_options.load(std::memory_order_relaxed) & KS_LAUNCH_PDL) != 0;
}
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ---------------------------------------------------------------- per-device caches

constexpr int kMaxDevices = 64;

struct DeviceSlot {
    std::once_flag once;
    int sm_count = 0;
    int l2_bytes = 0;
    cudaError_t err = cudaSuccess;
};
DeviceSlot g_devices[kMaxDevices];

std::mutex g_occ_mu;
std::unordered_map<uint64_t, int> g_occ;  // occupancy facts per (device, kernel, plan shape)

// Key of an occupancy fact: the device, what is asked (CTAs per SM or resident clusters), and
// every plan field that selects the kernel or changes its residency.
// Every field that selects the kernel or its resources: shared memory below 256 KiB (18 bits),
// block up to 1024 (11), stages (5), flags (4), cluster up to 16 (5), vectors per thread up to 8
// (4), kernel (3), op, dtype, the query kind, the warp-row team (8, 16 or a full warp) and the
// device.
uint64_t occ_key(int dev, ks_dtype_t d, bool fused, const ks_plan_t &p, bool clusters) {
    const uint64_t team = p.kernel == KS_KERNEL_WARP_ROW ? (p.team == 8 ? 1u : (p.team == 16 ? 2u : 0u)) : 0u;
    return ((uint64_t)(dev & 0x3F) << 56) | (team << 54) | ((uint64_t)clusters << 53) |
           ((uint64_t)(d & 0x3) << 51) | ((uint64_t)fused << 50) |
           ((uint64_t)(p.kernel & 0x7) << 47) | ((uint64_t)(p.vec_per_thread & 0xF) << 43) |
           ((uint64_t)(p.cluster & 0x1F) << 38) | ((uint64_t)(p.flags & 0xF) << 34) |
           ((uint64_t)(p.stages & 0x1F) << 29) | ((uint64_t)(p.block & 0x7FF) << 18) |
           (uint64_t)(p.smem_bytes & 0x3FFFF);
}

constexpr int kSmemLimit = 226 * 1024;  // dynamic ring; static smem and reserve fit in 227 KB
// Bytes of rows the two-pass kernels may have in flight together: the second pass re-reads each
// row from L2, so the grid keeps the first pass's rows inside three quarters of the device's L2
// (96 MiB when no device size is given, as in the pure-host ks_plan_launch). The
// one-CTA-per-row kernel never drops below one CTA per SM (for rows of 16384 vectors and more,
// measured: a full grid with some L2 misses beats fewer CTAs, 0.66-0.81 of the copy peak
// against 0.39-0.68 for fused rows).
constexpr int64_t kDefaultL2Bytes = 128ll << 20;  // when no device size is given
int64_t twopass_l2_budget(int64_t l2_bytes) { return (l2_bytes > 0 ? l2_bytes : kDefaultL2Bytes) / 4 * 3; }

int64_t twopass_grid_cap(int64_t hv, bool fused, int sm_count, int64_t l2_bytes) {
    const int64_t per_cta = hv * 16 * (fused ? 2 : 1);
    const int64_t cap = twopass_l2_budget(l2_bytes) / (per_cta > 0 ? per_cta : 1);
    return cap < sm_count ? sm_count : cap;
}

// Clusters of the split two-pass kernel: no more than keep their rows in flight (one per
// cluster, two for the pipelined kernel) within the L2 budget; then as few as give every cluster the same number of rows (a
// last wave that only some clusters run leaves the others' SMs idle), e.g. 768 rows on 152
// resident clusters run as 6 rows on each of 128 clusters instead of 5 or 6 on 152.
int64_t split_clusters(int64_t rows, int64_t resident, int64_t hv, bool fused, int rows_in_flight,
                       int64_t l2_bytes) {
    const int64_t row_bytes = hv * 16 * (fused ? 2 : 1) * (rows_in_flight > 1 ? rows_in_flight : 1);
    int64_t n = twopass_l2_budget(l2_bytes) / (row_bytes > 0 ? row_bytes : 1);
    n = n < resident ? n : resident;
    n = n < rows ? n : rows;
    n = n < 1 ? 1 : n;
    const int64_t waves = ceil_div(rows, n);
    return ceil_div(rows, waves);
}
constexpr int kRingHeader = 128;  // the staged kernel's mbarriers, ahead of its ring

// Checks that a plan fits the call (see ks_rms_norm_planned) and fills the derived fields.
ks_status_t check_plan(ks_plan_t &p, bool fused, int64_t rows, int64_t hidden, int e,
                       bool aligned16) {
    const int per_vec = 16 / e;
    const bool vec_ok = aligned16 && hidden % per_vec == 0;
    const int64_t hv = vec_ok ? hidden / per_vec : 0;
    if (p.block < 32 || p.block % 32 != 0)
        return fail(KS_ERR_INVALID_ARGUMENT, "plan block %d is not a positive multiple of 32", p.block);
    const bool split_req = p.kernel == KS_KERNEL_TWOPASS_ROW && p.cluster >= 2;
    if (split_req && (p.stages < 0 || p.stages > 2))
        return fail(KS_ERR_INVALID_ARGUMENT, "split two-pass plan: stages 0, 1 (one row in flight) or 2 "
                    "(two rows), got %d", p.stages);
    p.stages = (p.kernel == KS_KERNEL_BULK_ROW || split_req) ? p.stages : 0;
    p.smem_bytes = 0;
    const bool split_bulk = p.kernel == KS_KERNEL_BULK_ROW && p.cluster >= 2;
    const bool split_twopass = p.kernel == KS_KERNEL_TWOPASS_ROW && p.cluster >= 2;
    p.cluster = (p.kernel == KS_KERNEL_CLUSTER_ROW || split_bulk || split_twopass) ? p.cluster : 0;
    if (p.flags & ~(KS_PLAN_NO_PREFETCH | KS_PLAN_PDL | KS_PLAN_SMEM_ROWS))
        return fail(KS_ERR_INVALID_ARGUMENT, "unknown plan flags 0x%x", (unsigned)p.flags);
    if ((p.flags & KS_PLAN_SMEM_ROWS) && !(split_bulk && !fused && p.stages >= 2))
        return fail(KS_ERR_INVALID_ARGUMENT, "KS_PLAN_SMEM_ROWS: the plain op's staged kernel split "
                    "over a cluster, 2 or more stages");
    int64_t rows_per_cta = 1;
    switch (p.kernel) {
    case KS_KERNEL_WARP_ROW:
        if (!vec_ok) return fail(KS_ERR_INVALID_ARGUMENT, "vector kernel needs 16-byte rows and pointers");
        if (p.vec_per_thread != 1 && p.vec_per_thread != 2 && p.vec_per_thread != 4 &&
            p.vec_per_thread != 6 && p.vec_per_thread != 8)
            return fail(KS_ERR_INVALID_ARGUMENT, "warp-row kernel takes 1, 2, 4, 6 or 8 vectors");
        if (p.team == 0) p.team = 32;  // a plan made without a team: a warp per row
        if (p.team != 8 && p.team != 16 && p.team != 32)
            return fail(KS_ERR_INVALID_ARGUMENT, "warp-row team must be 8, 16 or 32 lanes (got %d)", p.team);
        if (p.team < 32 && p.vec_per_thread > 4)
            return fail(KS_ERR_INVALID_ARGUMENT, "8- and 16-lane teams take 1, 2 or 4 vectors per lane");
        if ((int64_t)p.team * p.vec_per_thread < hv || p.block > 256)
            return fail(KS_ERR_INVALID_ARGUMENT, "warp-row plan does not cover the row or block > 256");
        rows_per_cta = p.block / p.team;
        break;
    case KS_KERNEL_CTA_ROW:
    case KS_KERNEL_BULK_ROW: {
        if (!vec_ok) return fail(KS_ERR_INVALID_ARGUMENT, "vector kernel needs 16-byte rows and pointers");
        const bool bulk = p.kernel == KS_KERNEL_BULK_ROW;
        // the staged ring: 4 vectors per thread; split over a cluster, also 8 for the plain op
        const bool bulk_v = p.vec_per_thread == 4 || (split_bulk && !fused && p.vec_per_thread == 8);
        if (bulk ? !bulk_v : (p.vec_per_thread != 2 && p.vec_per_thread != 4))
            return fail(KS_ERR_INVALID_ARGUMENT, "unsupported vectors per thread %d", p.vec_per_thread);
        if (split_bulk && p.cluster > ((p.flags & KS_PLAN_SMEM_ROWS) ? 16 : 8))
            return fail(KS_ERR_INVALID_ARGUMENT, "cluster of %d CTAs (2..8 supported; 2..16 with "
                        "KS_PLAN_SMEM_ROWS)", p.cluster);
        const int C = split_bulk ? p.cluster : 1;
        const int64_t slice = ceil_div(hv, C);
        if ((C - 1) * slice >= hv)
            return fail(KS_ERR_INVALID_ARGUMENT, "a cluster of %d leaves a CTA without vectors", C);
        // the shared-memory rows kernel holds only the weight in registers: 1024 threads at 4
        const bool smem_rows = (p.flags & KS_PLAN_SMEM_ROWS) && p.vec_per_thread == 4;
        const int bound = bulk ? (smem_rows ? 1024 : 512) : (p.vec_per_thread == 2 ? 1024 : 512);
        if ((int64_t)p.block * p.vec_per_thread < slice || p.block > bound)
            return fail(KS_ERR_INVALID_ARGUMENT, "CTA-row plan does not cover the row or block > %d", bound);
        p.team = p.block * C;
        if (bulk) {
            const int64_t stage = slice * 16 * (fused ? 2 : 1);
            if (p.stages < 1 || p.stages > 16 || kRingHeader + stage * p.stages > kSmemLimit)
                return fail(KS_ERR_INVALID_ARGUMENT, "staged ring of %d stages does not fit", p.stages);
            p.smem_bytes = (int32_t)(kRingHeader + stage * p.stages);
        }
        break;
    }
    case KS_KERNEL_CLUSTER_ROW: {
        if (!vec_ok) return fail(KS_ERR_INVALID_ARGUMENT, "vector kernel needs 16-byte rows and pointers");
        if (p.vec_per_thread != 1 && p.vec_per_thread != 2 && p.vec_per_thread != 4)
            return fail(KS_ERR_INVALID_ARGUMENT, "cluster-row kernel takes 1, 2 or 4 vectors");
        if (p.cluster < 2 || p.cluster > 8)
            return fail(KS_ERR_INVALID_ARGUMENT, "cluster of %d CTAs (2..8 supported)", p.cluster);
        const int64_t slice = ceil_div(hv, p.cluster);
        if ((int64_t)p.block * p.vec_per_thread < slice || p.block > 512)
            return fail(KS_ERR_INVALID_ARGUMENT, "cluster-row plan does not cover its slice or block > 512");
        p.team = p.block * p.cluster;
        break;
    }
    case KS_KERNEL_TWOPASS_ROW:
        if (!vec_ok) return fail(KS_ERR_INVALID_ARGUMENT, "vector kernel needs 16-byte rows and pointers");
        if (p.vec_per_thread != 2 && p.vec_per_thread != 4)
            return fail(KS_ERR_INVALID_ARGUMENT, "two-pass kernel takes 2 or 4 vectors per step");
        if (p.block > 1024) return fail(KS_ERR_INVALID_ARGUMENT, "two-pass block > 1024");
        if (split_twopass) {
            if (p.cluster > 8)
                return fail(KS_ERR_INVALID_ARGUMENT, "cluster of %d CTAs (2..8 supported)", p.cluster);
            const int64_t slice = ceil_div(hv, p.cluster);
            if ((p.cluster - 1) * slice >= hv)
                return fail(KS_ERR_INVALID_ARGUMENT, "a cluster of %d leaves a CTA without vectors",
                            p.cluster);
        }
        p.team = p.block * (split_twopass ? p.cluster : 1);
        break;
    case KS_KERNEL_SCALAR:
        if (p.block > 1024) return fail(KS_ERR_INVALID_ARGUMENT, "scalar block > 1024");
        p.vec_per_thread = 0;
        p.team = p.block;
        break;
    default:
        return fail(KS_ERR_INVALID_ARGUMENT, "unknown kernel %d", p.kernel);
    }
    p.rows_per_pass = rows_per_cta;  // per CTA here; scaled by the grid once it is known
    (void)rows;
    return KS_SUCCESS;
}

int query_blocks_per_sm(ks_dtype_t d, const ks_plan_t &p, bool fused) {
    switch (d) {
    case KS_DTYPE_BF16: return blocks_per_sm_bf16(p, fused);
    case KS_DTYPE_F16: return blocks_per_sm_f16(p, fused);
    default: return blocks_per_sm_f32(p, fused);
    }
}

int query_max_clusters(ks_dtype_t d, const ks_plan_t &p, bool fused) {
    switch (d) {
    case KS_DTYPE_BF16: return max_clusters_bf16(p, fused);
    case KS_DTYPE_F16: return max_clusters_f16(p, fused);
    default: return max_clusters_f32(p, fused);
    }
}

// Cached occupancy facts of a plan's kernel on a device: CTAs per SM, and for cluster plans the
// clusters that can be resident at once (0 = the query failed).
int cached_query(int dev, ks_dtype_t dtype, bool fused, const ks_plan_t &p, bool clusters) {
    const uint64_t key = occ_key(dev, dtype, fused, p, clusters);
    std::lock_guard<std::mutex> lock(g_occ_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
    const int v = clusters ? query_max_clusters(dtype, p, fused) : query_blocks_per_sm(dtype, p, fused);
    if (v > 0) g_occ.emplace(key, v);
    return v;
}

ks_status_t run(bool fused, void *out, const void *x, void *res, const void *w, int64_t rows,
                int64_t hidden, float eps, ks_dtype_t dtype, ks_stream_t stream,
                const ks_plan_t *forced) {
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
    if (misaligned(e, out, x, w, fused ? res : nullptr))
        return fail(KS_ERR_INVALID_ARGUMENT, "a pointer is not aligned to the %d-byte element", e);
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

    const uintptr_t align = (uintptr_t)out | (uintptr_t)x | (uintptr_t)w | (fused ? (uintptr_t)res : 0);
    const bool aligned16 = (align & 15u) == 0;
    ks_plan_t p;
    ks_status_t st;
    if (forced) {  // an explicit plan is an argument too: checked before any CUDA call
        p = *forced;
        st = check_plan(p, fused, rows, hidden, e, aligned16);
        if (st != KS_SUCCESS) return st;
    }

    // ---- device facts (cached per device)
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
    if (dev < 0 || dev >= kMaxDevices) return fail(KS_ERR_CUDA, "device ordinal %d out of range", dev);
    DeviceSlot &slot = g_devices[dev];
    std::call_once(slot.once, [&] {
        slot.err = cudaDeviceGetAttribute(&slot.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (slot.err == cudaSuccess)
            slot.err = cudaDeviceGetAttribute(&slot.l2_bytes, cudaDevAttrL2CacheSize, dev);
    });
    if (slot.err != cudaSuccess)
        return fail(KS_ERR_CUDA, "querying the SM count and L2 size: %s", cudaGetErrorString(slot.err));
    if (!forced) {
        st = plan(fused ? 1 : 0, rows, hidden, dtype, aligned16, slot.sm_count, 0, slot.l2_bytes, &p);
        if (st != KS_SUCCESS) return st;
    }
    const int32_t pdl = forced ? (p.flags & KS_PLAN_PDL)
                               : ((g_launch_options.load(std::memory_order_relaxed) & KS_LAUNCH_PDL)
                                      ? KS_PLAN_PDL : 0);

    const int bps = cached_query(dev, dtype, fused, p, false);
    if (bps <= 0) return fail(KS_ERR_CUDA, "kernel %d (block %d) cannot be resident", p.kernel, p.block);
    if (forced && p.cluster >= 2) {
        // whole clusters: one row per cluster per pass
        const int64_t cap = (int64_t)slot.sm_count * bps / p.cluster;
        int64_t clusters = forced->grid > 0 ? forced->grid / p.cluster : cap;
        clusters = clusters < 1 ? 1 : clusters;
        clusters = clusters < rows ? clusters : rows;
        p.grid = clusters * p.cluster;
        p.rows_per_pass = clusters;
    } else if (forced) {
        const int64_t per_cta = p.rows_per_pass;
        const int64_t ctas = ceil_div(rows, per_cta);
        const int64_t cap = (int64_t)slot.sm_count * bps;
        p.grid = forced->grid > 0 ? (forced->grid < ctas ? forced->grid : ctas) : (ctas < cap ? ctas : cap);
        if (forced->grid <= 0 && p.kernel == KS_KERNEL_TWOPASS_ROW) {
            const int64_t l2cap = twopass_grid_cap(hidden / (16 / e), fused, slot.sm_count,
                                                   slot.l2_bytes);
            if (p.grid > l2cap) p.grid = l2cap;
        }
        p.rows_per_pass = p.grid * per_cta;
    } else {
        st = plan(fused ? 1 : 0, rows, hidden, dtype, aligned16, slot.sm_count, bps, slot.l2_bytes, &p);
        if (st != KS_SUCCESS) return st;
    }
    if (p.cluster >= 2) {
        // A persistent grid of clusters must be resident at once (a cluster left for a second
        // wave would start only after a resident one has finished all its rows): cap it by the
        // device's own count, which the placement of clusters on GPCs can make smaller than
        // SMs * CTAs per SM / cluster.
        const int resident = cached_query(dev, dtype, fused, p, true);
        if (resident <= 0)
            return fail(KS_ERR_CUDA, "no cluster of %d x %d threads can be resident", p.cluster, p.block);
        if (p.grid / p.cluster > resident) {
            p.grid = (int64_t)resident * p.cluster;
            p.rows_per_pass = resident;
        }
        if (p.kernel == KS_KERNEL_TWOPASS_ROW && !(forced && forced->grid > 0)) {
            const int64_t n = split_clusters(rows, p.grid / p.cluster, hidden / (16 / e), fused,
                                             p.stages == 2 ? 2 : 1, slot.l2_bytes);
            p.grid = n * p.cluster;
            p.rows_per_pass = n;
        }
    }

    p.flags = (p.flags & ~KS_PLAN_PDL) | pdl;
    RowArgs a;
    a.out = fused ? const_cast<void *>(x) : out;
    a.x = x;
    a.res = res;
    a.w = w;
    a.rows = rows;
    a.hidden = hidden;
    a.hv = (p.kernel == KS_KERNEL_SCALAR) ? 0 : hidden / (16 / e);
    a.eps = eps;
    a.stages = p.stages;
    a.l2_prefetch = (p.kernel == KS_KERNEL_TWOPASS_ROW && !(p.flags & KS_PLAN_NO_PREFETCH)) ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (dtype) {
    case KS_DTYPE_BF16: ce = launch_bf16(p, fused, a, s); break;
    case KS_DTYPE_F16: ce = launch_f16(p, fused, a, s); break;
    default: ce = launch_f32(p, fused, a, s); break;
    }
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "launch: %s", cudaGetErrorString(ce));
    return KS_SUCCESS;
}


// Host heuristic (after the pages' rule of sizing the launch from the row width: Triton
// Kernels, "Kernels" table, rmsnorm row; Kernscope, "Triton CUDA backend"):
//  * many rows (more than SMs) of 1..2048 vectors (bf16/fp16 H <= 16384, fp32 H <= 8192): the
//    band table below, one per dtype and op, generated from a plan-contexts sweep (8- and 16-lane
//    teams and warps per row, CTA rows at 2 or 4 vectors per thread, each with and without
//    prefetch, the staged ring and the two-pass kernel, each timed in two contexts); the ring and
//    the two-pass kernel only with at least 4 rows per SM, the band's one-pass fallback otherwise;
//  * at most SMs rows of at most 128 vectors: one warp per row, 1/2/4 vectors per lane (the
//    fewest that cover the row), next row prefetched, one row per CTA;
//  * latency regime (rows <= SMs, so each CTA gets at most one row) of 129..2048 vectors:
//    prefetch has nothing to fetch: the widest fused rows (>= 1792 vectors, at most SMs/8 rows)
//    go to a cluster of 8 CTAs per row, plain rows of at most 1024 vectors take 2 vectors per
//    thread, and the rest 4 (a graph-replay sweep of 1..333 rows found no gain in warp rows
//    there);
//  * rows wider than 2048 vectors (bf16/fp16 H > 16384, fp32 H > 8192): the two-pass kernel,
//    one CTA per row reading it twice (the second time from L2), any width; few rows (at most
//    SMs/8) of up to 16384 vectors split over a cluster of 8 CTAs instead, and rows that outgrow
//    L2 together over a cluster of 2..8 CTAs (split_row);
//  * anything else (H not a multiple of the vector, unaligned pointers): the scalar two-pass
//    kernel.
// The grid is persistent: at most sm_count * blocks_per_sm CTAs (for cluster plans, whole
// clusters, which the launch caps again by the device's count of resident clusters; for the
// two-pass kernel, no more CTAs than keep their rows in flight within 3/4 of the device's L2,
// but at least one per SM).
namespace {

// Many rows of 1..2048 vectors: one band table per dtype and op. A band covers the widths up to
// its `hi` (from the previous band's hi + 1) and names a launch:
//   E / e  an 8-lane team per row with / without prefetch (4 rows per warp), at the fewest of 1,
//          2 or 4 vectors per lane that cover the row (rows of at most 32 vectors);
//   H / h  the same with 16-lane teams (2 rows per warp; rows of at most 64 vectors);
//   W / w  a warp per row at the fewest of 1, 2, 4, 6 or 8 vectors per lane that cover the row:
//          up to 8 warps per 256-thread CTA at 1, 2 or 4 vectors (rows of at most 128 vectors),
//          4 rows per 128-thread CTA at 6 or 8;
//   T / t  a CTA per row at 2 vectors per thread, with / without prefetch;
//   F / f  the same at 4 vectors per thread;
//   R      the staged ring, 2 stages;
//   P      the two-pass kernel in its default shape;
// and a fallback for fewer than 4 rows per SM, where the ring and the two-pass kernel have too
// few rows to keep busy (the fallback is the code itself for the one-pass launches).
// The tables are generated, not edited: a plan-contexts sweep on GB300 times every launch at each
// measured width in two contexts (steady state, and right after a kernel with a large
// shared-memory carveout), a plan's score is the worse of the two, and the tables are the fewest
// bands such that at every measured width the band's launch scores within a point of the copy
// peak of the best launch there (bench.py --plan-bands-record / --plan-bands-derive; the
// measured record is committed in bands/ beside this file, and a CPU test re-derives the tables
// from it and checks every default plan against it).
struct RowBand {
    int32_t hi;     // the band's widest row, in 16-byte vectors
    char code;      // the launch
    char fallback;  // the launch with fewer than 4 rows per SM
};
constexpr int64_t kBandLo = 1, kBandHi = 2048;
// BEGIN GENERATED ROW BANDS
constexpr RowBand kRowBandsF32Plain[] = {{4, 'e', 'e'}, {8, 'E', 'E'}, {14, 'e', 'e'}, {16, 'E', 'E'}, {24, 'e', 'e'}, {32, 'E', 'E'}, {52, 'h', 'h'}, {64, 'H', 'H'}, {108, 'w', 'w'}, {124, 'W', 'W'}, {128, 'F', 'F'}, {152, 'w', 'w'}, {200, 'f', 'f'}, {248, 'W', 'W'}, {256, 'T', 'T'}, {480, 'f', 'f'}, {512, 'T', 'T'}, {608, 'f', 'f'}, {640, 'T', 'T'}, {992, 'f', 'f'}, {1344, 'P', 'f'}, {1536, 'f', 'f'}, {1888, 'P', 'f'}, {2048, 'f', 'f'}};
constexpr RowBand kRowBandsF32Fused[] = {{7, 'e', 'e'}, {8, 'E', 'E'}, {14, 'e', 'e'}, {16, 'E', 'E'}, {24, 'e', 'e'}, {32, 'E', 'E'}, {44, 'h', 'h'}, {64, 'H', 'H'}, {76, 'w', 'w'}, {92, 't', 't'}, {116, 'W', 'W'}, {128, 'F', 'F'}, {152, 't', 't'}, {192, 'T', 'T'}, {208, 't', 't'}, {248, 'T', 'T'}, {256, 'W', 'W'}, {296, 't', 't'}, {320, 'T', 'T'}, {360, 't', 't'}, {384, 'T', 'T'}, {416, 't', 't'}, {512, 'F', 'F'}, {768, 't', 't'}, {960, 'P', 't'}, {1152, 't', 't'}, {1600, 'f', 'f'}, {2048, 'P', 'f'}};
constexpr RowBand kRowBandsF16Plain[] = {{14, 'e', 'e'}, {16, 'E', 'E'}, {28, 'e', 'e'}, {32, 'E', 'E'}, {60, 'h', 'h'}, {64, 'H', 'H'}, {112, 'w', 'w'}, {124, 'f', 'f'}, {128, 'W', 'W'}, {188, 'w', 'w'}, {192, 'f', 'f'}, {200, 'w', 'w'}, {248, 'f', 'f'}, {256, 'W', 'W'}, {1536, 'f', 'f'}, {2048, 'P', 'f'}};
constexpr RowBand kRowBandsF16Fused[] = {{14, 'e', 'e'}, {16, 'E', 'E'}, {20, 'e', 'e'}, {24, 'h', 'h'}, {32, 'E', 'E'}, {44, 'h', 'h'}, {52, 'w', 'w'}, {64, 'H', 'H'}, {84, 'w', 'w'}, {92, 'f', 'f'}, {112, 't', 't'}, {128, 'W', 'W'}, {136, 'w', 'w'}, {176, 't', 't'}, {196, 'f', 'f'}, {248, 't', 't'}, {256, 'T', 'T'}, {576, 't', 't'}, {672, 'f', 'f'}, {768, 't', 't'}, {992, 'f', 'f'}, {1152, 't', 't'}, {1536, 'f', 'f'}, {1824, 'R', 't'}, {2048, 'P', 't'}};
constexpr RowBand kRowBandsBf16Plain[] = {{14, 'e', 'e'}, {16, 'E', 'E'}, {28, 'e', 'e'}, {32, 'H', 'H'}, {60, 'h', 'h'}, {64, 'W', 'W'}, {108, 'w', 'w'}, {124, 'W', 'W'}, {128, 'T', 'T'}, {144, 'w', 'w'}, {192, 'W', 'W'}, {208, 'w', 'w'}, {240, 'f', 'f'}, {256, 'W', 'W'}, {480, 'f', 'f'}, {512, 'F', 'F'}, {576, 'f', 'f'}, {640, 'F', 'F'}, {736, 'f', 'f'}, {768, 'F', 'F'}, {1152, 'f', 'f'}, {1280, 'F', 'F'}, {1536, 'f', 'f'}, {2048, 'P', 'f'}};
constexpr RowBand kRowBandsBf16Fused[] = {{12, 'e', 'e'}, {16, 'E', 'E'}, {20, 'e', 'e'}, {24, 'E', 'E'}, {32, 'H', 'H'}, {40, 'h', 'h'}, {64, 'H', 'H'}, {84, 'w', 'w'}, {128, 'W', 'W'}, {136, 'w', 'w'}, {168, 't', 't'}, {200, 'F', 'F'}, {312, 't', 't'}, {320, 'F', 'F'}, {576, 't', 't'}, {672, 'f', 'f'}, {864, 'F', 'F'}, {992, 'f', 'f'}, {1152, 't', 't'}, {1472, 'f', 'f'}, {2048, 'F', 'F'}};
// END GENERATED ROW BANDS

// The widest row (in vectors) a one-pass code's launch covers (0: not a one-pass code).
constexpr int64_t code_reach(char c) {
    return (c == 'E' || c == 'e') ? 32
         : (c == 'H' || c == 'h') ? 64
         : (c == 'W' || c == 'w') ? 256
         : (c == 'T' || c == 't' || c == 'F' || c == 'f') ? kBandHi : 0;
}

// Whether a table is well formed: widths rising to kBandHi, team and warp launches only where
// they cover the row, fallbacks one-pass launches, every code known.
template <size_t N>
constexpr bool bands_ok(const RowBand (&b)[N]) {
    for (size_t i = 0; i < N; ++i) {
        if (b[i].hi < kBandLo || b[i].hi > kBandHi || (i > 0 && b[i].hi <= b[i - 1].hi)) return false;
        const char c = b[i].code, f = b[i].fallback;
        const bool one_pass = code_reach(c) > 0;
        if (!(one_pass || c == 'R' || c == 'P') || code_reach(f) == 0) return false;
        if (one_pass && f != c) return false;
        if ((one_pass && b[i].hi > code_reach(c)) || b[i].hi > code_reach(f)) return false;
    }
    return b[N - 1].hi == kBandHi;
}
static_assert(bands_ok(kRowBandsF32Plain) && bands_ok(kRowBandsF32Fused) &&
                  bands_ok(kRowBandsF16Plain) && bands_ok(kRowBandsF16Fused) &&
                  bands_ok(kRowBandsBf16Plain) && bands_ok(kRowBandsBf16Fused),
              "a row band table is malformed");
// Indexed [dtype code][op].
const RowBand *const kRowBands[3][2] = {
    {kRowBandsF32Plain, kRowBandsF32Fused},
    {kRowBandsF16Plain, kRowBandsF16Fused},
    {kRowBandsBf16Plain, kRowBandsBf16Fused},
};

void cta_row(ks_plan_t *p, int64_t hv, int v, bool prefetch) {
    p->kernel = KS_KERNEL_CTA_ROW;
    p->vec_per_thread = v;
    p->block = (int32_t)round_up(ceil_div(hv, v), 32);
    p->team = p->block;
    p->flags = prefetch ? 0 : KS_PLAN_NO_PREFETCH;
}

void bulk_row(ks_plan_t *p, int64_t hv, bool fused, int64_t stages) {
    const int64_t stage = hv * 16 * (fused ? 2 : 1);
    p->kernel = KS_KERNEL_BULK_ROW;
    p->vec_per_thread = 4;
    p->block = (int32_t)round_up(ceil_div(hv, 4), 32);
    p->team = p->block;
    p->flags = 0;
    p->stages = (int32_t)stages;
    p->smem_bytes = (int32_t)(kRingHeader + stages * stage);
}

// The two-pass kernel's launch shape, from the plan sweep: plain rows 4 vectors per thread per
// step on 256 threads up to 4096 vectors, 512 up to 8192, 1024 beyond; fused rows 2 vectors on
// 512 threads up to 4096 vectors and 1024 beyond (fp32 rows of at most 2048 vectors: 4 on 256).
void twopass_row(ks_plan_t *p, int64_t hv, bool fused, ks_dtype_t dtype) {
    p->kernel = KS_KERNEL_TWOPASS_ROW;
    p->flags = KS_PLAN_NO_PREFETCH;
    if (!fused) {
        p->vec_per_thread = 4;
        p->block = hv <= 4096 ? 256 : (hv <= 8192 ? 512 : 1024);
    } else if (dtype == KS_DTYPE_F32 && hv <= 2048) {
        p->vec_per_thread = 4;
        p->block = 256;
    } else {
        p->vec_per_thread = 2;
        p->block = hv <= 4096 ? 512 : 1024;
    }
    p->team = p->block;
}

// The band plan for many rows (more than SMs) of 1..2048 vectors; returns the rows each CTA
// handles.
int64_t band_row(ks_plan_t *p, int64_t hv, int64_t rows, int sm_count, bool fused,
                 ks_dtype_t dtype) {
    const RowBand *b = kRowBands[(int)dtype][fused ? 1 : 0];
    while (hv > b->hi) ++b;
    const char c = rows >= 4 * (int64_t)sm_count ? b->code : b->fallback;
    switch (c) {
    case 'E':
    case 'e':
    case 'H':
    case 'h':
    case 'W':
    case 'w': {
        p->kernel = KS_KERNEL_WARP_ROW;
        p->team = (c == 'E' || c == 'e') ? 8 : ((c == 'H' || c == 'h') ? 16 : 32);
        p->flags = (c == 'E' || c == 'H' || c == 'W') ? 0 : KS_PLAN_NO_PREFETCH;
        int v = 1;
        while ((int64_t)p->team * v < hv) v = v < 4 ? 2 * v : v + 2;  // 1, 2, 4, 6, 8
        p->vec_per_thread = v;
        if (v >= 6) {
            p->block = 128;
            return 4;
        }
        // up to 8 warps per CTA, but never fewer CTAs than SMs when the rows allow it
        const int64_t per_warp = 32 / p->team;
        int64_t warps = ceil_div(rows, (int64_t)sm_count * per_warp);
        warps = warps < 1 ? 1 : (warps > 8 ? 8 : warps);
        p->block = (int32_t)(32 * warps);
        return warps * per_warp;
    }
    case 'T':
    case 't':
        cta_row(p, hv, 2, c == 'T');
        return 1;
    case 'F':
    case 'f':
        cta_row(p, hv, 4, c == 'F');
        return 1;
    case 'R':
        bulk_row(p, hv, fused, 2);
        return 1;
    default:
        twopass_row(p, hv, fused, dtype);
        return 1;
    }
}

// Many wide rows: the two-pass kernel split over a cluster. Measured on GB300 (plan sweep, 384 MiB
// per tensor, bf16/fp16), against 0.66-0.81 of the copy peak with one CTA per row (whose last wave,
// at 10 rows per CTA, left SMs idle, and whose rows in flight outgrew L2 for fused rows):
//  * plain rows: C = clamp(hv / 4096, 2, 8) CTAs, slices of about 4096 vectors (64 KiB) read 1024
//    vectors a step by 256 threads at 4 vectors, each slice asked into L2 as the row starts;
//    0.83-0.86 at 16384 and 32768 vectors (two rows in flight measured 0.79-0.87, no better);
//  * fused rows: C = clamp(hv / 2048, 2, 8) CTAs, slices of about 2048 vectors, 512 threads at 2
//    vectors, two rows in flight per cluster (the next row's first pass in the loop of this row's
//    second, so every CTA reads DRAM and writes together); 0.93-0.95 at 8192 vectors, 0.91-0.93 at
//    16384 and 32768, against 0.80-0.90 with one row in flight.
void split_row(ks_plan_t *p, int64_t hv, bool fused) {
    const int64_t c = hv / (fused ? 2048 : 4096);
    p->kernel = KS_KERNEL_TWOPASS_ROW;
    p->cluster = (int32_t)(c < 2 ? 2 : (c > 8 ? 8 : c));
    p->vec_per_thread = fused ? 2 : 4;
    p->block = fused ? 512 : 256;
    p->team = p->block * p->cluster;
    p->flags = fused ? KS_PLAN_NO_PREFETCH : 0;
    p->stages = fused ? 2 : 0;
}

// Many rows wider than 2048 vectors whose tensors exceed L2: one band table per dtype and op,
// generated from a plan sweep on GB300 (384 MiB per tensor, every launch timed back to back) by
// the rule of the narrow tables (the fewest bands within a point of each measured width's best),
// over the one-CTA two-pass kernel, the two-pass kernel split over a cluster, the
// register-resident cluster kernel and the staged kernel split over a cluster. A band names a
// full launch: kernel, CTAs per cluster (0: one CTA per row), block (0: fitted to the slice,
// ceil(ceil(hv / cluster) / v) rounded up to a warp), vectors per thread (per step), stages and
// flags (bench.py --wide-bands-record / --wide-bands-derive; the measured record is committed in
// bands/ beside this file, and a CPU test re-derives the tables from it).
struct WideBand {
    int32_t hi;
    int8_t kernel;
    int8_t cluster;
    int16_t block;
    int8_t v;
    int8_t stages;
    int8_t flags;
};
constexpr int64_t kWideLo = 2049, kWideHi = 32768;
// BEGIN GENERATED WIDE BANDS
constexpr WideBand kWideBandsF32Plain[] = {{2304, 6, 0, 256, 4, 0, 1}, {2560, 4, 2, 0, 8, 3, 8}, {2816, 6, 0, 512, 4, 0, 0}, {3584, 4, 4, 0, 8, 2, 8}, {4096, 4, 2, 0, 8, 4, 0}, {4608, 4, 2, 0, 8, 3, 0}, {5120, 4, 2, 0, 4, 4, 8}, {6144, 4, 2, 0, 4, 3, 8}, {7168, 4, 8, 0, 4, 4, 8}, {9216, 4, 4, 0, 8, 4, 0}, {10240, 4, 8, 0, 4, 4, 8}, {12288, 4, 4, 0, 4, 4, 8}, {14336, 4, 4, 0, 4, 3, 8}, {16384, 4, 8, 0, 8, 3, 8}, {20480, 6, 4, 512, 2, 0, 0}, {32768, 4, 8, 0, 8, 2, 0}};
constexpr WideBand kWideBandsF32Fused[] = {{2304, 4, 2, 0, 4, 2, 0}, {3072, 6, 0, 512, 2, 0, 1}, {4096, 6, 2, 256, 4, 2, 1}, {5120, 4, 4, 0, 4, 2, 0}, {6144, 4, 8, 0, 4, 2, 0}, {8192, 6, 4, 256, 4, 2, 1}, {10240, 6, 4, 512, 2, 2, 1}, {16384, 4, 8, 0, 4, 3, 0}, {20480, 6, 8, 512, 2, 2, 1}, {28672, 6, 8, 256, 4, 2, 1}, {32768, 6, 4, 512, 4, 2, 1}};
constexpr WideBand kWideBandsF16Plain[] = {{2304, 4, 4, 0, 8, 2, 0}, {3072, 6, 0, 256, 4, 0, 1}, {4096, 6, 0, 512, 4, 0, 0}, {5120, 6, 0, 512, 2, 0, 0}, {7168, 4, 2, 0, 8, 2, 0}, {8192, 4, 2, 0, 8, 3, 8}, {14336, 4, 8, 0, 8, 2, 0}, {16384, 4, 4, 0, 8, 3, 8}, {24576, 6, 4, 256, 4, 2, 1}, {28672, 6, 4, 512, 2, 0, 0}, {32768, 4, 8, 0, 8, 2, 0}};
constexpr WideBand kWideBandsF16Fused[] = {{2560, 6, 0, 512, 2, 0, 1}, {3072, 4, 2, 0, 4, 2, 0}, {3584, 4, 8, 0, 4, 4, 0}, {5120, 6, 2, 512, 2, 2, 1}, {7168, 4, 4, 0, 4, 3, 0}, {12288, 6, 4, 512, 2, 2, 1}, {14336, 6, 4, 256, 4, 2, 1}, {32768, 6, 8, 256, 4, 2, 1}};
constexpr WideBand kWideBandsBf16Plain[] = {{2304, 6, 0, 512, 2, 0, 0}, {2560, 4, 2, 0, 8, 4, 0}, {2816, 6, 0, 256, 4, 0, 1}, {3072, 4, 2, 0, 8, 4, 8}, {3584, 6, 0, 512, 4, 0, 0}, {4096, 4, 4, 0, 8, 4, 8}, {4608, 4, 4, 0, 8, 3, 8}, {5120, 4, 4, 0, 8, 4, 0}, {6144, 4, 4, 0, 8, 4, 8}, {7168, 4, 2, 0, 8, 3, 8}, {8192, 4, 2, 0, 4, 3, 8}, {10240, 4, 8, 0, 8, 3, 8}, {14336, 4, 4, 0, 8, 2, 0}, {16384, 4, 4, 0, 4, 3, 8}, {28672, 6, 4, 512, 2, 2, 1}, {32768, 4, 8, 0, 8, 2, 0}};
constexpr WideBand kWideBandsBf16Fused[] = {{2304, 4, 8, 0, 4, 2, 0}, {2816, 4, 2, 0, 4, 2, 0}, {3072, 6, 0, 512, 2, 0, 1}, {3584, 6, 2, 512, 2, 2, 1}, {4096, 6, 2, 256, 4, 2, 1}, {5120, 6, 2, 512, 2, 2, 1}, {7168, 4, 8, 0, 4, 2, 0}, {10240, 6, 4, 512, 2, 2, 1}, {14336, 6, 4, 256, 4, 2, 1}, {16384, 4, 8, 0, 4, 3, 0}, {28672, 6, 8, 512, 2, 2, 1}, {32768, 6, 4, 512, 4, 2, 1}};
// END GENERATED WIDE BANDS

// Whether a wide table is well formed: widths rising to kWideHi, kernels that take rows this
// wide, clusters of 2..8 CTAs where the kernel splits rows (2..16 for the shared-memory rows
// kernel).
template <size_t N>
constexpr bool wide_bands_ok(const WideBand (&b)[N]) {
    for (size_t i = 0; i < N; ++i) {
        if (b[i].hi < kWideLo || b[i].hi > kWideHi || (i > 0 && b[i].hi <= b[i - 1].hi)) return false;
        const int k = b[i].kernel, c = b[i].cluster;
        const bool split = k == KS_KERNEL_BULK_ROW || k == KS_KERNEL_CLUSTER_ROW ||
                           (k == KS_KERNEL_TWOPASS_ROW && c != 0);
        if (k != KS_KERNEL_TWOPASS_ROW && k != KS_KERNEL_BULK_ROW && k != KS_KERNEL_CLUSTER_ROW)
            return false;
        const int cmax = (k == KS_KERNEL_BULK_ROW && (b[i].flags & KS_PLAN_SMEM_ROWS)) ? 16 : 8;
        if (split && (c < 2 || c > cmax)) return false;
        if (k == KS_KERNEL_TWOPASS_ROW && (b[i].block <= 0 || (b[i].v != 2 && b[i].v != 4))) return false;
        if (k == KS_KERNEL_BULK_ROW && (b[i].block != 0 || b[i].stages < 1 || (b[i].v != 4 && b[i].v != 8)))
            return false;
    }
    return b[N - 1].hi == kWideHi;
}
static_assert(wide_bands_ok(kWideBandsF32Plain) && wide_bands_ok(kWideBandsF32Fused) &&
                  wide_bands_ok(kWideBandsF16Plain) && wide_bands_ok(kWideBandsF16Fused) &&
                  wide_bands_ok(kWideBandsBf16Plain) && wide_bands_ok(kWideBandsBf16Fused),
              "a wide band table is malformed");
// Indexed [dtype code][op].
const WideBand *const kWideBands[3][2] = {
    {kWideBandsF32Plain, kWideBandsF32Fused},
    {kWideBandsF16Plain, kWideBandsF16Fused},
    {kWideBandsBf16Plain, kWideBandsBf16Fused},
};

// The wide band plan for a row of hv (2049..32768) vectors. Returns false when the band's launch
// does not fit this width (a fitted block over 512 threads or a ring over the shared-memory
// limit), and the caller keeps the general rules.
bool wide_band_row(ks_plan_t *p, int64_t hv, bool fused, ks_dtype_t dtype) {
    const WideBand *b = kWideBands[(int)dtype][fused ? 1 : 0];
    while (hv > b->hi) ++b;
    const int C = b->cluster;
    const int64_t slice = C >= 2 ? ceil_div(hv, C) : hv;
    if (C >= 2 && (C - 1) * slice >= hv) return false;  // a CTA without vectors
    int64_t block = b->block;
    if (block == 0) block = round_up(ceil_div(slice, b->v), 32);
    const bool wide_block = b->kernel == KS_KERNEL_TWOPASS_ROW ||
                            (b->kernel == KS_KERNEL_BULK_ROW && (b->flags & KS_PLAN_SMEM_ROWS) && b->v == 4);
    if (block > (wide_block ? 1024 : 512)) return false;
    if (b->kernel == KS_KERNEL_BULK_ROW) {
        const int64_t smem = kRingHeader + (int64_t)b->stages * slice * 16 * (fused ? 2 : 1);
        if (smem > kSmemLimit || (fused && b->v != 4)) return false;
        p->smem_bytes = (int32_t)smem;
    }
    p->kernel = b->kernel;
    p->cluster = C;
    p->block = (int32_t)block;
    p->vec_per_thread = b->v;
    p->stages = b->stages;
    p->flags = b->flags;
    p->team = p->block * (C >= 2 ? C : 1);
    return true;
}

}  // namespace

ks_status_t plan(int op, int64_t rows, int64_t hidden, ks_dtype_t dtype, bool aligned16,
                 int sm_count, int blocks_per_sm, int64_t l2_bytes, ks_plan_t *p) {
    if (!p) return fail(KS_ERR_INVALID_ARGUMENT, "plan pointer is NULL");
    memset(p, 0, sizeof *p);
    const int elem = elem_bytes(dtype);
    if (elem == 0) return fail(KS_ERR_UNSUPPORTED_DTYPE, "dtype code %d is not a ks_dtype_t", (int)dtype);
    if (op != 0 && op != 1) return fail(KS_ERR_INVALID_ARGUMENT, "op must be 0 to 4");
    if (hidden <= 0 || rows < 0 || sm_count <= 0 || blocks_per_sm < 0)
        return fail(KS_ERR_INVALID_ARGUMENT, "bad plan arguments");
    if (rows == 0) {
        p->kernel = KS_KERNEL_NONE;
        return KS_SUCCESS;
    }
    const bool fused = op == 1;
    const int per_vec = 16 / elem;
    const bool vec_ok = aligned16 && hidden % per_vec == 0;
    const int64_t hv = vec_ok ? hidden / per_vec : 0;
    int64_t rows_per_cta = 1;
    if (vec_ok && hv <= 128 && rows <= sm_count) {
        // Few narrow rows: a warp per row, the fewest vectors per lane that cover it.
        p->kernel = KS_KERNEL_WARP_ROW;
        p->vec_per_thread = hv <= 32 ? 1 : (hv <= 64 ? 2 : 4);
        p->team = 32;
        int64_t teams = ceil_div(rows, sm_count);
        teams = teams < 1 ? 1 : (teams > 8 ? 8 : teams);
        rows_per_cta = teams;
        p->block = (int32_t)(32 * teams);
    } else if (vec_ok && hv <= 2048 && rows <= sm_count) {
        // Latency regime, from a graph-replay sweep of few rows.
        if (fused && hv >= 1792 && rows * 8 <= sm_count) {
            p->kernel = KS_KERNEL_CLUSTER_ROW;
            p->cluster = 8;
            p->vec_per_thread = 1;
            p->block = (int32_t)round_up(ceil_div(hv, 8), 32);
            p->team = p->block * 8;
        } else if (!fused && hv <= 1024) {
            cta_row(p, hv, 2, true);
        } else {
            cta_row(p, hv, 4, fused);
        }
    } else if (vec_ok && hv <= kBandHi) {
        // Many rows: the measured band table.
        rows_per_cta = band_row(p, hv, rows, sm_count, fused, dtype);
    } else if (vec_ok && hv > 2048 && rows * 8 <= sm_count && hv <= 16384) {
        // Few rows wider than one CTA's registers: each row split over a cluster of 8 CTAs (the
        // register-resident cluster kernel), so the row's bytes come in over 8 SMs.
        const int64_t slice = ceil_div(hv, 8);
        p->kernel = KS_KERNEL_CLUSTER_ROW;
        p->cluster = 8;
        p->vec_per_thread = slice <= 512 ? 1 : (slice <= 1024 ? 2 : 4);
        p->block = (int32_t)round_up(ceil_div(slice, p->vec_per_thread), 32);
        p->team = p->block * 8;
    } else if (vec_ok && hv <= kWideHi && rows >= 4 * (int64_t)sm_count &&
               rows * hv * 32 > (l2_bytes > 0 ? l2_bytes : kDefaultL2Bytes) &&
               wide_band_row(p, hv, fused, dtype)) {
        // Many wide rows past L2: the measured wide band table.
    } else if (vec_ok && (hv > 8192 || (fused && hv > 4096)) &&
               rows * hv * 32 > (l2_bytes > 0 ? l2_bytes : kDefaultL2Bytes)) {
        // Very wide rows, more than L2 holds: the two-pass kernel split over a cluster. (Rows that
        // fit in L2 run faster one CTA per row: a probe of 76..1216 rows measured the one-CTA
        // kernel ahead up to about the L2 size, e.g. fused 8192-vector rows 0.82 against 0.76 at
        // 456 rows, 112 MiB, and the split kernels ahead beyond, 0.86 against 0.79 at 912 rows.)
        split_row(p, hv, fused);
    } else if (vec_ok && hv > 2048) {
        // Wider rows, more of them: the two-pass kernel (no width limit; the second pass from L2).
        twopass_row(p, hv, fused, dtype);
    } else {
        p->kernel = KS_KERNEL_SCALAR;
        int64_t b = round_up(ceil_div(hidden, 8), 32);
        p->block = (int32_t)(b < 32 ? 32 : (b > 1024 ? 1024 : b));
        p->team = p->block;
    }
    if (p->cluster >= 2) {  // whole clusters, one row each per pass
        int64_t clusters = rows;
        const int64_t cap = (int64_t)sm_count * blocks_per_sm / p->cluster;
        if (blocks_per_sm > 0 && clusters > cap) clusters = cap < 1 ? 1 : cap;
        if (p->kernel == KS_KERNEL_TWOPASS_ROW)
            clusters = split_clusters(rows, clusters, hv, fused, p->stages == 2 ? 2 : 1, l2_bytes);
        else  // as few clusters as give every cluster the same number of rows
            clusters = ceil_div(rows, ceil_div(rows, clusters));
        p->grid = clusters * p->cluster;
        p->rows_per_pass = clusters;
        return KS_SUCCESS;
    }
    const int64_t ctas = ceil_div(rows, rows_per_cta);
    const int64_t cap = (int64_t)sm_count * blocks_per_sm;
    p->grid = (blocks_per_sm > 0 && ctas > cap) ? cap : ctas;
    if (p->kernel == KS_KERNEL_TWOPASS_ROW) {
        const int64_t l2cap = twopass_grid_cap(hv, fused, sm_count, l2_bytes);
        if (p->grid > l2cap) p->grid = l2cap;
    }
    p->rows_per_pass = p->grid * rows_per_cta;
    return KS_SUCCESS;
}

}  // namespace ks

extern "C" {

ks_status_t ks_rms_norm(void *out, const void *x, const void *weight, int64_t rows,
                        int64_t hidden, float eps, ks_dtype_t dtype, ks_stream_t stream) {
    return ks::run(false, out, x, nullptr, weight, rows, hidden, eps, dtype, stream, nullptr);
}

ks_status_t ks_fused_add_rms_norm(void *x, void *residual, const void *weight, int64_t rows,
                                  int64_t hidden, float eps, ks_dtype_t dtype,
                                  ks_stream_t stream) {
    return ks::run(true, x, x, residual, weight, rows, hidden, eps, dtype, stream, nullptr);
}

ks_status_t ks_rms_norm_planned(void *out, const void *x, const void *weight, int64_t rows,
                                int64_t hidden, float eps, ks_dtype_t dtype,
                                const ks_plan_t *plan, ks_stream_t stream) {
    if (!plan) return ks::fail(KS_ERR_INVALID_ARGUMENT, "plan is NULL");
    return ks::run(false, out, x, nullptr, weight, rows, hidden, eps, dtype, stream, plan);
}

ks_status_t ks_fused_add_rms_norm_planned(void *x, void *residual, const void *weight,
                                          int64_t rows, int64_t hidden, float eps,
                                          ks_dtype_t dtype, const ks_plan_t *plan,
                                          ks_stream_t stream) {
    if (!plan) return ks::fail(KS_ERR_INVALID_ARGUMENT, "plan is NULL");
    return ks::run(true, x, x, residual, weight, rows, hidden, eps, dtype, stream, plan);
}

ks_status_t ks_device_faults(int32_t *flags, int32_t clear) {
    if (!flags) return ks::fail(KS_ERR_INVALID_ARGUMENT, "flags is NULL");
    *flags = 0;
    const int parts[4] = {ks::fault_flags_bf16(clear != 0), ks::fault_flags_f16(clear != 0),
                          ks::fault_flags_f32(clear != 0), ks::fault_flags_ops(clear != 0)};
    for (int v : parts) {
        if (v < 0) return ks::fail(KS_ERR_CUDA, "reading the device fault words failed");
        *flags |= v;
    }
    return KS_SUCCESS;
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
    if (op >= 2 && op <= 4) {
        if (!plan) return ks::fail(KS_ERR_INVALID_ARGUMENT, "plan pointer is NULL");
        if (hidden <= 0 || rows < 0 || sm_count <= 0)
            return ks::fail(KS_ERR_INVALID_ARGUMENT, "bad plan arguments");
        return ks::op_plan(op, rows, hidden, dtype, aligned16 != 0, sm_count, plan);
    }
    return ks::plan(op, rows, hidden, dtype, aligned16 != 0, sm_count, blocks_per_sm, 0, plan);
}

ks_status_t ks_set_launch_options(int32_t options) {
    if (options & ~KS_LAUNCH_PDL)
        return ks::fail(KS_ERR_INVALID_ARGUMENT, "unknown launch option bits 0x%x", (unsigned)options);
    ks::g_launch_options.store(options, std::memory_order_relaxed);
    return KS_SUCCESS;
}

int32_t ks_get_launch_options(void) { return ks::g_launch_options.load(std::memory_order_relaxed); }

int32_t ks_version(void) { return 100; }

}  // extern "C"
