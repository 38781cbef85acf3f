// Host-resident rows (ks_rms_norm_host, ks_fused_add_rms_norm_host). Two modes, host code only:
//
// Direct (workspace == NULL): page-locked host memory is mapped into the device's address space,
// and on Grace-Blackwell the GPU reaches it over the coherent NVLink-C2C link, so the row kernels
// read and write the host rows themselves: every byte crosses the link once each way, with no
// staging copy. The library first asks the runtime (cudaPointerGetAttributes) for the device view
// of both ends of every host buffer and refuses the call unless each is page-locked, mapped, and
// contiguous in that view; no kernel is launched on memory the device cannot address.
//
// Staged (a device workspace is given): the rows are copied to the device in chunks, normalised
// there, and copied back, with the three stages of consecutive chunks overlapping.
//
// The caller's device workspace is split into kSlots slots. Chunk i uses slot i % kSlots and
// moves through three library-owned streams: `up` copies its rows in, `work` runs the row kernel
// on the slot in place, `down` copies the results out. Events order each stage after the one
// before it and each reuse of a slot after the previous chunk's copy-out from that slot, so with
// three slots the copy-in of chunk i+1, the kernel of chunk i and the copy-out of chunk i-1 run
// at once (copy engines in both directions plus the SMs). The caller's stream is joined on entry
// (everything before it on that stream happens first) and on exit (everything after it waits for
// the last copy-out).
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "ks_internal.h"

namespace ks {
namespace {

constexpr int kSlots = 3;
constexpr int kMaxDevices = 64;
constexpr int64_t kAlign = 256;

struct Pipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t up = nullptr, work = nullptr, down = nullptr;
    cudaEvent_t enter = nullptr;
    cudaEvent_t up_done[kSlots] = {}, work_done[kSlots] = {}, down_done[kSlots] = {};
};
Pipe g_pipes[kMaxDevices];

cudaError_t init_pipe(Pipe &p) {
    if (p.ready) return cudaSuccess;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&p.up, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p.work, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&p.enter, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int s = 0; s < kSlots; ++s) {
        if ((e = cudaEventCreateWithFlags(&p.up_done[s], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.work_done[s], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&p.down_done[s], cudaEventDisableTiming)) != cudaSuccess)
            return e;
    }
    p.ready = true;
    return cudaSuccess;
}

int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// The device address of host buffer [p, p+nbytes) if it is page-locked memory mapped into the
// device's address space as one contiguous range; NULL otherwise. Only queries, no access.
void *device_view(const void *p, int64_t nbytes) {
    cudaPointerAttributes a{}, b{};
    const char *first = static_cast<const char *>(p);
    const char *last = first + (nbytes - 1);
    if (cudaPointerGetAttributes(&a, first) != cudaSuccess ||
        cudaPointerGetAttributes(&b, last) != cudaSuccess) {
        (void)cudaGetLastError();  // a failed query leaves no sticky state
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || b.type != cudaMemoryTypeHost || !a.devicePointer ||
        !b.devicePointer)
        return nullptr;
    if (static_cast<char *>(b.devicePointer) - static_cast<char *>(a.devicePointer) != nbytes - 1)
        return nullptr;
    return a.devicePointer;
}

}  // namespace

// Rows per chunk for a workspace: a slot holds the chunk's x rows (and, fused, its residual
// rows after them at the next 256-byte boundary). 0 if not even one row fits.
int64_t host_chunk_rows(bool fused, int64_t hidden, int e, int64_t workspace_bytes) {
    const int64_t slot = (workspace_bytes / kSlots) / kAlign * kAlign;
    const int64_t row = hidden * e;
    if (slot <= 0 || row <= 0) return 0;
    if (!fused) return slot / row;
    int64_t n = slot / (2 * row);
    while (n > 0 && round_up(n * row, kAlign) + n * row > slot) --n;
    return n;
}

ks_status_t run_host(bool fused, void *out, const void *x, void *res, const void *w,
                     int64_t rows, int64_t hidden, float eps, ks_dtype_t dtype, void *ws,
                     int64_t ws_bytes, ks_stream_t stream) {
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
    if (rows == 0) return KS_SUCCESS;
    if (!out || !x || !w || (fused && !res))
        return fail(KS_ERR_INVALID_ARGUMENT, "NULL pointer with rows > 0");
    if (misaligned(e, out, x, w, fused ? res : nullptr))
        return fail(KS_ERR_INVALID_ARGUMENT, "a pointer is not aligned to the %d-byte element", e);
    const int64_t row_bytes = hidden * e, nbytes = rows * row_bytes;
    if (fused) {
        if (overlaps(x, nbytes, res, nbytes))
            return fail(KS_ERR_OVERLAP, "x and residual storage overlap");
    } else if (out != x && overlaps(out, nbytes, x, nbytes)) {
        return fail(KS_ERR_OVERLAP, "out partially overlaps x (only out == x is allowed)");
    }
    if (!ws) {
        // ---- direct mode: the kernels address the host rows over the link
        void *xd = device_view(x, nbytes);
        void *od = fused ? xd : device_view(out, nbytes);
        void *rd = fused ? device_view(res, nbytes) : nullptr;
        if (!xd || !od || (fused && !rd))
            return fail(KS_ERR_INVALID_ARGUMENT,
                        "without a workspace every host buffer must be page-locked memory mapped "
                        "into the device's address space");
        return run(fused, od, xd, rd, w, rows, hidden, eps, dtype, stream, nullptr);
    }
    if (ws_bytes <= 0) return fail(KS_ERR_INVALID_ARGUMENT, "workspace_bytes must be > 0");
    if (misaligned(e, ws))
        return fail(KS_ERR_INVALID_ARGUMENT, "the workspace is not aligned to the %d-byte element", e);
    if (overlaps(ws, ws_bytes, w, row_bytes))
        return fail(KS_ERR_OVERLAP, "workspace and weight storage overlap");
    const int64_t chunk = host_chunk_rows(fused, hidden, e, ws_bytes);
    if (chunk < 1)
        return fail(KS_ERR_INVALID_ARGUMENT, "workspace of %lld bytes holds no row in each of %d slots",
                    (long long)ws_bytes, kSlots);

    // ---- device resources (created once per device)
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
    if (dev < 0 || dev >= kMaxDevices) return fail(KS_ERR_CUDA, "device ordinal %d out of range", dev);
    Pipe &p = g_pipes[dev];
    std::lock_guard<std::mutex> lock(p.mu);
    if ((ce = init_pipe(p)) != cudaSuccess)
        return fail(KS_ERR_CUDA, "creating the pipeline streams: %s", cudaGetErrorString(ce));

    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    const int64_t slot_bytes = (ws_bytes / kSlots) / kAlign * kAlign;
    const int64_t res_off = round_up(chunk * row_bytes, kAlign);
    char *base = static_cast<char *>(ws);
    const char *xs = static_cast<const char *>(x);
    char *os = static_cast<char *>(fused ? const_cast<void *>(x) : out);
    char *rs = static_cast<char *>(res);
    ks_status_t st = KS_SUCCESS;
    int last = 0;
    auto cuda_fail = [&](const char *what) {
        st = fail(KS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(ce));
    };

    if ((ce = cudaEventRecord(p.enter, caller)) != cudaSuccess ||
        (ce = cudaStreamWaitEvent(p.up, p.enter, 0)) != cudaSuccess) {
        cuda_fail("joining the caller's stream");
        return st;
    }
    for (int64_t i = 0, r0 = 0; r0 < rows; ++i, r0 += chunk) {
        const int s = (int)(i % kSlots);
        const int64_t n = (rows - r0 < chunk) ? rows - r0 : chunk;
        const int64_t off = r0 * row_bytes, len = n * row_bytes;
        char *sx = base + s * slot_bytes;
        char *sr = sx + res_off;
        // copy in, after the previous copy-out from this slot (this call's or an earlier one's)
        if ((ce = cudaStreamWaitEvent(p.up, p.down_done[s], 0)) != cudaSuccess ||
            (ce = cudaMemcpyAsync(sx, xs + off, len, cudaMemcpyDefault, p.up)) != cudaSuccess ||
            (fused && (ce = cudaMemcpyAsync(sr, rs + off, len, cudaMemcpyDefault, p.up)) != cudaSuccess) ||
            (ce = cudaEventRecord(p.up_done[s], p.up)) != cudaSuccess ||
            (ce = cudaStreamWaitEvent(p.work, p.up_done[s], 0)) != cudaSuccess) {
            cuda_fail("copying rows in");
            break;
        }
        // normalise in place on the slot
        st = run(fused, sx, sx, fused ? sr : nullptr, w, n, hidden, eps, dtype, p.work, nullptr);
        if (st != KS_SUCCESS) break;
        // copy out
        if ((ce = cudaEventRecord(p.work_done[s], p.work)) != cudaSuccess ||
            (ce = cudaStreamWaitEvent(p.down, p.work_done[s], 0)) != cudaSuccess ||
            (ce = cudaMemcpyAsync(os + off, sx, len, cudaMemcpyDefault, p.down)) != cudaSuccess ||
            (fused && (ce = cudaMemcpyAsync(rs + off, sr, len, cudaMemcpyDefault, p.down)) != cudaSuccess) ||
            (ce = cudaEventRecord(p.down_done[s], p.down)) != cudaSuccess) {
            cuda_fail("copying rows out");
            break;
        }
        last = s;
    }
    // The caller's stream waits for the last copy-out (the down stream runs in order), also on
    // the error paths, so nothing the call enqueued outlives the caller's view of it.
    cudaError_t je = cudaEventRecord(p.down_done[last], p.down);
    if (je == cudaSuccess) je = cudaStreamWaitEvent(caller, p.down_done[last], 0);
    if (st == KS_SUCCESS && je != cudaSuccess) {
        ce = je;
        cuda_fail("joining the caller's stream");
    }
    return st;
}

}  // namespace ks

extern "C" {

ks_status_t ks_rms_norm_host(void *out, const void *x, const void *weight, int64_t rows,
                             int64_t hidden, float eps, ks_dtype_t dtype, void *workspace,
                             int64_t workspace_bytes, ks_stream_t stream) {
    return ks::run_host(false, out, x, nullptr, weight, rows, hidden, eps, dtype, workspace,
                        workspace_bytes, stream);
}

ks_status_t ks_fused_add_rms_norm_host(void *x, void *residual, const void *weight, int64_t rows,
                                       int64_t hidden, float eps, ks_dtype_t dtype,
                                       void *workspace, int64_t workspace_bytes,
                                       ks_stream_t stream) {
    return ks::run_host(true, x, x, residual, weight, rows, hidden, eps, dtype, workspace,
                        workspace_bytes, stream);
}

int64_t ks_host_chunk_rows(int32_t op, int64_t hidden, ks_dtype_t dtype, int64_t workspace_bytes) {
    const int e = ks::elem_bytes(dtype);
    if (e == 0 || hidden <= 0 || (op != 0 && op != 1)) return -1;
    return ks::host_chunk_rows(op == 1, hidden, e, workspace_bytes);
}

}  // extern "C"
