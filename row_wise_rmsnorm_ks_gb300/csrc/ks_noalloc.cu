// ks_fused_add_rms_norm_host_noalloc: the staged host-buffer fused residual-add RMSNorm with its
// device workspace built into the library, for callers that must not allocate device memory.
//
// Who needs it: code whose device memory is owned by someone else's allocator and is not allowed
// to call cudaMalloc itself (a plugin inside a framework or an inference server that budgets
// every byte of the GPU), and latency-sensitive loops where cudaMalloc/cudaFree would stall
// (cudaFree synchronises the device). Such a caller has its rows in host memory and a stream,
// but no device buffer to lend as a workspace.
//
// The workspace is the file-scope array below: kScratchBytes of device memory that every GPU
// which loads this library holds until the process exits. Host code cannot use the array's name
// as a device address (on the host it names a shadow variable), so the first call on each device
// asks the runtime for the real address with cudaGetSymbolAddress, with that device current, and
// keeps it once the lookup succeeds. That first call should therefore come before any stream
// capture. Nothing here calls cudaMalloc, cudaFree or any other allocating routine.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "ks_internal.h"

namespace ks {
namespace {

// 24 MiB: three 8 MiB slots, enough for a chunk of 256 rows of bf16 x and residual at H = 8192;
// one row of x plus one of residual must fit a slot (about 2M bf16 elements of hidden).
constexpr int64_t kScratchBytes = 24ll << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
// The scratch array's device address per device, looked up under the mutex until a lookup
// succeeds: a failed lookup (say, an error left pending by earlier work on the device) is not
// kept, so a later call tries again.
struct ScratchSlot {
    std::mutex mu;
    void *ptr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];

}  // namespace
}  // namespace ks

extern "C" ks_status_t ks_fused_add_rms_norm_host_noalloc(void *x, void *residual,
                                                          const void *weight, int64_t rows,
                                                          int64_t hidden, float eps,
                                                          ks_dtype_t dtype, ks_stream_t stream) {
    using namespace ks;
    // Argument checks before any CUDA call, including the size limit of the built-in scratch.
    const int e = elem_bytes(dtype);
    if (e == 0) return fail(KS_ERR_UNSUPPORTED_DTYPE, "dtype code %d is not a ks_dtype_t", (int)dtype);
    if (hidden <= 0)
        return fail(KS_ERR_INVALID_ARGUMENT, "hidden must be > 0 (got %lld)", (long long)hidden);
    if (rows < 0) return fail(KS_ERR_INVALID_ARGUMENT, "rows must be >= 0 (got %lld)", (long long)rows);
    if (!std::isfinite(eps) || !(eps > 0.0f))
        return fail(KS_ERR_INVALID_ARGUMENT, "eps must be finite and > 0 (got %g)", (double)eps);
    if (hidden > INT64_MAX / (2 * e))
        return fail(KS_ERR_INVALID_ARGUMENT, "hidden %lld times twice the element size overflows int64",
                    (long long)hidden);
    if (host_chunk_rows(true, hidden, e, kScratchBytes) < 1)
        return fail(KS_ERR_INVALID_ARGUMENT,
                    "hidden %lld is too wide: one row of x and one of residual (%lld bytes) do not "
                    "fit a slot of the %lld-byte built-in scratch (3 slots)",
                    (long long)hidden, (long long)(2 * hidden * e), (long long)kScratchBytes);
    if (rows == 0) return KS_SUCCESS;
    if (!x || !residual || !weight) return fail(KS_ERR_INVALID_ARGUMENT, "NULL pointer with rows > 0");
    if (misaligned(e, x, residual, weight))
        return fail(KS_ERR_INVALID_ARGUMENT, "a pointer is not aligned to the %d-byte element", e);

    // Set-up, once per device (until it succeeds), with that device current: the scratch array's
    // device address.
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return fail(KS_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
    if (dev < 0 || dev >= kMaxDevices) return fail(KS_ERR_CUDA, "device ordinal %d out of range", dev);
    ScratchSlot &slot = g_scratch[dev];
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(slot.mu);
        if (!slot.ptr) {
            void *p = nullptr;
            ce = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (ce != cudaSuccess || !p) {
                (void)cudaGetLastError();
                return fail(KS_ERR_CUDA, "locating the built-in scratch: %s",
                            cudaGetErrorString(ce != cudaSuccess ? ce : cudaErrorInvalidSymbol));
            }
            slot.ptr = p;
        }
        scratch = slot.ptr;
    }

    // The staged path with the built-in scratch as its workspace. Each chunk's rows are copied
    // into a slot before the kernel reads them, so nothing in the scratch needs to start at zero.
    return run_host(true, x, x, residual, weight, rows, hidden, eps, dtype, scratch,
                    kScratchBytes, stream);
}
