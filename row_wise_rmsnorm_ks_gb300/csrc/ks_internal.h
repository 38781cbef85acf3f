// Declarations shared by the translation units of libks (host side only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ks.h"

namespace ks {

// Arguments every row kernel receives, passed by value in the kernel parameter space.
struct RowArgs {
    void *out;          // plain: y (may be exactly x); fused: x, written in place
    const void *x;      // the input rows
    void *res;          // fused: residual, read then written in place; plain: unused
    const void *w;      // weight [hidden]
    int64_t rows;
    int64_t hidden;     // H, the real row width (the divisor of the mean)
    int64_t hv;         // H / elements-per-16-byte-vector (vector kernels)
    float eps;
    int32_t stages;     // staged kernel: rows in the shared-memory ring
    int32_t l2_prefetch;  // two-pass kernels: each row's slice asked into L2 as the row starts
};

// Records a failure detail for ks_last_error() on this thread and returns `s`.
ks_status_t fail(ks_status_t s, const char *fmt, ...);
// Element size of a dtype in bytes (0 for an unknown code).
int elem_bytes(ks_dtype_t d);
// Whether [a, a+na) and [b, b+nb) share a byte.
bool overlaps(const void *a, int64_t na, const void *b, int64_t nb);
// True when any of the (non-NULL) pointers is not a multiple of the element size e: every kernel
// accesses whole elements, so such a pointer is an argument error.
bool misaligned(int e, const void *a, const void *b = nullptr, const void *c = nullptr,
                const void *d = nullptr);
// The checked launch path behind every device-pointer entry point (forced == NULL: heuristic).
ks_status_t run(bool fused, void *out, const void *x, void *res, const void *w, int64_t rows,
                int64_t hidden, float eps, ks_dtype_t dtype, ks_stream_t stream,
                const ks_plan_t *forced);

// The host-buffer path behind ks_*_host: direct when ws is NULL, staged through ws otherwise.
ks_status_t run_host(bool fused, void *out, const void *x, void *res, const void *w,
                     int64_t rows, int64_t hidden, float eps, ks_dtype_t dtype, void *ws,
                     int64_t ws_bytes, ks_stream_t stream);
// Rows per staged chunk for a workspace of ws_bytes (0 if a slot holds no row).
int64_t host_chunk_rows(bool fused, int64_t hidden, int e, int64_t ws_bytes);

// Whether ks_set_launch_options turned programmatic dependent launch on.
bool launch_pdl_enabled();

// Host heuristic: fills *p from the shape, the dtype and the device's SM count and L2 size
// (l2_bytes <= 0: a GB300's). blocks_per_sm == 0 leaves grid at one pass over the rows.
ks_status_t plan(int op, int64_t rows, int64_t hidden, ks_dtype_t dtype, bool aligned16,
                 int sm_count, int blocks_per_sm, int64_t l2_bytes, ks_plan_t *p);

// The next operators' default launch plan (op 2 SwiGLU with hidden = d, 3 Softmax, 4 LayerNorm),
// pure host code; grid left 0 (sized from the occupancy at launch).
ks_status_t op_plan(int op, int64_t rows, int64_t hidden, ks_dtype_t dtype, bool aligned16,
                    int sm_count, ks_plan_t *p);

// Per-dtype launchers (one translation unit each). `blocks_per_sm` queries the occupancy of the
// kernel the plan names; `max_clusters` how many of its clusters can be resident at once (plans
// with cluster >= 2; 0 if the query fails); `launch` enqueues it.
int blocks_per_sm_bf16(const ks_plan_t &p, bool fused);
int blocks_per_sm_f16(const ks_plan_t &p, bool fused);
int blocks_per_sm_f32(const ks_plan_t &p, bool fused);
int max_clusters_bf16(const ks_plan_t &p, bool fused);
int max_clusters_f16(const ks_plan_t &p, bool fused);
int max_clusters_f32(const ks_plan_t &p, bool fused);
// Reads (and with `clear`, zeroes) the device fault word of each translation unit's kernels on
// the current device; returns the OR of them, or -1 if the read failed.
int fault_flags_bf16(bool clear);
int fault_flags_f16(bool clear);
int fault_flags_f32(bool clear);
int fault_flags_ops(bool clear);
cudaError_t launch_bf16(const ks_plan_t &p, bool fused, const RowArgs &a, cudaStream_t s);
cudaError_t launch_f16(const ks_plan_t &p, bool fused, const RowArgs &a, cudaStream_t s);
cudaError_t launch_f32(const ks_plan_t &p, bool fused, const RowArgs &a, cudaStream_t s);

}  // namespace ks
