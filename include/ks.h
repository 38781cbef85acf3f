/*
 * ks.h -- C ABI of libks: row-wise RMSNorm and fused residual-add RMSNorm on NVIDIA GB300
 * (sm_103a).
 *
 * Boundary style (kernel-set, "Operators"): every entry point returns a ks_status_t and takes
 * device pointers plus a ks_stream_t. No torch or C++ types cross this boundary.
 *
 * Semantics (Kernscope, "Numerical contract" and "API contract / Inputs"):
 *
 *   rms_norm:            for each row i of x viewed as [rows, hidden] (row-major, contiguous)
 *                          x32   = fp32(x[i, :])
 *                          scale = rsqrt(sum_j(x32_j^2) / hidden + eps)          (FP32)
 *                          out[i, j] = cast((x32_j * scale) * fp32(weight[j]))
 *   fused_add_rms_norm:  s = fp32(x[i, :]) + fp32(residual[i, :])                (one FP32 add)
 *                          residual[i, :] = cast(s)                               (in place)
 *                          x[i, :] = cast((s_j * rsqrt(mean(s^2) + eps)) * fp32(weight[j]))
 *                        normalising the FP32 s, not the value rounded into residual.
 *
 * cast() rounds to nearest, ties to even, to the element type (+-inf on fp16 overflow, NaN
 * stays NaN). rsqrt is the correctly rounded FP32 reciprocal square root; the sum of squares is
 * accumulated in FP32 in an order of the library's choosing (per-thread chains, a warp-shuffle
 * tree, then warps in order). That order follows the launch shape the heuristic picks from
 * (rows, hidden, dtype): results are bitwise reproducible for a given call shape on a given
 * device, but two calls whose row counts select different launch shapes may differ in the last
 * bit of some outputs (never in the residual, whose rounding is unique).
 *
 * Ownership and threading: the caller owns all memory; the library never allocates device or
 * pinned memory and keeps no state apart from a per-device cache of SM counts and kernel
 * occupancies. Calls are asynchronous on `stream`: a successful return means the work was
 * enqueued, and a fault in the kernel surfaces at the caller's next synchronisation. All entry
 * points are thread-safe. weight is read-only.
 *
 * Error behaviour: every argument check happens before any CUDA call, so an invalid call returns
 * its status without touching the device (and works on a machine without a GPU). The statuses:
 *   KS_ERR_INVALID_ARGUMENT   hidden <= 0, rows < 0, a NULL pointer with rows > 0, a pointer
 *                             that is not a multiple of the element size (2 or 4 bytes), eps
 *                             not finite or not > 0, or a byte size that overflows int64;
 *   KS_ERR_UNSUPPORTED_DTYPE  dtype outside ks_dtype_t;
 *   KS_ERR_OVERLAP            fused: any two of the x, residual, weight byte ranges overlap;
 *                             plain: out overlaps weight, or overlaps x without being exactly x;
 *   KS_ERR_CUDA               querying the device or launching failed (see ks_last_error()).
 * rows == 0 is legal (empty input) and returns KS_SUCCESS with no launch.
 */
#ifndef KS_H_
#define KS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of x, residual, out and weight (all four share it). */
typedef enum ks_dtype {
    KS_DTYPE_F32 = 0,
    KS_DTYPE_F16 = 1,
    KS_DTYPE_BF16 = 2
} ks_dtype_t;

typedef enum ks_status {
    KS_SUCCESS = 0,
    KS_ERR_INVALID_ARGUMENT = 1,
    KS_ERR_UNSUPPORTED_DTYPE = 2,
    KS_ERR_OVERLAP = 3,
    KS_ERR_CUDA = 4
} ks_status_t;

/* A cudaStream_t passed as an opaque handle; NULL is the legacy default stream. */
typedef void *ks_stream_t;

/*
 * RMSNorm (Kernscope, "Numerical contract / RMSNorm"; inputs per "API contract / Inputs").
 *   out     device pointer, [rows, hidden] elements of dtype; may be exactly x (in place).
 *   x       device pointer, [rows, hidden] elements of dtype, read-only unless out == x.
 *   weight  device pointer, [hidden] elements of dtype, read-only.
 *   rows    number of rows (the flattened leading dimensions); >= 0.
 *   hidden  row width (the last dimension); > 0.
 *   eps     finite, > 0; added to the mean square in FP32.
 * Pointers must be aligned to the element size (else KS_ERR_INVALID_ARGUMENT); 16-byte aligned
 * pointers with hidden*sizeof(element) a multiple of 16 take the vectorised kernels, anything
 * else a scalar kernel with the same arithmetic.
 */
ks_status_t ks_rms_norm(void *out, const void *x, const void *weight, int64_t rows,
                        int64_t hidden, float eps, ks_dtype_t dtype, ks_stream_t stream);

/*
 * Fused residual-add RMSNorm, in place on both x and residual (Kernscope, "Numerical contract /
 * Fused residual-add RMSNorm"; "API contract / Inputs": same shape, storage regions that do not
 * overlap, x and residual modified in place, inference only).
 *   x         device pointer, [rows, hidden]: input x; on return the normalised output.
 *   residual  device pointer, [rows, hidden]: input residual; on return cast(x + residual).
 *   weight    device pointer, [hidden], read-only.
 *   rows, hidden, eps, dtype, stream as for ks_rms_norm.
 */
ks_status_t ks_fused_add_rms_norm(void *x, void *residual, const void *weight, int64_t rows,
                                  int64_t hidden, float eps, ks_dtype_t dtype,
                                  ks_stream_t stream);

/* Static, human-readable name of a status ("KS_SUCCESS", ...); "KS_UNKNOWN_STATUS" otherwise. */
const char *ks_status_string(ks_status_t status);

/* Detail of the most recent non-success status returned on the calling thread (which check
 * failed, or the CUDA error string). Valid until the next ks_* call on that thread. */
const char *ks_last_error(void);

/*
 * Launch plan, for introspection and tests. A pure host function: no CUDA call. The plan
 * depends on the dtype (the heuristic was set per dtype from a sweep of every variant), the row
 * width in 16-byte vectors and the row count; grid is an upper bound when cluster >= 2 (the
 * launch caps whole clusters by what the device can hold resident).
 *   op              0 = rms_norm, 1 = fused_add_rms_norm, 2 = silu_and_mul (hidden = d, the
 *                   output row's width), 3 = softmax, 4 = layer_norm.
 *   aligned16       non-zero when every pointer of the call is 16-byte aligned.
 *   sm_count        multiprocessors of the device (152 on GB300).
 *   blocks_per_sm   resident CTAs per SM for the chosen kernel (0: plan the CTA shape only and
 *                   leave grid at the number of CTAs one pass over the rows needs). Ops 2..4
 *                   ignore it and leave grid 0: their launches size the grid from the kernel's
 *                   occupancy on the device.
 * On success *plan describes the launch the entry points would make. For ops 0 and 1 the L2
 * budget of the two-pass kernels is taken as 96 MiB (about three quarters of a GB300's L2);
 * the entry points use three quarters of the device's own L2.
 */
typedef struct ks_plan {
    int32_t kernel;         /* KS_KERNEL_* below */
    int32_t vec_per_thread; /* 16-byte vectors per thread and tensor (vector kernels): warp
                               rows 1, 2, 4, 6 or 8 (teams of 8 or 16 lanes: 1, 2 or 4); CTA
                               rows 2 or 4; staged rows 4 (split over a cluster, also 8 for the
                               plain op); cluster rows 1, 2 or 4; two-pass 2 or 4 per step */
    int32_t team;           /* threads per row: for warp rows 8, 16 or 32 lanes (several rows
                               per warp below 32; an explicit plan's 0 means 32), else block
                               (CTA per row) or block * cluster */
    int32_t block;          /* threads per CTA */
    int64_t grid;           /* CTAs launched */
    int64_t rows_per_pass;  /* rows in flight per pass over the grid (grid * rows per CTA) */
    int32_t stages;         /* staged kernel: rows in each CTA's shared-memory ring (else 0) */
    int32_t smem_bytes;     /* staged kernel: dynamic shared memory per CTA (else 0) */
    int32_t flags;          /* KS_PLAN_* bits below */
    int32_t cluster;        /* CTAs per cluster, one cluster per row: the cluster-row kernel
                               (2..8), or the staged or two-pass kernel split over a cluster
                               (2..8, the staged kernel with KS_PLAN_SMEM_ROWS 2..16; 0 or 1:
                               one CTA per row); 0 for the other kernels */
} ks_plan_t;

/* Plan flags. KS_PLAN_NO_PREFETCH: the register kernels (warp and CTA rows) load each row when
 * they reach it instead of loading the next row before reducing the current one (fewer
 * registers, so more resident CTAs). KS_PLAN_PDL: launch with programmatic stream serialization
 * (programmatic dependent launch), so the kernel may be scheduled while the previous kernel in
 * the stream finishes; it waits for that kernel's writes before its first memory access. */
#define KS_PLAN_NO_PREFETCH 1
#define KS_PLAN_PDL 2
/* KS_PLAN_AFFINE_SMEM (LayerNorm's staged ring only): the weight and bias rows live in the CTA's
 * shared memory beside the ring instead of in every thread's registers (fewer registers, so more
 * resident CTAs); the ring's shared memory grows by a row per array given. */
#define KS_PLAN_AFFINE_SMEM 4
/* KS_PLAN_SMEM_ROWS (RMSNorm without the residual, the staged kernel split over a cluster, 2 or
 * more stages): each row slice stays in its shared-memory stage through both passes instead of
 * moving into registers, and the CTA keeps two rows in flight, so one row's cluster exchange
 * overlaps the next row's sum of squares. vec_per_thread (4 or 8) then sizes only the weight
 * slice each thread holds. */
#define KS_PLAN_SMEM_ROWS 8

enum {
    KS_KERNEL_NONE = 0,     /* rows == 0: nothing is launched */
    KS_KERNEL_WARP_ROW = 1, /* one warp per row, row in registers, 16-byte vectors */
    KS_KERNEL_CTA_ROW = 2,  /* one CTA per row, row in registers, 16-byte vectors */
    KS_KERNEL_SCALAR = 3,   /* one CTA per row, element loads, two passes over the row */
    KS_KERNEL_BULK_ROW = 4, /* one CTA per row, rows streamed through a shared-memory ring by
                               bulk asynchronous copies, 4 vectors per thread; with cluster >= 2
                               the row is split over a cluster, each CTA streaming its slice of
                               ceil(hv / cluster) vectors through its own ring, partial sums
                               sent to every CTA of the cluster by asynchronous shared-memory
                               stores that complete on the receiver's mbarrier (rows too wide
                               for one CTA's registers) */
    KS_KERNEL_CLUSTER_ROW = 5, /* one cluster of `cluster` CTAs per row (few wide rows): each CTA
                                  holds a slice in registers and reduces it, partials exchanged
                                  in distributed shared memory */
    KS_KERNEL_TWOPASS_ROW = 6, /* one CTA per row, any width: the row read twice with 16-byte
                                  vectors (sum of squares, then outputs; the second pass from
                                  L2), vec_per_thread (2 or 4) vectors per thread in flight per
                                  step; the grid is capped so the rows in flight fit in L2,
                                  down to one CTA per SM. With cluster >= 2 each row is split
                                  over a cluster: CTA q runs both passes on its slice of
                                  ceil(hv / cluster) vectors and the slice sums reach every
                                  CTA of the cluster by asynchronous shared-memory stores that
                                  complete on the receiver's mbarrier;
                                  stages 2 keeps two rows in flight per cluster (the next
                                  row's first pass in the same loop as this row's second).
                                  Softmax and LayerNorm: their multi-pass wide kernel */
    KS_KERNEL_FLAT = 7         /* SwiGLU only: a grid-stride walk over all rows' vectors */
};

/*
 * What the kernel codes mean for the next operators (ks_silu_and_mul_planned,
 * ks_softmax_planned, ks_layer_norm_planned; ks_plan_launch with op 2..4):
 *   SwiGLU     KS_KERNEL_FLAT (block <= 256), KS_KERNEL_CTA_ROW (the row-structured kernel,
 *              its block fitted to the row with at most `block` threads, 32..256),
 *              KS_KERNEL_SCALAR (element loads, block <= 256).
 *   Softmax,   KS_KERNEL_WARP_ROW (a warp per row, vec_per_thread 2, 4, 6 or 8, block / 32
 *   LayerNorm  rows per CTA, block <= 128), KS_KERNEL_CTA_ROW (vec_per_thread 1, 2 or 4,
 *              block <= 512, block * vec_per_thread >= the row's vectors),
 *              KS_KERNEL_BULK_ROW (LayerNorm only: the staged ring, vec_per_thread 4,
 *              `stages` 2..8, block * 4 >= the row's vectors, block <= 512, or 1024 with
 *              KS_PLAN_AFFINE_SMEM), KS_KERNEL_TWOPASS_ROW (the multi-pass wide kernel, vec_per_thread
 *              4, block <= 1024 for Softmax and 512 for LayerNorm), KS_KERNEL_SCALAR
 *              (element loads, block <= 1024).
 * KS_PLAN_NO_PREFETCH picks the variant that loads each row when it comes: Softmax warp rows at
 * any vector count and CTA rows at 4 vectors (LayerNorm always prefetches; the flag is refused
 * there). A grid > 0 caps the CTAs launched; 0 sizes the grid from the occupancy.
 */

ks_status_t ks_plan_launch(int32_t op, int64_t rows, int64_t hidden, ks_dtype_t dtype,
                           int32_t aligned16, int32_t sm_count, int32_t blocks_per_sm,
                           ks_plan_t *plan);

/*
 * The same two operations with an explicit launch plan instead of the built-in heuristic (a
 * tuning hook: a plan from ks_plan_launch, edited). Semantics, arguments and errors are those of
 * ks_rms_norm / ks_fused_add_rms_norm, plus KS_ERR_INVALID_ARGUMENT when the plan does not fit
 * the call: a vector kernel on unaligned pointers or on a width that is not a multiple of 16
 * bytes, team * vec_per_thread vectors short of the row, a warp-row team other than 8, 16 or 32
 * lanes (or more than 4 vectors a lane on a team of 8 or 16), a block that is not a multiple of 32 or
 * exceeds the kernel's bound (warp rows 256, CTA rows 1024 at 2 vectors and 512 at 4, staged
 * rows 512, cluster rows 512, scalar 1024), a staged ring (stages 1..16) over 226 KB of shared
 * memory (per CTA: stages * slice * 16 bytes, twice that for the fused op), or a cluster outside
 * 2..8 CTAs (2..16 with KS_PLAN_SMEM_ROWS) whose slices (ceil(hv / cluster) vectors, at most
 * block * vec_per_thread each) do not cover the row or leave a CTA without vectors; a plan the
 * device cannot hold resident (e.g. a cluster of 16 it cannot place) gives KS_ERR_CUDA before any
 * launch. grid <= 0 lets the library size the persistent grid; cluster grids are whole clusters,
 * capped by the number the device can hold resident at once. smem_bytes and rows_per_pass are
 * recomputed. The plan is read, never written.
 */
ks_status_t ks_rms_norm_planned(void *out, const void *x, const void *weight, int64_t rows,
                                int64_t hidden, float eps, ks_dtype_t dtype,
                                const ks_plan_t *plan, ks_stream_t stream);
ks_status_t ks_fused_add_rms_norm_planned(void *x, void *residual, const void *weight,
                                          int64_t rows, int64_t hidden, float eps,
                                          ks_dtype_t dtype, const ks_plan_t *plan,
                                          ks_stream_t stream);

/*
 * Device-side faults of the current device: the OR of the fault words the kernels set (bit 0,
 * KS_FAULT_WAIT_TIMEOUT: a staged kernel gave up waiting for a bulk copy after about 2 s, left
 * its row loop and returned; its outputs are then incomplete). Reading synchronises with the
 * device. clear != 0 zeroes the words after reading. KS_ERR_CUDA if the read fails.
 */
#define KS_FAULT_WAIT_TIMEOUT 1
ks_status_t ks_device_faults(int32_t *flags, int32_t clear);

/*
 * The same two operations on rows held in host memory, for callers whose activations are not on
 * the device. Two modes:
 *   - direct (workspace == NULL): every host buffer must be page-locked memory mapped into the
 *     device's address space (cudaHostAlloc / cudaHostRegister; on Grace-Blackwell the GPU
 *     reaches it over the coherent NVLink-C2C link). The kernels read and write the host rows in
 *     place, on `stream`, with no staging copy. The library checks both ends of each buffer with
 *     cudaPointerGetAttributes first and returns KS_ERR_INVALID_ARGUMENT, launching nothing, if
 *     any is not page-locked, mapped and contiguous.
 *   - staged (workspace != NULL): any memory cudaMemcpy reads (pinned for the copies to overlap).
 *     The rows go in chunks through `workspace`, device memory the caller owns, split into 3
 *     slots; a chunk is as many rows as a slot holds (fused: x rows, then residual rows at the
 *     next 256-byte boundary; see ks_host_chunk_rows). Chunk i's copy to the device, the kernel
 *     on chunk i-1 and chunk i-2's copy back run at once on three streams the library creates
 *     once per device; the caller's `stream` is joined at entry (work queued on it earlier
 *     happens first) and at exit (work queued on it later waits for the last copy back).
 *     Calls that share a workspace must be ordered on one stream.
 * Both modes return once the work is queued: host buffers must stay valid and are complete only
 * after `stream` reaches that point.
 *   out, x, residual  host pointers, [rows, hidden]; rms_norm allows out == x; fused updates x
 *                     and residual in place.
 *   weight            device pointer, [hidden], read-only; must not overlap the workspace.
 *   workspace         device pointer or NULL (direct mode); workspace_bytes its size.
 * Errors as for the device entry points, plus KS_ERR_INVALID_ARGUMENT when a staged slot cannot
 * hold one row or a direct-mode buffer is not mapped, and KS_ERR_CUDA when the library's streams
 * cannot be created or a copy fails.
 */
ks_status_t ks_rms_norm_host(void *out, const void *x, const void *weight, int64_t rows,
                             int64_t hidden, float eps, ks_dtype_t dtype, void *workspace,
                             int64_t workspace_bytes, ks_stream_t stream);
ks_status_t ks_fused_add_rms_norm_host(void *x, void *residual, const void *weight, int64_t rows,
                                       int64_t hidden, float eps, ks_dtype_t dtype,
                                       void *workspace, int64_t workspace_bytes,
                                       ks_stream_t stream);

/* Rows per chunk the *_host entry points use for this workspace size (op 0 = rms_norm, 1 =
 * fused); 0 if a slot holds no row, -1 for invalid arguments. Pure host function. */
int64_t ks_host_chunk_rows(int32_t op, int64_t hidden, ks_dtype_t dtype, int64_t workspace_bytes);

/*
 * Fused residual-add RMSNorm of host rows, staged through device scratch memory built into the
 * library, so the call allocates nothing. (No counterpart in the source pages: this is a
 * convenience of this library.)
 *
 * For callers that cannot call cudaMalloc: code whose device memory belongs to another
 * allocator (a plugin in a framework or serving process that accounts for every byte on the
 * GPU) and latency-sensitive loops where cudaMalloc/cudaFree would stall the device. They have
 * host rows and a stream but no device buffer to lend; this entry point behaves like
 * ks_fused_add_rms_norm_host with a workspace, except that the workspace is a fixed 24 MiB array
 * inside the library that every GPU loading the library holds until the process exits.
 *   x, residual   host pointers (pinned for the copies to overlap), [rows, hidden], in place.
 *   weight        device pointer, [hidden], read-only.
 *   rows, hidden, eps, dtype, stream as for ks_fused_add_rms_norm_host.
 * Limit: one row of x plus one of residual must fit a third of the 24 MiB (hidden up to about
 * 2M bf16/fp16 or 1M fp32 elements); wider rows return KS_ERR_INVALID_ARGUMENT, launching
 * nothing. Any number of rows is processed, in chunks.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current (a lookup that fails is not kept: the next call tries again); make that
 * first call before any stream capture. All calls on a device share the one array and it keeps
 * the last call's contents (nothing in it needs to start at zero); calls whose GPU work overlaps
 * would race on it, so order them, e.g. on one stream. The library's own per-device copy and
 * kernel streams already queue each reuse of a third of the array after the previous copy out
 * of it, so consecutive calls of one process, from any of its streams, do not overlap there.
 */
ks_status_t ks_fused_add_rms_norm_host_noalloc(void *x, void *residual, const void *weight,
                                               int64_t rows, int64_t hidden, float eps,
                                               ks_dtype_t dtype, ks_stream_t stream);

/*
 * Process-wide launch options for the entry points that choose their own plan (all but the
 * *_planned ones, whose plan carries its flags). KS_LAUNCH_PDL: launch every row kernel with
 * programmatic dependent launch (see KS_PLAN_PDL), which hides launch latency in chains of small
 * kernels such as a decode step. Off by default. Unknown bits return KS_ERR_INVALID_ARGUMENT.
 * ks_get_launch_options returns the current bits.
 */
#define KS_LAUNCH_PDL 1
ks_status_t ks_set_launch_options(int32_t options);
int32_t ks_get_launch_options(void);

/*
 * SwiGLU activation (Kernscope, "Numerical contract / SwiGLU activation"): for x of shape
 * [rows, 2d], gate = fp32(x[:, :d]), up = fp32(x[:, d:]),
 * out[:, j] = cast((gate_j * sigmoid(gate_j)) * up_j) with sigmoid(g) = 1 / (1 + exp(-g)), FP32
 * throughout (exp within 2 ulp, the reciprocal an IEEE division).
 *   out  device pointer, [rows, d], must not overlap x.
 *   x    device pointer, [rows, 2d], read-only.
 *   rows >= 0 (0: nothing launched); d > 0 (it may be odd).
 * Errors as for ks_rms_norm (KS_ERR_OVERLAP if out overlaps x).
 */
ks_status_t ks_silu_and_mul(void *out, const void *x, int64_t rows, int64_t d, ks_dtype_t dtype,
                            ks_stream_t stream);

/*
 * Softmax over the last axis (Kernscope, "Numerical contract / Softmax"):
 * z = fp32(x) - max(fp32(x)), out = cast(exp(z) / sum(exp(z))). A row with NaN or +inf, or a
 * row that is all -inf, comes out NaN; -inf entries of a row with finite values come out 0.
 *   out  device pointer, [rows, hidden]; may be exactly x.
 *   x    device pointer, [rows, hidden].
 *   rows >= 0, hidden > 0. Errors as for ks_rms_norm.
 */
ks_status_t ks_softmax(void *out, const void *x, int64_t rows, int64_t hidden, ks_dtype_t dtype,
                       ks_stream_t stream);

/*
 * LayerNorm over the last axis (named on kernel-set's operator list, "Operators"; read as the
 * standard definition with FP32 steps): mean = sum(x)/H, var = sum((x - mean)^2)/H, rstd =
 * rsqrt(var + eps) correctly rounded, out = cast((((x - mean) * rstd) * w) + b).
 *   out           device pointer, [rows, hidden]; may be exactly x.
 *   weight, bias  device pointers, [hidden], or NULL (then 1 and 0); read-only.
 *   eps           finite, > 0. Errors as for ks_rms_norm.
 */
ks_status_t ks_layer_norm(void *out, const void *x, const void *weight, const void *bias,
                          int64_t rows, int64_t hidden, float eps, ks_dtype_t dtype,
                          ks_stream_t stream);

/*
 * The three operators above with an explicit launch plan instead of the built-in choice (a
 * tuning hook, as ks_rms_norm_planned is for RMSNorm: a plan from ks_plan_launch with op 2, 3 or
 * 4, edited; the kernel codes as listed after the KS_KERNEL_* enum). Arguments, semantics and
 * errors are those of the plain entry points, plus KS_ERR_INVALID_ARGUMENT, before any CUDA
 * call, for a NULL plan or one that does not fit the call (an unknown kernel for the operator, a
 * vector kernel on rows or pointers that are not 16-byte aligned, a team that does not cover the
 * row, a block or ring outside the kernel's bounds, a variant that does not exist). The plan is
 * read, never written; its derived fields are recomputed.
 */
ks_status_t ks_silu_and_mul_planned(void *out, const void *x, int64_t rows, int64_t d,
                                    ks_dtype_t dtype, const ks_plan_t *plan, ks_stream_t stream);
ks_status_t ks_softmax_planned(void *out, const void *x, int64_t rows, int64_t hidden,
                               ks_dtype_t dtype, const ks_plan_t *plan, ks_stream_t stream);
ks_status_t ks_layer_norm_planned(void *out, const void *x, const void *weight, const void *bias,
                                  int64_t rows, int64_t hidden, float eps, ks_dtype_t dtype,
                                  const ks_plan_t *plan, ks_stream_t stream);

/* Library version, major*10000 + minor*100 + patch. */
int32_t ks_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KS_H_ */
