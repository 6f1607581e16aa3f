/*
 * cake_rmsnorm.h -- C ABI of a training RMSNorm for one NVIDIA GB300 (sm_103a).
 *
 * The operation (the pages give names, dtypes and shapes, not formulas; the
 * formulas below are the standard RMSNorm and its exact gradient):
 *
 *   forward   h     = x                     (plain rows), or
 *             h     = bf16(x + residual)    (fused residual add; h is also
 *                                            returned as h_new)
 *             rstd  = 1 / sqrt(mean_j(h_j^2) + eps)        FP32, per row
 *             y_j   = bf16(h_j * rstd * w_j)
 *   backward  g_j   = dy_j * w_j,  xhat_j = h_j * rstd,  c = mean_j(g_j * xhat_j)
 *             dx_j  = bf16(rstd * (g_j - xhat_j * c) [+ dh_j])
 *             dw_j  = sum over all rows of dy_j * h_j * rstd      FP32
 *
 * Sources (page title, then the part of the page):
 *   - outputs and dtypes (y/dx BF16, rstd/dw FP32), the two backward modes
 *     sharing one forward, the per-head views and the `res` / `w32` routes:
 *     "Speedups ... GB300 windows" commit (#8577) quoted on the page of
 *     "feat(cake_rmsnorm): opt-in non-deterministic weight gradient for the
 *     autograd RMSNorm - #8208", intro and "Key"; PR #8899 page, first
 *     paragraph.
 *   - `deterministic` (default true): true gives a dw that is bitwise
 *     reproducible, false allows a single-kernel form whose dw is not; dx is
 *     bitwise identical across calls in both modes: #8208 page, description.
 *   - the deterministic backward is a pair: a main kernel that writes
 *     CTA-partial dw into a workspace, then a fixed-order dw reduce: #8577
 *     commit, intro; the workspace entry points: #8208 page, description.
 *   - per-head views: query [T, 24, 256] with strides (12288, 512, 1) and key
 *     [T, 4, 256], one shared w[256]: #8208 page, description.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     allocates nothing and never synchronises the host; every launch is
 *     asynchronous on `stream` (NULL = the legacy default stream).  A
 *     workspace must be 256-byte aligned.
 *   - A tensor is described by cake_tensor: base pointer plus element strides
 *     between tokens and between heads; the hidden dimension is contiguous.
 *     Row r of a [T, nh, H] view is (t, k) = (r / nh, r % nh).
 *   - Activations (x, residual, y, h_new, dy, dh, dx) are BF16; w is BF16 or
 *     FP32 (w_dtype); rstd and dw are FP32.
 *   - H must be a positive multiple of 8 and at most CAKE_MAX_HIDDEN; every
 *     activation base pointer and w must be 16-byte aligned and every stride a
 *     multiple of 8 elements (16 bytes), else CAKE_ERR_UNSUPPORTED.
 *   - rows = T * nh must be below 2^31.
 *   - Output views (y, h_new, dx) may not have rows that share memory, else
 *     CAKE_ERR_INVALID.  dx may not share memory with dy, x or dh; y and
 *     h_new may not share memory with each other, and share memory with an
 *     input only as exactly the same view (in place); else CAKE_ERR_INVALID.
 *   - Return codes come from host-side validation and from the CUDA launch
 *     (cudaGetLastError).  Faults that happen later on the device surface at
 *     the caller's next synchronisation, as with any CUDA call; the kernels'
 *     own bounded waits report through cake_rmsnorm_device_status().
 */
#ifndef CAKE_RMSNORM_H
#define CAKE_RMSNORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CAKE_ABI_VERSION 1
#define CAKE_MAX_HIDDEN 8192

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *cake_stream_t;

typedef enum {
    CAKE_OK = 0,
    CAKE_ERR_INVALID = 1,     /* null pointer, negative size, bad enum */
    CAKE_ERR_UNSUPPORTED = 2, /* H or alignment outside what the kernels take */
    CAKE_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    CAKE_ERR_CUDA = 4,        /* a CUDA runtime call failed */
    CAKE_ERR_TIMEOUT = 5      /* a kernel's bounded wait ran out (device status) */
} cake_status;

typedef enum { CAKE_BF16 = 0, CAKE_FP32 = 1 } cake_dtype;

/* Shape of the row set: T tokens, nh heads per token, H elements per row.
 * Plain [T, H] rows are nh = 1. */
typedef struct {
    int64_t tokens;
    int64_t heads;
    int64_t hidden;
} cake_shape;

/* A BF16 activation tensor: element (t, k, j) lives at
 * data + t*stride_token + k*stride_head + j. */
typedef struct {
    void *data;
    int64_t stride_token;
    int64_t stride_head;
} cake_tensor;

/*
 * Forward.  x: input rows.  residual: NULL or a tensor whose data is NULL for
 * plain rows; otherwise h = bf16(x + residual) is normalised and written to
 * h_new (required then, NULL otherwise).  w: [H] of w_dtype.  eps: added to
 * the mean square in FP32.  y: output rows.  rstd: [T*nh] FP32, row-major
 * over (t, k).  T = 0 is a no-op returning CAKE_OK.
 * The same kernels serve both backward modes, so y, rstd and h_new do not
 * depend on any mode, and a recomputed forward is bitwise equal to the first.
 */
cake_status cake_rmsnorm_fwd(const cake_shape *shape, const cake_tensor *x,
                             const cake_tensor *residual, const void *w,
                             cake_dtype w_dtype, float eps, const cake_tensor *y,
                             const cake_tensor *h_new, float *rstd,
                             cake_stream_t stream);

/*
 * Bytes of workspace cake_rmsnorm_bwd needs for this shape and mode
 * (0 only for T = 0): enough for every form the call may run.  The workspace
 * holds, in separate regions, the counters of the one-kernel forms, the FP64
 * column accumulators of the atomic single kernel, the CTA partials of the
 * pair and of the grid form, and the tree form's group totals.
 */
size_t cake_rmsnorm_bwd_workspace_size(const cake_shape *shape, cake_dtype w_dtype,
                                       int deterministic);

/*
 * Zero a workspace before its first use (an asynchronous memset on stream).
 * The single kernel needs its accumulator region to start at zero and leaves
 * it at zero again when it completes, so this is needed once per workspace
 * (and again only after a CAKE_ERR_TIMEOUT).  Calls that share a workspace
 * must be ordered on one stream.
 */
cake_status cake_rmsnorm_bwd_workspace_init(void *workspace, size_t workspace_bytes,
                                            cake_stream_t stream);

/*
 * Backward.  dy: gradient of y.  x: the normalised input (x for plain rows,
 * the saved h_new on the residual route).  rstd: the forward's FP32 rstd.
 * dh: NULL, or the gradient that reaches h_new directly on the residual route
 * (added into dx, which is then the gradient of both x and residual).
 * dx: output rows (may not share memory with dy, x or dh).  dw: [H] FP32,
 * overwritten.
 * deterministic != 0: the main + fixed-order reduce pair; dw is bitwise
 * reproducible for equal inputs and shape.  deterministic == 0: the window
 * table may pick a single-kernel form where one is faster than the pair, and
 * dw is then not guaranteed bitwise reproducible; on GB300 none is faster at
 * any measured shape, so the table runs the pair in both modes
 * (cake_rmsnorm_bwd_forced selects a single kernel).  A row set of at most
 * 24576 elements (T * nh * H) runs as one CTA whose main kernel writes dw
 * itself: one launch in both modes.  dx is the same bits in every mode and
 * variant.  T = 0: dw is zero-filled and CAKE_OK returned.
 */
cake_status cake_rmsnorm_bwd(const cake_shape *shape, const cake_tensor *dy,
                             const cake_tensor *x, const float *rstd, const void *w,
                             cake_dtype w_dtype, const cake_tensor *dh,
                             const cake_tensor *dx, float *dw, void *workspace,
                             size_t workspace_bytes, int deterministic,
                             cake_stream_t stream);

/*
 * The deterministic pair's two halves, for callers that schedule or time them
 * separately.  cake_rmsnorm_bwd(..., deterministic = 1, ...) is exactly
 * cake_rmsnorm_bwd_main followed by cake_rmsnorm_bwd_reduce on the same
 * stream, shape and workspace.
 *
 * _main: dx, plus one dw partial per CTA written into the workspace
 * (force_accum: -1 = the table's choice, else a cake_dw_accum).  dw is not
 * written.
 * _reduce: dw[j] = the partials of column j summed in a fixed order; reads
 * the partials the preceding _main call left in `workspace`.  has_dh must
 * match that call.
 */
cake_status cake_rmsnorm_bwd_main(const cake_shape *shape, const cake_tensor *dy,
                                  const cake_tensor *x, const float *rstd, const void *w,
                                  cake_dtype w_dtype, const cake_tensor *dh,
                                  const cake_tensor *dx, float *dw, void *workspace,
                                  size_t workspace_bytes, int force_accum,
                                  cake_stream_t stream);

cake_status cake_rmsnorm_bwd_reduce(const cake_shape *shape, int has_dh, float *dw,
                                    void *workspace, size_t workspace_bytes,
                                    cake_stream_t stream);

/* ---- variant table (host only; usable without a GPU) ------------------- */

/* How the per-thread dw column sums accumulate over a CTA's rows. */
typedef enum {
    CAKE_DW_PLAIN = 0,  /* FP32 running sum */
    CAKE_DW_BLOCKED = 1, /* FP32 sums over blocks of rows, folded into a
                            compensated (hi, lo) pair */
    CAKE_DW_TWOSUM = 2, /* error-free TwoSum per element, with the product's
                            rounding error kept as well */
    CAKE_DW_KAHAN = 3   /* Kahan-compensated FP32 sum of the rounded products */
} cake_dw_accum;

typedef struct {
    int single;        /* 0: main + fixed-order reduce pair; 1: single kernel,
                          FP64 atomics; 2: single kernel, fixed-order reduce
                          by the last-arriving CTAs (deterministic); 3:
                          single cooperative kernel, a grid barrier, then a
                          fixed-order reduce of a column slice by every CTA
                          (deterministic); 4: single kernel of one thread-block
                          cluster (ctas <= 16) whose CTAs keep their partials
                          in shared memory and reduce a column slice each
                          over the cluster's distributed shared memory, in
                          CTA order (deterministic; no workspace) */
    int dw_accum;      /* cake_dw_accum */
    int vec_per_thread; /* 16-byte vectors of a row held by each thread */
    int warps_per_row; /* warps that share one row (1 where lanes_per_row is 16 or 8) */
    int row_groups;    /* row groups (of warps_per_row warps) per CTA */
    int rows_per_group; /* rows each group owns per pipeline stage (1, 2 or 4) */
    int stages;        /* depth of the shared-memory ring */
    int ctas;          /* CTAs launched (P, also the number of dw partials) */
    int64_t rows_per_cta; /* contiguous rows each CTA owns */
    size_t smem_bytes; /* dynamic shared memory per CTA */
    int lanes_per_row; /* 32 x warps_per_row lanes, or 16 or 8: rows of part
                          of a warp, 32 / lanes_per_row per warp
                          (= rows_per_group) */
} cake_variant;

/*
 * Fill *out with the variant the window table picks for this shape, weight
 * dtype, mode and residual gradient.  force_single (0 to 4 as in
 * cake_variant.single) / force_accum (-1 = let the table decide) override
 * the table, as the tests that sweep every variant do; deterministic = 1
 * refuses force_single = 1 with CAKE_ERR_INVALID; force_single = 2 needs a
 * row layout of 8 columns per thread with one row per group or of 16
 * columns per thread (the table's choice for H <= 512 and for 1032 to
 * 1336), else CAKE_ERR_UNSUPPORTED.
 */
cake_status cake_rmsnorm_bwd_select(const cake_shape *shape, cake_dtype w_dtype,
                                    int deterministic, int has_dh, int force_single,
                                    int force_accum, cake_variant *out);

/* cake_rmsnorm_bwd with the variant forced as in cake_rmsnorm_bwd_select. */
cake_status cake_rmsnorm_bwd_forced(const cake_shape *shape, const cake_tensor *dy,
                                    const cake_tensor *x, const float *rstd,
                                    const void *w, cake_dtype w_dtype,
                                    const cake_tensor *dh, const cake_tensor *dx,
                                    float *dw, void *workspace, size_t workspace_bytes,
                                    int deterministic, int force_single,
                                    int force_accum, cake_stream_t stream);

/* ---- backward from and to host memory -------------------------------------
 * For rows that live in host memory (a training step whose activations were
 * offloaded, or a caller measuring the whole path from the host).  The rows
 * go to the device in `chunks` row chunks (1 .. 64, fewer if there are fewer
 * rows); the copy of one chunk in, the main kernel of the one before and the
 * copy of dx out of the one before that overlap, on `stream` (the kernels)
 * and two copy streams the library creates on a device at its first such
 * call and keeps.  One fixed-order reduce over the CTA partials of every
 * chunk then gives dw, so dw is bitwise reproducible for a given shape and
 * chunk count in both modes (its bits differ from cake_rmsnorm_bwd's, whose
 * partition is different); dx is the same bits as cake_rmsnorm_bwd's.
 *
 *   dy, x, rstd, dh (NULL: none), dx: HOST pointers to dense rows: [T*nh, H]
 *     BF16 with row stride H (a per-head view is passed as its T*nh rows),
 *     rstd [T*nh] FP32.  Page-locked memory lets the copies run
 *     asynchronously and overlap; pageable memory works but serialises.
 *   w: HOST pointer, [H] of w_dtype.  dw: HOST pointer, [H] FP32, overwritten.
 *   staging: DEVICE memory owned by the caller, 256-byte aligned, of at least
 *     cake_rmsnorm_bwd_host_staging_size() bytes (3 slots of chunk inputs and
 *     dx, the weight, dw and every chunk's partials), else CAKE_ERR_WORKSPACE.
 *   stream: must belong to the current device (else CAKE_ERR_INVALID); the
 *     call's copies and kernels come after earlier work on `stream`, and later
 *     work on `stream` comes after them: dx and dw are in host memory once
 *     `stream` has reached that point.  Calls on one device are enqueued one
 *     at a time; they share the copy streams.
 *   T = 0: dw is zero-filled on the host at once and CAKE_OK returned.
 */
size_t cake_rmsnorm_bwd_host_staging_size(const cake_shape *shape, cake_dtype w_dtype, int has_dh,
                                          int chunks);

cake_status cake_rmsnorm_bwd_host(const cake_shape *shape, const void *dy, const void *x,
                                  const float *rstd, const void *w, cake_dtype w_dtype,
                                  const void *dh, void *dx, float *dw, void *staging,
                                  size_t staging_bytes, int chunks, int deterministic,
                                  cake_stream_t stream);

/* ---- backward without caller scratch -------------------------------------
 * No counterpart in the pages: an addition of this library.
 *
 * Some callers cannot allocate device memory for the library -- code inside
 * a framework that owns every allocation, or a path that must not call
 * cudaMalloc (it can synchronise the device) in the middle of a step.
 * cake_rmsnorm_bwd_noalloc is the non-deterministic backward (the single
 * kernel, dx identical to cake_rmsnorm_bwd) with its scratch -- the CTA
 * arrival counter and the FP64 column accumulators -- in a library-owned
 * device array of 512 + 8 * CAKE_NOALLOC_MAX_HIDDEN bytes (64.5 KiB), which
 * every GPU that loads the library holds until the process exits.  The
 * caller still passes every input and output (same meaning as
 * cake_rmsnorm_bwd).  It allocates nothing and frees nothing.
 *   - hidden > CAKE_NOALLOC_MAX_HIDDEN: CAKE_ERR_WORKSPACE (the built-in
 *     scratch is too small); other argument errors as cake_rmsnorm_bwd.
 *   - The first call on a device looks up the array's device address with
 *     that device current and caches it; make that first call before any
 *     stream capture.  `stream` must belong to the current device, else
 *     CAKE_ERR_INVALID.
 *   - Every call clears the scratch it uses (an asynchronous memset) before
 *     its kernel.  All calls share the one array, so calls that overlap on
 *     the GPU (different streams, or several host threads) race: order them
 *     on one stream.
 */
#define CAKE_NOALLOC_MAX_HIDDEN 8192

cake_status cake_rmsnorm_bwd_noalloc(const cake_shape *shape, const cake_tensor *dy,
                                     const cake_tensor *x, const float *rstd, const void *w,
                                     cake_dtype w_dtype, const cake_tensor *dh,
                                     const cake_tensor *dx, float *dw, cake_stream_t stream);

/* ---- testing the timeout path ----------------------------------------------
 * No counterpart in the pages: an addition of this library, for tests.
 *
 * Every wait in the kernels is bounded; one that runs out sets the device
 * status to CAKE_ERR_TIMEOUT and the kernel returns instead of hanging.  This
 * entry point makes such a wait run out on purpose, from the host, so that a
 * test can check that path: it runs the cooperative grid form of the
 * backward (cake_rmsnorm_bwd_forced with force_single = 3) with its grid
 * barrier expecting one arrival more than the launch has CTAs, and with every
 * bounded wait limited to wait_limit_us microseconds (1 .. 1000000, else
 * CAKE_ERR_INVALID).  The barrier cannot complete, so each CTA gives up after
 * the limit, sets CAKE_ERR_TIMEOUT and returns: the launch ends by itself and
 * the CUDA context stays usable.  dx is written; dw is not.  The barrier's
 * arrival counter is left non-zero, so re-initialise the workspace
 * (cake_rmsnorm_bwd_workspace_init) before its next use, and read and clear
 * the status with cake_rmsnorm_device_status(&code, 1).  Other arguments as
 * cake_rmsnorm_bwd_forced.
 */
cake_status cake_rmsnorm_bwd_timeout_test(const cake_shape *shape, const cake_tensor *dy,
                                          const cake_tensor *x, const float *rstd, const void *w,
                                          cake_dtype w_dtype, const cake_tensor *dx, float *dw,
                                          void *workspace, size_t workspace_bytes,
                                          uint32_t wait_limit_us, cake_stream_t stream);

/*
 * Diagnostics: for the kernel a call with these arguments would launch, the
 * CTAs per SM the table plans for (*planned) and the number the CUDA runtime
 * reports can be resident (*resident).  backward = 0 asks about the forward
 * (has_extra: with residual); backward = 1 about the backward (has_extra:
 * with dh; deterministic and force_accum as in cake_rmsnorm_bwd_select).
 * A plan asks for no more CTAs than fit, so *planned <= *resident.
 */
cake_status cake_rmsnorm_plan_occupancy(const cake_shape *shape, int backward, int has_extra,
                                        int deterministic, int force_accum, int *planned,
                                        int *resident);

/* ---- status ------------------------------------------------------------ */

/* Static text for a status code. */
const char *cake_status_str(cake_status status);

/*
 * Read the device status word that kernels set when a bounded wait runs out
 * (CAKE_OK or CAKE_ERR_TIMEOUT) on the current device; clear != 0 resets it.
 * Synchronises the device.  Returns CAKE_ERR_CUDA if the read itself fails.
 */
cake_status cake_rmsnorm_device_status(int *code, int clear);

/* CAKE_ABI_VERSION of the loaded library. */
int cake_rmsnorm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CAKE_RMSNORM_H */
