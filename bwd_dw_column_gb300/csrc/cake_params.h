// cake_params.h -- launch parameters shared by the host launchers and the
// kernels (plain structs, passed by value as __grid_constant__ arguments).
#pragma once

#include <cstddef>
#include <cstdint>

namespace cake {

// Default limit of every bounded wait in the kernels: one that has not
// completed after this long is treated as a hang -- the kernel records
// CAKE_ERR_TIMEOUT in its status word and leaves its loop.  The limit travels
// in the launch parameters (wait_ns), so a test can shorten it.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Bytes at the start of a CTA's dynamic shared memory for the mbarriers, the
// per-row reduction slots and flags; the staging ring follows.
constexpr int kMiscBytes = 1024;

// Shared memory for the FP32 copy of w, rounded up to 1 KB so that the ring
// after it stays 1 KB aligned.
__host__ __device__ constexpr unsigned weight_smem_bytes(int H) { return ((unsigned)H * 4u + 1023u) & ~1023u; }

// Largest CTA (consumer warps + the producer warp) a row kernel with VPT
// vectors per thread is compiled for; it caps the registers per thread at
// 65536 / threads.
__host__ __device__ constexpr int kMaxThreadsFor(int vpt) { return vpt == 1 ? 832 : 416; }
// Largest CTA of the backward build whose groups own two rows per stage (one
// group of up to 16 warps and the producer).  A CTA's warps spread over the
// SM's four register files of 16384, so its 17 warps (5 per file) leave 96
// registers a thread.
constexpr int kMaxThreadsR2 = 544;
// Named barriers: 1 + g for row group g when a row spans several warps, and
// the consumer-wide barrier after them (hardware barrier ids are 0..15).  A
// plan whose rows span several warps has at most kMaxRowGroupBarriers groups.
constexpr int kMaxRowGroupBarriers = 14;
constexpr int kConsumerBarrier = kMaxRowGroupBarriers + 1;

// How the backward turns the CTAs' dw partials into dw (cake_variant.single):
// the pair (main kernel + fixed-order reduce kernel), one kernel with FP64
// atomics, one kernel with a fixed-order two-level reduce by the
// last-arriving CTAs (groups of kTreeGroup CTAs), or one cooperative kernel
// whose CTAs meet at a grid barrier and then each reduce a slice of the
// columns in fixed order.
// And (kFormCluster) one cluster of up to kMaxCluster CTAs whose partials
// stay in their own shared memory: after the cluster's CTAs have all written
// theirs, CTA c sums slice c of the columns over every CTA's partial in CTA
// order (distributed shared memory), with no workspace and no second kernel.
constexpr int kFormPair = 0;
constexpr int kFormAtomic = 1;
constexpr int kFormTree = 2;
constexpr int kFormGrid = 3;
constexpr int kFormCluster = 4;
constexpr int kTreeGroup = 16;
constexpr int kMaxCluster = 16;
// Copies (banks) of the single kernel's FP64 column accumulators, at most.
constexpr int kMaxAccBanks = 8;

// Per-thread dw accumulation forms (same values as cake_dw_accum).
#define CAKE_DWM_PLAIN 0
#define CAKE_DWM_BLOCKED 1
#define CAKE_DWM_TWOSUM 2
#define CAKE_DWM_KAHAN 3

// A BF16 [T, nh, H] view.  Row r = (t, k) = (r / nh, r % nh) starts at
// base + t*st + k*sh (elements).  When the rows are equally spaced
// (nh == 1, or st == nh*sh) `uniform` is set and row r is at base + r*row_stride.
struct RowView {
    const uint16_t *base;
    int64_t st, sh;
    int64_t row_stride;
    int uniform;
    int dense; // uniform and row_stride == H: a run of rows is one contiguous block
};

// How a CTA is organised, shared by all kernels of the row pipeline.
//   consumer warps = groups * warps_per_row; one extra producer warp issues the
//   bulk copies.  A pipeline stage holds `groups` rows (one per group) of each
//   staged tensor.
struct Layout {
    int H;              // elements per row
    int nvec;           // H / 8: 16-byte vectors per row
    int warps_per_row;  // W
    int groups;         // NG
    int rows_per_group; // rows a group owns per stage (1; the backward 2, or 32 / lanes_per_row)
    int lanes_per_row;  // the backward: 32 (rows of whole warps), 16 or 8 (rows of part of a warp)
    int stages;         // ring depth
    int lo_bytes;       // backward, blocked dw sums: the per-thread compensated pairs kept in
                        // shared memory ([2 or 4 * VPT float4][consumer threads]); 0 otherwise
    int ntens;          // tensors staged per row (x[, residual] / x, dy[, dh])
    uint32_t rows;      // total rows R = T * nh
    uint32_t nh;
    uint32_t rows_per_cta; // contiguous rows per CTA (the last CTA may own fewer)
    float inv_h;        // 1.0f / H
};

struct FwdParams {
    Layout L;
    RowView x, res;     // res.base == nullptr: plain rows
    const void *w;      // [H] BF16 or FP32
    int w_f32;
    float eps;
    uint16_t *y;
    int64_t y_st, y_sh, y_row_stride;
    int y_uniform;
    uint16_t *h_new;
    int64_t hn_st, hn_sh, hn_row_stride;
    int hn_uniform;
    float *rstd;
    int *status;
    uint64_t wait_ns;   // limit of every bounded wait
};

struct BwdParams {
    Layout L;
    RowView x, dy, dh;  // staged tensors; dh.base == nullptr: no dh
    const float *rstd;
    const void *w;
    int w_f32;
    uint16_t *dx;
    int64_t dx_st, dx_sh, dx_row_stride;
    int dx_uniform;
    float *dw;          // [H]
    float2 *partials;   // pair: [ctas][H] (hi, lo)
    double *acc;        // single: [banks][H] FP64 column accumulators (zero between calls)
    int banks;          // single: copies of the accumulators (1..kMaxAccBanks, at most the CTA count)
    unsigned int *tree_cnt; // tree: [0] groups done, [1 + g] CTAs of group g done (zero between calls)
    float2 *group_totals;   // tree: [ceil(P / kTreeGroup)][H] (hi, lo)
    unsigned int *grid_cnt; // grid: CTA arrivals at the barrier (zero between calls)
    unsigned int *grid_gen; // grid: barrier generation (advances every call)
    unsigned int *arrivals; // single: CTA arrival counter (zero between calls)
    int block_rows;     // blocked accumulation: rows per FP32 block
    int *status;
    uint64_t wait_ns;   // limit of every bounded wait
    int grid_extra;     // grid form: arrivals its barrier expects beyond the CTA count (0; the
                        // timeout test sets 1 so that the barrier never completes)
    int cluster;        // cluster form: CTAs in the (one) cluster, which is the whole grid
    int direct_dw;      // pair of one CTA: the main kernel writes dw itself (no reduce launch)
};

struct ReduceParams {
    const float2 *partials; // [P][H]
    int P, H;
    float *dw;
    int slices;             // 1, 2, 4 or 8: partial ranges per column per warp
};

} // namespace cake
