// cake_bwd.cu -- training RMSNorm backward for sm_103a: launch dispatch over
// the forms (instantiated in cake_bwd_<form>.cu from the template in
// cake_bwd.cuh), the deterministic pair's fixed-order reduce kernel, and the
// kernels' device status word.
#include <mutex>

#include "cake_bwd.cuh"

namespace cake {

__device__ int g_bwd_status;

// Device address of the status word, looked up once per device.
static cudaError_t status_ptr(int **out)
{
    static std::mutex mu;
    static int *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        e = cudaGetSymbolAddress((void **)&addr[dev], g_bwd_status);
        if (e != cudaSuccess)
            return e;
    }
    *out = addr[dev];
    return cudaSuccess;
}

// Fixed-order reduction of the pair's CTA partials.  A CTA owns C columns
// (C = 32 / S) and 16 warps; lane = (slice s, column c).  The P partials of a
// column are split into 16*S contiguous ranges in ascending order, range
// w*S + s summed (compensated, ascending p, 8 loads in flight) by slice s of
// warp w.  The ranges are then combined in range order: the S slices of a
// column within each warp, then the 16 warps.  Small H gets more CTAs.
constexpr int kReduceWarps = 16;

__global__ void __launch_bounds__(32 * kReduceWarps) dw_reduce_kernel(const __grid_constant__ ReduceParams rp)
{
    __shared__ float2 part[kReduceWarps][32];
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = rp.slices, C = 32 / S;
    const int sl = lane / C, col = lane - sl * C;
    const int j = blockIdx.x * C + col;
    const int nrange = kReduceWarps * S;
    const int per = (rp.P + nrange - 1) / nrange;
    const int p0 = (warp * S + sl) * per;
    const int p1 = min(rp.P, p0 + per);
    float hi = 0.f, lo = 0.f;
    if (j < rp.H) {
        for (int q = p0; q < p1; q += 8) {
            float2 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = q + u < p1 ? __ldcg(rp.partials + (size_t)(q + u) * rp.H + j) : make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                comp_add(hi, lo, v[u].x);
                lo = __fadd_rn(lo, v[u].y);
            }
        }
    }
    // slices of a column, in slice order, into slice 0
    for (int t = 1; t < S; ++t) {
        const float h2 = __shfl_sync(0xffffffffu, hi, t * C + col);
        const float l2 = __shfl_sync(0xffffffffu, lo, t * C + col);
        if (sl == 0) {
            comp_add(hi, lo, h2);
            lo = __fadd_rn(lo, l2);
        }
    }
    if (sl == 0)
        part[warp][col] = make_float2(hi, lo);
    __syncthreads();
    if (warp == 0 && sl == 0 && j < rp.H) {
        float h = part[0][col].x, l = part[0][col].y;
        for (int w = 1; w < kReduceWarps; ++w) {
            comp_add(h, l, part[w][col].x);
            l = __fadd_rn(l, part[w][col].y);
        }
        rp.dw[j] = __fadd_rn(h, l);
    }
}

// ------------------------------------------------------------------ launch

// The row build of a layout: rows of part of a warp -- 5 half a warp at
// two 8-column vectors per thread, 6 half a warp at one, 7 a quarter at one,
// 8 a quarter at two, 9 an eighth at two (one warp per group, 32 / lanes rows
// per warp and group); 1 two rows per
// group of one vector per thread; 4 rows of one warp at 8 columns per
// thread; 0 otherwise; -1 for a combination no build serves.
static int row_build(int vpt, int W, int rpg, int lanes, int threads)
{
    if (lanes == 16 || lanes == 8 || lanes == 4) {
        if (W != 1 || rpg != 32 / lanes || threads > kMaxThreadsFor(vpt))
            return -1;
        if (lanes == 16)
            return vpt == 2 ? 5 : vpt == 1 ? 6 : -1;
        if (lanes == 8)
            return vpt == 1 ? 7 : vpt == 2 ? 8 : -1;
        return vpt == 2 ? 9 : -1;
    }
    if (lanes != 32)
        return -1;
    if (rpg == 2)
        return vpt == 1 && threads <= kMaxThreadsR2 ? 1 : -1;
    return vpt == 1 && W == 1 ? 4 : 0;
}

cudaError_t launch_bwd_rows(const BwdParams &p, int vpt, int single, int dwm, int ctas, size_t smem,
                            cudaStream_t stream)
{
    BwdParams q = p;
    if (q.status == nullptr) {
        cudaError_t e = status_ptr(&q.status);
        if (e != cudaSuccess)
            return e;
    }
    const int rb = row_build(vpt, q.L.warps_per_row, q.L.rows_per_group, q.L.lanes_per_row,
                             32 * (q.L.groups * q.L.warps_per_row + 1));
    if (rb < 0)
        return cudaErrorInvalidValue;
    switch (single) {
    case kFormPair: return launch_bwd_form<kFormPair>(q, vpt, rb, dwm, ctas, smem, stream);
    case kFormAtomic: return launch_bwd_form<kFormAtomic>(q, vpt, rb, dwm, ctas, smem, stream);
    case kFormTree: return launch_bwd_form<kFormTree>(q, vpt, rb, dwm, ctas, smem, stream);
    case kFormGrid: return launch_bwd_form<kFormGrid>(q, vpt, rb, dwm, ctas, smem, stream);
    case kFormCluster: return launch_bwd_form<kFormCluster>(q, vpt, rb, dwm, ctas, smem, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dw_reduce(const ReduceParams &rp, cudaStream_t stream)
{
    // launched as a programmatic dependent of the main kernel before it in
    // the stream: its CTAs may start early and block in griddepcontrol.wait
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rp.H + 32 / rp.slices - 1) / (32 / rp.slices)));
    cfg.blockDim = dim3(32 * kReduceWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, dw_reduce_kernel, rp);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

cudaError_t occupancy_bwd(int vpt, int w, int rpg, int lanes, int single, int dwm, int threads, size_t smem, int *n)
{
    const int rb = row_build(vpt, w, rpg, lanes, threads);
    if (rb < 0)
        return cudaErrorInvalidValue;
    switch (single) {
    case kFormPair: return occ_bwd_form<kFormPair>(vpt, rb, dwm, threads, smem, n);
    case kFormAtomic: return occ_bwd_form<kFormAtomic>(vpt, rb, dwm, threads, smem, n);
    case kFormTree: return occ_bwd_form<kFormTree>(vpt, rb, dwm, threads, smem, n);
    case kFormGrid: return occ_bwd_form<kFormGrid>(vpt, rb, dwm, threads, smem, n);
    case kFormCluster: return occ_bwd_form<kFormCluster>(vpt, rb, dwm, threads, smem, n);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t bwd_status(int *code, int clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(code, g_bwd_status, sizeof(int));
    if (e == cudaSuccess && clear) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(int));
    }
    return e;
}

} // namespace cake
