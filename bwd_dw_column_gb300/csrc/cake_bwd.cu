// cake_bwd.cu -- training RMSNorm backward for sm_103a.
//
// Per row (the standard RMSNorm gradient; the pages fix the outputs and their
// dtypes -- dx BF16, dw FP32 -- in the "Speedups ... GB300 windows" commit
// (#8577) quoted on the PR #8208 page, intro):
//   g_j = dy_j * w_j, xhat_j = h_j * rstd, c = (1/H) sum_j g_j * xhat_j,
//   dx_j = bf16(rstd * (g_j - xhat_j * c) [+ dh_j]),
// and over rows, the FP32 column sum dw_j = sum_r dy_rj * h_rj * rstd_r.
//
// Two backward forms, as the pages describe them:
//   * the deterministic pair (#8577 commit, intro: "the main kernel +
//     fixed-order dw reduce"): `bwd_rows_kernel<..., SINGLE=false>` writes one
//     compensated (hi, lo) dw partial per CTA into the workspace, then
//     `dw_reduce_kernel` sums the partials of each column in a fixed order
//     (programmatic dependent launch hides its launch);
//   * the single kernel (#8208 page, description: FP64 dw column sums, not
//     bitwise reproducible): `bwd_rows_kernel<..., SINGLE=true>` adds each
//     CTA's partial into FP64 column accumulators with L2 atomics; the CTA that
//     arrives last converts them to FP32 dw and zeroes the accumulators and the
//     arrival counter for the next call.  Nobody waits for anybody.
// dx is computed by the same code in every form, with a reduction order fixed
// by the row layout (VPT, W) alone, so it is bitwise identical across modes,
// variants and calls (#8208 page, description; #8253 commit: "dx is bitwise
// identical across every one" of the window edges).
//
// Per-thread dw accumulation over the CTA's rows (DWM), the pages' kernel
// kinds restated: plain FP32 sums; blocked FP32 sums folded into a
// compensated pair ("kb", PR #8899 page, window list); TwoSum per-thread sums
// with the product's rounding error kept (#8208 page, description; #8253
// commit: "the twosum forms").
#include "cake_launch.h"
#include "cake_rows.cuh"

namespace cake {

__device__ int g_bwd_status;

template <int VPT, int DWM, bool SINGLE>
__global__ void __launch_bounds__(VPT == 1 ? 576 : 512) bwd_rows_kernel(const __grid_constant__ BwdParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Layout &L = p.L;
    const Smem s = carve_smem(smem_raw, L);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = L.warps_per_row;
    const int consumer_warps = L.groups * W;
    const Chunk c = cta_chunk(L);

    init_ring(s, L);
    pdl_wait();

    if (warp == consumer_warps) {
        // producer warp: warm L2 with this CTA's rstd segment, then stream rows
        for (uint32_t r = c.r0 + lane * 32; r < c.r_end; r += 32 * 32)
            prefetch_l2(p.rstd + r);
        const RowView views[3] = {p.x, p.dy, p.dh};
        produce<3>(s, L, c, views, L.ntens, p.status);
        return;
    }

    const int gid = warp / W, wig = warp - gid * W;
    const int gtid = wig * 32 + lane;
    const int nvec = L.nvec;
    const bool has_dh = L.ntens == 3;

    float wf[VPT][8];
    load_weight<VPT>(p.w, p.w_f32, nvec, gtid, W, wf);

    // dw accumulators for this thread's columns
    float hi[VPT][8], lo[VPT][8], blk[VPT][8];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            hi[k][e] = 0.f;
            if (DWM != 0)
                lo[k][e] = 0.f;
            if (DWM == 1)
                blk[k][e] = 0.f;
        }
    int blk_rows = 0;

    auto rs_of_tile = [&](uint32_t tile) {
        const uint32_t r = c.r0 + tile * c.tile_rows + gid;
        return (tile < c.ntiles && r < c.r_end) ? __ldg(p.rstd + r) : 0.f;
    };
    float rs_cur = rs_of_tile(0);

    bool abort = false;
    uint32_t slot = 0;
    for (uint32_t it = 0; it < c.ntiles && !abort; ++it) {
        const float rs_next = rs_of_tile(it + 1);
        const uint32_t st = it % L.stages;
        abort = !mbar_wait(smem_addr(&s.full[st]), (it / L.stages) & 1);
        const uint8_t *stage = s.ring + st * s.stage_bytes;
        const uint32_t r = c.r0 + it * c.tile_rows + gid;
        if (r < c.r_end) { // uniform across the group
            const float rs = rs_cur;
            const uint4 *xs = reinterpret_cast<const uint4 *>(stage + gid * L.H * 2);
            const uint4 *dys = reinterpret_cast<const uint4 *>(stage + s.tens_bytes + gid * L.H * 2);
            const uint4 *dhs = reinterpret_cast<const uint4 *>(stage + 2 * s.tens_bytes + gid * L.H * 2);

            // pass 1: c = (1/H) sum g*xhat, fixed order: e within a vector, then k,
            // then the group reduction
            float dot = 0.f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * 32 * W + gtid;
                if (v < nvec) {
                    float xf[8], df[8];
                    unpack8(xs[v], xf);
                    unpack8(dys[v], df);
                    float d8 = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        d8 = fmaf(__fmul_rn(df[e], wf[k][e]), __fmul_rn(xf[e], rs), d8);
                    dot = __fadd_rn(dot, d8);
                }
            }
            const float tot = group_sum(dot, s, L, gid, wig, lane, slot++, abort);
            const float cc = __fmul_rn(tot, L.inv_h);

            // pass 2 (re-reads the staged row): dx and the dw terms
            uint16_t *dxrow = p.dx + out_off(p.dx_st, p.dx_sh, p.dx_row_stride, p.dx_uniform, r, L.nh);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * 32 * W + gtid;
                if (v < nvec && !abort) {
                    float xf[8], df[8], o[8];
                    unpack8(xs[v], xf);
                    unpack8(dys[v], df);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float g = __fmul_rn(df[e], wf[k][e]);
                        const float xh = __fmul_rn(xf[e], rs);
                        o[e] = __fmul_rn(fmaf(-xh, cc, g), rs);
                    }
                    if (has_dh) {
                        float hf[8];
                        unpack8(dhs[v], hf);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            o[e] = __fadd_rn(o[e], hf[e]);
                    }
                    __stcs(reinterpret_cast<uint4 *>(dxrow) + v, pack8(o));
                    // dw terms: dy*h is exact in FP32; one rounding for *rstd
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float a = __fmul_rn(df[e], xf[e]);
                        if (DWM == 0) {
                            hi[k][e] = fmaf(a, rs, hi[k][e]);
                        } else if (DWM == 1) {
                            blk[k][e] = fmaf(a, rs, blk[k][e]);
                        } else {
                            const float pr = __fmul_rn(a, rs);
                            const float pe = fmaf(a, rs, -pr);
                            float sum, err;
                            two_sum(hi[k][e], pr, sum, err);
                            hi[k][e] = sum;
                            lo[k][e] = __fadd_rn(lo[k][e], __fadd_rn(err, pe));
                        }
                    }
                }
            }
            if (DWM == 1 && ++blk_rows == p.block_rows) {
                blk_rows = 0;
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        comp_add(hi[k][e], lo[k][e], blk[k][e]);
                        blk[k][e] = 0.f;
                    }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&s.empty[st]));
        rs_cur = rs_next;
    }
    if (abort && lane == 0)
        set_status(p.status, kStatusTimeout);
    if (DWM == 0) {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                lo[k][e] = 0.f;
    }
    if (DWM == 1) {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                comp_add(hi[k][e], lo[k][e], blk[k][e]);
    }
    if (!SINGLE)
        pdl_launch_dependents();

    // ---- combine the row groups' partials in group order (shared memory)
    consumer_sync(L);
    float2 *comb = reinterpret_cast<float2 *>(s.ring);
    const int ncol = nvec * 8;
    if (L.groups > 1) {
        if (gid > 0) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * 32 * W + gtid;
                if (v < nvec)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        comb[(gid - 1) * ncol + v * 8 + e] = make_float2(hi[k][e], lo[k][e]);
            }
        }
        consumer_sync(L);
        if (gid == 0) {
            for (int g = 1; g < L.groups; ++g) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = k * 32 * W + gtid;
                    if (v < nvec)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float2 o = comb[(g - 1) * ncol + v * 8 + e];
                            comp_add(hi[k][e], lo[k][e], o.x);
                            lo[k][e] = __fadd_rn(lo[k][e], o.y);
                        }
                }
            }
        }
    }

    if (!SINGLE) {
        if (gid == 0) {
            float4 *dst = reinterpret_cast<float4 *>(p.partials + (size_t)blockIdx.x * ncol);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * 32 * W + gtid;
                if (v < nvec)
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        dst[v * 4 + e / 2] = make_float4(hi[k][e], lo[k][e], hi[k][e + 1], lo[k][e + 1]);
            }
        }
        return;
    }

    // ---- single kernel: FP64 column accumulation, the last CTA finalises
    if (gid == 0) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * 32 * W + gtid;
            if (v < nvec)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    atomicAdd(p.acc + v * 8 + e, (double)hi[k][e] + (double)lo[k][e]);
        }
        __threadfence();
    }
    consumer_sync(L);
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(p.arrivals, 1u);
        s.flag[1] = (prev == gridDim.x - 1);
    }
    consumer_sync(L);
    if (s.flag[1]) {
        __threadfence();
        const int nthr = consumer_warps * 32;
        for (int j = threadIdx.x; j < ncol; j += nthr) {
            const unsigned long long bits =
                atomicExch(reinterpret_cast<unsigned long long *>(p.acc + j), 0ull);
            p.dw[j] = (float)__longlong_as_double((long long)bits);
        }
        if (threadIdx.x == 0)
            atomicExch(p.arrivals, 0u);
    }
}

// Fixed-order reduction of the pair's CTA partials: column j of dw is the
// compensated sum of partials[p][j] over p ascending, split into 8 contiguous
// ranges (one per warp) that are then combined in warp order.
__global__ void __launch_bounds__(256) dw_reduce_kernel(const __grid_constant__ ReduceParams rp)
{
    __shared__ float2 part[8][32];
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x * 32 + lane;
    const int per = (rp.P + 7) / 8;
    const int p0 = warp * per;
    const int p1 = min(rp.P, p0 + per);
    float hi = 0.f, lo = 0.f;
    if (j < rp.H) {
        int q = p0;
        for (; q + 4 <= p1; q += 4) {
            float2 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = __ldcg(rp.partials + (size_t)(q + u) * rp.H + j);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                comp_add(hi, lo, v[u].x);
                lo += v[u].y;
            }
        }
        for (; q < p1; ++q) {
            const float2 v = __ldcg(rp.partials + (size_t)q * rp.H + j);
            comp_add(hi, lo, v.x);
            lo += v.y;
        }
    }
    part[warp][lane] = make_float2(hi, lo);
    __syncthreads();
    if (warp == 0 && j < rp.H) {
        float h = part[0][lane].x, l = part[0][lane].y;
        for (int w = 1; w < 8; ++w) {
            comp_add(h, l, part[w][lane].x);
            l += part[w][lane].y;
        }
        rp.dw[j] = h + l;
    }
}

// ------------------------------------------------------------------ launch

template <int VPT, int DWM, bool SINGLE>
static cudaError_t launch_rows(const BwdParams &p, int ctas, size_t smem, cudaStream_t stream)
{
    auto kern = bwd_rows_kernel<VPT, DWM, SINGLE>;
    cudaError_t e = ensure_smem_attr((const void *)kern, smem);
    if (e != cudaSuccess)
        return e;
    const int threads = 32 * (p.L.groups * p.L.warps_per_row + 1);
    kern<<<ctas, threads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int VPT>
static cudaError_t launch_vpt(const BwdParams &p, int single, int dwm, int ctas, size_t smem,
                              cudaStream_t stream)
{
    if (single) {
        if (dwm == 0) return launch_rows<VPT, 0, true>(p, ctas, smem, stream);
        if (dwm == 1) return launch_rows<VPT, 1, true>(p, ctas, smem, stream);
        return launch_rows<VPT, 2, true>(p, ctas, smem, stream);
    }
    if (dwm == 0) return launch_rows<VPT, 0, false>(p, ctas, smem, stream);
    if (dwm == 1) return launch_rows<VPT, 1, false>(p, ctas, smem, stream);
    return launch_rows<VPT, 2, false>(p, ctas, smem, stream);
}

cudaError_t launch_bwd_rows(const BwdParams &p, int vpt, int single, int dwm, int ctas, size_t smem,
                            cudaStream_t stream)
{
    BwdParams q = p;
    if (q.status == nullptr) {
        cudaError_t e = cudaGetSymbolAddress((void **)&q.status, g_bwd_status);
        if (e != cudaSuccess)
            return e;
    }
    switch (vpt) {
    case 1: return launch_vpt<1>(q, single, dwm, ctas, smem, stream);
    case 2: return launch_vpt<2>(q, single, dwm, ctas, smem, stream);
    case 3: return launch_vpt<3>(q, single, dwm, ctas, smem, stream);
    case 4: return launch_vpt<4>(q, single, dwm, ctas, smem, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dw_reduce(const ReduceParams &rp, cudaStream_t stream)
{
    // launched as a programmatic dependent of the main kernel before it in
    // the stream: its CTAs may start early and block in griddepcontrol.wait
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rp.H + 31) / 32));
    cfg.blockDim = dim3(256);
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
