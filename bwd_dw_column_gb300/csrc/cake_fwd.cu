// cake_fwd.cu -- training RMSNorm forward for sm_103a.
//
// Per row (standard RMSNorm; the pages fix the outputs -- y BF16 and rstd
// FP32 -- in the "Speedups ... GB300 windows" commit (#8577) quoted on the
// PR #8208 page, intro, and the residual route's BF16 output h_new in its
// "Key"):
//   h    = x, or h = bf16(x + residual)     (written to h_new)
//   rstd = 1 / sqrt((1/H) sum_j h_j^2 + eps)   FP32
//   y_j  = bf16((h_j * rstd) * w_j)
// One program serves both backward modes (#8253 commit: the forward is the
// same in both, so y, rstd and h_new are bitwise equal across modes); the
// sum of squares has a reduction order fixed by the row layout, so a
// recomputed forward (the checkpointed "2xfwd+bwd" step) is bitwise equal.
#include "cake_launch.h"
#include "cake_rows.cuh"

namespace cake {

__device__ int g_fwd_status;

template <int VPT>
__global__ void __launch_bounds__(VPT == 1 ? 576 : 512) fwd_rows_kernel(const __grid_constant__ FwdParams p)
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
        const RowView views[2] = {p.x, p.res};
        produce<2>(s, L, c, views, L.ntens, p.status);
        return;
    }

    const int gid = warp / W, wig = warp - gid * W;
    const int gtid = wig * 32 + lane;
    const int nvec = L.nvec;
    const bool has_res = L.ntens == 2;

    float wf[VPT][8];
    load_weight<VPT>(p.w, p.w_f32, nvec, gtid, W, wf);

    bool abort = false;
    uint32_t slot = 0;
    for (uint32_t it = 0; it < c.ntiles && !abort; ++it) {
        const uint32_t st = it % L.stages;
        abort = !mbar_wait(smem_addr(&s.full[st]), (it / L.stages) & 1);
        const uint8_t *stage = s.ring + st * s.stage_bytes;
        const uint32_t r = c.r0 + it * c.tile_rows + gid;
        if (r < c.r_end) { // uniform across the group
            const uint4 *xs = reinterpret_cast<const uint4 *>(stage + gid * L.H * 2);
            const uint4 *rsd = reinterpret_cast<const uint4 *>(stage + s.tens_bytes + gid * L.H * 2);
            // h = x, or bf16(x + residual) (the FP32 sum of two BF16 values
            // rounds to the same BF16 value as the exact sum)
            auto load_h = [&](int v) {
                uint4 h = xs[v];
                if (has_res) {
                    float a[8], b[8], t[8];
                    unpack8(h, a);
                    unpack8(rsd[v], b);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        t[e] = __fadd_rn(a[e], b[e]);
                    h = pack8(t);
                }
                return h;
            };
            // pass 1: sum of squares, fixed order: e within a vector, then k,
            // then the group reduction
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * 32 * W + gtid;
                if (v < nvec) {
                    float hf[8];
                    unpack8(load_h(v), hf);
                    float s8 = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        s8 = fmaf(hf[e], hf[e], s8);
                    ss = __fadd_rn(ss, s8);
                }
            }
            const float tot = group_sum(ss, s, L, gid, wig, lane, slot++, abort);
            const float rs = 1.0f / sqrtf(__fadd_rn(__fmul_rn(tot, L.inv_h), p.eps));

            // pass 2 (re-reads the staged row): y and h_new
            uint16_t *yrow = p.y + out_off(p.y_st, p.y_sh, p.y_row_stride, p.y_uniform, r, L.nh);
            uint16_t *hrow = has_res
                                 ? p.h_new + out_off(p.hn_st, p.hn_sh, p.hn_row_stride, p.hn_uniform, r, L.nh)
                                 : nullptr;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * 32 * W + gtid;
                if (v < nvec && !abort) {
                    const uint4 h = load_h(v);
                    float hf[8], o[8];
                    unpack8(h, hf);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        o[e] = __fmul_rn(__fmul_rn(hf[e], rs), wf[k][e]);
                    __stcs(reinterpret_cast<uint4 *>(yrow) + v, pack8(o));
                    if (has_res)
                        __stcs(reinterpret_cast<uint4 *>(hrow) + v, h);
                }
            }
            if (gtid == 0 && !abort)
                p.rstd[r] = rs;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&s.empty[st]));
    }
    if (abort && lane == 0)
        set_status(p.status, kStatusTimeout);
}

template <int VPT>
static cudaError_t launch_fwd_vpt(const FwdParams &p, int ctas, size_t smem, cudaStream_t stream)
{
    auto kern = fwd_rows_kernel<VPT>;
    cudaError_t e = ensure_smem_attr((const void *)kern, smem);
    if (e != cudaSuccess)
        return e;
    const int threads = 32 * (p.L.groups * p.L.warps_per_row + 1);
    kern<<<ctas, threads, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdParams &p, int vpt, int ctas, size_t smem, cudaStream_t stream)
{
    FwdParams q = p;
    if (q.status == nullptr) {
        cudaError_t e = cudaGetSymbolAddress((void **)&q.status, g_fwd_status);
        if (e != cudaSuccess)
            return e;
    }
    switch (vpt) {
    case 1: return launch_fwd_vpt<1>(q, ctas, smem, stream);
    case 2: return launch_fwd_vpt<2>(q, ctas, smem, stream);
    case 3: return launch_fwd_vpt<3>(q, ctas, smem, stream);
    case 4: return launch_fwd_vpt<4>(q, ctas, smem, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t fwd_status(int *code, int clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(code, g_fwd_status, sizeof(int));
    if (e == cudaSuccess && clear) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(int));
    }
    return e;
}

} // namespace cake
