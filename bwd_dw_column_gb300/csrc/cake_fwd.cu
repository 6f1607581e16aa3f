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
// recomputed forward (a checkpointed step runs the forward again before the
// backward) is bitwise equal.
#include <mutex>

#include "cake_launch.h"
#include "cake_rows.cuh"

namespace cake {

__device__ int g_fwd_status;

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
        e = cudaGetSymbolAddress((void **)&addr[dev], g_fwd_status);
        if (e != cudaSuccess)
            return e;
    }
    *out = addr[dev];
    return cudaSuccess;
}

// LPR < 32: rows of LPR lanes (16, 8 or 4), 32 / LPR per warp and row group --
// lanes [s * LPR, (s + 1) * LPR) hold the group's row s of a tile, and one
// log2(LPR)-step butterfly sums all of them; a thread's vectors are
// k * LPR + lane % LPR.  Otherwise a row spans the group's W warps.
template <int VPT, int LPR = 32>
__global__ void __launch_bounds__(kMaxThreadsFor(VPT), 1) fwd_rows_kernel(const __grid_constant__ FwdParams p)
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
        produce<2>(s, L, c, views, L.ntens, p.status, p.wait_ns);
        return;
    }

    const int gid = warp / W, wig = warp - gid * W;
    const int gtid = wig * 32 + lane;
    const int nvec = L.nvec;
    const bool has_res = L.ntens == 2;
    constexpr bool SUB = LPR < 32;
    constexpr int RG = SUB ? 32 / LPR : 1; // rows a group owns per tile
    const int sub = SUB ? lane / LPR : 0;
    const int ltid = SUB ? lane % LPR : gtid;
    const int vstride = SUB ? LPR : 32 * W;

    stage_weight(s, L, p.w, p.w_f32);
    // a thread's columns are the same on every row: its weights stay in
    // registers up to 24 columns per thread (GB300, T = 65536: H = 640 and
    // 8192 5 %, H = 4096 4 %, H = 6144 2 % faster; H = 5120 1 % slower, where
    // 24 columns on 7 warps then fit two CTAs per SM instead of three)
    constexpr bool kWreg = VPT <= 3;
    float2 wreg[kWreg ? VPT : 1][4];
    if constexpr (kWreg)
#pragma unroll
        for (int k = 0; k < VPT; ++k)
            weight_pairs(s, L, k * vstride + ltid < nvec ? k * vstride + ltid : 0, wreg[k]);

    bool abort = false;
    uint32_t slot = 0;
    uint32_t st = 0, ph = 0; // ring slot of tile `it` and the parity of its round
    for (uint32_t it = 0; it < c.ntiles && !abort; ++it) {
        abort = !mbar_wait(smem_addr(&s.full[st]), ph, p.wait_ns);
        const uint8_t *stage = s.ring + st * s.stage_bytes;
        const uint32_t gbase = c.r0 + it * c.tile_rows + gid * RG; // the group's first row
        const uint32_t r = gbase + sub;                           // this thread's row
        if (gbase < c.r_end) { // uniform across the group
            const bool live = r < c.r_end; // all but the last rows of a tile of part-warp rows
            const int tr = gid * RG + sub;
            const uint4 *xs = reinterpret_cast<const uint4 *>(stage + tr * L.H * 2);
            const uint4 *rsd = reinterpret_cast<const uint4 *>(stage + s.tens_bytes + tr * L.H * 2);
            // h = x, or bf16(x + residual): the FP32 sum of two BF16 values
            // rounds to the same BF16 value as their exact sum.  Sum of
            // squares: even / odd columns in the two lanes in the order of k
            // and q, then lane 0 + lane 1, then the group reduction.
            float2 h2[VPT][4];
            uint4 hraw[VPT];
            float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * vstride + ltid;
                uint4 h = make_uint4(0, 0, 0, 0);
                if (live && v < nvec) {
                    h = xs[v];
                    if (has_res) {
                        const uint4 rr = rsd[v];
                        uint32_t o[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            o[q] = pack2(add2(bf2(word(h, q)), bf2(word(rr, q))));
                        h = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                hraw[k] = h;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    h2[k][q] = bf2(word(h, q));
                    ss2 = fma2(h2[k][q], h2[k][q], ss2);
                }
            }
            const float ss = __fadd_rn(ss2.x, ss2.y);
            float tot = ss;
            if constexpr (SUB) {
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1)
                    tot += __shfl_xor_sync(0xffffffffu, tot, o);
                abort = __any_sync(0xffffffffu, abort);
            } else {
                tot = group_sum(ss, s, L, gid, wig, lane, slot++, abort);
            }
            const float rs = 1.0f / sqrtf(__fadd_rn(__fmul_rn(tot, L.inv_h), p.eps));
            const float2 rs2 = make_float2(rs, rs);

            uint16_t *yrow = p.y + out_off(p.y_st, p.y_sh, p.y_row_stride, p.y_uniform, r, L.nh);
            uint16_t *hrow = has_res
                                 ? p.h_new + out_off(p.hn_st, p.hn_sh, p.hn_row_stride, p.hn_uniform, r, L.nh)
                                 : nullptr;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * vstride + ltid;
                if (live && v < nvec && !abort) {
                    float2 w2[4];
                    if constexpr (kWreg) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            w2[q] = wreg[k][q];
                    } else {
                        weight_pairs(s, L, v, w2);
                    }
                    uint32_t o[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        o[q] = pack2(mul2(mul2(h2[k][q], rs2), w2[q]));
                    __stcs(reinterpret_cast<uint4 *>(yrow) + v, make_uint4(o[0], o[1], o[2], o[3]));
                    if (has_res)
                        __stcs(reinterpret_cast<uint4 *>(hrow) + v, hraw[k]);
                }
            }
            if (live && ltid == 0 && !abort)
                p.rstd[r] = rs;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&s.empty[st]));
        if (++st == (uint32_t)L.stages) {
            st = 0;
            ph ^= 1u;
        }
    }
    if (abort && lane == 0)
        set_status(p.status, kStatusTimeout);
}

template <int VPT, int LPR>
static cudaError_t launch_fwd_vpt(const FwdParams &p, int ctas, size_t smem, cudaStream_t stream)
{
    auto kern = fwd_rows_kernel<VPT, LPR>;
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
        cudaError_t e = status_ptr(&q.status);
        if (e != cudaSuccess)
            return e;
    }
    const int lanes = q.L.lanes_per_row;
    if (lanes != 32) {
        // rows of part of a warp: one warp per group, 32 / lanes rows per group
        if (q.L.warps_per_row != 1 || q.L.rows_per_group * lanes != 32)
            return cudaErrorInvalidValue;
        if (lanes == 16 && vpt == 1) return launch_fwd_vpt<1, 16>(q, ctas, smem, stream);
        if (lanes == 16 && vpt == 2) return launch_fwd_vpt<2, 16>(q, ctas, smem, stream);
        if (lanes == 8 && vpt == 1) return launch_fwd_vpt<1, 8>(q, ctas, smem, stream);
        if (lanes == 8 && vpt == 2) return launch_fwd_vpt<2, 8>(q, ctas, smem, stream);
        if (lanes == 4 && vpt == 2) return launch_fwd_vpt<2, 4>(q, ctas, smem, stream);
        return cudaErrorInvalidValue;
    }
    switch (vpt) {
    case 1: return launch_fwd_vpt<1, 32>(q, ctas, smem, stream);
    case 2: return launch_fwd_vpt<2, 32>(q, ctas, smem, stream);
    case 3: return launch_fwd_vpt<3, 32>(q, ctas, smem, stream);
    case 4: return launch_fwd_vpt<4, 32>(q, ctas, smem, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <int VPT, int LPR>
static cudaError_t occ_fwd(int threads, size_t smem, int *n)
{
    auto kern = fwd_rows_kernel<VPT, LPR>;
    cudaError_t e = ensure_smem_attr((const void *)kern, smem);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, threads, smem);
}

cudaError_t occupancy_fwd(int vpt, int lanes, int threads, size_t smem, int *n)
{
    if (lanes == 16 && vpt == 1) return occ_fwd<1, 16>(threads, smem, n);
    if (lanes == 16 && vpt == 2) return occ_fwd<2, 16>(threads, smem, n);
    if (lanes == 8 && vpt == 1) return occ_fwd<1, 8>(threads, smem, n);
    if (lanes == 8 && vpt == 2) return occ_fwd<2, 8>(threads, smem, n);
    if (lanes == 4 && vpt == 2) return occ_fwd<2, 4>(threads, smem, n);
    if (lanes != 32) return cudaErrorInvalidValue;
    switch (vpt) {
    case 1: return occ_fwd<1, 32>(threads, smem, n);
    case 2: return occ_fwd<2, 32>(threads, smem, n);
    case 3: return occ_fwd<3, 32>(threads, smem, n);
    case 4: return occ_fwd<4, 32>(threads, smem, n);
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
