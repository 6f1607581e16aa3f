// cake_bwd.cuh -- training RMSNorm backward for sm_103a: the row kernel
// template and its launchers.  Each translation unit cake_bwd_<form>.cu
// instantiates one form for every row layout and dw accumulation, so the
// forms compile in parallel; cake_bwd.cu holds the dispatch and the pair's
// reduce kernel.
//
// Per row (the standard RMSNorm gradient; the pages fix the outputs and their
// dtypes -- dx BF16, dw FP32 -- in the "Speedups ... GB300 windows" commit
// (#8577) quoted on the PR #8208 page, intro):
//   g_j = dy_j * w_j, xhat_j = h_j * rstd, c = (1/H) sum_j g_j * xhat_j,
//   dx_j = bf16(rstd * (g_j - xhat_j * c) [+ dh_j]),
// and over rows, the FP32 column sum dw_j = sum_r dy_rj * h_rj * rstd_r.
//
// The two backward forms the pages describe, and two more one-kernel forms:
//   * the deterministic pair (#8577 commit, intro: a main kernel, then a
//     fixed-order dw reduce): `bwd_rows_kernel<..., FORM=0, ...>` writes one
//     compensated (hi, lo) dw partial per CTA into the workspace, then
//     `dw_reduce_kernel` sums the partials of each column in a fixed order
//     (programmatic dependent launch hides its launch);
//   * the single kernel (#8208 page, description: FP64 dw column sums, not
//     bitwise reproducible): FORM=1 adds each CTA's partial into FP64 column
//     accumulators with L2 atomics; the CTA that arrives last converts them to
//     FP32 dw and zeroes the accumulators and the arrival counter for the next
//     call.  Nobody waits for anybody;
//   * the tree form (FORM=2): the last CTA of each group of CTAs sums its
//     group's partials, and the last group the group totals, in fixed order;
//   * the grid form (FORM=3): a cooperative launch whose CTAs meet at one
//     bounded grid barrier, then each reduces a slice of the columns in fixed
//     order.
// dx is computed by the same code in every form, with a reduction order fixed
// by the row layout (VPT, W) alone, so it is bitwise identical across modes,
// variants and calls (#8208 page, description; the #8253 commit states that
// dx does not change across the window edges).
//
// Per-thread dw accumulation over the CTA's rows (DWM), the pages' kernel
// kinds restated: plain FP32 sums; blocked FP32 sums folded into a
// compensated pair ("kb", PR #8899 page, window list); TwoSum per-thread sums
// with the product's rounding error kept (#8208 page, description; #8253
// commit, which names the TwoSum forms).
#pragma once

#include "cake_launch.h"
#include "cake_rows.cuh"

namespace cake {

// Where slot m = 4 v + q of a row group's partial sits in shared memory (in
// float4 units from the group's base): the four slots of vector v together,
// permuted by bits 1-2 of v, so that eight lanes on consecutive vectors
// writing one q, and eight lanes on consecutive slots reading, each touch
// eight different 16-byte bank quads (GB300: 0.3-0.5 us off a one-row call).
__device__ __forceinline__ int comb_slot(int v, int q) { return 4 * v + (q ^ ((v >> 1) & 3)); }

// Slot m = 4 v + q of the CTA partial (columns 8 v + 2 q and the next one,
// float4 (hi.x, lo.x, hi.y, lo.y)) summed over the row groups' partials in
// shared memory (at shared address comb, [group][comb_slot]) in group order,
// four groups' loads in flight at a time.
__device__ __forceinline__ float4 slot_sum(uint32_t comb, int nvec, int groups, int m)
{
    const int v = m >> 2, q = m & 3;
    const uint32_t base = comb + 16u * (uint32_t)comb_slot(v, q);
    const uint32_t gstride = 64u * (uint32_t)nvec;
    float4 a = ld_shared_f4(base);
    for (int g0 = 1; g0 < groups; g0 += 4) {
        float4 b[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            b[u] = g0 + u < groups ? ld_shared_f4(base + (uint32_t)(g0 + u) * gstride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (g0 + u < groups) {
                comp_add(a.x, a.y, b[u].x);
                a.y = __fadd_rn(a.y, b[u].y);
                comp_add(a.z, a.w, b[u].z);
                a.w = __fadd_rn(a.w, b[u].w);
            }
    }
    return a;
}

// The pair's CTA partial to global memory (or, for a pair of one CTA, dw
// itself: hi + lo rounded once, the bits the reduce of one partial gives).
__device__ __forceinline__ void emit_pair_body(uint32_t comb, int nvec, int groups, int nthr, float4 *dst, float2 *dw,
                                               int direct)
{
    for (int m = (int)threadIdx.x; m < 4 * nvec; m += nthr) {
        const float4 a = slot_sum(comb, nvec, groups, m);
        if (direct)
            dw[m] = make_float2(__fadd_rn(a.x, a.y), __fadd_rn(a.z, a.w));
        else
            dst[m] = a;
    }
}
// The same as a called function, for the build whose row loop uses every
// register a thread may have (32 columns per thread with Kahan sums): inlined
// there, its addressing is hoisted into the loop and spills.  Elsewhere the
// call costs more than it saves (GB300: about 0.5 us of a one-row call,
// although ptxas gives the called function no stack frame).
static __device__ __noinline__ void emit_pair_partial(uint32_t comb, int nvec, int groups, int nthr, float4 *dst,
                                                      float2 *dw, int direct)
{
    emit_pair_body(comb, nvec, groups, nthr, dst, dw, direct);
}

template <int VPT, int DWM, int FORM, int R2, bool KEEP, bool W1, int LPR = 32>
__device__ __forceinline__ void bwd_rows(const BwdParams &p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Layout &L = p.L;
    const Smem s = carve_smem(smem_raw, L);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = W1 ? 1 : L.warps_per_row; // W1: rows of one warp, known at compile time
    const int consumer_warps = L.groups * W;
    const Chunk c = cta_chunk(L);

    // cluster form: two mbarriers at the end of the misc area, each expecting
    // one arrival from every CTA of the cluster -- `ready` (its partial is in
    // its shared memory) and `done` (it has finished reading the others')
    uint64_t *cl_bar = reinterpret_cast<uint64_t *>(smem_raw + kMiscBytes - 32);
    if constexpr (FORM == kFormCluster) {
        if (threadIdx.x == 0) {
            mbar_init(smem_addr(&cl_bar[0]), (uint32_t)p.cluster);
            mbar_init(smem_addr(&cl_bar[1]), (uint32_t)p.cluster);
        }
    }
    init_ring(s, L);
    if constexpr (FORM == kFormCluster)
        cluster_sync_all(); // every CTA's barriers exist before any remote arrival
    pdl_wait();

    if (warp == consumer_warps) {
        // producer warp: warm L2 with this CTA's rstd segment, then stream rows
        for (uint32_t r = c.r0 + lane * 32; r < c.r_end; r += 32 * 32)
            prefetch_l2(p.rstd + r);
        const RowView views[3] = {p.x, p.dy, p.dh};
        produce<3>(s, L, c, views, L.ntens, p.status, p.wait_ns);
        return;
    }

    const int gid = warp / W, wig = warp - gid * W;
    const int gtid = wig * 32 + lane;
    const int nvec = L.nvec;
    const bool has_dh = L.ntens == 3;
    // LPR < 32: rows of LPR lanes (16 or 8), 32 / LPR per warp -- lanes
    // [s * LPR, (s + 1) * LPR) hold the group's row s of a tile, so one
    // log2(LPR)-step butterfly reduces them all; a thread's vectors are
    // k * LPR + lane % LPR.  Otherwise a row spans the group's W warps and a
    // thread's vectors are k * 32 * W + gtid.
    constexpr bool SUB = LPR < 32;
    const int sub = SUB ? lane / LPR : 0;
    const int ltid = SUB ? lane % LPR : gtid;
    const int vstride = SUB ? LPR : 32 * W;
    const bool owner = !SUB || sub == 0; // holds the combined partial at the end
    constexpr int RG = SUB ? 32 / LPR : R2; // rows a group owns per tile

    // This thread's rows of tile `tile`: gid*RG + sub + i, i < R2.
    auto rs_of = [&](uint32_t tile, int i) {
        const uint32_t r = c.r0 + tile * c.tile_rows + gid * RG + sub + i;
        return (tile < c.ntiles && r < c.r_end) ? __ldg(p.rstd + r) : 0.f;
    };
    // rstd of this group's rows, loaded kAhead tiles ahead (a register ring);
    // the first loads go out before the weight is staged, so that their
    // latency overlaps the weight's
    constexpr int kAhead = R2 == 1 ? 4 : 2;
    float rsr[kAhead][R2];
#pragma unroll
    for (int d = 0; d < kAhead; ++d)
#pragma unroll
        for (int i = 0; i < R2; ++i)
            rsr[d][i] = rs_of(d, i);

    // (with 8 columns per thread the element-wise staging measured 3-6 %
    // faster over a whole T = 65536 step, although it costs up to 3 us more
    // at small T)
    stage_weight<VPT != 1>(s, L, p.w, p.w_f32);
    // with 8 columns per thread (or 16 on rows of half a warp) a thread's
    // columns are the same on every row: keep their weights in registers
    // instead of reading shared memory per row (GB300: 3 % off the main
    // kernel for rows of 256 and 640 with plain or blocked sums; the Kahan
    // and TwoSum builds would spill, so they keep reading shared memory)
    constexpr bool kWreg = (VPT == 1 || SUB) && (DWM == CAKE_DWM_PLAIN || DWM == CAKE_DWM_BLOCKED);
    float2 wreg[kWreg ? VPT : 1][4];
    if constexpr (kWreg)
#pragma unroll
        for (int k = 0; k < VPT; ++k)
            weight_pairs(s, L, k * vstride + ltid < nvec ? k * vstride + ltid : 0, wreg[k]);

    // dw accumulators for this thread's columns (pairs of adjacent columns):
    // the partial is hi + lo in every form.
    float2 hi[VPT][4], lo[VPT][4], blk[VPT][4];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            hi[k][q] = make_float2(0.f, 0.f);
            lo[k][q] = make_float2(0.f, 0.f);
            blk[k][q] = make_float2(0.f, 0.f);
        }
    // Blocked sums keep the compensated pair in shared memory (this thread's
    // own slots: planes [0, 2 VPT) the low parts, [2 VPT, 4 VPT) the high
    // parts with 8 columns per thread), so the row loop holds only the block
    // sums -- the registers of the plain sum.  Wider layouts keep the high
    // parts in registers.
    constexpr bool kHiSmem = DWM == CAKE_DWM_BLOCKED && VPT == 1;
    const int nct = consumer_warps * 32;
    auto plane = [&](int i) -> float4 & { return s.lo[i * nct + threadIdx.x]; };
    auto get4 = [&](int i, float2 &a, float2 &b) {
        const float4 v = plane(i);
        a = make_float2(v.x, v.y);
        b = make_float2(v.z, v.w);
    };
    auto put4 = [&](int i, float2 a, float2 b) { plane(i) = make_float4(a.x, a.y, b.x, b.y); };
    // fold the block sums into the pair: (hi, lo) += blk, blk = 0
    auto fold = [&]() {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float2 h[4], l[4], e[4];
            if constexpr (kHiSmem) {
                get4(2 * VPT + 2 * k, h[0], h[1]);
                get4(2 * VPT + 2 * k + 1, h[2], h[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    h[q] = hi[k][q];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float2 sum;
                two_sum2(h[q], blk[k][q], sum, e[q]);
                h[q] = sum;
                blk[k][q] = make_float2(0.f, 0.f);
            }
            get4(2 * k, l[0], l[1]);
            get4(2 * k + 1, l[2], l[3]);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                l[q] = add2(l[q], e[q]);
            put4(2 * k, l[0], l[1]);
            put4(2 * k + 1, l[2], l[3]);
            if constexpr (kHiSmem) {
                put4(2 * VPT + 2 * k, h[0], h[1]);
                put4(2 * VPT + 2 * k + 1, h[2], h[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    hi[k][q] = h[q];
            }
        }
    };
    if (DWM == CAKE_DWM_BLOCKED)
#pragma unroll
        for (int k = 0; k < (kHiSmem ? 4 : 2) * VPT; ++k)
            plane(k) = make_float4(0.f, 0.f, 0.f, 0.f);
    int blk_rows = 0;


    bool abort = false;
    uint32_t slot = 0;
    uint32_t st = 0, ph = 0; // ring slot of tile `it` and the parity of its round
    for (uint32_t it = 0; it < c.ntiles && !abort; ++it) {
        float rsn[R2];
#pragma unroll
        for (int i = 0; i < R2; ++i)
            rsn[i] = rs_of(it + kAhead, i);
        abort = !mbar_wait(smem_addr(&s.full[st]), ph, p.wait_ns);
        const uint8_t *stage = s.ring + st * s.stage_bytes;
        const uint32_t gbase = c.r0 + it * c.tile_rows + gid * RG; // the group's first row
        const uint32_t rbase = gbase + sub;                           // this thread's first row
        const int nrow = rbase < c.r_end ? (int)min((uint32_t)R2, c.r_end - rbase) : 0; // uniform in the group but for SUB
        if (gbase < c.r_end) {
            // One pass over each staged row: m = dy*w and the row dot sum m*h
            // (even / odd columns in the two lanes, in the order of k and q;
            // then lane 0 + lane 1; then the group reduction), and the dw
            // terms dy*h*rstd (dy*h is exact in FP32), rows in order.
            // VPT == 1 keeps x and m in registers for the dx step; wider
            // layouts re-read the staged row instead (fewer registers).
            constexpr bool kKeep = (VPT == 1 || SUB) && KEEP;
            float2 x2[R2][kKeep ? VPT : 1][4], m2[R2][kKeep ? VPT : 1][4];
            float dot[R2];
#pragma unroll
            for (int i = 0; i < R2; ++i) {
                dot[i] = 0.f;
                if (i >= nrow)
                    continue;
                const int tr = gid * RG + sub + i;
                const float rs = rsr[0][i];
                const float2 rs2 = make_float2(rs, rs);
                const float2 nrs2 = make_float2(-rs, -rs);
                const uint4 *xs = reinterpret_cast<const uint4 *>(stage + tr * L.H * 2);
                const uint4 *dys = reinterpret_cast<const uint4 *>(stage + s.tens_bytes + tr * L.H * 2);
                float2 dot2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = k * vstride + ltid;
                    uint4 xr = make_uint4(0, 0, 0, 0), dr = make_uint4(0, 0, 0, 0);
                    if (v < nvec) {
                        xr = xs[v];
                        dr = dys[v];
                    }
                    float2 w2[4];
                    if constexpr (kWreg) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            w2[q] = wreg[k][q];
                    } else {
                        weight_pairs(s, L, v < nvec ? v : 0, w2);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 xv = bf2(word(xr, q));
                        const float2 d2 = bf2(word(dr, q));
                        const float2 mv = mul2(d2, w2[q]);
                        if (kKeep) {
                            x2[i][kKeep ? k : 0][q] = xv;
                            m2[i][kKeep ? k : 0][q] = mv;
                        }
                        dot2 = fma2(mv, xv, dot2);
                        const float2 a2 = mul2(d2, xv);
                        if (DWM == CAKE_DWM_PLAIN) {
                            hi[k][q] = fma2(a2, rs2, hi[k][q]);
                        } else if (DWM == CAKE_DWM_BLOCKED) {
                            blk[k][q] = fma2(a2, rs2, blk[k][q]);
                        } else if (DWM == CAKE_DWM_TWOSUM) {
                            // npr = -RN(a*rs); pe = a*rs - RN(a*rs) exactly (FMA);
                            // Knuth's TwoSum of hi and RN(a*rs) written with npr:
                            // s = hi + pr, e = (hi - (s - (s - hi))) + (pr - (s - hi));
                            // lo collects e and pe
                            const float2 npr = mul2(a2, nrs2);
                            const float2 pe = fma2(a2, rs2, npr);
                            const float2 sm = sub2(hi[k][q], npr);
                            const float2 bp = sub2(sm, hi[k][q]);
                            const float2 ap = sub2(sm, bp);
                            const float2 e = sub2(sub2(hi[k][q], ap), add2(npr, bp));
                            hi[k][q] = sm;
                            lo[k][q] = add2(lo[k][q], add2(e, pe));
                        } else {
                            // Kahan: lo holds the negated running compensation
                            const float2 y = fma2(a2, rs2, lo[k][q]);
                            const float2 t = add2(hi[k][q], y);
                            lo[k][q] = add2(sub2(hi[k][q], t), y);
                            hi[k][q] = t;
                        }
                    }
                }
                dot[i] = __fadd_rn(dot2.x, dot2.y);
            }
            float tot[R2];
            if constexpr (SUB) {
                // every row of the warp at once: a butterfly within each row's lanes
                tot[0] = dot[0];
#pragma unroll
                for (int o = LPR / 2; o > 0; o >>= 1)
                    tot[0] += __shfl_xor_sync(0xffffffffu, tot[0], o);
                abort = __any_sync(0xffffffffu, abort);
            } else {
                group_sum_n<R2, W1 ? 1 : 0>(dot, tot, s, L, gid, wig, lane, slot++, abort);
            }

#pragma unroll
            for (int i = 0; i < R2; ++i) {
                if (i >= nrow)
                    continue;
                const int tr = gid * RG + sub + i;
                const float rs = rsr[0][i];
                const float2 rs2 = make_float2(rs, rs);
                // dx_j = rs*(g_j - xhat_j*c) = m_j*rs - h_j*kk, kk = ((tot/H)*rs)*rs*rs:
                // each product by rs brings kk back towards the scale of g, so no
                // intermediate leaves FP32's range before the result does
                const float kk = __fmul_rn(__fmul_rn(__fmul_rn(__fmul_rn(tot[i], L.inv_h), rs), rs), rs);
                const float2 nk2 = make_float2(-kk, -kk);
                const uint4 *xs = reinterpret_cast<const uint4 *>(stage + tr * L.H * 2);
                const uint4 *dys = reinterpret_cast<const uint4 *>(stage + s.tens_bytes + tr * L.H * 2);
                const uint4 *dhs = reinterpret_cast<const uint4 *>(stage + 2 * s.tens_bytes + tr * L.H * 2);
                uint16_t *dxrow =
                    p.dx + out_off(p.dx_st, p.dx_sh, p.dx_row_stride, p.dx_uniform, rbase + i, L.nh);
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = k * vstride + ltid;
                    if (v < nvec && !abort) {
                        uint4 hv = make_uint4(0, 0, 0, 0);
                        if (has_dh)
                            hv = dhs[v];
                        uint4 xr2 = make_uint4(0, 0, 0, 0), dr2 = make_uint4(0, 0, 0, 0);
                        float2 w2[4];
                        if (!kKeep) {
                            xr2 = xs[v];
                            dr2 = dys[v];
                            if constexpr (kWreg) {
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    w2[q] = wreg[k][q];
                            } else {
                                weight_pairs(s, L, v, w2);
                            }
                        }
                        uint32_t o[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 xv = kKeep ? x2[i][kKeep ? k : 0][q] : bf2(word(xr2, q));
                            const float2 mv = kKeep ? m2[i][kKeep ? k : 0][q] : mul2(bf2(word(dr2, q)), w2[q]);
                            float2 d = fma2(mv, rs2, mul2(xv, nk2));
                            if (has_dh)
                                d = add2(d, bf2(word(hv, q)));
                            o[q] = pack2(d);
                        }
                        __stcs(reinterpret_cast<uint4 *>(dxrow) + v, make_uint4(o[0], o[1], o[2], o[3]));
                    }
                }
            }
            if (DWM == CAKE_DWM_BLOCKED && (blk_rows += nrow) >= p.block_rows) {
                blk_rows = 0;
                fold();
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&s.empty[st]));
        if (++st == (uint32_t)L.stages) {
            st = 0;
            ph ^= 1u;
        }
#pragma unroll
        for (int d = 0; d + 1 < kAhead; ++d)
#pragma unroll
            for (int i = 0; i < R2; ++i)
                rsr[d][i] = rsr[d + 1][i];
#pragma unroll
        for (int i = 0; i < R2; ++i)
            rsr[kAhead - 1][i] = rsn[i];
    }
    if (abort && lane == 0)
        set_status(p.status, kStatusTimeout);
    if (DWM == CAKE_DWM_BLOCKED) {
        fold();
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            get4(2 * k, lo[k][0], lo[k][1]);
            get4(2 * k + 1, lo[k][2], lo[k][3]);
            if constexpr (kHiSmem) {
                get4(2 * VPT + 2 * k, hi[k][0], hi[k][1]);
                get4(2 * VPT + 2 * k + 1, hi[k][2], hi[k][3]);
            }
        }
    }
    if constexpr (SUB) {
        // the lanes of rows 1 .. 32 / LPR - 1 summed the tile's other rows
        // over the same columns as row 0's lanes: fold their partials into
        // row 0's, in a fixed order (pairs 16 apart, then 8 apart)
#pragma unroll
        for (int d = 16; d >= LPR; d >>= 1)
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float hx = __shfl_down_sync(0xffffffffu, hi[k][q].x, d);
                    const float lx = __shfl_down_sync(0xffffffffu, lo[k][q].x, d);
                    const float hy = __shfl_down_sync(0xffffffffu, hi[k][q].y, d);
                    const float ly = __shfl_down_sync(0xffffffffu, lo[k][q].y, d);
                    comp_add(hi[k][q].x, lo[k][q].x, hx);
                    lo[k][q].x = __fadd_rn(lo[k][q].x, lx);
                    comp_add(hi[k][q].y, lo[k][q].y, hy);
                    lo[k][q].y = __fadd_rn(lo[k][q].y, ly);
                }
    }

    // ---- the CTA partial.  Every row group writes its partial to shared
    // memory ([group][comb_slot(v, q)] float4 (hi.x, lo.x, hi.y, lo.y), free
    // of bank conflicts), then every consumer thread sums whole slots over
    // the groups in group order -- slot m = 4 v + q holds columns 8 v + 2 q
    // and the next one -- so the combine is spread over the CTA instead of
    // left to one group.
    consumer_sync(L);
    float4 *comb = reinterpret_cast<float4 *>(s.ring);
    const int ncol = nvec * 8;
    const int nslot = 4 * nvec;
    const int nthr = consumer_warps * 32;
    // The row groups that owned a row of this CTA.  Every sum starts at +0
    // and round-to-nearest never turns a sum into -0, so the other groups'
    // partials are +0 and adding them changes no bit: the combine reads the
    // live groups only, in the same order (GB300: 0.8-1.2 us off a one-row
    // call at H = 1536-6144, where one group of several is live).
    const uint32_t crows = c.r_end > c.r0 ? c.r_end - c.r0 : 0u;
    const int live = max(1, min(L.groups, (int)((crows + (uint32_t)RG - 1u) / (uint32_t)RG)));
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * vstride + ltid;
        if (owner && v < nvec && gid < live)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                comb[gid * nslot + comb_slot(v, q)] = make_float4(hi[k][q].x, lo[k][q].x, hi[k][q].y, lo[k][q].y);
    }
    consumer_sync(L);
    // calls emit(m, slot) for each of this thread's slots of the CTA partial
    auto for_each_slot = [&](auto &&emit) {
        for (int m = (int)threadIdx.x; m < nslot; m += nthr)
            emit(m, slot_sum(smem_addr(comb), nvec, live, m));
    };

    if constexpr (FORM == kFormCluster) {
        // ---- cluster form: the CTA's partial goes to its own shared memory
        // (the drained ring, past the combine buffer), as float2 (hi, lo) per
        // column; thread 0 then tells every CTA of the cluster, and each CTA,
        // once all have told it, reduces its slice of the columns over the
        // cluster's partials in CTA order.
        float4 *mine = comb + L.groups * nslot;
        for_each_slot([&](int m, float4 a) { mine[m] = a; });
        consumer_sync(L);
        const uint32_t C = (uint32_t)p.cluster;
        if (threadIdx.x == 0) {
            fence_acq_rel_cluster();
            for (uint32_t r = 0; r < C; ++r)
                mbar_arrive_remote(map_to_rank(smem_addr(&cl_bar[0]), r));
        }
        // thread 0 waits (bounded) and shares the outcome, so that the whole
        // CTA either reads the partials or leaves together
        if (threadIdx.x == 0)
            s.flag[2] = mbar_wait_cluster(smem_addr(&cl_bar[0]), 0, p.wait_ns);
        consumer_sync(L);
        if (!s.flag[2]) {
            // some CTA never published its partial: read nothing remote
            if (threadIdx.x == 0)
                set_status(p.status, kStatusTimeout);
            return;
        }
        fence_acq_rel_cluster();
        const uint32_t rank = cluster_ctarank();
        const int per = (ncol + (int)C - 1) / (int)C;
        const int j0 = (int)rank * per, j1 = min(ncol, j0 + per);
        const uint32_t base = smem_addr(mine);
        for (int j = j0 + (int)threadIdx.x; j < j1; j += consumer_warps * 32) {
            // CTA order, four remote loads in flight at a time
            float h = 0.f, l = 0.f;
            for (int r0 = 0; r0 < (int)C; r0 += 4) {
                float2 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    v[u] = r0 + u < (int)C ? ld_cluster_f2(map_to_rank(base + 8u * (uint32_t)j, (uint32_t)(r0 + u)))
                                           : make_float2(0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (r0 + u < (int)C) {
                        comp_add(h, l, v[u].x);
                        l = __fadd_rn(l, v[u].y);
                    }
            }
            p.dw[j] = __fadd_rn(h, l);
        }
        // this CTA's remote reads are complete: tell every CTA, and keep this
        // CTA's shared memory until every CTA has finished reading it
        consumer_sync(L);
        if (threadIdx.x == 0) {
            for (uint32_t r = 0; r < C; ++r)
                mbar_arrive_remote(map_to_rank(smem_addr(&cl_bar[1]), r));
            if (!mbar_wait_cluster(smem_addr(&cl_bar[1]), 0, p.wait_ns))
                set_status(p.status, kStatusTimeout);
        }
        return;
    }

    if constexpr (FORM == kFormPair) {
        // the CTA partial, or for a pair of one CTA dw itself (the reduce of
        // a single partial would give the same bits, hi + lo rounded once)
        float4 *dst = reinterpret_cast<float4 *>(p.partials + (size_t)blockIdx.x * ncol);
        if constexpr (VPT >= 4 && DWM == CAKE_DWM_KAHAN)
            emit_pair_partial(smem_addr(comb), nvec, live, nthr, dst, reinterpret_cast<float2 *>(p.dw), p.direct_dw);
        else
            emit_pair_body(smem_addr(comb), nvec, live, nthr, dst, reinterpret_cast<float2 *>(p.dw), p.direct_dw);
        // the reduce may launch once every CTA has written its partial (GB300:
        // 1-2 us faster at T = 4096 than a trigger before the group combine)
        pdl_launch_dependents();
        return;
    }
    if (FORM != kFormAtomic) {
        float4 *dst = reinterpret_cast<float4 *>(p.partials + (size_t)blockIdx.x * ncol);
        for_each_slot([&](int m, float4 a) { dst[m] = a; });
        if (FORM == kFormGrid) {
            // ---- cooperative form: every CTA's partial is written; after
            // the grid barrier CTA b reduces columns [b*C, (b+1)*C), one
            // column per warp at a time: lane l sums the partials of CTAs
            // [l*per, (l+1)*per) in ascending order (compensated), then the
            // 32 lane sums merge in a butterfly whose every step is
            // symmetric, so the result is the same on every lane and run.
            consumer_sync(L);
            if (threadIdx.x == 0)
                s.flag[1] = grid_barrier(p.grid_cnt, p.grid_gen, gridDim.x + (uint32_t)p.grid_extra, p.wait_ns);
            consumer_sync(L);
            if (!s.flag[1]) {
                if (threadIdx.x == 0)
                    set_status(p.status, kStatusTimeout);
                return;
            }
            const int P = (int)gridDim.x;
            const int C = (ncol + P - 1) / P;
            const int c0 = (int)blockIdx.x * C, c1 = min(ncol, c0 + C);
            const int per = (P + 31) / 32;
            const int q0 = lane * per, q1 = min(P, q0 + per);
            for (int j = c0 + warp; j < c1; j += consumer_warps) {
                float h = 0.f, l = 0.f;
                for (int q = q0; q < q1; q += 4) {
                    float2 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        v[u] = q + u < q1 ? __ldcg(p.partials + (size_t)(q + u) * ncol + j) : make_float2(0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        comp_add(h, l, v[u].x);
                        l = __fadd_rn(l, v[u].y);
                    }
                }
#pragma unroll
                for (int o = 1; o < 32; o <<= 1)
                    comp_merge(h, l, __shfl_xor_sync(0xffffffffu, h, o), __shfl_xor_sync(0xffffffffu, l, o));
                if (lane == 0)
                    p.dw[j] = __fadd_rn(h, l);
            }
            return;
        }
        // ---- one-kernel fixed-order reduce: the last CTA to arrive among
        // the kTreeGroup CTAs of its group sums their partials in CTA order
        // into the group's total; the last group to finish sums the group
        // totals in group order.  Nobody waits; the arithmetic order does not
        // depend on who arrives last.
        __threadfence();
        consumer_sync(L);
        const int grp = blockIdx.x / kTreeGroup;
        const int ngroups = (gridDim.x + kTreeGroup - 1) / kTreeGroup;
        if (threadIdx.x == 0) {
            const int n_g = min(kTreeGroup, (int)gridDim.x - grp * kTreeGroup);
            const unsigned prev = atomicAdd(p.tree_cnt + 1 + grp, 1u);
            s.flag[1] = (prev == (unsigned)n_g - 1);
        }
        consumer_sync(L);
        if (!s.flag[1])
            return;
        __threadfence();
        const int nthr = consumer_warps * 32;
        const int p0 = grp * kTreeGroup, p1 = min((int)gridDim.x, p0 + kTreeGroup);
        for (int j = threadIdx.x; j < ncol; j += nthr) {
            float2 v[kTreeGroup];
#pragma unroll
            for (int u = 0; u < kTreeGroup; ++u)
                v[u] = p0 + u < p1 ? __ldcg(p.partials + (size_t)(p0 + u) * ncol + j) : make_float2(0.f, 0.f);
            float h = 0.f, l = 0.f;
#pragma unroll
            for (int u = 0; u < kTreeGroup; ++u) {
                comp_add(h, l, v[u].x);
                l = __fadd_rn(l, v[u].y);
            }
            p.group_totals[(size_t)grp * ncol + j] = make_float2(h, l);
        }
        __threadfence();
        consumer_sync(L);
        if (threadIdx.x == 0) {
            atomicExch(p.tree_cnt + 1 + grp, 0u);
            const unsigned prev = atomicAdd(p.tree_cnt, 1u);
            s.flag[2] = (prev == (unsigned)ngroups - 1);
        }
        consumer_sync(L);
        if (!s.flag[2])
            return;
        __threadfence();
        for (int j = threadIdx.x; j < ncol; j += nthr) {
            float h = 0.f, l = 0.f;
            for (int g2 = 0; g2 < ngroups; ++g2) {
                const float2 v = __ldcg(p.group_totals + (size_t)g2 * ncol + j);
                comp_add(h, l, v.x);
                l = __fadd_rn(l, v.y);
            }
            p.dw[j] = __fadd_rn(h, l);
        }
        if (threadIdx.x == 0)
            atomicExch(p.tree_cnt, 0u);
        return;
    }

    // ---- single kernel: FP64 column accumulation into one of `banks` copies
    // of the accumulators (CTA b adds into bank b % banks, which spreads the
    // L2 atomics); the last CTA to arrive sums the banks and finalises
    {
        double *acc = p.acc + (size_t)(blockIdx.x % p.banks) * ncol;
        for_each_slot([&](int m, float4 a) {
            atomicAdd(acc + 2 * m, (double)a.x + (double)a.y);
            atomicAdd(acc + 2 * m + 1, (double)a.z + (double)a.w);
        });
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
            // every bank's load issued before the sum (banks in ascending order)
            double v[kMaxAccBanks];
#pragma unroll
            for (int b = 0; b < kMaxAccBanks; ++b)
                v[b] = b < p.banks ? __ldcg(p.acc + (size_t)b * ncol + j) : 0.0;
            double sum = 0.0;
#pragma unroll
            for (int b = 0; b < kMaxAccBanks; ++b)
                if (b < p.banks) {
                    sum += v[b];
                    p.acc[(size_t)b * ncol + j] = 0.0;
                }
            p.dw[j] = (float)sum;
        }
        if (threadIdx.x == 0)
            atomicExch(p.arrivals, 0u);
    }
}

// The row kernels, by row build RB: 0 one row per group; 1 two rows per
// group (one group of up to 16 warps and the producer per CTA), keeping x and
// dy*w of both rows in registers; 4 one row per group for rows of one warp
// (H <= 256), with that width known to the compiler; rows of part of a warp:
// 5 (VPT = 2) and 6 (VPT = 1) half a warp, two rows per warp; 7 (VPT = 1)
// and 8 (VPT = 2) a quarter, four rows per warp; 9 (VPT = 2) an eighth,
// eight rows per warp.  The bounds cap the registers a thread may use
// so that the largest CTA fits: 72 (26 warps), 96 (17 warps), 128 (13 warps).
template <int VPT, int DWM, int FORM, int RB>
__global__ void __launch_bounds__(RB == 1 ? kMaxThreadsR2 : kMaxThreadsFor(VPT), 1)
    bwd_rows_kernel(const __grid_constant__ BwdParams p)
{
    bwd_rows<VPT, DWM, FORM, RB == 1 ? 2 : 1, true, RB == 4 || RB >= 5,
             RB == 5 || RB == 6 ? 16 : RB == 7 || RB == 8 ? 8 : RB == 9 ? 4 : 32>(p);
}

// ------------------------------------------------------------------ launch

template <int VPT, int DWM, int FORM, int RB>
static cudaError_t launch_rows(const BwdParams &p, int ctas, size_t smem, cudaStream_t stream)
{
    const int threads = 32 * (p.L.groups * p.L.warps_per_row + 1);
    auto kern = bwd_rows_kernel<VPT, DWM, FORM, RB>;
    cudaError_t e = ensure_smem_attr((const void *)kern, smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // the grid form's CTAs wait for one another: the launch must guarantee
    // that they are all resident at once (it fails otherwise); the cluster
    // form is one cluster of all its CTAs, co-scheduled by the hardware
    cudaLaunchAttribute attr[1];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (FORM == kFormGrid) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.numAttrs = 1;
    }
    if (FORM == kFormCluster) {
        if (p.cluster < 1 || p.cluster > kMaxCluster || ctas != p.cluster)
            return cudaErrorInvalidValue;
        if (p.cluster > 8) {
            e = cudaFuncSetAttribute((const void *)kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess)
                return e;
        }
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)p.cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
        // refuse a cluster the device cannot hold rather than launch it
        int nclusters = 0;
        e = cudaOccupancyMaxActiveClusters(&nclusters, (const void *)kern, &cfg);
        if (e != cudaSuccess)
            return e;
        if (nclusters < 1)
            return cudaErrorInvalidConfiguration;
    }
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <int VPT, int FORM, int RB>
static cudaError_t launch_dwm(const BwdParams &p, int dwm, int ctas, size_t smem, cudaStream_t stream)
{
    if (dwm == 0) return launch_rows<VPT, 0, FORM, RB>(p, ctas, smem, stream);
    if (dwm == 1) return launch_rows<VPT, 1, FORM, RB>(p, ctas, smem, stream);
    if (dwm == 2) return launch_rows<VPT, 2, FORM, RB>(p, ctas, smem, stream);
    return launch_rows<VPT, 3, FORM, RB>(p, ctas, smem, stream);
}

template <int VPT, int DWM, int FORM, int RB>
static cudaError_t occ_rows(int threads, size_t smem, int *n)
{
    const void *kern = (const void *)bwd_rows_kernel<VPT, DWM, FORM, RB>;
    cudaError_t e = ensure_smem_attr(kern, smem);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, threads, smem);
}

template <int VPT, int FORM, int RB>
static cudaError_t occ_dwm(int dwm, int threads, size_t smem, int *n)
{
    if (dwm == 0) return occ_rows<VPT, 0, FORM, RB>(threads, smem, n);
    if (dwm == 1) return occ_rows<VPT, 1, FORM, RB>(threads, smem, n);
    if (dwm == 2) return occ_rows<VPT, 2, FORM, RB>(threads, smem, n);
    return occ_rows<VPT, 3, FORM, RB>(threads, smem, n);
}

// One form's launcher and occupancy query over the row builds it is compiled
// for: (VPT, RB) = (1, 0), (1, 1), (1, 4), (1, 6), (1, 7), (2, 0), (2, 5),
// (3, 0), (4, 0); the tree form only (1, 0), which also serves rows of one
// warp, (1, 6), (1, 7), (2, 0) and (2, 5).
template <int FORM>
cudaError_t launch_bwd_form(const BwdParams &p, int vpt, int rb, int dwm, int ctas, size_t smem,
                            cudaStream_t stream)
{
    if (vpt == 2 && rb == 5) return launch_dwm<2, FORM, 5>(p, dwm, ctas, smem, stream);
    if (vpt == 1 && rb == 6) return launch_dwm<1, FORM, 6>(p, dwm, ctas, smem, stream);
    if (vpt == 1 && rb == 7) return launch_dwm<1, FORM, 7>(p, dwm, ctas, smem, stream);
    if (vpt == 2 && rb == 8) return launch_dwm<2, FORM, 8>(p, dwm, ctas, smem, stream);
    if (vpt == 2 && rb == 9) return launch_dwm<2, FORM, 9>(p, dwm, ctas, smem, stream);
    if constexpr (FORM == kFormTree) {
        if (vpt == 2 && rb == 0) return launch_dwm<2, FORM, 0>(p, dwm, ctas, smem, stream);
        return vpt == 1 && rb != 1 ? launch_dwm<1, FORM, 0>(p, dwm, ctas, smem, stream) : cudaErrorInvalidValue;
    } else {
        if (vpt == 1 && rb == 1) return launch_dwm<1, FORM, 1>(p, dwm, ctas, smem, stream);
        if (vpt == 1 && rb == 4) return launch_dwm<1, FORM, 4>(p, dwm, ctas, smem, stream);
        if (rb != 0) return cudaErrorInvalidValue;
        switch (vpt) {
        case 1: return launch_dwm<1, FORM, 0>(p, dwm, ctas, smem, stream);
        case 2: return launch_dwm<2, FORM, 0>(p, dwm, ctas, smem, stream);
        case 3: return launch_dwm<3, FORM, 0>(p, dwm, ctas, smem, stream);
        case 4: return launch_dwm<4, FORM, 0>(p, dwm, ctas, smem, stream);
        default: return cudaErrorInvalidValue;
        }
    }
}

template <int FORM>
cudaError_t occ_bwd_form(int vpt, int rb, int dwm, int threads, size_t smem, int *n)
{
    if (vpt == 2 && rb == 5) return occ_dwm<2, FORM, 5>(dwm, threads, smem, n);
    if (vpt == 1 && rb == 6) return occ_dwm<1, FORM, 6>(dwm, threads, smem, n);
    if (vpt == 1 && rb == 7) return occ_dwm<1, FORM, 7>(dwm, threads, smem, n);
    if (vpt == 2 && rb == 8) return occ_dwm<2, FORM, 8>(dwm, threads, smem, n);
    if (vpt == 2 && rb == 9) return occ_dwm<2, FORM, 9>(dwm, threads, smem, n);
    if constexpr (FORM == kFormTree) {
        if (vpt == 2 && rb == 0) return occ_dwm<2, FORM, 0>(dwm, threads, smem, n);
        return vpt == 1 && rb != 1 ? occ_dwm<1, FORM, 0>(dwm, threads, smem, n) : cudaErrorInvalidValue;
    } else {
        if (vpt == 1 && rb == 1) return occ_dwm<1, FORM, 1>(dwm, threads, smem, n);
        if (vpt == 1 && rb == 4) return occ_dwm<1, FORM, 4>(dwm, threads, smem, n);
        if (rb != 0) return cudaErrorInvalidValue;
        switch (vpt) {
        case 1: return occ_dwm<1, FORM, 0>(dwm, threads, smem, n);
        case 2: return occ_dwm<2, FORM, 0>(dwm, threads, smem, n);
        case 3: return occ_dwm<3, FORM, 0>(dwm, threads, smem, n);
        case 4: return occ_dwm<4, FORM, 0>(dwm, threads, smem, n);
        default: return cudaErrorInvalidValue;
        }
    }
}

#define CAKE_BWD_FORM_DECL(F)                                                                            \
    extern template cudaError_t launch_bwd_form<F>(const BwdParams &, int, int, int, int, size_t, cudaStream_t); \
    extern template cudaError_t occ_bwd_form<F>(int, int, int, int, size_t, int *);
CAKE_BWD_FORM_DECL(kFormPair)
CAKE_BWD_FORM_DECL(kFormAtomic)
CAKE_BWD_FORM_DECL(kFormTree)
CAKE_BWD_FORM_DECL(kFormGrid)
CAKE_BWD_FORM_DECL(kFormCluster)
#undef CAKE_BWD_FORM_DECL

} // namespace cake
