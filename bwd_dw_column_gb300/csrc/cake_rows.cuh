// cake_rows.cuh -- the row pipeline shared by the forward and backward kernels.
//
// CTA organisation (all kernels of this library that stream rows):
//   * warps [0, groups*W) are consumers; a "row group" of W warps owns one row
//     at a time, each thread holding VPT 16-byte vectors of that row in
//     registers (vector v = k*32*W + thread-in-group, k < VPT);
//   * the last warp is the producer: it streams the CTA's contiguous chunk of
//     rows into a `stages`-deep shared-memory ring with cp.async.bulk copies
//     (one per row, or one per stage when the rows are dense) that complete on
//     the stage's `full` mbarrier; consumers release a stage on its `empty`
//     mbarrier (one arrival per consumer warp);
//   * the per-row reductions (sum of squares, sum of g*xhat) are a warp
//     butterfly plus, when W > 1, a fixed-order sum of the W warp partials
//     through shared memory behind one named barrier per row.
// No CTA ever waits on another CTA.  Every mbarrier wait is bounded
// (the launch's wait_ns); a wait that runs out sets the status word to
// CAKE_ERR_TIMEOUT and the CTA leaves its loop after draining its own copies.
#pragma once

#include "cake_device.cuh"

namespace cake {

constexpr int kStatusTimeout = 5; // == CAKE_ERR_TIMEOUT

struct Smem {
    uint64_t *full;   // [stages]
    uint64_t *empty;  // [stages]
    float *red;       // [groups][2][R2][W] (groups * W * R2 <= 50: 400 bytes)
    int *flag;        // [4]
    float *wsm;       // [H] the weight as FP32, staged once per CTA
    float4 *lo;       // blocked dw sums: [2 or 4 * VPT][consumer threads] compensated pairs
    uint8_t *ring;    // stages * stage_bytes
    uint32_t stage_bytes;
    uint32_t tens_bytes; // bytes of one tensor in one stage
};

__device__ __forceinline__ Smem carve_smem(uint8_t *base, const Layout &L)
{
    Smem s;
    s.full = reinterpret_cast<uint64_t *>(base);
    s.empty = s.full + L.stages;
    s.red = reinterpret_cast<float *>(base + 16 * 2 * 8); // 256 B of barriers first
    s.flag = reinterpret_cast<int *>(base + kMiscBytes - 16);
    s.wsm = reinterpret_cast<float *>(base + kMiscBytes);
    s.lo = reinterpret_cast<float4 *>(base + kMiscBytes + weight_smem_bytes(L.H));
    s.ring = base + kMiscBytes + weight_smem_bytes(L.H) + L.lo_bytes;
    s.tens_bytes = (uint32_t)L.groups * L.rows_per_group * L.H * 2;
    s.stage_bytes = s.tens_bytes * L.ntens;
    return s;
}

// Thread 0 initialises the ring's barriers; everyone syncs once.
__device__ __forceinline__ void init_ring(const Smem &s, const Layout &L)
{
    if (threadIdx.x == 0) {
        const int consumer_warps = L.groups * L.warps_per_row;
        for (int i = 0; i < L.stages; ++i) {
            mbar_init(smem_addr(&s.full[i]), 1);
            mbar_init(smem_addr(&s.empty[i]), consumer_warps);
        }
        s.flag[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
}

struct Chunk {
    uint32_t r0, r_end, ntiles, tile_rows;
};

__device__ __forceinline__ Chunk cta_chunk(const Layout &L)
{
    Chunk c;
    c.r0 = blockIdx.x * L.rows_per_cta;
    uint32_t e = c.r0 + L.rows_per_cta;
    c.r_end = e < L.rows ? e : L.rows;
    c.tile_rows = (uint32_t)L.groups * L.rows_per_group;
    c.ntiles = c.r_end > c.r0 ? (c.r_end - c.r0 + c.tile_rows - 1) / c.tile_rows : 0;
    return c;
}

// Producer warp: stream `ntens` tensors of the chunk into the ring.
// views[i] is the i-th staged tensor.  Returns false on a timeout.
template <int NT>
__device__ __forceinline__ void produce(const Smem &s, const Layout &L, const Chunk &c,
                                       const RowView (&views)[NT], int ntens, int *status, uint64_t wait_ns)
{
    const int lane = threadIdx.x & 31;
    const uint64_t pol = policy_evict_first();
    const uint32_t row_bytes = (uint32_t)L.H * 2;
    bool ok = true;
    uint32_t it = 0;
    uint32_t st = 0, ph = 0; // ring slot of tile `it` and the parity of its round
    for (; it < c.ntiles; ++it) {
        if (it >= (uint32_t)L.stages) {
            // the previous round of this slot was released by the consumers
            bool got = mbar_wait(smem_addr(&s.empty[st]), ph ^ 1u, wait_ns);
            got = __all_sync(0xffffffffu, got);
            if (!got) {
                if (lane == 0)
                    set_status(status, kStatusTimeout);
                ok = false;
                break;
            }
        }
        const uint32_t row0 = c.r0 + it * c.tile_rows;
        const uint32_t left = c.r_end - row0;
        const uint32_t n = left < c.tile_rows ? left : c.tile_rows;
        const uint32_t full_bar = smem_addr(&s.full[st]);
        if (lane == 0)
            mbar_arrive_expect_tx(full_bar, (uint32_t)ntens * n * row_bytes);
        __syncwarp();
        const uint32_t stage_base = smem_addr(s.ring) + st * s.stage_bytes;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t >= ntens)
                break;
            const RowView &v = views[t];
            const uint32_t dst = stage_base + t * s.tens_bytes;
            if (v.dense) {
                if (lane == 0)
                    bulk_g2s(dst, v.base + (int64_t)row0 * v.row_stride, n * row_bytes, full_bar, pol);
            } else {
                for (uint32_t q = lane; q < n; q += 32)
                    bulk_g2s(dst + q * row_bytes, v.base + row_off(v, row0 + q, L.nh), row_bytes,
                             full_bar, pol);
            }
        }
        if (++st == (uint32_t)L.stages) {
            st = 0;
            ph ^= 1u;
        }
    }
    // Never leave copies in flight: wait (bounded) for the last issued stages.
    const uint32_t issued = it;
    const uint32_t first = issued > (uint32_t)L.stages ? issued - L.stages : 0;
    for (uint32_t j = first; j < issued; ++j) {
        if (!mbar_wait(smem_addr(&s.full[j % L.stages]), (j / L.stages) & 1, wait_ns)) {
            if (lane == 0)
                set_status(status, kStatusTimeout);
        }
    }
    (void)ok;
}

// Per-row group reduction: a warp butterfly, then (W > 1) lane i of every
// warp of the group reads warp i's partial and a second butterfly sums them
// (zeros past W), so every warp of the group ends with the same value in the
// same fixed order.  `abort` is OR-ed across the group.  `slot` toggles per
// row, so one barrier per row suffices.
__device__ __forceinline__ float group_sum(float v, const Smem &s, const Layout &L, int gid,
                                           int wig, int lane, uint32_t slot, bool &abort)
{
    v = warp_sum(v);
    const int W = L.warps_per_row;
    if (W == 1) {
        abort = __any_sync(0xffffffffu, abort);
        return v;
    }
    float *red = s.red + (gid * 2 + (slot & 1)) * W;
    if (lane == 0)
        red[wig] = v;
    abort = named_sync_or(1 + gid, 32 * W, abort);
    return warp_sum(lane < W ? red[lane] : 0.f);
}

// group_sum for N rows at once: the N butterflies interleave, and with
// W > 1 one barrier serves all N rows.  Same order per row as group_sum.
template <int N, int WC = 0>
__device__ __forceinline__ void group_sum_n(const float (&v)[N], float (&out)[N], const Smem &s,
                                            const Layout &L, int gid, int wig, int lane, uint32_t slot,
                                            bool &abort)
{
#pragma unroll
    for (int n = 0; n < N; ++n)
        out[n] = v[n];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int n = 0; n < N; ++n)
            out[n] += __shfl_xor_sync(0xffffffffu, out[n], o);
    const int W = WC ? WC : L.warps_per_row; // WC: rows of WC warps known at compile time
    if (W == 1) {
        abort = __any_sync(0xffffffffu, abort);
        return;
    }
    float *red = s.red + (gid * 2 + (slot & 1)) * W * N;
    if (lane == 0)
#pragma unroll
        for (int n = 0; n < N; ++n)
            red[n * W + wig] = out[n];
    abort = named_sync_or(1 + gid, 32 * W, abort);
#pragma unroll
    for (int n = 0; n < N; ++n)
        out[n] = lane < W ? red[n * W + lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int n = 0; n < N; ++n)
            out[n] += __shfl_xor_sync(0xffffffffu, out[n], o);
}

__device__ __forceinline__ void consumer_sync(const Layout &L)
{
    named_sync(kConsumerBarrier, 32 * L.groups * L.warps_per_row);
}

// Consumer threads stage w (BF16 or FP32) into shared memory as FP32, then
// sync among themselves; the producer warp does not take part.  Two planes:
// plane 0 holds columns 0-3 of every 8-column vector, plane 1 columns 4-7, so
// that a warp reading its vectors' weights with 16-byte loads touches
// consecutive addresses (no bank conflicts).
template <bool VEC = true>
__device__ __forceinline__ void stage_weight(const Smem &s, const Layout &L, const void *w, int w_f32)
{
    const int nthr = 32 * L.groups * L.warps_per_row;
    if (!VEC) { // one element per thread and round
        const int half = L.nvec * 4;
        for (int j = threadIdx.x; j < L.H; j += nthr) {
            const float v = w_f32 ? static_cast<const float *>(w)[j]
                                  : __uint_as_float((uint32_t)static_cast<const uint16_t *>(w)[j] << 16);
            const int vec = j >> 3, e = j & 7;
            s.wsm[(e >> 2) * half + vec * 4 + (e & 3)] = v;
        }
        consumer_sync(L);
        return;
    }
    // One 16-byte vector of w (8 BF16) or two (8 FP32) per consumer thread
    // and round, all loads of a round issued before its stores (w is 16-byte
    // aligned: the host checks it).
    constexpr int U = 2;
    float4 *wsm = reinterpret_cast<float4 *>(s.wsm);
    for (int v0 = threadIdx.x; v0 < L.nvec; v0 += U * nthr) {
        float4 a[U], b[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * nthr;
            if (v < L.nvec) {
                if (w_f32) {
                    a[u] = __ldg(static_cast<const float4 *>(w) + 2 * v);
                    b[u] = __ldg(static_cast<const float4 *>(w) + 2 * v + 1);
                } else {
                    const uint4 r = __ldg(static_cast<const uint4 *>(w) + v);
                    a[u] = make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
                    b[u] = make_float4(__uint_as_float(r.z << 16), __uint_as_float(r.z & 0xffff0000u),
                                       __uint_as_float(r.w << 16), __uint_as_float(r.w & 0xffff0000u));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * nthr;
            if (v < L.nvec) {
                wsm[v] = a[u];
                wsm[L.nvec + v] = b[u];
            }
        }
    }
    consumer_sync(L);
}

// The 8 weights of vector v as four FP32 pairs.
__device__ __forceinline__ void weight_pairs(const Smem &s, const Layout &L, int v, float2 (&w2)[4])
{
    const float4 a = reinterpret_cast<const float4 *>(s.wsm)[v];
    const float4 b = reinterpret_cast<const float4 *>(s.wsm)[L.nvec + v];
    w2[0] = make_float2(a.x, a.y);
    w2[1] = make_float2(a.z, a.w);
    w2[2] = make_float2(b.x, b.y);
    w2[3] = make_float2(b.z, b.w);
}

__device__ __forceinline__ int64_t out_off(int64_t st, int64_t sh, int64_t row_stride, int uniform,
                                           uint32_t r, uint32_t nh)
{
    if (uniform)
        return (int64_t)r * row_stride;
    const uint32_t t = r / nh, k = r - t * nh;
    return (int64_t)t * st + (int64_t)k * sh;
}

} // namespace cake
