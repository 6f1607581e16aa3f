// cake_device.cuh -- sm_103a building blocks shared by the forward and
// backward kernels: mbarrier + bulk-copy (TMA) staging, bounded waits, BF16
// packing, group reductions and compensated sums.  Hand-written PTX.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "cake_params.h"

namespace cake {

// ----------------------------------------------------------------- timing

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One bounded test of a phase: a thread whose phase is not complete may be
// suspended by the hardware until it completes or the hint (ns) runs out, so
// waiting warps do not spin on the issue slots.
constexpr uint32_t kSuspendHintNs = 1000000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if it
// has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 3u) == 0 && globaltimer_ns() - t0 > limit_ns)
            return false;
    }
}

// ------------------------------------------------- thread-block clusters

// This CTA's rank within its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster (a hardware barrier: all threads
// reach it unconditionally at kernel start, before any can leave).
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same shared-memory location in CTA
// `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem), "r"(rank));
    return r;
}

__device__ __forceinline__ void fence_acq_rel_cluster()
{
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// Arrive on an mbarrier of another CTA of the cluster, releasing this
// thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// A non-blocking test (no suspension): the cluster form's waits are short
// and a suspended waiter on a remotely completed phase measured slow.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for a phase whose arrivals come from other CTAs of the cluster
// (acquiring their writes at cluster scope).  False after limit_ns.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        __nanosleep(32);
        if ((i & 15u) == 0 && globaltimer_ns() - t0 > limit_ns)
            return false;
    }
}

// Load a float4 from this CTA's shared memory.  Volatile, so that a batch of
// them is issued in program order after the barrier before it, and in flight
// together until their values are used.
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// Load a float2 from another CTA's shared memory (distributed shared memory).
__device__ __forceinline__ float2 ld_cluster_f2(uint32_t cluster_addr)
{
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(cluster_addr) : "memory");
    return v;
}

// -------------------------------------------------------- bulk copies (TMA)

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Global -> shared bulk copy completing on an mbarrier.  Both addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ------------------------------------------------- programmatic dependent launch

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------- named barriers

__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("barrier.sync.aligned %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_sync_or(int id, int threads, bool pred)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.red.or.pred.aligned po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)pred), "r"(id), "r"(threads)
        : "memory");
    return out != 0;
}

// -------------------------------------------------------------- BF16 packing

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Round two FP32 values to BF16 (nearest, ties to even) and pack (lo, hi).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Unpack one 16-byte vector of 8 BF16 values.
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8])
{
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                      pack_bf16(f[6], f[7]));
}

// ------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Error-free transformation: s + e == a + b exactly (Knuth's TwoSum; no
// ordering precondition on |a|, |b|).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    float bp = __fsub_rn(s, a);
    float ap = __fsub_rn(s, bp);
    e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// (hi, lo) += v, keeping hi + lo as the compensated sum.
__device__ __forceinline__ void comp_add(float &hi, float &lo, float v)
{
    float s, e;
    two_sum(hi, v, s, e);
    hi = s;
    lo = __fadd_rn(lo, e);
}

// --------------------------------------------------------- row addressing

// GPU-scope loads for a flag other CTAs publish.
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier of one thread per CTA (all CTAs co-resident: a
// cooperative launch).  cnt counts arrivals; the CTA whose arrival makes
// `target` resets it and advances gen, which the others wait on (target is
// the CTA count; a larger one never completes, which is how the timeout test
// makes this wait run out).  Before it the caller's CTA has synchronised, so
// the fence + add publishes the whole CTA's writes (a release; the acquire
// loads / fence make the other CTAs' writes visible to this CTA after its
// next barrier).  Returns false if gen has not moved within limit_ns.
__device__ __forceinline__ bool grid_barrier(uint32_t *cnt, uint32_t *gen, uint32_t target, uint64_t limit_ns)
{
    const uint32_t g0 = ld_relaxed_gpu(gen);
    __threadfence();
    if (atomicAdd(cnt, 1u) == target - 1) {
        atomicExch(cnt, 0u);
        __threadfence();
        atomicAdd(gen, 1u);
        return true;
    }
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ld_acquire_gpu(gen) != g0)
            return true;
        __nanosleep(64);
        if ((i & 15u) == 0 && globaltimer_ns() - t0 > limit_ns)
            return false;
    }
}

// (h, l) + (h2, l2) as a compensated pair, symmetric in its two operands
// (the result does not depend on their order).
__device__ __forceinline__ void comp_merge(float &h, float &l, float h2, float l2)
{
    float s, e;
    two_sum(h, h2, s, e);
    l = __fadd_rn(__fadd_rn(l, l2), e);
    h = s;
}

// Element offset of row r in a [T, nh, H] view.
__device__ __forceinline__ int64_t row_off(const RowView &v, uint32_t r, uint32_t nh)
{
    if (v.uniform)
        return (int64_t)r * v.row_stride;
    const uint32_t t = r / nh, k = r - t * nh;
    return (int64_t)t * v.st + (int64_t)k * v.sh;
}

__device__ __forceinline__ void set_status(int *status, int code)
{
    atomicExch(status, code);
}

}  // namespace cake

namespace cake {

// ------------------------------------------------------ packed FP32 pairs
// sm_100-family packed FP32 arithmetic (PTX add/sub/mul/fma .rn.f32x2):
// one instruction operates on two FP32 values held in a 64-bit register,
// each rounded to nearest even exactly as the scalar instruction would.

__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// a * b + c with one rounding per lane
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// BF16 pair (one 32-bit word: element 2i in the low half) -> FP32 pair.
__device__ __forceinline__ float2 bf2(uint32_t u) { return make_float2(bf16lo(u), bf16hi(u)); }

// FP32 pair -> BF16 pair, round to nearest even.
__device__ __forceinline__ uint32_t pack2(float2 v) { return pack_bf16(v.x, v.y); }

__device__ __forceinline__ uint32_t word(const uint4 &v, int q)
{
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// TwoSum on pairs: (s, e) with s + e == a + b exactly, lane by lane.
__device__ __forceinline__ void two_sum2(float2 a, float2 b, float2 &s, float2 &e)
{
    s = add2(a, b);
    const float2 bp = sub2(s, a);
    const float2 ap = sub2(s, bp);
    e = add2(sub2(a, ap), sub2(b, bp));
}

} // namespace cake
