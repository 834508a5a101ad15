// ptx.cuh -- thin inline-PTX wrappers used by the verify kernels (sm_103a):
// bulk (TMA) copies with mbarrier completion, thread-block-cluster barriers
// and distributed shared memory, packed bf16x2 / f32x2 arithmetic and the
// hardware base-2 exponential.
#pragma once
#include <cstdint>

namespace specv {

// ------------------------------------------------------------------ addresses
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Plain arrival (one count) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrival counting `count` at once.
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}

// try_wait with an explicit bound on how long the thread may be suspended
// (nanoseconds) before it polls again.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t phase, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(phase), "r"(ns)
        : "memory");
    return ok != 0;
}

// Non-blocking tests of a phase (mbarrier.test_wait never suspends the
// thread, unlike try_wait): for a loop that polls several things in turn.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}

// The same with acquire at cluster scope: once it returns true, what other
// CTAs of the cluster stored before their (release) arrivals on `bar` is
// visible to the calling thread.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}

// Nanoseconds of the global timer.
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// No wait in these kernels takes more than this (a correct call runs for
// microseconds); past it a wait gives up and the row reports a timeout.
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;

// Bounded wait on an mbarrier phase: gives up after `limit` polls or kWaitNs
// of wall-clock time, whichever comes first (each poll may itself suspend the
// thread for about a microsecond), and returns false, so that a lost
// completion ends the kernel with an error status instead of a hang.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t phase, uint32_t limit) {
    unsigned long long t0 = 0;
    for (uint32_t it = 0; it < limit; ++it) {
        if (mbar_try_wait(bar, phase)) return true;
        if ((it & 255) == 255) {
            const unsigned long long t = gtimer();
            if (t0 == 0)
                t0 = t;
            else if (t - t0 > kWaitNs)
                return false;
        }
    }
    return false;
}

// 1-D bulk copy global -> shared of this CTA, completion counted in bytes on
// `bar`.  src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Full cluster barrier with release/acquire semantics on shared memory of
// every CTA of the cluster (a hardware barrier: no polling loop).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of a cluster barrier (release on arrive, acquire on wait),
// for work between them.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ double ld_cluster_f64(uint32_t addr) {
    double v;
    asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t r;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
    return r;
}

// Stores into the shared memory of another CTA of the cluster (visible to
// it after the next cluster barrier); they do not wait for a reply.
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// A 16-byte store into the shared memory of a CTA of the cluster whose
// completion is counted, in bytes, on an mbarrier of that CTA (both
// addresses shared::cluster): the sender does not wait for it, and a thread
// that sees the barrier's phase complete sees the data.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
                 "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Named barrier 1 over the first 128 threads of the CTA (the consumer warps).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// ------------------------------------------------------------------ loads
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ unsigned short ld_shared_u16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// Streaming 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------------------ arithmetic
// 2^x on the special-function unit (relative error a few ulp; flushes
// subnormal results to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16x2 maximum (a NaN operand yields the other operand).
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bf16x2 maximum that propagates NaN.
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float max_nan_f32(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Maximum over the 32 lanes of a converged warp, in one instruction (NaN
// inputs are ignored unless every input is NaN).
__device__ __forceinline__ float warp_max_f32(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Packed pairs of fp32 (sm_100+ f32x2 instructions: one issue, two lanes).
struct f2 {
    unsigned long long v;
};

__device__ __forceinline__ f2 pack2(float a, float b) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void unpack2(f2 p, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(p.v));
}

__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
}

// a * b + c, one rounding per lane.
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
}

// ------------------------------------------------------------------ error-free sums
// Knuth's two-sum: s + e == a + b exactly (round to nearest).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) += (a_hi, a_lo) for unevaluated float pairs.
__device__ __forceinline__ void df_add(float& hi, float& lo, float a_hi, float a_lo) {
    float s, e;
    two_sum(hi, a_hi, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, a_lo));
}

// Unevaluated pairs of floats ("double-float"): value = hi + lo, |lo| small.
// All sums and comparisons of the stop-row weights use them: the GB300's
// float64 units are far too slow for the critical path.
struct df {
    float hi, lo;
};

__device__ __forceinline__ df df_make(float h, float l = 0.0f) { return df{h, l}; }

__device__ __forceinline__ df df_sum(df a, df b) {
    df r = a;
    df_add(r.hi, r.lo, b.hi, b.lo);
    return r;
}

__device__ __forceinline__ df df_neg(df a) { return df{-a.hi, -a.lo}; }

// a * b for a float b: exact product of the high parts plus the low part.
__device__ __forceinline__ df df_mul_f(df a, float b) {
    const float p = a.hi * b;
    const float e = fmaf(a.hi, b, -p);
    return df{p, fmaf(a.lo, b, e)};
}

// sign of a - b as -1, 0, +1 (to the pairs' precision)
__device__ __forceinline__ bool df_less(df a, df b) {
    float s, e;
    two_sum(a.hi, -b.hi, s, e);
    return s + (e + (a.lo - b.lo)) < 0.0f;
}

__device__ __forceinline__ float df_val(df a) { return a.hi + a.lo; }

__device__ __forceinline__ df df_shfl_up(df a, int off) {
    return df{__shfl_up_sync(0xffffffffu, a.hi, off), __shfl_up_sync(0xffffffffu, a.lo, off)};
}

__device__ __forceinline__ df df_shfl_down(df a, int off) {
    return df{__shfl_down_sync(0xffffffffu, a.hi, off), __shfl_down_sync(0xffffffffu, a.lo, off)};
}

__device__ __forceinline__ df df_shfl(df a, int src) {
    return df{__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}

// Warp-wide inclusive prefix sum of pairs, lane order.
__device__ __forceinline__ df df_warp_incl_scan(df v, int lane) {
    for (int off = 1; off < 32; off <<= 1) {
        const df o = df_shfl_up(v, off);
        if (lane >= off) v = df_sum(o, v);
    }
    return v;
}

// Warp-wide total of pairs (valid in lane 0), fixed tree order.
__device__ __forceinline__ df df_warp_total(df v) {
    for (int off = 16; off > 0; off >>= 1) v = df_sum(v, df_shfl_down(v, off));
    return v;
}

// log2(e) / T as a pair: the quotient of the high part of log2(e), its
// exact remainder (one fma), and the low part of log2(e).
__device__ __forceinline__ df log2e_over(float T) {
    const float l2e_hi = 1.44269502162933349609375f;  // float(log2 e)
    const float l2e_lo = 1.9259629911266175e-8f;     // log2 e - l2e_hi
    const float qh = l2e_hi / T;
    const float rem = fmaf(-qh, T, l2e_hi);
    const float ql = (rem + l2e_lo) / T;
    float h, l;
    two_sum(qh, ql, h, l);
    return df{h, l};
}

}  // namespace specv
