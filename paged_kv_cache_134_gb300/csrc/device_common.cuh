// Device-side helpers shared by the kernels: mbarriers, bulk async copies, bounded
// waits, element conversions.  All inline PTX follows the PTX ISA for sm_100-family
// targets (this library is built for sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "pagedkv.h"

#define PKV_DEV __device__ __forceinline__

// Every spin on an mbarrier gives up after this long and reports PKV_DEVERR_TIMEOUT.
#ifndef PKV_WAIT_LIMIT_NS
#define PKV_WAIT_LIMIT_NS 1000000000ull
#endif

PKV_DEV uint32_t smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

PKV_DEV uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: let the next kernel of the stream begin launching, and wait
// until the previous kernel has completed and its memory is visible (no-ops when the kernel was
// launched without the programmatic-serialization attribute).
PKV_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
PKV_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

PKV_DEV void set_error(unsigned int *err, unsigned int bits) {
    if (err) atomicOr(err, bits);
}

// ------------------------------------------------------------------ mbarrier

PKV_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

PKV_DEV void fence_mbarrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

PKV_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

PKV_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// raise the transaction count of the current phase without arriving (the arrival comes later)
PKV_DEV void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

PKV_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// non-blocking test: has the phase of `parity` completed?
PKV_DEV bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false after limit_ns
// without completion (checked every 256 tests), or after 2^31 tests whatever the clock says.
PKV_DEV bool mbar_wait_for(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < 0x80000000u; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// The kernels' wait: bounded by PKV_WAIT_LIMIT_NS.
PKV_DEV bool mbar_wait(uint64_t *bar, uint32_t parity) { return mbar_wait_for(bar, parity, PKV_WAIT_LIMIT_NS); }

// The same bounded wait with a suspend-time hint: a warp whose phase has not completed sleeps in
// the barrier until it completes (or the hint runs out) instead of re-testing it, which leaves the
// shared-memory pipe to the warps doing the work in kernels where many warps wait at once.  The
// first test is inline; the loop that keeps time for the wait limit is one out-of-line copy, so
// that the many wait sites of a large kernel stay small in the instruction cache.
PKV_DEV bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

static __device__ __noinline__ bool mbar_wait_sleep_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0; i < 0x80000000u; ++i) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

PKV_DEV bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint64_t limit_ns = PKV_WAIT_LIMIT_NS) {
    const uint32_t b = smem_u32(bar);
    return mbar_try_wait_sleep(b, parity) || mbar_wait_sleep_slow(b, parity, limit_ns);
}

// The same wait entirely inline, for kernels whose warps change their register budget
// (setmaxnreg), where a call to the out-of-line loop cannot be register-allocated.
PKV_DEV bool mbar_wait_hint(uint64_t *bar, uint32_t parity, uint64_t limit_ns = PKV_WAIT_LIMIT_NS) {
    const uint32_t b = smem_u32(bar);
    if (mbar_try_wait_sleep(b, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0; i < 0x80000000u; ++i) {
        if (mbar_try_wait_sleep(b, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// two-lane fp32 arithmetic (one instruction for both lanes): a * b + c and a + b; max of three
// (the softmax of the prefill kernels issues these per key pair instead of two scalar operations)
PKV_DEV float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}
PKV_DEV float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
PKV_DEV float2 add2(float2 a, float2 b) {
    unsigned long long ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

// ------------------------------------------------------------------ bulk async copy (1-D TMA)

// global -> shared, completion counted in bytes on `bar`.  dst/src 16-B aligned, bytes % 16 == 0.
PKV_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

PKV_DEV void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

PKV_DEV uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

PKV_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

PKV_DEV void named_barrier_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads: every thread leaves
// with the same answer, so a group of warps can agree to stop together (a warp that left on its
// own would leave the others waiting at the next barrier).
PKV_DEV bool named_barrier_and(uint32_t id, uint32_t nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// The same barrier reducing with OR: true on every thread if any of the nthreads passed true.
PKV_DEV bool named_barrier_or(uint32_t id, uint32_t nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ math

PKV_DEV float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// (a0, a1) += (x0, x1) * (y0, y1) as one packed fp32 FMA; each half is an IEEE fma, round to nearest
PKV_DEV void ffma2(float &a0, float &a1, float x0, float x1, float y0, float y1) {
    asm("{\n\t.reg .b64 ra, rx, ry;\n\t"
        "mov.b64 ra, {%0, %1};\n\tmov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\t"
        "fma.rn.f32x2 ra, rx, ry, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

// ------------------------------------------------------------------ element conversions

template <int DT>
struct ModelT;
template <>
struct ModelT<PKV_F16> {
    using T = __half;
    static PKV_DEV float to_f(T x) { return __half2float(x); }
    static PKV_DEV T from_f(float x) { return __float2half_rn(x); }
    // two floats -> one 32-bit word of two fp16 (round-to-nearest-even), `lo` in the low half
    static PKV_DEV uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
};
template <>
struct ModelT<PKV_BF16> {
    using T = __nv_bfloat16;
    static PKV_DEV float to_f(T x) { return __bfloat162float(x); }
    static PKV_DEV T from_f(float x) { return __float2bfloat16_rn(x); }
    static PKV_DEV uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
};

// 8 consecutive 16-bit elements (one uint4) -> 8 floats
template <int DT>
PKV_DEV void cvt8(const uint4 &u, float *f);
template <>
PKV_DEV void cvt8<PKV_F16>(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __half2float(__ushort_as_half(static_cast<unsigned short>(w[i] & 0xFFFFu)));
        f[2 * i + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(w[i] >> 16)));
    }
}
template <>
PKV_DEV void cvt8<PKV_BF16>(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// 8 consecutive E4M3 codes (one uint2) -> 8 floats (exact: every E4M3 value is an fp16 value)
PKV_DEV void cvt8_e4m3(const uint2 &u, float *f) {
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const unsigned short pair = static_cast<unsigned short>(w[i] >> (16 * j));
            uint32_t h2;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
            f[4 * i + 2 * j] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
            f[4 * i + 2 * j + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
        }
    }
}

// fp32 -> E4M3 pair: round to nearest-even, saturate to +-448, NaN -> 0x7F.
// Returns lo in bits 0..7 and hi in bits 8..15.
PKV_DEV uint32_t e4m3x2_from_f32(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    uint32_t v = r;
    if (isnan(lo)) v = (v & 0xFF00u) | 0x7Fu;
    if (isnan(hi)) v = (v & 0x00FFu) | 0x7F00u;
    return v;
}
