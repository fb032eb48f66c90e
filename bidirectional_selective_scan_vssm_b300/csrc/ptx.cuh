// Thin wrappers over the PTX instructions the scan kernels use: mbarriers,
// 1-D bulk async copies (the TMA engine's non-tensor form), proxy fences,
// packed f32x2 arithmetic and the MUFU exp2.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vssm {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase. Returns false if the phase has not
// completed within limit_ns, or after 2^28 polls whatever the timer says (the
// caller then reports a timeout and stops).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t polls = 0; !mbar_try_wait(bar, parity); ++polls) {
        if (global_timer_ns() - t0 > limit_ns || polls >= (1u << 28)) return false;
    }
    return true;
}

// Per-thread 16-byte async copy global -> shared (L2-cached only). Bytes past
// src_bytes (1..16) are zero-filled; dst and src must be 16-byte aligned.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Per-thread 16-byte async copy global -> shared of a whole block.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// Store v to global memory when pred holds (a predicated store, no branch).
// No memory clobber: the compiler may move other loads and stores across it;
// it stays ordered with the other volatile asm, fences included.
__device__ __forceinline__ void st_global_if(float *ptr, float v, bool pred)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p st.global.f32 [%0], %1;\n\t}" ::"l"(ptr),
                 "f"(v), "r"((unsigned)pred));
}

__device__ __forceinline__ void st_global_if(__nv_bfloat16 *ptr, __nv_bfloat16 v, bool pred)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p st.global.b16 [%0], %1;\n\t}" ::"l"(ptr),
                 "h"(*reinterpret_cast<unsigned short *>(&v)), "r"((unsigned)pred));
}

// cp_async16 issued only when pred holds (a predicated instruction; nothing is
// read or written otherwise).
__device__ __forceinline__ void cp_async16_if(void *dst, const void *src, bool pred)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t"
                 "@p cp.async.cg.shared.global [%0], [%1], 16;\n\t}" ::"r"(smem_addr(dst)),
                 "l"(src), "r"((unsigned)pred)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's committed copy groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Global -> shared bulk copy; completion is signalled on `bar` as transaction
// bytes. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Shared -> global bulk copy, tracked by the bulk async-group of this thread.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the source of every committed bulk store may be overwritten.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic-proxy global-memory accesses with later
// async-proxy (bulk copy) accesses of the same data.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- packed f32x2 arithmetic (sm_100+): one instruction, two fp32 lanes

struct f2 {
    uint64_t v;
};

__device__ __forceinline__ f2 pack2(float a, float b)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float2 unpack2(f2 a)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(a.v));
    return r;
}

__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return d;
}

// In-place forms: the accumulator keeps its register pair (a loop-carried
// state updated in place needs no copy at the loop's back edge).
// acc = a * acc + c
__device__ __forceinline__ void fma2_scale_acc(f2 &acc, f2 a, f2 c)
{
    asm("fma.rn.f32x2 %0, %1, %0, %2;" : "+l"(acc.v) : "l"(a.v), "l"(c.v));
}
// acc = a * b + acc
__device__ __forceinline__ void fma2_acc(f2 &acc, f2 a, f2 b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc.v) : "l"(a.v), "l"(b.v));
}

__device__ __forceinline__ f2 add2(f2 a, f2 b)
{
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}

__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}

// Two fp32 pairs from 16 bytes of shared memory (16-byte aligned), kept as
// 64-bit registers so they feed packed instructions without repacking.
__device__ __forceinline__ void lds_2xf2(const void *p, f2 &a, f2 &b)
{
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a.v), "=l"(b.v) : "r"(smem_addr(p)));
}

// (2^x.lo, 2^x.hi) of a pair, with the products a*b computed first: the
// argument, both MUFU results and the result pair stay in one register pair.
__device__ __forceinline__ f2 ex2_mul2(f2 a, f2 b)
{
    f2 d;
    asm("{\n\t.reg .b64 t;\n\t.reg .f32 lo, hi;\n\t"
        "mul.rn.f32x2 t, %1, %2;\n\t"
        "mov.b64 {lo, hi}, t;\n\t"
        "ex2.approx.ftz.f32 lo, lo;\n\t"
        "ex2.approx.ftz.f32 hi, hi;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(d.v) : "l"(a.v), "l"(b.v));
    return d;
}

// Same with a*b + c as the argument.
__device__ __forceinline__ f2 ex2_fma2(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("{\n\t.reg .b64 t;\n\t.reg .f32 lo, hi;\n\t"
        "fma.rn.f32x2 t, %1, %2, %3;\n\t"
        "mov.b64 {lo, hi}, t;\n\t"
        "ex2.approx.ftz.f32 lo, lo;\n\t"
        "ex2.approx.ftz.f32 hi, hi;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return d;
}

// 2^x on the MUFU unit.
__device__ __forceinline__ float ex2_mufu(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float tanh_mufu(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_mufu(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Invalidate a 128-byte line of global memory in L2 without writing it back
// (its contents become undefined). Used for scratch that has been read for
// the last time.
__device__ __forceinline__ void discard_l2(const void *p)
{
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Two fp32 values rounded (to nearest even) to bf16 and packed: lo in bits
// 0..15, hi in bits 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// softplus(v) = log(1 + exp(v)) = ln 2 * log2(1 + 2^(v * log2 e)) on the MUFU
// unit (absolute error about 1e-7, from lg2.approx). Above 15 it is v (the
// difference, log(1 + exp(-v)), is below 3.1e-7); below -30 it is 0 (the true
// value is below 1e-13), so a pre-activation of -inf gives a step of exactly 0.
__device__ __forceinline__ float softplus_f32(float v)
{
    const float s = 0.6931471805599453f * lg2_mufu(1.0f + ex2_mufu(v * 1.4426950408889634f));
    return v > 15.0f ? v : (v < -30.0f ? 0.0f : s);
}

}  // namespace vssm
