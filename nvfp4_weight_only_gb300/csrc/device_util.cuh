// device_util.cuh -- inline-PTX building blocks for sm_103a: mbarriers, the
// bulk-copy (TMA) engine, NVFP4 element conversions and the f16 tensor-core MMA.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace nvf {

// Longest a kernel waits on one mbarrier phase before it reports a timeout.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test, allowing the hardware to suspend the thread until the phase
// completes or hint_ns have passed, so waiting warps do not spin on the
// issue slots the working warps need.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Longest single suspension inside a bounded wait; the abort flag and the
// time limit are checked between suspensions.
constexpr uint32_t kSuspendHintNs = 20000;

// Waits for the phase with the given parity to complete.  Gives up (returns
// false) after limit_ns, or when *abort is set by another warp (noticed
// within one suspension).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, kSuspendHintNs)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// One bulk copy global -> shared through the TMA engine; completion is
// reported to `bar` as transaction bytes.  Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Same copy with an L2 eviction-priority hint (a createpolicy policy).
__device__ __forceinline__ void bulk_copy_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                                   uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// L2 policy that marks lines for early eviction (single-use streams).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// Load with acquire semantics at GPU scope.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Polls *p (acquire) until it reaches `target`.  Gives up (returns false)
// after limit_ns, or when *abort is set by another warp.
__device__ __forceinline__ bool wait_count_bounded(const int* p, int target,
                                                   const volatile int* abort,
                                                   unsigned long long limit_ns) {
    if (ld_acquire_gpu(p) >= target) return true;
    const unsigned long long t0 = global_timer_ns();
    unsigned pause = 32;  // ns, doubled up to 512 to keep the polling light
    for (;;) {
        __nanosleep(pause);
        if (pause < 512) pause *= 2;
        if (ld_acquire_gpu(p) >= target) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Four packed bytes of E2M1 pairs -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& a0, uint32_t& a1,
                                                  uint32_t& a2, uint32_t& a3) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
        : "r"(w));
}

// Two E4M3 bytes (low 16 bits of v) -> f16x2 (low byte -> low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
    uint32_t r;
    asm("{\n .reg .b16 h, hi;\n mov.b32 {h, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}"
        : "=r"(r)
        : "r"(v));
    return r;
}

// The same for the high two bytes of v (bytes 2, 3).
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t v) {
    uint32_t r;
    asm("{\n .reg .b16 lo, h;\n mov.b32 {lo, h}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}"
        : "=r"(r)
        : "r"(v));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// D += A * B for one m16n8k16 tile, f16 operands, f32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B for one m16n8k16 tile from a zero accumulator (C is the constant
// 0, D is write-only, so no accumulator registers need clearing).
__device__ __forceinline__ void mma_f16_16816_zero(float (&d)[4], uint32_t a0, uint32_t a1,
                                                   uint32_t a2, uint32_t a3, uint32_t b0,
                                                   uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Round-to-nearest-even, saturating conversion of one fp32 to an E4M3 byte.
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(v));
    return r & 0xFFu;
}

// Round-to-nearest-even, saturating conversion of one fp32 to an E2M1 code
// (4 bits).
__device__ __forceinline__ uint32_t f32_to_e2m1(float v) {
    uint32_t r;
    asm("{\n .reg .b8 b;\n cvt.rn.satfinite.e2m1x2.f32 b, %1, %1;\n cvt.u32.u8 %0, b;\n}"
        : "=r"(r)
        : "f"(v));
    return r & 0xFu;
}

// E4M3 byte -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    uint32_t h2 = e4m3x2_to_f16x2(b & 0xFFu);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

}  // namespace nvf
