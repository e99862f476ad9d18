// Device-side helpers shared by the libq2k kernels (sm_103a only).
//
// Q2_K block layout (mlx-native page "tests/deepseek_q2_k.rs", fixture fn
// block and fn reference_dequant): 84 bytes per 256 weights - scale bytes at
// 0..15 (low nibble sc, high nibble m), 2-bit quants at 16..79, f16 d at
// 80..81, f16 dmin at 82..83.  Weight k = 128 half + 32 j + 16 seg + lane is
// dl*q - ml with q = (qs[32 half + 16 seg + lane] >> 2j) & 3 and
// dl = d*(sc&15), ml = dmin*(sc>>4) taken from scale byte 8 half + 2 j + seg.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libq2k is written for sm_103a (Blackwell) only"
#endif

namespace q2k {

constexpr int kQK = 256;          // weights per super-block
constexpr int kBlockBytes = 84;   // bytes per super-block
constexpr int kWordsPerBlock = 21;

// Bits of the device error word (see q2k_device_error in q2k.h).
constexpr uint32_t kErrTimeoutFull = 1u;    // MMA issuer gave up waiting for a filled stage
constexpr uint32_t kErrTimeoutEmpty = 2u;   // a producer gave up waiting for a free stage
constexpr uint32_t kErrTimeoutAccum = 4u;   // epilogue gave up waiting for the accumulator
constexpr uint32_t kErrTimeoutDrain = 8u;   // teardown gave up waiting for in-flight MMAs
constexpr uint32_t kErrTimeoutGemv = 16u;   // GEMV gave up waiting for its weight copies

__device__ __forceinline__ float f16_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t ld_u32(const uint8_t* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}

// Read-only, streamed once: do not keep it in L1.
__device__ __forceinline__ uint32_t ldg_stream_u32(const uint8_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ---- programmatic dependent launch ------------------------------------------

// Block until the grids this one depends on have completed and their writes
// are visible (a no-op when the launch carries no programmatic dependency).
__device__ __forceinline__ void pdl_wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next grid in the stream to start launching.
__device__ __forceinline__ void pdl_allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- packed fp32 (sm_100+) --------------------------------------------------

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// ---- bulk asynchronous copies (TMA, non-tensor) ----------------------------

// Prefetch [src, src + bytes) into L2; src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Copy bytes (multiple of 16, both addresses 16-byte aligned) global -> shared,
// completing `bytes` transaction bytes on the mbarrier at `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ---- mbarrier (shared::cta) -------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the hardware may suspend the thread for up to
// `suspend_ns` until the phase completes (no instructions issued meanwhile).
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity,
                                                      uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed, but never for
// more than about `limit_ns`: on time-out (or when another thread of the CTA
// already timed out and raised *abort) set `err_bit` in *err, raise *abort
// and return false.  No wait in libq2k is unbounded.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, unsigned int* err,
                                                  uint32_t err_bit,
                                                  uint64_t limit_ns = 1000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_suspend(bar, parity, 1000u)) return true;
        if ((it & 7u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                atomicOr(err, err_bit);
                *abort = 1;
                return false;
            }
        }
    }
}

// As mbar_wait_bounded (kept as a separate entry for waiters off the critical
// path); both suspend in hardware between polls instead of spinning, so
// waiting threads take no issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_wait_backoff(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, unsigned int* err,
                                                  uint32_t err_bit, uint32_t max_sleep_ns,
                                                  uint64_t limit_ns = 1000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_suspend(bar, parity, max_sleep_ns < 1000u ? 1000u : max_sleep_ns))
            return true;
        if ((it & 7u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                atomicOr(err, err_bit);
                *abort = 1;
                return false;
            }
        }
    }
}

// Non-blocking test of a phase (one instruction, never suspends).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for warps that share their scheduler with busy warps: one
// test per poll and a short sleep between polls, so a waiting warp spends a
// handful of instructions per poll (the suspending try_wait form expands to
// a longer retry loop).  Same abort / time-out contract as mbar_wait_bounded.
__device__ __forceinline__ bool mbar_wait_lean(uint32_t bar, uint32_t parity, volatile int* abort,
                                               unsigned int* err, uint32_t err_bit,
                                               uint32_t sleep_ns,
                                               uint64_t limit_ns = 1000000000ull) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(sleep_ns);
        if (mbar_test_wait(bar, parity)) return true;
        if ((it & 15u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                atomicOr(err, err_bit);
                *abort = 1;
                return false;
            }
        }
    }
}

// ---- explicit shared-memory accesses (addresses from smem_u32) -------------

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

}  // namespace q2k
