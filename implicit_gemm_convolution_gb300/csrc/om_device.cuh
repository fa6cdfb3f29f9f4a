// om_device.cuh -- device-side building blocks shared by the library's kernels:
// the per-term arithmetic of the two bit-exact modes, the canonical-NaN store,
// mbarrier / TMA / cp.async wrappers in inline PTX, and bounded waits.
//
// Arithmetic follows the OneModel "Exact mode" page (rules 1-4 and section
// "Matrix product"): exact mode is round(acc + round(a*b)) with the multiply
// and the add rounded separately; fast mode ("Matrix product and convolution
// kernels" page, section "Fast mode") is one fused multiply-add per term.
// The library is compiled with -fmad=false and without -ftz, and uses the
// explicitly rounded _rn intrinsics, which the compiler never contracts.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace om {

enum Mode : int { kExact = 0, kFast = 1 };

// Bit of a translation unit's device status word set by a bounded wait that
// ran out; om_device_status() reads and clears the words.
constexpr unsigned kDevErrTimeout = 1u;

// Records a bounded wait that ran out: into the calling entry point's own
// status word when it has one (a word of the caller's workspace), else into
// the translation unit's device-wide word.
__device__ __forceinline__ void report_timeout(unsigned *call_status, unsigned *tu_word) {
    atomicOr(call_status != nullptr ? call_status : tu_word, kDevErrTimeout);
}

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ float canonical_nan(float v) {
    // Every stored NaN becomes the quiet NaN 0x7FC00000.
    return (v != v) ? __int_as_float(0x7FC00000) : v;
}

// The output epilogue's arithmetic, one binary32 operation per step:
// bias, then residual, then ReLU (keeps NaN, maps -0 and negatives to +0).
__device__ __forceinline__ float epilogue_value(float v, const float *bias, const float *res,
                                                int act) {
    if (bias) v = __fadd_rn(v, *bias);
    if (res) v = __fadd_rn(v, __ldg(res));
    if (act == 1 && !(v > 0.0f) && v == v) v = 0.0f;
    return v;
}

template <int MODE>
__device__ __forceinline__ float term(float acc, float a, float b) {
    if constexpr (MODE == kFast) {
        return __fmaf_rn(a, b, acc);
    } else {
        return __fadd_rn(acc, __fmul_rn(a, b));
    }
}

// Paired-lane fp32 instructions of sm_100+ (inline PTX, explicit .rn).
// Fast mode uses the paired fused multiply-add: one rounding per lane.
// Exact mode must keep the multiply and the add as two roundings. The
// assembler was measured to contract a paired multiply followed by a paired
// add into the paired fused multiply-add even when both carry .rn and even
// with --fmad=false, so exact mode pairs only the add: two scalar
// mul.rn.f32 (never contracted) feed one add.rn.f32x2. That form was checked
// bit for bit against the all-scalar form on the device and costs three
// issue slots per two terms instead of four.
__device__ __forceinline__ float mul_rn_scalar(float a, float b) {
    float r;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
    unsigned long long r;
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%1, %2};\n\t"
        "mov.b64 rb, {%3, %4};\n\t"
        "add.rn.f32x2 %0, ra, rb;\n\t}"
        : "=l"(r)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
    unsigned long long r;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%1, %2};\n\t"
        "mov.b64 rb, {%3, %4};\n\t"
        "mov.b64 rc, {%5, %6};\n\t"
        "fma.rn.f32x2 %0, ra, rb, rc;\n\t}"
        : "=l"(r)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}

// Two independent outputs: acc.x gets a.x*b.x, acc.y gets a.y*b.y, each lane
// rounded exactly like term<MODE>.
template <int MODE>
__device__ __forceinline__ float2 term2(float2 acc, float2 a, float2 b) {
    if constexpr (MODE == kFast) {
        return fma2_rn(a, b, acc);
    } else {
        return add2_rn(acc, make_float2(mul_rn_scalar(a.x, b.x), mul_rn_scalar(a.y, b.y)));
    }
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

// Wait for the phase with the given parity to complete; false after
// limit_ns (the caller records the error and leaves).
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity,
                                                unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_limit(bar, parity, kWaitLimitNs);
}

// Wait until the global flag *f is non-zero, with acquire ordering; false
// after limit_ns.
__device__ __forceinline__ bool acquire_flag(const unsigned *f, unsigned long long limit_ns) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v != 0) return true;
    const unsigned long long t0 = global_ns();
    do {
        __nanosleep(200);
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    } while (v == 0 && global_ns() - t0 <= limit_ns);
    return v != 0;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---------------------------------------------------------------- cp.async
// 4-byte copy global -> shared; src_bytes == 0 writes +0 without reading.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// 4-byte copy global -> shared when ok, else +0 written without reading src
// (src must still be a valid address).
__device__ __forceinline__ void cp_async_4_if(uint32_t dst, const void *src, bool ok) {
    asm volatile(
        "{\n\t.reg .pred skip;\n\tsetp.eq.u32 skip, %2, 0;\n\t"
        "cp.async.ca.shared.global [%0], [%1], 4, skip;\n\t}" ::"r"(dst),
        "l"(src), "r"(static_cast<uint32_t>(ok))
        : "memory");
}

// Two 32-bit integers from shared memory.
__device__ __forceinline__ int2 lds_int2(uint32_t a) {
    int2 v;
    asm volatile("ld.shared.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

// 16-byte copy global -> shared (both 16-byte aligned); src_bytes 0 or 16,
// 0 writes +0 without reading.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Arrive on bar once every cp.async this thread issued so far has landed.
// The barrier's expected count must include this arrival (.noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

}  // namespace om
