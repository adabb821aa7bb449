// Device-side helpers for libpkv kernels (sm_103a): mbarriers, bulk async
// copies into shared memory, bounded waits, and 16-bit / 8-bit unpacking.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

#include "pkv_internal.h"

namespace pkv {
namespace dev {

constexpr unsigned FULL_MASK = 0xffffffffu;

// A bounded wait gives up after about one second of device time.
constexpr uint64_t WAIT_LIMIT_NS = 1ull << 30;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed.  Gives up (and
// returns false) after WAIT_LIMIT_NS, or at once when *abort is set by any
// thread of the CTA; the caller then records the timeout and winds down.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (*abort)
                return false;
            if (globaltimer_ns() - t0 > WAIT_LIMIT_NS)
                return false;
        }
    }
}

// Wait until the shared counter *c reaches target (another thread of the
// CTA advances it).  Bounded like mbar_wait_bounded.
__device__ __forceinline__ bool count_wait_bounded(volatile int *c, int target,
                                                   volatile int *abort)
{
    if (*c >= target)
        return true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (*c >= target)
            return true;
        if ((it & 63u) == 0) {
            if (*abort)
                return false;
            if (globaltimer_ns() - t0 > WAIT_LIMIT_NS)
                return false;
        }
    }
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel of its stream is still
// running; grid_dependency_wait() blocks until that kernel has completed and
// its memory is visible, so it must come before the first global access.
// grid_dependents_launch() lets the next such kernel start early (it still
// waits for this one to finish before touching memory).  Both are no-ops for
// a kernel launched without the attribute.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host: launch kernel<<<grid, block, smem, stream>>>(args...) with
// programmatic stream serialization allowed, so that its launch and prologue
// overlap the tail of the previous kernel in the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Relaxed load at GPU scope (no ordering; pair with a fence to acquire).
__device__ __forceinline__ int ld_relaxed_gpu(const int *ptr)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// Bulk (non-tensor) async copy global -> this CTA's shared memory; completion
// is counted in bytes on the mbarrier.  dst, src 16-byte aligned; bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Asynchronous 16-byte (L2 only) and 8-byte copies global -> shared
// (cp.async): addresses aligned to the size.  Their completion reaches an
// mbarrier through cp_async_mbar_arrive.
__device__ __forceinline__ void cp_async_16b(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_8b(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

// One arrival on the mbarrier once every cp.async this thread issued before
// has landed.  The arrival is not added to the barrier's pending count: the
// barrier's expected arrival count must include it.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- unpacking -------------------------------------------------------------

// Two bf16 packed in a word -> two floats (exact: bf16 is the top half of f32).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float2 half2_to_float2(uint32_t w)
{
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
}

// Bytes 2J and 2J+1 of a word of biased int8 codes -> two exact floats: each
// biased byte becomes the low mantissa bits of 2^23, and one packed add takes
// 2^23 + 128 off both.
template <int J>
__device__ __forceinline__ void i8pair_to_float2(uint32_t biased, float &lo, float &hi)
{
    const float a = __uint_as_float(__byte_perm(biased, 0x4B000000u, 0x7440u + 2 * J));
    const float b = __uint_as_float(__byte_perm(biased, 0x4B000000u, 0x7441u + 2 * J));
    asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\t"
        "add.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "f"(a), "f"(b), "f"(-8388736.0f));
}

// 4-bit two's-complement codes, code j of a word in bits 4j..4j+3.
// Codes k and k+4 -> an fp16 pair, exactly: the biased code (code ^ 8 =
// code + 8) becomes the low mantissa bits of 1024 (0x6400), and 1032 (0x6408)
// is subtracted.
__device__ __forceinline__ uint32_t i4pair_to_half2(uint32_t w, int k)
{
    const uint32_t t = ((w >> (4 * k)) & 0x000F000Fu) ^ 0x64086408u;
    uint32_t h;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(t), "r"(0x64086408u));
    return h;
}

// Codes at bits 4..7 and 20..23 of w -> an fp16 pair, exactly, without a
// shift: the biased field lands 4 bits up in the mantissa of 1024, giving
// 1024 + 16 (code + 8); times 1/16 minus 72 is the code (every step exact).
__device__ __forceinline__ uint32_t i4pair_hi_to_half2(uint32_t w)
{
    const uint32_t t = (w & 0x00F000F0u) ^ 0x64806480u;
    uint32_t h;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(h) : "r"(t), "r"(0x2C002C00u), "r"(0xD480D480u));
    return h;
}

// Codes at bits 0..3 and 16..19 of w -> an fp16 pair, exactly.
__device__ __forceinline__ uint32_t i4pair_lo_to_half2(uint32_t w)
{
    const uint32_t t = (w & 0x000F000Fu) ^ 0x64086408u;
    uint32_t h;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(t), "r"(0x64086408u));
    return h;
}

// The code in the low 4 bits of x -> float, exactly (biased code in the
// mantissa of 2^23, minus 2^23 + 8).
__device__ __forceinline__ float i4_to_float(uint32_t x)
{
    return __uint_as_float((x & 0xFu) ^ 0x4B000008u) - 8388616.0f;
}

// Mixed-precision FMA: fp32 accumulate of the product of two bf16 (or fp16)
// halves taken from packed words; the product is exact in fp32.
__device__ __forceinline__ float fma_bf16x2(uint32_t a, uint32_t b, float c)
{
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 t;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 t, al, bl, %3;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, t;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float fma_f16x2(uint32_t a, uint32_t b, float c)
{
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 t;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 t, al, bl, %3;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, t;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}

}  // namespace dev
}  // namespace pkv
