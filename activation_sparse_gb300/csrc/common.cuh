// common.cuh -- device helpers shared by the kernels of the library:
// mbarrier / bulk-copy PTX wrappers with bounded waits, bf16 unpacking,
// order-preserving keys for radix selection, and the error word.
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/si.h"

namespace si {

constexpr int kWarp = 32;

// Upper bound on any spin in a kernel, in SM clock cycles (about 4 s at
// 2 GHz). A correct kernel never waits this long; when a wait runs out the
// kernel records SI_DEVERR_WAIT_TIMEOUT in the device error word and goes on
// without blocking. clock64() is the SM's own monotonic cycle counter (the
// global nanosecond timer can be stepped by the driver's time sync).
constexpr long long kWaitLimitCycles = 8000000000ll;
constexpr long long kDrainLimitCycles = 400000000ll;

__device__ __forceinline__ long long cycles() { return clock64(); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
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

// Bounded wait for the phase with the given parity to complete. Returns false
// when the limit runs out (recording SI_DEVERR_WAIT_TIMEOUT), or at once when
// some wait has already run out, so a faulty launch ends within one limit.
// Wait sites recorded with a timeout: kernel id in bits 8-15, barrier kind in
// bits 16-19 (see si.h).
enum : unsigned {
    kSiteDecode = 1u << 8, kSiteDenseAct = 2u << 8, kSiteTiered = 3u << 8, kSiteGemm = 4u << 8,
    kSiteFull = 1u << 16, kSiteEmpty = 2u << 16, kSiteFullB = 3u << 16, kSiteAccum = 4u << 16,
};

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err, unsigned site = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = cycles();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*reinterpret_cast<volatile unsigned*>(err) & SI_DEVERR_WAIT_TIMEOUT) return false;
            if (cycles() - t0 > kWaitLimitCycles) {
                atomicOr(err, SI_DEVERR_WAIT_TIMEOUT | site);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------- bulk copies

// 1-D bulk copy global -> this CTA's shared memory, completion counted in
// bytes on `bar`. dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
        "[%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 prefetch of a global range (a hint: no data dependency, no completion).
__device__ __forceinline__ void prefetch_l2(const void* src_gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// ------------------------------------------------ programmatic dependent launch

// Blocks until the grids this launch depends on have completed and their
// memory is visible (a no-op when the launch has no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next launch in the stream (if it was launched with programmatic
// stream serialization) start scheduling its CTAs before this grid finishes.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// -------------------------------------------------------------- named barrier

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- bf16 math

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// dot of 8 bf16 pairs packed in two uint4, accumulated into acc (fp32)
// acc + sum of the 8 products a[e] * b[e] of bf16 pairs, in element order.
// fma.rn.f32.bf16 takes the bf16 operands directly: their product is exact
// in float32 and is added with one rounding, so the result is bit for bit
// that of converting to float32 and calling fmaf, without the conversions.
__device__ __forceinline__ float fma_bf16x2(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

__device__ __forceinline__ float dot8(const uint4 a, const uint4 b, float acc) {
    acc = fma_bf16x2(a.x, b.x, acc);
    acc = fma_bf16x2(a.y, b.y, acc);
    acc = fma_bf16x2(a.z, b.z, acc);
    acc = fma_bf16x2(a.w, b.w, acc);
    return acc;
}

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
    f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
    f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// silu(g) * u, the SwiGLU activation (down_proj input)
__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// ------------------------------------------------------------ ordering keys

// Magnitude key: larger |f| <=> larger key (-0 and +0 equal). NaN ranks above inf.
__device__ __forceinline__ uint32_t abs_key(float f) { return __float_as_uint(f) & 0x7FFFFFFFu; }

// Value key: monotone map of float order onto uint32 order (-0 == +0).
__device__ __forceinline__ uint32_t value_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ------------------------------------------------------------------ host

// Lets `kernel` use all the dynamic shared memory the device offers (once per
// kernel and device). Launches then only need their own size to fit, whatever
// size an earlier launch of the same kernel used.
template <class K>
cudaError_t allow_max_smem(K kernel) {
    static std::mutex mu;
    static const void* done[64];
    static int done_dev[64];
    static int n_done = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void* fn = reinterpret_cast<const void*>(kernel);
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i] == fn && done_dev[i] == dev) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    if (n_done < 64) {
        done[n_done] = fn;
        done_dev[n_done] = dev;
        ++n_done;
    }
    return cudaSuccess;
}

}  // namespace si
