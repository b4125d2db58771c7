// Device helpers shared by the libxs_paged kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "xs_paged.h"

namespace xs {

// ------------------------------------------------------------------ dtypes

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f32(float x) { return x; }
    static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// Unpack a 16-byte vector of T into fp32 values (8 bf16 or 4 fp32).
__device__ __forceinline__ void unpack16(const uint4 &v, float *f, __nv_bfloat16 *) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4 &v, float *f, float *) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}

// 2^x with the hardware approximation (relative error ~2^-22; ex2 of -inf is +0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void raise_flag(int *err_flag, int bit) {
    if (err_flag) atomicOr(err_flag, bit);
}

// ------------------------------------------------------------------ debug bounds checks
// Compiled with -DXS_DEBUG_BOUNDS (the debug library), XS_BOUNDS(cond, flag)
// evaluates cond - that a computed global-memory index lies inside its
// buffer - and when it does not, ORs XS_FLAG_BOUNDS into *flag and yields
// false, so the guarded access is skipped.  It stands in for a device memory
// checker: the debug library runs the same cases as the release one and the
// flag must stay clear.  In release builds it is the constant true.
// Failed checks are also counted per translation unit (err_flag is optional),
// and xs_debug_bounds_failures() returns the sum over the library.
#ifdef XS_DEBUG_BOUNDS
static __device__ unsigned int g_bounds_failures;
__device__ __forceinline__ bool bounds_ok(bool ok, int *err_flag) {
    if (!ok) {
        raise_flag(err_flag, XS_FLAG_BOUNDS);
        atomicAdd(&g_bounds_failures, 1u);
    }
    return ok;
}
#define XS_BOUNDS(cond, err_flag) (::xs::bounds_ok(static_cast<bool>(cond), (err_flag)))
// This translation unit's count of failed checks on the current device
// (optionally cleared), or a negative XS_E* code.
#define XS_DEFINE_BOUNDS_COUNTER(fn)                                                       \
    int fn(int reset) {                                                                   \
        unsigned int v = 0;                                                               \
        if (cudaMemcpyFromSymbol(&v, ::xs::g_bounds_failures, sizeof(v)) != cudaSuccess) \
            return XS_EDEVICE;                                                            \
        if (reset) {                                                                      \
            const unsigned int z = 0;                                                     \
            if (cudaMemcpyToSymbol(::xs::g_bounds_failures, &z, sizeof(z)) != cudaSuccess) \
                return XS_EDEVICE;                                                        \
        }                                                                                 \
        return static_cast<int>(v);                                                       \
    }
#else
#define XS_BOUNDS(cond, err_flag) true
#define XS_DEFINE_BOUNDS_COUNTER(fn) \
    int fn(int) { return 0; }
#endif
// Per translation unit (kv_append.cu, paged_decode.cu, paged_prefill_tc.cu).
int bounds_failures_append(int reset);
int bounds_failures_decode(int reset);
int bounds_failures_prefill_tc(int reset);

// ------------------------------------------------------------------ mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// atomicAdd(ptr, v) on the threads where pred holds (returning the old
// value; 0 elsewhere) as one predicated instruction, so no branch forces the
// warp to wait for the result before it is used.
// Atomic add with acquire-release semantics at GPU scope: this thread's
// earlier writes (and those it has synchronized with) are released by it,
// and the writes released to the counter before are acquired.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *ptr, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v)
                 : "memory");
    return old;
}

__device__ __forceinline__ int atomic_add_if(int *ptr, int v, bool pred) {
    int old = 0;
    asm volatile(
        "{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q atom.global.add.u32 %0, [%1], %3;\n}"
        : "+r"(old)
        : "l"(ptr), "r"(static_cast<uint32_t>(pred)), "r"(v)
        : "memory");
    return old;
}

// Acquire-release fence at GPU scope: this thread's earlier memory operations
// (and those it has synchronized with) happen before its later ones, as
// seen by any thread of the GPU that synchronizes with it.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
// Orders this thread's earlier generic-proxy writes to global memory before
// later async-proxy operations (bulk copies) that read the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// The same for this CTA's shared memory (generic stores, then tensor-core or
// bulk-copy reads of them).
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Programmatic dependent launch (sm_90+): let the next grid on the stream be
// scheduled, and wait until the previous grid has completed with its memory
// writes visible.  Both return at once when the launch had no such dependency.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Bring `bytes` (a multiple of 16, 16-byte aligned) at global `src` into L2;
// a hint with no completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Non-blocking test of a phase (try_wait may suspend the thread for a while).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, giving up after
// `limit_ns` of wall time.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).  The source is read once: evict-first.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Dynamic shared memory the running launch was given (bytes).
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t n;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
    return n;
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ host-side checks

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int elem_bytes(int dtype) {
    return dtype == XS_F32 ? 4 : (dtype == XS_BF16 ? 2 : 0);
}

inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? XS_OK : XS_ELAUNCH;
}

}  // namespace xs
