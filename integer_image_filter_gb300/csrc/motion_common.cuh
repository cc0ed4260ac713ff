// motion_common.cuh -- device helpers shared by the motion and SSE kernels of
// libmotion_gb300 (sm_103a).  Nothing here is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>

namespace mg {

// The 5-tap integer Gaussian of the motion feature: t0 = t4 = 3571,
// t1 = t3 = 16004, t2 = 26386 (sum 65536).  Symmetric, so each pass is
// t0 (a + e) + t1 (b + d) + t2 c.
constexpr uint32_t kT0 = 3571u;
constexpr uint32_t kT1 = 16004u;
constexpr uint32_t kT2 = 26386u;
static_assert(2 * kT0 + 2 * kT1 + kT2 == 65536u, "taps must sum to 2^16");

// Mirror index for n >= 3 and -2 <= i <= n + 1, clamped into [0, n) for the
// positions a tile loads but never uses.
__device__ __forceinline__ int mirror_clamp(int i, int n) {
    i = i < 0 ? -i : i;
    i = i >= n ? 2 * n - i - 2 : i;
    i = i < 0 ? 0 : i;
    return i >= n ? n - 1 : i;
}

// 16-byte asynchronous global -> shared copy (L2 only), grouped by commit.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

}  // namespace mg

// ---------------------------------------------------------------- TMA / mbarrier
namespace mg {

__device__ __forceinline__ unsigned smem_u32(const void* p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before the
// asynchronous (TMA) writes it issues next.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile(
        "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// One potentially blocking test of an mbarrier phase (the hardware holds the
// warp for a short, implementation-defined time before reporting "not yet").
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for a phase of an mbarrier: gives up after `limit_cycles` SM
// clock cycles and returns false (the caller records the error and leaves);
// it never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity,
                                                  long long limit_cycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit_cycles) return false;
    }
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

}  // namespace mg

namespace mg {

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

}  // namespace mg
