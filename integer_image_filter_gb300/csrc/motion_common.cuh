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
