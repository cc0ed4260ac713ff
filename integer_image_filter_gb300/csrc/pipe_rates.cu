// pipe_rates.cu -- throughput of the instruction classes the motion kernels
// run, measured on the device they run on (libpipe_rates_gb300.so; not part
// of the motion library).  Each measurement is a kernel whose loop issues one
// instruction class many times over independent dependency chains, so that
// the pipe, not the latency of one chain, sets the rate.  Every block reads
// the SM clock before and after its loop; the rate is the lane-operations of
// all blocks divided by the SM count and by the largest block duration in SM
// clocks (the blocks of one launch all fit on the device at once).
//
// The result, lane-operations per clock per SM for each class, is the peak
// the integer co-bound of the motion kernels is taken against: their ncu
// instruction counts per pipe divided by these rates give the fewest clocks
// each pipe needs per launch.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace {

constexpr int kChains = 8;     // independent dependency chains per thread
constexpr int kUnroll = 16;    // operations per chain per loop iteration

struct Out {
    unsigned long long max_cycles;
    unsigned long long sink;
};

// One class per tag: op(x, y, k) returns the next value of a chain from its
// own value x and the neighbouring chain's value y (so that no two operations
// of a chain can be folded into one), k being loop-invariant.
struct OpImad {     // IMAD: a * b + c
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t k) const { return x * y + k; }
};
struct OpDp2a {     // IDP.2A: two 16 x 8 bit products and an add
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t k) const {
        return __dp2a_lo(x, y, k);
    }
};
struct OpDp4a {     // IDP.4A: four 8 x 8 bit products and an add
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t k) const {
        return __dp4a(x, y, k);
    }
};
struct OpIadd3 {    // IADD3: a + b - c
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t k) const { return x + y - k; }
};
struct OpShf {      // SHF: funnel shift of two registers by a register amount
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t k) const {
        return __funnelshift_r(x, y, k);
    }
};
struct OpPrmt {     // PRMT: byte permute of two registers
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t) const {
        return __byte_perm(x, y, 0x5140);
    }
};
struct OpSad {      // VABSDIFF: |a - b| + c
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t k) const { return __sad(x, y, k); }
};
struct OpLop3 {     // LOP3: a ^ (b & c)
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t k) const {
        uint32_t r;
        asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r) : "r"(x), "r"(y), "r"(k));
        return r;
    }
};
struct OpFfma {     // FFMA on the bit patterns as floats
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t k) const {
        return __float_as_uint(fmaf(__uint_as_float(x), __uint_as_float(y), __uint_as_float(k)));
    }
};
struct OpShfl {     // SHFL: a butterfly shuffle with a register lane mask
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t) const {
        return __shfl_xor_sync(0xffffffffu, x, y);
    }
};
struct OpMnmx {     // VIMNMX: unsigned minimum
    __device__ __forceinline__ uint32_t operator()(uint32_t x, uint32_t y, uint32_t) const { return min(x, y); }
};

template <typename Op>
__global__ void __launch_bounds__(256) rate_kernel(int iters, uint32_t seed, Out* out) {
    uint32_t v[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) v[c] = seed * (threadIdx.x + 1u) + (uint32_t)c * 0x45d9f3bu;
    const uint32_t k = (seed ^ 0x27d4eb2du) & 0x0f0f0f0fu;
    Op op;
    __syncthreads();
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            uint32_t nv[kChains];
#pragma unroll
            for (int c = 0; c < kChains; ++c) nv[c] = op(v[c], v[(c + 1) % kChains], k);
#pragma unroll
            for (int c = 0; c < kChains; ++c) v[c] = nv[c];
        }
    }
    const long long t1 = clock64();
    __syncthreads();
    uint32_t acc = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc ^= v[c];
    if (threadIdx.x == 0) atomicMax(&out->max_cycles, (unsigned long long)(t1 - t0));
    if (acc == 0x12345678u) out->sink = acc;   // keeps the chains live
}

// Shared-memory loads of 32 or 128 bits per lane, consecutive across the warp.
template <int WORDS>
__global__ void __launch_bounds__(256) lds_kernel(int iters, uint32_t seed, Out* out) {
    __shared__ __align__(16) uint32_t buf[256 * 4 + 64];
    for (int i = threadIdx.x; i < 256 * 4 + 64; i += blockDim.x) buf[i] = seed + i;
    __syncthreads();
    uint32_t acc = 0;
    const int lane = threadIdx.x & 31;
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll * 2; ++u) {
            const int off = (((u * 7 + i) & 7) * 32 + lane) * WORDS;
            const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(&buf[off]));
            if constexpr (WORDS == 4) {
                uint32_t x, y, z, w;
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(x), "=r"(y), "=r"(z), "=r"(w) : "r"(a));
                acc += x ^ w;
            } else {
                uint32_t x;
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x) : "r"(a));
                acc += x;
            }
        }
    }
    const long long t1 = clock64();
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(&out->max_cycles, (unsigned long long)(t1 - t0));
    if (acc == 0x12345678u) out->sink = acc;
}

template <typename K>
int run(K kernel, int ops_per_iter_per_thread, int iters, int blocks_per_sm, double* lanes_per_clk) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    Out* d = nullptr;
    if (cudaMalloc(&d, sizeof(Out)) != cudaSuccess) return 1;
    int rc = 0;
    for (int rep = 0; rep < 2 && !rc; ++rep) {   // the first launch warms up
        if (cudaMemset(d, 0, sizeof(Out)) != cudaSuccess) rc = 1;
        kernel<<<sms * blocks_per_sm, 256>>>(iters, 0x1234567u + rep, d);
        if (cudaDeviceSynchronize() != cudaSuccess) rc = 1;
    }
    Out h;
    std::memset(&h, 0, sizeof(h));
    if (!rc && cudaMemcpy(&h, d, sizeof(Out), cudaMemcpyDeviceToHost) != cudaSuccess) rc = 1;
    cudaFree(d);
    if (rc || h.max_cycles == 0) return 1;
    const double lane_ops = (double)blocks_per_sm * 256.0 * (double)iters * ops_per_iter_per_thread;
    *lanes_per_clk = lane_ops / (double)h.max_cycles;
    return 0;
}

}  // namespace

// Number of measured classes and their names (static strings).
extern "C" __attribute__((visibility("default"))) int pipe_rates_count(void) { return 13; }

extern "C" __attribute__((visibility("default"))) const char* pipe_rates_name(int i) {
    static const char* names[] = {"IMAD", "IDP.2A (dp2a)", "IDP.4A (dp4a)", "IADD3", "SHF", "PRMT",
                                  "VABSDIFF (sad)", "LOP3", "FFMA", "SHFL", "VIMNMX (min)",
                                  "LDS.32", "LDS.128"};
    return i >= 0 && i < 13 ? names[i] : "";
}

// Measures every class on the current device: out[i] receives lane-operations
// per SM clock per SM (shared-memory loads: bytes per clock per SM).
// Returns 0, or 1 when a CUDA call failed.
extern "C" __attribute__((visibility("default"))) int pipe_rates_measure(double* out) {
    const int it = 2048, bps = 4;   // 4 blocks of 256 threads per SM: 32 warps
    const int ops = kChains * kUnroll;
    int rc = 0;
    rc |= run(rate_kernel<OpImad>, ops, it, bps, &out[0]);
    rc |= run(rate_kernel<OpDp2a>, ops, it, bps, &out[1]);
    rc |= run(rate_kernel<OpDp4a>, ops, it, bps, &out[2]);
    rc |= run(rate_kernel<OpIadd3>, ops, it, bps, &out[3]);
    rc |= run(rate_kernel<OpShf>, ops, it, bps, &out[4]);
    rc |= run(rate_kernel<OpPrmt>, ops, it, bps, &out[5]);
    rc |= run(rate_kernel<OpSad>, ops, it, bps, &out[6]);
    rc |= run(rate_kernel<OpLop3>, ops, it, bps, &out[7]);
    rc |= run(rate_kernel<OpFfma>, ops, it, bps, &out[8]);
    rc |= run(rate_kernel<OpShfl>, ops, it / 4, bps, &out[9]);
    rc |= run(rate_kernel<OpMnmx>, ops, it, bps, &out[10]);
    double w = 0;
    rc |= run(lds_kernel<1>, kUnroll * 2, it, bps, &w);
    out[11] = w * 4.0;     // bytes per clock
    rc |= run(lds_kernel<4>, kUnroll * 2, it, bps, &w);
    out[12] = w * 16.0;
    return rc;
}
