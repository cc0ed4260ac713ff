// pipe_rates.cu -- throughput of the instruction classes the motion kernels
// run, and the HBM read-only, write-only and copy stream rates, measured on
// the device they run on (libpipe_rates_gb300.so; not part of the motion
// library).  Each measurement is a kernel whose loop issues one
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

// ---- HBM streams: read-only, write-only and copy, 16 bytes per lane access,
// four accesses in flight per thread, grid-stride over buffers far larger
// than the L2 (of the variants measured -- eight accesses in flight, one
// contiguous part per block -- the fastest read stream).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__global__ void __launch_bounds__(256) hbm_read_kernel(const uint4* __restrict__ src, size_t n16, Out* out) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = ld_stream(src + i), b = ld_stream(src + i + stride);
        const uint4 c = ld_stream(src + i + 2 * stride), d = ld_stream(src + i + 3 * stride);
        acc ^= a.x ^ a.w ^ b.y ^ b.z ^ c.x ^ c.w ^ d.y ^ d.z;
    }
    for (; i < n16; i += stride) {
        const uint4 a = ld_stream(src + i);
        acc ^= a.x ^ a.w;
    }
    if (acc == 0x12345678u) out->sink = acc;
}

__global__ void __launch_bounds__(256) hbm_write_kernel(uint4* __restrict__ dst, size_t n16, uint32_t v) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const uint4 w = make_uint4(v, v + 1, v + 2, v + 3);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = w;
}

__global__ void __launch_bounds__(256) hbm_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                       size_t n16) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = ld_stream(src + i), b = ld_stream(src + i + stride);
        const uint4 c = ld_stream(src + i + 2 * stride), d = ld_stream(src + i + 3 * stride);
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = ld_stream(src + i);
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

// HBM bandwidth of one stream kind on the current device: 0 read-only (4 GiB
// read), 1 write-only (4 GiB written), 2 copy (2 GiB read and 2 GiB written;
// both directions counted).  *gbs receives the best of 5 timed launches after
// one warm-up, in GB/s (10^9 bytes).  Returns 0, or 1 when a CUDA call failed.
extern "C" __attribute__((visibility("default"))) int hbm_stream_gbs(int kind, double* gbs) {
    if (kind < 0 || kind > 2 || !gbs) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    const size_t bytes = kind == 2 ? ((size_t)2 << 30) : ((size_t)4 << 30);
    const size_t n16 = bytes / 16;
    uint4 *a = nullptr, *b = nullptr;
    Out* o = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int rc = 0;
    if (cudaMalloc(&a, bytes) != cudaSuccess) rc = 1;
    if (!rc && kind == 2 && cudaMalloc(&b, bytes) != cudaSuccess) rc = 1;
    if (!rc && cudaMalloc(&o, sizeof(Out)) != cudaSuccess) rc = 1;
    if (!rc && cudaMemset(a, 1, bytes) != cudaSuccess) rc = 1;
    if (!rc && (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)) rc = 1;
    float best = 1e30f;
    const int grid = sms * 8;
    for (int rep = 0; rep < 6 && !rc; ++rep) {
        if (cudaEventRecord(e0) != cudaSuccess) { rc = 1; break; }
        if (kind == 0) hbm_read_kernel<<<grid, 256>>>(a, n16, o);
        else if (kind == 1) hbm_write_kernel<<<grid, 256>>>(a, n16, (uint32_t)rep);
        else hbm_copy_kernel<<<grid, 256>>>(a, b, n16);
        if (cudaEventRecord(e1) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess) { rc = 1; break; }
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) { rc = 1; break; }
        if (rep > 0 && ms < best) best = ms;
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(a);
    cudaFree(b);
    cudaFree(o);
    if (rc || best >= 1e29f) return 1;
    *gbs = (double)(kind == 2 ? 2 * bytes : bytes) / (best * 1e-3) / 1e9;
    return 0;
}
