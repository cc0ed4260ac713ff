// psnr_sse.cu -- per-plane squared-error sums SSE = sum (ref - dist)^2 for n
// picture pairs x (1 or 3) planes in ONE launch.
//
// "ADR-1392: CUDA motion, PSNR and moment kernels add one atomic per block,
// the motion SAD filters separably, and PSNR selects its plane with constant
// indices": Context (exact 64-bit sums, order-independent), Decision 1 (one
// atomic per block), Decision 3 (the plane is chosen by a branch over constant
// indices, never by indexing kernel parameters with a runtime value).
//
// GB300 form: each CTA owns a band of rows of one plane of one pair; the band's
// samples are streamed with 16-byte non-allocating loads, four loads in flight
// per thread; 8-bit squared differences use the byte-SIMD |a-b| followed by a
// 4-way dot product, exact in 32 bits per vector.
#include "motion_common.cuh"
#include "motion_internal.h"

namespace mg {

constexpr int SSE_NT = 256;
constexpr int SSE_UNROLL = 4;

// Squared differences of 16 bytes of samples.
__device__ __forceinline__ unsigned long long sse16_u8(const uint4 r, const uint4 d) {
    uint32_t s = 0;
    uint32_t t = __vabsdiffu4(r.x, d.x); s = __dp4a(t, t, s);
    t = __vabsdiffu4(r.y, d.y); s = __dp4a(t, t, s);
    t = __vabsdiffu4(r.z, d.z); s = __dp4a(t, t, s);
    t = __vabsdiffu4(r.w, d.w); s = __dp4a(t, t, s);
    return s;  // <= 16 * 255^2
}
__device__ __forceinline__ unsigned long long sq2_u16(uint32_t r, uint32_t d) {
    const uint32_t t = __vabsdiffu2(r, d);
    const unsigned long long lo = t & 0xffffu, hi = t >> 16;
    return lo * lo + hi * hi;
}
__device__ __forceinline__ unsigned long long sse16_u16(const uint4 r, const uint4 d) {
    return sq2_u16(r.x, d.x) + sq2_u16(r.y, d.y) + sq2_u16(r.z, d.z) + sq2_u16(r.w, d.w);
}

template <typename Pix>
__global__ void __launch_bounds__(SSE_NT) sse_kernel(const SseArgs a, int rows_per_block,
                                                     int blocks_y, int blocks_c, int vec) {
    constexpr int S = sizeof(Pix);
    const int per_pair = blocks_y + (a.planes == 3 ? 2 * blocks_c : 0);
    const int pair = blockIdx.x / per_pair;
    int rem = blockIdx.x - pair * per_pair;
    int plane, chunk;
    if (rem < blocks_y) {
        plane = 0;
        chunk = rem;
    } else {
        rem -= blocks_y;
        plane = rem < blocks_c ? 1 : 2;
        chunk = plane == 1 ? rem : rem - blocks_c;
    }
    // constant-index plane selection: no runtime index into the arguments
    const uint8_t* r;
    const uint8_t* d;
    long long rp, dp;
    int w, h;
    if (plane == 0) {
        r = a.ref_y + (long long)pair * a.stride_y;
        d = a.dist_y + (long long)pair * a.stride_y;
        rp = a.ref_pitch_y; dp = a.dist_pitch_y; w = a.w; h = a.h;
    } else if (plane == 1) {
        r = a.ref_u + (long long)pair * a.stride_uv;
        d = a.dist_u + (long long)pair * a.stride_uv;
        rp = a.pitch_uv; dp = a.pitch_uv; w = a.cw; h = a.ch;
    } else {
        r = a.ref_v + (long long)pair * a.stride_uv;
        d = a.dist_v + (long long)pair * a.stride_uv;
        rp = a.pitch_uv; dp = a.pitch_uv; w = a.cw; h = a.ch;
    }
    const int y0 = chunk * rows_per_block;
    const int rows = min(h - y0, rows_per_block);
    unsigned long long acc = 0;
    int scalar_from = 0;  // first column handled sample by sample
    if (vec) {
        const int nvec = (w * S) / 16;
        const int total = rows * nvec;
        int i = threadIdx.x;
        for (; i + (SSE_UNROLL - 1) * SSE_NT < total; i += SSE_UNROLL * SSE_NT) {
            uint4 rv[SSE_UNROLL], dv[SSE_UNROLL];
#pragma unroll
            for (int u = 0; u < SSE_UNROLL; ++u) {
                const int j = i + u * SSE_NT;
                const int y = j / nvec, v = j - y * nvec;
                rv[u] = ldg_stream16(r + (long long)(y0 + y) * rp + 16LL * v);
                dv[u] = ldg_stream16(d + (long long)(y0 + y) * dp + 16LL * v);
            }
#pragma unroll
            for (int u = 0; u < SSE_UNROLL; ++u)
                acc += (S == 1) ? sse16_u8(rv[u], dv[u]) : sse16_u16(rv[u], dv[u]);
        }
        for (; i < total; i += SSE_NT) {
            const int y = i / nvec, v = i - y * nvec;
            const uint4 rv = ldg_stream16(r + (long long)(y0 + y) * rp + 16LL * v);
            const uint4 dv = ldg_stream16(d + (long long)(y0 + y) * dp + 16LL * v);
            acc += (S == 1) ? sse16_u8(rv, dv) : sse16_u16(rv, dv);
        }
        scalar_from = nvec * 16 / S;
    }
    const int tail = w - scalar_from;
    if (tail > 0) {
        for (int i = threadIdx.x; i < rows * tail; i += SSE_NT) {
            const int y = i / tail, x = scalar_from + (i - y * tail);
            const long long ee =
                (long long)*reinterpret_cast<const Pix*>(r + (long long)(y0 + y) * rp + (long long)x * S) -
                (long long)*reinterpret_cast<const Pix*>(d + (long long)(y0 + y) * dp + (long long)x * S);
            acc += (unsigned long long)(ee * ee);
        }
    }
    // one atomic per block (ADR-1392 Decision 1)
    __shared__ unsigned long long part[SSE_NT / 32];
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        unsigned long long t = threadIdx.x < SSE_NT / 32 ? part[threadIdx.x] : 0ull;
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0 && rows > 0)
            atomicAdd(a.sse_out + (long long)pair * a.planes + plane, t);
    }
}

cudaError_t launch_sse(const SseArgs& a, cudaStream_t s, int sm_count, int* launches) {
    if (a.n <= 0) return cudaSuccess;
    const int S = a.bpc == 8 ? 1 : 2;
    const int vec =
        (((uintptr_t)a.ref_y | (uintptr_t)a.dist_y | (uintptr_t)a.ref_pitch_y | (uintptr_t)a.dist_pitch_y) % 16 == 0) &&
        (a.n == 1 || a.stride_y % 16 == 0) &&
        (a.planes == 1 || ((((uintptr_t)a.ref_u | (uintptr_t)a.dist_u | (uintptr_t)a.ref_v |
                             (uintptr_t)a.dist_v | (uintptr_t)a.pitch_uv) % 16 == 0) &&
                           (a.n == 1 || a.stride_uv % 16 == 0)));
    // rows per block: about 8 16-byte vectors per thread for the luma plane,
    // but never so many that one pair gives fewer blocks than SMs
    const int vec_per_row = (a.w * S + 15) / 16;
    int rpb = (SSE_NT * 8 + vec_per_row - 1) / vec_per_row;
    if (rpb < 1) rpb = 1;
    const long long want_blocks = 4LL * sm_count;
    if ((long long)a.n * ((a.h + rpb - 1) / rpb) < want_blocks) {
        long long per_pair = (want_blocks + a.n - 1) / a.n;
        rpb = (int)((a.h + per_pair - 1) / per_pair);
        if (rpb < 1) rpb = 1;
    }
    const int blocks_y = (a.h + rpb - 1) / rpb;
    const int blocks_c = a.planes == 3 ? (a.ch + rpb - 1) / rpb : 0;
    const long long grid = (long long)a.n * (blocks_y + 2LL * blocks_c);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    *launches += 1;
    if (S == 1)
        sse_kernel<uint8_t><<<(unsigned)grid, SSE_NT, 0, s>>>(a, rpb, blocks_y, blocks_c, vec);
    else
        sse_kernel<uint16_t><<<(unsigned)grid, SSE_NT, 0, s>>>(a, rpb, blocks_y, blocks_c, vec);
    return cudaGetLastError();
}

}  // namespace mg
