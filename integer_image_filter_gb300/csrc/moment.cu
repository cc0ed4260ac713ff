// moment.cu -- sums of the reference and distorted luma samples and of their
// squares for n picture pairs in ONE launch.
//
// "ADR-1392: CUDA motion, PSNR and moment kernels add one atomic per block,
// the motion SAD filters separably, and PSNR selects its plane with constant
// indices": Decision 6 (the moment kernel follows the PSNR layout and keeps
// four accumulators -- the reference and distorted sums and sums of squares --
// each added once per block), Context (exact 64-bit integer sums, so the order
// of the adds does not matter).
//
// GB300 form: each CTA owns a band of rows of one pair's luma, streamed with
// 16-byte non-allocating loads, four loads of each picture in flight per
// thread.  8-bit sums and squares are 4-way byte dot products (against ones
// and against the word itself), exact in 32 bits for a group of vectors and
// widened to 64 bits once per group.
#include "motion_common.cuh"
#include "motion_internal.h"

namespace mg {

constexpr int MOM_NT = 256;
constexpr int MOM_UNROLL = 4;

struct Mom {
    unsigned long long s_r = 0, s_d = 0, q_r = 0, q_d = 0;
};

// 16 bytes of 8-bit samples: sum and sum of squares, 32-bit partials (at most
// 16 * 255 and 16 * 255^2 per vector).
__device__ __forceinline__ void mom16_u8(const uint4 v, uint32_t& s, uint32_t& q) {
    s = __dp4a(v.x, 0x01010101u, s);
    q = __dp4a(v.x, v.x, q);
    s = __dp4a(v.y, 0x01010101u, s);
    q = __dp4a(v.y, v.y, q);
    s = __dp4a(v.z, 0x01010101u, s);
    q = __dp4a(v.z, v.z, q);
    s = __dp4a(v.w, 0x01010101u, s);
    q = __dp4a(v.w, v.w, q);
}
// 8 little-endian 16-bit samples: the sum fits 32 bits, the squares take 64.
__device__ __forceinline__ void mom2_u16(uint32_t w, uint32_t& s, unsigned long long& q) {
    const uint32_t lo = w & 0xffffu, hi = w >> 16;
    s += lo + hi;
    q += (unsigned long long)lo * lo + (unsigned long long)hi * hi;
}
__device__ __forceinline__ void mom16_u16(const uint4 v, uint32_t& s, unsigned long long& q) {
    mom2_u16(v.x, s, q);
    mom2_u16(v.y, s, q);
    mom2_u16(v.z, s, q);
    mom2_u16(v.w, s, q);
}

template <typename Pix>
__global__ void __launch_bounds__(MOM_NT) moment_kernel(const MomentArgs a, int rows_per_block,
                                                        int blocks_per_pair, int vec) {
    constexpr int S = sizeof(Pix);
    const int pair = blockIdx.x / blocks_per_pair;
    const int y0 = (blockIdx.x - pair * blocks_per_pair) * rows_per_block;
    const int rows = min(a.h - y0, rows_per_block);
    const uint8_t* r = a.ref + (long long)pair * a.stride;
    const uint8_t* d = a.dist + (long long)pair * a.stride;
    Mom m;
    int scalar_from = 0;  // first column handled sample by sample
    if (vec) {
        const int nvec = (a.w * S) / 16;
        const int total = rows * nvec;
        int i = threadIdx.x;
        for (; i + (MOM_UNROLL - 1) * MOM_NT < total; i += MOM_UNROLL * MOM_NT) {
            uint4 rv[MOM_UNROLL], dv[MOM_UNROLL];
#pragma unroll
            for (int u = 0; u < MOM_UNROLL; ++u) {
                const int j = i + u * MOM_NT;
                const int y = j / nvec, v = j - y * nvec;
                rv[u] = ldg_stream16(r + (long long)(y0 + y) * a.pitch + 16LL * v);
                dv[u] = ldg_stream16(d + (long long)(y0 + y) * a.pitch + 16LL * v);
            }
            uint32_t sr = 0, sd = 0;
            if constexpr (S == 1) {
                uint32_t qr = 0, qd = 0;   // <= 4 * 16 * 255^2
#pragma unroll
                for (int u = 0; u < MOM_UNROLL; ++u) {
                    mom16_u8(rv[u], sr, qr);
                    mom16_u8(dv[u], sd, qd);
                }
                m.q_r += qr;
                m.q_d += qd;
            } else {
#pragma unroll
                for (int u = 0; u < MOM_UNROLL; ++u) {
                    mom16_u16(rv[u], sr, m.q_r);
                    mom16_u16(dv[u], sd, m.q_d);
                }
            }
            m.s_r += sr;
            m.s_d += sd;
        }
        for (; i < total; i += MOM_NT) {
            const int y = i / nvec, v = i - y * nvec;
            const uint4 rv = ldg_stream16(r + (long long)(y0 + y) * a.pitch + 16LL * v);
            const uint4 dv = ldg_stream16(d + (long long)(y0 + y) * a.pitch + 16LL * v);
            uint32_t sr = 0, sd = 0;
            if constexpr (S == 1) {
                uint32_t qr = 0, qd = 0;
                mom16_u8(rv, sr, qr);
                mom16_u8(dv, sd, qd);
                m.q_r += qr;
                m.q_d += qd;
            } else {
                mom16_u16(rv, sr, m.q_r);
                mom16_u16(dv, sd, m.q_d);
            }
            m.s_r += sr;
            m.s_d += sd;
        }
        scalar_from = nvec * 16 / S;
    }
    const int tail = a.w - scalar_from;
    if (tail > 0) {
        for (int i = threadIdx.x; i < rows * tail; i += MOM_NT) {
            const int y = i / tail, x = scalar_from + (i - y * tail);
            const unsigned long long p =
                *reinterpret_cast<const Pix*>(r + (long long)(y0 + y) * a.pitch + (long long)x * S);
            const unsigned long long q =
                *reinterpret_cast<const Pix*>(d + (long long)(y0 + y) * a.pitch + (long long)x * S);
            m.s_r += p;
            m.s_d += q;
            m.q_r += p * p;
            m.q_d += q * q;
        }
    }
    // block reduction: warp sums through shared memory, then threads 0..3 each
    // add one accumulator's block sum with one atomic (ADR-1392 Decision 6)
    __shared__ unsigned long long part[4][MOM_NT / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    m.s_r = warp_sum(m.s_r);
    m.s_d = warp_sum(m.s_d);
    m.q_r = warp_sum(m.q_r);
    m.q_d = warp_sum(m.q_d);
    if (lane == 0) {
        part[0][warp] = m.s_r;
        part[1][warp] = m.s_d;
        part[2][warp] = m.q_r;
        part[3][warp] = m.q_d;
    }
    __syncthreads();
    if (warp == 0 && rows > 0) {
        if (lane < 4) {
            unsigned long long t = 0;
#pragma unroll
            for (int k = 0; k < MOM_NT / 32; ++k) t += part[lane][k];
            atomicAdd(a.out + 4LL * pair + lane, t);
        }
    }
}

cudaError_t launch_moment(const MomentArgs& a, cudaStream_t s, int sm_count, int* launches) {
    if (a.n <= 0) return cudaSuccess;
    const int S = a.bpc == 8 ? 1 : 2;
    const int vec = (((uintptr_t)a.ref | (uintptr_t)a.dist | (uintptr_t)a.pitch) % 16 == 0) &&
                    (a.n == 1 || a.stride % 16 == 0);
    // rows per block: about 8 16-byte vectors of each picture per thread, but
    // never so many that the launch has fewer than 4 blocks per SM
    const int vec_per_row = (a.w * S + 15) / 16;
    int rpb = (MOM_NT * 8 + vec_per_row - 1) / vec_per_row;
    if (rpb < 1) rpb = 1;
    const long long want_blocks = 4LL * sm_count;
    if ((long long)a.n * ((a.h + rpb - 1) / rpb) < want_blocks) {
        const long long per_pair = (want_blocks + a.n - 1) / a.n;
        rpb = (int)((a.h + per_pair - 1) / per_pair);
        if (rpb < 1) rpb = 1;
    }
    const int blocks_per_pair = (a.h + rpb - 1) / rpb;
    const long long grid = (long long)a.n * blocks_per_pair;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    *launches += 1;
    if (S == 1)
        moment_kernel<uint8_t><<<(unsigned)grid, MOM_NT, 0, s>>>(a, rpb, blocks_per_pair, vec);
    else
        moment_kernel<uint16_t><<<(unsigned)grid, MOM_NT, 0, s>>>(a, rpb, blocks_per_pair, vec);
    return cudaGetLastError();
}

}  // namespace mg
