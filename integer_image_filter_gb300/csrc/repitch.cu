// repitch.cu -- copies planes whose rows the Tensor Memory Accelerator cannot
// address (a base, row pitch or frame stride that is not a multiple of 16
// bytes) into a library-owned scratch with 16-byte-aligned rows, so that the
// motion kernel always streams its tiles with TMA boxes.
//
// One warp copies one row: lane k writes 16-byte chunks k, k + 32, ... of the
// destination row with one aligned store each, and reads the source bytes of
// the chunk with the widest loads the source alignment allows (G bytes, G the
// largest power of two up to 16 that divides every source base, pitch and
// stride), so no load leaves the source row.  The ragged last chunk of a row
// is read byte by byte; destination bytes past the row's samples are zero.
// The copy is bandwidth-bound: every source byte is read once and written once.
#include "bounds_check.cuh"
#include "motion_internal.h"

namespace mg {

namespace {

constexpr int RP_NT = 256;   // threads per CTA (8 rows in flight)

template <int G>
__device__ __forceinline__ uint4 load16(const uint8_t* p, [[maybe_unused]] Span src) {
    uint4 o;
    if constexpr (G == 16) {
        o = MG_LD(reinterpret_cast<const uint4*>(p), src.p, src.n);
    } else if constexpr (G == 8) {
        const uint2 a = MG_LD(reinterpret_cast<const uint2*>(p), src.p, src.n);
        const uint2 b = MG_LD(reinterpret_cast<const uint2*>(p + 8), src.p, src.n);
        o = make_uint4(a.x, a.y, b.x, b.y);
    } else if constexpr (G == 4) {
        const uint32_t* q = reinterpret_cast<const uint32_t*>(p);
        o = make_uint4(MG_LD(q, src.p, src.n), MG_LD(q + 1, src.p, src.n), MG_LD(q + 2, src.p, src.n),
                       MG_LD(q + 3, src.p, src.n));
    } else if constexpr (G == 2) {
        const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (uint32_t)MG_LD(q + 2 * i, src.p, src.n) | ((uint32_t)MG_LD(q + 2 * i + 1, src.p, src.n) << 16);
        o = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (uint32_t)MG_LD(p + 4 * i, src.p, src.n) | ((uint32_t)MG_LD(p + 4 * i + 1, src.p, src.n) << 8) |
                   ((uint32_t)MG_LD(p + 4 * i + 2, src.p, src.n) << 16) |
                   ((uint32_t)MG_LD(p + 4 * i + 3, src.p, src.n) << 24);
        o = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return o;
}

// The plane of index i, selected with constant indices (no runtime index into
// the kernel-parameter array, which would copy it to local memory).
__device__ __forceinline__ RepitchPlane plane_at(const RepitchArgs& a, int i) {
    return i == 0 ? a.p[0] : i == 1 ? a.p[1] : i == 2 ? a.p[2] : i == 3 ? a.p[3] : i == 4 ? a.p[4] : a.p[5];
}

template <int G>
__global__ void __launch_bounds__(RP_NT) repitch_kernel(const RepitchArgs a) {
    MG_BC_BEGIN(a.err);
#if MG_BOUNDS_CHECK
    __syncthreads();
#endif
    const int lane = threadIdx.x & 31;
    int rows_total = 0;
#pragma unroll
    for (int i = 0; i < kRepitchMaxPlanes; ++i)
        if (i < a.planes) rows_total += plane_at(a, i).rows;
    const long long items = (long long)a.n * rows_total;
    const long long warps = (long long)gridDim.x * (RP_NT / 32);
    for (long long it = (long long)blockIdx.x * (RP_NT / 32) + (threadIdx.x >> 5); it < items; it += warps) {
        // item -> (frame, plane, row)
        const int f = (int)(it / rows_total);
        int r = (int)(it - (long long)f * rows_total);
        int pi = 0;
        while (pi + 1 < a.planes && r >= plane_at(a, pi).rows) {
            r -= plane_at(a, pi).rows;
            ++pi;
        }
        const RepitchPlane P = plane_at(a, pi);
        [[maybe_unused]] const Span src{P.src, (size_t)plane_span(a.n, P.stride, P.rows, P.pitch, P.row_bytes, 1)};
        [[maybe_unused]] const Span dst{P.dst, (size_t)a.n * (size_t)P.dstride};
        const uint8_t* s = P.src + (long long)f * P.stride + (long long)r * P.pitch;
        uint8_t* d = P.dst + (long long)f * P.dstride + (long long)r * P.dpitch;
        const int chunks = (int)(P.dpitch / 16);
        for (int k = lane; k < chunks; k += 32) {
            const int b0 = 16 * k;
            uint4 o;
            if (b0 + 16 <= P.row_bytes) {
                o = load16<G>(s + b0, src);
            } else {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
                for (int i = 0; b0 + i < P.row_bytes; ++i)
                    w[i >> 2] |= (uint32_t)MG_LD(s + b0 + i, src.p, src.n) << (8 * (i & 3));
                o = make_uint4(w[0], w[1], w[2], w[3]);
            }
            MG_ST(reinterpret_cast<uint4*>(d + b0), o, dst.p, dst.n);
        }
    }
}

}  // namespace

int repitch_granule(const RepitchArgs& a) {
    unsigned long long bits = 16;
    for (int p = 0; p < a.planes; ++p)
        bits |= (unsigned long long)(uintptr_t)a.p[p].src | (unsigned long long)a.p[p].pitch |
                (a.n > 1 ? (unsigned long long)a.p[p].stride : 0ull);
    return (int)(bits & (~bits + 1));   // lowest set bit, at most 16
}

cudaError_t launch_repitch(const RepitchArgs& a, cudaStream_t s, int sm_count, int* launches) {
    if (a.n <= 0 || a.planes <= 0) return cudaSuccess;
    long long rows = 0;
    for (int p = 0; p < a.planes; ++p) rows += a.p[p].rows;
    const long long items = rows * a.n;
    long long blocks = (items + RP_NT / 32 - 1) / (RP_NT / 32);
    const long long cap = 8LL * (sm_count > 0 ? sm_count : 1);
    if (blocks > cap) blocks = cap;
    *launches += 1;
    switch (repitch_granule(a)) {
        case 16: repitch_kernel<16><<<(unsigned)blocks, RP_NT, 0, s>>>(a); break;
        case 8: repitch_kernel<8><<<(unsigned)blocks, RP_NT, 0, s>>>(a); break;
        case 4: repitch_kernel<4><<<(unsigned)blocks, RP_NT, 0, s>>>(a); break;
        case 2: repitch_kernel<2><<<(unsigned)blocks, RP_NT, 0, s>>>(a); break;
        default: repitch_kernel<1><<<(unsigned)blocks, RP_NT, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

}  // namespace mg
