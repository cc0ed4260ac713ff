// tile_geometry.cuh -- the output tile shared by the motion kernels: sizes of
// the staged regions and the small per-sample helpers of the 5-tap passes.
#pragma once

#include "bounds_check.cuh"
#include "motion_common.cuh"
#include "motion_internal.h"

namespace mg {

constexpr int TW = kTileW;         // output tile width, samples (128)
constexpr int TH = kTileH;         // output tile height, rows (32)
constexpr int NT = 256;            // threads per CTA
constexpr int NW = NT / 32;
constexpr int SVW = TW + 8;        // V tile row pitch (uint32); col j <-> x = x0 - 4 + j

// Staged regions of one frame (or picture pair) for one tile.  The luma box
// spans rows y0-2 .. y0+TH+1 and columns x0-HX .. x0+TW+HX-1 (HX = 16 bytes of
// samples, so every box starts on a 16-byte boundary); the fused form adds the
// distorted luma tile and the four 4:2:0 chroma tiles (ref U, dist U, ref V,
// dist V).  Every region is a multiple of 128 bytes.
template <typename Pix, int THT = TH>
struct Geo {
    static constexpr int S = sizeof(Pix);
    static constexpr int HX = 16 / S;
    static constexpr int RAW_W = TW + 2 * HX;
    static constexpr int RAW_ROWS = THT + 4;
    static constexpr int RAW_BYTES = RAW_ROWS * RAW_W * S;
    static constexpr int DIST_BYTES = THT * TW * S;
    static constexpr int CW = TW / 2, CH = THT / 2;
    static constexpr int C_BYTES = CH * CW * S;
    static constexpr int STAGE_MOTION = RAW_BYTES;
    static constexpr int STAGE_FUSED = RAW_BYTES + DIST_BYTES + 4 * C_BYTES;
    static constexpr int SV_BYTES = THT * SVW * 4;
    static_assert(RAW_BYTES % 128 == 0 && DIST_BYTES % 128 == 0 && C_BYTES % 128 == 0,
                  "regions must keep 128-byte alignment");
};

template <typename Pix> struct SseAcc;
template <> struct SseAcc<uint8_t> { using T = uint32_t; };            // 4096 * 255^2 < 2^32
template <> struct SseAcc<uint16_t> { using T = unsigned long long; };

__device__ __forceinline__ void unpack4(const uint8_t* p, uint32_t (&o)[4]) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    o[0] = w & 0xffu; o[1] = (w >> 8) & 0xffu; o[2] = (w >> 16) & 0xffu; o[3] = w >> 24;
}
__device__ __forceinline__ void unpack4(const uint16_t* p, uint32_t (&o)[4]) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    o[0] = w.x & 0xffffu; o[1] = w.x >> 16; o[2] = w.y & 0xffffu; o[3] = w.y >> 16;
}

// unpack4 of 4 samples that must lie inside [lo, lo + bytes) (checked build)
template <typename Pix>
__device__ __forceinline__ void unpack4_in(const Pix* p, const void* lo, size_t bytes, uint32_t (&o)[4]) {
    if (MG_OK(p, 4 * sizeof(Pix), lo, bytes))
        unpack4(p, o);
    else
        o[0] = o[1] = o[2] = o[3] = 0;
}

// One 5-tap pass with symmetric taps: (t0 (a + e) + t1 (b + d) + t2 c + rnd) >> sh.
__device__ __forceinline__ uint32_t vtap(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                         uint32_t e, uint32_t rnd, int sh) {
    return (kT0 * (a + e) + kT1 * (b + d) + kT2 * c + rnd) >> sh;
}

// motion_v2 helpers.  The blur of prev - cur is linear up to its roundings, so
// the vertical sum of the difference is the difference of the unrounded
// vertical sums X = t0 (a + e) + t1 (b + d) + t2 c of the two frames (exact:
// X < 2^32 for samples < 2^16); it is then rounded with a floor shift.
__device__ __forceinline__ uint32_t vsum(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                         uint32_t e) {
    return kT0 * (a + e) + kT1 * (b + d) + kT2 * c;
}
// floor((xp - x + rnd) / 2^sh): 32-bit for 8-bit samples (|xp - x| < 2^24),
// 64-bit above (33 bits with sign).
template <typename Pix>
__device__ __forceinline__ int vdiff(uint32_t xp, uint32_t x, uint32_t rnd, int sh) {
    if constexpr (sizeof(Pix) == 1)
        return ((int)xp - (int)x + (int)rnd) >> sh;
    else
        return (int)(((long long)xp - (long long)x + (long long)rnd) >> sh);
}
// The horizontal pass on signed V: the same window sums as horizontal_quad,
// the products and the rounding in 64 bits (|sum| < 2^32 + 2^15 needs 33
// bits with sign), floor shift >> 16.
__device__ __forceinline__ void horizontal_quad_signed(const int (&wv)[12], int (&b)[4]) {
    int w3 = wv[3] + wv[4] + wv[5];
    int w5 = w3 + wv[2] + wv[6];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i > 0) {
            w3 = w3 + wv[5 + i] - wv[2 + i];
            w5 = w5 + wv[6 + i] - wv[1 + i];
        }
        const long long t = (long long)kT0 * w5 + (long long)(kT1 - kT0) * w3 +
                            (long long)(kT2 - kT1) * wv[4 + i] + 32768LL;
        b[i] = (int)(t >> 16);
    }
}

}  // namespace mg
