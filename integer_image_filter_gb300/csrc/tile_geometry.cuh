// tile_geometry.cuh -- the output tile shared by the motion kernels: sizes of
// the staged regions and the small per-sample helpers of the 5-tap passes.
#pragma once

#include "motion_common.cuh"

namespace mg {

constexpr int TW = 128;            // output tile width, samples
constexpr int TH = 32;             // output tile height, rows
constexpr int NT = 256;            // threads per CTA
constexpr int NW = NT / 32;
constexpr int SVW = TW + 8;        // V tile row pitch (uint32); col j <-> x = x0 - 4 + j

// Staged regions of one frame (or picture pair) for one tile.  The luma box
// spans rows y0-2 .. y0+TH+1 and columns x0-HX .. x0+TW+HX-1 (HX = 16 bytes of
// samples, so every box starts on a 16-byte boundary); the fused form adds the
// distorted luma tile and the four 4:2:0 chroma tiles (ref U, dist U, ref V,
// dist V).  Every region is a multiple of 128 bytes.
template <typename Pix>
struct Geo {
    static constexpr int S = sizeof(Pix);
    static constexpr int HX = 16 / S;
    static constexpr int RAW_W = TW + 2 * HX;
    static constexpr int RAW_ROWS = TH + 4;
    static constexpr int RAW_BYTES = RAW_ROWS * RAW_W * S;
    static constexpr int DIST_BYTES = TH * TW * S;
    static constexpr int CW = TW / 2, CH = TH / 2;
    static constexpr int C_BYTES = CH * CW * S;
    static constexpr int STAGE_MOTION = RAW_BYTES;
    static constexpr int STAGE_FUSED = RAW_BYTES + DIST_BYTES + 4 * C_BYTES;
    static constexpr int SV_BYTES = TH * SVW * 4;
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

// One 5-tap pass with symmetric taps: (t0 (a + e) + t1 (b + d) + t2 c + rnd) >> sh.
__device__ __forceinline__ uint32_t vtap(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                         uint32_t e, uint32_t rnd, int sh) {
    return (kT0 * (a + e) + kT1 * (b + d) + kT2 * c + rnd) >> sh;
}

}  // namespace mg
