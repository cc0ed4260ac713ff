// motion_tma.cu -- the batched motion kernel (blur + SAD against the previous
// frame), optionally fused with the per-plane SSE of 4:2:0 pairs, fed by the
// Tensor Memory Accelerator.
//
// Structure (GB300 / sm_103a):
//  * One CTA owns a TW x TH output tile (128 x 32; 128 x 16 for motion-only
//    launches that fit in one wave) and walks the batch of frames (or one
//    chunk of it) in time order; B_prev of its tile stays in registers, so
//    every frame is read from HBM once ("Making it fast: three rounds on one
//    pipeline", Round 1 -- one kernel over all frames).
//  * Thread 0 keeps STAGES frames in flight: for each frame it issues 3-D tiled
//    TMA loads (cp.async.bulk.tensor, x / y / frame coordinates) of the luma
//    box with its 2-row and 16-byte halo -- and, fused, the distorted luma
//    tile and the four chroma tiles -- completing on that stage's mbarrier.
//    Out-of-frame parts of a box arrive zero-filled; tiles on the frame border
//    read rows through a per-CTA table of mirrored rows (i<0 -> -i,
//    i>=n -> 2n-i-2) and mirror the V columns of their own rows, so no tile
//    takes a sample-by-sample path and no block barrier is left in the frame
//    loop.  Full tiles on the left or right edge need only mirrored halo
//    columns: their halo lanes read the mirrored columns inside the frame, and
//    they run the interior copy of the frame loop.
//  * Blocks take the border tiles (top and bottom tile rows, a partial last
//    column) of every chunk first and the interior tiles after them in
//    row-major order (tile_of_block): the two kinds run different copies of
//    the frame loop, and an SM that runs both at once misses in its
//    instruction cache; adjacent interior tiles run together and share their
//    halos in L2.
//  * Separable blur: the vertical 5-tap pass once per sample (rounded >> bpc)
//    into a shared V tile, then the horizontal 5-tap pass (rounded >> 16)
//    ("ADR-1392: CUDA motion, PSNR and moment kernels add one atomic per
//    block, the motion SAD filters separably, ...", Decision 4).
//  * Per frame each warp reduces its partial sums with one warp-reduce
//    instruction and keeps them in lane (frame mod 32); every 32 frames the
//    warps add their lanes into the block's window sums in shared memory and
//    the last warp adds each accumulator of each frame to its 64-bit output
//    with ONE atomic (same page, Decision 1; integer sums are
//    order-independent, so the result is exact -- Context).
//  * Every mbarrier wait is bounded: on time-out a warp raises the device
//    error word and leaves instead of spinning; thread 0 waits (bounded) for
//    the copies it issued before the block exits.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <type_traits>

#include "motion_internal.h"
#include "tile_geometry.cuh"

namespace mg {

constexpr long long kWaitCycles = 1LL << 31;  // default wait bound: about one second

// The vertical 5-tap pass for one warp: 4 output rows x 128 columns, fed by 8
// staged rows at element offsets ro(0..7) from the lane's column src (lane =
// quad of 4 columns); result V (uint32) into the warp's own rows of sV, and
// the 4 centre-row words (the reference luma of the warp's output rows) for
// the squared error.  8-bit samples use byte-pair dot products: rows are
// interleaved two at a time so that one dp2a applies two taps to two rows of
// one column (exact: sums stay below 2^24).  `box` and `vrows` are the staged
// box and the warp's V rows (the bounds-checked build checks every access
// against them).
template <typename RowOff>
__device__ __forceinline__ void vertical_quad(const uint8_t* src, RowOff ro, uint32_t* dst,
                                              uint32_t rnd, int sh, uint32_t (&center)[4],
                                              [[maybe_unused]] Span box, [[maybe_unused]] Span vrows) {
    uint32_t wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) wv[i] = MG_LD(reinterpret_cast<const uint32_t*>(src + ro(i)), box.p, box.n);
#pragma unroll
    for (int i = 0; i < 4; ++i) center[i] = wv[i + 2];
    uint32_t lo[7], hi[7];  // rows (i, i+1): columns 0,1 in lo, columns 2,3 in hi
#pragma unroll
    for (int i = 0; i < 7; ++i) {
        lo[i] = __byte_perm(wv[i], wv[i + 1], 0x5140);
        hi[i] = __byte_perm(wv[i], wv[i + 1], 0x7362);
    }
    constexpr uint32_t T01 = kT0 | (kT1 << 16);   // taps of rows j, j+1
    constexpr uint32_t T23 = kT2 | (kT1 << 16);   // rows j+2, j+3 (t3 = t1)
    constexpr uint32_t T_4 = kT0 << 16;            // row j+4 as the upper row of (j+3, j+4)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 o;
        o.x = __dp2a_lo(T01, lo[j], __dp2a_lo(T23, lo[j + 2], __dp2a_lo(T_4, lo[j + 3], rnd))) >> sh;
        o.y = __dp2a_hi(T01, lo[j], __dp2a_hi(T23, lo[j + 2], __dp2a_hi(T_4, lo[j + 3], rnd))) >> sh;
        o.z = __dp2a_lo(T01, hi[j], __dp2a_lo(T23, hi[j + 2], __dp2a_lo(T_4, hi[j + 3], rnd))) >> sh;
        o.w = __dp2a_hi(T01, hi[j], __dp2a_hi(T23, hi[j + 2], __dp2a_hi(T_4, hi[j + 3], rnd))) >> sh;
        MG_ST(reinterpret_cast<uint4*>(dst + j * SVW), o, vrows.p, vrows.n);
    }
}
// The vertical pass of all 8 of a warp's rows at once: 12 staged rows, each
// loaded and interleaved (or unpacked) once, 8 V rows into the warp's V rows.
template <typename RowOff>
__device__ __forceinline__ void vertical_oct(const uint8_t* src, RowOff ro, uint32_t* dst, uint32_t rnd,
                                             int sh, uint32_t (&center)[8], [[maybe_unused]] Span box,
                                             [[maybe_unused]] Span vrows) {
    uint32_t wv[12];
#pragma unroll
    for (int i = 0; i < 12; ++i) wv[i] = MG_LD(reinterpret_cast<const uint32_t*>(src + ro(i)), box.p, box.n);
#pragma unroll
    for (int i = 0; i < 8; ++i) center[i] = wv[i + 2];
    uint32_t lo[11], hi[11];
#pragma unroll
    for (int i = 0; i < 11; ++i) {
        lo[i] = __byte_perm(wv[i], wv[i + 1], 0x5140);
        hi[i] = __byte_perm(wv[i], wv[i + 1], 0x7362);
    }
    constexpr uint32_t T01 = kT0 | (kT1 << 16);
    constexpr uint32_t T23 = kT2 | (kT1 << 16);
    constexpr uint32_t T_4 = kT0 << 16;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint4 o;
        o.x = __dp2a_lo(T01, lo[j], __dp2a_lo(T23, lo[j + 2], __dp2a_lo(T_4, lo[j + 3], rnd))) >> sh;
        o.y = __dp2a_hi(T01, lo[j], __dp2a_hi(T23, lo[j + 2], __dp2a_hi(T_4, lo[j + 3], rnd))) >> sh;
        o.z = __dp2a_lo(T01, hi[j], __dp2a_lo(T23, hi[j + 2], __dp2a_lo(T_4, hi[j + 3], rnd))) >> sh;
        o.w = __dp2a_hi(T01, hi[j], __dp2a_hi(T23, hi[j + 2], __dp2a_hi(T_4, hi[j + 3], rnd))) >> sh;
        MG_ST(reinterpret_cast<uint4*>(dst + j * SVW), o, vrows.p, vrows.n);
    }
}
template <typename RowOff>
__device__ __forceinline__ void vertical_oct(const uint16_t* src, RowOff ro, uint32_t* dst, uint32_t rnd,
                                             int sh, uint32_t (&center)[8], [[maybe_unused]] Span box,
                                             [[maybe_unused]] Span vrows) {
    uint32_t p[12][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) center[i] = 0;   // 16-bit SSE reloads its samples
#pragma unroll
    for (int i = 0; i < 12; ++i) unpack4_in(src + ro(i), box.p, box.n, p[i]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint4 o;
        o.x = vtap(p[j][0], p[j + 1][0], p[j + 2][0], p[j + 3][0], p[j + 4][0], rnd, sh);
        o.y = vtap(p[j][1], p[j + 1][1], p[j + 2][1], p[j + 3][1], p[j + 4][1], rnd, sh);
        o.z = vtap(p[j][2], p[j + 1][2], p[j + 2][2], p[j + 3][2], p[j + 4][2], rnd, sh);
        o.w = vtap(p[j][3], p[j + 1][3], p[j + 2][3], p[j + 3][3], p[j + 4][3], rnd, sh);
        MG_ST(reinterpret_cast<uint4*>(dst + j * SVW), o, vrows.p, vrows.n);
    }
}
template <typename RowOff>
__device__ __forceinline__ void vertical_quad(const uint16_t* src, RowOff ro, uint32_t* dst,
                                              uint32_t rnd, int sh, uint32_t (&center)[4],
                                              [[maybe_unused]] Span box, [[maybe_unused]] Span vrows) {
    uint32_t p[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) unpack4_in(src + ro(i), box.p, box.n, p[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i) center[i] = 0;  // 16-bit SSE reloads its samples
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 o;
        o.x = vtap(p[j][0], p[j + 1][0], p[j + 2][0], p[j + 3][0], p[j + 4][0], rnd, sh);
        o.y = vtap(p[j][1], p[j + 1][1], p[j + 2][1], p[j + 3][1], p[j + 4][1], rnd, sh);
        o.z = vtap(p[j][2], p[j + 1][2], p[j + 2][2], p[j + 3][2], p[j + 4][2], rnd, sh);
        o.w = vtap(p[j][3], p[j + 1][3], p[j + 2][3], p[j + 3][3], p[j + 4][3], rnd, sh);
        MG_ST(reinterpret_cast<uint4*>(dst + j * SVW), o, vrows.p, vrows.n);
    }
}

// The horizontal 5-tap pass of 4 outputs from V at columns -2 .. +9 around
// the quad: t0 W5 + (t1 - t0) W3 + (t2 - t1) c with the 5- and 3-wide window
// sums slid one column at a time (the same integers as the tap-by-tap sum,
// kept exact in uint32; three-input adds leave the multiplier pipe to the
// three products).
__device__ __forceinline__ void horizontal_quad(const uint32_t (&wv)[12], uint32_t (&b)[4]) {
    uint32_t w3 = wv[3] + wv[4] + wv[5];
    uint32_t w5 = w3 + wv[2] + wv[6];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i > 0) {
            w3 = w3 + wv[5 + i] - wv[2 + i];
            w5 = w5 + wv[6 + i] - wv[1 + i];
        }
        b[i] = (kT0 * w5 + (kT1 - kT0) * w3 + (kT2 - kT1) * wv[4 + i] + 32768u) >> 16;
    }
}

// Unrounded vertical sums of 4 rows x 4 columns (8 staged rows from src).
template <typename RowOff>
__device__ __forceinline__ void vertical_sums(const uint8_t* src, RowOff ro, uint32_t (&x)[4][4],
                                              [[maybe_unused]] Span box) {
    uint32_t wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) wv[i] = MG_LD(reinterpret_cast<const uint32_t*>(src + ro(i)), box.p, box.n);
    uint32_t lo[7], hi[7];
#pragma unroll
    for (int i = 0; i < 7; ++i) {
        lo[i] = __byte_perm(wv[i], wv[i + 1], 0x5140);
        hi[i] = __byte_perm(wv[i], wv[i + 1], 0x7362);
    }
    constexpr uint32_t T01 = kT0 | (kT1 << 16);
    constexpr uint32_t T23 = kT2 | (kT1 << 16);
    constexpr uint32_t T_4 = kT0 << 16;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        x[j][0] = __dp2a_lo(T01, lo[j], __dp2a_lo(T23, lo[j + 2], __dp2a_lo(T_4, lo[j + 3], 0u)));
        x[j][1] = __dp2a_hi(T01, lo[j], __dp2a_hi(T23, lo[j + 2], __dp2a_hi(T_4, lo[j + 3], 0u)));
        x[j][2] = __dp2a_lo(T01, hi[j], __dp2a_lo(T23, hi[j + 2], __dp2a_lo(T_4, hi[j + 3], 0u)));
        x[j][3] = __dp2a_hi(T01, hi[j], __dp2a_hi(T23, hi[j + 2], __dp2a_hi(T_4, hi[j + 3], 0u)));
    }
}
template <typename RowOff>
__device__ __forceinline__ void vertical_sums(const uint16_t* src, RowOff ro, uint32_t (&x)[4][4],
                                              [[maybe_unused]] Span box) {
    uint32_t p[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) unpack4_in(src + ro(i), box.p, box.n, p[i]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            x[j][i] = vsum(p[j][i], p[j + 1][i], p[j + 2][i], p[j + 3][i], p[j + 4][i]);
}
// Thread layout: 4 warps per CTA; on a tile of THT = 32 rows each warp owns
// RPW = 8 output rows.  The motion-only kernels run the vertical pass of all
// 8 rows at once into the warp's 8-row V buffer (each of the 12 staged rows
// loaded and interleaved once), and so does the 8-bit fused kernel with 2
// stages; the 16-bit fused and the motion_v2 kernels run two halves of 4 rows
// through a 4-row V buffer.  Eight rows per warp halve the per-frame cost of
// stage waits, reductions and loop control per pixel against four, and the 32
// halo values of a warp's rows then occupy every lane once.  Motion-only
// launches that fit in one wave of 32-row tiles run tiles of THT = 16 rows
// instead (4 rows per warp, at most 72 registers, 7 CTAs per SM): twice the
// blocks, each warp with half the work per frame.
template <int THT>
struct ShapeT {
    static_assert(THT == 32 || THT == 16, "tiles are 32 or 16 rows high");
    static constexpr int RPW = THT / 4;           // output rows per warp
    static constexpr int NWK = THT / RPW;         // warps per CTA
    static constexpr int NTK = NWK * 32;          // threads per CTA
    // resident CTAs per SM: 4 (<= 128 registers) for 32-row tiles, 7 (<= 72) for 16
    static constexpr int MINB = THT == 32 ? 4 : 7;
    // V rows of one vertical pass: 8 for the motion-only and 8-bit fused
    // kernels on 32-row tiles; 4 (two halves of a warp's 8 rows, or all of its
    // 4) otherwise
    template <typename Pix, bool FUSED, bool V2>
    static constexpr int VR = (RPW == 8 && !V2 && !(FUSED && sizeof(Pix) == 2)) ? 8 : 4;
    template <typename Pix, bool FUSED, bool V2>
    static constexpr int SV = NWK * VR<Pix, FUSED, V2> * SVW * 4;  // V buffers, bytes
    static constexpr int CRW = 16 / NWK;          // chroma rows per warp
    static constexpr int SPL = RPW;               // chroma samples per lane and plane
    static constexpr int LPR = 64 / SPL;          // lanes per chroma row
};

// V2: motion_v2, the blur of prev - cur (see vsum / vdiff); FUSED is false then.
// THT: tile rows (32, or 16 for motion-only launches under one wave).
template <typename Pix, bool FUSED, int STAGES, bool V2, int THT>
__global__ void __launch_bounds__(ShapeT<THT>::NTK, ShapeT<THT>::MINB)
    motion_tma_kernel(const __grid_constant__ TmaMaps maps, const TileArgs a) {
    static_assert(!(FUSED && V2), "motion_v2 has no fused form");
    static_assert(!FUSED || THT == 32, "the fused form runs 32-row tiles");
    constexpr int TH = THT;
    using G = Geo<Pix, THT>;
    using SH = ShapeT<THT>;
    constexpr int NWK = SH::NWK, NTK = SH::NTK, RPW = SH::RPW;
    using Acc = typename SseAcc<Pix>::T;
    constexpr int STAGE = FUSED ? G::STAGE_FUSED : G::STAGE_MOTION;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // TMA destinations must sit on 128-byte boundaries; the launch adds 128 B of slack
    unsigned char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    __shared__ __align__(8) uint64_t full[STAGES];   // TMA bytes landed
    __shared__ __align__(8) uint64_t empty[STAGES];  // every warp done with the stage
    // Block sums of a window of 32 frames, [window parity][accumulator][frame]:
    // every warp adds its sums once per window, the last warp to do so adds
    // them to the outputs (32 bits suffice for 8-bit samples: a tile's SAD is
    // at most 4096 x 65280 and its luma SSE 4096 x 255^2).
    using Win = typename std::conditional<sizeof(Pix) == 1, uint32_t, unsigned long long>::type;
    __shared__ __align__(16) Win wsum[2][4][32];
    __shared__ int wcount[2];
    // border tiles: element offset of the staged row that holds each staged
    // row after the mirror rule (frame-invariant, filled once)
    __shared__ int rowsrc[G::RAW_ROWS];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // each warp owns output rows RPW w .. RPW w + RPW-1 of the tile; its V rows are private
    constexpr int VR = SH::template VR<Pix, FUSED, V2>;   // V rows of one vertical pass
    uint32_t* sV = reinterpret_cast<uint32_t*>(smem + STAGES * STAGE) + warp * VR * SVW;
    [[maybe_unused]] const Span vrows{sV, VR * SVW * sizeof(uint32_t)};   // this warp's V rows
    // border tiles of every chunk first, interior tiles after them in row-major
    // order (tile_of_block)
    // this block's tile and frames (uniform chunks, or a split-tail launch)
    int tx, ty, f_begin, f_end;
    block_work(a.w, a.h, (a.w + TW - 1) / TW, (a.h + TH - 1) / TH, gridDim.z, a.n, a.chunk, a.tiles_a,
               a.chunk_b, blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z), &tx, &ty, &f_begin,
               &f_end, TH);
    const int x0 = tx * TW, y0 = ty * TH;
    const bool full_tile = (x0 + TW <= a.w) && (y0 + TH <= a.h);
    const bool pl = x0 == 0, pt = y0 == 0;
    const bool pr = x0 + TW + 2 > a.w, pb = y0 + TH + 2 > a.h;
    // interior copy of the frame loop: no mirrored rows, no partial columns
    const bool interior = full_tile && !pt && !pb;
    const uint32_t rnd = 1u << (a.bpc - 1);
    const int sh = a.bpc;
    const long long wait_cycles = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NWK);
        }
        fence_mbar_init();
        prefetch_tmap(&maps.raw);
        if (V2 && a.has_prev) prefetch_tmap(&maps.prev);
        if constexpr (FUSED) {
            prefetch_tmap(&maps.dist);
            prefetch_tmap(&maps.ru);
            prefetch_tmap(&maps.du);
            prefetch_tmap(&maps.rv);
            prefetch_tmap(&maps.dv);
        }
        wcount[0] = wcount[1] = 0;
    }
    for (int i = tid; i < 2 * 4 * 32; i += NTK) (&wsum[0][0][0])[i] = 0;
    MG_BC_BEGIN(a.err);
    if (tid < G::RAW_ROWS) {
        // mirror on read: the boxes arrive zero-filled outside the frame; a row
        // y0 - 2 + r outside [0, h) is read from its mirror, clamped into the
        // box for rows that only feed outputs outside the frame
        int y = y0 - 2 + tid;
        y = y < 0 ? -y : (y >= a.h ? 2 * a.h - 2 - y : y);
        int rr = y - (y0 - 2);
        rr = rr < 0 ? 0 : (rr > G::RAW_ROWS - 1 ? G::RAW_ROWS - 1 : rr);
        rowsrc[tid] = rr * G::RAW_W;
    }
    __syncthreads();

    // a chunk that starts after frame 0 starts one frame early to rebuild
    // B_prev (no outputs for it).  motion_v2 continuing an earlier call starts
    // from that call's last raw frame (the prev map) in the same way.
    const bool warm_prev = V2 && f_begin == 0 && a.has_prev;
    const bool warm = f_begin > 0 || warm_prev;
    const int first = f_begin - (warm ? 1 : 0);
    const int cnt = f_end - first;
    const bool use_prev = !V2 && !warm && a.has_prev;

    int issued = 0;  // thread 0: frames issued so far
    auto issue = [&](int l) {  // thread 0 only; l = frame index within the chunk
        issued = l + 1;
        const int s = l % STAGES;
        const int f = first + l;
        unsigned char* st = smem + s * STAGE;
        const bool luma_only = warm && l == 0;
        fence_proxy_async();
        mbar_arrive_expect_tx(&full[s], (luma_only ? G::RAW_BYTES : STAGE) + a.tx_extra);
        if (V2 && warm_prev && l == 0)
            tma_load_3d(st, &maps.prev, x0 - G::HX, y0 - 2, 0, &full[s]);
        else
            tma_load_3d(st, &maps.raw, x0 - G::HX, y0 - 2, f, &full[s]);
        if (FUSED && !luma_only) {
            tma_load_3d(st + G::RAW_BYTES, &maps.dist, x0, y0, f, &full[s]);
            unsigned char* sc = st + G::RAW_BYTES + G::DIST_BYTES;
            tma_load_3d(sc, &maps.ru, x0 / 2, y0 / 2, f, &full[s]);
            tma_load_3d(sc + G::C_BYTES, &maps.du, x0 / 2, y0 / 2, f, &full[s]);
            tma_load_3d(sc + 2 * G::C_BYTES, &maps.rv, x0 / 2, y0 / 2, f, &full[s]);
            tma_load_3d(sc + 3 * G::C_BYTES, &maps.dv, x0 / 2, y0 / 2, f, &full[s]);
        }
    };
    if (tid == 0) {
        const int pre = cnt < STAGES ? cnt : STAGES;
        for (int l = 0; l < pre; ++l) issue(l);
    }

    // this thread's outputs: rows RPW w + k, columns 4q .. 4q+3 (q = lane).
    // bp holds B of the previous frame -- for motion_v2 the previous frame's
    // unrounded vertical sums X, and hxp that of the thread's halo value
    const int q = lane;
    [[maybe_unused]] uint32_t hxp = 0;
    uint32_t bp[RPW][4];
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
        const int y = y0 + RPW * warp + k;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int x = x0 + 4 * q + i;
            bp[k][i] = (use_prev && y < a.h && x < a.w)
                           ? MG_LD(a.bprev + (long long)y * a.bprev_pitch + x, a.bprev,
                                   (size_t)a.h * a.bprev_pitch * sizeof(uint16_t))
                           : 0u;
        }
    }
    // valid columns of this thread's quad in each of its rows (edge tiles)
    int nvalid[RPW];
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
        int nv = (y0 + RPW * warp + k < a.h) ? a.w - (x0 + 4 * q) : 0;
        nvalid[k] = nv < 0 ? 0 : (nv > 4 ? 4 : nv);
    }
    // per-thread byte offsets inside a stage (the same for every stage)
    const int off_vcol = (G::HX + 4 * lane) * G::S;   // this lane's columns in staged row 0
    // halo row 0..RPW-1 and column; with 4-row warps lanes 16..31 repeat lanes 0..15
    const int halo_r = (lane >> 2) % RPW, halo_which = lane & 3;
    const int halo_off = halo_which == 0 ? -2 : halo_which == 1 ? -1 : halo_which == 2 ? TW : TW + 1;
    // an interior tile on the left or right frame edge reads a halo column
    // outside the frame from its mirror inside it (x < 0 -> -x, x >= w ->
    // 2w - 2 - x; here always within the staged box); border tiles mirror V
    // after the vertical pass instead
    int hsrc = halo_off;
    if (interior) {
        if (x0 + hsrc < 0) hsrc = -2 * x0 - hsrc;
        else if (x0 + hsrc >= a.w) hsrc = 2 * (a.w - x0) - 2 - hsrc;
    }
    const int off_hcol = (G::HX + hsrc) * G::S;   // the halo lane's column in staged row 0
    // only warps whose rows reach above row 0 or below row h - 1 read rows
    // through rowsrc
    const bool wmirror = (pt && RPW * warp < 2) || (pb && RPW * warp + RPW + 3 >= a.h - y0 + 2);
    const int off_ref = ((RPW * warp + 2) * G::RAW_W + G::HX + 4 * q) * G::S;   // row k: + k RAW_W S
    const int off_dist = G::RAW_BYTES + ((RPW * warp) * TW + 4 * q) * G::S;     // row k: + k TW S
    const int off_chroma = G::RAW_BYTES + G::DIST_BYTES +
                           ((SH::CRW * warp + lane / SH::LPR) * G::CW + SH::SPL * (lane % SH::LPR)) * G::S;
    // lane j holds the warp's sums of frame 32 m + j of the current window
    uint32_t acc_s = 0;
    [[maybe_unused]] Win acc_y = 0, acc_u = 0, acc_v = 0;
    // End of a window of 32 frames (or of the chunk) at frame l: each warp adds
    // its lanes to the block's window sums; the last warp to arrive adds them
    // to the 64-bit outputs, one atomic per frame and accumulator (ADR-1392,
    // Decision 1, with the atomics of 32 frames issued together) and clears
    // them.  Warps are at most STAGES frames apart, so two windows suffice.
    auto flush_window = [&](int l) {
        const int jl = (l & ~31) + lane;   // this lane's frame
        const bool v = jl <= l && first + jl >= 0;   // (a warm-up frame may be frame -1)
        const int wb = (l >> 5) & 1;
        if (v) {
            atomicAdd(&wsum[wb][0][lane], (Win)acc_s);
            if constexpr (FUSED) {
                atomicAdd(&wsum[wb][1][lane], acc_y);
                atomicAdd(&wsum[wb][2][lane], acc_u);
                atomicAdd(&wsum[wb][3][lane], acc_v);
            }
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&wcount[wb], 1) == NWK - 1;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
            __threadfence_block();
            if (v) {
                const long long g = first + jl;
                const unsigned long long t = atomicExch(&wsum[wb][0][lane], (Win)0);
                if (t && MG_OK(a.sad_out + g, 8, a.sad_out, (size_t)a.n * 8)) atomicAdd(a.sad_out + g, t);
                if constexpr (FUSED) {
                    const unsigned long long ty = atomicExch(&wsum[wb][1][lane], (Win)0);
                    const unsigned long long tu = atomicExch(&wsum[wb][2][lane], (Win)0);
                    const unsigned long long tv = atomicExch(&wsum[wb][3][lane], (Win)0);
                    if (MG_OK(a.sse_out + 3LL * g, 8, a.sse_out, (size_t)a.n * 24) &&
                        MG_OK(a.sse_out + 3LL * g + 2, 8, a.sse_out, (size_t)a.n * 24)) {
                        if (ty) atomicAdd(a.sse_out + 3LL * g, ty);
                        if (tu) atomicAdd(a.sse_out + 3LL * g + 1, tu);
                        if (tv) atomicAdd(a.sse_out + 3LL * g + 2, tv);
                    }
                }
            }
            if (lane == 0) wcount[wb] = 0;
        }
    };

    // The frame loop, compiled twice: for interior tiles (no mirrored rows, no
    // masks) and for tiles on the top or bottom border or with a partial
    // column.  A runtime test per frame costs the interior tiles several
    // percent.
    auto frames = [&](auto interior_tag) -> bool {
        constexpr bool INTERIOR = decltype(interior_tag)::value;
        for (int l = 0; l < cnt; ++l) {
            const int s = l % STAGES;
            const unsigned parity = (unsigned)(l / STAGES) & 1u;
            const bool ok = mbar_wait_bounded(&full[s], parity, wait_cycles);
            unsigned char* st = smem + s * STAGE;
            [[maybe_unused]] const Span box{st, (size_t)G::RAW_BYTES};   // the staged luma box
            // the stage of frame l-1 takes frame l+STAGES-1 as soon as every warp
            // has released it
            if (tid == 0 && l >= 1 && l + STAGES - 1 < cnt) {
                const int sp = (l - 1) % STAGES;
                // (a stage never released is left alone: the warps that wait for
                // its refill time out and report it)
                if (mbar_wait_bounded(&empty[sp], (unsigned)((l - 1) / STAGES) & 1u, wait_cycles))
                    issue(l + STAGES - 1);
            }
            // a stage that never landed: this warp records it and leaves (the
            // others then run out of stages and leave too)
            if (__any_sync(0xffffffffu, !ok)) {
                if (lane == 0 && a.err) atomicOr(a.err, 1);
                return false;
            }
            const bool remap = !INTERIOR && wmirror;   // warp-uniform

            // ---- halo columns (two on each side) of the warp's rows: lane = (row, column)
            uint32_t hv = 0;
            {
                const Pix* c = reinterpret_cast<const Pix*>(st + off_hcol);
                const int hr = RPW * warp + halo_r;
                uint32_t t[5];
#pragma unroll
                for (int k = 0; k < 5; ++k) {
                    const int ri = remap ? MG_LD(&rowsrc[hr + k], rowsrc, sizeof(rowsrc)) : (hr + k) * G::RAW_W;
                    t[k] = MG_LD(c + ri, box.p, box.n);
                }
                if constexpr (V2) {
                    const uint32_t x = vsum(t[0], t[1], t[2], t[3], t[4]);
                    hv = (uint32_t)vdiff<Pix>(hxp, x, rnd, sh);
                    hxp = x;
                } else {
                    hv = vtap(t[0], t[1], t[2], t[3], t[4], rnd, sh);
                }
            }
            [[maybe_unused]] const bool do_out = l > 0 || !warm;   // not the warm-up frame
            const bool do_sad = l > 0 || use_prev;
            uint32_t sad = 0;
            [[maybe_unused]] Acc sse_y = 0, sse_u = 0, sse_v = 0;
#pragma unroll
            for (int h = 0; h < RPW / VR; ++h) {
                if (h > 0) __syncwarp();   // the previous half has read the V rows
                // ---- vertical pass of VR rows (staged row r <-> y0 - 2 + r)
                [[maybe_unused]] uint32_t center[VR];
                if constexpr (VR == 8) {
                    const Pix* colv = reinterpret_cast<const Pix*>(st + off_vcol);
                    const int r0 = RPW * warp;
                    if (remap)
                        vertical_oct(colv, [&](int i) { return MG_LD(&rowsrc[r0 + i], rowsrc, sizeof(rowsrc)); },
                                     sV + 4 + 4 * lane, rnd, sh, center, box, vrows);
                    else
                        vertical_oct(colv, [=](int i) { return (r0 + i) * G::RAW_W; }, sV + 4 + 4 * lane, rnd, sh,
                                     center, box, vrows);
                } else if constexpr (V2) {
                    // V of prev - cur from this frame's sums and the previous frame's
                    uint32_t x[4][4];
                    const Pix* colv = reinterpret_cast<const Pix*>(st + off_vcol);
                    const int r0 = RPW * warp + 4 * h;
                    if (remap)
                        vertical_sums(colv, [&](int i) { return MG_LD(&rowsrc[r0 + i], rowsrc, sizeof(rowsrc)); }, x, box);
                    else
                        vertical_sums(colv, [=](int i) { return (r0 + i) * G::RAW_W; }, x, box);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4 o;
                        o.x = (uint32_t)vdiff<Pix>(bp[4 * h + j][0], x[j][0], rnd, sh);
                        o.y = (uint32_t)vdiff<Pix>(bp[4 * h + j][1], x[j][1], rnd, sh);
                        o.z = (uint32_t)vdiff<Pix>(bp[4 * h + j][2], x[j][2], rnd, sh);
                        o.w = (uint32_t)vdiff<Pix>(bp[4 * h + j][3], x[j][3], rnd, sh);
                        MG_ST(reinterpret_cast<uint4*>(sV + 4 + 4 * lane + j * SVW), o, vrows.p, vrows.n);
#pragma unroll
                        for (int i = 0; i < 4; ++i) bp[4 * h + j][i] = x[j][i];
                    }
                } else {
                    const Pix* colv = reinterpret_cast<const Pix*>(st + off_vcol);
                    const int r0 = RPW * warp + 4 * h;
                    if (remap)
                        vertical_quad(colv, [&](int i) { return MG_LD(&rowsrc[r0 + i], rowsrc, sizeof(rowsrc)); },
                                      sV + 4 + 4 * lane, rnd, sh, center, box, vrows);
                    else
                        vertical_quad(colv, [=](int i) { return (r0 + i) * G::RAW_W; },
                                      sV + 4 + 4 * lane, rnd, sh, center, box, vrows);
                }
                if ((lane >> 2) < RPW && halo_r / VR == h)
                    MG_ST(&sV[(halo_r % VR) * SVW + 4 + halo_off], hv, vrows.p, vrows.n);
                __syncwarp();
                if (!INTERIOR && (pl || pr)) {
                    // the column mirror on V (the vertical pass works per column):
                    // x = -1, -2 <- 1, 2 on the left edge, x = w + k <- w - 2 - k on
                    // the right edge, in this warp's VR V rows; no source is a target
                    if (lane < 4 * VR) {
                        const int row = lane >> 2, which = lane & 3;
                        int dc = -3, sc = 0;
                        if (which < 2) {
                            if (pl) { dc = -1 - which; sc = 1 + which; }
                        } else if (pr) {
                            const int k = which - 2;
                            dc = a.w - x0 + k;
                            sc = a.w - x0 - 2 - k;
                        }
                        if (dc >= -2 && dc <= TW + 1)
                            MG_ST(&sV[row * SVW + 4 + dc], MG_LD(&sV[row * SVW + 4 + sc], vrows.p, vrows.n),
                                  vrows.p, vrows.n);
                    }
                    __syncwarp();
                }

                // ---- horizontal pass, SAD against B_prev, squared errors
#pragma unroll
                for (int kk = 0; kk < VR; ++kk) {
                    const int k = VR * h + kk;
                    const uint32_t* v = sV + kk * SVW + 4 * q;
                    const uint4 A = MG_LD(reinterpret_cast<const uint4*>(v), vrows.p, vrows.n);
                    const uint4 Bq = MG_LD(reinterpret_cast<const uint4*>(v + 4), vrows.p, vrows.n);
                    const uint4 C = MG_LD(reinterpret_cast<const uint4*>(v + 8), vrows.p, vrows.n);
                    if constexpr (V2) {
                        // SAD of |blur(prev - cur)|; invalid samples add 0
                        const int wi[12] = {(int)A.x, (int)A.y, (int)A.z, (int)A.w, (int)Bq.x, (int)Bq.y,
                                            (int)Bq.z, (int)Bq.w, (int)C.x, (int)C.y, (int)C.z, (int)C.w};
                        int bd[4];
                        horizontal_quad_signed(wi, bd);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            sad = __sad((INTERIOR || full_tile || i < nvalid[k]) ? bd[i] : 0, 0, sad);
                        continue;
                    }
                    const uint32_t wv[12] = {A.x, A.y, A.z, A.w, Bq.x, Bq.y, Bq.z, Bq.w, C.x, C.y, C.z, C.w};
                    uint32_t b[4];
                    horizontal_quad(wv, b);
                    if (INTERIOR || full_tile) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) sad = __sad(b[i], bp[k][i], sad);
                    } else {
                        // an invalid sample compares with itself and adds 0
#pragma unroll
                        for (int i = 0; i < 4; ++i) sad = __sad(b[i], i < nvalid[k] ? bp[k][i] : b[i], sad);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) bp[k][i] = b[i];
                    if constexpr (FUSED) {
                        const Pix* dp = reinterpret_cast<const Pix*>(st + off_dist + k * TW * G::S);
                        if constexpr (sizeof(Pix) == 1) {
                            uint32_t d = __vabsdiffu4(
                                center[kk], MG_LD(reinterpret_cast<const uint32_t*>(dp), st + G::RAW_BYTES, G::DIST_BYTES));
                            if (!INTERIOR && !full_tile)
                                d &= nvalid[k] <= 0 ? 0u : (0xffffffffu >> (8 * (4 - nvalid[k])));
                            sse_y = __dp4a(d, d, sse_y);
                        } else {
                            uint32_t rf[4], ds[4];
                            unpack4_in(reinterpret_cast<const Pix*>(st + off_ref + k * G::RAW_W * G::S), box.p, box.n, rf);
                            unpack4_in(dp, st + G::RAW_BYTES, G::DIST_BYTES, ds);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const long long e = (long long)rf[i] - (long long)ds[i];
                                sse_y += (INTERIOR || i < nvalid[k]) ? (Acc)(e * e) : (Acc)0;
                            }
                        }
                    }
                }
            }
            if constexpr (FUSED) {
                // 4:2:0 chroma: 16 rows x 64 columns per plane; warp w takes rows
                // CRW w .. CRW w + CRW-1, SPL samples per lane; outside the picture
                // both sides were zero-filled, so they add 0
                const unsigned char* sc = st + off_chroma;
                [[maybe_unused]] const unsigned char* cb = st + G::RAW_BYTES + G::DIST_BYTES;   // chroma tiles
#pragma unroll
                for (int j = 0; j < SH::SPL / 4; ++j) {
                    const unsigned char* cj = sc + 4 * j * G::S;
                    if constexpr (sizeof(Pix) == 1) {
                        const uint32_t du = __vabsdiffu4(
                            MG_LD(reinterpret_cast<const uint32_t*>(cj), cb, G::C_BYTES),
                            MG_LD(reinterpret_cast<const uint32_t*>(cj + G::C_BYTES), cb + G::C_BYTES, G::C_BYTES));
                        const uint32_t dv = __vabsdiffu4(
                            MG_LD(reinterpret_cast<const uint32_t*>(cj + 2 * G::C_BYTES), cb + 2 * G::C_BYTES, G::C_BYTES),
                            MG_LD(reinterpret_cast<const uint32_t*>(cj + 3 * G::C_BYTES), cb + 3 * G::C_BYTES, G::C_BYTES));
                        sse_u = __dp4a(du, du, sse_u);
                        sse_v = __dp4a(dv, dv, sse_v);
                    } else {
                        uint32_t ru[4], du[4], rv[4], dv[4];
                        unpack4_in(reinterpret_cast<const Pix*>(cj), cb, G::C_BYTES, ru);
                        unpack4_in(reinterpret_cast<const Pix*>(cj + G::C_BYTES), cb + G::C_BYTES, G::C_BYTES, du);
                        unpack4_in(reinterpret_cast<const Pix*>(cj + 2 * G::C_BYTES), cb + 2 * G::C_BYTES, G::C_BYTES, rv);
                        unpack4_in(reinterpret_cast<const Pix*>(cj + 3 * G::C_BYTES), cb + 3 * G::C_BYTES, G::C_BYTES, dv);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const long long eu = (long long)ru[i] - (long long)du[i];
                            const long long ev = (long long)rv[i] - (long long)dv[i];
                            sse_u += (Acc)(eu * eu);
                            sse_v += (Acc)(ev * ev);
                        }
                    }
                }
            }
            // every lane has finished reading this stage: release it to the producer
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);

            // ---- warp sums of this frame into lane l mod 32
            const uint32_t wsad = __reduce_add_sync(0xffffffffu, sad);
            [[maybe_unused]] Win wy = 0, wu = 0, wvv = 0;
            if constexpr (FUSED) {
                if constexpr (sizeof(Pix) == 1) {
                    wy = __reduce_add_sync(0xffffffffu, sse_y);
                    wu = __reduce_add_sync(0xffffffffu, sse_u);
                    wvv = __reduce_add_sync(0xffffffffu, sse_v);
                } else {
                    wy = warp_sum(sse_y);
                    wu = warp_sum(sse_u);
                    wvv = warp_sum(sse_v);
                }
            }
            if (lane == (l & 31)) {
                acc_s = do_sad ? wsad : 0u;
                if constexpr (FUSED) {
                    acc_y = do_out ? wy : (Win)0;
                    acc_u = do_out ? wu : (Win)0;
                    acc_v = do_out ? wvv : (Win)0;
                }
            }
            if ((l & 31) == 31 || l == cnt - 1) flush_window(l);
        }
        return true;
    };
    const bool alive = interior ? frames(std::true_type{}) : frames(std::false_type{});
    if (tid == 0) {
        // no copy may still be landing in this block's shared memory when it
        // exits: wait (bounded) for the last phase of every stage issued
        for (int m = issued - STAGES < 0 ? 0 : issued - STAGES; m < issued; ++m)
            mbar_wait_bounded(&full[m % STAGES], (unsigned)(m / STAGES) & 1u, wait_cycles);
    }
    if (!alive) return;

    if (V2 && a.store_last && cnt > 0 && f_end == a.n) {
        // motion_v2 keeps the last raw frame for the next call: the tile's
        // samples from the last frame's stage (no stage is refilled after it)
        const Pix* raw = reinterpret_cast<const Pix*>(smem + ((cnt - 1) % STAGES) * STAGE);
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int y = y0 + RPW * warp + k;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int x = x0 + 4 * q + i;
                if (y < a.h && x < a.w)
                    MG_ST(reinterpret_cast<Pix*>(a.raw_out + (long long)y * a.raw_pitch) + x,
                          MG_LD(raw + (RPW * warp + k + 2) * G::RAW_W + G::HX + 4 * q + i, raw, G::RAW_BYTES),
                          a.raw_out, (size_t)a.h * a.raw_pitch);
            }
        }
        return;
    }
    if (a.store_last && cnt > 0 && f_end == a.n) {
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int y = y0 + RPW * warp + k;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int x = x0 + 4 * q + i;
                if (y < a.h && x < a.w)
                    MG_ST(a.bprev_out + (long long)y * a.bprev_pitch + x, (uint16_t)bp[k][i], a.bprev_out,
                          (size_t)a.h * a.bprev_pitch * sizeof(uint16_t));
            }
        }
    }
}

// ------------------------------------------------------------------ host side
// Frame chunks of a launch, sized by the SM count (ADR-1226): n frames over
// `tiles` tiles run as c chunks of CTAs, `slots` CTAs resident at once.  A
// chunk after the first pays one warm-up frame and every chunk its own
// pipeline fill (about half a frame):
//   cost(c) = (n + (c - 1) + c / 2) / n / eff,  waves = tiles c / slots.
// A launch under one wave leaves SMs idle but runs the CTAs it holds faster,
// so it pays a quarter of its idle share:
//   eff = waves / (1 + (1 / waves - 1) / 4)                  (waves <= 1).
// Past one wave the motion kernel (bound by instruction issue) pays for the
// idle slots of its last, partial wave in proportion p = min(1, 2.6 /
// waves^2) -- fully under ~1.6 waves, less and less as CTAs of many waves
// start at staggered times -- while motion_v2 (its 64-bit horizontal pass has
// long dependency chains) pays a quarter of them at any count:
//   eff = 1 / (1 + p (ceil(waves) / waves - 1)),  p as above or 1/4 (v2).
// Chunks keep at least 5 frames; c <= max_c.  Fitted to forced-chunk timings
// on GB300 with the block order of tile_of_block.  Motion: 1080p x 16 frames
// is fastest at one chunk (three as fast, two 2 % slower), x 32 at three (4 %
// over two); 4K x 16 and the 10-bit 4K x 32 at one; the 4K 4:2:0 x 50 pairs at
// two (2 % over one and three; a split tail, which plan_launch takes first,
// beats both by 1.7 %).  motion_v2: 1080p x 16 and x 32 at two (one is 13 % and
// 19 % slower), 10-bit 4K x 32 at one or two.
int plan_frame_chunks(long long tiles, long long slots, int n, int max_c, bool v2) {
    if (n <= 1 || tiles <= 0 || slots <= 0) return 1;
    int best_c = 1;
    double best = 1e30;
    for (int c = 1; c <= max_c && c <= n; ++c) {
        const int len = (n + c - 1) / c;
        if (c > 1 && len < 5) break;
        const int cz = (n + len - 1) / len;
        const double waves = (double)tiles * cz / (double)slots;
        double eff;
        if (waves <= 1.0) {
            eff = waves / (1.0 + 0.25 * (1.0 / waves - 1.0));
        } else {
            const double p = v2 ? 0.25 : std::min(1.0, 2.6 / (waves * waves));
            eff = 1.0 / (1.0 + p * (std::ceil(waves) / waves - 1.0));
        }
        const double work = (n + (cz - 1) + 0.5 * cz) / (double)n;
        const double cost = work / eff;
        if (cost < best - 1e-9) {
            best = cost;
            best_c = cz;
        }
    }
    return best_c;
}

long long plan_split_tail(long long tiles, long long slots, int n, int* tiles_a, int* chunk_b) {
    *tiles_a = 0;
    *chunk_b = 0;
    if (slots <= 0 || tiles <= slots) return 0;
    const long long rest = tiles % slots;
    if (rest == 0 || 2 * rest > slots) return 0;
    long long cb = slots / rest;
    if (cb > 8) cb = 8;
    while (cb > 1 && (n + cb - 1) / cb < 4) --cb;
    if (cb < 2) return 0;
    const int len = (int)((n + cb - 1) / cb);
    const long long chunks = (n + len - 1) / len;   // non-empty chunks
    *tiles_a = (int)(tiles - rest);
    *chunk_b = len;
    return (tiles - rest) + rest * chunks;
}

LaunchPlan plan_launch(long long tiles, long long slots, int n, bool v2, bool same_plane) {
    LaunchPlan p{n > 0 ? n : 1, 1, 0, 0, tiles};
    if (same_plane) return p;
    if (!v2) {
        const long long b = plan_split_tail(tiles, slots, n, &p.tiles_a, &p.chunk_b);
        if (b > 0) {
            p.blocks = b;
            return p;
        }
    }
    const int c = plan_frame_chunks(tiles, slots, n, 8, v2);
    p.chunk = (n + c - 1) / c;
    p.gz = (n + p.chunk - 1) / p.chunk;
    p.blocks = tiles * p.gz;
    if (v2 && c == 1) {
        const long long b = plan_split_tail(tiles, slots, n, &p.tiles_a, &p.chunk_b);
        if (b > 0) p.blocks = b;
    }
    return p;
}

namespace {

// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised exactly once even when several host threads get here together).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

bool encode(CUtensorMap* m, int bytes_per_sample, const void* base, int w, int h, int n,
            long long pitch, long long stride, int box_w, int box_h) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || !base) return false;
    if (n <= 1) stride = ((pitch * h) + 15) & ~15LL;  // never stepped through
    cuuint64_t dims[3] = {(cuuint64_t)w, (cuuint64_t)h, (cuuint64_t)(n > 0 ? n : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)pitch, (cuuint64_t)stride};
    cuuint32_t box[3] = {(cuuint32_t)box_w, (cuuint32_t)box_h, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        bytes_per_sample == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Resident CTAs of one kernel instance on the current device (all SMs), with
// its dynamic shared memory configured; cached per device (threads racing
// here compute and store the same value).
template <typename Pix, bool FUSED, int STAGES, bool V2, int THT>
cudaError_t resident_slots(int* slots) {
    using G = Geo<Pix, THT>;
    using SH = ShapeT<THT>;
    constexpr int STAGE = FUSED ? G::STAGE_FUSED : G::STAGE_MOTION;
    constexpr int SMEM = STAGES * STAGE + SH::template SV<Pix, FUSED, V2> + 128;
    static unsigned long long configured = 0;  // per device bit
    static int slots_per_dev[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(motion_tma_kernel<Pix, FUSED, STAGES, V2, THT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, bit, __ATOMIC_RELEASE);
    }
    int spm = __atomic_load_n(&slots_per_dev[dev & 63], __ATOMIC_RELAXED);
    if (spm == 0) {
        int per_sm = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, motion_tma_kernel<Pix, FUSED, STAGES, V2, THT>,
                                                          SH::NTK, SMEM);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        spm = (per_sm > 0 ? per_sm : 1) * sms;
        __atomic_store_n(&slots_per_dev[dev & 63], spm, __ATOMIC_RELAXED);
    }
    *slots = spm;
    return cudaSuccess;
}

template <typename Pix, bool FUSED, int STAGES, bool V2 = false, int THT = 32>
cudaError_t launch_tma_one(const TmaMaps& maps, const TileArgs& a, cudaStream_t s) {
    using G = Geo<Pix, THT>;
    using SH = ShapeT<THT>;
    constexpr int STAGE = FUSED ? G::STAGE_FUSED : G::STAGE_MOTION;
    constexpr int SMEM = STAGES * STAGE + SH::template SV<Pix, FUSED, V2> + 128;
    // Size the launch by the SM count (ADR-1226): plan_launch.
    int spm = 0;
    cudaError_t e = resident_slots<Pix, FUSED, STAGES, V2, THT>(&spm);
    if (e != cudaSuccess) return e;
    TileArgs b = a;
    constexpr int TH = THT;
    const long long tiles = (long long)((a.w + TW - 1) / TW) * ((a.h + TH - 1) / TH);
    // a launch that reads and writes the same resident plane keeps one chunk:
    // the last chunk's store must not overtake the first chunk's read
    const bool same_plane = !V2 && a.has_prev && a.bprev == a.bprev_out;
    const LaunchPlan p = plan_launch(tiles, spm, a.n, V2, same_plane);
    b.chunk = p.chunk;
    b.tiles_a = p.tiles_a;
    b.chunk_b = p.chunk_b;
    const dim3 grid = p.tiles_a > 0 ? dim3((unsigned)p.blocks, 1, 1)
                                    : dim3((a.w + TW - 1) / TW, (a.h + TH - 1) / TH, p.gz);
    motion_tma_kernel<Pix, FUSED, STAGES, V2, THT><<<grid, SH::NTK, SMEM, s>>>(maps, b);
    return cudaGetLastError();
}

// A motion-only launch whose 32-row tiles (in their planned chunks) fit in
// one wave leaves every block a long serial chain of frames at a fraction of
// the SMs' issue capacity; 16-row tiles with 4-row warps halve each warp's
// work per frame and run twice the blocks, more of them resident per SM.
template <typename Pix, int STAGES, bool V2>
cudaError_t choose_short_tiles(const TileArgs& a, bool* out) {
    int spm = 0;
    const cudaError_t e = resident_slots<Pix, false, STAGES, V2, TH>(&spm);
    if (e != cudaSuccess) return e;
    const long long tiles = (long long)((a.w + TW - 1) / TW) * ((a.h + TH - 1) / TH);
    const bool same_plane = !V2 && a.has_prev && a.bprev == a.bprev_out;
    *out = prefer_short_tiles(tiles, spm, a.n, same_plane ? 1 : 8, V2);
    return cudaSuccess;
}

}  // namespace

bool tma_usable(const TileArgs& a, bool fused) {
    if (!encode_fn() || !a.aligned16) return false;
    // TMA global strides must be multiples of 16 bytes below 2^40
    if (a.pitch_y % 16 || a.pitch_y >= (1LL << 40)) return false;
    if (a.n > 1 && (a.stride_y % 16 || a.stride_y >= (1LL << 40))) return false;
    if (fused) {
        if (a.pitch_uv % 16 || (a.n > 1 && a.stride_uv % 16)) return false;
    }
    return true;
}

cudaError_t launch_motion_tma(const TileArgs& a, bool fused, cudaStream_t s, int* launches,
                              bool* used) {
    *used = false;
    if (a.n <= 0) return cudaSuccess;
    if (!tma_usable(a, fused)) return cudaSuccess;
    const int S = a.bpc == 8 ? 1 : 2;
    // tile height first: the luma box of the tensor map is (tile rows + 4) high
    bool short_tiles = !fused && a.force_rows == kShortTileH;
    if (!fused && a.force_rows == 0) {
        const cudaError_t e = S == 1 ? choose_short_tiles<uint8_t, 4, false>(a, &short_tiles)
                                     : choose_short_tiles<uint16_t, 3, false>(a, &short_tiles);
        if (e != cudaSuccess) return e;
    }
    TmaMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const int rawW = TW + 2 * (16 / S), rawH = (short_tiles ? kShortTileH : TH) + 4;
    bool ok = encode(&maps.raw, S, a.ref_y, a.w, a.h, a.n, a.pitch_y, a.stride_y, rawW, rawH);
    if (fused) {
        ok = ok && encode(&maps.dist, S, a.dist_y, a.w, a.h, a.n, a.pitch_y, a.stride_y, TW, TH);
        ok = ok && encode(&maps.ru, S, a.ref_u, a.cw, a.ch, a.n, a.pitch_uv, a.stride_uv, TW / 2, TH / 2);
        ok = ok && encode(&maps.du, S, a.dist_u, a.cw, a.ch, a.n, a.pitch_uv, a.stride_uv, TW / 2, TH / 2);
        ok = ok && encode(&maps.rv, S, a.ref_v, a.cw, a.ch, a.n, a.pitch_uv, a.stride_uv, TW / 2, TH / 2);
        ok = ok && encode(&maps.dv, S, a.dist_v, a.cw, a.ch, a.n, a.pitch_uv, a.stride_uv, TW / 2, TH / 2);
    }
    if (!ok) return cudaSuccess;  // the caller falls back to the generic kernel
    *used = true;
    *launches += 1;
    // stages per CTA: as many as keep the CTAs resident beside the V buffers
    // (4 for 8-bit motion, 3 for 16-bit motion, 2 for pairs)
    if (fused)
        return S == 1 ? launch_tma_one<uint8_t, true, 2>(maps, a, s) : launch_tma_one<uint16_t, true, 2>(maps, a, s);
    if (S == 1)
        return short_tiles ? launch_tma_one<uint8_t, false, 4, false, kShortTileH>(maps, a, s)
                           : launch_tma_one<uint8_t, false, 4>(maps, a, s);
    return short_tiles ? launch_tma_one<uint16_t, false, 3, false, kShortTileH>(maps, a, s)
                       : launch_tma_one<uint16_t, false, 3>(maps, a, s);
}

cudaError_t launch_motion_v2_tma(const TileArgs& a, cudaStream_t s, int* launches, bool* used) {
    *used = false;
    if (a.n <= 0) return cudaSuccess;
    if (!tma_usable(a, false)) return cudaSuccess;
    if (a.has_prev && (a.raw_pitch % 16 || ((uintptr_t)a.raw_prev & 15))) return cudaSuccess;
    const int S = a.bpc == 8 ? 1 : 2;
    bool short_tiles = a.force_rows == kShortTileH;
    if (a.force_rows == 0) {
        const cudaError_t e = S == 1 ? choose_short_tiles<uint8_t, 4, true>(a, &short_tiles)
                                     : choose_short_tiles<uint16_t, 4, true>(a, &short_tiles);
        if (e != cudaSuccess) return e;
    }
    TmaMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    const int rawW = TW + 2 * (16 / S), rawH = (short_tiles ? kShortTileH : TH) + 4;
    bool ok = encode(&maps.raw, S, a.ref_y, a.w, a.h, a.n, a.pitch_y, a.stride_y, rawW, rawH);
    if (a.has_prev)
        ok = ok && encode(&maps.prev, S, a.raw_prev, a.w, a.h, 1, a.raw_pitch, 0, rawW, rawH);
    if (!ok) return cudaSuccess;  // the caller falls back to the generic kernel
    *used = true;
    *launches += 1;
    if (S == 1)
        return short_tiles ? launch_tma_one<uint8_t, false, 4, true, kShortTileH>(maps, a, s)
                           : launch_tma_one<uint8_t, false, 4, true>(maps, a, s);
    return short_tiles ? launch_tma_one<uint16_t, false, 3, true, kShortTileH>(maps, a, s)
                       : launch_tma_one<uint16_t, false, 4, true>(maps, a, s);
}

}  // namespace mg
