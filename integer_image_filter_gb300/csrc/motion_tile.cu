// motion_tile.cu -- batched integer motion kernel (blur + SAD against the
// previous frame), optionally fused with the per-plane SSE of 4:2:0 pairs.
//
// Design (GB300 / sm_103a):
//  * One CTA owns a TW x TH output tile and walks the whole batch of frames in
//    time order, so the previous frame's blurred tile B_prev never leaves the
//    SM (registers); each frame is read from HBM once ("Making it fast",
//    Round 1: one kernel over all frames; Round 2: no scratch rebuilt per call).
//  * The next frame's tile (luma with a 2-row / 16-byte halo, and in the fused
//    form the distorted luma and the four chroma tiles) is staged into shared
//    memory with 16-byte cp.async copies while the current frame is computed
//    (double buffer).  Tiles touching the frame border load sample by sample
//    with the mirror rule applied at load time.
//  * The blur is separable: the vertical 5-tap pass runs once per sample
//    (rounded >> bpc) into a shared V tile, the horizontal 5-tap pass reads it
//    (rounded >> 16) -- "ADR-1392: CUDA motion, PSNR and moment kernels add one
//    atomic per block, the motion SAD filters separably, ...", Decision 4.
//  * |B - B_prev| and (ref - dist)^2 are reduced per block with warp shuffles
//    and shared memory, then ONE 64-bit atomic per block per frame and per
//    accumulator (same page, Decision 1).  Integer sums are order-independent,
//    so the result is exact (same page, Context).
#include "motion_internal.h"
#include "tile_geometry.cuh"

namespace mg {

// A 16-byte asynchronous copy whose source and destination must stay inside
// their buffers (checked build; otherwise the plain copy).
__device__ __forceinline__ void cp_async16_in(void* dst, const void* src, [[maybe_unused]] Span d,
                                              [[maybe_unused]] Span s) {
    if (MG_OK(dst, 16, d.p, d.n) && MG_OK(src, 16, s.p, s.n)) cp_async16(dst, src);
}

// Stage frame f (luma fy with row pitch `pitch`; fused: the distorted luma
// and chroma of pair f) for the tile at (x0, y0).
template <typename Pix, bool FUSED>
__device__ __forceinline__ void load_stage(const TileArgs& a, int f, unsigned char* st,
                                           int x0, int y0, bool fast, const uint8_t* fy,
                                           long long pitch) {
    using G = Geo<Pix>;
    constexpr int S = G::S;
    const int tid = threadIdx.x;
    // the buffers every access below must stay in: the frame fy, the caller's
    // distorted luma and chroma planes, and this stage's regions
    [[maybe_unused]] const Span fy_span{fy, (size_t)plane_span(1, 0, a.h, pitch, a.w, S)};
    [[maybe_unused]] const Span box{st, (size_t)G::RAW_BYTES};
    if (fast) {
        constexpr int CHR = G::RAW_W * S / 16;
        const uint8_t* g0 = fy + (long long)(y0 - 2) * pitch + (long long)(x0 - G::HX) * S;
        for (int c = tid; c < G::RAW_ROWS * CHR; c += NT) {
            const int r = c / CHR, k = c - r * CHR;
            cp_async16_in(st + (r * G::RAW_W) * S + k * 16, g0 + (long long)r * pitch + k * 16, box, fy_span);
        }
        if constexpr (FUSED) {
            unsigned char* sd = st + G::RAW_BYTES;
            constexpr int CHD = TW * S / 16;
            const uint8_t* d0 = a.dist_y + (long long)f * a.stride_y + (long long)y0 * a.pitch_y +
                                (long long)x0 * S;
            const Span dist_span{a.dist_y, (size_t)plane_span(a.n, a.stride_y, a.h, a.pitch_y, a.w, S)};
            for (int c = tid; c < TH * CHD; c += NT) {
                const int r = c / CHD, k = c - r * CHD;
                cp_async16_in(sd + r * TW * S + k * 16, d0 + (long long)r * a.pitch_y + k * 16,
                              Span{sd, (size_t)G::DIST_BYTES}, dist_span);
            }
            constexpr int CHC = G::CW * S / 16;
            const long long coff = (long long)f * a.stride_uv + (long long)(y0 / 2) * a.pitch_uv +
                                   (long long)(x0 / 2) * S;
            unsigned char* sc = sd + G::DIST_BYTES;
            for (int c = tid; c < 4 * G::CH * CHC; c += NT) {
                const int p = c / (G::CH * CHC);
                const int rem = c - p * (G::CH * CHC);
                const int r = rem / CHC, k = rem - r * CHC;
                // constant-index plane selection (ADR-1392 Decision 3)
                const uint8_t* base = p == 0 ? a.ref_u : p == 1 ? a.dist_u : p == 2 ? a.ref_v : a.dist_v;
                cp_async16_in(sc + p * G::C_BYTES + r * G::CW * S + k * 16,
                              base + coff + (long long)r * a.pitch_uv + k * 16,
                              Span{sc + p * G::C_BYTES, (size_t)G::C_BYTES},
                              Span{base, (size_t)plane_span(a.n, a.stride_uv, a.ch, a.pitch_uv, a.cw, S)});
            }
        }
        return;
    }
    // border tile: sample loads with the mirror rule applied here
    Pix* raw = reinterpret_cast<Pix*>(st);
    for (int e = tid; e < G::RAW_ROWS * G::RAW_W; e += NT) {
        const int r = e / G::RAW_W, c = e - r * G::RAW_W;
        const int yy = mirror_clamp(y0 - 2 + r, a.h), xx = mirror_clamp(x0 - G::HX + c, a.w);
        MG_ST(&raw[e], MG_LD(reinterpret_cast<const Pix*>(fy + (long long)yy * pitch + (long long)xx * S),
                             fy_span.p, fy_span.n),
              box.p, box.n);
    }
    if constexpr (FUSED) {
        Pix* sd = reinterpret_cast<Pix*>(st + G::RAW_BYTES);
        const uint8_t* fd = a.dist_y + (long long)f * a.stride_y;
        for (int e = tid; e < TH * TW; e += NT) {
            const int r = e / TW, c = e - r * TW;
            const int y = y0 + r, x = x0 + c;
            // outside the picture the distorted sample repeats the staged
            // reference sample, so the squared error there is zero
            const bool in = (y < a.h) && (x < a.w);
            const uint8_t* src = in ? fd + (long long)y * a.pitch_y + (long long)x * S
                                    : fy + (long long)mirror_clamp(y, a.h) * pitch +
                                          (long long)mirror_clamp(x, a.w) * S;
            [[maybe_unused]] const Span src_span =
                in ? Span{fd, (size_t)plane_span(1, 0, a.h, a.pitch_y, a.w, S)} : fy_span;
            MG_ST(&sd[e], MG_LD(reinterpret_cast<const Pix*>(src), src_span.p, src_span.n), st + G::RAW_BYTES,
                  G::DIST_BYTES);
        }
        Pix* sc = reinterpret_cast<Pix*>(st + G::RAW_BYTES + G::DIST_BYTES);
        const long long foff = (long long)f * a.stride_uv;
        for (int e = tid; e < 4 * G::CH * G::CW; e += NT) {
            const int p = e / (G::CH * G::CW);
            const int rem = e - p * (G::CH * G::CW);
            const int r = rem / G::CW, c = rem - r * G::CW;
            const int y = y0 / 2 + r, x = x0 / 2 + c;
            const uint8_t* base = p == 0 ? a.ref_u : p == 1 ? a.dist_u : p == 2 ? a.ref_v : a.dist_v;
            Pix v = 0;
            if (y < a.ch && x < a.cw)
                v = MG_LD(reinterpret_cast<const Pix*>(base + foff + (long long)y * a.pitch_uv + (long long)x * S),
                          base, plane_span(a.n, a.stride_uv, a.ch, a.pitch_uv, a.cw, S));
            MG_ST(&sc[e], v, st + G::RAW_BYTES + G::DIST_BYTES, 4 * G::C_BYTES);
        }
    }
}

// V2: motion_v2, the blur of prev - cur (unrounded vertical sums of the
// previous frame kept per thread, floor shifts, SAD of |blur|); FUSED false.
template <typename Pix, bool FUSED, bool V2>
__global__ void __launch_bounds__(NT) motion_tile_kernel(const TileArgs a) {
    static_assert(!(FUSED && V2), "motion_v2 has no fused form");
    using G = Geo<Pix>;
    using Acc = typename SseAcc<Pix>::T;
    constexpr int STAGE = FUSED ? G::STAGE_FUSED : G::STAGE_MOTION;
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* sV = reinterpret_cast<uint32_t*>(smem + 2 * STAGE);
    [[maybe_unused]] const Span vtile{sV, (size_t)G::SV_BYTES};
    __shared__ unsigned long long red[NW][4];
#if MG_BOUNDS_CHECK
    MG_BC_BEGIN(a.err);
    __syncthreads();
#endif

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int x0 = blockIdx.x * TW, y0 = blockIdx.y * TH;
    const bool full = (x0 + TW <= a.w) && (y0 + TH <= a.h);
    const bool inner = (x0 - G::HX >= 0) && (x0 + TW + G::HX <= a.w) && (y0 - 2 >= 0) &&
                       (y0 + TH + 2 <= a.h);
    const bool fast = a.aligned16 && inner;
    const bool fast_prev = inner && (((uintptr_t)a.raw_prev | (uintptr_t)a.raw_pitch) % 16 == 0);
    // motion_v2 continuing an earlier call first re-derives the vertical sums
    // of that call's last raw frame (local frame 0, no output)
    const bool warm = V2 && a.has_prev;
    const int cnt = a.n + (warm ? 1 : 0);
    auto stage = [&](int l, unsigned char* st) {
        const int f = l - (warm ? 1 : 0);
        if (f < 0)
            load_stage<Pix, FUSED>(a, 0, st, x0, y0, fast_prev, a.raw_prev, a.raw_pitch);
        else
            load_stage<Pix, FUSED>(a, f, st, x0, y0, fast, a.ref_y + (long long)f * a.stride_y,
                                   a.pitch_y);
    };
    [[maybe_unused]] uint32_t xp[4][4] = {};   // motion_v2: this thread's vertical sums, previous frame
    [[maybe_unused]] uint32_t hxp = 0;          // and of its halo value
    const uint32_t rnd = 1u << (a.bpc - 1);
    const int sh = a.bpc;

    // horizontal-pass ownership: quad q of 4 columns, rows rbase + 8k
    const int q = lane, rbase = warp;
    uint32_t bp[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int y = y0 + rbase + 8 * k;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int x = x0 + 4 * q + i;
            bp[k][i] = (a.has_prev && y < a.h && x < a.w)
                           ? MG_LD(a.bprev + (long long)y * a.bprev_pitch + x, a.bprev,
                                   (size_t)a.h * a.bprev_pitch * sizeof(uint16_t))
                           : 0u;
        }
    }

    stage(0, smem);
    cp_async_commit();
    for (int l = 0; l < cnt; ++l) {
        const int f = l - (warm ? 1 : 0);   // frame index of the output (-1: warm-up)
        unsigned char* st = smem + (l & 1) * STAGE;
        if (l + 1 < cnt) stage(l + 1, smem + ((l + 1) & 1) * STAGE);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const Pix* raw = reinterpret_cast<const Pix*>(st);
        [[maybe_unused]] const Span box{st, (size_t)G::RAW_BYTES};
        // ---- vertical pass: 32 quads x 8 runs of 4 rows; raw row r <-> y0 - 2 + r
        {
            const Pix* src = raw + (warp * 4) * G::RAW_W + G::HX + 4 * lane;
            uint32_t p[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) unpack4_in(src + i * G::RAW_W, box.p, box.n, p[i]);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                uint4 o;
                if constexpr (V2) {
                    uint32_t x[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        x[i] = vsum(p[r][i], p[r + 1][i], p[r + 2][i], p[r + 3][i], p[r + 4][i]);
                    o.x = (uint32_t)vdiff<Pix>(xp[r][0], x[0], rnd, sh);
                    o.y = (uint32_t)vdiff<Pix>(xp[r][1], x[1], rnd, sh);
                    o.z = (uint32_t)vdiff<Pix>(xp[r][2], x[2], rnd, sh);
                    o.w = (uint32_t)vdiff<Pix>(xp[r][3], x[3], rnd, sh);
#pragma unroll
                    for (int i = 0; i < 4; ++i) xp[r][i] = x[i];
                } else {
                    o.x = vtap(p[r][0], p[r + 1][0], p[r + 2][0], p[r + 3][0], p[r + 4][0], rnd, sh);
                    o.y = vtap(p[r][1], p[r + 1][1], p[r + 2][1], p[r + 3][1], p[r + 4][1], rnd, sh);
                    o.z = vtap(p[r][2], p[r + 1][2], p[r + 2][2], p[r + 3][2], p[r + 4][2], rnd, sh);
                    o.w = vtap(p[r][3], p[r + 1][3], p[r + 2][3], p[r + 3][3], p[r + 4][3], rnd, sh);
                }
                MG_ST(reinterpret_cast<uint4*>(sV + (warp * 4 + r) * SVW + 4 + 4 * lane), o, vtile.p, vtile.n);
            }
            // the two halo columns on each side of the tile
            if (tid < 4 * TH) {
                const int r = tid >> 2, which = tid & 3;
                const int off = which == 0 ? -2 : which == 1 ? -1 : which == 2 ? TW : TW + 1;
                const Pix* s = raw + r * G::RAW_W + G::HX + off;
                uint32_t t[5];
#pragma unroll
                for (int k = 0; k < 5; ++k) t[k] = MG_LD(s + k * G::RAW_W, box.p, box.n);
                if constexpr (V2) {
                    const uint32_t x = vsum(t[0], t[1], t[2], t[3], t[4]);
                    MG_ST(&sV[r * SVW + 4 + off], (uint32_t)vdiff<Pix>(hxp, x, rnd, sh), vtile.p, vtile.n);
                    hxp = x;
                } else {
                    MG_ST(&sV[r * SVW + 4 + off], vtap(t[0], t[1], t[2], t[3], t[4], rnd, sh), vtile.p, vtile.n);
                }
            }
        }
        __syncthreads();

        // ---- horizontal pass, SAD against B_prev, SSE of the luma
        const bool do_sad = V2 ? l > 0 : (f > 0) || a.has_prev;
        uint32_t sad = 0;
        Acc sse_y = 0, sse_u = 0, sse_v = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = rbase + 8 * k;
            const uint32_t* v = sV + r * SVW + 4 * q;
            const uint4 A = MG_LD(reinterpret_cast<const uint4*>(v), vtile.p, vtile.n);
            const uint4 Bq = MG_LD(reinterpret_cast<const uint4*>(v + 4), vtile.p, vtile.n);
            const uint4 C = MG_LD(reinterpret_cast<const uint4*>(v + 8), vtile.p, vtile.n);
            if constexpr (V2) {
                const int wi[12] = {(int)A.x, (int)A.y, (int)A.z, (int)A.w, (int)Bq.x, (int)Bq.y,
                                    (int)Bq.z, (int)Bq.w, (int)C.x, (int)C.y, (int)C.z, (int)C.w};
                int bd[4];
                horizontal_quad_signed(wi, bd);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool ok = full || ((y0 + r < a.h) && (x0 + 4 * q + i < a.w));
                    sad = __sad(ok ? bd[i] : 0, 0, sad);
                }
                continue;
            }
            const uint32_t wv[12] = {A.x, A.y, A.z, A.w, Bq.x, Bq.y, Bq.z, Bq.w, C.x, C.y, C.z, C.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t b = (kT0 * (wv[2 + i] + wv[6 + i]) + kT1 * (wv[3 + i] + wv[5 + i]) +
                                    kT2 * wv[4 + i] + 32768u) >> 16;
                uint32_t d = b > bp[k][i] ? b - bp[k][i] : bp[k][i] - b;
                if (!full) {
                    const bool ok = (y0 + r < a.h) && (x0 + 4 * q + i < a.w);
                    d = ok ? d : 0u;
                }
                sad += d;
                bp[k][i] = b;
            }
            if constexpr (FUSED) {
                uint32_t rf[4], ds[4];
                unpack4_in(raw + (r + 2) * G::RAW_W + G::HX + 4 * q, box.p, box.n, rf);
                unpack4_in(reinterpret_cast<const Pix*>(st + G::RAW_BYTES) + r * TW + 4 * q, st + G::RAW_BYTES,
                           G::DIST_BYTES, ds);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = (int)rf[i] - (int)ds[i];
                    sse_y += (Acc)((long long)e * e);
                }
            }
        }
        if constexpr (FUSED) {
            const Pix* sc = reinterpret_cast<const Pix*>(st + G::RAW_BYTES + G::DIST_BYTES);
            constexpr int CE = G::CH * G::CW;
            const int off = (tid >> 4) * G::CW + 4 * (tid & 15);
            uint32_t ru[4], du[4], rv[4], dv[4];
            unpack4_in(sc + off, sc, G::C_BYTES, ru);
            unpack4_in(sc + CE + off, sc + CE, G::C_BYTES, du);
            unpack4_in(sc + 2 * CE + off, sc + 2 * CE, G::C_BYTES, rv);
            unpack4_in(sc + 3 * CE + off, sc + 3 * CE, G::C_BYTES, dv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int eu = (int)ru[i] - (int)du[i], ev = (int)rv[i] - (int)dv[i];
                sse_u += (Acc)((long long)eu * eu);
                sse_v += (Acc)((long long)ev * ev);
            }
        }

        // ---- one atomic per block per accumulator
        if (do_sad || FUSED) {
            sad = warp_sum(sad);
            if constexpr (FUSED) {
                sse_y = warp_sum(sse_y);
                sse_u = warp_sum(sse_u);
                sse_v = warp_sum(sse_v);
            }
            if (lane == 0) {
                red[warp][0] = sad;
                red[warp][1] = sse_y;
                red[warp][2] = sse_u;
                red[warp][3] = sse_v;
            }
        }
        __syncthreads();
        if ((do_sad || FUSED) && warp == 0) {
            unsigned long long t0 = lane < NW ? red[lane][0] : 0ull;
            unsigned long long t1 = 0, t2 = 0, t3 = 0;
            if constexpr (FUSED) {
                t1 = lane < NW ? red[lane][1] : 0ull;
                t2 = lane < NW ? red[lane][2] : 0ull;
                t3 = lane < NW ? red[lane][3] : 0ull;
            }
#pragma unroll
            for (int o = NW / 2; o > 0; o >>= 1) {
                t0 += __shfl_xor_sync(0xffffffffu, t0, o);
                if constexpr (FUSED) {
                    t1 += __shfl_xor_sync(0xffffffffu, t1, o);
                    t2 += __shfl_xor_sync(0xffffffffu, t2, o);
                    t3 += __shfl_xor_sync(0xffffffffu, t3, o);
                }
            }
            if (lane == 0 && do_sad && MG_OK(a.sad_out + f, 8, a.sad_out, (size_t)a.n * 8))
                atomicAdd(a.sad_out + f, t0);
            if constexpr (FUSED) {
                if (lane == 1 && MG_OK(a.sse_out + 3LL * f + 0, 8, a.sse_out, (size_t)a.n * 24))
                    atomicAdd(a.sse_out + 3LL * f + 0, t1);
                if (lane == 2 && MG_OK(a.sse_out + 3LL * f + 1, 8, a.sse_out, (size_t)a.n * 24))
                    atomicAdd(a.sse_out + 3LL * f + 1, t2);
                if (lane == 3 && MG_OK(a.sse_out + 3LL * f + 2, 8, a.sse_out, (size_t)a.n * 24))
                    atomicAdd(a.sse_out + 3LL * f + 2, t3);
            }
        }
    }

    if (V2 && a.store_last && a.n > 0) {
        // keep the last raw frame for the next call (the last stage; border
        // tiles staged it with the mirror applied, so take in-frame samples only)
        const Pix* raw = reinterpret_cast<const Pix*>(smem + ((cnt - 1) & 1) * STAGE);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = rbase + 8 * k, y = y0 + r;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int x = x0 + 4 * q + i;
                if (y < a.h && x < a.w)
                    MG_ST(reinterpret_cast<Pix*>(a.raw_out + (long long)y * a.raw_pitch) + x,
                          MG_LD(raw + (r + 2) * G::RAW_W + G::HX + 4 * q + i, raw, G::RAW_BYTES),
                          a.raw_out, (size_t)a.h * a.raw_pitch);
            }
        }
        return;
    }
    if (a.store_last && a.n > 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int y = y0 + rbase + 8 * k;
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

template <typename Pix, bool FUSED, bool V2 = false>
static cudaError_t launch_one(const TileArgs& a, cudaStream_t s) {
    using G = Geo<Pix>;
    constexpr int STAGE = FUSED ? G::STAGE_FUSED : G::STAGE_MOTION;
    constexpr int SMEM = 2 * STAGE + G::SV_BYTES;
    // the shared-memory opt-in is per device; remember which devices have it
    static unsigned long long configured = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        e = cudaFuncSetAttribute(motion_tile_kernel<Pix, FUSED, V2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured, bit, __ATOMIC_RELEASE);
    }
    dim3 grid((a.w + TW - 1) / TW, (a.h + TH - 1) / TH);
    motion_tile_kernel<Pix, FUSED, V2><<<grid, NT, SMEM, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_motion_tile(const TileArgs& a, bool fused, cudaStream_t s, int* launches) {
    if (a.n <= 0) return cudaSuccess;
    *launches += 1;
    if (a.bpc == 8) return fused ? launch_one<uint8_t, true>(a, s) : launch_one<uint8_t, false>(a, s);
    return fused ? launch_one<uint16_t, true>(a, s) : launch_one<uint16_t, false>(a, s);
}

cudaError_t launch_motion_v2_tile(const TileArgs& a, cudaStream_t s, int* launches) {
    if (a.n <= 0) return cudaSuccess;
    *launches += 1;
    if (a.bpc == 8) return launch_one<uint8_t, false, true>(a, s);
    return launch_one<uint16_t, false, true>(a, s);
}

}  // namespace mg
