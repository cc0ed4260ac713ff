// motion_internal.h -- host-side launch interface between the C-ABI layer and
// the kernels of libmotion_gb300.  Internal; not installed.
#pragma once

#include <cstdint>
#include <cstddef>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace mg {

// Arguments of one batched motion (+ optional fused 4:2:0 SSE) launch.  All
// plane pointers are byte pointers; pitches and strides are in bytes.  Passed
// by value and only ever read field by field (no runtime-indexed arrays).
struct TileArgs {
    const uint8_t* ref_y;
    const uint8_t* dist_y;
    const uint8_t* ref_u;
    const uint8_t* dist_u;
    const uint8_t* ref_v;
    const uint8_t* dist_v;
    long long pitch_y, pitch_uv, stride_y, stride_uv;
    int w, h, cw, ch, bpc, n;
    int has_prev;       // B of the previous frame is in bprev
    int store_last;     // write B of the last frame to bprev
    int aligned16;      // every plane base, pitch and stride is 16-byte aligned
    uint16_t* bprev;      // resident blurred plane read as B_prev (has_prev), bprev_pitch per row
    uint16_t* bprev_out;  // plane that receives B of the last frame (store_last)
    int bprev_pitch;
    unsigned long long* sad_out;  // [n], zeroed by the caller
    unsigned long long* sse_out;  // [n][3], zeroed by the caller (fused only)
    int* err;                     // device error word (bit 0: a stage wait timed out)
    int chunk;                    // TMA kernel: frames per CTA (grid.z = ceil(n / chunk))
    // TMA kernel, split tail (tiles_a > 0; see block_work): a one-dimensional
    // grid whose first tiles_a blocks take tiles 0 .. tiles_a-1 whole and whose
    // other blocks take the remaining tiles in chunks of chunk_b frames
    int tiles_a, chunk_b;
    int force_rows;               // motion-only TMA tile height: 0 chosen per launch, 32 or 16 forced
    long long wait_cycles;        // bound of every mbarrier wait (0: about one second)
    int tx_extra;                 // test hook: bytes a stage expects beyond its boxes (0)
    // motion_v2 (blur of prev - cur): the last raw frame of the previous call
    // (read when has_prev) and the plane that receives this call's last frame
    const uint8_t* raw_prev;      // w x h samples, raw_pitch bytes per row
    uint8_t* raw_out;
    long long raw_pitch;
};

// Tensor maps of one TMA launch (64-byte aligned, passed as a grid constant).
struct TmaMaps {
    CUtensorMap raw;              // reference luma, box (TW + 2 HX) x (TH + 4) x 1
    CUtensorMap dist;             // distorted luma, box TW x TH x 1
    CUtensorMap ru, du, rv, dv;   // chroma planes, box TW/2 x TH/2 x 1
    CUtensorMap prev;             // motion_v2: the previous call's last raw frame, box as raw
};

// Arguments of one batched SSE launch over n pairs x (1 or 3) planes.
struct SseArgs {
    const uint8_t* ref_y;
    const uint8_t* dist_y;
    const uint8_t* ref_u;
    const uint8_t* dist_u;
    const uint8_t* ref_v;
    const uint8_t* dist_v;
    long long ref_pitch_y, dist_pitch_y, pitch_uv, stride_y, stride_uv;
    int w, h, cw, ch, bpc, n, planes;  // planes: 1 (luma only) or 3
    unsigned long long* sse_out;       // [n][planes], zeroed by the caller
};

// Generic kernel: any pitch / alignment (sample loads on border tiles).
cudaError_t launch_motion_tile(const TileArgs& a, bool fused, cudaStream_t s,
                               int* launches);
// TMA kernel: 16-byte aligned layouts.  *used is false when the layout does not
// suit TMA (nothing launched; the caller falls back to launch_motion_tile).
cudaError_t launch_motion_tma(const TileArgs& a, bool fused, cudaStream_t s, int* launches,
                              bool* used);
// motion_v2 (the blur of prev - cur, floor rounding, SAD of |blur|): TMA
// kernel when the layout allows (*used), else the generic kernel.
cudaError_t launch_motion_v2_tma(const TileArgs& a, cudaStream_t s, int* launches, bool* used);
cudaError_t launch_motion_v2_tile(const TileArgs& a, cudaStream_t s, int* launches);
// Whether the TMA kernel can take a's planes (16-byte strides and bases; the
// driver's tensor-map encoder available).
bool tma_usable(const TileArgs& a, bool fused);
// The output tile of the motion kernels (the TMA kernel's TW x TH); the TMA
// kernel's motion-only launches under one wave take tiles of kShortTileH rows.
constexpr int kTileW = 128, kTileH = 32, kShortTileH = 16;
// The tile and frame chunk of block `lin` (x fastest, then y, then chunk) of a
// TMA launch over gx x gy tiles of th rows and gz chunks.  Tiles whose staged rows reach
// past the top or bottom frame edge (tile row 0 and the rows after niy), and
// a partial last tile column, run the border copy of the frame loop; all other
// tiles run the interior copy -- the left and right edge columns included,
// whose halo lanes read the mirrored columns inside the frame instead.  The
// border tiles of every chunk come first, then the interior tiles in row-major
// order, so that horizontally and vertically adjacent tiles run at the same
// time and share their halo columns and rows in L2; an SM that ran both
// copies of the loop at once would miss in its instruction cache, and in this
// order only the first wave mixes them.  A bijection of [0, gx gy gz).
__host__ __device__ inline void tile_of_block(int w, int h, int gx, int gy, int gz, int lin,
                                              int* tx, int* ty, int* cz, int th = kTileH) {
    const int niy = h >= th + 2 ? (h - th - 2) / th : 0;   // interior rows 1..niy
    const int nfull = w / kTileW;                                       // full columns 0..nfull-1
    const int ni = nfull * niy, nb = gx * gy - ni;
    if (lin >= nb * gz) {
        const int idx = lin - nb * gz;
        *cz = idx / ni;
        const int r = idx - *cz * ni;
        *ty = 1 + r / nfull;
        *tx = r % nfull;
        return;
    }
    *cz = lin / nb;
    const int r = lin - *cz * nb;
    const int nbr = (gy - niy) * gx;   // whole border rows: row 0 and rows after niy
    if (r < nbr) {
        const int k = r / gx;
        *tx = r % gx;
        *ty = k == 0 ? 0 : niy + k;
    } else {                           // rows 1..niy: the partial last column
        const int rr = r - nbr, per = gx - nfull;
        *ty = 1 + rr / per;
        *tx = nfull + rr % per;
    }
}
// The work of block `lin` of a TMA launch over n frames of w x h in tiles of
// th rows: its tile (tile_of_block order) and frames [*f_begin, *f_end).  Uniform launches
// (tiles_a == 0) run gx x gy x gz blocks, each tile in gz chunks of `chunk`
// frames.  Split-tail launches (tiles_a > 0) run tiles_a whole tiles first
// and then the other tiles in chunks of chunk_b frames, chunk-major, so that
// the last blocks to start are short.  A block whose chunk starts after frame
// 0 also blurs the frame before it (no output for that frame).
__host__ __device__ inline void block_work(int w, int h, int gx, int gy, int gz, int n, int chunk,
                                           int tiles_a, int chunk_b, int lin, int* tx, int* ty,
                                           int* f_begin, int* f_end, int th = kTileH) {
    int cz = 0, len = chunk > 0 ? chunk : n;
    if (tiles_a > 0) {
        int t = lin, dz;
        len = n;
        if (lin >= tiles_a) {
            const int tb = gx * gy - tiles_a;
            const int r = lin - tiles_a;
            cz = r / tb;
            t = tiles_a + (r - cz * tb);
            len = chunk_b;
        }
        tile_of_block(w, h, gx, gy, 1, t, tx, ty, &dz, th);
    } else {
        tile_of_block(w, h, gx, gy, gz, lin, tx, ty, &cz, th);
    }
    *f_begin = cz * len;
    *f_end = *f_begin + len < n ? *f_begin + len : n;
}
// The split-tail plan of a one-chunk launch of `tiles` tiles over `slots`
// resident blocks (host only): when the tiles fill more than one wave and
// the last wave is at most half full, the tiles of the full waves stay whole
// (*tiles_a) and the rest are split into chunks of *chunk_b frames (at least
// 4, a tile's last chunk the remainder; at most 8 chunks, as many as the last
// wave has room for);
// returns the block count, or 0 (and *tiles_a = 0) for no split.
long long plan_split_tail(long long tiles, long long slots, int n, int* tiles_a, int* chunk_b);

// Chunks of a TMA launch (host only): n frames over `tiles` tiles with
// `slots` CTAs resident on the device at once; 1 <= result <= max_c; v2
// selects the motion_v2 kernel's constants.
int plan_frame_chunks(long long tiles, long long slots, int n, int max_c, bool v2 = false);
// The plan of a TMA launch (host only): chunks of `chunk` frames over gz
// chunks (tiles_a == 0), or a split tail (tiles_a > 0, see block_work).  The
// motion and fused kernels take the split tail whenever the one-chunk launch
// has one (whole tiles keep their frames; only the last wave's tiles pay a
// warm-up frame); motion_v2 takes it only when plan_frame_chunks picks one
// chunk; a launch that continues in place (same_plane) always runs one chunk.
struct LaunchPlan {
    int chunk, gz, tiles_a, chunk_b;
    long long blocks;
};
LaunchPlan plan_launch(long long tiles, long long slots, int n, bool v2, bool same_plane);
// Whether a motion-only TMA launch takes tiles of kShortTileH rows (host
// only): its tiles32 tiles of kTileH rows, in their planned chunks, fit in
// one wave of slots32 resident CTAs.
inline bool prefer_short_tiles(long long tiles32, long long slots32, int n, int max_c, bool v2) {
    return tiles32 * plan_frame_chunks(tiles32, slots32, n, max_c, v2) <= slots32;
}
cudaError_t launch_sse(const SseArgs& a, cudaStream_t s, int sm_count, int* launches);

// Copies of planes into rows the TMA can address (repitch.cu): n frames of
// `rows` rows of row_bytes bytes, source rows `pitch` and frames `stride` bytes
// apart, destination rows dpitch (a multiple of 16) and frames dstride apart.
constexpr int kRepitchMaxPlanes = 6;
struct RepitchPlane {
    const uint8_t* src;
    long long pitch, stride;
    uint8_t* dst;
    long long dpitch, dstride;
    int row_bytes, rows;
};
struct RepitchArgs {
    RepitchPlane p[kRepitchMaxPlanes];
    int planes, n;
    int* err;   // device error word (the bounds-checked build reports failed checks here)
};
// The largest power of two up to 16 dividing every source base, pitch and stride.
int repitch_granule(const RepitchArgs& a);
cudaError_t launch_repitch(const RepitchArgs& a, cudaStream_t s, int sm_count, int* launches);

// Moment sums of n luma pairs (sum ref, sum dist, sum ref^2, sum dist^2).
struct MomentArgs {
    const uint8_t* ref;
    const uint8_t* dist;
    long long pitch, stride;        // shared by both pictures
    int w, h, bpc, n;
    unsigned long long* out;        // [n][4], zeroed by the caller
};
cudaError_t launch_moment(const MomentArgs& a, cudaStream_t s, int sm_count, int* launches);

// Adds to the library-wide kernel launch count (motion_kernel_launch_count).
void note_launches(int n);

// Host-side argument checks shared by the entry points (motion_capi.cu); each
// returns MOTION_OK or a MOTION_ERR_* code of include/motion.h.
// Bytes per sample: 1 at 8 bits, 2 above.
int sample_bytes(int bpc);
// bpc in [8, 16], 3 <= w, h <= MOTION_MAX_DIM.
int check_dims(int w, int h, int bpc);
// n planes of w samples per row, rows `pitch` bytes apart, planes `stride`
// bytes apart: a non-null base, pitch >= w samples, 2-byte alignment for
// uint16 samples, pitch <= 2^40, stride <= 2^46, n strides within 2^48.
int check_layout(const void* p, size_t pitch, size_t stride, int n, int w, int bpc);

}  // namespace mg
