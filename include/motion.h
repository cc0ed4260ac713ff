/*
 * motion.h -- C ABI of the GB300 integer motion / PSNR-SSE library
 * (libmotion_gb300.so, built for sm_103a).
 *
 * What it computes (the integer motion feature of a video-quality pipeline):
 *   For each frame F (h rows x w columns, bpc bits per sample):
 *     V[y][x] = (sum_k t_k F[mirror(y+k-2, h)][x] + 2^(bpc-1)) >> bpc
 *     B[y][x] = (sum_k t_k V[y][mirror(x+k-2, w)] + 2^15) >> 16
 *   with t = {3571, 16004, 26386, 16004, 3571} (sum 65536) and
 *   mirror(i, n) = i < 0 ? -i : (i >= n ? 2n - i - 2 : i);
 *     SAD_i     = sum_{y,x} |B_i[y][x] - B_{i-1}[y][x]|   (uint64, exact)
 *     score_i   = ((double)SAD_i / 256.0) / (double)(w * h)
 *     motion2_i = min(score_i, score_{i+1})
 *   and, per plane of a reference/distorted pair,
 *     SSE = sum (ref - dist)^2                             (uint64, exact).
 *
 * Sources, by page title and section:
 *   "ADR-1392: CUDA motion, PSNR and moment kernels add one atomic per block,
 *   the motion SAD filters separably, and PSNR selects its plane with constant
 *   indices" -- Context (one integer per pixel summed into one 64-bit value,
 *   equal to the CPU bit for bit; order-independent, so any reduction order is
 *   exact), Decision 1 (one atomic per block), Decision 3 (planes selected with
 *   constant indices), Decision 4 (vertical pass first, rounded >> bpc, then
 *   the horizontal taps, rounded >> 16).
 *   "ADR-1380: The CUDA SpEED twins are device-resident ..." -- Decision
 *   (submit enqueues on the caller's stream; one small readback per frame).
 *   "Making it fast: three rounds on one pipeline" -- Round 1 (batched launches,
 *   one kernel over all frames), Round 2 (no allocation on the hot path).
 *
 * Conventions for every entry point:
 *   - Return 0 (MOTION_OK) on success or a MOTION_ERR_* code; nothing is written
 *     to an output on error.  motion_strerror() names a code.
 *   - Device errors: the motion kernels never spin without bound.  A stage
 *     wait that runs out (about one second), or a failed check in the
 *     bounds-checked build, sets a sticky device error word (one per context;
 *     one per device for the allocation-free entry point) and the kernel
 *     leaves, so its results are incomplete.  The calls that wait for their
 *     results anyway (motion_submit, which reads the word in the same 16-byte
 *     readback as the SAD, and the two host-buffer calls, which read it after
 *     their final synchronisation) return MOTION_ERR_DEVICE and write no
 *     output; the asynchronous calls cannot see it, and motion_device_error
 *     (motion_noalloc_device_error) is their collect step.  Whenever the word
 *     is found set it is cleared and the context's sequences restart (the next
 *     frame has SAD 0), since the resident planes may be incomplete (the
 *     per-frame result readback behind the stream, ADR-1380 Decision).
 *   - "d_" pointers are device memory (cudaMalloc / PyTorch CUDA tensors) owned
 *     by the caller; "h_" pointers are host memory owned by the caller (pinned
 *     memory gives full copy speed; pageable memory works).
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Device-result calls only enqueue work on it.
 *   - Samples are uint8 when bpc == 8 and little-endian uint16 when
 *     9 <= bpc <= 16.  Values >= 2^bpc violate a precondition and give
 *     unspecified (but memory-safe) results.  uint16 planes must be 2-byte
 *     aligned (pointer, pitch and frame stride).
 *   - pitch / stride arguments are in BYTES; a pitch above 2^40, a frame
 *     stride above 2^46 or n frames spanning more than 2^48 bytes is
 *     MOTION_ERR_INVALID_ARGUMENT.
 *   - Frames must be at least 3 x 3 (the mirror rule needs n >= 3) and at most
 *     MOTION_MAX_DIM on each side.
 *   - Calls on one context must not overlap (one stream per context, or
 *     ordered by the caller); distinct contexts are independent and may be
 *     driven from different host threads at the same time (the library's
 *     one-time set-up -- driver entry point, launch attributes, occupancy --
 *     is safe under that race).  motion_inject_alloc_failure is process-wide.
 *   - CUDA graphs: the device-result calls (motion_submit_batch,
 *     motion_v2_submit_batch, motion_psnr_yuv420_batch, psnr_sse,
 *     psnr_sse_yuv420_batch, moment_sums_batch) enqueue only stream work (an
 *     output memset and their kernels) and motion_reset changes host state only,
 *     so a stream capture of them replays the same computation.  A context's sequence state (which
 *     resident plane holds the previous frame's blur, whether there is one)
 *     advances when a call is captured, not when it is replayed: capture a
 *     sequence that starts with motion_reset and every replay computes it
 *     from its first frame; a direct call after a replay continues from the
 *     replay's last frame.  Make one direct call of each kind before
 *     capturing (motion_v2 allocates its raw planes on its first call).  The
 *     host-buffer and single-frame calls (motion_psnr_yuv420_batch_host,
 *     motion_submit) synchronise and are not capturable.  A call whose planes
 *     are not 16-byte aligned adds one copy kernel (see motion_set_kernel_path)
 *     and allocates its scratch the first time: make it once directly too.
 */
#ifndef MOTION_GB300_H
#define MOTION_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOTION_MAX_DIM 32768

#if defined(__GNUC__)
#define MOTION_API __attribute__((visibility("default")))
#else
#define MOTION_API
#endif

enum motion_status {
    MOTION_OK = 0,
    MOTION_ERR_INVALID_ARGUMENT = 1,   /* NULL pointer, n < 0, bad plane index, layout too large */
    MOTION_ERR_FRAME_TOO_SMALL = 2,     /* w < 3 or h < 3 */
    MOTION_ERR_UNSUPPORTED_BITDEPTH = 3,/* bpc outside [8, 16] */
    MOTION_ERR_BAD_PITCH = 4,           /* pitch < w * sample size, or misaligned uint16 layout */
    MOTION_ERR_TOO_LARGE = 5,           /* w or h > MOTION_MAX_DIM */
    MOTION_ERR_CUDA = 6,                /* a CUDA runtime call failed (motion_last_cuda_error) */
    MOTION_ERR_OUT_OF_MEMORY = 7,       /* device or pinned allocation failed */
    MOTION_ERR_NO_DEVICE = 8,           /* no CUDA device visible */
    MOTION_ERR_WRONG_DEVICE = 9,        /* called with a device other than the context's */
    MOTION_ERR_DEVICE = 10              /* a kernel set the device error word: results incomplete */
};

typedef struct motion_ctx motion_ctx;  /* opaque, library-owned */

/* Create a motion context for frames of w x h samples at bpc bits on the
 * current CUDA device.  All device scratch (two w*h uint16 planes that take
 * turns holding the previous frame's blur, so that one launch can read one and
 * write the other) is allocated here, never on a submit.  *out receives the
 * handle. */
MOTION_API int motion_init(int w, int h, int bpc, motion_ctx** out);

/* Free the context and its device memory.  NULL is accepted. */
MOTION_API int motion_destroy(motion_ctx* ctx);

/* Start a new sequence: the next frame submitted has SAD 0 / score 0. */
MOTION_API int motion_reset(motion_ctx* ctx);

/* Submit ONE frame (device memory, pitch_bytes between rows).  Enqueues the
 * blur + SAD on `stream`, waits for it, and returns the frame's SAD against
 * the previously submitted frame (0 for the first frame of a sequence) and its
 * score.  Either output pointer may be NULL.  Follows the submit / collect
 * pattern with one small readback per frame (ADR-1380, Decision): 16 bytes,
 * the SAD and the context's device error word; if the word is set the call
 * returns MOTION_ERR_DEVICE, writes neither output, clears the word and
 * restarts the sequence. */
MOTION_API int motion_submit(motion_ctx* ctx, const void* d_frame, size_t pitch_bytes,
                  void* stream, uint64_t* sad_out, double* score_out);

/* Submit n frames in ONE launch (ADR-1392 Decision 1; "Making it fast",
 * Round 1, batched launches).  Frame i starts at d_frames + i*frame_stride
 * bytes.  d_sad_out (device, n uint64) receives SAD_i against frame i-1; SAD_0
 * is against the last frame of the previous submit on this context, or 0 at
 * the start of a sequence.  Asynchronous: only enqueues on `stream`.  n == 0
 * is a no-op. */
MOTION_API int motion_submit_batch(motion_ctx* ctx, const void* d_frames, int n,
                        size_t frame_stride_bytes, size_t pitch_bytes,
                        void* stream, uint64_t* d_sad_out);

/* motion_v2 over n frames in ONE launch ("ADR-1392: CUDA motion, PSNR and
 * moment kernels add one atomic per block, ...", Decision 4: stage prev - cur,
 * vertical 5-tap pass with the CPU's rounding (>> bpc), then the 5 horizontal
 * taps (>> 16)).  With the same taps and mirror rule as motion_submit_batch,
 * each frame i gives the blur Bd of D = F_{i-1} - F_i, where a right shift
 * of a negative sum rounds towards minus infinity, and d_sad_out[i] =
 * sum |Bd| (device uint64[n]).  SAD_0 is against the last frame of the
 * previous motion_v2 call on this context, or 0 at the start of a sequence
 * (motion_reset starts one).  The context keeps the last raw frame in two
 * planes of its own that alternate between calls; the first motion_v2 call
 * on a context allocates them (2 w h bytes per sample).  The motion_v2
 * sequence state is independent of motion_submit_batch's.  Frame layout,
 * alignment handling, asynchrony and errors as motion_submit_batch. */
MOTION_API int motion_v2_submit_batch(motion_ctx* ctx, const void* d_frames, int n,
                                      size_t frame_stride_bytes, size_t pitch_bytes,
                                      void* stream, uint64_t* d_sad_out);

/* Fused pass over n 4:2:0 reference/distorted picture pairs in ONE launch:
 * motion SAD on the reference luma (continuing the context's sequence, as
 * motion_submit_batch) and SSE of each plane Y, U, V of every pair.
 * Luma planes are ctx w x h; chroma planes ceil(w/2) x ceil(h/2).  Reference
 * and distorted pictures share one layout: pitch_y / pitch_uv between rows,
 * stride_y / stride_uv between pairs.  d_sad_out: device uint64[n];
 * d_sse_out: device uint64[n][3] (Y, U, V).  Asynchronous. */
MOTION_API int motion_psnr_yuv420_batch(motion_ctx* ctx, int n,
                             const void* d_ref_y, const void* d_ref_u,
                             const void* d_ref_v, const void* d_dist_y,
                             const void* d_dist_u, const void* d_dist_v,
                             size_t pitch_y, size_t pitch_uv,
                             size_t stride_y, size_t stride_uv, void* stream,
                             uint64_t* d_sad_out, uint64_t* d_sse_out);

/* The same fused pass with HOST pictures and HOST results: the library copies
 * chunks of pairs host->device into its own staging buffers (allocated on the
 * first call and kept; size them with motion_reserve_host_staging to keep the
 * first call allocation-free) on two streams so that copies overlap the
 * kernels, and copies the results back through a pinned result buffer the
 * context keeps (grown to n pairs when a call needs more; the caller's result
 * arrays may be pageable).  Blocks until h_sad_out (uint64[n]) and h_sse_out
 * (uint64[n][3]) are written.  Host planes are tightly packed with the given
 * pitches and strides.  Pinned host memory recommended for the pictures.
 * After the last chunk the context's device error word is read: if a kernel
 * set it the call returns MOTION_ERR_DEVICE, writes no output, clears the
 * word and restarts the sequence. */
MOTION_API int motion_psnr_yuv420_batch_host(motion_ctx* ctx, int n,
                                  const void* h_ref_y, const void* h_ref_u,
                                  const void* h_ref_v, const void* h_dist_y,
                                  const void* h_dist_u, const void* h_dist_v,
                                  size_t pitch_y, size_t pitch_uv,
                                  size_t stride_y, size_t stride_uv,
                                  uint64_t* h_sad_out, uint64_t* h_sse_out);

/* motion_submit_batch with HOST frames and HOST results: n frames
 * (frame_stride bytes apart, rows pitch bytes apart, as motion_submit_batch)
 * are copied host->device in chunks of frames_per_chunk frames (0 picks about
 * 256 MB of frames, 1 to 256) into the context's staging sets on one stream
 * while the motion kernel of the previous chunk runs on another ("Making it
 * fast" -- the upload is the wall-time bottleneck; the same pipeline as
 * motion_psnr_yuv420_batch_host, whose staging sets it shares and grows when
 * needed).  The frames continue the context's sequence (SAD_0 against the last
 * frame of the previous call, device or host).  Blocks until h_sad_out
 * (uint64[n]) is written; pinned host frames give full copy speed.  Errors as
 * motion_submit_batch, plus MOTION_ERR_BAD_PITCH if consecutive host frames
 * overlap; after a CUDA error the sequence may have advanced by the chunks
 * that ran.  MOTION_ERR_DEVICE as motion_psnr_yuv420_batch_host. */
MOTION_API int motion_submit_batch_host(motion_ctx* ctx, const void* h_frames, int n,
                                        size_t frame_stride_bytes, size_t pitch_bytes,
                                        int frames_per_chunk, uint64_t* h_sad_out);

/* Allocate the two device staging sets, result buffers and streams used by
 * motion_psnr_yuv420_batch_host, for chunks of `pairs_per_chunk` pairs whose
 * planes are stride_y / stride_uv bytes apart (0 picks about 256 MB of
 * pictures per chunk, 1 to 64 pairs, so the two sets take about 512 MB of
 * device memory; a stride of 0 means tightly packed rows).  Kept until
 * destroy; a later call with a larger need reallocates. */
MOTION_API int motion_reserve_host_staging(motion_ctx* ctx, int pairs_per_chunk,
                                size_t stride_y, size_t stride_uv);

/* SSE of one plane pair (ADR-1392 Context / Decision 2): d_sse_out (device,
 * one uint64) receives sum (ref - dist)^2.  Stateless; asynchronous. */
MOTION_API int psnr_sse(const void* d_ref, const void* d_dist, size_t ref_pitch,
             size_t dist_pitch, int w, int h, int bpc, void* stream,
             uint64_t* d_sse_out);

/* SSE of all three planes of n 4:2:0 pairs in ONE launch, planes selected
 * with constant indices (ADR-1392 Decision 3).  Layout as in
 * motion_psnr_yuv420_batch; d_sse_out: device uint64[n][3].  Stateless. */
MOTION_API int psnr_sse_yuv420_batch(int w, int h, int bpc, int n,
                          const void* d_ref_y, const void* d_ref_u,
                          const void* d_ref_v, const void* d_dist_y,
                          const void* d_dist_u, const void* d_dist_v,
                          size_t pitch_y, size_t pitch_uv, size_t stride_y,
                          size_t stride_uv, void* stream, uint64_t* d_sse_out);

/* Moment sums of n picture pairs' luma planes in ONE launch ("ADR-1392: CUDA
 * motion, PSNR and moment kernels add one atomic per block, ...", Decision 6:
 * four accumulators -- the reference and distorted sums and sums of squares --
 * each added once per block; Context: exact 64-bit integer sums).
 * d_ref / d_dist: device w x h planes, `pitch` bytes between rows and `stride`
 * bytes between pairs (one layout for both pictures; pairs must not overlap);
 * uint8 samples for bpc 8, little-endian uint16 for bpc 9..16.  d_out: device
 * uint64[n][4] = {sum ref, sum dist, sum ref^2, sum dist^2}, zeroed and then
 * written by the call.  Asynchronous on `stream` (a cudaStream_t, NULL for the
 * legacy default stream).  w, h >= 1.  16-byte aligned pointers, pitch and
 * stride take the vector path; any other layout is served sample by sample.
 * Errors: MOTION_ERR_UNSUPPORTED_BITDEPTH, MOTION_ERR_INVALID_ARGUMENT (n < 0,
 * w or h < 1, null pointers), MOTION_ERR_TOO_LARGE, MOTION_ERR_BAD_PITCH,
 * MOTION_ERR_CUDA; nothing is launched on error.  n == 0 is a no-op. */
MOTION_API int moment_sums_batch(int w, int h, int bpc, int n, const void* d_ref,
                                 const void* d_dist, size_t pitch, size_t stride,
                                 void* stream, uint64_t* d_out);

/* Host, no GPU: the moments from moment sums, each sum over the sample count
 * w*h in double -- out[i][0..3] = mean of ref, mean of dist, mean square of
 * ref, mean square of dist (the first and second moments of each picture).
 * sums: host uint64[n][4]; out: host double[n][4]. */
MOTION_API int moments_from_sums(const uint64_t* sums, int n, int w, int h, double* out);

/* Host helper: score_i = (SAD_i / 256) / (w h) and motion2_i =
 * min(score_i, score_{i+1}); motion2_{n-1} = score_{n-1} unless next_score
 * (the score of the frame after the last, e.g. from the next shard) is
 * non-NULL.  All pointers are host memory. */
MOTION_API int motion_scores_from_sad(const uint64_t* sad, int n, int w, int h,
                           const double* next_score, double* score,
                           double* motion2);

/* Host helper: mse = SSE / n_samples and psnr_db = 10 log10((2^bpc-1)^2 /
 * mse), +inf when SSE == 0 (no cap). */
MOTION_API int psnr_from_sse(uint64_t sse, uint64_t n_samples, int bpc, double* mse,
                  double* psnr_db);

/* Kernel selection for a context (diagnostics and tests): MOTION_PATH_AUTO
 * always uses the TMA kernel -- planes whose base, pitch or frame stride is
 * not a multiple of 16 bytes are first copied, in one more launch, into a
 * scratch the context owns with 16-byte-aligned rows (allocated by the first
 * such call, n frames' or pairs' worth up to motion_set_copy_limit, grown
 * when a call needs more, freed by motion_destroy); MOTION_PATH_GENERIC
 * always uses the generic kernel, which reads any layout in place;
 * MOTION_PATH_TMA_32 and MOTION_PATH_TMA_16 are MOTION_PATH_AUTO with the
 * tile height of the motion-only launches (motion and motion_v2) fixed at
 * 128 x 32 or 128 x 16 instead of chosen per launch (motion_launch_shape).
 * Results are identical on every path. */
#define MOTION_PATH_AUTO 0
#define MOTION_PATH_GENERIC 1
#define MOTION_PATH_TMA_32 2
#define MOTION_PATH_TMA_16 3
MOTION_API int motion_set_kernel_path(motion_ctx* ctx, int path);

/* The most scratch the copy of MOTION_PATH_AUTO may use for one launch, in
 * bytes (0, the default: 1 GiB).  A call whose planes need the copy and do
 * not fit runs as several launches of as many frames (or pairs) as fit, each
 * continuing the sequence; results are the same. */
MOTION_API int motion_set_copy_limit(motion_ctx* ctx, size_t bytes);

/* Diagnostic, host only, no GPU: the number of frame chunks (1..8) a batched
 * launch of n frames of w x h in 128 x 32 tiles splits into on a device where
 * `resident_ctas` motion CTAs run at once (4 per SM on GB300: 608).  The launch sizing
 * follows "ADR-1226: Size the CUDA AIM CM launch by SM count, not by a fixed
 * rows-per-thread": chunks after the first re-blur one warm-up frame, and
 * the count balances that work against the idle part of the last wave.  This
 * is the plan of the motion and fused kernels' uniform launches (a launch
 * that splits its tail instead, see motion_launch_blocks, runs its full waves
 * in one chunk); motion_v2 launches weigh a partial last wave less (1080p x
 * 16 frames: two chunks).
 * *chunks_out (host int) receives the count.  Errors:
 * MOTION_ERR_INVALID_ARGUMENT (w, h < 1, n < 0, resident_ctas < 1, NULL
 * chunks_out).  A launch that continues a sequence in place (the
 * allocation-free entry point) always uses one chunk. */
MOTION_API int motion_plan_chunks(int w, int h, int n, int resident_ctas, int* chunks_out);

/* Diagnostic, host only, no GPU: the output tile and frame chunk that block
 * `block` of a batched TMA launch of w x h frames in `chunks` chunks works on
 * (blocks counted x fastest, then y, then chunk, over ceil(w/128) x
 * ceil(h/32) x chunks blocks).  The tiles that read mirrored rows (the top
 * tile row and the rows whose halo passes the bottom edge) or hold a partial
 * last column come first for every chunk, then the other tiles in row-major
 * order -- the full tiles of the left and right edges among them, which read
 * their mirrored halo columns directly -- so that after the first wave an SM
 * runs one kind of frame loop at a time and neighbouring tiles share their
 * halos in L2.  tile_out (host int[3]) receives
 * {tile column, tile row, chunk}.  Errors: MOTION_ERR_INVALID_ARGUMENT (w, h
 * outside 1..32768, chunks outside 1..8, block outside the launch, NULL
 * tile_out). */
MOTION_API int motion_tile_order(int w, int h, int chunks, long long block, int* tile_out);

/* Diagnostic, host only, no GPU: the tile height of a batched motion-only
 * launch (motion_v2 when v2 != 0; the fused 4:2:0 launches always take 32):
 * 16 when its 128 x 32 tiles, in their motion_plan_chunks chunks, fit in one
 * wave of `resident_ctas` resident CTAs (608 on GB300), else 32.  Under one
 * wave each block runs a long serial chain of frames on SMs that are not
 * full; 128 x 16 tiles give twice the blocks, each warp 4 output rows instead
 * of 8, and 7 CTAs per SM instead of 4 (1080p x 16 frames: 1020 blocks of 16
 * rows instead of 510 of 32).  *tile_rows (host int) receives 16 or 32.
 * Errors: MOTION_ERR_INVALID_ARGUMENT (w, h outside 1..32768, n < 1,
 * resident_ctas < 1, NULL tile_rows). */
MOTION_API int motion_launch_shape(int w, int h, int n, int v2, int resident_ctas, int* tile_rows);

/* Diagnostic, host only, no GPU: the blocks of a batched motion launch of n
 * frames of w x h in tiles of 128 x tile_rows (32 or 16, see
 * motion_launch_shape) on a device where `resident_ctas` blocks of that tile
 * run at once (GB300: 608 of 32 rows, 1064 of 16).  The launch is sized by
 * the SM count ("ADR-1226: Size the CUDA AIM CM launch by SM count, not by a
 * fixed rows-per-thread"): a launch of more than a wave whose last wave
 * would be at most half full keeps the tiles of its full waves whole (one
 * chunk of all n frames) and splits the other tiles into chunks (of at least
 * 4 frames but the last, at most 8 per tile), so that the blocks that start
 * last are short (the fused 4K 4:2:0 launch of 50 pairs: 1824 whole tiles and
 * 216 tiles in two chunks of 25); other launches run their frames in
 * motion_plan_chunks chunks.  A chunk that starts after frame
 * 0 blurs the frame before it as well (no output for it).  *blocks_out (host)
 * receives the block count; for 0 <= block < that count, work_out (host
 * int[4]) receives {tile column, tile row, first frame, end frame} of that
 * block (block < 0: the count only).  Errors: MOTION_ERR_INVALID_ARGUMENT (w,
 * h outside 1..32768, n < 1, tile_rows not 16 or 32, resident_ctas < 1, NULL
 * blocks_out, block past the launch or NULL work_out).  The allocation-free
 * entry point, which continues in place, never splits. */
MOTION_API int motion_launch_blocks(int w, int h, int n, int tile_rows, int resident_ctas, long long block,
                                    int* work_out, long long* blocks_out);

/* Test hook for allocation failures (not part of the method): the nth
 * device or pinned-host allocation the library makes from now on (1 = the
 * next one) fails with MOTION_ERR_OUT_OF_MEMORY without reaching the driver;
 * 0 turns it off.  Library-wide.  Every entry point that allocates (init,
 * the first motion_v2 call, the first call that needs the copy scratch, the
 * host-buffer staging and result buffers) then returns the error, frees what
 * it had allocated for that call, and leaves the context usable.  Errors:
 * MOTION_ERR_INVALID_ARGUMENT for nth < 0. */
MOTION_API int motion_inject_alloc_failure(int nth);

/* Test hook for the kernels' bounded waits (not part of the method):
 * while on, TMA launches on this context expect 16 bytes per stage more than
 * their boxes deliver, so no stage wait can complete, and bound every wait at
 * about 2 ms; the kernels then set bit 0 of the device error word and leave.
 * Results of such launches are incomplete.  Turn it off to compute again. */
MOTION_API int motion_set_stall_injection(motion_ctx* ctx, int on);

/* The collect step of the asynchronous calls: read and clear the context's
 * device error word after waiting for the device.  Bit 0 set means a
 * kernel's bounded wait for a staged tile ran out, bit 1 a failed check in
 * the bounds-checked build; the results written since the previous read are
 * then incomplete, and the context's sequences restart (the next frame has
 * SAD 0).  *flags receives the word; the return is MOTION_OK when it could be
 * read. */
MOTION_API int motion_device_error(motion_ctx* ctx, int* flags);

/* Largest frame of motion_submit_batch_noalloc: rows of round_up(w, 8)
 * samples times h must not exceed this (3840x2160 and 4096x2048 fit). */
#define MOTION_NOALLOC_MAX_SAMPLES (8u * 1024u * 1024u)

/* Batched motion SAD that allocates nothing (not part of the method: it
 * exists for callers that may not allocate device memory -- a host program
 * that owns all device memory through its own pool and forbids libraries to
 * call cudaMalloc, or a latency-critical loop where an allocation, which can
 * synchronise the device, is not acceptable).  Same result as
 * motion_submit_batch on a context of size w x h at bpc bits, without a
 * context: the previous frame's blurred plane is kept in a fixed 16 MiB array
 * built into the library (MOTION_NOALLOC_MAX_SAMPLES uint16 values; every GPU
 * that loads the library holds it until the process exits).  continue_sequence
 * = 0 starts a sequence (SAD_0 = 0); 1 compares frame 0 with the last frame of
 * the previous call on this device, which must have had the same w, h and bpc
 * (else MOTION_ERR_INVALID_ARGUMENT).  Frames larger than the array give
 * MOTION_ERR_TOO_LARGE.  d_sad_out (device, n uint64) is zeroed on `stream`
 * and filled asynchronously.  The first call on a device, with that device
 * current, looks up the array's device address (no allocation); make that
 * first call before any stream capture.  All calls on a device share the one
 * array and keep the last call's contents: calls that overlap on the GPU race,
 * so order them on one stream.  Host threads calling at once are serialised
 * around the library's per-device bookkeeping, but their GPU work still
 * races: order them.  Layouts are checked as for motion_submit_batch
 * (pitch <= 2^40, frame stride <= 2^46, n frames within 2^48 bytes).  A
 * bounded wait that runs out sets this device's error word, which only
 * motion_noalloc_device_error reads. */
MOTION_API int motion_submit_batch_noalloc(const void* d_frames, int n, int w, int h, int bpc,
                                           size_t frame_stride_bytes, size_t pitch_bytes,
                                           int continue_sequence, void* stream,
                                           uint64_t* d_sad_out);

/* The collect step of motion_submit_batch_noalloc (not part of the method):
 * waits for `stream`, then reads and clears the current device's error word
 * of the allocation-free calls (bits as motion_device_error).  A set word
 * means the SADs written since the previous read are incomplete and so may be
 * the built-in plane: the next call with continue_sequence = 1 is refused
 * (MOTION_ERR_INVALID_ARGUMENT) until one starts a sequence.  Allocates
 * nothing.  *flags receives the word. */
MOTION_API int motion_noalloc_device_error(void* stream, int* flags);

/* Test hook for the allocation-free calls' bounded waits (not part of the
 * method), process-wide: while on, their TMA launches expect 16 bytes per stage
 * more than their boxes deliver and bound every wait at about 2 ms, so the
 * kernels set bit 0 of the error word and leave. */
MOTION_API int motion_noalloc_set_stall_injection(int on);

/* Number of this library's kernels launched by the calls above since load. */
MOTION_API uint64_t motion_kernel_launch_count(void);

/* Human-readable name of a status code (static string). */
MOTION_API const char* motion_strerror(int code);

/* The last CUDA error seen by a MOTION_ERR_CUDA return (cudaError_t value). */
MOTION_API int motion_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOTION_GB300_H */
