/*
 * oracle.c -- plain, slow, single-threaded CPU definition of the integer motion
 * feature and the per-plane PSNR squared-error sum.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file: only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library; the two agree only because both follow the same definition.
 *
 * Sources (cited by page title and section):
 *   [ADR-1392] "ADR-1392: CUDA motion, PSNR and moment kernels add one atomic per
 *              block, the motion SAD filters separably, and PSNR selects its plane
 *              with constant indices".
 *              Context: every sum is one integer per pixel accumulated into a
 *              single 64-bit value that must equal the CPU's bit for bit.
 *              Decision 4: the blur is separable -- a vertical 5-tap pass with the
 *              CPU's rounding (>> bpc) first, then the 5 horizontal taps (>> 16);
 *              the integers equal those of the per-output loop.
 *   The filter constants are this library's definition of the integer motion
 *   blur: taps {3571, 16004, 26386, 16004, 3571} (sum 65536), mirror boundaries
 *   i < 0 -> -i, i >= n -> 2n - i - 2, rounding by adding half before each shift,
 *   score = SAD / 256 / (w*h), motion2 = min(score(prev,cur), score(cur,next)).
 *
 * Readings of points the pages leave open (each is listed in the design notes):
 *   - Reading A: each frame is blurred, then |B_cur - B_prev| is summed (not the
 *     blur of the signed difference).
 *   - The first frame of a sequence has SAD 0 and score 0.
 *   - motion2 of the last frame is its own score (no next frame).
 *   - w and h must be >= 3 (the mirror rule leaves [0, n) for n < 3).
 *   - bpc in [8, 16]; samples are uint8 for bpc == 8, little-endian uint16
 *     otherwise; sample values >= 2^bpc are a precondition violation.
 *
 * Arithmetic: every sum is exact in uint32 for sample values < 2^16
 * (65535 * 65536 + 2^15 < 2^32); SAD and SSE accumulate in uint64.
 *
 * Two further quantities of the same page:
 *   - Moment sums [ADR-1392, Decision 6 and Context]: for a picture pair, the
 *     sums of the reference and distorted luma samples and of their squares,
 *     four exact uint64 accumulators; the moments are those sums over the
 *     sample count (mean and mean square), in double.
 *   - motion_v2 [ADR-1392, Decision 4]: the separable blur applied to the
 *     signed difference prev - cur of two consecutive frames, with the same
 *     taps, mirror and rounding constants; a right shift of a negative sum
 *     rounds towards minus infinity (floor), and the SAD is the sum of the
 *     absolute blurred values.  Sums need 33 bits with sign, so the
 *     arithmetic is int64 here.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_API
#define ORACLE_API __attribute__((visibility("default")))
#endif

/* The 5 taps of the integer Gaussian, k = 0..4 for offsets -2..+2. */
static const uint32_t oracle_taps[5] = {3571u, 16004u, 26386u, 16004u, 3571u};

/* Mirror boundary: reflect about the edge sample, the edge itself not repeated. */
ORACLE_API int oracle_mirror(int i, int n)
{
#if defined(ORACLE_PLANT_MIRROR_REPEAT)
    /* planted mistake (tests only): edge-repeating reflection */
    if (i < 0) return -i - 1;
    if (i >= n) return 2 * n - i - 1;
    return i;
#else
    if (i < 0) return -i;
    if (i >= n) return 2 * n - i - 2;
    return i;
#endif
}

static uint32_t sample_at(const unsigned char* base, size_t pitch, int bpc,
                          int y, int x)
{
    const unsigned char* row = base + (size_t)y * pitch;
    if (bpc == 8) return row[x];
    /* little-endian uint16 sample, assembled byte by byte */
    return (uint32_t)row[2 * (size_t)x] | ((uint32_t)row[2 * (size_t)x + 1] << 8);
}

static int args_ok(int w, int h, int bpc)
{
    return w >= 3 && h >= 3 && bpc >= 8 && bpc <= 16;
}

/*
 * Blur one frame.  out receives B as h rows of w uint16 values (row-major,
 * pitch w).  Returns 0, or -1 on a bad argument or allocation failure.
 *
 *   V[y][x] = (sum_k t_k * F[mirror(y+k-2, h)][x] + 2^(bpc-1)) >> bpc
 *   B[y][x] = (sum_k t_k * V[y][mirror(x+k-2, w)] + 2^15) >> 16
 * [ADR-1392, Decision 4]: vertical pass first, rounded >> bpc; then horizontal,
 * rounded >> 16.
 */
ORACLE_API int oracle_blur(const void* frame, int w, int h, size_t pitch_bytes,
                           int bpc, uint16_t* out)
{
    if (!frame || !out || !args_ok(w, h, bpc)) return -1;
    const unsigned char* src = (const unsigned char*)frame;
    uint32_t* V = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)w * (size_t)h);
    if (!V) return -1;

    const uint32_t vround = 1u << (bpc - 1);
    for (int y = 0; y < h; ++y) {
        for (int x = 0; x < w; ++x) {
            uint32_t s = 0;
            for (int k = 0; k < 5; ++k) {
#if defined(ORACLE_PLANT_HFIRST)
                int xx = oracle_mirror(x + k - 2, w);         /* planted: passes swapped */
                s += oracle_taps[k] * sample_at(src, pitch_bytes, bpc, y, xx);
#else
                int yy = oracle_mirror(y + k - 2, h);
                s += oracle_taps[k] * sample_at(src, pitch_bytes, bpc, yy, x);
#endif
            }
#if defined(ORACLE_PLANT_NO_VROUND)
            V[(size_t)y * w + x] = s >> bpc;              /* planted: rounding dropped */
#elif defined(ORACLE_PLANT_VSHIFT8)
            V[(size_t)y * w + x] = (s + 128u) >> 8;        /* planted: 8-bit shift at any depth */
#else
            V[(size_t)y * w + x] = (s + vround) >> bpc;
#endif
        }
    }
    for (int y = 0; y < h; ++y) {
        for (int x = 0; x < w; ++x) {
            uint32_t s = 0;
            for (int k = 0; k < 5; ++k) {
#if defined(ORACLE_PLANT_SWAP_MIRROR_N)
                int xx = oracle_mirror(x + k - 2, h);       /* planted: wrong extent */
                if (xx >= w) xx = w - 1;
                s += oracle_taps[k] * V[(size_t)y * w + xx];
#elif defined(ORACLE_PLANT_HFIRST)
                int yy = oracle_mirror(y + k - 2, h);
                s += oracle_taps[k] * V[(size_t)yy * w + x];
#else
                int xx = oracle_mirror(x + k - 2, w);
                s += oracle_taps[k] * V[(size_t)y * w + xx];
#endif
            }
#if defined(ORACLE_PLANT_NO_HROUND)
            out[(size_t)y * w + x] = (uint16_t)(s >> 16);
#else
            out[(size_t)y * w + x] = (uint16_t)((s + 32768u) >> 16);
#endif
        }
    }
    free(V);
    return 0;
}

/* SAD of two blurred planes of n samples each: sum |a_i - b_i| in uint64. */
ORACLE_API uint64_t oracle_sad(const uint16_t* a, const uint16_t* b, size_t n)
{
    uint64_t acc = 0;
    for (size_t i = 0; i < n; ++i) {
        int d = (int)a[i] - (int)b[i];
        acc += (uint64_t)(d < 0 ? -d : d);
    }
    return acc;
}

/*
 * Motion SAD over a sequence of n frames stored frame_stride bytes apart.
 * sad_out[0] = 0 (no previous frame); sad_out[i] = SAD(B_i, B_{i-1}).
 * Each frame is blurred once and compared with the previous frame's blur.
 */
ORACLE_API int oracle_motion_sad_sequence(const void* frames, int n,
                                          size_t frame_stride, int w, int h,
                                          size_t pitch_bytes, int bpc,
                                          uint64_t* sad_out)
{
    if (n < 0 || (n > 0 && (!frames || !sad_out)) || !args_ok(w, h, bpc)) return -1;
    if (n == 0) return 0;
    size_t npx = (size_t)w * (size_t)h;
    uint16_t* prev = (uint16_t*)malloc(sizeof(uint16_t) * npx);
    uint16_t* cur = (uint16_t*)malloc(sizeof(uint16_t) * npx);
    if (!prev || !cur) { free(prev); free(cur); return -1; }
    const unsigned char* base = (const unsigned char*)frames;
    int rc = 0;
    for (int i = 0; i < n && rc == 0; ++i) {
        rc = oracle_blur(base + (size_t)i * frame_stride, w, h, pitch_bytes, bpc, cur);
        if (rc) break;
        sad_out[i] = (i == 0) ? 0 : oracle_sad(cur, prev, npx);
        uint16_t* t = prev; prev = cur; cur = t;
    }
    free(prev);
    free(cur);
    return rc;
}

/*
 * Per-plane squared-error sum, SSE = sum (ref - dist)^2 in uint64.
 * [ADR-1392, Context]: one integer per pixel summed into a 64-bit value.
 */
ORACLE_API uint64_t oracle_sse(const void* ref, const void* dist, int w, int h,
                               size_t ref_pitch, size_t dist_pitch, int bpc)
{
    if (!ref || !dist || w <= 0 || h <= 0 || bpc < 8 || bpc > 16) return 0;
    const unsigned char* r = (const unsigned char*)ref;
    const unsigned char* d = (const unsigned char*)dist;
    uint64_t acc = 0;
    for (int y = 0; y < h; ++y) {
        for (int x = 0; x < w; ++x) {
            int64_t e = (int64_t)sample_at(r, ref_pitch, bpc, y, x)
                      - (int64_t)sample_at(d, dist_pitch, bpc, y, x);
            acc += (uint64_t)(e * e);
        }
    }
    return acc;
}

/*
 * Scores from SADs, in double:
 *   score_i   = ((double)SAD_i / 256.0) / (double)(w*h)
 *   motion2_i = min(score_i, score_{i+1}); motion2_{n-1} = score_{n-1}.
 * next_score, when not NULL, is the score of the frame after the last one (a
 * sequence continued elsewhere); it then takes part in motion2_{n-1}.
 */
ORACLE_API int oracle_scores(const uint64_t* sad, int n, int w, int h,
                             const double* next_score, double* score,
                             double* motion2)
{
    if (n < 0 || (n > 0 && (!sad || !score || !motion2)) || w <= 0 || h <= 0) return -1;
    const double area = (double)w * (double)h;
    for (int i = 0; i < n; ++i)
        score[i] = ((double)sad[i] / 256.0) / area;
    for (int i = 0; i < n; ++i) {
        double nxt;
        int has_next = 1;
        if (i + 1 < n) nxt = score[i + 1];
        else if (next_score) nxt = *next_score;
        else { nxt = 0.0; has_next = 0; }
        motion2[i] = has_next ? (score[i] < nxt ? score[i] : nxt) : score[i];
    }
    return 0;
}

/*
 * Moment sums of one picture pair [ADR-1392, Decision 6: four accumulators,
 * the reference and distorted sums and sums of squares; Context: exact 64-bit
 * integer sums].  out[0] = sum ref, out[1] = sum dist, out[2] = sum ref^2,
 * out[3] = sum dist^2.  Returns 0, or -1 on a bad argument.
 */
ORACLE_API int oracle_moment_sums(const void* ref, const void* dist, int w, int h,
                                  size_t ref_pitch, size_t dist_pitch, int bpc,
                                  uint64_t* out)
{
    if (!ref || !dist || !out || w <= 0 || h <= 0 || bpc < 8 || bpc > 16) return -1;
    const unsigned char* r = (const unsigned char*)ref;
    const unsigned char* d = (const unsigned char*)dist;
    uint64_t s_r = 0, s_d = 0, q_r = 0, q_d = 0;
#if defined(ORACLE_PLANT_MOMENT_SKIP_LAST_ROW)
    h -= 1;   /* planted mistake (tests only): the last row is left out */
#endif
    for (int y = 0; y < h; ++y) {
        for (int x = 0; x < w; ++x) {
            const uint64_t a = sample_at(r, ref_pitch, bpc, y, x);
            const uint64_t b = sample_at(d, dist_pitch, bpc, y, x);
            s_r += a;
            s_d += b;
            q_r += a * a;
#if defined(ORACLE_PLANT_MOMENT_SQUARE_OF_REF)
            q_d += a * a;   /* planted mistake (tests only): ref squared twice */
#else
            q_d += b * b;
#endif
        }
    }
    out[0] = s_r;
    out[1] = s_d;
    out[2] = q_r;
    out[3] = q_d;
    return 0;
}

/*
 * Moments from moment sums, in double: each sum over the sample count w*h
 * (the first moments are the means, the second the mean squares).
 */
ORACLE_API int oracle_moments(const uint64_t* sums, int n, int w, int h, double* out)
{
    if (n < 0 || (n > 0 && (!sums || !out)) || w <= 0 || h <= 0) return -1;
    const double count = (double)w * (double)h;
    for (int i = 0; i < 4 * n; ++i) out[i] = (double)sums[i] / count;
    return 0;
}

/* Floor of a / 2^k for a signed a (an arithmetic right shift). */
static int64_t floor_shift(int64_t a, int k)
{
#if defined(ORACLE_PLANT_V2_TRUNCATE)
    /* planted mistake (tests only): division that truncates towards zero */
    return a / ((int64_t)1 << k);
#else
    const int64_t q = a / ((int64_t)1 << k);
    return (q * ((int64_t)1 << k) > a) ? q - 1 : q;
#endif
}

/*
 * motion_v2 blur of the signed difference of two frames, as h rows of w int32
 * values [ADR-1392, Decision 4: stage prev - cur, vertical pass with the CPU's
 * rounding (>> bpc), then the 5 horizontal taps (>> 16)]:
 *   D[y][x]  = prev[y][x] - cur[y][x]
 *   V[y][x]  = floor((sum_k t_k * D[mirror(y+k-2, h)][x] + 2^(bpc-1)) / 2^bpc)
 *   Bd[y][x] = floor((sum_k t_k * V[y][mirror(x+k-2, w)] + 2^15) / 2^16)
 * Returns 0, or -1 on a bad argument or allocation failure.
 */
ORACLE_API int oracle_blur_diff(const void* prev, const void* cur, int w, int h,
                                size_t pitch_bytes, int bpc, int32_t* out)
{
    if (!prev || !cur || !out || !args_ok(w, h, bpc)) return -1;
    int64_t* v = (int64_t*)malloc(sizeof(int64_t) * (size_t)w * (size_t)h);
    if (!v) return -1;
    const unsigned char* p = (const unsigned char*)prev;
    const unsigned char* c = (const unsigned char*)cur;
    const int64_t vround = (int64_t)1 << (bpc - 1);
    for (int y = 0; y < h; ++y) {
        for (int x = 0; x < w; ++x) {
            int64_t acc = 0;
            for (int k = 0; k < 5; ++k) {
                const int yy = oracle_mirror(y + k - 2, h);
#if defined(ORACLE_PLANT_V2_CUR_MINUS_PREV)
                /* planted mistake (tests only): the difference taken the other way */
                const int64_t dd = (int64_t)sample_at(c, pitch_bytes, bpc, yy, x)
                                 - (int64_t)sample_at(p, pitch_bytes, bpc, yy, x);
#else
                const int64_t dd = (int64_t)sample_at(p, pitch_bytes, bpc, yy, x)
                                 - (int64_t)sample_at(c, pitch_bytes, bpc, yy, x);
#endif
                acc += (int64_t)oracle_taps[k] * dd;
            }
            v[(size_t)y * w + x] = floor_shift(acc + vround, bpc);
        }
    }
    for (int y = 0; y < h; ++y) {
        for (int x = 0; x < w; ++x) {
            int64_t acc = 0;
            for (int k = 0; k < 5; ++k) {
                const int xx = oracle_mirror(x + k - 2, w);
                acc += (int64_t)oracle_taps[k] * v[(size_t)y * w + xx];
            }
            out[(size_t)y * w + x] = (int32_t)floor_shift(acc + 32768, 16);
        }
    }
    free(v);
    return 0;
}

/*
 * motion_v2 SADs over a sequence of n frames stored frame_stride bytes apart:
 * sad_out[0] = 0 (no previous frame); sad_out[i] = sum |Bd(F_{i-1}, F_i)|.
 */
ORACLE_API int oracle_motion_v2_sequence(const void* frames, int n, size_t frame_stride,
                                         int w, int h, size_t pitch_bytes, int bpc,
                                         uint64_t* sad_out)
{
    if (n < 0 || (n > 0 && (!frames || !sad_out)) || !args_ok(w, h, bpc)) return -1;
    if (n == 0) return 0;
    const size_t npx = (size_t)w * (size_t)h;
    int32_t* b = (int32_t*)malloc(sizeof(int32_t) * npx);
    if (!b) return -1;
    const unsigned char* base = (const unsigned char*)frames;
    sad_out[0] = 0;
    int rc = 0;
    for (int i = 1; i < n && rc == 0; ++i) {
        rc = oracle_blur_diff(base + (size_t)(i - 1) * frame_stride, base + (size_t)i * frame_stride,
                              w, h, pitch_bytes, bpc, b);
        if (rc) break;
        uint64_t acc = 0;
        for (size_t j = 0; j < npx; ++j) acc += (uint64_t)(b[j] < 0 ? -(int64_t)b[j] : (int64_t)b[j]);
        sad_out[i] = acc;
    }
    free(b);
    return rc;
}
