// motion_capi.cu -- the C ABI of libmotion_gb300: argument validation, the
// motion context (resident previous blurred plane, result slot, host staging),
// launch planning, and the host-buffer pipeline.  See include/motion.h for
// the contract of every entry point.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "motion.h"
#include "motion_internal.h"

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_last_cuda_error{0};
// test hook (motion_inject_alloc_failure): the k-th allocation from now fails
// without reaching the driver; 0 = off
std::atomic<int> g_fail_alloc_in{0};

bool injected_alloc_failure() {
    int k = g_fail_alloc_in.load();
    while (k > 0) {
        if (g_fail_alloc_in.compare_exchange_weak(k, k - 1)) return k == 1;
    }
    return false;
}

// Every device and pinned allocation of the library goes through these two.
cudaError_t dev_alloc(void** p, size_t bytes) {
    if (injected_alloc_failure()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}
cudaError_t host_alloc(void** p, size_t bytes) {
    if (injected_alloc_failure()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaHostAlloc(p, bytes, cudaHostAllocDefault);
}

int cuda_fail(cudaError_t e) {
    g_last_cuda_error.store((int)e);
    return e == cudaErrorMemoryAllocation ? MOTION_ERR_OUT_OF_MEMORY : MOTION_ERR_CUDA;
}
#define MG_CUDA(call)                               \
    do {                                            \
        cudaError_t e_ = (call);                    \
        if (e_ != cudaSuccess) return cuda_fail(e_); \
    } while (0)

using mg::check_dims;
using mg::check_layout;
using mg::sample_bytes;

bool aligned16(const void* p, size_t pitch, size_t stride, int n) {
    return (((uintptr_t)p | pitch) % 16 == 0) && (n <= 1 || stride % 16 == 0);
}

int current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    return MOTION_OK;
}

}  // namespace

namespace mg {
void note_launches(int n) { g_launches += (uint64_t)n; }

int sample_bytes(int bpc) { return bpc == 8 ? 1 : 2; }

int check_dims(int w, int h, int bpc) {
    if (bpc < 8 || bpc > 16) return MOTION_ERR_UNSUPPORTED_BITDEPTH;
    if (w < 3 || h < 3) return MOTION_ERR_FRAME_TOO_SMALL;
    if (w > MOTION_MAX_DIM || h > MOTION_MAX_DIM) return MOTION_ERR_TOO_LARGE;
    return MOTION_OK;
}

// A plane layout: rows of w samples, pitch bytes apart; n planes stride apart.
int check_layout(const void* p, size_t pitch, size_t stride, int n, int w, int bpc) {
    if (!p) return MOTION_ERR_INVALID_ARGUMENT;
    const size_t s = (size_t)sample_bytes(bpc);
    if (pitch < (size_t)w * s) return MOTION_ERR_BAD_PITCH;
    if (s == 2 && (((uintptr_t)p & 1) || (pitch & 1) || (n > 1 && (stride & 1))))
        return MOTION_ERR_BAD_PITCH;
    if (pitch > (size_t)1 << 40 || stride > (size_t)1 << 46) return MOTION_ERR_INVALID_ARGUMENT;
    // n frames stride apart must fit a 48-bit address space (no frame offset wraps)
    if (n > 1 && stride > ((size_t)1 << 48) / (size_t)n) return MOTION_ERR_INVALID_ARGUMENT;
    return MOTION_OK;
}
}  // namespace mg

struct motion_ctx {
    int device = -1;
    int w = 0, h = 0, bpc = 8, cw = 0, ch = 0;
    int sm_count = 0;
    int bprev_pitch = 0;            // elements per row of the resident plane
    uint16_t* d_bprev[2] = {nullptr, nullptr};  // previous frame's blurred plane, ping-pong
    int cur = 0;                    // index of the plane that holds B_{i-1}
    int has_prev = 0;
    // device error word (bit 0: a bounded wait ran out; bit 1: a failed check in
    // the bounds-checked build): the low half of d_slot[1], so that one 16-byte
    // copy reads a frame's SAD and the word together
    int* d_err = nullptr;
    int force_generic = 0;          // diagnostics: always use the generic kernel
    int force_rows = 0;             // diagnostics: TMA tile height of motion-only launches (0: chosen)
    int stall_injection = 0;        // test hook: stage waits that can never complete
    unsigned long long* d_slot = nullptr;   // [0]: single-submit SAD, [1]: error word
    unsigned long long* h_slot = nullptr;   // pinned readback of d_slot (16 bytes)
    // host-buffer pipeline
    int stage_pairs = 0;
    size_t stage_stride_y = 0, stage_stride_uv = 0;
    size_t stage_set_bytes = 0, stage_res_n = 0;   // bytes of each staging set, results per set
    uint8_t* d_stage[2] = {nullptr, nullptr};
    unsigned long long* d_res[2] = {nullptr, nullptr};
    cudaStream_t s_copy = nullptr, s_comp = nullptr;
    cudaEvent_t ev_in[2] = {nullptr, nullptr}, ev_done[2] = {nullptr, nullptr};
    // pinned result staging of a host-buffer call (SAD + 3 SSE per pair), so
    // that its device-to-host copies stay asynchronous and the next chunk's
    // uploads are queued without waiting for this chunk's kernel
    unsigned long long* h_res = nullptr;
    size_t h_res_pairs = 0;
    // motion_v2: the last raw frame of the sequence, two planes that alternate
    // (allocated by the first motion_v2 call), rows raw_pitch bytes apart
    uint8_t* d_raw[2] = {nullptr, nullptr};
    size_t raw_pitch = 0;
    int raw_cur = 0;
    int v2_has_prev = 0;
    // planes a call passes with rows the TMA cannot address are first copied
    // here with 16-byte-aligned rows (allocated by the first such call, grown
    // when a call needs more)
    uint8_t* d_rp = nullptr;
    size_t rp_bytes = 0;
    size_t rp_limit = 0;            // most bytes of one copy (0: 1 GiB); longer calls go in parts
};

namespace {

int ctx_device_ok(const motion_ctx* c) {
    int dev = -1;
    int rc = current_device(&dev);
    if (rc) return rc;
    return dev == c->device ? MOTION_OK : MOTION_ERR_WRONG_DEVICE;
}

void free_staging(motion_ctx* c) {
    for (int k = 0; k < 2; ++k) {
        if (c->d_stage[k]) cudaFree(c->d_stage[k]);
        if (c->d_res[k]) cudaFree(c->d_res[k]);
        if (c->ev_in[k]) cudaEventDestroy(c->ev_in[k]);
        if (c->ev_done[k]) cudaEventDestroy(c->ev_done[k]);
        c->d_stage[k] = nullptr;
        c->d_res[k] = nullptr;
        c->ev_in[k] = c->ev_done[k] = nullptr;
    }
    if (c->s_copy) cudaStreamDestroy(c->s_copy);
    if (c->s_comp) cudaStreamDestroy(c->s_comp);
    c->s_copy = c->s_comp = nullptr;
    c->stage_pairs = 0;
    c->stage_set_bytes = c->stage_res_n = 0;
    if (c->h_res) cudaFreeHost(c->h_res);
    c->h_res = nullptr;
    c->h_res_pairs = 0;
}

// The two staging sets of the host-buffer calls: at least set_bytes each and
// res_n uint64 results each (grown, never shrunk), their events and streams.
int reserve_stage(motion_ctx* c, size_t set_bytes, size_t res_n) {
    if (c->d_stage[0] && c->stage_set_bytes >= set_bytes && c->stage_res_n >= res_n) return MOTION_OK;
    if (set_bytes < c->stage_set_bytes) set_bytes = c->stage_set_bytes;
    if (res_n < c->stage_res_n) res_n = c->stage_res_n;
    free_staging(c);
    for (int k = 0; k < 2; ++k) {
        MG_CUDA(dev_alloc(reinterpret_cast<void**>(&c->d_stage[k]), set_bytes));
        MG_CUDA(dev_alloc(reinterpret_cast<void**>(&c->d_res[k]), sizeof(unsigned long long) * res_n));
        MG_CUDA(cudaEventCreateWithFlags(&c->ev_in[k], cudaEventDisableTiming));
        MG_CUDA(cudaEventCreateWithFlags(&c->ev_done[k], cudaEventDisableTiming));
    }
    MG_CUDA(cudaStreamCreateWithFlags(&c->s_copy, cudaStreamNonBlocking));
    MG_CUDA(cudaStreamCreateWithFlags(&c->s_comp, cudaStreamNonBlocking));
    c->stage_set_bytes = set_bytes;
    c->stage_res_n = res_n;
    return MOTION_OK;
}

// The pinned result buffer of the host-buffer calls: at least n uint64.
int reserve_host_results(motion_ctx* c, size_t n) {
    if (c->h_res_pairs * 4 >= n) return MOTION_OK;
    if (c->h_res) cudaFreeHost(c->h_res);
    c->h_res = nullptr;
    c->h_res_pairs = 0;
    const size_t pairs = (n + 3) / 4;
    MG_CUDA(host_alloc(reinterpret_cast<void**>(&c->h_res), sizeof(unsigned long long) * 4 * pairs));
    c->h_res_pairs = pairs;
    return MOTION_OK;
}

// Planes whose base, pitch or frame stride the TMA cannot take are copied
// into the context's scratch with 16-byte-aligned rows (one bandwidth-bound
// launch), and `a` is pointed at the copies, so the TMA kernel serves every
// layout; the generic kernel stays for motion_set_kernel_path(GENERIC).
int repitch_for_tma(motion_ctx* c, mg::TileArgs& a, bool fused, cudaStream_t s) {
    if (c->force_generic || a.n <= 0 || mg::tma_usable(a, fused)) return MOTION_OK;
    const long long S = sample_bytes(c->bpc);
    const long long py = ((long long)c->w * S + 15) & ~15LL, sy = py * c->h;
    const long long puv = ((long long)c->cw * S + 15) & ~15LL, suv = puv * c->ch;
    const size_t need = (size_t)a.n * (size_t)(fused ? 2 * sy + 4 * suv : sy);
    if (c->rp_bytes < need) {
        if (c->d_rp) cudaFree(c->d_rp);
        c->d_rp = nullptr;
        c->rp_bytes = 0;
        MG_CUDA(dev_alloc(reinterpret_cast<void**>(&c->d_rp), need));
        c->rp_bytes = need;
    }
    mg::RepitchArgs r;
    std::memset(&r, 0, sizeof(r));
    r.n = a.n;
    r.err = c->d_err;
    const uint8_t* src[6] = {a.ref_y, a.dist_y, a.ref_u, a.dist_u, a.ref_v, a.dist_v};
    uint8_t* base = c->d_rp;
    r.planes = fused ? 6 : 1;
    for (int p = 0; p < r.planes; ++p) {
        const bool luma = p < 2;
        mg::RepitchPlane& q = r.p[p];
        q.src = src[p];
        q.pitch = luma ? a.pitch_y : a.pitch_uv;
        q.stride = luma ? a.stride_y : a.stride_uv;
        q.dst = base;
        q.dpitch = luma ? py : puv;
        q.dstride = luma ? sy : suv;
        q.row_bytes = (int)((luma ? c->w : c->cw) * S);
        q.rows = luma ? c->h : c->ch;
        base += (size_t)a.n * (size_t)q.dstride;
    }
    int launched = 0;
    const cudaError_t e = mg::launch_repitch(r, s, c->sm_count, &launched);
    g_launches += (uint64_t)launched;
    if (e != cudaSuccess) return cuda_fail(e);
    a.ref_y = r.p[0].dst;
    a.pitch_y = py;
    a.stride_y = sy;
    if (fused) {
        a.dist_y = r.p[1].dst;
        a.ref_u = r.p[2].dst;
        a.dist_u = r.p[3].dst;
        a.ref_v = r.p[4].dst;
        a.dist_v = r.p[5].dst;
        a.pitch_uv = puv;
        a.stride_uv = suv;
    }
    a.aligned16 = 1;
    return MOTION_OK;
}

// The TMA kernel (after repitch_for_tma, for any layout), or the generic
// kernel when motion_set_kernel_path asks for it.
// Frames (or pairs) of one launch whose planes the copy kernel re-pitches:
// as many as fit the context's copy limit, at least one; all of them when the
// planes need no copy.
int frames_per_copy(const motion_ctx* c, const mg::TileArgs& a, bool fused) {
    if (c->force_generic || a.n <= 1 || mg::tma_usable(a, fused)) return a.n;
    const long long S = sample_bytes(c->bpc);
    const long long py = ((long long)c->w * S + 15) & ~15LL, puv = ((long long)c->cw * S + 15) & ~15LL;
    const size_t per = (size_t)(fused ? 2 * py * c->h + 4 * puv * c->ch : py * c->h);
    const size_t limit = c->rp_limit ? c->rp_limit : ((size_t)1 << 30);
    const size_t m = limit / per;
    return m < 1 ? 1 : (m >= (size_t)a.n ? a.n : (int)m);
}

// The planes of frames [f0, f0 + m) of a launch.
mg::TileArgs frames_slice(const mg::TileArgs& a, int f0, int m) {
    mg::TileArgs b = a;
    b.n = m;
    b.ref_y = a.ref_y + (long long)f0 * a.stride_y;
    if (a.dist_y) b.dist_y = a.dist_y + (long long)f0 * a.stride_y;
    if (a.ref_u) b.ref_u = a.ref_u + (long long)f0 * a.stride_uv;
    if (a.dist_u) b.dist_u = a.dist_u + (long long)f0 * a.stride_uv;
    if (a.ref_v) b.ref_v = a.ref_v + (long long)f0 * a.stride_uv;
    if (a.dist_v) b.dist_v = a.dist_v + (long long)f0 * a.stride_uv;
    if (a.sad_out) b.sad_out = a.sad_out + f0;
    if (a.sse_out) b.sse_out = a.sse_out + 3LL * f0;
    return b;
}

int launch_motion_one(motion_ctx* c, mg::TileArgs a, bool fused, cudaStream_t s);

// A launch, in parts when its planes need the copy kernel and do not fit the
// copy limit (each part continues the sequence of the one before).
int launch_motion(motion_ctx* c, mg::TileArgs a, bool fused, cudaStream_t s) {
    const int m = frames_per_copy(c, a, fused);
    if (m >= a.n) return launch_motion_one(c, a, fused, s);
    for (int f0 = 0; f0 < a.n; f0 += m) {
        mg::TileArgs b = frames_slice(a, f0, (a.n - f0) < m ? (a.n - f0) : m);
        b.has_prev = c->has_prev;
        b.bprev = c->d_bprev[c->cur];
        b.bprev_out = c->d_bprev[c->cur ^ 1];
        const int rc = launch_motion_one(c, b, fused, s);
        if (rc) return rc;
    }
    return MOTION_OK;
}

int launch_motion_one(motion_ctx* c, mg::TileArgs a, bool fused, cudaStream_t s) {
    int rc = repitch_for_tma(c, a, fused, s);
    if (rc) return rc;
    int launched = 0;
    bool used = false;
    cudaError_t e = cudaSuccess;
    if (!c->force_generic) e = mg::launch_motion_tma(a, fused, s, &launched, &used);
    if (e == cudaSuccess && !used) e = mg::launch_motion_tile(a, fused, s, &launched);
    g_launches += (uint64_t)launched;
    if (e != cudaSuccess) return cuda_fail(e);
    c->has_prev = 1;
    c->cur ^= 1;   // the plane just written holds B of the last frame
    return MOTION_OK;
}

mg::TileArgs motion_args(motion_ctx* c, int n) {
    mg::TileArgs a;
    std::memset(&a, 0, sizeof(a));
    a.w = c->w;
    a.h = c->h;
    a.cw = c->cw;
    a.ch = c->ch;
    a.bpc = c->bpc;
    a.n = n;
    a.has_prev = c->has_prev;
    a.store_last = 1;
    a.bprev = c->d_bprev[c->cur];
    a.bprev_out = c->d_bprev[c->cur ^ 1];
    a.bprev_pitch = c->bprev_pitch;
    a.err = c->d_err;
    a.force_rows = c->force_rows;
    if (c->stall_injection) {
        a.tx_extra = 16;               // the stage expects 16 bytes that never arrive
        a.wait_cycles = 1LL << 22;     // and gives up after about 2 ms
    }
    return a;
}

int validate_yuv(const motion_ctx* c, int n, const void* ry, const void* ru, const void* rv,
                 const void* dy, const void* du, const void* dv, size_t pitch_y,
                 size_t pitch_uv, size_t stride_y, size_t stride_uv) {
    int rc;
    if ((rc = check_layout(ry, pitch_y, stride_y, n, c->w, c->bpc))) return rc;
    if ((rc = check_layout(dy, pitch_y, stride_y, n, c->w, c->bpc))) return rc;
    if ((rc = check_layout(ru, pitch_uv, stride_uv, n, c->cw, c->bpc))) return rc;
    if ((rc = check_layout(rv, pitch_uv, stride_uv, n, c->cw, c->bpc))) return rc;
    if ((rc = check_layout(du, pitch_uv, stride_uv, n, c->cw, c->bpc))) return rc;
    if ((rc = check_layout(dv, pitch_uv, stride_uv, n, c->cw, c->bpc))) return rc;
    return MOTION_OK;
}

int launch_fused(motion_ctx* c, int n, const void* ry, const void* ru, const void* rv,
                 const void* dy, const void* du, const void* dv, size_t pitch_y,
                 size_t pitch_uv, size_t stride_y, size_t stride_uv, cudaStream_t s,
                 uint64_t* d_sad, uint64_t* d_sse) {
    MG_CUDA(cudaMemsetAsync(d_sad, 0, sizeof(uint64_t) * (size_t)n, s));
    MG_CUDA(cudaMemsetAsync(d_sse, 0, sizeof(uint64_t) * 3 * (size_t)n, s));
    mg::TileArgs a = motion_args(c, n);
    a.ref_y = (const uint8_t*)ry;
    a.ref_u = (const uint8_t*)ru;
    a.ref_v = (const uint8_t*)rv;
    a.dist_y = (const uint8_t*)dy;
    a.dist_u = (const uint8_t*)du;
    a.dist_v = (const uint8_t*)dv;
    a.pitch_y = (long long)pitch_y;
    a.pitch_uv = (long long)pitch_uv;
    a.stride_y = (long long)stride_y;
    a.stride_uv = (long long)stride_uv;
    a.aligned16 = aligned16(ry, pitch_y, stride_y, n) && aligned16(dy, pitch_y, stride_y, n) &&
                  aligned16(ru, pitch_uv, stride_uv, n) && aligned16(rv, pitch_uv, stride_uv, n) &&
                  aligned16(du, pitch_uv, stride_uv, n) && aligned16(dv, pitch_uv, stride_uv, n);
    a.sad_out = (unsigned long long*)d_sad;
    a.sse_out = (unsigned long long*)d_sse;
    return launch_motion(c, a, true, s);
}

// A kernel of this context set the device error word: clear it on `s`, start
// the sequences afresh (the resident planes may be incomplete) and report it.
int device_failed(motion_ctx* c, cudaStream_t s) {
    MG_CUDA(cudaMemsetAsync(c->d_err, 0, sizeof(int), s));
    MG_CUDA(cudaStreamSynchronize(s));
    c->has_prev = 0;
    c->v2_has_prev = 0;
    return MOTION_ERR_DEVICE;
}

// Queue the read of the error word into h_slot[1] on `s` (the host-buffer
// calls check it after their final synchronisation).
int queue_error_read(motion_ctx* c, cudaStream_t s) {
    c->h_slot[1] = 0;
    MG_CUDA(cudaMemcpyAsync(&c->h_slot[1], c->d_err, sizeof(int), cudaMemcpyDeviceToHost, s));
    return MOTION_OK;
}

}  // namespace

extern "C" {

int motion_init(int w, int h, int bpc, motion_ctx** out) {
    if (!out) return MOTION_ERR_INVALID_ARGUMENT;
    *out = nullptr;
    int rc = check_dims(w, h, bpc);
    if (rc) return rc;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        cudaGetLastError();
        return MOTION_ERR_NO_DEVICE;
    }
    motion_ctx* c = new (std::nothrow) motion_ctx();
    if (!c) return MOTION_ERR_OUT_OF_MEMORY;
    c->w = w;
    c->h = h;
    c->bpc = bpc;
    c->cw = (w + 1) / 2;
    c->ch = (h + 1) / 2;
    c->bprev_pitch = (w + 7) & ~7;
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);
    if (e == cudaSuccess)
        e = dev_alloc(reinterpret_cast<void**>(&c->d_bprev[0]), sizeof(uint16_t) * (size_t)c->bprev_pitch * (size_t)h);
    if (e == cudaSuccess)
        e = dev_alloc(reinterpret_cast<void**>(&c->d_bprev[1]), sizeof(uint16_t) * (size_t)c->bprev_pitch * (size_t)h);
    if (e == cudaSuccess) e = dev_alloc(reinterpret_cast<void**>(&c->d_slot), 2 * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(c->d_slot, 0, 2 * sizeof(unsigned long long));
    if (e == cudaSuccess) c->d_err = reinterpret_cast<int*>(c->d_slot + 1);
    if (e == cudaSuccess) e = host_alloc(reinterpret_cast<void**>(&c->h_slot), 2 * sizeof(unsigned long long));
    if (e != cudaSuccess) {
        motion_destroy(c);
        return cuda_fail(e);
    }
    *out = c;
    return MOTION_OK;
}

int motion_destroy(motion_ctx* c) {
    if (!c) return MOTION_OK;
    int prev = -1;
    cudaGetDevice(&prev);
    if (c->device >= 0) cudaSetDevice(c->device);
    free_staging(c);
    if (c->d_bprev[0]) cudaFree(c->d_bprev[0]);
    if (c->d_bprev[1]) cudaFree(c->d_bprev[1]);
    if (c->d_raw[0]) cudaFree(c->d_raw[0]);
    if (c->d_raw[1]) cudaFree(c->d_raw[1]);
    if (c->d_rp) cudaFree(c->d_rp);
    if (c->d_slot) cudaFree(c->d_slot);   // holds the error word too
    if (c->h_slot) cudaFreeHost(c->h_slot);
    if (prev >= 0) cudaSetDevice(prev);
    delete c;
    return MOTION_OK;
}

int motion_reset(motion_ctx* c) {
    if (!c) return MOTION_ERR_INVALID_ARGUMENT;
    c->has_prev = 0;
    c->v2_has_prev = 0;
    return MOTION_OK;
}

int motion_submit_batch(motion_ctx* c, const void* d_frames, int n, size_t frame_stride,
                        size_t pitch, void* stream, uint64_t* d_sad_out) {
    if (!c || n < 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (n == 0) return MOTION_OK;
    if (!d_sad_out) return MOTION_ERR_INVALID_ARGUMENT;
    int rc = check_layout(d_frames, pitch, frame_stride, n, c->w, c->bpc);
    if (rc) return rc;
    if ((rc = ctx_device_ok(c))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    MG_CUDA(cudaMemsetAsync(d_sad_out, 0, sizeof(uint64_t) * (size_t)n, s));
    mg::TileArgs a = motion_args(c, n);
    a.ref_y = (const uint8_t*)d_frames;
    a.pitch_y = (long long)pitch;
    a.stride_y = (long long)frame_stride;
    a.aligned16 = aligned16(d_frames, pitch, frame_stride, n);
    a.sad_out = (unsigned long long*)d_sad_out;
    return launch_motion(c, a, false, s);
}

int motion_v2_submit_batch(motion_ctx* c, const void* d_frames, int n, size_t frame_stride,
                           size_t pitch, void* stream, uint64_t* d_sad_out) {
    if (!c || n < 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (n == 0) return MOTION_OK;
    if (!d_sad_out) return MOTION_ERR_INVALID_ARGUMENT;
    int rc = check_layout(d_frames, pitch, frame_stride, n, c->w, c->bpc);
    if (rc) return rc;
    if ((rc = ctx_device_ok(c))) return rc;
    const size_t s_bytes = (size_t)sample_bytes(c->bpc);
    if (!c->d_raw[0] || !c->d_raw[1]) {
        // both planes or neither: a failed second allocation leaves no half state
        const size_t pitch_r = ((size_t)c->w * s_bytes + 15) & ~(size_t)15;
        uint8_t* p[2] = {nullptr, nullptr};
        cudaError_t e = dev_alloc(reinterpret_cast<void**>(&p[0]), pitch_r * (size_t)c->h);
        if (e == cudaSuccess) e = dev_alloc(reinterpret_cast<void**>(&p[1]), pitch_r * (size_t)c->h);
        if (e != cudaSuccess) {
            if (p[0]) cudaFree(p[0]);
            return cuda_fail(e);
        }
        if (c->d_raw[0]) cudaFree(c->d_raw[0]);
        if (c->d_raw[1]) cudaFree(c->d_raw[1]);
        c->d_raw[0] = p[0];
        c->d_raw[1] = p[1];
        c->raw_pitch = pitch_r;
        c->raw_cur = 0;
        c->v2_has_prev = 0;
    }
    cudaStream_t s = (cudaStream_t)stream;
    MG_CUDA(cudaMemsetAsync(d_sad_out, 0, sizeof(uint64_t) * (size_t)n, s));
    mg::TileArgs a = motion_args(c, n);
    a.ref_y = (const uint8_t*)d_frames;
    a.pitch_y = (long long)pitch;
    a.stride_y = (long long)frame_stride;
    a.aligned16 = aligned16(d_frames, pitch, frame_stride, n);
    a.sad_out = (unsigned long long*)d_sad_out;
    a.bprev = a.bprev_out = nullptr;
    a.raw_pitch = (long long)c->raw_pitch;
    const int m = frames_per_copy(c, a, false);
    for (int f0 = 0; f0 < n; f0 += m) {
        mg::TileArgs b = frames_slice(a, f0, (n - f0) < m ? (n - f0) : m);
        b.has_prev = c->v2_has_prev;
        b.raw_prev = c->d_raw[c->raw_cur];
        b.raw_out = c->d_raw[c->raw_cur ^ 1];
        if ((rc = repitch_for_tma(c, b, false, s))) return rc;
        int launched = 0;
        bool used = false;
        cudaError_t e = cudaSuccess;
        if (!c->force_generic) e = mg::launch_motion_v2_tma(b, s, &launched, &used);
        if (e == cudaSuccess && !used) e = mg::launch_motion_v2_tile(b, s, &launched);
        g_launches += (uint64_t)launched;
        if (e != cudaSuccess) return cuda_fail(e);
        c->v2_has_prev = 1;
        c->raw_cur ^= 1;   // the plane just written holds the last frame
    }
    return MOTION_OK;
}

int motion_submit(motion_ctx* c, const void* d_frame, size_t pitch, void* stream,
                  uint64_t* sad_out, double* score_out) {
    if (!c) return MOTION_ERR_INVALID_ARGUMENT;
    cudaStream_t s = (cudaStream_t)stream;
    int rc = motion_submit_batch(c, d_frame, 1, 0, pitch, stream, (uint64_t*)c->d_slot);
    if (rc) return rc;
    // one readback: the SAD and, beside it, the device error word
    MG_CUDA(cudaMemcpyAsync(c->h_slot, c->d_slot, 2 * sizeof(unsigned long long),
                            cudaMemcpyDeviceToHost, s));
    MG_CUDA(cudaStreamSynchronize(s));
    if ((int)(uint32_t)c->h_slot[1] != 0) return device_failed(c, s);
    const uint64_t sad = (uint64_t)c->h_slot[0];
    if (sad_out) *sad_out = sad;
    if (score_out) *score_out = ((double)sad / 256.0) / ((double)c->w * (double)c->h);
    return MOTION_OK;
}

int motion_psnr_yuv420_batch(motion_ctx* c, int n, const void* ry, const void* ru,
                             const void* rv, const void* dy, const void* du, const void* dv,
                             size_t pitch_y, size_t pitch_uv, size_t stride_y,
                             size_t stride_uv, void* stream, uint64_t* d_sad_out,
                             uint64_t* d_sse_out) {
    if (!c || n < 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (n == 0) return MOTION_OK;
    if (!d_sad_out || !d_sse_out) return MOTION_ERR_INVALID_ARGUMENT;
    int rc = validate_yuv(c, n, ry, ru, rv, dy, du, dv, pitch_y, pitch_uv, stride_y, stride_uv);
    if (rc) return rc;
    if ((rc = ctx_device_ok(c))) return rc;
    return launch_fused(c, n, ry, ru, rv, dy, du, dv, pitch_y, pitch_uv, stride_y, stride_uv,
                        (cudaStream_t)stream, d_sad_out, d_sse_out);
}

int motion_reserve_host_staging(motion_ctx* c, int pairs_per_chunk, size_t stride_y,
                                size_t stride_uv) {
    if (!c || pairs_per_chunk < 0) return MOTION_ERR_INVALID_ARGUMENT;
    int rc = ctx_device_ok(c);
    if (rc) return rc;
    const size_t s = (size_t)sample_bytes(c->bpc);
    if (stride_y == 0) stride_y = (size_t)c->w * s * (size_t)c->h;
    if (stride_uv == 0) stride_uv = (size_t)c->cw * s * (size_t)c->ch;
    if (pairs_per_chunk == 0) {
        // about 256 MB of pictures per chunk (copies of that size run at the
        // host link's rate; 64 MB chunks lost ~4 %), at least one pair
        const size_t pair_bytes = 2 * (stride_y + 2 * stride_uv);
        pairs_per_chunk = (int)(((size_t)256 << 20) / (pair_bytes ? pair_bytes : 1));
        if (pairs_per_chunk < 1) pairs_per_chunk = 1;
        if (pairs_per_chunk > 64) pairs_per_chunk = 64;
    }
    if (c->stage_pairs >= pairs_per_chunk && c->stage_stride_y >= stride_y &&
        c->stage_stride_uv >= stride_uv && c->d_stage[0])
        return MOTION_OK;
    rc = reserve_stage(c, 2 * (size_t)pairs_per_chunk * (stride_y + 2 * stride_uv),
                       4 * (size_t)pairs_per_chunk);
    if (rc) return rc;
    c->stage_pairs = pairs_per_chunk;
    c->stage_stride_y = stride_y;
    c->stage_stride_uv = stride_uv;
    return MOTION_OK;
}

int motion_psnr_yuv420_batch_host(motion_ctx* c, int n, const void* ry, const void* ru,
                                  const void* rv, const void* dy, const void* du,
                                  const void* dv, size_t pitch_y, size_t pitch_uv,
                                  size_t stride_y, size_t stride_uv, uint64_t* h_sad_out,
                                  uint64_t* h_sse_out) {
    if (!c || n < 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (n == 0) return MOTION_OK;
    if (!h_sad_out || !h_sse_out) return MOTION_ERR_INVALID_ARGUMENT;
    int rc = validate_yuv(c, n, ry, ru, rv, dy, du, dv, pitch_y, pitch_uv, stride_y, stride_uv);
    if (rc) return rc;
    if ((rc = ctx_device_ok(c))) return rc;
    const size_t s = (size_t)sample_bytes(c->bpc);
    if (stride_y < pitch_y * (size_t)(c->h - 1) + (size_t)c->w * s ||
        stride_uv < pitch_uv * (size_t)(c->ch - 1) + (size_t)c->cw * s)
        return MOTION_ERR_BAD_PITCH;  // host pairs must not overlap
    if ((rc = motion_reserve_host_staging(c, c->stage_pairs, stride_y, stride_uv))) return rc;
    if ((rc = reserve_host_results(c, 4 * (size_t)n))) return rc;
    unsigned long long* h_sad = c->h_res;
    unsigned long long* h_sse = c->h_res + n;
    const int P = c->stage_pairs;
    const size_t ybytes = (size_t)P * stride_y, cbytes = (size_t)P * stride_uv;
    const void* src[6] = {ry, ru, rv, dy, du, dv};
    const int nchunks = (n + P - 1) / P;
    for (int ci = 0; ci < nchunks; ++ci) {
        const int k = ci & 1;
        const int first = ci * P;
        const int m = (n - first) < P ? (n - first) : P;
        uint8_t* dst[6];
        dst[0] = c->d_stage[k];
        dst[1] = dst[0] + ybytes;
        dst[2] = dst[1] + cbytes;
        dst[3] = dst[2] + cbytes;
        dst[4] = dst[3] + ybytes;
        dst[5] = dst[4] + cbytes;
        // the staging set k is free once the kernel of chunk ci-2 has finished
        MG_CUDA(cudaStreamWaitEvent(c->s_copy, c->ev_done[k], 0));
        for (int p = 0; p < 6; ++p) {
            const bool luma = (p == 0 || p == 3);
            const size_t stride = luma ? stride_y : stride_uv;
            const size_t last = luma ? pitch_y * (size_t)(c->h - 1) + (size_t)c->w * s
                                     : pitch_uv * (size_t)(c->ch - 1) + (size_t)c->cw * s;
            const size_t bytes = (size_t)(m - 1) * stride + last;
            MG_CUDA(cudaMemcpyAsync(dst[p], (const uint8_t*)src[p] + (size_t)first * stride, bytes,
                                    cudaMemcpyHostToDevice, c->s_copy));
        }
        MG_CUDA(cudaEventRecord(c->ev_in[k], c->s_copy));
        MG_CUDA(cudaStreamWaitEvent(c->s_comp, c->ev_in[k], 0));
        uint64_t* d_sad = (uint64_t*)c->d_res[k];
        uint64_t* d_sse = d_sad + P;
        rc = launch_fused(c, m, dst[0], dst[1], dst[2], dst[3], dst[4], dst[5], pitch_y, pitch_uv,
                          stride_y, stride_uv, c->s_comp, d_sad, d_sse);
        if (rc) return rc;
        MG_CUDA(cudaMemcpyAsync(h_sad + first, d_sad, sizeof(uint64_t) * (size_t)m,
                                cudaMemcpyDeviceToHost, c->s_comp));
        MG_CUDA(cudaMemcpyAsync(h_sse + 3 * (size_t)first, d_sse, sizeof(uint64_t) * 3 * (size_t)m,
                                cudaMemcpyDeviceToHost, c->s_comp));
        MG_CUDA(cudaEventRecord(c->ev_done[k], c->s_comp));
    }
    if ((rc = queue_error_read(c, c->s_comp))) return rc;
    MG_CUDA(cudaStreamSynchronize(c->s_comp));
    if ((int)(uint32_t)c->h_slot[1] != 0) return device_failed(c, c->s_comp);
    std::memcpy(h_sad_out, h_sad, sizeof(uint64_t) * (size_t)n);
    std::memcpy(h_sse_out, h_sse, sizeof(uint64_t) * 3 * (size_t)n);
    return MOTION_OK;
}

int motion_submit_batch_host(motion_ctx* c, const void* h_frames, int n, size_t frame_stride,
                             size_t pitch, int frames_per_chunk, uint64_t* h_sad_out) {
    if (!c || n < 0 || frames_per_chunk < 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (n == 0) return MOTION_OK;
    if (!h_sad_out) return MOTION_ERR_INVALID_ARGUMENT;
    int rc = check_layout(h_frames, pitch, frame_stride, n, c->w, c->bpc);
    if (rc) return rc;
    if ((rc = ctx_device_ok(c))) return rc;
    const size_t last = pitch * (size_t)(c->h - 1) + (size_t)c->w * (size_t)sample_bytes(c->bpc);
    if (n > 1 && frame_stride < last) return MOTION_ERR_BAD_PITCH;   // host frames must not overlap
    const size_t slot = n > 1 ? frame_stride : last;
    int F = frames_per_chunk;
    if (F == 0) {
        // about 256 MB of frames per chunk (copies of that size run at the host
        // link's rate), 1 to 256 frames
        const size_t f = ((size_t)256 << 20) / slot;
        F = f < 1 ? 1 : (f > 256 ? 256 : (int)f);
    }
    if (F > n) F = n;
    if ((rc = reserve_stage(c, (size_t)(F - 1) * slot + last, (size_t)F))) return rc;
    if ((rc = reserve_host_results(c, (size_t)n))) return rc;
    unsigned long long* h_sad = c->h_res;
    const int nchunks = (n + F - 1) / F;
    for (int ci = 0; ci < nchunks; ++ci) {
        const int k = ci & 1;
        const int first = ci * F;
        const int m = (n - first) < F ? (n - first) : F;
        // the staging set k is free once the kernel of chunk ci-2 has finished
        MG_CUDA(cudaStreamWaitEvent(c->s_copy, c->ev_done[k], 0));
        MG_CUDA(cudaMemcpyAsync(c->d_stage[k], (const uint8_t*)h_frames + (size_t)first * slot,
                                (size_t)(m - 1) * slot + last, cudaMemcpyHostToDevice, c->s_copy));
        MG_CUDA(cudaEventRecord(c->ev_in[k], c->s_copy));
        MG_CUDA(cudaStreamWaitEvent(c->s_comp, c->ev_in[k], 0));
        unsigned long long* d_sad = c->d_res[k];
        MG_CUDA(cudaMemsetAsync(d_sad, 0, sizeof(uint64_t) * (size_t)m, c->s_comp));
        mg::TileArgs a = motion_args(c, m);
        a.ref_y = c->d_stage[k];
        a.pitch_y = (long long)pitch;
        a.stride_y = (long long)slot;
        a.aligned16 = aligned16(c->d_stage[k], pitch, slot, m);
        a.sad_out = d_sad;
        if ((rc = launch_motion(c, a, false, c->s_comp))) return rc;
        MG_CUDA(cudaMemcpyAsync(h_sad + first, d_sad, sizeof(uint64_t) * (size_t)m,
                                cudaMemcpyDeviceToHost, c->s_comp));
        MG_CUDA(cudaEventRecord(c->ev_done[k], c->s_comp));
    }
    if ((rc = queue_error_read(c, c->s_comp))) return rc;
    MG_CUDA(cudaStreamSynchronize(c->s_comp));
    if ((int)(uint32_t)c->h_slot[1] != 0) return device_failed(c, c->s_comp);
    std::memcpy(h_sad_out, h_sad, sizeof(uint64_t) * (size_t)n);
    return MOTION_OK;
}

int psnr_sse(const void* d_ref, const void* d_dist, size_t ref_pitch, size_t dist_pitch, int w,
             int h, int bpc, void* stream, uint64_t* d_sse_out) {
    if (bpc < 8 || bpc > 16) return MOTION_ERR_UNSUPPORTED_BITDEPTH;
    if (w < 1 || h < 1) return MOTION_ERR_INVALID_ARGUMENT;
    if (w > MOTION_MAX_DIM || h > MOTION_MAX_DIM) return MOTION_ERR_TOO_LARGE;
    if (!d_sse_out) return MOTION_ERR_INVALID_ARGUMENT;
    int rc;
    if ((rc = check_layout(d_ref, ref_pitch, 0, 1, w, bpc))) return rc;
    if ((rc = check_layout(d_dist, dist_pitch, 0, 1, w, bpc))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    MG_CUDA(cudaMemsetAsync(d_sse_out, 0, sizeof(uint64_t), s));
    int dev = 0, sms = 0;
    MG_CUDA(cudaGetDevice(&dev));
    MG_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    mg::SseArgs a;
    std::memset(&a, 0, sizeof(a));
    a.ref_y = (const uint8_t*)d_ref;
    a.dist_y = (const uint8_t*)d_dist;
    a.ref_pitch_y = (long long)ref_pitch;
    a.dist_pitch_y = (long long)dist_pitch;
    a.w = w;
    a.h = h;
    a.bpc = bpc;
    a.n = 1;
    a.planes = 1;
    a.sse_out = (unsigned long long*)d_sse_out;
    int launched = 0;
    cudaError_t e = mg::launch_sse(a, s, sms, &launched);
    g_launches += (uint64_t)launched;
    if (e != cudaSuccess) return cuda_fail(e);
    return MOTION_OK;
}

int psnr_sse_yuv420_batch(int w, int h, int bpc, int n, const void* ry, const void* ru,
                          const void* rv, const void* dy, const void* du, const void* dv,
                          size_t pitch_y, size_t pitch_uv, size_t stride_y, size_t stride_uv,
                          void* stream, uint64_t* d_sse_out) {
    if (bpc < 8 || bpc > 16) return MOTION_ERR_UNSUPPORTED_BITDEPTH;
    if (w < 1 || h < 1 || n < 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (w > MOTION_MAX_DIM || h > MOTION_MAX_DIM) return MOTION_ERR_TOO_LARGE;
    if (n == 0) return MOTION_OK;
    if (!d_sse_out) return MOTION_ERR_INVALID_ARGUMENT;
    const int cw = (w + 1) / 2, ch = (h + 1) / 2;
    int rc;
    if ((rc = check_layout(ry, pitch_y, stride_y, n, w, bpc))) return rc;
    if ((rc = check_layout(dy, pitch_y, stride_y, n, w, bpc))) return rc;
    if ((rc = check_layout(ru, pitch_uv, stride_uv, n, cw, bpc))) return rc;
    if ((rc = check_layout(rv, pitch_uv, stride_uv, n, cw, bpc))) return rc;
    if ((rc = check_layout(du, pitch_uv, stride_uv, n, cw, bpc))) return rc;
    if ((rc = check_layout(dv, pitch_uv, stride_uv, n, cw, bpc))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    MG_CUDA(cudaMemsetAsync(d_sse_out, 0, sizeof(uint64_t) * 3 * (size_t)n, s));
    int dev = 0, sms = 0;
    MG_CUDA(cudaGetDevice(&dev));
    MG_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    mg::SseArgs a;
    std::memset(&a, 0, sizeof(a));
    a.ref_y = (const uint8_t*)ry;
    a.dist_y = (const uint8_t*)dy;
    a.ref_u = (const uint8_t*)ru;
    a.dist_u = (const uint8_t*)du;
    a.ref_v = (const uint8_t*)rv;
    a.dist_v = (const uint8_t*)dv;
    a.ref_pitch_y = (long long)pitch_y;
    a.dist_pitch_y = (long long)pitch_y;
    a.pitch_uv = (long long)pitch_uv;
    a.stride_y = (long long)stride_y;
    a.stride_uv = (long long)stride_uv;
    a.w = w;
    a.h = h;
    a.cw = cw;
    a.ch = ch;
    a.bpc = bpc;
    a.n = n;
    a.planes = 3;
    a.sse_out = (unsigned long long*)d_sse_out;
    int launched = 0;
    cudaError_t e = mg::launch_sse(a, s, sms, &launched);
    g_launches += (uint64_t)launched;
    if (e != cudaSuccess) return cuda_fail(e);
    return MOTION_OK;
}

int moment_sums_batch(int w, int h, int bpc, int n, const void* d_ref, const void* d_dist,
                      size_t pitch, size_t stride, void* stream, uint64_t* d_out) {
    if (bpc < 8 || bpc > 16) return MOTION_ERR_UNSUPPORTED_BITDEPTH;
    if (w < 1 || h < 1 || n < 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (w > MOTION_MAX_DIM || h > MOTION_MAX_DIM) return MOTION_ERR_TOO_LARGE;
    if (n == 0) return MOTION_OK;
    if (!d_out) return MOTION_ERR_INVALID_ARGUMENT;
    int rc;
    if ((rc = check_layout(d_ref, pitch, stride, n, w, bpc))) return rc;
    if ((rc = check_layout(d_dist, pitch, stride, n, w, bpc))) return rc;
    if (n > 1 && stride < pitch * (size_t)(h - 1) + (size_t)w * (size_t)sample_bytes(bpc))
        return MOTION_ERR_BAD_PITCH;
    cudaStream_t s = (cudaStream_t)stream;
    MG_CUDA(cudaMemsetAsync(d_out, 0, sizeof(uint64_t) * 4 * (size_t)n, s));
    int dev = 0, sms = 0;
    MG_CUDA(cudaGetDevice(&dev));
    MG_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    mg::MomentArgs a;
    std::memset(&a, 0, sizeof(a));
    a.ref = (const uint8_t*)d_ref;
    a.dist = (const uint8_t*)d_dist;
    a.pitch = (long long)pitch;
    a.stride = (long long)stride;
    a.w = w;
    a.h = h;
    a.bpc = bpc;
    a.n = n;
    a.out = (unsigned long long*)d_out;
    int launched = 0;
    cudaError_t e = mg::launch_moment(a, s, sms, &launched);
    g_launches += (uint64_t)launched;
    if (e != cudaSuccess) return cuda_fail(e);
    return MOTION_OK;
}

int moments_from_sums(const uint64_t* sums, int n, int w, int h, double* out) {
    if (n < 0 || w <= 0 || h <= 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (n > 0 && (!sums || !out)) return MOTION_ERR_INVALID_ARGUMENT;
    const double count = (double)w * (double)h;
    for (int i = 0; i < 4 * n; ++i) out[i] = (double)sums[i] / count;
    return MOTION_OK;
}

int motion_scores_from_sad(const uint64_t* sad, int n, int w, int h, const double* next_score,
                           double* score, double* motion2) {
    if (n < 0 || w <= 0 || h <= 0) return MOTION_ERR_INVALID_ARGUMENT;
    if (n > 0 && (!sad || !score || !motion2)) return MOTION_ERR_INVALID_ARGUMENT;
    const double area = (double)w * (double)h;
    for (int i = 0; i < n; ++i) score[i] = ((double)sad[i] / 256.0) / area;
    for (int i = 0; i < n; ++i) {
        if (i + 1 < n)
            motion2[i] = std::fmin(score[i], score[i + 1]);
        else
            motion2[i] = next_score ? std::fmin(score[i], *next_score) : score[i];
    }
    return MOTION_OK;
}

int psnr_from_sse(uint64_t sse, uint64_t n_samples, int bpc, double* mse, double* psnr_db) {
    if (n_samples == 0 || bpc < 8 || bpc > 16) return MOTION_ERR_INVALID_ARGUMENT;
    const double m = (double)sse / (double)n_samples;
    if (mse) *mse = m;
    if (psnr_db) {
        const double peak = (double)((1u << bpc) - 1u);
        *psnr_db = sse == 0 ? INFINITY : 10.0 * std::log10(peak * peak / m);
    }
    return MOTION_OK;
}

int motion_set_kernel_path(motion_ctx* c, int path) {
    if (!c || path < MOTION_PATH_AUTO || path > MOTION_PATH_TMA_16)
        return MOTION_ERR_INVALID_ARGUMENT;
    c->force_generic = path == MOTION_PATH_GENERIC;
    c->force_rows = path == MOTION_PATH_TMA_32 ? mg::kTileH : path == MOTION_PATH_TMA_16 ? mg::kShortTileH : 0;
    return MOTION_OK;
}

int motion_plan_chunks(int w, int h, int n, int resident_ctas, int* chunks_out) {
    if (w < 1 || h < 1 || n < 0 || resident_ctas < 1 || !chunks_out)
        return MOTION_ERR_INVALID_ARGUMENT;
    const long long tiles = (long long)((w + mg::kTileW - 1) / mg::kTileW) *
                            ((h + mg::kTileH - 1) / mg::kTileH);
    *chunks_out = mg::plan_frame_chunks(tiles, resident_ctas, n, 8);
    return MOTION_OK;
}

int motion_tile_order(int w, int h, int chunks, long long block, int* tile_out) {
    if (w < 1 || h < 1 || w > 32768 || h > 32768 || chunks < 1 || chunks > 8 || !tile_out)
        return MOTION_ERR_INVALID_ARGUMENT;
    const int gx = (w + mg::kTileW - 1) / mg::kTileW, gy = (h + mg::kTileH - 1) / mg::kTileH;
    if (block < 0 || block >= (long long)gx * gy * chunks) return MOTION_ERR_INVALID_ARGUMENT;
    mg::tile_of_block(w, h, gx, gy, chunks, (int)block, &tile_out[0], &tile_out[1], &tile_out[2]);
    return MOTION_OK;
}

int motion_launch_blocks(int w, int h, int n, int tile_rows, int resident_ctas, long long block, int* work_out,
                         long long* blocks_out) {
    if (w < 1 || h < 1 || w > 32768 || h > 32768 || n < 1 || resident_ctas < 1 || !blocks_out ||
        (tile_rows != mg::kTileH && tile_rows != mg::kShortTileH))
        return MOTION_ERR_INVALID_ARGUMENT;
    const int gx = (w + mg::kTileW - 1) / mg::kTileW, gy = (h + tile_rows - 1) / tile_rows;
    const long long tiles = (long long)gx * gy;
    const mg::LaunchPlan p = mg::plan_launch(tiles, resident_ctas, n, false, false);
    *blocks_out = p.blocks;
    if (block < 0) return MOTION_OK;   // the count only
    if (block >= p.blocks || !work_out) return MOTION_ERR_INVALID_ARGUMENT;
    mg::block_work(w, h, gx, gy, p.gz, n, p.chunk, p.tiles_a, p.chunk_b, (int)block, &work_out[0], &work_out[1],
                   &work_out[2], &work_out[3], tile_rows);
    return MOTION_OK;
}

int motion_launch_shape(int w, int h, int n, int v2, int resident_ctas, int* tile_rows) {
    if (w < 1 || h < 1 || w > 32768 || h > 32768 || n < 1 || resident_ctas < 1 || !tile_rows)
        return MOTION_ERR_INVALID_ARGUMENT;
    const long long tiles = (long long)((w + mg::kTileW - 1) / mg::kTileW) * ((h + mg::kTileH - 1) / mg::kTileH);
    *tile_rows = mg::prefer_short_tiles(tiles, resident_ctas, n, 8, v2 != 0) ? mg::kShortTileH : mg::kTileH;
    return MOTION_OK;
}

int motion_set_copy_limit(motion_ctx* c, size_t bytes) {
    if (!c) return MOTION_ERR_INVALID_ARGUMENT;
    c->rp_limit = bytes;
    return MOTION_OK;
}

int motion_inject_alloc_failure(int nth) {
    if (nth < 0) return MOTION_ERR_INVALID_ARGUMENT;
    g_fail_alloc_in.store(nth);
    return MOTION_OK;
}

int motion_set_stall_injection(motion_ctx* c, int on) {
    if (!c) return MOTION_ERR_INVALID_ARGUMENT;
    c->stall_injection = on ? 1 : 0;
    return MOTION_OK;
}

int motion_device_error(motion_ctx* c, int* flags) {
    if (!c || !flags) return MOTION_ERR_INVALID_ARGUMENT;
    int rc = ctx_device_ok(c);
    if (rc) return rc;
    MG_CUDA(cudaDeviceSynchronize());
    int v = 0;
    MG_CUDA(cudaMemcpy(&v, c->d_err, sizeof(int), cudaMemcpyDeviceToHost));
    MG_CUDA(cudaMemset(c->d_err, 0, sizeof(int)));
    if (v) {
        // the resident planes may be incomplete: the next call starts a sequence
        c->has_prev = 0;
        c->v2_has_prev = 0;
    }
    *flags = v;
    return MOTION_OK;
}

uint64_t motion_kernel_launch_count(void) { return g_launches.load(); }

int motion_last_cuda_error(void) { return g_last_cuda_error.load(); }

const char* motion_strerror(int code) {
    switch (code) {
        case MOTION_OK: return "ok";
        case MOTION_ERR_INVALID_ARGUMENT: return "invalid argument";
        case MOTION_ERR_FRAME_TOO_SMALL: return "frame smaller than 3x3";
        case MOTION_ERR_UNSUPPORTED_BITDEPTH: return "bits per sample outside [8, 16]";
        case MOTION_ERR_BAD_PITCH: return "pitch, stride or alignment does not fit the samples";
        case MOTION_ERR_TOO_LARGE: return "frame larger than MOTION_MAX_DIM";
        case MOTION_ERR_CUDA: return "CUDA runtime error";
        case MOTION_ERR_OUT_OF_MEMORY: return "out of memory";
        case MOTION_ERR_NO_DEVICE: return "no CUDA device";
        case MOTION_ERR_WRONG_DEVICE: return "current device is not the context's device";
        case MOTION_ERR_DEVICE:
            return "a kernel reported a device error (a bounded wait ran out or a bounds check "
                   "failed); results incomplete, sequence restarted";
        default: return "unknown status";
    }
}

}  // extern "C"
