// motion_noalloc.cu -- the allocation-free form of the batched motion submit.
//
// Some callers cannot allocate device memory: a host application that hands
// all device memory out through its own pool and does not let libraries call
// cudaMalloc, or a latency-critical loop in which an allocation (which can
// synchronise the device) is not acceptable.  For them this entry point keeps
// the one piece of scratch the motion kernel needs between calls -- the
// previous frame's blurred plane -- in a fixed array compiled into the
// library, instead of in memory that a context allocates.
//
// The array is static device memory: every GPU that loads the library holds
// it until the process exits.  Host code cannot use the array's name as a
// device address (it names a host-side stand-in), so the entry point asks the
// runtime for the device address once per device, on its first call on that
// device with the device current, and keeps it.
//
// The kernels report a bounded wait that ran out (or, in the bounds-checked
// build, a failed check) in a device error word beside the array; the call
// that enqueues them cannot see it without waiting, so
// motion_noalloc_device_error reads and clears it, and a set word makes the
// next call start a new sequence instead of continuing from an incomplete
// plane.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "motion.h"
#include "motion_internal.h"

namespace {

// The previous frame's blurred plane, rows of round_up(w, 8) uint16 values.
constexpr size_t kNoallocSamples = MOTION_NOALLOC_MAX_SAMPLES;
static __device__ __align__(256) uint16_t g_noalloc_bprev[kNoallocSamples];
// Device error word of the kernels launched from here (bounded waits).
static __device__ __align__(256) int g_noalloc_err;

constexpr int kMaxDevices = 64;
struct DeviceSlot {
    uint16_t* bprev = nullptr;   // device address of g_noalloc_bprev on this device
    int* err = nullptr;          // device address of g_noalloc_err on this device
    // the sequence the array currently continues (written by the last call)
    int w = 0, h = 0, bpc = 0;
    bool valid = false;
};
DeviceSlot g_slots[kMaxDevices];
// Guards every slot's host-side fields: host threads calling at once on one
// device are serialised here (their launches still race on the GPU array
// unless the caller orders them).
std::mutex g_slots_mu;
// test hook (motion_noalloc_set_stall_injection): stage waits that can never
// complete, bounded at about 2 ms
bool g_stall_injection = false;

// With g_slots_mu held.
int setup_device(int dev, DeviceSlot** out) {
    if (dev < 0 || dev >= kMaxDevices) return MOTION_ERR_INVALID_ARGUMENT;
    DeviceSlot& s = g_slots[dev];
    if (!s.bprev) {
        void* p = nullptr;
        void* e = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_bprev) != cudaSuccess ||
            cudaGetSymbolAddress(&e, g_noalloc_err) != cudaSuccess) {
            cudaGetLastError();
            return MOTION_ERR_CUDA;
        }
        s.bprev = static_cast<uint16_t*>(p);
        s.err = static_cast<int*>(e);
    }
    *out = &s;
    return MOTION_OK;
}

}  // namespace

extern "C" int motion_submit_batch_noalloc(const void* d_frames, int n, int w, int h, int bpc,
                                           size_t frame_stride, size_t pitch,
                                           int continue_sequence, void* stream,
                                           uint64_t* d_sad_out) {
    if (n < 0) return MOTION_ERR_INVALID_ARGUMENT;
    int rc = mg::check_dims(w, h, bpc);
    if (rc) return rc;
    const size_t bprev_pitch = ((size_t)w + 7) & ~(size_t)7;
    if (bprev_pitch * (size_t)h > kNoallocSamples) return MOTION_ERR_TOO_LARGE;
    if (n == 0) return MOTION_OK;
    if (!d_sad_out) return MOTION_ERR_INVALID_ARGUMENT;
    if ((rc = mg::check_layout(d_frames, pitch, frame_stride, n, w, bpc))) return rc;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOTION_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_slots_mu);
    DeviceSlot* slot = nullptr;
    if ((rc = setup_device(dev, &slot))) return rc;
    // continuing needs the array to hold the last frame of a sequence of the
    // same size and depth
    if (continue_sequence && !(slot->valid && slot->w == w && slot->h == h && slot->bpc == bpc))
        return MOTION_ERR_INVALID_ARGUMENT;

    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(d_sad_out, 0, sizeof(uint64_t) * (size_t)n, st) != cudaSuccess) {
        cudaGetLastError();
        return MOTION_ERR_CUDA;
    }
    mg::TileArgs a;
    std::memset(&a, 0, sizeof(a));
    a.ref_y = (const uint8_t*)d_frames;
    a.pitch_y = (long long)pitch;
    a.stride_y = (long long)frame_stride;
    a.w = w;
    a.h = h;
    a.cw = (w + 1) / 2;
    a.ch = (h + 1) / 2;
    a.bpc = bpc;
    a.n = n;
    a.has_prev = continue_sequence ? 1 : 0;
    a.store_last = 1;
    a.aligned16 = ((((uintptr_t)d_frames) | pitch) % 16 == 0) && (n <= 1 || frame_stride % 16 == 0);
    a.bprev = slot->bprev;
    a.bprev_out = slot->bprev;   // one array: a continuing launch stays in one chunk
    a.bprev_pitch = (int)bprev_pitch;
    a.sad_out = (unsigned long long*)d_sad_out;
    a.err = slot->err;
    if (g_stall_injection) {
        a.tx_extra = 16;               // the stage expects 16 bytes that never arrive
        a.wait_cycles = 1LL << 22;     // and gives up after about 2 ms
    }
    int launched = 0;
    bool used = false;
    cudaError_t e = mg::launch_motion_tma(a, false, st, &launched, &used);
    if (e == cudaSuccess && !used) e = mg::launch_motion_tile(a, false, st, &launched);
    mg::note_launches(launched);
    if (e != cudaSuccess) return MOTION_ERR_CUDA;
    slot->w = w;
    slot->h = h;
    slot->bpc = bpc;
    slot->valid = true;
    return MOTION_OK;
}

extern "C" int motion_noalloc_device_error(void* stream, int* flags) {
    if (!flags) return MOTION_ERR_INVALID_ARGUMENT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOTION_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_slots_mu);
    DeviceSlot* slot = nullptr;
    int rc = setup_device(dev, &slot);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    int v = 0;
    // the word is read after the stream's earlier work, then cleared on it
    if (cudaMemcpyAsync(&v, slot->err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemsetAsync(slot->err, 0, sizeof(int), st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return MOTION_ERR_CUDA;
    }
    if (v) slot->valid = false;   // the array's plane may be incomplete
    *flags = v;
    return MOTION_OK;
}

extern "C" int motion_noalloc_set_stall_injection(int on) {
    std::lock_guard<std::mutex> lock(g_slots_mu);
    g_stall_injection = on != 0;
    return MOTION_OK;
}
