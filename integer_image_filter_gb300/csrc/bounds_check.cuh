// bounds_check.cuh -- software bounds checks for the motion kernels.
//
// The bounds-checked build (compiled with MG_BOUNDS_CHECK=1 into a library of
// its own) checks every shared- and global-memory access of the motion
// kernels against the buffer it must stay in: the stage region a TMA box or a
// cp.async copy landed in, the warp's rows of the V tile, the caller's planes
// and output arrays.  An access outside its buffer, or not aligned to its
// width, is skipped (a load yields 0) and sets bit 1 (value 2) of the
// context's device error word.  The normal build compiles every macro below
// to the plain access, so both builds run the same arithmetic.
#pragma once

#include <cstddef>
#include <cstdint>

#ifndef MG_BOUNDS_CHECK
#define MG_BOUNDS_CHECK 0
#endif

namespace mg {

constexpr int kErrBounds = 2;   // device error word bit of a failed bounds check

#if MG_BOUNDS_CHECK
// the error word of the running launch: set by thread 0 before the block's
// first barrier (every checked access comes after it)
static __shared__ int* bc_err;

__device__ __forceinline__ void bc_begin(int* err) {
    if (threadIdx.x == 0) bc_err = err;
}

// [p, p + n) inside [lo, lo + bytes) and p aligned to n (n is the access width)
__device__ __forceinline__ bool bc_ok(const void* p, size_t n, const void* lo, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(lo);
    const bool ok = a >= b && a + n <= b + bytes && (a & (n - 1)) == 0;
    if (!ok && bc_err) atomicOr(bc_err, kErrBounds);
    return ok;
}

template <typename T>
__device__ __forceinline__ T bc_ld(const T* p, const void* lo, size_t bytes) {
    return bc_ok(p, sizeof(T), lo, bytes) ? *p : T{};
}

template <typename T>
__device__ __forceinline__ void bc_st(T* p, const T& v, const void* lo, size_t bytes) {
    if (bc_ok(p, sizeof(T), lo, bytes)) *p = v;
}

#define MG_BC_BEGIN(err) ::mg::bc_begin(err)
#define MG_LD(p, lo, bytes) ::mg::bc_ld((p), (lo), (size_t)(bytes))
#define MG_ST(p, v, lo, bytes) ::mg::bc_st((p), (v), (lo), (size_t)(bytes))
#define MG_OK(p, n, lo, bytes) ::mg::bc_ok((p), (size_t)(n), (lo), (size_t)(bytes))
#else
#define MG_BC_BEGIN(err) ((void)0)
#define MG_LD(p, lo, bytes) (*(p))
#define MG_ST(p, v, lo, bytes) (*(p) = (v))
#define MG_OK(p, n, lo, bytes) true
#endif

// A buffer an access must stay in (the checked build); unused otherwise.
struct Span {
    const void* p;
    size_t n;
};

// Bytes from the first sample of n planes (frames `stride` bytes apart, rows
// `pitch` bytes apart) to the end of the last sample of the last plane.
__host__ __device__ __forceinline__ long long plane_span(int n, long long stride, int h, long long pitch,
                                                         int w, int s) {
    return (n > 1 ? (long long)(n - 1) * stride : 0) + (long long)(h - 1) * pitch + (long long)w * s;
}

}  // namespace mg
