// bounds.cuh -- the kernels' output stores, with the bounds check of the
// library's debug build.
//
// Every store of a code, scale or output element goes through store_out(),
// which also takes the byte range [lo, hi) that the call declared for that
// buffer: from the first byte of the buffer to the last byte the call's shape
// and leading dimension reach.  In the debug build (compiled with
// NVFP4_BOUNDS_CHECK) a store whose bytes do not all lie in that range is
// skipped and counted in a device word of its translation unit, which
// nvfp4_testing_bounds_violations (nvfp4_testing.h) reads and clears; nothing
// traps, so a check that fires leaves the GPU usable.  In the regular build
// store_out() is the plain store and the ranges are never read.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

// Bytes [lo, hi) a kernel may write in one output buffer.
struct Extent {
    uintptr_t lo, hi;
};

// Host: the range of `bytes` bytes from p, less the test-support shrink (the
// debug build's nvfp4_testing_bounds_shrink; 0 otherwise).
Extent extent_of(const void* p, int64_t bytes);

// Host: the range of a row-major [rows][ld] buffer of which each row holds
// `row_bytes` bytes in use (the last row ends after them).
inline Extent extent_rows(const void* p, int64_t rows, int64_t ld_bytes, int64_t row_bytes) {
    return extent_of(p, rows > 0 ? (rows - 1) * ld_bytes + row_bytes : 0);
}

#ifdef NVFP4_BOUNDS_CHECK
// Stores skipped by the check in this translation unit.
static __device__ unsigned int g_bounds_violations;
#endif

template <typename T>
__device__ __forceinline__ void store_out(T* p, const T& v, const Extent& e) {
#ifdef NVFP4_BOUNDS_CHECK
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if (a < e.lo || a + sizeof(T) > e.hi) {
        atomicAdd(&g_bounds_violations, 1u);
        return;
    }
#else
    (void)e;
#endif
    *p = v;
}

// Host: add this translation unit's count of skipped stores to *n and clear
// it (synchronous; nothing to do in the regular build).
inline cudaError_t bounds_read_and_clear_local(uint64_t* n) {
#ifdef NVFP4_BOUNDS_CHECK
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_bounds_violations, sizeof(v));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_bounds_violations, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
    *n += v;
#else
    (void)n;
#endif
    return cudaSuccess;
}

}  // namespace nvfp4
