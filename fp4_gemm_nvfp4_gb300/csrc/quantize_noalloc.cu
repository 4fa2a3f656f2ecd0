// quantize_noalloc.cu -- nvfp4_quantize for callers that cannot provide device
// scratch memory.
//
// The regular quantizer asks its caller for a small device workspace (the
// per-CTA amax partials of its first pass).  Some callers have no way to get
// one: a plugin whose host runtime owns every device allocation and hands the
// plugin only its input and output buffers, or code that must not allocate
// once it is running (cudaMalloc can synchronize the device, and can fail
// under memory pressure at the worst moment).  This entry point takes the
// workspace from a fixed array that lives in the library itself instead.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nvfp4.h"
#include "kernels.h"

namespace {

// The scratch: room for the amax partials of both orientations.  Every GPU
// that loads the library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = nvfp4::kQuantizeWorkspaceBytes;   // 32 KiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch on the current device.  The name
// g_noalloc_scratch is only a host-side handle in host code; the address must
// be looked up once per device, with that device current.
nvfp4_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return NVFP4_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return NVFP4_OK;
}

}  // namespace

extern "C" NVFP4_API nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                                         nvfp4_scaling scaling, nvfp4_rounding rounding,
                                                         uint64_t seed, uint64_t stream_id, int orientations,
                                                         const nvfp4_tensor* out_row, const nvfp4_tensor* out_col,
                                                         nvfp4_stream_t stream) {
    // The scratch must hold the workspace this shape needs; larger needs are
    // refused rather than overrun.
    if (nvfp4_quantize_workspace_size(rows, cols, orientations) > kNoAllocScratchBytes)
        return NVFP4_ERR_WORKSPACE;
    void* scratch = nullptr;
    const nvfp4_status s = scratch_for_current_device(&scratch);
    if (s != NVFP4_OK) return s;
    return nvfp4_quantize(x, rows, cols, ld_x, scaling, rounding, seed, stream_id, orientations, out_row, out_col,
                          scratch, kNoAllocScratchBytes, stream);
}
