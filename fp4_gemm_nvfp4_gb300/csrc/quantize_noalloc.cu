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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nvfp4.h"
#include "kernels.h"

namespace {

// The scratch: room for the amax partials of both orientations.  Every GPU
// that loads the library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = 32 * 1024;
static_assert(nvfp4::kQuantizeWorkspaceBytes <= kNoAllocScratchBytes,
              "the quantizer's workspace must fit the library-held scratch");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// Per device: the context the address was looked up in and the address.  A
// device reset, or a primary context released and created again, loads the
// module anew (possibly elsewhere), so the address is looked up again
// whenever the current context's id changes.
unsigned long long g_scratch_ctx[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the calling thread's current context (0 if there is none yet).
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return false;
    *id = 0;
    return !ctx || get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch in the current context.  In host code the
// name g_noalloc_scratch is only a host-side handle; the device address is
// looked up with that device current (cudaGetSymbolAddress, which also makes
// the runtime's primary context current if none was) and cached per device
// and context.
nvfp4_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) return NVFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return NVFP4_ERR_CUDA;
        if (!current_context_id(&ctx) || ctx == 0) return NVFP4_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
        g_scratch_ctx[dev] = ctx;
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
