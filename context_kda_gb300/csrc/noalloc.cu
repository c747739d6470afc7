// kda_forward_segmented_noalloc: the whole segmented forward with its workspace
// in a fixed device array owned by the library, for callers that cannot
// allocate device memory themselves.
//
// Who needs it: code that is handed only its input and output buffers by a host
// framework that owns every device allocation (a plugin inside an inference
// engine, for instance) and has no allocator it may call, and code that must not
// call cudaMalloc in its steady-state loop because an allocation there can
// synchronise the device and stall other work.  The pages have no counterpart to
// this entry point.
//
// The scratch is a file-scope __device__ array of KDA_NOALLOC_SCRATCH_BYTES
// (32 MiB).  Every GPU that loads the library holds it until the process
// exits.  Host code cannot use the array's name as a device address, so the
// first call on each device looks the address up with cudaGetSymbolAddress
// (with that device current) and caches it; later calls on that device reuse
// the cached address.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(KDA_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int kda_forward_segmented_noalloc(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                             const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                             const float *g, const float *beta, const float *h0,
                                             float scale, kda_bf16 *o, float *final_state, void *stream)
{
    const size_t need = kda_workspace_bytes(plan, H);
    if (need == 0) return KDA_ERR_INVALID_ARG;
    if (need > kScratchBytes) return KDA_ERR_WORKSPACE;
    void *ws = nullptr;
    const cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) {
        kda::record_cuda_error(static_cast<int>(e));
        return KDA_ERR_CUDA;
    }
    // Every workspace region (qhat, final-state transitions, A, B, S_in) is written in
    // full before it is read within one call, so nothing left by an earlier call needs
    // clearing.
    return kda_forward_segmented(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, final_state, ws,
                                 kScratchBytes, stream);
}
