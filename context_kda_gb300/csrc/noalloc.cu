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
// (with that device current) and caches it.  The cache is keyed on the
// context's unique id as well as the device: after cudaDeviceReset, or when the
// primary context is destroyed and created again, the module is loaded anew and
// the next call looks the address up again instead of reusing a stale one.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(KDA_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // id of the context the address belongs to

// Device address of g_noalloc_scratch in the current context (looked up once per device and context).
cudaError_t scratch_address(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned long long ctx = 0;
    e = kda::current_context_id(&ctx);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
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
