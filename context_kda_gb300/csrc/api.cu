// C ABI entry points of libkda (declared and documented in include/kda.h).
//
// Every call validates its arguments on the host and enqueues nothing when it
// rejects them; no call allocates, frees or synchronises.  There is no
// fallback path (cuLA PR #110, "feat(cp): add opt-in NVSHMEM CP state handoff",
// §Supported configuration: request an error instead of fallback).
#include <cstdint>
#include <mutex>

#include "kda_internal.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return KDA_OK;
    g_last_cuda_error = static_cast<int>(e);
    return KDA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A host plan is accepted when kda_plan_check accepts it.  The check re-plans, so the plans
// already accepted are remembered by (length, checksum, T, N, S); a plan whose words hash to a
// remembered entry is accepted after the O(length) checksum pass alone.
struct PlanKey {
    int32_t total, checksum, T, N, S;
    bool operator==(const PlanKey &o) const
    {
        return total == o.total && checksum == o.checksum && T == o.T && N == o.N && S == o.S;
    }
};
std::mutex g_plan_mutex;
PlanKey g_plan_seen[16];
int g_plan_seen_n = 0, g_plan_seen_next = 0;

bool plan_ok(const int32_t *plan)
{
    if (!plan) return false;
    if (plan[KDA_PH_MAGIC] != KDA_PLAN_MAGIC || plan[KDA_PH_VERSION] != KDA_PLAN_VERSION) return false;
    if (plan[KDA_PH_TOTAL] < KDA_PLAN_HEADER_WORDS) return false;
    const uint32_t sum = kda::plan_checksum_words(plan, static_cast<size_t>(plan[KDA_PH_TOTAL]));
    if (sum != static_cast<uint32_t>(plan[KDA_PH_CHECKSUM])) return false;
    const PlanKey key{plan[KDA_PH_TOTAL], plan[KDA_PH_CHECKSUM], plan[KDA_PH_T], plan[KDA_PH_N], plan[KDA_PH_S]};
    {
        std::lock_guard<std::mutex> lock(g_plan_mutex);
        for (int i = 0; i < g_plan_seen_n; ++i)
            if (g_plan_seen[i] == key) return true;
    }
    if (kda_plan_check(plan) != KDA_OK) return false;
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    g_plan_seen[g_plan_seen_next] = key;
    g_plan_seen_next = (g_plan_seen_next + 1) % 16;
    if (g_plan_seen_n < 16) ++g_plan_seen_n;
    return true;
}

size_t round256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

constexpr int kBlockedMinSegments = 16;   // fewer segments always compose by the chain

bool layout(const int32_t *plan, int32_t H, size_t off[7])
{
    if (!plan_ok(plan) || H < 1) return false;
    const size_t h = static_cast<size_t>(H), K = kda::KD, V = kda::VD;
    const size_t sizes[6] = {
        h * static_cast<size_t>(plan[KDA_PH_TCONT]) * K * 2,                 // qhat (bf16)
        static_cast<size_t>(plan[KDA_PH_NFIN]) * h * K * K * 4,              // fin transitions
        static_cast<size_t>(plan[KDA_PH_NCHUNKS]) * h * KDA_PACKAGE_BYTES,   // chunk packages
        static_cast<size_t>(plan[KDA_PH_S]) * h * K * K * 4,                 // A
        static_cast<size_t>(plan[KDA_PH_S]) * h * K * V * 4,                 // B
        static_cast<size_t>(plan[KDA_PH_S]) * h * K * V * 4,                 // S_in
    };
    size_t pos = 0;
    for (int i = 0; i < 6; ++i) {
        off[i] = pos;
        pos = round256(pos + sizes[i]);
    }
    // from 16 segments on, room for the two-level scan's group totals and incoming states after S_in
    if (plan[KDA_PH_S] >= kBlockedMinSegments) pos = round256(pos + kda::scan_scratch_bytes(plan, H));
    off[6] = pos;
    return true;
}

// The composition schedule of the fused entry points: the two-level scan where its estimated depth,
// counted in products per CTA over the waves the device's SMs need, is below the chain's.
bool use_blocked_scan(const int32_t *plan, int32_t H)
{
    const long long S = plan[KDA_PH_S];
    if (S < kBlockedMinSegments) return false;
    const long long sm = kda::sm_count(), m = kda::scan_group_size(static_cast<int>(S)), G = (S + m - 1) / m;
    auto waves = [&](long long ctas) { return (ctas + sm - 1) / sm; };
    const long long chain = waves(4LL * H) * S;
    const long long blocked = waves(8LL * H * G) * (m + 1) + (G - 1) + waves(4LL * H * G) * (m + 1);
    return blocked < chain;
}

bool inputs_ok(const void *q, const void *k, const void *v, const float *g, const float *beta,
               const float *h0)
{
    if (!q || !k || !v || !g || !beta) return false;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta)) return false;
    if (h0 && !aligned16(h0)) return false;
    return true;
}

size_t S_in_bytes(const int32_t *plan, int32_t H)
{
    return static_cast<size_t>(plan[KDA_PH_S]) * static_cast<size_t>(H) * kda::KD * kda::VD * 4;
}

kda::Workspace carve(void *ws, const size_t off[7])
{
    char *b = static_cast<char *>(ws);
    return kda::Workspace{reinterpret_cast<uint16_t *>(b + off[0]), reinterpret_cast<float *>(b + off[1]),
                          reinterpret_cast<unsigned char *>(b + off[2]), reinterpret_cast<float *>(b + off[3]),
                          reinterpret_cast<float *>(b + off[4]), reinterpret_cast<float *>(b + off[5])};
}

// Bytes of the qhat + fin regions that kda_apply_boundary reads.
size_t boundary_bytes(const size_t off[7]) { return off[2]; }
// Bytes of the qhat + fin + package regions that kda_segment_forward uses.
size_t segment_bytes(const size_t off[7]) { return off[3]; }

}  // namespace

extern "C" const char *kda_status_string(int status)
{
    switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case KDA_ERR_WORKSPACE: return "buffer too small";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_TIMEOUT: return "device wait timed out";
    case KDA_ERR_RANGE: return "decay out of the chunkwise range";
    default: return "unknown status";
    }
}

extern "C" int kda_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int kda_selftest_wait_expiry(void *stream)
{
    return cuda_status(kda::launch_wait_expiry_probe(static_cast<cudaStream_t>(stream)));
}

extern "C" int kda_selftest_state_abort(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                        const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const float *g,
                                        const float *beta, const float *h0, float scale, kda_bf16 *o, float *A,
                                        float *B, float *final_state, void *ws, size_t ws_bytes, void *stream)
{
    size_t off[7];
    if (!layout(plan, H, off) || !plan_dev) return KDA_ERR_INVALID_ARG;
    if (plan[KDA_PH_MAXPIECE] <= KDA_CHUNK) return KDA_ERR_INVALID_ARG;   // needs a piece of two chunks
    if (!inputs_ok(q, k, v, g, beta, h0)) return KDA_ERR_INVALID_ARG;
    if (!o || !A || !B || !final_state || !aligned16(o) || !aligned16(A) || !aligned16(B) ||
        !aligned16(final_state))
        return KDA_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws)) return KDA_ERR_INVALID_ARG;
    if (ws_bytes < off[3]) return KDA_ERR_WORKSPACE;
    const kda::Workspace w = carve(ws, off);
    return cuda_status(kda::launch_state_abort_selftest(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, A, B,
                                                        final_state, w.qhat, w.afin, w.pkg,
                                                        static_cast<cudaStream_t>(stream)));
}

extern "C" int kda_device_status(void)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        return KDA_ERR_CUDA;
    }
    int worst = KDA_OK;
    for (int st : {kda::take_prep_status(), kda::take_state_status(), kda::take_compose_status(),
                   kda::take_boundary_status(), kda::take_backward_status(), kda::take_reverse_status()})
        if (st != KDA_OK && worst == KDA_OK) worst = st;
    return worst;
}

namespace kda {
void record_cuda_error(int err) { g_last_cuda_error = err; }

PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_f32_rows(CUtensorMap *m, const void *ptr, uint64_t rows, uint32_t cols, uint32_t box_rows)
{
    auto fn = tmap_encode_fn();
    if (!fn || rows == 0) return false;
    const cuuint64_t dims[2] = {cols, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
    const cuuint32_t box[2] = {32, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f32_rows128(CUtensorMap *m, const void *ptr, uint64_t rows, uint32_t box_rows)
{
    return encode_f32_rows(m, ptr, rows, 128, box_rows);
}

bool encode_rows_3d(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, uint32_t elem, int H, int T,
                    uint32_t inner, uint32_t box_rows)
{
    auto fn = tmap_encode_fn();
    if (!fn || T <= 0) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {128ull * elem, 128ull * elem * static_cast<cuuint64_t>(H)};
    const cuuint32_t box[3] = {inner, 1, box_rows};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Unique id of the calling thread's current context (driver entry points, looked up once).
cudaError_t current_context_id(unsigned long long *id)
{
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    if (!get_current || !get_id) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    if (!ctx) {   // nothing current yet on this thread: the runtime would use the primary context
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaSetDevice(dev);   // initialises and binds the primary context
        if (e != cudaSuccess) return e;
        if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
    }
    if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    return cudaSuccess;
}

// The dynamic shared-memory limit of a kernel, set once per (kernel, context): the attribute
// belongs to the function in the current context, so after cudaDeviceReset (a new context id) it
// is set again.
cudaError_t set_dynamic_smem(const void *fn, int bytes)
{
    unsigned long long ctx = 0;
    cudaError_t e = current_context_id(&ctx);
    if (e != cudaSuccess) return e;
    struct Done {
        const void *fn;
        unsigned long long ctx;
        int bytes;
    };
    static std::mutex mu;
    static Done done[64];
    static int n_done = 0, next = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n_done; ++i)
            if (done[i].fn == fn && done[i].ctx == ctx && done[i].bytes >= bytes) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    done[next] = Done{fn, ctx, bytes};
    next = (next + 1) % 64;
    if (n_done < 64) ++n_done;
    return cudaSuccess;
}

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}
}  // namespace kda

extern "C" int kda_workspace_layout(const int32_t *plan, int32_t H, size_t off[7])
{
    if (!off) return KDA_ERR_INVALID_ARG;
    return layout(plan, H, off) ? KDA_OK : KDA_ERR_INVALID_ARG;
}

extern "C" size_t kda_workspace_bytes(const int32_t *plan, int32_t H)
{
    size_t off[7];
    return layout(plan, H, off) ? off[6] : 0;
}

extern "C" int kda_segment_forward(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                   const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                   const float *g, const float *beta, const float *h0, float scale,
                                   kda_bf16 *o, float *A, float *B, float *final_state,
                                   void *ws, size_t ws_bytes, void *stream)
{
    size_t off[7];
    if (!layout(plan, H, off) || !plan_dev) return KDA_ERR_INVALID_ARG;
    if (!inputs_ok(q, k, v, g, beta, h0)) return KDA_ERR_INVALID_ARG;
    if (!o || !A || !B || !final_state || !aligned16(o) || !aligned16(A) || !aligned16(B) ||
        !aligned16(final_state))
        return KDA_ERR_INVALID_ARG;
    if (segment_bytes(off) > 0 && (!ws || !aligned16(ws))) return KDA_ERR_INVALID_ARG;
    if (ws_bytes < segment_bytes(off)) return KDA_ERR_WORKSPACE;
    const kda::Workspace w = carve(ws, off);
    return cuda_status(kda::launch_chunk_forward(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, A, B,
                                                 final_state, w.qhat, w.afin, w.pkg,
                                                 static_cast<cudaStream_t>(stream)));
}

extern "C" int kda_compose_summaries(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                     const float *A, const float *B, const float *h0, float *S_in,
                                     void *stream)
{
    size_t off[7];
    if (!layout(plan, H, off) || !plan_dev) return KDA_ERR_INVALID_ARG;
    if (!A || !B || !S_in || !aligned16(A) || !aligned16(B) || !aligned16(S_in)) return KDA_ERR_INVALID_ARG;
    if (h0 && !aligned16(h0)) return KDA_ERR_INVALID_ARG;
    return cuda_status(kda::launch_compose(plan, plan_dev, H, A, B, h0, S_in, static_cast<cudaStream_t>(stream)));
}

extern "C" size_t kda_scan_workspace_bytes(const int32_t *plan, int32_t H)
{
    size_t off[7];
    if (!layout(plan, H, off)) return 0;
    return kda::scan_scratch_bytes(plan, H);
}

extern "C" int kda_compose_summaries_blocked(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                             const float *A, const float *B, const float *h0, float *S_in,
                                             void *ws, size_t ws_bytes, void *stream)
{
    size_t off[7];
    if (!layout(plan, H, off) || !plan_dev) return KDA_ERR_INVALID_ARG;
    if (!A || !B || !S_in || !aligned16(A) || !aligned16(B) || !aligned16(S_in)) return KDA_ERR_INVALID_ARG;
    if (h0 && !aligned16(h0)) return KDA_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KDA_ERR_INVALID_ARG;
    if (ws_bytes < kda::scan_scratch_bytes(plan, H)) return KDA_ERR_WORKSPACE;
    return cuda_status(kda::launch_compose_blocked(plan, plan_dev, H, A, B, h0, S_in, ws,
                                                   static_cast<cudaStream_t>(stream)));
}

extern "C" int kda_apply_boundary(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                  const float *S_in, const void *ws, size_t ws_bytes, kda_bf16 *o,
                                  float *final_state, void *stream)
{
    size_t off[7];
    if (!layout(plan, H, off) || !plan_dev) return KDA_ERR_INVALID_ARG;
    if (!S_in || !o || !final_state || !aligned16(S_in) || !aligned16(o) || !aligned16(final_state))
        return KDA_ERR_INVALID_ARG;
    if (boundary_bytes(off) > 0 && (!ws || !aligned16(ws))) return KDA_ERR_INVALID_ARG;
    if (ws_bytes < boundary_bytes(off)) return KDA_ERR_WORKSPACE;
    const kda::Workspace w = carve(const_cast<void *>(ws), off);
    return cuda_status(kda::launch_boundary(plan, plan_dev, H, S_in, w.qhat, w.afin, o, final_state,
                                            static_cast<cudaStream_t>(stream)));
}

extern "C" int kda_forward_segmented(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                     const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                     const float *g, const float *beta, const float *h0, float scale,
                                     kda_bf16 *o, float *final_state, void *ws, size_t ws_bytes,
                                     void *stream)
{
    size_t off[7];
    if (!layout(plan, H, off) || !plan_dev) return KDA_ERR_INVALID_ARG;
    if (!inputs_ok(q, k, v, g, beta, h0)) return KDA_ERR_INVALID_ARG;
    if (!o || !final_state || !aligned16(o) || !aligned16(final_state)) return KDA_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws)) return KDA_ERR_INVALID_ARG;
    if (ws_bytes < off[6]) return KDA_ERR_WORKSPACE;
    const kda::Workspace w = carve(ws, off);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = cuda_status(kda::launch_chunk_forward(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, w.A, w.B,
                                                   final_state, w.qhat, w.afin, w.pkg, s));
    if (rc != KDA_OK) return rc;
    rc = cuda_status(use_blocked_scan(plan, H)
                         ? kda::launch_compose_blocked(plan, plan_dev, H, w.A, w.B, h0, w.S_in,
                                                       static_cast<char *>(ws) + round256(off[5] + S_in_bytes(plan, H)), s)
                         : kda::launch_compose(plan, plan_dev, H, w.A, w.B, h0, w.S_in, s));
    if (rc != KDA_OK) return rc;
    return cuda_status(kda::launch_boundary(plan, plan_dev, H, w.S_in, w.qhat, w.afin, o, final_state, s));
}

extern "C" int kda_forward_two_pass(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                    const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                                    const float *g, const float *beta, const float *h0, float scale,
                                    kda_bf16 *o, float *final_state, void *ws, size_t ws_bytes, void *stream)
{
    size_t off[7];
    if (!layout(plan, H, off) || !plan_dev) return KDA_ERR_INVALID_ARG;
    if (!inputs_ok(q, k, v, g, beta, h0)) return KDA_ERR_INVALID_ARG;
    if (!o || !final_state || !aligned16(o) || !aligned16(final_state)) return KDA_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws)) return KDA_ERR_INVALID_ARG;
    if (ws_bytes < off[6]) return KDA_ERR_WORKSPACE;
    const kda::Workspace w = carve(ws, off);
    return cuda_status(kda::launch_two_pass(plan, plan_dev, H, q, k, v, g, beta, h0, scale, o, w.A, w.B, w.S_in,
                                            final_state, w.pkg, static_cast<cudaStream_t>(stream)));
}

namespace {

constexpr int kBackwardGrid = 152;   // CTAs of the backward's chunk and piece kernels (grid-stride)

// Regions of the backward's workspace after the forward's: o and final states of the forward run it
// needs (not returned), the chunk start states and end gradients, the segment end gradients and
// continuing pieces' incoming-state gradients, the CTAs' scratch, and each chunk's terms for the chains.
bool backward_layout(const int32_t *plan, int32_t H, size_t off[10])
{
    size_t fw[7];
    if (!layout(plan, H, fw)) return false;
    const size_t h = static_cast<size_t>(H), K = kda::KD, V = kda::VD;
    const size_t T = static_cast<size_t>(plan[KDA_PH_T]), N = static_cast<size_t>(plan[KDA_PH_N]);
    const size_t S = static_cast<size_t>(plan[KDA_PH_S]), C = static_cast<size_t>(plan[KDA_PH_NCHUNKS]);
    const size_t sizes[9] = {T * h * V * 2, N * h * K * V * 4, h * C * K * V * 4, h * C * K * V * 4,
                             S * h * K * V * 4, S * h * K * V * 4,
                             static_cast<size_t>(kBackwardGrid) * kda::backward_scratch_floats() * 4,
                             h * C * kda::BT_FLOATS * 4, h * C * kda::RIMG_UNIT};
    size_t pos = fw[6];
    for (int i = 0; i < 9; ++i) {
        off[i] = pos;
        pos = round256(pos + sizes[i]);
    }
    off[9] = pos;
    return true;
}

}  // namespace

extern "C" size_t kda_backward_workspace_bytes(const int32_t *plan, int32_t H)
{
    size_t off[10];
    return backward_layout(plan, H, off) ? off[9] : 0;
}

extern "C" int kda_backward_segmented(const int32_t *plan, const int32_t *plan_dev, int32_t H,
                                      const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v, const float *g,
                                      const float *beta, const float *h0, float scale, const kda_bf16 *dout,
                                      const float *dfinal, float *dq, float *dk, float *dv, float *dg,
                                      float *dbeta, float *dh0, void *ws, size_t ws_bytes, void *stream)
{
    size_t fw[7], off[10];
    if (!layout(plan, H, fw) || !backward_layout(plan, H, off) || !plan_dev) return KDA_ERR_INVALID_ARG;
    if (!inputs_ok(q, k, v, g, beta, h0)) return KDA_ERR_INVALID_ARG;
    if (!dout || !aligned16(dout) || (dfinal && !aligned16(dfinal)) || (dh0 && !aligned16(dh0)))
        return KDA_ERR_INVALID_ARG;
    if (!dq || !dk || !dv || !dg || !dbeta || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(dg) || !aligned16(dbeta))
        return KDA_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws)) return KDA_ERR_INVALID_ARG;
    if (ws_bytes < off[9]) return KDA_ERR_WORKSPACE;
    const kda::Workspace w = carve(ws, fw);
    char *b = static_cast<char *>(ws);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the forward's local pass and composition: S_in, the segment transitions A and the final-state
    // transitions of continuing pieces
    // (its preparation in backward mode also leaves each chunk's FP32 terms and operand images)
    int rc = cuda_status(kda::launch_chunk_forward(plan, plan_dev, H, q, k, v, g, beta, h0, scale,
                                                   reinterpret_cast<uint16_t *>(b + off[0]), w.A, w.B,
                                                   reinterpret_cast<float *>(b + off[1]), w.qhat, w.afin, w.pkg, s,
                                                   reinterpret_cast<unsigned char *>(b + off[8]),
                                                   reinterpret_cast<float *>(b + off[7])));
    if (rc != KDA_OK) return rc;
    rc = cuda_status(use_blocked_scan(plan, H)
                         ? kda::launch_compose_blocked(plan, plan_dev, H, w.A, w.B, h0, w.S_in,
                                                       b + round256(fw[5] + S_in_bytes(plan, H)), s)
                         : kda::launch_compose(plan, plan_dev, H, w.A, w.B, h0, w.S_in, s));
    if (rc != KDA_OK) return rc;
    // every piece again from its true incoming state, recording each chunk's start state
    rc = cuda_status(kda::launch_state_record(plan, plan_dev, H, h0, w.S_in, w.pkg,
                                              reinterpret_cast<uint16_t *>(b + off[0]),
                                              reinterpret_cast<float *>(b + off[1]),
                                              reinterpret_cast<float *>(b + off[2]), s));
    if (rc != KDA_OK) return rc;
    return cuda_status(kda::launch_backward(
        plan, plan_dev, H, q, k, v, g, beta, scale, dout, dfinal, w.A, w.afin,
        reinterpret_cast<const float *>(b + off[2]), reinterpret_cast<float *>(b + off[3]),
        reinterpret_cast<float *>(b + off[4]), reinterpret_cast<float *>(b + off[5]), w.S_in,
        reinterpret_cast<const float *>(b + off[1]), reinterpret_cast<float *>(b + off[7]),
        reinterpret_cast<unsigned char *>(b + off[8]),
        reinterpret_cast<float *>(b + off[6]), kBackwardGrid, dq, dk, dv, dg, dbeta, dh0, s));
}
