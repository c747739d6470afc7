// Composition of the segment summaries into each segment's incoming state.
//
// cuLA PR #136 ("feat(kda): add cuDNN concatenated-summary Kimi CP", §Summary):
// affine summary composition in FP32.  With the seed (0, h0) in front of the
// first segment, the prefix composition (A_{j-1},B_{j-1}) o ... o (0, h0) always
// has a zero transition, so the incoming state is its state part:
//     S_in[0] = h0[first sequence],
//     S_in[j] = h0[s]                            if sequence s starts at b_j,
//             = B[j-1]                           if a sequence starts inside j-1,
//             = A[j-1] S_in[j-1] + B[j-1]        otherwise (a "step").
// The value columns are independent, so each CTA carries a 32-column slice of
// one head's state through all segments.  A step is one tcgen05 product
// D = A[j-1] S_in[j-1] (M = 128 rows, N = 32, K = 128) with both operands split
// into bf16 hi/lo and three products accumulated in FP32 in TMEM.
//
// The chain is pipelined so that a step costs its product and a short
// epilogue, not a memory round trip:
// - Transitions arrive by tiled TMA (four 32-column boxes, 128-byte swizzle)
//   into two staging buffers, two steps ahead (the L2 is warmed one step
//   further), and the worker warps split each into bf16 hi/lo straight into
//   TMEM, the A operand of its product, one step ahead while the previous
//   product runs; two TMEM operand buffers alternate.
// - The slice an iteration adds (B[j-1] or h0) arrives by TMA into one of two
//   buffers, two iterations ahead.
// - The epilogue adds it to the product, writes S_in[j] into one of two output
//   buffers that a TMA store drains, and splits S_in[j] into the bf16 hi/lo
//   shared-memory operand of the next product.
// - An issuer warp issues the products and the transition copies; an I/O warp
//   the stores and the slice copies.
// Every mbarrier has one waiting role that can fall at most one phase behind
// its arrivals, so parity waits never alias: the issuer waits once per step,
// the I/O warp once per iteration on the barrier of that iteration's parity.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int NS = 32;                     // value columns per CTA
constexpr int NC = NS / 2;                 // columns per epilogue thread
constexpr uint32_t CS_S = 2048;            // state operand (rows k, cols c), read MN-major
constexpr uint32_t SOP = NS / 8 * CS_S;    // one bf16 part of the state operand (8 KiB)
constexpr uint32_t STG = 65536;            // one fp32 transition, 4 swizzled boxes of 32 columns
constexpr uint32_t SLICE = 16384;          // one fp32 slice box (128 rows x 32 columns, swizzled)
constexpr uint32_t OFF_STG = 0;                       // two transition staging buffers
constexpr uint32_t OFF_VAL = OFF_STG + 2 * STG;       // two incoming slices (B[j-1] or h0)
constexpr uint32_t OFF_OUT = OFF_VAL + 2 * SLICE;     // two S_in slices on their way out
constexpr uint32_t OFF_SOP = OFF_OUT + 2 * SLICE;     // state operand hi | lo
constexpr uint32_t SMEM_BYTES = OFF_SOP + 2 * SOP;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;    // room to align the base to 1024 bytes
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");

// TMEM columns: the accumulator, then two transition operands (hi: k pairs in 64 columns, lo after)
constexpr uint32_t TM_D = 0;
constexpr uint32_t TM_A = 128;             // operand buffer b at TM_A + 128 b: hi [0, 64), lo [64, 128)
constexpr uint32_t TM_COLS = 512;

__device__ int g_compose_status;

enum { IN_SEED = 0, IN_UPDATE = 1, IN_STEP = 2 };

__device__ __forceinline__ int in_kind(const PlanView &pv, int j)
{
    if (j == 0 || (pv.seg(j)[1] & KDA_SEG_STARTS_SEQ)) return IN_SEED;
    return (pv.seg(j - 1)[1] & KDA_SEG_HAS_RESET) ? IN_UPDATE : IN_STEP;
}

// First segment >= j whose incoming state is a step (S if none).
__device__ __forceinline__ int next_step(const PlanView &pv, int j)
{
    const int S = pv.S();
    while (j < S && in_kind(pv, j) != IN_STEP) ++j;
    return j;
}

constexpr int NWORK = 256;                 // 8 worker warps
constexpr int NT = NWORK + 64;             // + issuer warp + I/O warp
constexpr int MMA_TID = NWORK, IO_TID = NWORK + 32;

__global__ void __launch_bounds__(NT, 1)
compose_tc(const int32_t *__restrict__ plan, PlanSig sig, int H, int has_h0, const float *__restrict__ A_raw,
           const __grid_constant__ CUtensorMap tm_A, const __grid_constant__ CUtensorMap tm_B,
           const __grid_constant__ CUtensorMap tm_h0, const __grid_constant__ CUtensorMap tm_S)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_mbar;      // a step's product is done (one arrival per step)
    __shared__ __align__(8) uint64_t s_mready;    // workers -> issuer: a step's operands are in place
    __shared__ __align__(8) uint64_t s_abar[2];   // transition staged, per staging buffer
    __shared__ __align__(8) uint64_t s_vbar[2];   // incoming slice staged, per buffer
    __shared__ __align__(8) uint64_t s_oready[2]; // workers -> I/O: iteration done, per parity
    __shared__ __align__(8) uint64_t s_ofree[2];  // I/O -> workers: output buffer read by its store
    __shared__ uint32_t s_tmem;
    if (!plan_matches(plan, sig)) {   // not the plan the launch was sized from: touch nothing
        if (threadIdx.x == 0) record_status(&g_compose_status, KDA_ERR_INVALID_ARG);
        return;
    }
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = (warp >> 2) & 1;
    const int nsl = VD / NS;
    const int h = blockIdx.x / nsl, col0 = (blockIdx.x % nsl) * NS;
    const int S = pv.S();
    const int r = quad * 32 + lane;   // state row (and TMEM lane) of this worker
    const int cl = half * NC;         // its first column within the slice
    const uint32_t sbase = smem_u32(smem);
    const uint32_t mbar = smem_u32(&s_mbar), mready = smem_u32(&s_mready);
    const bool worker = tid < NWORK, issuer = tid == MMA_TID, io = tid == IO_TID;

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(mready, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_abar[i]), 1);
            mbar_init(smem_u32(&s_vbar[i]), 1);
            mbar_init(smem_u32(&s_oready[i]), 1);
            mbar_init(smem_u32(&s_ofree[i]), 1);
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    grid_dep_wait();     // the summaries come from the previous kernel
    grid_dep_launch();   // the fix-up may be scheduled on SMs this kernel leaves

    auto needs_vals = [&](int j) { return in_kind(pv, j) != IN_SEED || has_h0; };
    auto is_step = [&](int j) { return j < S && in_kind(pv, j) == IN_STEP; };
    // issuer: the transition of step j (segment j - 1) into staging buffer b
    auto fetch_A = [&](int j, int b) {
        const uint32_t bar = smem_u32(&s_abar[b]);
        const int y = ((j - 1) * H + h) * KD;
        mbar_arrive_expect_tx(bar, STG);
#pragma unroll
        for (int bx = 0; bx < 4; ++bx) tma_load_2d(sbase + OFF_STG + b * STG + bx * SLICE, &tm_A, 32 * bx, y, bar);
    };
    // I/O thread: the slice iteration j adds (B[j-1] or h0) into buffer j & 1
    auto fetch_vals = [&](int j) {
        const uint32_t bar = smem_u32(&s_vbar[j & 1]);
        mbar_arrive_expect_tx(bar, SLICE);
        const uint32_t dst = sbase + OFF_VAL + (j & 1) * SLICE;
        if (in_kind(pv, j) == IN_SEED)
            tma_load_2d(dst, &tm_h0, col0, (pv.seg(j)[0] * H + h) * KD, bar);
        else
            tma_load_2d(dst, &tm_B, col0, ((j - 1) * H + h) * KD, bar);
    };

    bool ok = true;
    if (worker) {
        bool bad = false;
        uint32_t n_step = 0;                       // steps whose product this thread has consumed
        uint32_t n_conv = 0;                       // transitions split into TMEM so far
        uint32_t v_count[2] = {0, 0};              // slices consumed per buffer
        for (int j = 0; j < S; ++j) {
            // (a) the next step's transition: staging -> TMEM operand (bf16 hi | lo); lane = row r,
            //     this thread's half of the columns k
            if (is_step(j + 1)) {
                const int b = n_conv & 1;
                if (!mbar_wait_warp(smem_u32(&s_abar[b]), (n_conv >> 1) & 1)) bad = true;
                ++n_conv;
                const unsigned char *stg = smem + OFF_STG + b * STG;
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int bx = 0; bx < 2; ++bx) {
                    const unsigned char *box = stg + (2 * half + bx) * SLICE;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const float4 x = *reinterpret_cast<const float4 *>(box + sw128(r, ch));
                        split_bf16x2(x.x, x.y, hi[bx * 16 + 2 * ch], lo[bx * 16 + 2 * ch]);
                        split_bf16x2(x.z, x.w, hi[bx * 16 + 2 * ch + 1], lo[bx * 16 + 2 * ch + 1]);
                    }
                }
                const uint32_t ta = tbase + (static_cast<uint32_t>(quad * 32) << 16) + TM_A + b * 128 + half * 32;
                tmem_st32_nowait(ta, hi);
                tmem_st32_nowait(ta + 64, lo);
                tmem_wait_st();
            }
            // (b) this step's product
            float st[NC];
            if (is_step(j)) {
                if (!mbar_wait_warp(mbar, n_step & 1)) bad = true;
                ++n_step;
                fence_after();
                tmem_ld16(tbase + (static_cast<uint32_t>(quad * 32) << 16) + TM_D + cl, st);
            } else {
#pragma unroll
                for (int e = 0; e < NC; ++e) st[e] = 0.f;
            }
            // (c) + B[j-1] or h0
            if (needs_vals(j)) {
                const int b = j & 1;
                if (!mbar_wait_warp(smem_u32(&s_vbar[b]), v_count[b]++ & 1)) bad = true;
                const unsigned char *vb = smem + OFF_VAL + b * SLICE;
#pragma unroll
                for (int m = 0; m < NC / 4; ++m) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(vb + sw128(r, cl / 4 + m));
                    st[4 * m] += b4.x;
                    st[4 * m + 1] += b4.y;
                    st[4 * m + 2] += b4.z;
                    st[4 * m + 3] += b4.w;
                }
            }
            // (d) S_in[j] into output buffer j & 1, once the store of iteration j - 2 has read it
            {
                const int b = j & 1;
                if (j >= 2 && !mbar_wait_warp(smem_u32(&s_ofree[b]), ((j - 2) >> 1) & 1)) bad = true;
                unsigned char *ob = smem + OFF_OUT + b * SLICE;
#pragma unroll
                for (int m = 0; m < NC / 4; ++m)
                    *reinterpret_cast<float4 *>(ob + sw128(r, cl / 4 + m)) =
                        make_float4(st[4 * m], st[4 * m + 1], st[4 * m + 2], st[4 * m + 3]);
            }
            // (e) S_in[j] as the next product's operand (rows k = r, cols c), bf16 hi | lo
            if (is_step(j + 1)) {
#pragma unroll
                for (int m = 0; m < NC / 8; ++m) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) split_bf16x2(st[8 * m + 2 * p], st[8 * m + 2 * p + 1], hi[p], lo[p]);
                    const uint32_t off = static_cast<uint32_t>((cl / 8 + m) * CS_S + (r >> 3) * 128 + (r & 7) * 16);
                    *reinterpret_cast<uint4 *>(smem + OFF_SOP + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(smem + OFF_SOP + SOP + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            // (f) hand the iteration over: the next product's operands to the issuer, the output
            //     buffer and the consumed slice buffer to the I/O warp
            fence_async_smem();
            fence_before();
            if (bar_or1(NWORK, bad)) {
                ok = false;
                break;
            }
            if (tid == 0) {
                if (is_step(j + 1)) mbar_arrive(mready);
                mbar_arrive(smem_u32(&s_oready[j & 1]));
            }
        }
        if (bad) ok = false;
    } else if (issuer) {
        // per step n (in order): once its operands are in place, its product; then the transition
        // of step n + 2 into the staging buffer step n's transition was split from
        int j_cur = next_step(pv, 1);
        int j_ahead = j_cur < S ? next_step(pv, j_cur + 1) : S;
        uint32_t n = 0, n_fetch[2] = {0, 0};
        if (j_cur < S) {
            fetch_A(j_cur, 0);
            n_fetch[0] = 1;
        }
        if (j_ahead < S) {
            fetch_A(j_ahead, 1);
            n_fetch[1] = 1;
        }
        while (j_cur < S) {
            if (!(ok = mbar_wait(mready, n & 1))) break;
            fence_after();
            {
                const uint32_t id = idesc_bf16(128, NS, 0, 1);
                const uint32_t ta = tbase + TM_A + (n & 1) * 128;
                const uint32_t s_hi = sbase + OFF_SOP;
                const uint32_t aop[3] = {ta, ta, ta + 64}, sop[3] = {s_hi, s_hi + SOP, s_hi};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ta(tbase + TM_D, aop[ps] + kk * 8, sdesc(sop[ps] + kk * 256, 128, CS_S), id,
                                    (ps | kk) != 0);
                commit(mbar);
            }
            // staging buffer n & 1 was split before this step's handoff: it takes step n + 2
            const int j_next = j_ahead < S ? next_step(pv, j_ahead + 1) : S;
            if (j_next < S) {
                fetch_A(j_next, n & 1);
                ++n_fetch[n & 1];
                const int j_warm = next_step(pv, j_next + 1);   // and the L2 warms the one after
                if (j_warm < S) {
                    const float *pa = A_raw + static_cast<size_t>((j_warm - 1) * H + h) * KD * KD;
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(pa), "r"(STG) : "memory");
                }
            }
            ++n;
            j_cur = j_ahead;
            j_ahead = j_next;
        }
        if (!ok) record_status(&g_compose_status, KDA_ERR_TIMEOUT);
        // whatever happened elsewhere, the products and copies this role issued land before the CTA
        // frees its tensor memory (bounded waits; immediate when the workers consumed them)
        if (n) mbar_wait(mbar, (n - 1) & 1);
        for (int b = 0; b < 2; ++b)
            if (n_fetch[b]) mbar_wait(smem_u32(&s_abar[b]), (n_fetch[b] - 1) & 1);
    } else if (io) {
        // per iteration j: once the workers hand it over, the store of S_in[j] and the copy of the
        // slice iteration j + 2 adds (into the buffer iteration j read)
        uint32_t n_fetch[2] = {0, 0};
        if (needs_vals(0)) {
            fetch_vals(0);
            ++n_fetch[0];
        }
        if (S > 1 && needs_vals(1)) {
            fetch_vals(1);
            ++n_fetch[1];
        }
        for (int j = 0; j < S; ++j) {
            if (!(ok = mbar_wait(smem_u32(&s_oready[j & 1]), (j >> 1) & 1))) break;
            tma_store_2d(&tm_S, col0, (j * H + h) * KD, sbase + OFF_OUT + (j & 1) * SLICE);
            bulk_commit_group();
            if (j + 2 < S && needs_vals(j + 2)) {
                fetch_vals(j + 2);
                ++n_fetch[j & 1];
            }
            bulk_wait_read_all();                      // output buffer j & 1 has been read
            mbar_arrive(smem_u32(&s_ofree[j & 1]));
        }
        if (!ok) record_status(&g_compose_status, KDA_ERR_TIMEOUT);
        bulk_wait_all();
        for (int b = 0; b < 2; ++b)
            if (n_fetch[b]) mbar_wait(smem_u32(&s_vbar[b]), (n_fetch[b] - 1) & 1);
    }
    // A role whose wait gave up has recorded it; every role has let its own copies and products land
    // above, so the tensor memory can be freed.
    if (!__syncthreads_and(ok) && tid == 0) record_status(&g_compose_status, KDA_ERR_TIMEOUT);
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

cudaError_t launch_compose(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *A,
                           const float *B, const float *h0, float *S_in, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    const int S = pv.S();
    if (S <= 0) return cudaSuccess;
    const uint64_t rows = static_cast<uint64_t>(S) * H * KD;
    CUtensorMap tA, tB, tH, tS;
    if (!encode_f32_rows128(&tA, A, rows, KD) || !encode_f32_rows128(&tB, B, rows, KD) ||
        !encode_f32_rows128(&tS, S_in, rows, KD))
        return cudaErrorInvalidValue;
    if (h0) {
        if (!encode_f32_rows128(&tH, h0, static_cast<uint64_t>(pv.N()) * H * KD, KD)) return cudaErrorInvalidValue;
    } else {
        tH = tB;   // never read: no segment takes a seed from h0
    }
    cudaError_t err =
        cudaFuncSetAttribute(compose_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_ALLOC));
    if (err != cudaSuccess) return err;
    return launch_dependent(compose_tc, dim3(H * (VD / NS)), dim3(NT), SMEM_ALLOC, stream, plan_dev,
                            plan_sig(plan_host), H, h0 ? 1 : 0, A, tA, tB, tH, tS);
}

// The status word of this file's kernel: read and cleared (the caller has synchronised the device).
int take_compose_status()
{
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_compose_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_compose_status, &z, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return v;
}

}  // namespace kda
