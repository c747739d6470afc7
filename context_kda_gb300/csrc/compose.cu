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
// All global traffic is tiled TMA with the 128-byte swizzle: each transition
// arrives one step ahead and is split while the previous step's MMA runs; the
// B (or h0) slice a step adds arrives in a 16 KiB buffer where the epilogue
// forms S_in[j] in place, and one TMA store writes it out.  Eight warps split
// operands and run the epilogue; a ninth warp issues the MMAs and the
// transition loads, and a tenth owns the slice loads and stores, so neither
// the split nor the copies wait on MMA issue.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int NS = 32;                     // value columns per CTA
constexpr int NC = NS / 2;                 // columns per epilogue thread
constexpr uint32_t LBO_A = 2048;           // transition operand (rows r, cols k), K-major
constexpr uint32_t TILE_A = 16 * LBO_A;
constexpr uint32_t CS_S = 2048;            // state operand (rows k, cols c), read MN-major
constexpr uint32_t SOP = NS / 8 * CS_S;
constexpr uint32_t OFF_AOP = 0;                       // two buffers, each hi | lo
constexpr uint32_t OFF_SOP = OFF_AOP + 4 * TILE_A;    // hi | lo
constexpr uint32_t OFF_STG = OFF_SOP + 2 * SOP;       // fp32 transition, 4 swizzled boxes of 32 columns
constexpr uint32_t OFF_BS = OFF_STG + 65536;          // fp32 slice, one swizzled box (B / h0 in, S_in out)
constexpr uint32_t SMEM_BYTES = OFF_BS + 16384;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;    // room to align the base to 1024 bytes
constexpr uint32_t TM_COLS = 32;

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

constexpr int NT = 320;                    // 8 worker warps + MMA warp + I/O warp
constexpr int MMA_TID = 256, IO_TID = 288;

__global__ void __launch_bounds__(NT, 1)
compose_tc(const int32_t *__restrict__ plan, PlanSig sig, int H, int has_h0, const __grid_constant__ CUtensorMap tm_A,
           const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_h0,
           const __grid_constant__ CUtensorMap tm_S)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_mbar, s_abar, s_bbar;
    __shared__ uint32_t s_tmem;
    if (!plan_matches(plan, sig)) {   // not the plan the launch was sized from: touch nothing
        if (threadIdx.x == 0) record_status(&g_compose_status, KDA_ERR_INVALID_ARG);
        return;
    }
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int nsl = VD / NS;
    const int h = blockIdx.x / nsl, col0 = (blockIdx.x % nsl) * NS;
    const int S = pv.S();
    const int r = quad * 32 + lane;   // state row held by this thread in the epilogue
    const int cl = half * NC;         // its first column within the slice
    const uint32_t sbase = smem_u32(smem);
    const uint32_t mbar = smem_u32(&s_mbar), abar = smem_u32(&s_abar), bbar = smem_u32(&s_bbar);
    const bool io = tid == IO_TID;           // slice loads and stores
    const bool issuer = tid == MMA_TID;      // MMAs and transition loads
    const bool worker = tid < 256;

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(abar, 1);
        mbar_init(bbar, 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    grid_dep_wait();     // the summaries come from the previous kernel
    grid_dep_launch();   // the fix-up may be scheduled on SMs this kernel leaves
    uint32_t a_phase = 0, b_phase = 0, mma_phase = 0;
    bool ok = true, a_pending = false, b_pending = false;
    int n_conv = 0, n_mma = 0;   // transitions split so far / steps issued so far

    auto needs_vals = [&](int j) { return in_kind(pv, j) != IN_SEED || has_h0; };
    auto fetch_A = [&](int step) {   // issuer: transition of segment step-1, four 32-column boxes
        const int y = ((step - 1) * H + h) * KD;
        mbar_arrive_expect_tx(abar, 65536u);
#pragma unroll
        for (int b = 0; b < 4; ++b) tma_load_2d(sbase + OFF_STG + b * 16384, &tm_A, 32 * b, y, abar);
    };
    auto fetch_vals = [&](int j) {   // I/O thread: the slice segment j's incoming state starts from
        mbar_arrive_expect_tx(bbar, 16384u);
        if (in_kind(pv, j) == IN_SEED)
            tma_load_2d(sbase + OFF_BS, &tm_h0, col0, (pv.seg(j)[0] * H + h) * KD, bbar);
        else
            tma_load_2d(sbase + OFF_BS, &tm_B, col0, ((j - 1) * H + h) * KD, bbar);
    };
    // staged transition -> operand buffer b (rows r, cols k) as bf16 hi | lo; lanes take consecutive rows
    auto convert_A = [&](int b) {
        a_pending = false;
        ++n_conv;
        const uint32_t par = a_phase++ & 1;   // every thread tracks the phases; workers wait
        if (!worker) return;
        ok &= mbar_wait(abar, par);
        const uint32_t base = OFF_AOP + static_cast<uint32_t>(b) * 2 * TILE_A;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int id = tid + 256 * i, rr = id & 127, kc = id >> 7;   // 8-column chunk kc of row rr
            const unsigned char *box = smem + OFF_STG + (kc >> 2) * 16384;
            const float4 x0 = *reinterpret_cast<const float4 *>(box + sw128(rr, (kc & 3) * 2));
            const float4 x1 = *reinterpret_cast<const float4 *>(box + sw128(rr, (kc & 3) * 2 + 1));
            uint32_t hi[4], lo[4];
            split_bf16x2(x0.x, x0.y, hi[0], lo[0]);
            split_bf16x2(x0.z, x0.w, hi[1], lo[1]);
            split_bf16x2(x1.x, x1.y, hi[2], lo[2]);
            split_bf16x2(x1.z, x1.w, hi[3], lo[3]);
            const uint32_t off = cm_off(rr, kc * 8, LBO_A);
            *reinterpret_cast<uint4 *>(smem + base + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(smem + base + TILE_A + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    };

    {
        const int s0 = next_step(pv, 1);
        if (s0 < S) {
            if (issuer) fetch_A(s0);
            a_pending = true;
        }
        if (needs_vals(0)) {
            if (io) fetch_vals(0);
            b_pending = true;
        }
    }

    for (int j = 0; j < S; ++j) {
        const bool step = in_kind(pv, j) == IN_STEP;
        float st[NC];
        if (step) {
            if (issuer) {
                fence_after();
                const uint32_t id = idesc_bf16(128, NS, 0, 1);
                const uint32_t a_hi = sbase + OFF_AOP + static_cast<uint32_t>(n_mma & 1) * 2 * TILE_A;
                const uint32_t s_hi = sbase + OFF_SOP;
                const uint32_t aop[3] = {a_hi, a_hi, a_hi + TILE_A}, sop[3] = {s_hi, s_hi + SOP, s_hi};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tbase, sdesc(aop[ps] + kk * 2 * LBO_A, LBO_A), sdesc(sop[ps] + kk * 256, 128, CS_S),
                                 id, (ps | kk) != 0);
                commit(mbar);
            }
            ++n_mma;
            // split the next step's transition while this one runs
            const int nxt = next_step(pv, j + 1);
            if (nxt < S && n_conv == n_mma) {
                convert_A(n_conv & 1);
                fence_async_smem();
                __syncthreads();   // staging read by all threads
                const int nn = next_step(pv, nxt + 1);
                if (nn < S) {
                    if (issuer) fetch_A(nn);
                    a_pending = true;
                }
            }
            const uint32_t par = mma_phase++ & 1;
            if (worker) {
                ok &= mbar_wait(mbar, par);
                fence_after();
                float d[NC];
                tmem_ld16(tbase + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(cl), d);
#pragma unroll
                for (int e = 0; e < NC; ++e) st[e] = d[e];
            }
        } else {
#pragma unroll
            for (int e = 0; e < NC; ++e) st[e] = 0.f;
        }
        // S_in[j] = (step ? D : 0) + (B[j-1] or h0 or 0), formed in the slice buffer
        if (needs_vals(j)) {
            b_pending = false;
            const uint32_t par = b_phase++ & 1;
            if (worker) ok &= mbar_wait(bbar, par);
#pragma unroll
            for (int m = 0; m < NC / 4 && worker; ++m) {
                const float4 b4 = *reinterpret_cast<const float4 *>(smem + OFF_BS + sw128(r, cl / 4 + m));
                st[4 * m] += b4.x;
                st[4 * m + 1] += b4.y;
                st[4 * m + 2] += b4.z;
                st[4 * m + 3] += b4.w;
            }
        } else {
            __syncthreads();   // the previous store has finished reading the buffer (the I/O thread waited)
        }
        if (worker) {
#pragma unroll
            for (int m = 0; m < NC / 4; ++m)
                *reinterpret_cast<float4 *>(smem + OFF_BS + sw128(r, cl / 4 + m)) =
                    make_float4(st[4 * m], st[4 * m + 1], st[4 * m + 2], st[4 * m + 3]);
        }
        bool fetch_after = false;
        if (j + 1 < S && in_kind(pv, j + 1) == IN_STEP) {
            if (n_conv == n_mma) {   // not split yet (no step ran since it was staged)
                convert_A(n_conv & 1);
                fetch_after = next_step(pv, j + 2) < S;
            }
            // S_in[j] -> state operand (rows k = r, cols c) as bf16 hi | lo
#pragma unroll
            for (int m = 0; m < NC / 8 && worker; ++m) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) split_bf16x2(st[8 * m + 2 * p], st[8 * m + 2 * p + 1], hi[p], lo[p]);
                const uint32_t off = static_cast<uint32_t>((cl / 8 + m) * CS_S + (r >> 3) * 128 + (r & 7) * 16);
                *reinterpret_cast<uint4 *>(smem + OFF_SOP + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(smem + OFF_SOP + SOP + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        fence_async_smem();
        fence_before();
        const bool all_ok = __syncthreads_and(ok);
        if (io && all_ok) {
            tma_store_2d(&tm_S, col0, (j * H + h) * KD, sbase + OFF_BS);
            bulk_commit_group();
            bulk_wait_read_all();   // the buffer is free again
            if (j + 1 < S && needs_vals(j + 1)) fetch_vals(j + 1);
        }
        if (!all_ok) break;
        if (j + 1 < S && needs_vals(j + 1)) b_pending = true;
        if (fetch_after) {
            if (issuer) fetch_A(next_step(pv, j + 2));
            a_pending = true;
        }
    }
    if (io) bulk_wait_all();
    if (!__syncthreads_and(ok)) {
        // a wait gave up: record it, and let copies and products still in flight land before the CTA exits
        if (issuer) {
            record_status(&g_compose_status, KDA_ERR_TIMEOUT);
            if (a_pending) mbar_wait(abar, a_phase & 1);
            mbar_wait(mbar, mma_phase & 1);
        }
        if (io && b_pending) mbar_wait(bbar, b_phase & 1);
        __syncthreads();
    }
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
    return launch_dependent(compose_tc, dim3(H * (VD / NS)), dim3(NT), SMEM_ALLOC, stream, plan_dev, plan_sig(plan_host), H,
                            h0 ? 1 : 0, tA,
                            tB, tH, tS);
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
