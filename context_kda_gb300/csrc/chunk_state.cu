// Serial state pass of the chunkwise KDA forward over one piece (segment x sequence), with the
// segment summaries: state columns (outputs, state update B, final states) and transition
// columns (qhat, transition A).
//
// Per chunk, from the package the preparation kernel wrote (W, Qt, masked QK, Kh, exp(Gamma_C),
// Ut) and the chunk-start state X:
//   U = Ut - W X,   O = Qt X + QK U,   X' = Diag(exp Gamma_C) (X + Kh^T U)
// (the KDA gated delta rule unrolled over a chunk; cuLA PR #110, "feat(cp): add opt-in NVSHMEM
// CP state handoff", §Supported configuration: BF16 inputs, FP32 state).  The transition
// columns run the same recurrence on P (K x K) with zero values from P = I at the piece start,
// so their 'outputs' are qhat_t = scale P_t^T q_t and their end state is the piece's transition
// (cuLA PR #136, "feat(kda): add cuDNN concatenated-summary Kimi CP", §Summary:
// preceding_transition).
//
// Mapping.  One CTA per (work item, head): 8 worker warps and an issuer warp.  The state lives
// transposed in TMEM (lane c, column k) as an FP32 accumulator and, split into bf16 hi/lo, in
// shared memory as the A operand of W X and Qt X.  Per chunk the chain is: (W X)^T = X^T W^T
// (3-term) -> workers form U^T = Ut^T - (W X)^T and split it -> O^T += U^T QK^T (1-term),
// X^T += U^T Kh (3-term) -> workers decay X and split it for the next chunk, then store O.
// Qt X (1-term) runs right after W X.  The package arrives by bulk copies one chunk ahead
// (W and Qt once Qt X has read the previous ones; QK, Kh and the decay double-buffered); Ut
// goes straight into registers, also one chunk ahead.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

// ---- shared-memory map (bytes from the dynamic base; bf16 tiles, hi then lo where split) ------
constexpr uint32_t OFF_XT = 0;          // X^T: rows c (128), cols k (128), CS 2048, hi | lo   2 x 32768
constexpr uint32_t OFF_P1 = 65536;      // package bytes [PK_W, PK_P1_END): W hi | lo, Qt hi   49152
constexpr uint32_t P2_BYTES = PK_P2_END - PK_QK;   // QK, Kh hi | lo, exp(Gamma_C)          41472
constexpr uint32_t OFF_P2 = OFF_P1 + PK_P1_END;    // two buffers of P2_BYTES
constexpr uint32_t OFF_UT = OFF_P2 + 2 * P2_BYTES;  // U^T: rows c, cols r (64), CS 2048, hi | lo;
                                                    // then the row-major O tile for the stores
constexpr uint32_t SMEM_BYTES = OFF_UT + 32768;
constexpr uint32_t T128 = 32768, T64 = 16384;
// offsets inside a P2 buffer
constexpr uint32_t P2_QK = 0, P2_KH = PK_KH - PK_QK, P2_GC = PK_GC - PK_QK;

// ---- TMEM columns --------------------------------------------------------------------------
constexpr uint32_t TM_WX = 0;     // (W X)^T (64 cols)
constexpr uint32_t TM_O = 64;     // O^T (64 cols)
constexpr uint32_t TM_X = 128;    // X^T (128 cols)
constexpr uint32_t TM_COLS = 256;

constexpr int NWORK = 256;             // worker threads
constexpr int NTHREADS = NWORK + 32;   // plus the issuer warp
constexpr int ISSUER = NWORK;
enum { HO_X = 0, HO_U = 1 };           // worker -> issuer handoffs of a chunk

__device__ int g_state_status;   // set to KDA_ERR_TIMEOUT when a bounded wait expires

// Writes 8 consecutive values as bf16 hi and lo (two 16-byte stores).
__device__ __forceinline__ void st_split8(unsigned char *hi, unsigned char *lo, const float *x)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) split_bf16x2(x[2 * p], x[2 * p + 1], h[p], l[p]);
    *reinterpret_cast<uint4 *>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

__global__ void __launch_bounds__(NTHREADS, 1)
chunk_state_tc(const int32_t *__restrict__ plan, int H, const float *__restrict__ h0,
               const unsigned char *__restrict__ pkg, uint16_t *__restrict__ o, float *__restrict__ A,
               float *__restrict__ B, float *__restrict__ fin_state, uint16_t *__restrict__ qhat,
               float *__restrict__ afin)
{
    extern __shared__ __align__(16) unsigned char base[];
    __shared__ __align__(8) uint64_t s_mbar;      // W X, then the output / state products
    __shared__ __align__(8) uint64_t s_mbar_o;    // Qt X (W and Qt read)
    __shared__ __align__(8) uint64_t s_pbar1;     // package part 1 landed
    __shared__ __align__(8) uint64_t s_pbar2[2];  // package part 2 landed, per buffer
    __shared__ __align__(8) uint64_t s_hbar[2];   // worker -> issuer handoffs
    __shared__ uint32_t s_tmem;
    const uint32_t sbase = smem_u32(base);

    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;          // TMEM lane quadrant, column half
    const bool worker = tid < NWORK, issuer = tid == ISSUER;
    const int item = blockIdx.x / H, h = blockIdx.x % H;
    const int32_t *it = pv.item(item);
    const int p = it[0], kind = it[1];
    const int32_t *pc = pv.piece(p);
    const int start = pc[PC_START], len = pc[PC_LEN], seq = pc[PC_SEQ], seg = pc[PC_SEG];
    const int flags = pc[PC_FLAGS], row0 = pc[PC_ROW], fin = pc[PC_FIN];
    const int64_t T_cont = pv.T_cont();
    const int nch = (len + CH - 1) / CH;
    // global index of the piece's first chunk (chunks are numbered piece by piece): each warp sums
    // the earlier pieces' chunk counts, its lanes taking every 32nd piece
    int c0 = 0;
    for (int i = lane; i < p; i += 32) c0 += (pv.piece(i)[PC_LEN] + CH - 1) / CH;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) c0 += __shfl_xor_sync(0xffffffffu, c0, sh);
    auto pk_of = [&](int ci) {
        return pkg + (static_cast<size_t>(h) * pv.n_chunks() + c0 + ci) * KDA_PACKAGE_BYTES;
    };
    const uint32_t mbar = smem_u32(&s_mbar), mbar_o = smem_u32(&s_mbar_o), pbar1 = smem_u32(&s_pbar1);

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(mbar_o, 1);
        mbar_init(pbar1, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_pbar2[i]), 1);
            mbar_init(smem_u32(&s_hbar[i]), 1);
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);  // this warp's lane quadrant
    const int c_lane = quad * 32 + lane;                                     // state column of this thread

    // package parts by bulk copy (issuer thread)
    auto load_p1 = [&](int ci) {
        mbar_arrive_expect_tx(pbar1, PK_P1_END);
        bulk_g2s(sbase + OFF_P1, pk_of(ci) + PK_W, PK_P1_END, pbar1);
    };
    auto load_p2 = [&](int ci) {
        const uint32_t bar = smem_u32(&s_pbar2[ci & 1]);
        mbar_arrive_expect_tx(bar, P2_BYTES);
        bulk_g2s(sbase + OFF_P2 + (ci & 1) * P2_BYTES, pk_of(ci) + PK_QK, P2_BYTES, bar);
    };
    if (issuer && nch > 0) {
        load_p1(0);
        load_p2(0);
    }

    bool aborted = false;   // all workers agree on it (OR-reduced at barriers)
    bool bad = false;       // a bounded wait of this thread gave up
    uint32_t phase = 0;
    auto wait_mma = [&]() {
        if (!mbar_wait_warp(mbar, phase & 1)) bad = true;
        ++phase;
        fence_after();
    };
    // Workers hand a set of shared-memory operands over to the issuer: every writer fences its
    // generic-proxy stores for the tensor core, the workers meet on named barrier 1 (OR-reducing
    // their wait failures, so all of them take the same abort decision), and one of them arrives.
    auto handoff = [&](int which) -> bool {
        fence_async_smem();
        fence_before();
        const bool ab = bar_or1(NWORK, bad);
        if (!ab && tid == 0) mbar_arrive(smem_u32(&s_hbar[which]));
        return ab;
    };
    // Ut^T row c_lane, columns hw*32 .. +32 of chunk ci, into registers (state columns only); the
    // package holds it as [hw][m][c] float4 groups, so each load of a warp reads 512 contiguous bytes
    float4 ut[8];
    auto load_ut = [&](int ci) {
        if (kind != 0 || ci >= nch) return;
        const float4 *src = reinterpret_cast<const float4 *>(pk_of(ci) + PK_U) + hw * 8 * 128 + c_lane;
#pragma unroll
        for (int m = 0; m < 8; ++m) ut[m] = src[m * 128];
    };

    if (worker) {
        // ---- piece start: X^T into TMEM (fp32) and its bf16 split into shared memory
        {
            const bool from_h0 = kind == 0 && (flags & KDA_PIECE_FIRST) && h0 != nullptr;
            const float *src = h0 + (static_cast<size_t>(seq) * H + h) * KD * VD;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float x[32];
                const int k0 = hw * 64 + half * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int kk = k0 + j;
                    x[j] = kind == 1 ? (kk == c_lane ? 1.f : 0.f) : (from_h0 ? src[kk * VD + c_lane] : 0.f);
                }
                tmem_st32(tl + TM_X + k0, x);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    st_split8(base + OFF_XT + cm_off(c_lane, k0 + 8 * m, 2048),
                              base + OFF_XT + T128 + cm_off(c_lane, k0 + 8 * m, 2048), x + 8 * m);
            }
            load_ut(0);
            aborted = handoff(HO_X);   // -> W X, Qt X
        }
        for (int ci = 0; ci < nch && !aborted; ++ci) {
            const int t0 = start + ci * CH;
            const int L = min(CH, len - ci * CH);

            // ================= U^T = Ut^T - (W X)^T, split into the A operand of the next products ===
            wait_mma();
            {
                float d[32];
                tmem_ld32(tl + TM_WX + hw * 32, d);   // (W X)^T[c = c_lane][r = hw*32 + j]
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float4 u4 = kind == 0 ? ut[m] : make_float4(0.f, 0.f, 0.f, 0.f);
                    d[4 * m] = u4.x - d[4 * m];
                    d[4 * m + 1] = u4.y - d[4 * m + 1];
                    d[4 * m + 2] = u4.z - d[4 * m + 2];
                    d[4 * m + 3] = u4.w - d[4 * m + 3];
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t off = cm_off(c_lane, hw * 32 + 8 * m, 2048);
                    st_split8(base + OFF_UT + off, base + OFF_UT + T64 + off, d + 8 * m);
                }
                aborted = handoff(HO_U);   // -> O^T += U^T QK^T, X^T += U^T Kh
            }
            if (aborted) break;
            load_ut(ci + 1);

            // ================= outputs (or qhat) to HBM; new X^T split into shared memory =============
            wait_mma();
            {
                // O^T and this thread's half of X^T (X + Kh^T U) in one batch of TMEM reads
                uint32_t od[32], xa[32], xb[32];
                tmem_ld32_nowait(tl + TM_O + hw * 32, od);   // O^T[c][r = hw*32 + j]
                tmem_ld32_nowait(tl + TM_X + hw * 64, xa);
                tmem_ld32_nowait(tl + TM_X + hw * 64 + 32, xb);
                tmem_wait_ld();
                reg_fence32(od);
                reg_fence32(xa);
                reg_fence32(xb);
                const float *gc = reinterpret_cast<const float *>(base + OFF_P2 + (ci & 1) * P2_BYTES + P2_GC);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int k0 = hw * 64 + half * 32;
                    float x[32];   // Diag(exp Gamma_C) (X + Kh^T U)
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(half ? xb[j] : xa[j]) * gc[k0 + j];
                    tmem_st32(tl + TM_X + k0, x);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        st_split8(base + OFF_XT + cm_off(c_lane, k0 + 8 * m, 2048),
                                  base + OFF_XT + T128 + cm_off(c_lane, k0 + 8 * m, 2048), x + 8 * m);
                }
                aborted = handoff(HO_X);   // -> next chunk's W X, Qt X (they overlap the stores below)
                if (aborted) break;
                // O^T[c][r] -> row-major bf16 tile in the U^T region (free: its products have completed),
                // then 16-byte coalesced stores: outputs for state columns, qhat for transition columns
                {
                    uint16_t *so = reinterpret_cast<uint16_t *>(base + OFF_UT);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        so[(hw * 32 + j) * 128 + c_lane] = f32_to_bf16_bits(__uint_as_float(od[j]));
                }
                bar_sync1(NWORK);
                uint16_t *const dst_row0 = kind == 0 ? o + (static_cast<size_t>(t0) * H + h) * VD
                                                     : qhat + (static_cast<size_t>(h) * T_cont + row0 + ci * CH) * KD;
                const size_t row_stride = kind == 0 ? static_cast<size_t>(H) * VD : KD;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int id = tid + 256 * i, r = id >> 4, c16 = id & 15;
                    if (r < L)
                        *reinterpret_cast<uint4 *>(dst_row0 + r * row_stride + c16 * 8) =
                            *reinterpret_cast<const uint4 *>(base + OFF_UT + r * 256 + c16 * 16);
                }
                bar_sync1(NWORK);   // the O tile is read before the next U^T overwrites it
            }
        }
    } else if (issuer) {
        // Issuer: per chunk, W X and Qt X once the state split is in, the output / state products
        // once U^T is; package parts are staged one chunk ahead.
        bool ok = true;
        int n_p1 = nch > 0 ? 1 : 0, n_p2[2] = {nch > 0 ? 1 : 0, 0};
        for (int ci = 0; ci < nch && ok; ++ci) {
            const uint32_t par = ci & 1;
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_X]), par))) break;
            if (ci + 1 < nch) {   // its buffer's previous chunk (ci - 1) is fully consumed
                load_p2(ci + 1);
                ++n_p2[(ci + 1) & 1];
            }
            if (!(ok = mbar_wait(pbar1, par))) break;
            fence_after();
            {
                // (W X)^T = X^T W^T (3-term; W read MN-major)
                const uint32_t idw = idesc_bf16(128, 64, 0, 1);
                const uint32_t aoff[3] = {0, 0, T128}, boff[3] = {0, T64, 0};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tbase + TM_WX, sdesc(sbase + OFF_XT + aoff[ps] + kk * 2 * 2048, 2048),
                                 sdesc(sbase + OFF_P1 + PK_W + boff[ps] + kk * 256, 128, 2048), idw, (ps | kk) != 0);
                commit(mbar);
                // O^T = X^T Qt^T (1-term)
                const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase + TM_O, sdesc(sbase + OFF_XT + kk * 2 * 2048, 2048),
                             sdesc(sbase + OFF_P1 + PK_Q + kk * 2 * 1024, 1024), id, kk != 0);
                commit(mbar_o);
            }
            if (!(ok = mbar_wait(mbar_o, par))) break;
            if (ci + 1 < nch) {   // W and Qt have been read
                load_p1(ci + 1);
                ++n_p1;
            }
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_U]), par))) break;
            if (!(ok = mbar_wait(smem_u32(&s_pbar2[ci & 1]), (ci >> 1) & 1))) break;
            fence_after();
            {
                const unsigned char *p2 = base + OFF_P2 + (ci & 1) * P2_BYTES;
                const uint32_t s2 = smem_u32(p2);
                // O^T += U^T QK^T (1-term)
                const uint32_t id64 = idesc_bf16(128, 64), id128 = idesc_bf16(128, 128, 0, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tbase + TM_O, sdesc(sbase + OFF_UT + kk * 2 * 2048, 2048),
                             sdesc(s2 + P2_QK + kk * 2 * 1024, 1024), id64, 1);
                // X^T += U^T Kh (3-term; Kh read MN-major)
                const uint32_t aoff[3] = {0, 0, T64}, boff[3] = {0, T64, 0};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tbase + TM_X, sdesc(sbase + OFF_UT + aoff[ps] + kk * 2 * 2048, 2048),
                                 sdesc(s2 + P2_KH + boff[ps] + kk * 256, 128, 1024), id128, 1);
                commit(mbar);
            }
        }
        if (!ok) {   // a wait gave up: record it and let the staged copies land (bounded waits)
            atomicExch(&g_state_status, KDA_ERR_TIMEOUT);
            if (n_p1) mbar_wait(pbar1, (n_p1 - 1) & 1);
            for (int b = 0; b < 2; ++b)
                if (n_p2[b]) mbar_wait(smem_u32(&s_pbar2[b]), (n_p2[b] - 1) & 1);
        }
    }

    // ---- piece end: summaries and final states (X[k][c] from TMEM lane c, column k)
    if (worker && !aborted) {
        const size_t mat = static_cast<size_t>(KD) * VD;
        const bool seg_last = flags & KDA_PIECE_SEG_LAST, seq_end = flags & KDA_PIECE_SEQ_END;
        float *dst0 = nullptr, *dst1 = nullptr;
        if (kind == 0) {
            if (seg_last) dst0 = B + (static_cast<size_t>(seg) * H + h) * mat;
            if (seq_end) dst1 = fin_state + (static_cast<size_t>(seq) * H + h) * mat;
            if (seg_last && (pv.seg(seg)[1] & KDA_SEG_HAS_RESET)) {
                float *za = A + (static_cast<size_t>(seg) * H + h) * KD * KD;
                for (int e = tid; e < KD * KD / 4; e += NWORK)
                    reinterpret_cast<float4 *>(za)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        } else {
            if (seg_last) dst0 = A + (static_cast<size_t>(seg) * H + h) * KD * KD;
            if (seq_end) dst1 = afin + (static_cast<size_t>(fin) * H + h) * KD * KD;
        }
        if (dst0 || dst1) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int k0 = hw * 64 + half * 32;
                float x[32];
                tmem_ld32(tl + TM_X + k0, x);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (dst0) dst0[(k0 + j) * VD + c_lane] = x[j];
                    if (dst1) dst1[(k0 + j) * VD + c_lane] = x[j];
                }
            }
        }
    } else if (worker && tid == 0) {
        atomicExch(&g_state_status, KDA_ERR_TIMEOUT);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

cudaError_t launch_chunk_state(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *h0,
                               const unsigned char *pkg, uint16_t *o, float *A, float *B, float *final_state,
                               uint16_t *qhat, float *afin, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    const long long blocks = static_cast<long long>(pv.n_items()) * H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t err = cudaFuncSetAttribute(chunk_state_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(SMEM_BYTES));
    if (err != cudaSuccess) return err;
    chunk_state_tc<<<static_cast<unsigned>(blocks), NTHREADS, SMEM_BYTES, stream>>>(plan_dev, H, h0, pkg, o, A, B,
                                                                                    final_state, qhat, afin);
    return cudaGetLastError();
}

// The local chunkwise forward: the chunk-parallel preparation, then the serial state pass.
cudaError_t launch_chunk_forward(const int32_t *plan_host, const int32_t *plan_dev, int H,
                                 const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const float *g, const float *beta, const float *h0, float scale,
                                 uint16_t *o, float *A, float *B, float *final_state,
                                 uint16_t *qhat, float *afin, unsigned char *pkg, cudaStream_t stream)
{
    cudaError_t err = launch_chunk_prep(plan_host, plan_dev, H, q, k, v, g, beta, scale, pkg, stream);
    if (err != cudaSuccess) return err;
    return launch_chunk_state(plan_host, plan_dev, H, h0, pkg, o, A, B, final_state, qhat, afin, stream);
}

}  // namespace kda
