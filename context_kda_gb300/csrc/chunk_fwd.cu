// Chunkwise KDA forward of one piece (segment x sequence) on the tcgen05 tensor
// cores, with the segment summaries: state columns (outputs, state update B,
// final states) and transition columns (qhat, transition A).
//
// Algebra (per chunk of C = 64 rows, Gamma_r = cumulative g within the chunk):
//   kt_r = exp(Gamma_r) k_r, kh_i = exp(-Gamma_i) k_i, qt_r = scale exp(Gamma_r) q_r,
//   M[r,i] = beta_r (kt_r . kh_i) for i < r,   T' = (I + M)^-1 Diag(beta),
//   Ut = T' V,   U = Ut - T' (Kt X)   (= Ut - W X with W = T' Kt),
//   O = Qt X + ((Qt Kh^T) masked to i <= r) U,
//   X' = Diag(exp Gamma_C) (X + Kh^T U)   (= Diag(exp Gamma_C) X + Kb^T U with
//        kb_i = exp(Gamma_C - Gamma_i) k_i).
// This is the KDA gated delta rule (cuLA PR #110, "feat(cp): add opt-in NVSHMEM
// CP state handoff", §Supported configuration: BF16 inputs, FP32 state) unrolled
// over a chunk: writing u_r = beta_r (v_r - (Diag(exp g_r) X_{r-1})^T k_r) for
// every row gives (I + M) U = Diag(beta) (V - Kt X).
//
// The transition columns run the same recurrence on P (K x K) with zero values
// from P = I at the piece start, so their 'outputs' are qhat_t = scale P_t^T q_t
// and their end state is the piece's transition (cuLA PR #136, "feat(kda): add
// cuDNN concatenated-summary Kimi CP", §Summary: preceding_transition).
//
// Mapping.  One CTA per (work item, head): 256 threads, 128 state columns c.
// The state lives transposed in TMEM (lane c, column k) as an FP32 accumulator;
// every contraction is a tcgen05.mma (M = 128, bf16 operands in shared memory,
// FP32 accumulation in TMEM).  Operand tiles are written row by row with
// 16-byte stores; the transposed operands (Kt^T, Kb^T, V^T, W) are the same
// row-major tiles read MN-major.  The contractions that feed the state and the
// summaries (Kt Kh^T, Kt X, Ut, T' (Kt X), Kh^T U) use a three-term bf16 split
// (hi*hi + hi*lo + lo*hi, ~2^-17 relative per product) so the FP32 state and
// summaries stay within 1e-4; the output-only ones (Qt X, masked QK U) use one
// term.  The 64 x 64 unit-triangular inverse is solved on the CUDA cores in
// FP32 (16 x 16 blocks) while the tensor core forms Qt X and Kt X from the
// chunk-start state (issued by a warp the inverse leaves idle).  Each chunk's raw rows are staged in shared memory
// by tiled TMA loads (128-byte swizzle) issued while the previous chunk finishes.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

// ---- shared-memory map (bytes from the 16-byte aligned dynamic base) ------------------------
// Tiles are bf16, hi and lo halves back to back; CS = chunk-column stride (see tc.cuh).
constexpr uint32_t OFF_XT = 0;        // X^T: rows c (128), cols k (128), CS 2048           2 x 32768
constexpr uint32_t OFF_KQ = 65536;    // [Kt; Qt]: rows r / 64 + r, cols k, CS 2048          2 x 32768
constexpr uint32_t OFF_MT = 131072;   // M (fp32 64 x 64) + T (fp32 64 x 64, at +16384); then -(Kt X)^T:
//   rows c (128), cols i (64), CS 2048                                                   2 x 16384
constexpr uint32_t OFF_KH = 163840;   // Kh: rows i (64), cols k, CS 1024                    2 x 16384
constexpr uint32_t OFF_VT = 196608;   // V: rows r (64), cols v, CS 1024 (16384) + T': rows r, cols i,
//   CS 1024 (2 x 8192 at +16384); then U^T: rows c (128), cols r (64), CS 2048          2 x 16384
constexpr uint32_t OFF_MISC = 229376;
constexpr uint32_t OFF_BETA = OFF_MISC;         // 64 fp32
constexpr uint32_t OFF_GC = OFF_MISC + 256;     // 128 fp32: exp(Gamma_C)
constexpr uint32_t OFF_GSUM = OFF_MISC + 768;   // 2 x 128 fp32: per-half decay sums
constexpr uint32_t SMEM_BYTES = OFF_MISC + 1792;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;   // room to align the base to 1024 bytes
constexpr uint32_t T128 = 32768, T64 = 16384;
constexpr uint32_t OFF_M32 = OFF_MT, OFF_T32 = OFF_MT + 16384;
constexpr uint32_t OFF_TP = OFF_VT + 16384;          // T' hi | lo (8192 each)
constexpr uint32_t OFF_QKL = OFF_KQ + T128 + 1024;   // masked QK (bf16) in the Qt rows of the lo tile
constexpr uint32_t OFF_QT_HI = OFF_KQ + 1024;        // Qt rows of the hi tile
// Raw rows of the next chunk, loaded by tiled TMA copies (128-byte swizzle, 1024-aligned boxes of
// 64 rows x 128 bytes): q, k, v as two 64-column boxes each, g as four 32-column boxes.
constexpr uint32_t BOX = 8192;
constexpr uint32_t STG_Q = OFF_KQ, STG_K = OFF_KQ + 2 * BOX, STG_V = OFF_KQ + 4 * BOX, STG_G = OFF_MT;

// ---- TMEM columns --------------------------------------------------------------------------
constexpr uint32_t TM_D1 = 0;     // [KK; QK] (64 cols)
constexpr uint32_t TM_KX = 64;    // (Kt X)^T
constexpr uint32_t TM_U = 128;    // Ut^T, then U^T
constexpr uint32_t TM_O = 192;    // O^T (64 cols)
constexpr uint32_t TM_X = 256;    // X^T (128 cols)
constexpr uint32_t TM_COLS = 512;

constexpr float LOG2E = 1.4426950408889634f;

__device__ int g_chunk_status;   // set to KDA_ERR_TIMEOUT when a bounded wait expires

// fp32 64 x 64 scratch with the 16-byte chunk index XOR-swizzled by the row
__device__ __forceinline__ float *f32_at(unsigned char *base, uint32_t off, int r, int i)
{
    return reinterpret_cast<float *>(base + off + r * 256 + (((i >> 2) ^ (r & 15)) << 4) + (i & 3) * 4);
}


// Writes 8 consecutive values as bf16 hi and lo (two 16-byte stores).
__device__ __forceinline__ void st_split8(unsigned char *hi, unsigned char *lo, const float *x)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) split_bf16x2(x[2 * p], x[2 * p + 1], h[p], l[p]);
    *reinterpret_cast<uint4 *>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 w, float *x)
{
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        x[2 * p] = __uint_as_float(ww[p] << 16);
        x[2 * p + 1] = __uint_as_float(ww[p] & 0xFFFF0000u);
    }
}

constexpr int NWORK = 256;        // worker threads (8 warps): operands, inverse, epilogues
constexpr int NTHREADS = NWORK + 32;   // plus one warp whose lane 0 issues every MMA and TMA load
constexpr int ISSUER = NWORK;
enum { HO_A = 0, HO_D = 1, HO_E = 2, HO_H = 3 };   // worker -> issuer handoffs of a chunk

__global__ void __launch_bounds__(NTHREADS, 1)
chunk_forward_tc(const int32_t *__restrict__ plan, int H, const uint16_t *__restrict__ q,
                 const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                 const float *__restrict__ g, const float *__restrict__ beta,
                 const float *__restrict__ h0, float scale, uint16_t *__restrict__ o,
                 float *__restrict__ A, float *__restrict__ B, float *__restrict__ fin_state,
                 float *__restrict__ qhat, float *__restrict__ afin,
                 const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_mbar;
    __shared__ __align__(8) uint64_t s_ldbar;
    __shared__ __align__(8) uint64_t s_mbar2;
    __shared__ __align__(8) uint64_t s_hbar[4];
    __shared__ uint32_t s_tmem;
    unsigned char *const base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(base);
    float *const s_beta = reinterpret_cast<float *>(base + OFF_BETA);
    float *const s_gc = reinterpret_cast<float *>(base + OFF_GC);
    float *const s_gsum = reinterpret_cast<float *>(base + OFF_GSUM);

    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;          // TMEM lane quadrant, column half
    const int item = blockIdx.x / H, h = blockIdx.x % H;
    const int32_t *it = pv.item(item);
    const int p = it[0], kind = it[1];
    const int32_t *pc = pv.piece(p);
    const int start = pc[PC_START], len = pc[PC_LEN], seq = pc[PC_SEQ], seg = pc[PC_SEG];
    const int flags = pc[PC_FLAGS], row0 = pc[PC_ROW], fin = pc[PC_FIN];
    const int64_t T_cont = pv.T_cont();
    const uint32_t mbar = smem_u32(&s_mbar);
    const uint32_t ldbar = smem_u32(&s_ldbar);
    const uint32_t mbar2 = smem_u32(&s_mbar2);   // the state products issued with [KK; QK]
    const bool worker = tid < NWORK, issuer = tid == ISSUER;

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(ldbar, 1);
        mbar_init(mbar2, 1);
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&s_hbar[i]), 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);  // this warp's lane quadrant
    const int c_lane = quad * 32 + lane;                                     // state column of this thread
    uint32_t phase = 0, phase2 = 0;
    bool aborted = false;   // all workers agree on it (OR-reduced at barriers)
    bool bad = false;       // a bounded wait of this thread gave up

    auto wait_mma = [&]() {
        if (!mbar_wait(mbar, phase & 1)) bad = true;
        ++phase;
        fence_after();
    };

    // Stage the raw rows of chunk cn (q, k, g, and v for state columns) with tiled TMA copies
    // issued by the issuer thread; rows past the end of the tensor arrive as zeros, rows past the
    // piece are masked when read.  beta of that chunk goes to a register of the first 64 workers.
    uint32_t ld_phase = 0;
    float beta_next = 0.f;
    auto issue_tma = [&](int cn) {
        const int t0n = start + cn * CH;
        mbar_arrive_expect_tx(ldbar, (kind == 0 ? 6u : 4u) * BOX + 4u * BOX);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(sbase + STG_Q + half * BOX, &tm_q, half * 64, h, t0n, ldbar);
            tma_load_3d(sbase + STG_K + half * BOX, &tm_k, half * 64, h, t0n, ldbar);
            if (kind == 0) tma_load_3d(sbase + STG_V + half * BOX, &tm_v, half * 64, h, t0n, ldbar);
        }
#pragma unroll
        for (int qtr = 0; qtr < 4; ++qtr) tma_load_3d(sbase + STG_G + qtr * BOX, &tm_g, qtr * 32, h, t0n, ldbar);
    };
    auto load_beta = [&](int cn) {
        const int t0n = start + cn * CH;
        const int Ln = min(CH, len - cn * CH);
        if (tid < 64) beta_next = (tid < Ln) ? beta[static_cast<size_t>(t0n + tid) * H + h] : 0.f;
    };
    if (issuer) issue_tma(0);
    load_beta(0);

    // ---- piece start: X^T into TMEM (fp32) and its bf16 split into shared memory
    if (worker) {
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
        fence_before();
        fence_async_smem();
    }
    __syncthreads();

    // ---- MMA groups, issued by the issuer thread once the workers hand the operands over.
    // [KK; QK] = [Kt; Qt] Kh^T (3-term) -> mbar
    auto mma_kkqk = [&]() {
        const uint32_t id = idesc_bf16(128, 64);
        const uint32_t aoff[3] = {0, 0, T128}, boff[3] = {0, T64, 0};
#pragma unroll
        for (int ps = 0; ps < 3; ++ps)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tbase + TM_D1, sdesc(sbase + OFF_KQ + aoff[ps] + kk * 2 * 2048, 2048),
                         sdesc(sbase + OFF_KH + boff[ps] + kk * 2 * 1024, 1024), id, (ps | kk) != 0);
        commit(mbar);
    };
    // O^T = X^T Qt^T (1-term) and (Kt X)^T = X^T Kt^T (3-term): only the chunk-start state and the
    // decayed rows, so they run while the workers solve the inverse -> mbar2
    auto mma_state = [&]() {
        const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tbase + TM_O, sdesc(sbase + OFF_XT + kk * 2 * 2048, 2048),
                     sdesc(sbase + OFF_QT_HI + kk * 2 * 2048, 2048), id, kk != 0);
        const uint32_t xoff[3] = {0, 0, T128}, toff[3] = {0, T128, 0};
#pragma unroll
        for (int ps = 0; ps < 3; ++ps)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tbase + TM_KX, sdesc(sbase + OFF_XT + xoff[ps] + kk * 2 * 2048, 2048),
                         sdesc(sbase + OFF_KQ + toff[ps] + kk * 2 * 2048, 2048), id, (ps | kk) != 0);
        commit(mbar2);
    };
    // Ut^T = V^T T'^T (2-term; V^T is the row-major V tile read MN-major), state columns only
    auto mma_ut = [&]() {
        const uint32_t id = idesc_bf16(128, 64, 1, 0);
#pragma unroll
        for (int ps = 0; ps < 2; ++ps)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tbase + TM_U, sdesc(sbase + OFF_VT + kk * 256, 128, 1024),
                         sdesc(sbase + OFF_TP + ps * 8192 + kk * 2 * 1024, 1024), id, (ps | kk) != 0);
    };
    // U^T (+)= -(Kt X)^T T'^T (3-term) -> mbar
    auto mma_u = [&]() {
        const uint32_t id = idesc_bf16(128, 64);
        const uint32_t aoff[3] = {0, 0, T64}, boff[3] = {0, 8192, 0};
#pragma unroll
        for (int ps = 0; ps < 3; ++ps)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tbase + TM_U, sdesc(sbase + OFF_MT + aoff[ps] + kk * 2 * 2048, 2048),
                         sdesc(sbase + OFF_TP + boff[ps] + kk * 2 * 1024, 1024), id, (kind == 0) || ((ps | kk) != 0));
        commit(mbar);
    };
    // O^T += U^T QK^T (1-term); X^T += U^T Kh (3-term, Kh read MN-major) -> mbar
    auto mma_out = [&]() {
        const uint32_t id64 = idesc_bf16(128, 64), id128 = idesc_bf16(128, 128, 0, 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tbase + TM_O, sdesc(sbase + OFF_VT + kk * 2 * 2048, 2048),
                     sdesc(sbase + OFF_QKL + kk * 2 * 2048, 2048), id64, 1);
        const uint32_t aoff[3] = {0, 0, T64}, boff[3] = {0, T64, 0};
#pragma unroll
        for (int ps = 0; ps < 3; ++ps)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tbase + TM_X, sdesc(sbase + OFF_VT + aoff[ps] + kk * 2 * 2048, 2048),
                         sdesc(sbase + OFF_KH + boff[ps] + kk * 256, 128, 1024), id128, 1);
        commit(mbar);
    };
    // Workers hand a set of shared-memory operands over to the issuer: every writer fences its
    // generic-proxy stores for the tensor core, the workers meet, and one of them arrives.
    // Returns true when some worker's wait gave up (then nothing is handed over).
    auto handoff = [&](int which) -> bool {
        fence_async_smem();
        fence_before();
        const bool ab = bar_or1(NWORK, bad);
        if (!ab && tid == 0) mbar_arrive(smem_u32(&s_hbar[which]));
        return ab;
    };

    const int nch = (len + CH - 1) / CH;
    if (worker) {
        for (int ci = 0; ci < nch && !aborted; ++ci) {
            const int t0 = start + ci * CH;
            const int L = min(CH, len - ci * CH);

            // ================= A: staged rows -> decayed keys / queries / values in operand tiles =====
            {
                if (!mbar_wait(ldbar, ld_phase & 1)) bad = true;
                ++ld_phase;
                // A1: log2-scaled cumulative decay per key channel, in place over the staged g
                //     (32 rows per thread: load all, scan in registers, store once)
                {
                    const int kc = tid & 127, hr = tid >> 7;
                    unsigned char *gq = base + STG_G + (kc >> 5) * BOX + (kc & 3) * 4;
                    const int gch = (kc & 31) >> 2;
                    float gv[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) gv[j] = *reinterpret_cast<const float *>(gq + sw128(hr * 32 + j, gch));
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        acc += (hr * 32 + j < L) ? gv[j] * LOG2E : 0.f;
                        gv[j] = acc;
                    }
                    s_gsum[hr * 128 + kc] = acc;
                    if (tid < 64) s_beta[tid] = beta_next;
                    bar_sync1(NWORK);
                    const float off = hr ? s_gsum[kc] : 0.f;
                    if (hr == 0) s_gc[kc] = ex2_ftz(s_gsum[kc] + s_gsum[128 + kc]);   // exp(Gamma_C)
#pragma unroll
                    for (int j = 0; j < 32; ++j) *reinterpret_cast<float *>(gq + sw128(hr * 32 + j, gch)) = gv[j] + off;
                    bar_sync1(NWORK);
                }
                // A2: each thread takes four (row, 8-column) pieces of the staged rows into registers;
                //     the lanes of a warp hold consecutive rows of one piece column
                const int pr = tid & 63, pcg = tid >> 6;
                float gam[4][8];
                uint4 kw[4], qw[4], vw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = pr, c8 = (pcg + 4 * i) * 8;
                    const unsigned char *gb = base + STG_G + (c8 >> 5) * BOX;
                    const int gch = (c8 & 31) >> 2;
                    const float4 a = *reinterpret_cast<const float4 *>(gb + sw128(r, gch));
                    const float4 b = *reinterpret_cast<const float4 *>(gb + sw128(r, gch + 1));
                    gam[i][0] = a.x; gam[i][1] = a.y; gam[i][2] = a.z; gam[i][3] = a.w;
                    gam[i][4] = b.x; gam[i][5] = b.y; gam[i][6] = b.z; gam[i][7] = b.w;
                    const bool ok = r < L;
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t bo = (c8 >> 6) * BOX + sw128(r, (c8 & 63) >> 3);
                    kw[i] = ok ? *reinterpret_cast<const uint4 *>(base + STG_K + bo) : z;
                    qw[i] = ok ? *reinterpret_cast<const uint4 *>(base + STG_Q + bo) : z;
                    vw[i] = (ok && kind == 0) ? *reinterpret_cast<const uint4 *>(base + STG_V + bo) : z;
                }
                bar_sync1(NWORK);   // staging consumed: every region may be rewritten from here
                // A3: Kt, Qt (stacked), Kh as bf16 hi/lo and V as bf16, one row piece at a time
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = pr, c8 = (pcg + 4 * i) * 8;
                    float kf[8], qf[8], kt[8], qt[8], kh[8];
                    bf16x8_to_f32(kw[i], kf);
                    bf16x8_to_f32(qw[i], qf);
#pragma unroll
                    for (int e8 = 0; e8 < 8; ++e8) {
                        const float G = gam[i][e8];
                        const float e = ex2_ftz(G), ei = ex2_ftz(-G);
                        kt[e8] = e * kf[e8];
                        qt[e8] = scale * e * qf[e8];
                        kh[e8] = ei * kf[e8];
                    }
                    const uint32_t o_r = cm_off(r, c8, 2048), o_q = cm_off(64 + r, c8, 2048), o_64 = cm_off(r, c8, 1024);
                    st_split8(base + OFF_KQ + o_r, base + OFF_KQ + T128 + o_r, kt);
                    st_split8(base + OFF_KQ + o_q, base + OFF_KQ + T128 + o_q, qt);
                    st_split8(base + OFF_KH + o_64, base + OFF_KH + T64 + o_64, kh);
                    if (kind == 0) *reinterpret_cast<uint4 *>(base + OFF_VT + o_64) = vw[i];
                }
                aborted = handoff(HO_A);   // -> [KK; QK], then Qt X and Kt X
            }
            if (aborted) break;

            // ================= B: [KK; QK] = [Kt; Qt] Kh^T  (3-term split) =================
            wait_mma();

            // ================= C: M (fp32, beta-scaled, strictly lower) and masked QK (bf16) =====
            {
                float d[32];
                tmem_ld32(tl + TM_D1 + hw * 32, d);
                if (quad < 2) {
                    const int r = c_lane;
                    const float br = s_beta[r];
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        float4 m4;
                        const int i0 = hw * 32 + 4 * j4;
                        m4.x = (i0 + 0 < r) ? br * d[4 * j4 + 0] : 0.f;
                        m4.y = (i0 + 1 < r) ? br * d[4 * j4 + 1] : 0.f;
                        m4.z = (i0 + 2 < r) ? br * d[4 * j4 + 2] : 0.f;
                        m4.w = (i0 + 3 < r) ? br * d[4 * j4 + 3] : 0.f;
                        *reinterpret_cast<float4 *>(f32_at(base, OFF_M32, r, i0)) = m4;
                    }
                } else {
                    const int r = c_lane - 64;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        uint32_t w[4];
#pragma unroll
                        for (int p2 = 0; p2 < 4; ++p2) {
                            const int i0 = hw * 32 + 8 * m + 2 * p2;
                            w[p2] = bf16x2_bits(i0 <= r ? d[8 * m + 2 * p2] : 0.f, i0 + 1 <= r ? d[8 * m + 2 * p2 + 1] : 0.f);
                        }
                        *reinterpret_cast<uint4 *>(base + OFF_QKL + cm_off(r, hw * 32 + 8 * m, 2048)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                fence_before();
                aborted = bar_or1(NWORK, bad);
            }
            if (aborted) break;

            // ================= D: T = (I + M)^-1 in 16 x 16 blocks (fp32, CUDA cores) =========
            // Diagonal blocks t_b by forward substitution; then each 32 x 32 half as
            // [t_0 0; -t_1 M_10 t_0  t_1], and the whole as [T_lo 0; -T_hi M_hi,lo T_lo  T_hi].
            {
                if (tid < 64) {   // column jj of diagonal block b; each solved entry updates all later rows
                    const int b = tid >> 4, jj = tid & 15, r0 = 16 * b;
                    float x[16], sacc[16];
#pragma unroll
                    for (int rr = 0; rr < 16; ++rr) sacc[rr] = 0.f;
#pragma unroll
                    for (int rr = 0; rr < 16; ++rr) {
                        x[rr] = (rr == jj) ? 1.f : ((rr < jj) ? 0.f : -sacc[rr]);
#pragma unroll
                        for (int r2 = rr + 1; r2 < 16; ++r2)
                            sacc[r2] = fmaf(*f32_at(base, OFF_M32, r0 + r2, r0 + rr), x[rr], sacc[r2]);
                    }
#pragma unroll
                    for (int rr = 0; rr < 16; ++rr) *f32_at(base, OFF_T32, r0 + rr, r0 + jj) = x[rr];
                }
                bar_sync1(NWORK);
                // Thread -> group g of 64 (one 16 x 16 output block), row rr, four adjacent columns c4..c4+3.
                // Intermediate products Y_ij go to the unused upper-triangle block (j, i) of M.
                const int g = tid >> 6, rr = (tid >> 2) & 15, c4 = (tid & 3) * 4;
                // y += A[ar + rr][ac + 0..15] * B[br + 0..15][bc + c4 .. c4 + 3]
                auto blk_fma = [&](float4 &y, uint32_t offa, int ar, int ac, uint32_t offb, int br, int bc) {
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {
                        const float4 av = *reinterpret_cast<const float4 *>(f32_at(base, offa, ar + rr, ac + 4 * m4));
                        const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float4 bv =
                                *reinterpret_cast<const float4 *>(f32_at(base, offb, br + 4 * m4 + e, bc + c4));
                            y.x = fmaf(aa[e], bv.x, y.x);
                            y.y = fmaf(aa[e], bv.y, y.y);
                            y.z = fmaf(aa[e], bv.z, y.z);
                            y.w = fmaf(aa[e], bv.w, y.w);
                        }
                    }
                };
                const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
                // halves: Y_10 = M_10 t_0, Y_32 = M_32 t_2 (groups 0, 1), then T_10, T_32 = -t_i Y
                if (g < 2) {
                    const int i = 1 + 2 * g, j = 2 * g;
                    float4 y = z4;
                    blk_fma(y, OFF_M32, 16 * i, 16 * j, OFF_T32, 16 * j, 16 * j);
                    *reinterpret_cast<float4 *>(f32_at(base, OFF_M32, 16 * j + rr, 16 * i + c4)) = y;
                }
                bar_sync1(NWORK);
                if (g < 2) {
                    const int i = 1 + 2 * g, j = 2 * g;
                    float4 t = z4;
                    blk_fma(t, OFF_T32, 16 * i, 16 * i, OFF_M32, 16 * j, 16 * i);
                    *reinterpret_cast<float4 *>(f32_at(base, OFF_T32, 16 * i + rr, 16 * j + c4)) =
                        make_float4(-t.x, -t.y, -t.z, -t.w);
                }
                bar_sync1(NWORK);
                // whole: Y_ij = sum_{k=j..1} M_ik T_kj, then T_ij = -sum_{k=2..i} T_ik Y_kj (i = 2, 3; j = 0, 1)
                {
                    const int i = 2 + (g >> 1), j = g & 1;
                    float4 y = z4;
                    blk_fma(y, OFF_M32, 16 * i, 16 * j, OFF_T32, 16 * j, 16 * j);
                    if (j == 0) blk_fma(y, OFF_M32, 16 * i, 16, OFF_T32, 16, 0);
                    *reinterpret_cast<float4 *>(f32_at(base, OFF_M32, 16 * j + rr, 16 * i + c4)) = y;
                    bar_sync1(NWORK);
                    float4 t = z4;
                    blk_fma(t, OFF_T32, 16 * i, 32, OFF_M32, 16 * j, 32);
                    if (i == 3) blk_fma(t, OFF_T32, 48, 48, OFF_M32, 16 * j, 48);
                    *reinterpret_cast<float4 *>(f32_at(base, OFF_T32, 16 * i + rr, 16 * j + c4)) =
                        make_float4(-t.x, -t.y, -t.z, -t.w);
                    bar_sync1(NWORK);
                }
                // T' = T Diag(beta) as bf16 hi/lo (rows r, cols i), zero above the diagonal
                {
                    // lanes: 8 consecutive rows x four 16-column groups (conflict-free row-piece reads)
                    const int r = ((tid >> 5) << 3) | (tid & 7), i0 = ((tid >> 3) & 3) * 16;
                    float tv[16];
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {
                        const float4 t4 = *reinterpret_cast<const float4 *>(f32_at(base, OFF_T32, r, i0 + 4 * m4));
                        const float tt[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = i0 + 4 * m4 + e;
                            tv[4 * m4 + e] = (i <= r) ? tt[e] * s_beta[i] : 0.f;
                        }
                    }
                    st_split8(base + OFF_TP + cm_off(r, i0, 1024), base + OFF_TP + 8192 + cm_off(r, i0, 1024), tv);
                    st_split8(base + OFF_TP + cm_off(r, i0 + 8, 1024), base + OFF_TP + 8192 + cm_off(r, i0 + 8, 1024),
                              tv + 8);
                }
                aborted = handoff(HO_D);   // -> Ut^T = V^T T'^T
            }
            if (aborted) break;

            // ================= E: U^T = Ut^T - (Kt X)^T T'^T; Ut^T = V^T T'^T (2-term, V^T the row-major
            //                     V tile read MN-major), the product term 3-term from -(Kt X)^T in smem
            {
                if (!mbar_wait(mbar2, phase2 & 1)) bad = true;
                ++phase2;
                fence_after();
                float d[32];
                tmem_ld32(tl + TM_KX + hw * 32, d);   // (Kt X)^T[c = c_lane][i = hw*32 + j]
#pragma unroll
                for (int j = 0; j < 32; ++j) d[j] = -d[j];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t off = cm_off(c_lane, hw * 32 + 8 * m, 2048);
                    st_split8(base + OFF_MT + off, base + OFF_MT + T64 + off, d + 8 * m);
                }
                aborted = handoff(HO_E);   // -> U^T += -(Kt X)^T T'^T
            }
            if (aborted) break;
            wait_mma();

            // ================= H: U^T (rows c, cols r) hi/lo into shared memory ====================
            {
                float d[32];
                tmem_ld32(tl + TM_U + hw * 32, d);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t off = cm_off(c_lane, hw * 32 + 8 * m, 2048);
                    st_split8(base + OFF_VT + off, base + OFF_VT + T64 + off, d + 8 * m);
                }
                aborted = handoff(HO_H);   // -> O^T += U^T QK^T, X^T += U^T Kh
            }
            if (aborted) break;

            // ================= I: O^T += U^T QK^T (1-term); X^T += U^T Kh (3-term, Kh read MN-major) ==
            wait_mma();

            // ================= J: outputs (or qhat) to HBM; new X^T split into shared memory ========
            if (ci + 1 < nch) load_beta(ci + 1);   // the issuer stages the rows once I has completed
            {
                // O^T[c][r] -> row-major O tile in the free V/U region, then 16-byte coalesced stores;
                // the state half X^T[c][hw*64 .. +64) is read in the same batch
                uint32_t od[32], xa[32], xb[32];
                tmem_ld32_nowait(tl + TM_O + hw * 32, od);   // O^T[c][r = hw*32 + j]
                tmem_ld32_nowait(tl + TM_X + hw * 64, xa);
                tmem_ld32_nowait(tl + TM_X + hw * 64 + 32, xb);
                tmem_wait_ld();
                reg_fence32(od);
                reg_fence32(xa);
                reg_fence32(xb);
                float d[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) d[j] = __uint_as_float(od[j]);
                if (kind == 0) {
                    uint16_t *so = reinterpret_cast<uint16_t *>(base + OFF_VT);
#pragma unroll
                    for (int j = 0; j < 32; ++j) so[(hw * 32 + j) * 128 + c_lane] = f32_to_bf16_bits(d[j]);
                } else {
                    float *so = reinterpret_cast<float *>(base + OFF_VT);
#pragma unroll
                    for (int j = 0; j < 32; ++j) so[(hw * 32 + j) * 128 + c_lane] = d[j];
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int k0 = hw * 64 + half * 32;
                    float x[32];   // X + Kh^T U, then Diag(exp Gamma_C)
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(half ? xb[j] : xa[j]) * s_gc[k0 + j];
                    tmem_st32(tl + TM_X + k0, x);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        st_split8(base + OFF_XT + cm_off(c_lane, k0 + 8 * m, 2048),
                                  base + OFF_XT + T128 + cm_off(c_lane, k0 + 8 * m, 2048), x + 8 * m);
                }
                fence_before();
                fence_async_smem();
                aborted = bar_or1(NWORK, bad);
                if (kind == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int id = tid + 256 * i, r = id >> 4, c16 = id & 15;
                        if (r < L)
                            *reinterpret_cast<uint4 *>(o + (static_cast<size_t>(t0 + r) * H + h) * VD + c16 * 8) =
                                *reinterpret_cast<const uint4 *>(base + OFF_VT + r * 256 + c16 * 16);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int id = tid + 256 * i, r = id >> 5, c32 = id & 31;
                        if (r < L)
                            *reinterpret_cast<uint4 *>(qhat + (static_cast<size_t>(h) * T_cont + row0 + ci * CH + r) * KD +
                                                       c32 * 4) =
                                *reinterpret_cast<const uint4 *>(base + OFF_VT + r * 512 + c32 * 16);
                    }
                }
            }
        }
    } else if (issuer) {
        // Issuer: for each chunk, wait for the workers' handoffs and issue the MMA groups; stage the
        // next chunk's rows once the output products (the last readers of the staging regions) finish.
        bool ok = true;
        int last_tma = 0;
        for (int ci = 0; ci < nch && ok; ++ci) {
            const uint32_t par = ci & 1;
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_A]), par))) break;
            fence_after();
            mma_kkqk();
            mma_state();
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_D]), par))) break;
            fence_after();
            if (kind == 0) mma_ut();
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_E]), par))) break;
            fence_after();
            mma_u();
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_H]), par))) break;
            fence_after();
            mma_out();
            if (ci + 1 < nch) {
                // mbar phases per chunk: [KK; QK], U, outputs; the last is the one pending now
                if (!(ok = mbar_wait(mbar, (3 * ci + 2) & 1))) break;
                issue_tma(ci + 1);
                last_tma = ci + 1;
            }
        }
        if (!ok) {
            atomicExch(&g_chunk_status, KDA_ERR_TIMEOUT);
            mbar_wait(ldbar, last_tma & 1);   // bounded: let the last staged copy land
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
                for (int e = tid; e < KD * KD / 4; e += 256)
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
        atomicExch(&g_chunk_status, KDA_ERR_TIMEOUT);
    }
    fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

namespace {

// [T][H][128] tensor as a 3-D map (inner dim first) with a box of 'inner' x 1 x 64 rows.
bool encode_rows(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, uint32_t elem, int H, int T,
                 uint32_t inner)
{
    auto fn = tmap_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {128ull * elem, 128ull * elem * static_cast<cuuint64_t>(H)};
    const cuuint32_t box[3] = {inner, 1, 64};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_forward(const int32_t *plan_host, const int32_t *plan_dev, int H,
                                 const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const float *g, const float *beta, const float *h0, float scale,
                                 uint16_t *o, float *A, float *B, float *final_state,
                                 float *qhat, float *afin, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    const long long blocks = static_cast<long long>(pv.n_items()) * H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap tq, tk, tv, tg;
    const int T = pv.T();
    if (!encode_rows(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64) ||
        !encode_rows(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64) ||
        !encode_rows(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64) ||
        !encode_rows(&tg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, T, 32))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(chunk_forward_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(SMEM_ALLOC));
    if (err != cudaSuccess) return err;
    chunk_forward_tc<<<static_cast<unsigned>(blocks), NTHREADS, SMEM_ALLOC, stream>>>(
        plan_dev, H, q, k, v, g, beta, h0, scale, o, A, B, final_state, qhat, afin, tq, tk, tv, tg);
    return cudaGetLastError();
}

}  // namespace kda
