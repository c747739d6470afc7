// Chunk-parallel preparation of the chunkwise KDA forward: everything about a 64-token chunk of
// one head that does not depend on the state entering it.
//
// Algebra (per chunk of C = 64 rows, Gamma_r = cumulative g within the chunk):
//   kt_r = exp(Gamma_r) k_r, kh_i = exp(-Gamma_i) k_i, qt_r = scale exp(Gamma_r) q_r,
//   M[r,i] = beta_r (kt_r . kh_i) for i < r,   T' = (I + M)^-1 Diag(beta),
//   W = T' Kt,   Ut = T' V,   QK = (Qt Kh^T) masked to i <= r.
// The state pass then needs only these: with X the chunk-start state,
//   U = Ut - W X,   O = Qt X + QK U,   X' = Diag(exp Gamma_C) (X + Kh^T U).
// This is the KDA gated delta rule (cuLA PR #110, "feat(cp): add opt-in NVSHMEM CP state
// handoff", §Supported configuration: BF16 inputs, FP32 state) unrolled over a chunk: writing
// u_r = beta_r (v_r - (Diag(exp g_r) X_{r-1})^T k_r) for every row gives (I + M) U = Diag(beta)
// (V - Kt X).  The intra-chunk transform runs once per (chunk, head) here, on all SMs, instead
// of once per piece column set inside the serial pass.
//
// Mapping.  A persistent CTA per SM walks (chunk, head) units: 8 worker warps build the operand
// tiles and solve the inverse on the CUDA cores; lane 0 of a ninth warp issues the tcgen05 MMAs
// (M = 128, bf16 operands in shared memory, FP32 accumulators in TMEM) and lane 0 of a tenth the
// TMA loads that stage the next unit's rows.  The products that feed the state (Kt Kh^T, W) use a three-term
// bf16 split (hi*hi + hi*lo + lo*hi, ~2^-17 relative); Ut two terms (V is exact in bf16); Qt Kh^T, an
// output product, two (Qt's low part is zero).
// Results go straight from registers to the unit's package in the workspace with 16-byte
// stores, each tile already in the layout the state pass's MMAs read.  A unit's W and Ut products
// run while the workers start the next unit; the workers read W back from TMEM and store it while
// they wait for the next unit's [KK; QK], and four warps store Ut while two solve the next
// unit's diagonal blocks.
//
// Backward mode (BWD): the same pass also leaves what the backward reads of each unit, in the layouts
// its kernels use: the FP32 terms Ut (row-major) and S = strictly_lower(Kt Kh^T), and the bf16 hi/lo
// images of Kh, Qt, the masked QK, W (as W^T: rows k, cols r), exp(Gamma_C), T = (I + M)^-1 (lower),
// Diag(beta) Kt and Diag(beta) V.  Qt then enters [KK; QK] with its low part too, so QK is a full
// three-term product.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

// ---- shared-memory map (bytes from the 1024-byte aligned dynamic base) ------------------------
constexpr uint32_t OFF_KQ = 0;        // [Kt; Qt]: rows r / 64 + r, cols k, CS 2048, hi | lo       2 x 32768
constexpr uint32_t OFF_MT = 65536;    // g staging (four 32-column boxes)
constexpr uint32_t OFF_KH = 98304;    // Kh: rows i (64), cols k, CS 1024, hi | lo                2 x 16384
//   then (once [KK; QK] has read it) M (fp32 64 x 64) + T (fp32 64 x 64, at +16384)
constexpr uint32_t OFF_VT = 131072;   // V: rows r (64), cols v, CS 1024                            16384
constexpr uint32_t OFF_TP = 147456;   // T': rows r, cols i, CS 1024, hi | lo                      2 x 8192
constexpr uint32_t OFF_MISC = 163840;
constexpr uint32_t OFF_BETA = OFF_MISC;         // 64 fp32
constexpr uint32_t OFF_GC = OFF_MISC + 256;     // 128 fp32: exp(Gamma_C)
constexpr uint32_t OFF_NEXT = OFF_MISC + 1792;  // staged unit: beta (64 fp32), then its row count
// Raw rows of a unit, loaded by tiled TMA copies (128-byte swizzle, 1024-aligned boxes of 64 rows
// x 128 bytes) into their own regions: q, k, v as two 64-column boxes each, g as four 32-column
// boxes.  The next unit's copies are issued once this unit's rows are in registers.
constexpr uint32_t BOX = 8192;
constexpr uint32_t OFF_SQKV = 166912;
constexpr uint32_t STG_Q = OFF_SQKV, STG_K = OFF_SQKV + 2 * BOX, STG_V = OFF_SQKV + 4 * BOX, STG_G = OFF_MT;
constexpr uint32_t SMEM_BYTES = OFF_SQKV + 6 * BOX;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;   // room to align the base to 1024 bytes
constexpr uint32_t T128 = 32768, T64 = 16384;
constexpr uint32_t OFF_M32 = OFF_KH, OFF_T32 = OFF_KH + 16384;
static_assert(OFF_NEXT + 260 <= OFF_SQKV && OFF_SQKV % 1024 == 0, "staging region");

// ---- TMEM columns --------------------------------------------------------------------------
constexpr uint32_t TM_D1 = 0;     // [KK; QK] (64 cols)
constexpr uint32_t TM_W = 64;     // W^T
constexpr uint32_t TM_U = 128;    // Ut^T
constexpr uint32_t TM_COLS = 256;

constexpr int NWORK = 256;             // worker threads
constexpr int NTHREADS = NWORK + 64;   // plus the issuer (MMAs) and producer (row copies) warps
constexpr int ISSUER = NWORK;
constexpr int PRODUCER = NWORK + 32;
enum { HO_A = 0, HO_D = 1, HO_S = 2 };  // worker -> issuer handoffs of a unit (HO_S: staging read)

constexpr float LOG2E = 1.4426950408889634f;

__device__ int g_prep_status;   // set to KDA_ERR_TIMEOUT when a bounded wait expires

// fp32 64 x 64 scratch with the 16-byte chunk index XOR-swizzled by the row
__device__ __forceinline__ float *f32_at(unsigned char *base, uint32_t off, int r, int i)
{
    return reinterpret_cast<float *>(base + off + r * 256 + (((i >> 2) ^ (r & 15)) << 4) + (i & 3) * 4);
}

// 8 consecutive values as bf16 hi and lo words (4 + 4 packed pairs).
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) split_bf16x2(x[2 * p], x[2 * p + 1], h[p], l[p]);
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Writes 8 consecutive values as bf16 hi and lo (two 16-byte stores).
__device__ __forceinline__ void st_split8(unsigned char *hi, unsigned char *lo, const float *x)
{
    uint4 h, l;
    split8(x, h, l);
    *reinterpret_cast<uint4 *>(hi) = h;
    *reinterpret_cast<uint4 *>(lo) = l;
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

template <bool BWD>
__global__ void __launch_bounds__(NTHREADS, 1)
chunk_prep_tc(const int32_t *__restrict__ plan, PlanSig sig, int H, long long n_units, const float *__restrict__ beta,
              float scale, unsigned char *__restrict__ pkg, const __grid_constant__ CUtensorMap tm_q,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_g, unsigned char *__restrict__ bimg, float *__restrict__ bterms)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_mbar;
    __shared__ __align__(8) uint64_t s_ldbar;    // q, k, v rows landed
    __shared__ __align__(8) uint64_t s_gbar;     // g rows landed
    __shared__ __align__(8) uint64_t s_hbar[3];
    __shared__ uint32_t s_tmem;
    if (!plan_matches(plan, sig)) {   // not the plan the launch was sized from: touch nothing
        if (threadIdx.x == 0) record_status(&g_prep_status, KDA_ERR_INVALID_ARG);
        return;
    }
    unsigned char *const base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(base);
    float *const s_beta = reinterpret_cast<float *>(base + OFF_BETA);
    float *const s_gc = reinterpret_cast<float *>(base + OFF_GC);

    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;          // TMEM lane quadrant, column half
    const bool worker = tid < NWORK, issuer = tid == ISSUER, producer_warp = warp == PRODUCER / 32;
    const uint32_t mbar = smem_u32(&s_mbar), ldbar = smem_u32(&s_ldbar), gbar = smem_u32(&s_gbar);

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(ldbar, 1);
        mbar_init(gbar, 1);
        for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&s_hbar[i]), 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);  // this warp's lane quadrant
    const int c_lane = quad * 32 + lane;                                     // TMEM lane of this thread

    // unit u = head * n_chunks + chunk, so a head's chunks (and their packages, at
    // pkg + u * KDA_PACKAGE_BYTES) are consecutive; each CTA takes a contiguous run of units
    const int n_chunks = pv.n_chunks();
    const int32_t *const chunk_tab = pv.chunk(0);   // records of 4 words: piece, start, rows, index
    const long long u_begin = n_units * blockIdx.x / gridDim.x, u_end = n_units * (blockIdx.x + 1) / gridDim.x;
    // units are walked in order by (chunk, head) counters: no 64-bit division per unit
    struct UnitPos {
        int ch, h;
    };
    const UnitPos pos_begin{static_cast<int>(u_begin % n_chunks), static_cast<int>(u_begin / n_chunks)};
    auto advance = [&](UnitPos &q) {
        if (++q.ch == n_chunks) {
            q.ch = 0;
            ++q.h;
        }
    };
    // Rows of a unit (q, k, v, g) by tiled TMA copies; rows past the end of the tensor arrive as
    // zeros, rows past the chunk are masked when read.
    auto issue_rows = [&](int t0, int h) {
        mbar_arrive_expect_tx(ldbar, 6u * BOX);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(sbase + STG_Q + half * BOX, &tm_q, half * 64, h, t0, ldbar);
            tma_load_3d(sbase + STG_K + half * BOX, &tm_k, half * 64, h, t0, ldbar);
            tma_load_3d(sbase + STG_V + half * BOX, &tm_v, half * 64, h, t0, ldbar);
        }
        mbar_arrive_expect_tx(gbar, 4u * BOX);
#pragma unroll
        for (int qtr = 0; qtr < 4; ++qtr) tma_load_3d(sbase + STG_G + qtr * BOX, &tm_g, qtr * 32, h, t0, gbar);
    };
    // The producer warp stages a unit: its beta and row count into shared memory (all lanes), then
    // (lane 0) arms the row barriers, whose release orders those writes before the workers' waits,
    // and issues the row copies.
    float *const s_beta_next = reinterpret_cast<float *>(base + OFF_NEXT);
    int *const s_L_next = reinterpret_cast<int *>(base + OFF_NEXT + 256);
    auto load_beta = [&](int t0, int L, int h, float (&b)[2]) {   // issued early, used at staging
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = lane + 32 * e;
            b[e] = i < L ? beta[static_cast<size_t>(t0 + i) * H + h] : 0.f;
        }
    };
    auto stage_unit = [&](int t0, int L, int h, const float (&b)[2]) {
        s_beta_next[lane] = b[0];
        s_beta_next[lane + 32] = b[1];
        if (lane == 0) *s_L_next = L;
        __syncwarp();
        if (lane == 0) issue_rows(t0, h);
    };
    if (producer_warp && u_begin < u_end) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_q) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_k) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_v) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_g) : "memory");
        }
        const int t0 = chunk_tab[4 * pos_begin.ch + 1], L = chunk_tab[4 * pos_begin.ch + 2];
        float b[2];
        load_beta(t0, L, pos_begin.h, b);
        stage_unit(t0, L, pos_begin.h, b);
    }

    // the bf16 low part of the Qt rows (64 .. 127) of the stacked [Kt; Qt] operand: zero for good
    if (worker) {
        for (int e = tid; e < 16 * 64; e += NWORK) {   // 16 column chunks x 64 rows x 16 bytes
            const int ch = e >> 6, r = 64 + (e & 63);
            *reinterpret_cast<uint4 *>(base + OFF_KQ + T128 + cm_off(r, ch * 8, 2048)) = make_uint4(0u, 0u, 0u, 0u);
        }
    }

    bool aborted = false;   // all workers agree on it (OR-reduced at barriers)
    bool bad = false;       // a bounded wait of this thread gave up
    uint32_t phase = 0;
    auto wait_mma = [&]() {
        if (!mbar_wait(mbar, phase & 1)) bad = true;
        ++phase;
        fence_after();
    };
    // Workers hand their shared-memory operands over to the issuer: every writer fences its
    // generic-proxy stores for the tensor core, the workers meet on named barrier 1 (OR-reducing
    // their wait failures), and one of them arrives.
    auto handoff = [&](int which) -> bool {
        fence_async_smem();
        fence_before();
        const bool ab = bar_or1(NWORK, bad);
        if (!ab && tid == 0) mbar_arrive(smem_u32(&s_hbar[which]));
        return ab;
    };

    // W^T of a unit (already complete) from TMEM into its package
    auto store_w = [&](long long u) {
        unsigned char *const pk = pkg + static_cast<size_t>(u) * KDA_PACKAGE_BYTES;
        unsigned char *const im = BWD ? bimg + static_cast<size_t>(u) * RIMG_UNIT : nullptr;
        {
            float x[32];
            tmem_ld32(tl + TM_W + hw * 32, x);   // W^T[k = c_lane][r = hw*32 + j]
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint4 hi, lo;
                split8(x + 8 * m, hi, lo);
                const uint32_t off = cm_off(c_lane, hw * 32 + 8 * m, 2048);
                *reinterpret_cast<uint4 *>(pk + PK_W + off) = hi;
                *reinterpret_cast<uint4 *>(pk + PK_W + T64 + off) = lo;
                if constexpr (BWD) {
                    *reinterpret_cast<uint4 *>(im + RIMG_W + off) = hi;
                    *reinterpret_cast<uint4 *>(im + RIMG_W + T64 + off) = lo;
                }
            }
        }
    };
    // Ut^T by the threads of column half hw_of (all 32-column halves when one warp per quadrant
    // does it: hw_of < 0)
    auto store_ut = [&](long long u, int hw_of) {
        unsigned char *const pk = pkg + static_cast<size_t>(u) * KDA_PACKAGE_BYTES;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            const int hh = hw_of < 0 ? half : hw_of;
            if (hw_of >= 0 && half > 0) break;
            float x[32];
            tmem_ld32(tl + TM_U + hh * 32, x);   // Ut^T[c = c_lane][r = hh*32 + j]
            // Ut^T as [hh][m][c] float4 groups: a warp's store (and the state pass's load) of one
            // group covers 512 contiguous bytes
            float4 *ut = reinterpret_cast<float4 *>(pk + PK_U) + hh * 8 * 128 + c_lane;
#pragma unroll
            for (int m = 0; m < 8; ++m) ut[m * 128] = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
            if constexpr (BWD) {   // Ut row-major: a warp's store covers 128 contiguous bytes of a row
                float *const ur = bterms + static_cast<size_t>(u) * BT_FLOATS + BT_UT + (hh * 32) * VD + c_lane;
#pragma unroll
                for (int j = 0; j < 32; ++j) ur[j * VD] = x[j];
            }
        }
    };

    if (worker) {
        int n = 0;
        for (long long u = u_begin; u < u_end && !aborted; ++u, ++n) {
            unsigned char *const pk = pkg + static_cast<size_t>(u) * KDA_PACKAGE_BYTES;
            unsigned char *const im = BWD ? bimg + static_cast<size_t>(u) * RIMG_UNIT : nullptr;
            float *const bt = BWD ? bterms + static_cast<size_t>(u) * BT_FLOATS : nullptr;
            int L;

            // ================= A: staged rows -> decayed keys / queries / values =====================
            {
                if (!mbar_wait_warp(gbar, n & 1)) bad = true;
                L = *s_L_next;   // staged with the rows (read before this unit's staging handoff)
                // A1: log2-scaled cumulative decay per key channel, in place over the staged g: each
                //     thread scans 8 rows x 4 channels (16-byte loads), the 8 row groups' totals meet
                //     in the Kh region (free until A3 writes this unit's Kh), each thread adds the
                //     totals of the groups above its own and stores its rows back
                {
                    const int cq = tid & 31, rg = tid >> 5;   // channels 4 cq .. 4 cq + 3, rows 8 rg .. 8 rg + 7
                    unsigned char *gq = base + STG_G + (cq >> 3) * BOX;
                    const int gch = cq & 7;
                    float4 gv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) gv[j] = *reinterpret_cast<const float4 *>(gq + sw128(rg * 8 + j, gch));
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const bool ok = rg * 8 + j < L;
                        acc.x += ok ? gv[j].x * LOG2E : 0.f;
                        acc.y += ok ? gv[j].y * LOG2E : 0.f;
                        acc.z += ok ? gv[j].z * LOG2E : 0.f;
                        acc.w += ok ? gv[j].w * LOG2E : 0.f;
                        gv[j] = acc;
                    }
                    float4 *const gtot = reinterpret_cast<float4 *>(base + OFF_KH);   // [row group][channel quad]
                    gtot[rg * 32 + cq] = acc;
                    if (tid < 64) s_beta[tid] = s_beta_next[tid];
                    bar_sync1(NWORK);
                    float4 off = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int g2 = 0; g2 < 7; ++g2) {
                        const float4 t = gtot[g2 * 32 + cq];
                        if (g2 < rg) {
                            off.x += t.x;
                            off.y += t.y;
                            off.z += t.z;
                            off.w += t.w;
                        }
                    }
                    if (rg == 7) {
                        // Gamma_C log2 e per channel; below 2^-112 the decayed operands and their bf16 low
                        // parts leave the normal fp32 range (NaN or inf in g lands here too)
                        const float4 gs = make_float4(off.x + acc.x, off.y + acc.y, off.z + acc.z, off.w + acc.w);
                        if (!(gs.x >= -112.f && gs.y >= -112.f && gs.z >= -112.f && gs.w >= -112.f))
                            record_status(&g_prep_status, KDA_ERR_RANGE);
                        const float4 gcv = make_float4(ex2_ftz(gs.x), ex2_ftz(gs.y), ex2_ftz(gs.z), ex2_ftz(gs.w));
                        reinterpret_cast<float4 *>(s_gc)[cq] = gcv;
                        reinterpret_cast<float4 *>(pk + PK_GC)[cq] = gcv;
                        if constexpr (BWD) reinterpret_cast<float4 *>(im + RIMG_GC)[cq] = gcv;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4 *>(gq + sw128(rg * 8 + j, gch)) =
                            make_float4(gv[j].x + off.x, gv[j].y + off.y, gv[j].z + off.z, gv[j].w + off.w);
                    bar_sync1(NWORK);
                }
                // A2: each thread takes four (row, 8-column) pieces of the staged rows into registers;
                //     the lanes of a warp hold consecutive rows of one piece column
                if (!mbar_wait_warp(ldbar, n & 1)) bad = true;
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
                    vw[i] = ok ? *reinterpret_cast<const uint4 *>(base + STG_V + bo) : z;
                }
                bar_sync1(NWORK);   // staging consumed: the next unit's rows may land
                if (tid == 0) mbar_arrive(smem_u32(&s_hbar[HO_S]));
                if (n > 0) wait_mma();   // the previous unit's W / Ut have read the operand tiles
                // A3: Kt, Qt (stacked), Kh as bf16 hi/lo and V as bf16 in shared memory; Qt hi and Kh
                //     hi/lo also into the package (lanes hold consecutive rows: 512 contiguous bytes)
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
                    uint4 hi, lo;
                    split8(kt, hi, lo);
                    *reinterpret_cast<uint4 *>(base + OFF_KQ + o_r) = hi;
                    *reinterpret_cast<uint4 *>(base + OFF_KQ + T128 + o_r) = lo;
                    if constexpr (BWD) {   // Diag(beta) Kt and Diag(beta) V for the gradient pass
                        const float br = s_beta[r];
                        float bx[8], vf[8];
#pragma unroll
                        for (int e8 = 0; e8 < 8; ++e8) bx[e8] = br * kt[e8];
                        split8(bx, hi, lo);
                        *reinterpret_cast<uint4 *>(im + RIMG_BKT + o_64) = hi;
                        *reinterpret_cast<uint4 *>(im + RIMG_BKT + T64 + o_64) = lo;
                        bf16x8_to_f32(vw[i], vf);
#pragma unroll
                        for (int e8 = 0; e8 < 8; ++e8) bx[e8] = br * vf[e8];
                        split8(bx, hi, lo);
                        *reinterpret_cast<uint4 *>(im + RIMG_BV + o_64) = hi;
                        *reinterpret_cast<uint4 *>(im + RIMG_BV + T64 + o_64) = lo;
                    }
                    if constexpr (BWD) {
                        // the backward's QK and Qt take the full split
                        split8(qt, hi, lo);
                        *reinterpret_cast<uint4 *>(base + OFF_KQ + o_q) = hi;
                        *reinterpret_cast<uint4 *>(base + OFF_KQ + T128 + o_q) = lo;
                        *reinterpret_cast<uint4 *>(pk + PK_Q + o_64) = hi;
                        *reinterpret_cast<uint4 *>(im + RIMG_QT + o_64) = hi;
                        *reinterpret_cast<uint4 *>(im + RIMG_QT + T64 + o_64) = lo;
                    } else {
                        // Qt only feeds the masked scores QK, single-term like every output product: its
                        // bf16 low part stays zero (cleared once at the start), one conversion per pair
                        hi = make_uint4(bf16x2_bits(qt[0], qt[1]), bf16x2_bits(qt[2], qt[3]),
                                        bf16x2_bits(qt[4], qt[5]), bf16x2_bits(qt[6], qt[7]));
                        *reinterpret_cast<uint4 *>(base + OFF_KQ + o_q) = hi;
                        *reinterpret_cast<uint4 *>(pk + PK_Q + o_64) = hi;
                    }
                    split8(kh, hi, lo);
                    *reinterpret_cast<uint4 *>(base + OFF_KH + o_64) = hi;
                    *reinterpret_cast<uint4 *>(base + OFF_KH + T64 + o_64) = lo;
                    *reinterpret_cast<uint4 *>(pk + PK_KH + o_64) = hi;
                    *reinterpret_cast<uint4 *>(pk + PK_KH + T64 + o_64) = lo;
                    if constexpr (BWD) {
                        *reinterpret_cast<uint4 *>(im + RIMG_KH + o_64) = hi;
                        *reinterpret_cast<uint4 *>(im + RIMG_KH + T64 + o_64) = lo;
                    }
                    *reinterpret_cast<uint4 *>(base + OFF_VT + o_64) = vw[i];
                }
                aborted = handoff(HO_A);   // -> [KK; QK]
            }
            if (aborted) break;
            if (n > 0) store_w(u - 1);   // while [KK; QK] runs

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
                        float4 s4, m4;
                        const int i0 = hw * 32 + 4 * j4;
                        s4.x = (i0 + 0 < r) ? d[4 * j4 + 0] : 0.f;
                        s4.y = (i0 + 1 < r) ? d[4 * j4 + 1] : 0.f;
                        s4.z = (i0 + 2 < r) ? d[4 * j4 + 2] : 0.f;
                        s4.w = (i0 + 3 < r) ? d[4 * j4 + 3] : 0.f;
                        m4 = make_float4(br * s4.x, br * s4.y, br * s4.z, br * s4.w);
                        *reinterpret_cast<float4 *>(f32_at(base, OFF_M32, r, i0)) = m4;
                        if constexpr (BWD) *reinterpret_cast<float4 *>(bt + BT_S + r * 64 + i0) = s4;
                    }
                } else {
                    const int r = c_lane - 64;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t off = cm_off(r, hw * 32 + 8 * m, 1024);
                        if constexpr (BWD) {
                            float qk[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) qk[e] = hw * 32 + 8 * m + e <= r ? d[8 * m + e] : 0.f;
                            uint4 hi, lo;
                            split8(qk, hi, lo);
                            *reinterpret_cast<uint4 *>(pk + PK_QK + off) = hi;
                            *reinterpret_cast<uint4 *>(im + RIMG_QK + off) = hi;
                            *reinterpret_cast<uint4 *>(im + RIMG_QK + 8192 + off) = lo;
                        } else {
                            uint32_t w[4];
#pragma unroll
                            for (int p2 = 0; p2 < 4; ++p2) {
                                const int i0 = hw * 32 + 8 * m + 2 * p2;
                                w[p2] = bf16x2_bits(i0 <= r ? d[8 * m + 2 * p2] : 0.f,
                                                    i0 + 1 <= r ? d[8 * m + 2 * p2 + 1] : 0.f);
                            }
                            *reinterpret_cast<uint4 *>(pk + PK_QK + off) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
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
            // warps 4 - 7 (one per TMEM lane quadrant) store the previous unit's Ut^T meanwhile: its
            // columns stay valid until this unit's T' is handed over
            if (n > 0 && tid >= 128) store_ut(u - 1, -1);
            if (tid < 64) {   // column jj of diagonal block b, row by row: x_r = -sum_{i<r} M[r][i] x_i
                const int b = tid >> 4, jj = tid & 15, r0 = 16 * b;
                float x[16];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    float s0 = 0.f, s1 = 0.f;   // two partial sums: half the dependent chain
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {   // the block row's entries in 16-byte loads
                        if (4 * m4 < rr) {
                            const float4 mv =
                                *reinterpret_cast<const float4 *>(f32_at(base, OFF_M32, r0 + rr, r0 + 4 * m4));
                            const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (4 * m4 + e < rr) {
                                    if (e & 1) s1 = fmaf(mm[e], x[4 * m4 + e], s1);
                                    else s0 = fmaf(mm[e], x[4 * m4 + e], s0);
                                }
                            }
                        }
                    }
                    x[rr] = (rr == jj) ? 1.f : ((rr < jj) ? 0.f : -(s0 + s1));
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
                float tfull[BWD ? 16 : 1];   // (backward mode) T itself, for its image
#pragma unroll
                for (int m4 = 0; m4 < 4; ++m4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(f32_at(base, OFF_T32, r, i0 + 4 * m4));
                    const float tt[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = i0 + 4 * m4 + e;
                        const float t = (i <= r) ? tt[e] : 0.f;   // T, zero above the diagonal
                        tv[4 * m4 + e] = t * s_beta[i];
                        if constexpr (BWD) tfull[4 * m4 + e] = t;
                    }
                }
                if constexpr (BWD) {   // T's image for the gradient pass (rows r, cols i)
                    uint4 hi, lo;
                    split8(tfull, hi, lo);
                    *reinterpret_cast<uint4 *>(im + RIMG_T + cm_off(r, i0, 1024)) = hi;
                    *reinterpret_cast<uint4 *>(im + RIMG_T + 8192 + cm_off(r, i0, 1024)) = lo;
                    split8(tfull + 8, hi, lo);
                    *reinterpret_cast<uint4 *>(im + RIMG_T + cm_off(r, i0 + 8, 1024)) = hi;
                    *reinterpret_cast<uint4 *>(im + RIMG_T + 8192 + cm_off(r, i0 + 8, 1024)) = lo;
                }
                st_split8(base + OFF_TP + cm_off(r, i0, 1024), base + OFF_TP + 8192 + cm_off(r, i0, 1024), tv);
                st_split8(base + OFF_TP + cm_off(r, i0 + 8, 1024), base + OFF_TP + 8192 + cm_off(r, i0 + 8, 1024),
                          tv + 8);
            }
                aborted = handoff(HO_D);   // -> W^T = Kt^T T'^T, Ut^T = V^T T'^T
            }

        }
        if (!aborted && n > 0) {   // the last unit's W / Ut
            wait_mma();
            if (!bar_or1(NWORK, bad)) {
                store_w(u_end - 1);
                store_ut(u_end - 1, hw);
            }
            else aborted = true;
        }
    } else if (issuer) {
        // Issuer: per unit, [KK; QK] once the operand tiles are in, then W and Ut once T' is.
        bool ok = true;
        int n = 0;
        for (long long u = u_begin; u < u_end && ok; ++u, ++n) {
            const uint32_t par = n & 1;
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_A]), par))) break;
            fence_after();
            {
                const uint32_t id = idesc_bf16(128, 64);
                const uint32_t aoff[3] = {0, 0, T128}, boff[3] = {0, T64, 0};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tbase + TM_D1, sdesc(sbase + OFF_KQ + aoff[ps] + kk * 2 * 2048, 2048),
                                 sdesc(sbase + OFF_KH + boff[ps] + kk * 2 * 1024, 1024), id, (ps | kk) != 0);
                commit(mbar);
            }
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_D]), par))) break;
            fence_after();
            {
                // W^T = Kt^T T'^T (3-term; Kt^T is the row-major Kt tile read MN-major)
                const uint32_t id = idesc_bf16(128, 64, 1, 0);
                const uint32_t aoff[3] = {0, 0, T128}, boff[3] = {0, 8192, 0};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tbase + TM_W, sdesc(sbase + OFF_KQ + aoff[ps] + kk * 256, 128, 2048),
                                 sdesc(sbase + OFF_TP + boff[ps] + kk * 2 * 1024, 1024), id, (ps | kk) != 0);
                // Ut^T = V^T T'^T (2-term)
#pragma unroll
                for (int ps = 0; ps < 2; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tbase + TM_U, sdesc(sbase + OFF_VT + kk * 256, 128, 1024),
                                 sdesc(sbase + OFF_TP + ps * 8192 + kk * 2 * 1024, 1024), id, (ps | kk) != 0);
                commit(mbar);
            }
        }
        if (!ok) record_status(&g_prep_status, KDA_ERR_TIMEOUT);
    } else if (producer_warp) {
        // Producer warp: the next unit once this unit's staged rows and metadata are read (a TMA unit
        // busy with earlier boxes stalls the thread that issues more, which must not be the MMA
        // issuer; the row count and beta loads ride along off the workers' path)
        bool ok = true;
        int n = 0;
        int last = 0;   // unit count of the last staged copies
        UnitPos ipos = pos_begin;
        advance(ipos);   // the unit staged next
        for (long long u = u_begin; u + 1 < u_end && ok; ++u, ++n) {
            const int t0_next = chunk_tab[4 * ipos.ch + 1], L_next = chunk_tab[4 * ipos.ch + 2];
            float b[2];
            load_beta(t0_next, L_next, ipos.h, b);   // in flight during the wait
            if (!(ok = mbar_wait_warp(smem_u32(&s_hbar[HO_S]), n & 1))) break;
            stage_unit(t0_next, L_next, ipos.h, b);
            advance(ipos);
            last = n + 1;
        }
        if (!ok && lane == 0) record_status(&g_prep_status, KDA_ERR_TIMEOUT);
        if (lane == 0 && u_begin < u_end) {   // bounded: every staged copy lands before the CTA exits
            mbar_wait(ldbar, last & 1);
            mbar_wait(gbar, last & 1);
        }
    }
    if (worker && aborted && tid == 0) record_status(&g_prep_status, KDA_ERR_TIMEOUT);
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

cudaError_t launch_chunk_prep(const int32_t *plan_host, const int32_t *plan_dev, int H, const uint16_t *q,
                              const uint16_t *k, const uint16_t *v, const float *g, const float *beta, float scale,
                              unsigned char *pkg, cudaStream_t stream, unsigned char *bimg, float *bterms)
{
    const PlanView pv{plan_host};
    const long long n_units = static_cast<long long>(pv.n_chunks()) * H;
    if (n_units <= 0) return cudaSuccess;
    const int T = pv.T();
    CUtensorMap tq, tk, tv, tg;
    if (!encode_rows_3d(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64) ||
        !encode_rows_3d(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64) ||
        !encode_rows_3d(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, T, 64) ||
        !encode_rows_3d(&tg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, T, 32))
        return cudaErrorInvalidValue;
    const bool bwd = bimg != nullptr && bterms != nullptr;
    if ((bimg != nullptr) != (bterms != nullptr)) return cudaErrorInvalidValue;
    const void *fn = bwd ? reinterpret_cast<const void *>(chunk_prep_tc<true>)
                         : reinterpret_cast<const void *>(chunk_prep_tc<false>);
    cudaError_t err = set_dynamic_smem(fn, static_cast<int>(SMEM_ALLOC));
    if (err != cudaSuccess) return err;
    const long long grid = n_units < sm_count() ? n_units : sm_count();
    const PlanSig sig = plan_sig(plan_host);
    if (bwd)
        chunk_prep_tc<true><<<static_cast<unsigned>(grid), NTHREADS, SMEM_ALLOC, stream>>>(
            plan_dev, sig, H, n_units, beta, scale, pkg, tq, tk, tv, tg, bimg, bterms);
    else
        chunk_prep_tc<false><<<static_cast<unsigned>(grid), NTHREADS, SMEM_ALLOC, stream>>>(
            plan_dev, sig, H, n_units, beta, scale, pkg, tq, tk, tv, tg, nullptr, nullptr);
    return cudaGetLastError();
}

// The status word of this file's kernel: read and cleared (the caller has synchronised the device).
int take_prep_status()
{
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_prep_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_prep_status, &z, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return v;
}

}  // namespace kda
