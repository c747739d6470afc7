// Segment-parallel backward of the KDA forward: gradients of q, k, v, g, beta and h0.
//
// The pages name the backward's inputs only: cuLA PR #136 ("feat(kda): add cuDNN
// concatenated-summary Kimi CP", §Summary and its walkthrough's sequence diagram: the following
// FP32 summaries are gathered during the backward), and cuLA PR #110 ("feat(cp): add opt-in
// NVSHMEM CP state handoff", §Correctness) checks the output and Q/K/V/g/beta gradients.  The loss
// is L = sum_t <do_t, o_t> + sum_seq <dfinal, S_end>.  Per 64-token chunk, with the chunk's terms
// (Gamma = in-chunk cumulative g, Kt = e^Gamma k, Kh = e^-Gamma k, Qt = scale e^Gamma q,
// M = Diag(beta) strictly_lower(Kt Kh^T), T = (I + M)^-1, W = T Diag(beta) Kt, Ut = T Diag(beta) V,
// QK = lower(Qt Kh^T), Dc = Diag(e^Gamma_C)) the forward is
//     U = Ut - W X,   O = Qt X + QK U,   X' = Dc (X + Kh^T U),
// and its reverse, given the gradient G of X', is
//     DG = Dc G,   dU = Kh DG + QK^T dO,   dX = DG + Qt^T dO - W^T dU.
// The chunk's input gradients follow from (X, G, dO) by the chain rule through the terms above.
//
// Steps (after the forward's own preparation, state pass and composition, which give S_in, the
// segment transitions A and the final-state transitions of continuing pieces):
//  0. every (chunk, head) in parallel: the chunk's FP32 terms (Ut, S) for the gradient pass and the bf16
//     operand images (Kh, Qt, QK, W, Dc, T, Diag(beta) Kt, Diag(beta) V) of the reverse chains and the
//     gradient pass, which the forward's preparation writes in its backward mode (the caller launches
//     it), and dO's image;
//  1. every piece from its true incoming state (h0, or S_in of its segment), recording each chunk's
//     start state X_c as the image of X_c^T: the forward's state pass in its output mode (the caller
//     launches it);
//  2. (reverse.cu) every piece that continues a sequence, backwards from a zero end gradient: the gradient of its
//     incoming state through its own outputs, Qd (the qhat do^T sum of the pages' summaries);
//  3. the following summaries, last segment first: the gradient of the state crossing the end of
//     segment j is dfinal of a sequence that ends there, or Qd[j+1] plus the transposed map of the
//     continuing piece of segment j+1 (A[j+1]^T, or P_end^T of a piece that ends its sequence
//     there, on dfinal) applied to the gradient at that piece's end;
//  4. (reverse.cu) every piece backwards from its true end gradient, recording each chunk's DG_c = Dc G_c
//     (G_c its end gradient) as the image of DG_c^T and giving dh0 at a sequence start;
//  5. every (chunk, head) in parallel: dq, dk, dv, dg, dbeta from (X_c, DG_c, dO).
//
// The gradient pass here runs every product on the tensor cores, its operands bf16 hi/lo images brought
// into shared memory by bulk copies (a three-term split accumulated in FP32 in TMEM), and keeps the
// results that later steps read in a private scratch area in global memory (FP32 where an element-wise
// step reads them, as images where a product does), which keeps every step a literal transcription of
// the formulas above.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int BT = 256;                      // threads per CTA
constexpr int CK = 64 * KD;                  // a 64 x 128 chunk matrix
constexpr int CC = 64 * 64;                  // a 64 x 64 chunk matrix
constexpr int SQ = KD * VD;                  // a 128 x 128 state

__device__ int g_bwd_status;

// Per-CTA scratch (floats): the FP32 product results an element-wise step reads (dKh, dQt, dKt: 64 x 128;
// d(beta Kt) and d(beta V) side by side in one 64 x 256 array; dM: 64 x 64), row vectors (gc, beta,
// dGamma_C), then bf16 hi/lo images (bytes / 4) of the products' results that later products read (U, dQK,
// dU, dW, dT, T^T dT, dM).  About 0.34 MB: the working areas of all CTAs fit in the L2.
enum : int {
    S_DKH = 0, S_DQT = S_DKH + CK, S_DKT = S_DQT + CK, S_DBKV = S_DKT + CK,   // [d(beta Kt) | d(beta V)]: 64 x 256
    S_DM = S_DBKV + 2 * CK, S_GC = S_DM + CC, S_BT = S_GC + KD, S_DGC = S_BT + 64,
    S_IMG = (S_DGC + KD + 255) & ~255,
    S_UI = S_IMG, S_DQKI = S_UI + CK, S_DUI = S_DQKI + CC, S_DWI = S_DUI + CK, S_DTI = S_DWI + CK,
    S_T64I = S_DTI + CC, S_DMI = S_T64I + CC, S_IMG_END = S_DMI + CC,
    SCRATCH_FLOATS = S_IMG_END
};

static_assert(BT_UT == 0 && BT_S == CK && BT_FLOATS == BT_S + CC, "the chunk terms' layout");

// Dynamic shared memory of the backward's kernels: both operands of one product, k-major.
constexpr size_t BWD_SMEM = 6ull * 32768 + 1024;   // the operand tiles of a two-term product, aligned to 1024 bytes

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
// Orders this thread's generic-proxy global writes before later bulk (async-proxy) reads of them.
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ float4 add4(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ float4 sub4(float4 a, float4 b) { return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }
// 8 bf16 (16 bytes) as fp32
__device__ __forceinline__ void bf16x8(uint4 w, float *x)
{
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        x[2 * p] = __uint_as_float(ww[p] << 16);
        x[2 * p + 1] = __uint_as_float(ww[p] & 0xFFFF0000u);
    }
}
// 4 bf16 (8 bytes) as fp32
__device__ __forceinline__ float4 bf4(uint2 w)
{
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
}
__device__ __forceinline__ float4 mul4(float4 a, float4 b) { return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w); }
__device__ __forceinline__ float4 scl4(float s, float4 a) { return make_float4(s * a.x, s * a.y, s * a.z, s * a.w); }
__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) v += __shfl_xor_sync(0xffffffffu, v, sh);
    return v;
}

// Tensor-core state of a CTA: the accumulator's TMEM columns, the products' mbarrier and the parity
// of its next phase, and a flag raised when a bounded wait gave up (every later product of the CTA
// is then skipped, and the kernel reports KDA_ERR_TIMEOUT).
__shared__ __align__(8) uint64_t s_tc_bar;
__shared__ __align__(8) uint64_t s_tc_ld;   // a product's operand images landed (bulk copies)
__shared__ uint32_t s_tc_tmem, s_tc_phase, s_tc_fail, s_tc_ldph;
constexpr uint32_t TC_COLS = 256;

__device__ void tc_begin()
{
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&s_tc_bar), 1);
        mbar_init(smem_u32(&s_tc_ld), 1);
        s_tc_phase = 0;
        s_tc_fail = 0;
        s_tc_ldph = 0;
    }
    if (threadIdx.x < 32) tmem_alloc(smem_u32(&s_tc_tmem), TC_COLS);
    fence_before();
    __syncthreads();
    fence_after();
}

__device__ void tc_end()
{
    fence_before();
    __syncthreads();
    fence_after();
    if (threadIdx.x == 0 && s_tc_fail) record_status(&g_bwd_status, KDA_ERR_TIMEOUT);
    if (threadIdx.x < 32) tmem_dealloc(s_tc_tmem, TC_COLS);
}

// The operand tiles in dynamic shared memory (1024-byte aligned): A hi | lo (128 x K bf16 each), then
// B hi | lo (N x K bf16 each).
__device__ __forceinline__ unsigned char *tc_tiles()
{
    extern __shared__ __align__(16) unsigned char bsm_raw[];
    return bsm_raw + ((1024u - (smem_u32(bsm_raw) & 1023u)) & 1023u);
}

// One term A B of a product, both operands as images in global memory: the bf16 hi/lo split of the
// operand as it lies (R rows of its contiguous index, chunk stride R * 16, lo R * C * 2 bytes after hi; a
// single image holds only hi, the operand being exact in bf16, and the products with its lo part are
// skipped), brought in by bulk copies.  A(m, k) is the image's [k][m] when the product transposes A (rows k),
// else [m][k]; B(k, n) likewise [n][k] or [k][n].  b2, when set (untransposed B only), is a second image whose
// columns follow b's: B = [b | b2].
struct Term {
    const unsigned char *a, *b, *b2;
    bool a_single, b_single;
};
__device__ __forceinline__ Term term(const unsigned char *a, const unsigned char *b, bool a_single = false,
                                     bool b_single = false, const unsigned char *b2 = nullptr)
{
    return Term{a, b, b2, a_single, b_single};
}

// The output of a product: C[m][n] = out_rows[m] * (alpha * sum of the terms + in_rows[m] * cin[m][n]),
// each factor or input omitted when its pointer is null; MASK 1 keeps n <= m, MASK 2 n < m (zero
// elsewhere).  c may be null; img, when set, receives the result's bf16 hi/lo image as it lies (M rows).
struct Out {
    float *c;
    int ldc;
    float alpha;
    const float *cin;
    int ldcin;
    const float *in_rows;
    const float *out_rows;
    unsigned char *img;
};
__device__ __forceinline__ Out out(float *c, int ldc, float alpha = 1.f, const float *cin = nullptr, int ldcin = 0,
                                   const float *in_rows = nullptr, const float *out_rows = nullptr)
{
    return Out{c, ldc, alpha, cin, ldcin, in_rows, out_rows, nullptr};
}
__device__ __forceinline__ Out out_img(Out o, unsigned char *img)
{
    o.img = img;
    return o;
}

// An M x N product of one or two terms (K1- and K2-long sums; K2 = 0: one term; M, K in {64, 128}, N in
// {64, 128}, or 256 for a one-term product with no accumulated input)
// by all threads of the CTA.  Every operand is an image of its bf16 hi/lo split as it lies (rows of its
// contiguous index, chunk stride: its rows x 16), brought into the no-swizzle canonical tiles by bulk copies
// and read by the tensor core K-major or MN-major accordingly, so nothing is transposed on the way; each
// term is the split hi*hi + hi*lo + lo*hi (~2^-16 relative; without the products of a single operand's
// absent lo part), both terms accumulate in FP32 in one TMEM accumulator, M = 128 (a 64-row A fills half
// the lanes: the rows the tensor core reads past it land in lanes that are never read).  The accumulated
// input is loaded while the tensor core works.
template <int M, int N, int K1, bool TA1, bool TB1, int K2 = 0, bool TA2 = false, bool TB2 = false, int MASK = 0>
__device__ void product(const Term t1, const Term t2, const Out o)
{
    static_assert((M == 64 || M == 128) && (N == 64 || N == 128 || (N == 256 && K2 == 0 && !TB1)) &&
                      (K1 == 64 || K1 == 128) && (K2 == 0 || K2 == 64 || K2 == 128), "shapes");
    if (s_tc_fail) return;   // uniform: written before the previous product's closing barrier
    const int tid = threadIdx.x;
    constexpr int K2E = K2 ? K2 : 64;   // shapes of the (unused when K2 = 0) second term
    constexpr int RA1 = TA1 ? K1 : M, CA1 = TA1 ? M : K1, RB1 = TB1 ? N : K1, CB1 = TB1 ? K1 : N;
    constexpr int RA2 = TA2 ? K2E : M, CA2 = TA2 ? M : K2E, RB2 = TB2 ? N : K2E, CB2 = TB2 ? K2E : N;
    constexpr uint32_t CSA1 = RA1 * 16, CSB1 = RB1 * 16, CSA2 = RA2 * 16, CSB2 = RB2 * 16;
    constexpr uint32_t A1B = 128 * K1 * 2, B1B = N * K1 * 2, A2B = 128 * K2E * 2, B2B = N * K2E * 2;
    static_assert(2 * (A1B + B1B + (K2 ? A2B + B2B : 0)) <= BWD_SMEM - 1024, "the operand tiles fit");
    unsigned char *const a1h = tc_tiles(), *const a1l = a1h + A1B, *const b1h = a1l + A1B, *const b1l = b1h + B1B;
    unsigned char *const a2h = b1l + B1B, *const a2l = a2h + A2B, *const b2h = a2l + A2B, *const b2l = b2h + B2B;
    if (tid == 0) {   // the operands: bulk copies into the tiles, counted on s_tc_ld
        const uint32_t ld = smem_u32(&s_tc_ld);
        uint32_t bytes = 0;
        auto part = [&](bool single, uint32_t nbytes) { bytes += single ? nbytes : 2 * nbytes; };
        part(t1.a_single, RA1 * CA1 * 2);
        part(t1.b_single, RB1 * CB1 * 2);
        if (K2 != 0) {
            part(t2.a_single, RA2 * CA2 * 2);
            part(t2.b_single, RB2 * CB2 * 2);
        }
        mbar_arrive_expect_tx(ld, bytes);
        auto copy = [&](const unsigned char *img, bool single, uint32_t nbytes, unsigned char *hi, unsigned char *lo) {
            bulk_g2s(smem_u32(hi), img, nbytes, ld);
            if (!single) bulk_g2s(smem_u32(lo), img + nbytes, nbytes, ld);
        };
        copy(t1.a, t1.a_single, RA1 * CA1 * 2, a1h, a1l);
        if (t1.b2) {   // B = [b | b2]: each image fills half of the tile's column chunks
            copy(t1.b, t1.b_single, RB1 * CB1, b1h, b1l);
            copy(t1.b2, t1.b_single, RB1 * CB1, b1h + RB1 * CB1, b1l + RB1 * CB1);
        } else {
            copy(t1.b, t1.b_single, RB1 * CB1 * 2, b1h, b1l);
        }
        if (K2 != 0) {
            copy(t2.a, t2.a_single, RA2 * CA2 * 2, a2h, a2l);
            copy(t2.b, t2.b_single, RB2 * CB2 * 2, b2h, b2l);
        }
    }
    __syncthreads();   // every thread reads the phase of this product's barrier after the previous one's update
    fence_after();
    const uint32_t ph = s_tc_phase, tmem = s_tc_tmem, bar = smem_u32(&s_tc_bar);
    if (tid == 0) {
        const bool ld_ok = mbar_wait(smem_u32(&s_tc_ld), s_tc_ldph);
        s_tc_ldph ^= 1u;
        if (!ld_ok) s_tc_fail = 1;
        bool first = true;
        // the split terms of one A B pair: hi hi, hi lo (unless B is single), lo hi (unless A is single)
        auto issue = [&](int K, bool ta, bool tb, uint32_t ah_, uint32_t al_, uint32_t bh_, uint32_t bl_, uint32_t csa,
                         uint32_t csb, bool a_single, bool b_single) {
            const uint32_t id = idesc_bf16(128, N, ta ? 1 : 0, tb ? 0 : 1);
            const uint32_t ah[3] = {ah_, ah_, al_}, bh[3] = {bh_, bl_, bh_};
            const bool use[3] = {true, !b_single, !a_single};
            for (int ps = 0; ps < 3; ++ps) {
                if (!use[ps]) continue;
                for (int kk = 0; kk < K / 16; ++kk) {
                    const uint64_t ad = ta ? sdesc(ah[ps] + kk * 256, 128, csa) : sdesc(ah[ps] + kk * 2 * csa, csa, 128);
                    const uint64_t bd = tb ? sdesc(bh[ps] + kk * 2 * csb, csb, 128) : sdesc(bh[ps] + kk * 256, 128, csb);
                    mma_bf16(tmem, ad, bd, id, first ? 0u : 1u);
                    first = false;
                }
            }
        };
        if (ld_ok) {
            issue(K1, TA1, TB1, smem_u32(a1h), smem_u32(a1l), smem_u32(b1h), smem_u32(b1l), CSA1, CSB1, t1.a_single,
                  t1.b_single);
            if constexpr (K2 != 0)
                issue(K2, TA2, TB2, smem_u32(a2h), smem_u32(a2l), smem_u32(b2h), smem_u32(b2l), CSA2, CSB2,
                      t2.a_single, t2.b_single);
        }
        commit(bar);   // (with nothing issued, it arrives at once: the readers see the failure flag)
    }
    // row m = this thread's TMEM lane, columns hw * N/2 .. + N/2; the accumulated input is loaded
    // while the tensor core works
    const int warp = tid >> 5, quad = warp & 3, hw = warp >> 2;
    const int m = quad * 32 + (tid & 31), n0 = hw * (N / 2);
    const bool live = quad * 32 < M;
    constexpr int NOLD = N <= 128 ? N / 8 : 1;   // (N = 256: no accumulated input)
    float4 old[NOLD];
    if constexpr (N <= 128) {
        const float f = (o.cin && live) ? (o.in_rows ? o.in_rows[m] : 1.f) : 0.f;
#pragma unroll
        for (int q4 = 0; q4 < N / 8; ++q4)
            old[q4] = (o.cin && live) ? scl4(f, ld4(o.cin + m * o.ldcin + n0 + 4 * q4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float fo = (o.out_rows && live) ? o.out_rows[m] : 1.f;
    const bool ok = mbar_wait_warp(bar, ph);
    fence_after();
    if (ok && live) {
        float *const crow = o.c ? o.c + m * o.ldc + n0 : nullptr;
#pragma unroll
        for (int j0 = 0; j0 < N / 2; j0 += 32) {
            float d[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + n0 + j0, d);
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                float r[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float ov = 0.f;
                    if constexpr (N <= 128) {
                        const float4 o4 = old[(j0 + 8 * q8 + e) / 4];
                        ov = (e & 3) == 0 ? o4.x : (e & 3) == 1 ? o4.y : (e & 3) == 2 ? o4.z : o4.w;
                    }
                    r[e] = fo * (o.alpha * d[8 * q8 + e] + ov);
                    if constexpr (MASK != 0) {
                        const int n = n0 + j0 + 8 * q8 + e;
                        if (MASK == 1 ? n > m : n >= m) r[e] = 0.f;
                    }
                }
                if (crow) {
                    st4(crow + j0 + 8 * q8, make_float4(r[0], r[1], r[2], r[3]));
                    st4(crow + j0 + 8 * q8 + 4, make_float4(r[4], r[5], r[6], r[7]));
                }
                if (o.img) {   // the result's image as it lies: rows m (M of them), chunk stride M * 16
                    uint32_t hh[4], ll[4];
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) split_bf16x2(r[2 * pp], r[2 * pp + 1], hh[pp], ll[pp]);
                    const uint32_t off = cm_off(m, n0 + j0 + 8 * q8, M * 16);
                    *reinterpret_cast<uint4 *>(o.img + off) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
                    *reinterpret_cast<uint4 *>(o.img + M * N * 2 + off) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                }
            }
        }
    }
    if (!ok) s_tc_fail = 1;
    if (o.img) fence_async_global();
    fence_before();
    __syncthreads();
    if (tid == 0) s_tc_phase = ph ^ 1u;
}

// The chunk's row scalars into scratch sc: beta (rows past L zero) and gc = e^Gamma_C (from the chunk's
// image, the values the reverse chains decayed with).
__device__ void chunk_rows(float *sc, int t0, int L, int h, int H, const float *beta, const unsigned char *im)
{
    const int tid = threadIdx.x;
    if (tid < 64) sc[S_BT + tid] = tid < L ? beta[static_cast<size_t>(t0 + tid) * H + h] : 0.f;
    else if (tid < 64 + KD / 4)
        st4(sc + S_GC + 4 * (tid - 64), ld4(reinterpret_cast<const float *>(im + RIMG_GC) + 4 * (tid - 64)));
    __syncthreads();
}

#define BWD_PLAN_CHECK()                                                                  \
    if (!plan_matches(plan, sig)) {                                                       \
        if (threadIdx.x == 0 && blockIdx.x == 0) record_status(&g_bwd_status, KDA_ERR_INVALID_ARG); \
        return;                                                                           \
    }

// 0. every (chunk, head): dO's bf16 image (rows r x cols v, rows past the chunk zero) into the unit's images;
//    the lanes of a warp take consecutive rows of one 8-column piece, so each store writes 512 contiguous bytes
__global__ void __launch_bounds__(BT) bwd_do_images(const int32_t *plan, PlanSig sig, int H, const uint16_t *dout,
                                                    unsigned char *img)
{
    BWD_PLAN_CHECK();
    const PlanView pv{plan};
    const int n_chunks = pv.n_chunks();
    for (long long unit = blockIdx.x; unit < static_cast<long long>(n_chunks) * H; unit += gridDim.x) {
        const int h = static_cast<int>(unit / n_chunks), c = static_cast<int>(unit % n_chunks);
        const int32_t *cr = pv.chunk(c);
        const int t0 = cr[1], L = cr[2];
        unsigned char *const dst = img + static_cast<size_t>(unit) * RIMG_UNIT + RIMG_DO;
        uint4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int pc = threadIdx.x + i * BT, r = pc & 63, c8 = (pc >> 6) * 8;
            w[i] = r < L ? *reinterpret_cast<const uint4 *>(dout + (static_cast<size_t>(t0 + r) * H + h) * VD + c8)
                         : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int pc = threadIdx.x + i * BT, r = pc & 63, c8 = (pc >> 6) * 8;
            *reinterpret_cast<uint4 *>(dst + cm_off(r, c8, RIMG_CS)) = w[i];
        }
    }
}

// 3. The following summaries, per (head, 16-column slice), last segment first:
//    G_end[j] = dfinal of the sequence ending at b_{j+1}, if one does; otherwise, with p the
//    continuing piece that opens segment j+1,
//    G_end[j] = Qd[j+1] + (P_end(p)^T dfinal[seq] if p ends its sequence, else A[j+1]^T G_end[j+1]).
constexpr int CMP_COLS = 16;                               // gradient columns per CTA
constexpr int CMP_SMEM = (KD * KD + KD * CMP_COLS) * 4;   // the map's matrix and the gradient's column slice

__global__ void __launch_bounds__(BT, 1) bwd_compose(const int32_t *plan, PlanSig sig, int H, const float *A,
                                                  const float *afin, const float *dfinal, const float *Qd,
                                                  float *G_end)
{
    extern __shared__ __align__(16) float csm[];
    BWD_PLAN_CHECK();
    const PlanView pv{plan};
    constexpr int NSL = VD / CMP_COLS;   // slices per head
    const int h = blockIdx.x / NSL, col0 = (blockIdx.x % NSL) * CMP_COLS;
    const int S = pv.S(), N = pv.N(), T = pv.T();
    const int32_t *cu = pv.cu();
    const int tid = threadIdx.x;
    for (int j = S - 1; j >= 0; --j) {
        const int b = pv.bounds()[j + 1];
        float *out = G_end + (static_cast<size_t>(j) * H + h) * SQ;
        int ends = -1;   // the sequence ending exactly at b
        for (int s = 0; s < N; ++s)
            if (cu[s + 1] == b) ends = s;
        if (ends >= 0 || b == T) {
            const float *df = (dfinal && ends >= 0) ? dfinal + (static_cast<size_t>(ends) * H + h) * SQ : nullptr;
            for (int e = tid; e < KD * CMP_COLS; e += BT) {
                const int r = e / CMP_COLS, c = col0 + e % CMP_COLS;
                out[r * VD + c] = df ? df[r * VD + c] : 0.f;
            }
            __syncthreads();
            continue;
        }
        const int p = pv.seg(j + 1)[2];            // first piece of segment j + 1: it continues a sequence
        const int32_t *pc = pv.piece(p);
        const float *qd = Qd + (static_cast<size_t>(j + 1) * H + h) * SQ;
        const float *Mt;                            // the transposed map's matrix and the gradient it acts on
        const float *gin;
        if (pc[PC_FLAGS] & KDA_PIECE_SEQ_END) {
            Mt = afin + (static_cast<size_t>(pc[PC_FIN]) * H + h) * KD * KD;
            gin = dfinal ? dfinal + (static_cast<size_t>(pc[PC_SEQ]) * H + h) * SQ : nullptr;
        } else {
            Mt = A + (static_cast<size_t>(j + 1) * H + h) * KD * KD;
            gin = G_end + (static_cast<size_t>(j + 1) * H + h) * SQ;
        }
        // out[r][c] = qd[r][c] + sum_i Mt[i][r] gin[i][c]  (2 rows x 4 columns per thread), with Mt and this
        // CTA's column slice of gin staged in shared memory first (every 16-byte load of a thread in flight)
        const int rr = (tid >> 2) * 2, cc = col0 + (tid & 3) * 4;
        float *const sM = csm, *const sG = csm + KD * KD;
        if (gin) {
            float4 mv[16], gv[2];
#pragma unroll
            for (int i = 0; i < 16; ++i) mv[i] = ld4(Mt + 4 * (tid + i * BT));
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = tid + i * BT;   // row e / 4, columns 4 (e % 4) .. + 3 of the slice
                gv[i] = ld4(gin + (e >> 2) * VD + col0 + 4 * (e & 3));
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) st4(sM + 4 * (tid + i * BT), mv[i]);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = tid + i * BT;
                st4(sG + (e >> 2) * CMP_COLS + 4 * (e & 3), gv[i]);
            }
        }
        float acc[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a) {
            const float4 q4 = ld4(qd + (rr + a) * VD + cc);
            acc[a][0] = q4.x;
            acc[a][1] = q4.y;
            acc[a][2] = q4.z;
            acc[a][3] = q4.w;
        }
        __syncthreads();   // the staged operands are in; every read of G_end[j + 1] is done before G_end[j]
                           // is written (other slices of the same rows belong to other CTAs)
        if (gin) {
#pragma unroll 8
            for (int i = 0; i < KD; ++i) {
                const float2 m2 = *reinterpret_cast<const float2 *>(sM + i * KD + rr);
                const float4 x4 = ld4(sG + i * CMP_COLS + (cc - col0));
                const float m[2] = {m2.x, m2.y}, x[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) acc[a][bb] = fmaf(m[a], x[bb], acc[a][bb]);
            }
        }
#pragma unroll
        for (int a = 0; a < 2; ++a) st4(out + (rr + a) * VD + cc, make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]));
        __syncthreads();
    }
}

// 5. every (chunk, head): the input gradients of the chunk's rows from (X_c, G_c, dO)
__global__ void __launch_bounds__(BT, 1) bwd_grads(const int32_t *plan, PlanSig sig, int H, const uint16_t *q,
                                                const uint16_t *k, const uint16_t *v, const float *g,
                                                const float *beta, float scale, const uint16_t *dout,
                                                const float *xs, const float *gs, const float *S_in,
                                                const float *fin_out, const float *terms, const unsigned char *img,
                                                float *dq, float *dk, float *dv, float *dg, float *dbeta,
                                                float *scratch)
{
    BWD_PLAN_CHECK();
    tc_begin();
    const PlanView pv{plan};
    float *sc = scratch + static_cast<size_t>(blockIdx.x) * SCRATCH_FLOATS;
    const int n_chunks = pv.n_chunks();
    const int tid = threadIdx.x;
    for (int unit = blockIdx.x; unit < n_chunks * H; unit += gridDim.x) {
        const int h = unit / n_chunks, c = unit % n_chunks;
        const int32_t *cr = pv.chunk(c);
        const int t0 = cr[1], L = cr[2];
        const unsigned char *im = img + static_cast<size_t>(unit) * RIMG_UNIT;
        chunk_rows(sc, t0, L, h, H, beta, im);
        const float *tm = terms + static_cast<size_t>(unit) * BT_FLOATS;   // Ut, S
        // Every operand comes as a bf16 hi/lo image by bulk copies: X (the chunk's start state) and DG = Dc G
        // (G its end-state gradient) as the images of X^T and DG^T the chains recorded (rows v, cols k); Kh,
        // QK, Qt, W (as W^T), dO, T, Diag(beta) Kt and Diag(beta) V as the chunk's operand images; and every
        // product whose result feeds another leaves its result as an image
        const unsigned char *const xt = reinterpret_cast<const unsigned char *>(xs + (static_cast<size_t>(h) * n_chunks + c) * SQ);
        const unsigned char *const dgt = reinterpret_cast<const unsigned char *>(gs + (static_cast<size_t>(h) * n_chunks + c) * SQ);
        // the state after the chunk: the next chunk's recorded image, or the piece's end state (FP32 K x V: the
        // final state of a sequence that ends there, else the state entering the next segment)
        const unsigned char *xn_img = nullptr;
        const float *xn = nullptr;
        {
            const int32_t *pc = pv.piece(cr[0]);
            if (cr[3] + 1 < (pc[PC_LEN] + CH - 1) / CH) xn_img = xt + SQ * 4;
            else if (pc[PC_FLAGS] & KDA_PIECE_SEQ_END) xn = fin_out + (static_cast<size_t>(pc[PC_SEQ]) * H + h) * SQ;
            else xn = S_in + (static_cast<size_t>(pc[PC_SEG] + 1) * H + h) * SQ;
        }
        unsigned char *const sci = reinterpret_cast<unsigned char *>(sc);
        unsigned char *const ui = sci + 4 * S_UI, *const dqki = sci + 4 * S_DQKI;
        const unsigned char *const ti = im + RIMG_T, *const bkti = im + RIMG_BKT;   // T, Diag(beta) Kt
        unsigned char *const dui = sci + 4 * S_DUI, *const dwi = sci + 4 * S_DWI, *const dti = sci + 4 * S_DTI;
        unsigned char *const t64i = sci + 4 * S_T64I, *const dmi = sci + 4 * S_DMI;
        float *dKh = sc + S_DKH, *dQt = sc + S_DQT, *dM = sc + S_DM, *dKt = sc + S_DKT;
        const Term none = term(nullptr, nullptr);
        __syncthreads();
        // U = Ut - W X (W from the image of W^T as it lies)
        product<64, VD, KD, true, true>(term(im + RIMG_W, xt), none,
                                        out_img(out(nullptr, 0, -1.f, tm + BT_UT, VD), ui));
        // dQK = lower(dO U^T)
        product<64, 64, VD, false, true, 0, false, false, 1>(term(im + RIMG_DO, ui, true, false), none,
                                                             out_img(out(nullptr, 0), dqki));
        // dU = Kh DG + QK^T dO
        product<64, VD, KD, false, true, 64, true, false>(term(im + RIMG_KH, dgt),
                                                          term(im + RIMG_QK, im + RIMG_DO, false, true),
                                                          out_img(out(nullptr, 0), dui));
        // dKh = U DG^T + dQK^T Qt
        product<64, KD, VD, false, false, 64, true, false>(term(ui, dgt), term(dqki, im + RIMG_QT),
                                                           out(dKh, KD));
        // dGamma_C[k] = gc[k] sum_v G[k][v] (X + Kh^T U)[k][v] = sum_v DG[k][v] X'[k][v] / gc[k], with
        // X' = Diag(gc) (X + Kh^T U) the state after the chunk (images read as hi + lo): each thread takes the 8
        // columns k of chunk kc for 8 rows v of group vg, then the 16 groups of a half-warp are summed
        {
            const int kc = tid >> 4, vg = tid & 15;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
            for (int i = 0; i < 8; ++i) {
                const int vv = vg * 8 + i;
                const uint32_t o = cm_off(vv, kc * 8, 2048);
                const uint4 dh = *reinterpret_cast<const uint4 *>(dgt + o), dl = *reinterpret_cast<const uint4 *>(dgt + 32768 + o);
                float d[8], dlo[8], xv[8];
                bf16x8(dh, d);
                bf16x8(dl, dlo);
                if (xn_img) {
                    float xlo[8];
                    bf16x8(*reinterpret_cast<const uint4 *>(xn_img + o), xv);
                    bf16x8(*reinterpret_cast<const uint4 *>(xn_img + 32768 + o), xlo);
#pragma unroll
                    for (int e = 0; e < 8; ++e) xv[e] += xlo[e];
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) xv[e] = xn[(kc * 8 + e) * VD + vv];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(d[e] + dlo[e], xv[e], acc[e]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
#pragma unroll
                for (int sh = 8; sh > 0; sh >>= 1) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], sh);
            }
            if (vg == 0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) sc[S_DGC + kc * 8 + e] = acc[e] / sc[S_GC + kc * 8 + e];
            }
        }
        // dQt = dO X^T + dQK Kh
        product<64, KD, VD, false, false, 64, false, false>(term(im + RIMG_DO, xt, true, false),
                                                            term(dqki, im + RIMG_KH), out(dQt, KD));
        // dW = -dU X^T
        product<64, KD, VD, false, false>(term(dui, xt), none, out_img(out(nullptr, 0, -1.f), dwi));
        // dT = dW (beta Kt)^T + dU (beta V)^T
        product<64, 64, KD, false, true, VD, false, true>(term(dwi, bkti),
                                                          term(dui, im + RIMG_BV), out_img(out(nullptr, 0), dti));
        // d(beta Kt) = T^T dW, d(beta V) = T^T dU
        // (one product: B = [dW | dU], N = 256)
        product<64, KD + VD, 64, true, false>(term(ti, dwi, false, false, dui), none, out(sc + S_DBKV, KD + VD));
        // dM = strictly_lower(-T^T dT T^T)
        product<64, 64, 64, true, false>(term(ti, dti), none, out_img(out(nullptr, 0), t64i));
        product<64, 64, 64, false, true, 0, false, false, 2>(term(t64i, ti), none,
                                                             out_img(out(dM, 64, -1.f), dmi));
        // dKt = beta (d(beta Kt) + dM Kh);  dKh += dM^T (beta Kt);  dv = beta d(beta V)
        product<64, KD, 64, false, false>(term(dmi, im + RIMG_KH), none,
                                          out(dKt, KD, 1.f, sc + S_DBKV, KD + VD, nullptr, sc + S_BT));
        product<64, KD, 64, true, false>(term(dmi, bkti), none, out(dKh, KD, 1.f, dKh, KD));
        __syncthreads();
        // The rows' input gradients in one pass.  Each thread holds rows 8 rg .. 8 rg + 7 and columns
        // 4 cq .. 4 cq + 3 (of K, and of V for v and d(beta V); of the 64-wide dM and S rows on lanes cq < 16).
        // Gamma = cumulative g down the rows (the row groups' totals met in shared memory); per row, with
        // E = e^Gamma and Ei = e^-Gamma:
        //   dq = scale E dQt,  dk = E dKt + Ei dKh,  dv = beta d(beta V),
        //   dbeta = rowsum(d(beta Kt) E k) + rowsum(d(beta V) v) + rowsum(dM S)  (a warp sum per row),
        //   dGamma = Kt dKt - Kh dKh + Qt dQt = k (E dKt - Ei dKh) + q dq  (+ dGamma_C on the last row),
        // and dg is its reverse cumulative sum (the row groups' totals met in shared memory again).
        {
            extern __shared__ __align__(16) float bsm[];
            float4 *const tot = reinterpret_cast<float4 *>(bsm);   // [row group][channel quad]
            const int cq = tid & 31, rg = tid >> 5;
            float4 gam[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = rg * 8 + j;
                gam[j] = r < L ? ld4(g + (static_cast<size_t>(t0 + r) * H + h) * KD + 4 * cq) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc = add4(acc, gam[j]);
                    gam[j] = acc;
                }
                tot[rg * 32 + cq] = acc;
                __syncthreads();
                float4 off = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int g2 = 0; g2 < 7; ++g2) {
                    const float4 t = tot[g2 * 32 + cq];
                    if (g2 < rg) off = add4(off, t);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) gam[j] = add4(gam[j], off);
                __syncthreads();   // the totals are read: the suffix sums below reuse the array
            }
            float4 suf[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = rg * 8 + j;
                const bool live = r < L;
                const size_t gi = (static_cast<size_t>(t0 + r) * H + h) * KD + 4 * cq;   // (V = K columns)
                const int e = r * KD + 4 * cq;
                const uint2 kw = live ? *reinterpret_cast<const uint2 *>(k + gi) : make_uint2(0u, 0u);
                const uint2 qw = live ? *reinterpret_cast<const uint2 *>(q + gi) : make_uint2(0u, 0u);
                const uint2 vw = live ? *reinterpret_cast<const uint2 *>(v + gi) : make_uint2(0u, 0u);
                const float4 dkt = ld4(dKt + e), dkh = ld4(dKh + e), dqt = ld4(dQt + e);
                const float4 dbk = ld4(sc + S_DBKV + r * (KD + VD) + 4 * cq), dbv = ld4(sc + S_DBKV + r * (KD + VD) + KD + 4 * cq);
                float4 ms = make_float4(0.f, 0.f, 0.f, 0.f), sv = ms;
                if (cq < 16) {
                    ms = ld4(dM + r * 64 + 4 * cq);
                    sv = ld4(tm + BT_S + r * 64 + 4 * cq);
                }
                const float4 G = gam[j];
                const float4 ea = make_float4(expf(G.x), expf(G.y), expf(G.z), expf(G.w));
                const float4 ei = make_float4(expf(-G.x), expf(-G.y), expf(-G.z), expf(-G.w));
                const float4 a = mul4(ea, dkt), b = mul4(ei, dkh);
                const float4 dqv = scl4(scale, mul4(ea, dqt));
                const float4 kf = bf4(kw);
                const float br = sc[S_BT + r];
                if (live) {
                    st4(dq + gi, dqv);
                    st4(dk + gi, add4(a, b));
                    st4(dv + gi, scl4(br, dbv));
                }
                suf[j] = add4(mul4(kf, sub4(a, b)), mul4(bf4(qw), dqv));
                const float part = warp_sum(dot4(dbk, mul4(ea, kf)) + dot4(dbv, bf4(vw)) + dot4(ms, sv));
                if (cq == 0 && live) dbeta[static_cast<size_t>(t0 + r) * H + h] = part;
            }
            if (L - 1 >= rg * 8 && L - 1 < rg * 8 + 8) {
                const float4 dgc = ld4(sc + S_DGC + 4 * cq);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (rg * 8 + j == L - 1) suf[j] = add4(suf[j], dgc);
            }
#pragma unroll
            for (int j = 6; j >= 0; --j) suf[j] = add4(suf[j], suf[j + 1]);
            tot[rg * 32 + cq] = suf[0];
            __syncthreads();
            float4 off = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int g2 = 1; g2 < 8; ++g2) {
                const float4 t = tot[g2 * 32 + cq];
                if (g2 > rg) off = add4(off, t);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = rg * 8 + j;
                if (r < L) st4(dg + (static_cast<size_t>(t0 + r) * H + h) * KD + 4 * cq, add4(suf[j], off));
            }
        }
        __syncthreads();
    }
    tc_end();
}

}  // namespace

size_t backward_scratch_floats() { return static_cast<size_t>(SCRATCH_FLOATS); }

cudaError_t launch_backward(const int32_t *plan_host, const int32_t *plan_dev, int H, const uint16_t *q,
                            const uint16_t *k, const uint16_t *v, const float *g, const float *beta, float scale,
                            const uint16_t *dout, const float *dfinal, const float *A, const float *afin,
                            const float *xs, float *gs, float *G_end, float *Qd, const float *S_in,
                            const float *fin_out, float *terms, unsigned char *img, float *scratch, int grid, float *dq,
                            float *dk, float *dv, float *dg, float *dbeta, float *dh0, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    const PlanSig sig = plan_sig(plan_host);
    cudaError_t err = set_dynamic_smem(reinterpret_cast<const void *>(bwd_grads), static_cast<int>(BWD_SMEM));
    if (err != cudaSuccess) return err;
    const long long n_units = static_cast<long long>(pv.n_chunks()) * H;
    if (n_units > 0) {
        const unsigned blocks = static_cast<unsigned>(n_units < 4096 ? n_units : 4096);
        bwd_do_images<<<blocks, BT, 0, stream>>>(plan_dev, sig, H, dout, img);
        err = cudaGetLastError();
    }
    if (err != cudaSuccess) return err;
    if (pv.n_cont() > 0) {
        err = launch_reverse_tc(plan_host, plan_dev, H, false, img, dfinal, G_end, Qd, gs, dh0, stream);
        if (err != cudaSuccess) return err;
    }
    if ((err = set_dynamic_smem(reinterpret_cast<const void *>(bwd_compose), CMP_SMEM)) != cudaSuccess) return err;
    bwd_compose<<<H * (VD / CMP_COLS), BT, CMP_SMEM, stream>>>(plan_dev, sig, H, A, afin, dfinal, Qd, G_end);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    err = launch_reverse_tc(plan_host, plan_dev, H, true, img, dfinal, G_end, Qd, gs, dh0, stream);
    if (err != cudaSuccess) return err;
    bwd_grads<<<grid, BT, BWD_SMEM, stream>>>(plan_dev, sig, H, q, k, v, g, beta, scale, dout, xs, gs, S_in, fin_out,
                                              terms, img, dq, dk, dv, dg, dbeta, scratch);
    return cudaGetLastError();
}

int take_backward_status()
{
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_bwd_status, &z, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return v;
}

}  // namespace kda
