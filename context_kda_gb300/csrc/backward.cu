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
//  0. every (chunk, head) in parallel: the chunk's terms that the chains need (W, Ut, Kh, Qt, QK, Dc);
//  1. every piece from its true incoming state (h0, or S_in of its segment), recording each chunk's
//     start state X_c;
//  2. every piece that continues a sequence, backwards from a zero end gradient: the gradient of its
//     incoming state through its own outputs, Qd (the qhat do^T sum of the pages' summaries);
//  3. the following summaries, last segment first: the gradient of the state crossing the end of
//     segment j is dfinal of a sequence that ends there, or Qd[j+1] plus the transposed map of the
//     continuing piece of segment j+1 (A[j+1]^T, or P_end^T of a piece that ends its sequence
//     there, on dfinal) applied to the gradient at that piece's end;
//  4. every piece backwards from its true end gradient, recording each chunk's end gradient G_c and
//     giving dh0 at a sequence start;
//  5. every (chunk, head) in parallel: dq, dk, dv, dg, dbeta from (X_c, G_c, dO).
//
// This implementation computes in FP32 on the CUDA cores: each CTA keeps its chunk's matrices in a
// private scratch area in global memory (L2-resident) and runs every product by staging both
// operands in shared memory, which keeps every step a literal transcription of the formulas above.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int BT = 256;                      // threads per CTA
constexpr int CK = 64 * KD;                  // a 64 x 128 chunk matrix
constexpr int CC = 64 * 64;                  // a 64 x 64 chunk matrix
constexpr int SQ = KD * VD;                  // a 128 x 128 state

__device__ int g_bwd_status;

// Per-CTA scratch (floats): three states, twenty 64 x 128 and eight 64 x 64 matrices, vectors.
enum : int {
    S_X = 0, S_G = S_X + SQ, S_Y = S_G + SQ,
    S_KT = S_Y + SQ, S_KH = S_KT + CK, S_QT = S_KH + CK, S_VF = S_QT + CK, S_E = S_VF + CK, S_EI = S_E + CK,
    S_W = S_EI + CK, S_UT = S_W + CK, S_U = S_UT + CK, S_DO = S_U + CK, S_DU = S_DO + CK, S_DKH = S_DU + CK,
    S_DQT = S_DKH + CK, S_DW = S_DQT + CK, S_DKT = S_DW + CK, S_BKT = S_DKT + CK, S_BV = S_BKT + CK,
    S_DBKT = S_BV + CK, S_DBV = S_DBKT + CK, S_TMP = S_DBV + CK,
    S_M = S_TMP + CK, S_S = S_M + CC, S_T = S_S + CC, S_QK = S_T + CC, S_DQK = S_QK + CC, S_DT = S_DQK + CC,
    S_DM = S_DT + CC, S_T64 = S_DM + CC,
    S_GC = S_T64 + CC, S_BT = S_GC + KD, S_DGC = S_BT + 64, S_DBETA = S_DGC + KD,
    SCRATCH_FLOATS = S_DBETA + 64
};

// The terms a chain step needs, stored per (head, chunk) by the terms pass (floats): W, Ut, Kh, Qt
// (64 x 128 each), QK (64 x 64), exp(Gamma_C) (128).
enum : int { TM_W = 0, TM_UT = CK, TM_KH = 2 * CK, TM_QT = 3 * CK, TM_QK = 4 * CK, TM_GC = 4 * CK + CC,
             TERMS_FLOATS = TM_GC + KD };

// A matrix operand in global scratch: element (r, c) = t ? p[c * ld + r] : p[r * ld + c].
struct Mat {
    const float *p;
    int ld;
    bool t;
};
__device__ __forceinline__ Mat mat(const float *p, int ld) { return Mat{p, ld, false}; }
__device__ __forceinline__ Mat tr(const float *p, int ld) { return Mat{p, ld, true}; }

// Dynamic shared memory of the backward's kernels: both operands of one product, k-major.
constexpr int SM_PAD = 4;
constexpr int SM_LD = 128 + SM_PAD;
constexpr size_t BWD_SMEM = 2ull * 128 * SM_LD * sizeof(float);

// Micro-tile product over operands already in shared memory: As[k][m] (M x K), Bs[k][n] (K x N);
// thread (ty, tx) of a 16 x 16 grid computes rows ty*MR .. +MR and columns tx*NR .. +NR.
template <int MR, int NR>
__device__ __forceinline__ void gemm_core(int K, const float *As, const float *Bs, float *C, int ldc, float alpha,
                                          bool acc)
{
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float c[MR][NR];
#pragma unroll
    for (int i = 0; i < MR; ++i)
#pragma unroll
        for (int j = 0; j < NR; ++j) c[i][j] = 0.f;
    for (int k = 0; k < K; ++k) {
        float a[MR], b[NR];
#pragma unroll
        for (int i = 0; i < MR; i += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(As + k * SM_LD + ty * MR + i);
            a[i] = v.x; a[i + 1] = v.y; a[i + 2] = v.z; a[i + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < NR; j += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(Bs + k * SM_LD + tx * NR + j);
            b[j] = v.x; b[j + 1] = v.y; b[j + 2] = v.z; b[j + 3] = v.w;
        }
#pragma unroll
        for (int i = 0; i < MR; ++i)
#pragma unroll
            for (int j = 0; j < NR; ++j) c[i][j] = fmaf(a[i], b[j], c[i][j]);
    }
#pragma unroll
    for (int i = 0; i < MR; ++i)
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            float *d = C + (ty * MR + i) * ldc + tx * NR + j;
            *d = alpha * c[i][j] + (acc ? *d : 0.f);
        }
}

// C(m, n) = alpha * sum_k A(m, k) B(k, n) (+ C(m, n) when acc), for an M x N result (M, N in {64, 128})
// and K-long sums (K in {64, 128}), operands 16-byte aligned with leading dimensions a multiple of 4, by
// all threads of the CTA: both operands are staged in shared memory
// (k-major) in one pass, then every thread accumulates its micro-tile over the whole K.
__device__ void gemm(int M, int N, int K, Mat A, Mat B, float *C, int ldc, float alpha, bool acc)
{
    extern __shared__ __align__(16) float bsm[];
    float *As = bsm, *Bs = bsm + 128 * SM_LD;
    const int tid = threadIdx.x;
    __syncthreads();
    // 16-byte loads along the contiguous index; M, N, K are powers of two (64 or 128, K >= 64)
    const int lm = __ffs(M) - 1, ln = __ffs(N) - 1, lk = __ffs(K) - 1;
    if (A.t) {            // A(m, k) = p[k * ld + m]: rows of m, stored as they come
        for (int e = tid; e < (K * M) >> 2; e += BT) {
            const int k = e >> (lm - 2), m4 = (e & ((M >> 2) - 1)) << 2;
            *reinterpret_cast<float4 *>(As + k * SM_LD + m4) = *reinterpret_cast<const float4 *>(A.p + k * A.ld + m4);
        }
    } else {              // A(m, k) = p[m * ld + k]: rows of k, transposed into As; a warp takes 16 rows m
                          // x 2 vectors, so its scattered stores fall in 32 distinct banks
        for (int e = tid; e < (K * M) >> 2; e += BT) {
            const int rest = e >> 4, kv = rest & ((K >> 2) - 1);
            const int m = ((rest >> (lk - 2)) << 4) | (e & 15), k4 = kv << 2;
            const float4 v = *reinterpret_cast<const float4 *>(A.p + m * A.ld + k4);
            As[(k4 + 0) * SM_LD + m] = v.x;
            As[(k4 + 1) * SM_LD + m] = v.y;
            As[(k4 + 2) * SM_LD + m] = v.z;
            As[(k4 + 3) * SM_LD + m] = v.w;
        }
    }
    if (B.t) {            // B(k, n) = p[n * ld + k]: rows of k, transposed into Bs (16 rows n x 2 vectors a warp)
        for (int e = tid; e < (K * N) >> 2; e += BT) {
            const int rest = e >> 4, kv = rest & ((K >> 2) - 1);
            const int n = ((rest >> (lk - 2)) << 4) | (e & 15), k4 = kv << 2;
            const float4 v = *reinterpret_cast<const float4 *>(B.p + n * B.ld + k4);
            Bs[(k4 + 0) * SM_LD + n] = v.x;
            Bs[(k4 + 1) * SM_LD + n] = v.y;
            Bs[(k4 + 2) * SM_LD + n] = v.z;
            Bs[(k4 + 3) * SM_LD + n] = v.w;
        }
    } else {              // B(k, n) = p[k * ld + n]: rows of n, stored as they come
        for (int e = tid; e < (K * N) >> 2; e += BT) {
            const int k = e >> (ln - 2), n4 = (e & ((N >> 2) - 1)) << 2;
            *reinterpret_cast<float4 *>(Bs + k * SM_LD + n4) = *reinterpret_cast<const float4 *>(B.p + k * B.ld + n4);
        }
    }
    __syncthreads();
    if (M == 128 && N == 128) gemm_core<8, 8>(K, As, Bs, C, ldc, alpha, acc);
    else if (M == 128) gemm_core<8, 4>(K, As, Bs, C, ldc, alpha, acc);
    else if (N == 128) gemm_core<4, 8>(K, As, Bs, C, ldc, alpha, acc);
    else gemm_core<4, 4>(K, As, Bs, C, ldc, alpha, acc);
    __syncthreads();
}

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// The chunk's terms into scratch sc (rows past L are zero): Kt, Kh, Qt, V, E = e^Gamma, Ei = e^-Gamma,
// gc = e^Gamma_C, beta, M, S = strictly_lower(Kt Kh^T), T, W, Ut, QK, and Diag(beta) Kt, Diag(beta) V.
__device__ void chunk_terms(float *sc, int t0, int L, int h, int H, const uint16_t *q, const uint16_t *k,
                            const uint16_t *v, const float *g, const float *beta, float scale)
{
    const int tid = threadIdx.x;
    float *Kt = sc + S_KT, *Kh = sc + S_KH, *Qt = sc + S_QT, *Vf = sc + S_VF, *E = sc + S_E, *Ei = sc + S_EI;
    for (int e = tid; e < CK; e += BT) {
        const int r = e >> 7, c = e & 127;
        const bool ok = r < L;
        const size_t gi = (static_cast<size_t>(t0 + r) * H + h) * KD + c;
        Kt[e] = ok ? bf(k[gi]) : 0.f;       // raw k for now
        Qt[e] = ok ? bf(q[gi]) : 0.f;       // raw q for now
        Vf[e] = ok ? bf(v[gi]) : 0.f;
        E[e] = ok ? g[gi] : 0.f;            // g for now
    }
    for (int r = tid; r < 64; r += BT) sc[S_BT + r] = r < L ? beta[static_cast<size_t>(t0 + r) * H + h] : 0.f;
    __syncthreads();
    if (tid < KD) {                           // Gamma: cumulative sum down the rows, per channel
        float acc = 0.f;
        for (int r = 0; r < 64; ++r) {
            acc += E[r * KD + tid];
            E[r * KD + tid] = acc;
        }
        sc[S_GC + tid] = expf(acc);
    }
    __syncthreads();
    for (int e = tid; e < CK; e += BT) {
        const float G = E[e], ex = expf(G), exi = expf(-G), kv = Kt[e];
        Kt[e] = ex * kv;
        Kh[e] = exi * kv;
        Qt[e] = scale * ex * Qt[e];
        E[e] = ex;
        Ei[e] = exi;
    }
    __syncthreads();
    gemm(64, 64, KD, mat(Kt, KD), tr(Kh, KD), sc + S_S, 64, 1.f, false);
    gemm(64, 64, KD, mat(Qt, KD), tr(Kh, KD), sc + S_QK, 64, 1.f, false);
    for (int e = tid; e < CC; e += BT) {
        const int r = e >> 6, i = e & 63;
        const float s = i < r ? sc[S_S + e] : 0.f;
        sc[S_S + e] = s;
        sc[S_M + e] = sc[S_BT + r] * s;
        if (i > r) sc[S_QK + e] = 0.f;
    }
    for (int e = tid; e < CK; e += BT) {
        const float b = sc[S_BT + (e >> 7)];
        sc[S_BKT + e] = b * Kt[e];
        sc[S_BV + e] = b * Vf[e];
    }
    __syncthreads();
    // T = (I + M)^-1 by forward substitution, one column per thread: T[j][j] = 1,
    // T[r][j] = -sum_{j <= i < r} M[r][i] T[i][j]; M in shared memory (read by every thread alike),
    // the column in registers
    {
        extern __shared__ __align__(16) float bsm[];
        for (int e = tid; e < CC; e += BT) bsm[e] = sc[S_M + e];
        __syncthreads();
        if (tid < 64) {
            const int j = tid;
            float t[64];
#pragma unroll
            for (int r = 0; r < 64; ++r) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < r; ++i) s = fmaf(bsm[r * 64 + i], t[i], s);
                t[r] = r < j ? 0.f : (r == j ? 1.f : -s);
            }
#pragma unroll
            for (int r = 0; r < 64; ++r) sc[S_T + r * 64 + j] = t[r];
        }
        __syncthreads();
    }
    gemm(64, KD, 64, mat(sc + S_T, 64), mat(sc + S_BKT, KD), sc + S_W, KD, 1.f, false);
    gemm(64, VD, 64, mat(sc + S_T, 64), mat(sc + S_BV, VD), sc + S_UT, VD, 1.f, false);
}

// The chunk's output gradients rows into scratch (zero past L), bf16 -> fp32.
__device__ void load_do(float *sc, int t0, int L, int h, int H, const uint16_t *dout)
{
    for (int e = threadIdx.x; e < CK; e += BT) {
        const int r = e >> 7, c = e & 127;
        sc[S_DO + e] = r < L ? bf(dout[(static_cast<size_t>(t0 + r) * H + h) * VD + c]) : 0.f;
    }
    __syncthreads();
}

// X <- Dc (X + Kh^T (Ut - W X)), the chunk's terms at tm
__device__ void forward_step(float *sc, const float *tm)
{
    float *X = sc + S_X, *U = sc + S_U;
    for (int e = threadIdx.x; e < CK; e += BT) U[e] = tm[TM_UT + e];
    gemm(64, VD, KD, mat(tm + TM_W, KD), mat(X, VD), U, VD, -1.f, true);
    gemm(KD, VD, 64, tr(tm + TM_KH, KD), mat(U, VD), X, VD, 1.f, true);
    for (int e = threadIdx.x; e < SQ; e += BT) X[e] *= tm[TM_GC + (e >> 7)];
    __syncthreads();
}

// G <- DG + Qt^T dO - W^T (Kh DG + QK^T dO), DG = Dc G (the gradient reaching the chunk start), the chunk's
// terms at tm
__device__ void reverse_step(float *sc, const float *tm)
{
    float *G = sc + S_G, *DG = sc + S_Y, *dU = sc + S_DU;
    for (int e = threadIdx.x; e < SQ; e += BT) DG[e] = tm[TM_GC + (e >> 7)] * G[e];
    __syncthreads();
    gemm(64, VD, KD, mat(tm + TM_KH, KD), mat(DG, VD), dU, VD, 1.f, false);
    gemm(64, VD, 64, tr(tm + TM_QK, 64), mat(sc + S_DO, VD), dU, VD, 1.f, true);
    for (int e = threadIdx.x; e < SQ; e += BT) G[e] = DG[e];
    __syncthreads();
    gemm(KD, VD, 64, tr(tm + TM_QT, KD), mat(sc + S_DO, VD), G, VD, 1.f, true);
    gemm(KD, VD, 64, tr(tm + TM_W, KD), mat(dU, VD), G, VD, -1.f, true);
}

// Plan helpers
struct PieceInfo {
    int start, len, seq, seg, flags, nch, c0;   // c0: global index of the piece's first chunk
};
__device__ PieceInfo piece_info(const PlanView &pv, int p)
{
    const int32_t *pc = pv.piece(p);
    PieceInfo pi{pc[PC_START], pc[PC_LEN], pc[PC_SEQ], pc[PC_SEG], pc[PC_FLAGS], (pc[PC_LEN] + CH - 1) / CH, 0};
    int c0 = 0;
    for (int i = 0; i < p; ++i) c0 += (pv.piece(i)[PC_LEN] + CH - 1) / CH;
    pi.c0 = c0;
    return pi;
}

#define BWD_PLAN_CHECK()                                                                  \
    if (!plan_matches(plan, sig)) {                                                       \
        if (threadIdx.x == 0 && blockIdx.x == 0) record_status(&g_bwd_status, KDA_ERR_INVALID_ARG); \
        return;                                                                           \
    }

// 0. every (chunk, head) in parallel: the terms the chains need, stored at terms[h][c]
__global__ void __launch_bounds__(BT) bwd_terms(const int32_t *plan, PlanSig sig, int H, const uint16_t *q,
                                                const uint16_t *k, const uint16_t *v, const float *g,
                                                const float *beta, float scale, float *terms, float *scratch)
{
    BWD_PLAN_CHECK();
    const PlanView pv{plan};
    float *sc = scratch + static_cast<size_t>(blockIdx.x) * SCRATCH_FLOATS;
    const int n_chunks = pv.n_chunks();
    for (int unit = blockIdx.x; unit < n_chunks * H; unit += gridDim.x) {
        const int h = unit / n_chunks, c = unit % n_chunks;
        const int32_t *cr = pv.chunk(c);
        chunk_terms(sc, cr[1], cr[2], h, H, q, k, v, g, beta, scale);
        float *tm = terms + static_cast<size_t>(unit) * TERMS_FLOATS;
        for (int e = threadIdx.x; e < CK; e += BT) {
            tm[TM_W + e] = sc[S_W + e];
            tm[TM_UT + e] = sc[S_UT + e];
            tm[TM_KH + e] = sc[S_KH + e];
            tm[TM_QT + e] = sc[S_QT + e];
        }
        for (int e = threadIdx.x; e < CC; e += BT) tm[TM_QK + e] = sc[S_QK + e];
        for (int e = threadIdx.x; e < KD; e += BT) tm[TM_GC + e] = sc[S_GC + e];
        __syncthreads();
    }
}

// 1. every piece from its true incoming state, recording X_c = xs[h][c] for each of its chunks
__global__ void __launch_bounds__(BT) bwd_states(const int32_t *plan, PlanSig sig, int H, const float *terms,
                                                 const float *h0, const float *S_in, float *xs, float *scratch)
{
    BWD_PLAN_CHECK();
    const PlanView pv{plan};
    float *sc = scratch + static_cast<size_t>(blockIdx.x) * SCRATCH_FLOATS;
    const int n_items = pv.n_pieces() * H;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int p = item / H, h = item % H;
        const PieceInfo pi = piece_info(pv, p);
        const float *src = nullptr;
        if (pi.flags & KDA_PIECE_FIRST) {
            if (h0) src = h0 + (static_cast<size_t>(pi.seq) * H + h) * SQ;
        } else {
            src = S_in + (static_cast<size_t>(pi.seg) * H + h) * SQ;
        }
        for (int e = threadIdx.x; e < SQ; e += BT) sc[S_X + e] = src ? src[e] : 0.f;
        __syncthreads();
        for (int ci = 0; ci < pi.nch; ++ci) {
            const size_t unit = static_cast<size_t>(h) * pv.n_chunks() + pi.c0 + ci;
            float *dst = xs + unit * SQ;
            for (int e = threadIdx.x; e < SQ; e += BT) dst[e] = sc[S_X + e];
            forward_step(sc, terms + unit * TERMS_FLOATS);
        }
        __syncthreads();
    }
}

// 2 (LOCAL) / 4 (TRUE). Pieces backwards over their chunks.  LOCAL: pieces that continue a sequence,
// from a zero end gradient; the gradient reaching the piece start is Qd[seg].  TRUE: every piece from
// its true end gradient (dfinal of its sequence when it ends it, else G_end[seg]); records G_c =
// gs[h][c], the gradient of each chunk's end state, and gives dh0 at a sequence start.
template <bool TRUE_PASS>
__global__ void __launch_bounds__(BT) bwd_reverse(const int32_t *plan, PlanSig sig, int H, const float *terms,
                                                  const uint16_t *dout, const float *dfinal, const float *G_end,
                                                  float *Qd, float *gs, float *dh0, float *scratch)
{
    BWD_PLAN_CHECK();
    const PlanView pv{plan};
    float *sc = scratch + static_cast<size_t>(blockIdx.x) * SCRATCH_FLOATS;
    const int n_items = pv.n_pieces() * H;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int p = item / H, h = item % H;
        const PieceInfo pi = piece_info(pv, p);
        if (!TRUE_PASS && !(pi.flags & KDA_PIECE_CONT)) continue;
        const float *src = nullptr;
        if (TRUE_PASS) {
            if (pi.flags & KDA_PIECE_SEQ_END) {
                if (dfinal) src = dfinal + (static_cast<size_t>(pi.seq) * H + h) * SQ;
            } else {
                src = G_end + (static_cast<size_t>(pi.seg) * H + h) * SQ;
            }
        }
        for (int e = threadIdx.x; e < SQ; e += BT) sc[S_G + e] = src ? src[e] : 0.f;
        __syncthreads();
        for (int ci = pi.nch - 1; ci >= 0; --ci) {
            const size_t unit = static_cast<size_t>(h) * pv.n_chunks() + pi.c0 + ci;
            if (TRUE_PASS) {
                float *dst = gs + unit * SQ;
                for (int e = threadIdx.x; e < SQ; e += BT) dst[e] = sc[S_G + e];
            }
            const int t0 = pi.start + ci * CH, L = min(CH, pi.len - ci * CH);
            load_do(sc, t0, L, h, H, dout);
            reverse_step(sc, terms + unit * TERMS_FLOATS);
        }
        __syncthreads();
        float *dst = nullptr;
        if (!TRUE_PASS) dst = Qd + (static_cast<size_t>(pi.seg) * H + h) * SQ;
        else if ((pi.flags & KDA_PIECE_FIRST) && dh0) dst = dh0 + (static_cast<size_t>(pi.seq) * H + h) * SQ;
        if (dst)
            for (int e = threadIdx.x; e < SQ; e += BT) dst[e] = sc[S_G + e];
        __syncthreads();
    }
}

// 3. The following summaries, per (head, 32-column slice), last segment first:
//    G_end[j] = dfinal of the sequence ending at b_{j+1}, if one does; otherwise, with p the
//    continuing piece that opens segment j+1,
//    G_end[j] = Qd[j+1] + (P_end(p)^T dfinal[seq] if p ends its sequence, else A[j+1]^T G_end[j+1]).
__global__ void __launch_bounds__(BT) bwd_compose(const int32_t *plan, PlanSig sig, int H, const float *A,
                                                  const float *afin, const float *dfinal, const float *Qd,
                                                  float *G_end)
{
    BWD_PLAN_CHECK();
    const PlanView pv{plan};
    const int h = blockIdx.x / 4, col0 = (blockIdx.x % 4) * 32;
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
            for (int e = tid; e < KD * 32; e += BT) {
                const int r = e >> 5, c = col0 + (e & 31);
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
        // out[r][c] = qd[r][c] + sum_i Mt[i][r] gin[i][c]  (4 rows x 4 columns per thread)
        const int rr = (tid >> 3) * 4, cc = col0 + (tid & 7) * 4;
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) acc[a][bb] = qd[(rr + a) * VD + cc + bb];
        if (gin)
            for (int i = 0; i < KD; ++i) {
                float m[4], x[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) m[a] = Mt[i * KD + rr + a];
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) x[bb] = gin[i * VD + cc + bb];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) acc[a][bb] = fmaf(m[a], x[bb], acc[a][bb]);
            }
        __syncthreads();   // every read of G_end[j + 1] is done before G_end[j] is written (other slices
                           // of the same rows belong to other CTAs and are not touched here)
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) out[(rr + a) * VD + cc + bb] = acc[a][bb];
        __syncthreads();
    }
}

// 5. every (chunk, head): the input gradients of the chunk's rows from (X_c, G_c, dO)
__global__ void __launch_bounds__(BT) bwd_grads(const int32_t *plan, PlanSig sig, int H, const uint16_t *q,
                                                const uint16_t *k, const uint16_t *v, const float *g,
                                                const float *beta, float scale, const uint16_t *dout,
                                                const float *xs, const float *gs, float *dq, float *dk, float *dv,
                                                float *dg, float *dbeta, float *scratch)
{
    BWD_PLAN_CHECK();
    const PlanView pv{plan};
    float *sc = scratch + static_cast<size_t>(blockIdx.x) * SCRATCH_FLOATS;
    const int n_chunks = pv.n_chunks();
    const int tid = threadIdx.x;
    for (int unit = blockIdx.x; unit < n_chunks * H; unit += gridDim.x) {
        const int h = unit / n_chunks, c = unit % n_chunks;
        const int32_t *cr = pv.chunk(c);
        const int t0 = cr[1], L = cr[2];
        chunk_terms(sc, t0, L, h, H, q, k, v, g, beta, scale);
        load_do(sc, t0, L, h, H, dout);
        float *X = sc + S_X, *G = sc + S_G, *DG = sc + S_Y;
        const float *xsrc = xs + (static_cast<size_t>(h) * n_chunks + c) * SQ;
        const float *gsrc = gs + (static_cast<size_t>(h) * n_chunks + c) * SQ;
        for (int e = tid; e < SQ; e += BT) {
            X[e] = xsrc[e];
            G[e] = gsrc[e];
            DG[e] = sc[S_GC + (e >> 7)] * gsrc[e];
        }
        float *U = sc + S_U, *dU = sc + S_DU, *dKh = sc + S_DKH, *dQt = sc + S_DQT, *dW = sc + S_DW;
        float *dQK = sc + S_DQK, *dT = sc + S_DT, *dM = sc + S_DM, *dKt = sc + S_DKT;
        for (int e = tid; e < CK; e += BT) U[e] = sc[S_UT + e];
        __syncthreads();
        gemm(64, VD, KD, mat(sc + S_W, KD), mat(X, VD), U, VD, -1.f, true);            // U = Ut - W X
        gemm(64, VD, KD, mat(sc + S_KH, KD), mat(DG, VD), dU, VD, 1.f, false);         // dU = Kh DG
        gemm(64, KD, VD, mat(U, VD), tr(DG, VD), dKh, KD, 1.f, false);                  // dKh = U DG^T
        // dGamma_C[k] = sum_c G[k][c] gc[k] (X + Kh^T U)[k][c]: Y = X + Kh^T U in place of DG
        for (int e = tid; e < SQ; e += BT) DG[e] = X[e];
        __syncthreads();
        gemm(KD, VD, 64, tr(sc + S_KH, KD), mat(U, VD), DG, VD, 1.f, true);
        if (tid < KD) {
            float s = 0.f;
            for (int cc = 0; cc < VD; ++cc) s = fmaf(G[tid * VD + cc], DG[tid * VD + cc], s);
            sc[S_DGC + tid] = s * sc[S_GC + tid];
        }
        __syncthreads();
        gemm(64, KD, VD, mat(sc + S_DO, VD), tr(X, VD), dQt, KD, 1.f, false);          // dQt = dO X^T
        gemm(64, 64, VD, mat(sc + S_DO, VD), tr(U, VD), dQK, 64, 1.f, false);          // dO U^T
        for (int e = tid; e < CC; e += BT)
            if ((e & 63) > (e >> 6)) dQK[e] = 0.f;                                      // lower incl. diagonal
        __syncthreads();
        gemm(64, VD, 64, tr(sc + S_QK, 64), mat(sc + S_DO, VD), dU, VD, 1.f, true);    // dU += QK^T dO
        gemm(64, KD, 64, mat(dQK, 64), mat(sc + S_KH, KD), dQt, KD, 1.f, true);         // dQt += dQK Kh
        gemm(64, KD, 64, tr(dQK, 64), mat(sc + S_QT, KD), dKh, KD, 1.f, true);          // dKh += dQK^T Qt
        gemm(64, KD, VD, mat(dU, VD), tr(X, VD), dW, KD, -1.f, false);                  // dW = -dU X^T
        gemm(64, 64, KD, mat(dW, KD), tr(sc + S_BKT, KD), dT, 64, 1.f, false);          // dT = dW (bKt)^T
        gemm(64, 64, VD, mat(dU, VD), tr(sc + S_BV, VD), dT, 64, 1.f, true);            //    + dU (bV)^T
        gemm(64, KD, 64, tr(sc + S_T, 64), mat(dW, KD), sc + S_DBKT, KD, 1.f, false);   // d(bKt) = T^T dW
        gemm(64, VD, 64, tr(sc + S_T, 64), mat(dU, VD), sc + S_DBV, VD, 1.f, false);    // d(bV) = T^T dU
        // dM = strictly_lower(-T^T dT T^T)
        gemm(64, 64, 64, tr(sc + S_T, 64), mat(dT, 64), sc + S_T64, 64, 1.f, false);
        gemm(64, 64, 64, mat(sc + S_T64, 64), tr(sc + S_T, 64), dM, 64, -1.f, false);
        for (int e = tid; e < CC; e += BT)
            if ((e & 63) >= (e >> 6)) dM[e] = 0.f;
        __syncthreads();
        // dKt = beta (d(bKt) + dM Kh);  dKh += dM^T (beta Kt);  dv = beta d(bV)
        gemm(64, KD, 64, mat(dM, 64), mat(sc + S_KH, KD), dKt, KD, 1.f, false);
        gemm(64, KD, 64, tr(dM, 64), mat(sc + S_BKT, KD), dKh, KD, 1.f, true);
        // dbeta = rowsum(d(bKt) Kt) + rowsum(d(bV) V) + rowsum(dM S)
        if (tid < 64) {
            const int r = tid;
            float s = 0.f;
            for (int cc = 0; cc < KD; ++cc) s = fmaf(sc[S_DBKT + r * KD + cc], sc[S_KT + r * KD + cc], s);
            for (int cc = 0; cc < VD; ++cc) s = fmaf(sc[S_DBV + r * VD + cc], sc[S_VF + r * VD + cc], s);
            for (int i = 0; i < 64; ++i) s = fmaf(dM[r * 64 + i], sc[S_S + r * 64 + i], s);
            sc[S_DBETA + r] = s;
        }
        for (int e = tid; e < CK; e += BT) {
            const float b = sc[S_BT + (e >> 7)];
            dKt[e] = b * (sc[S_DBKT + e] + dKt[e]);
        }
        __syncthreads();
        // dGamma = Kt dKt - Kh dKh + Qt dQt (+ dGamma_C on the last row), dg its reverse cumulative sum;
        // dq = scale E dQt, dk = E dKt + Ei dKh, dv = beta d(bV)
        if (tid < KD) {
            float acc = 0.f;
            for (int r = 63; r >= 0; --r) {
                const int e = r * KD + tid;
                float dG = sc[S_KT + e] * dKt[e] - sc[S_KH + e] * dKh[e] + sc[S_QT + e] * dQt[e];
                if (r == L - 1) dG += sc[S_DGC + tid];
                acc += dG;
                if (r < L) dg[(static_cast<size_t>(t0 + r) * H + h) * KD + tid] = acc;
            }
        }
        for (int e = tid; e < CK; e += BT) {
            const int r = e >> 7, cc = e & 127;
            if (r < L) {
                const size_t o = (static_cast<size_t>(t0 + r) * H + h) * KD + cc;
                dq[o] = scale * sc[S_E + e] * dQt[e];
                dk[o] = sc[S_E + e] * dKt[e] + sc[S_EI + e] * dKh[e];
                dv[o] = sc[S_BT + r] * sc[S_DBV + e];
            }
        }
        for (int r = tid; r < L; r += BT) dbeta[static_cast<size_t>(t0 + r) * H + h] = sc[S_DBETA + r];
        __syncthreads();
    }
}

}  // namespace

size_t backward_scratch_floats() { return static_cast<size_t>(SCRATCH_FLOATS); }
size_t backward_terms_floats() { return static_cast<size_t>(TERMS_FLOATS); }

cudaError_t launch_backward(const int32_t *plan_host, const int32_t *plan_dev, int H, const uint16_t *q,
                            const uint16_t *k, const uint16_t *v, const float *g, const float *beta,
                            const float *h0, float scale, const uint16_t *dout, const float *dfinal,
                            const float *A, const float *afin, const float *S_in, float *xs, float *gs,
                            float *G_end, float *Qd, float *terms, float *scratch, int grid, float *dq, float *dk,
                            float *dv, float *dg, float *dbeta, float *dh0, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    const PlanSig sig = plan_sig(plan_host);
    for (auto fn : {reinterpret_cast<const void *>(bwd_terms), reinterpret_cast<const void *>(bwd_states),
                    reinterpret_cast<const void *>(bwd_reverse<false>),
                    reinterpret_cast<const void *>(bwd_reverse<true>), reinterpret_cast<const void *>(bwd_grads)}) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(BWD_SMEM));
        if (e != cudaSuccess) return e;
    }
    bwd_terms<<<grid, BT, BWD_SMEM, stream>>>(plan_dev, sig, H, q, k, v, g, beta, scale, terms, scratch);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    bwd_states<<<grid, BT, BWD_SMEM, stream>>>(plan_dev, sig, H, terms, h0, S_in, xs, scratch);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (pv.n_cont() > 0) {
        bwd_reverse<false><<<grid, BT, BWD_SMEM, stream>>>(plan_dev, sig, H, terms, dout, dfinal, G_end, Qd, gs, dh0,
                                                           scratch);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    bwd_compose<<<H * 4, BT, 0, stream>>>(plan_dev, sig, H, A, afin, dfinal, Qd, G_end);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    bwd_reverse<true><<<grid, BT, BWD_SMEM, stream>>>(plan_dev, sig, H, terms, dout, dfinal, G_end, Qd, gs, dh0,
                                                      scratch);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    bwd_grads<<<grid, BT, BWD_SMEM, stream>>>(plan_dev, sig, H, q, k, v, g, beta, scale, dout, xs, gs, dq, dk, dv, dg,
                                       dbeta, scratch);
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
