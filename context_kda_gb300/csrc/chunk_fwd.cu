// Chunkwise KDA forward of one piece (segment x sequence), with the segment
// summaries: state columns (outputs, state update B, final states) and
// transition columns (qhat, transition A).
//
// Algebra (per chunk of C = 64 rows, Gamma_r = cumulative g within the chunk):
//   kt_r = exp(Gamma_r) k_r, kh_i = exp(-Gamma_i) k_i, kb_i = exp(Gamma_C - Gamma_i) k_i,
//   qt_r = scale exp(Gamma_r) q_r,
//   M[r,i] = beta_r (kt_r . kh_i) for i < r,   T = (I + M)^-1,
//   W = T Diag(beta) Kt,   Ut = T Diag(beta) V,
//   U = Ut - W S,   O = Qt S + ((Qt Kh^T) masked to i <= r) U,
//   S' = Diag(exp Gamma_C) S + Kb^T U.
// This is the KDA gated delta rule (cuLA PR #110, "feat(cp): add opt-in NVSHMEM
// CP state handoff", §Supported configuration: BF16 inputs, FP32 state) unrolled
// over a chunk: writing u_r = beta_r (v_r - (Diag(exp g_r) S_{r-1})^T k_r) for
// every row gives (I + M) U = Diag(beta) (V - Kt S).
//
// The transition columns run the same recurrence on P (K x K) with zero values
// from P = I at the piece start, so their 'outputs' are qhat_t = scale P_t^T q_t
// and their end state is the piece's transition (cuLA PR #136, "feat(kda): add
// cuDNN concatenated-summary Kimi CP", §Summary: preceding_transition).
//
// This kernel keeps everything on the FP32 CUDA cores: one CTA per
// (work item, head), 256 threads, the 128-column state slice in registers
// (thread = column c, key half hf).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int LDA = 132;  // row stride (floats) of 64 x 128 tiles, 16-byte aligned rows
constexpr int LDH = 129;  // row stride of the kh / kb tile (odd: conflict-free column reads)
constexpr int LDM = 65;   // row stride of 64 x 64 tiles

struct SmemV0 {
    float kb[CH * LDA];   // beta * kt, then W
    float kh[CH * LDH];   // kh, then kb (decay to chunk end)
    float qt[CH * LDA];   // scaled qt
    float vv[CH * LDA];   // beta * v, then Ut, then U
    float rd[CH * LDA];   // Gamma, then T (stride LDM), then partial-sum exchange
    float mt[CH * LDM];   // M
    float qk[CH * LDM];   // masked Qt Kh^T
    float bt[CH];         // beta
    float gc[KD];         // exp(Gamma_C)
};

__global__ void __launch_bounds__(256, 1)
chunk_forward_v0(const int32_t *__restrict__ plan, int H, const uint16_t *__restrict__ q,
                 const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                 const float *__restrict__ g, const float *__restrict__ beta,
                 const float *__restrict__ h0, float scale, uint16_t *__restrict__ o,
                 float *__restrict__ A, float *__restrict__ B, float *__restrict__ fin_state,
                 float *__restrict__ qhat, float *__restrict__ afin)
{
    extern __shared__ float4 smem_raw[];
    SmemV0 &sm = *reinterpret_cast<SmemV0 *>(smem_raw);
    const PlanView pv{plan};
    const int tid = threadIdx.x;
    const int c = tid & 127, hf = tid >> 7;
    const int item = blockIdx.x / H, h = blockIdx.x % H;
    const int32_t *it = pv.item(item);
    const int p = it[0], kind = it[1];
    const int32_t *pc = pv.piece(p);
    const int start = pc[PC_START], len = pc[PC_LEN], seq = pc[PC_SEQ], seg = pc[PC_SEG];
    const int flags = pc[PC_FLAGS], row0 = pc[PC_ROW], fin = pc[PC_FIN];
    const int64_t T_cont = pv.T_cont();

    // thread's slice of the state / transition: rows hf*64 + i, column c
    float st[64];
    if (kind == 0) {
        const bool from_h0 = (flags & KDA_PIECE_FIRST) && h0 != nullptr;
        const float *src = h0 + (static_cast<size_t>(seq) * H + h) * KD * VD;
#pragma unroll
        for (int i = 0; i < 64; ++i) st[i] = from_h0 ? src[(hf * 64 + i) * VD + c] : 0.f;
    } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) st[i] = (hf * 64 + i == c) ? 1.f : 0.f;
    }

    const int nch = (len + CH - 1) / CH;
    for (int ci = 0; ci < nch; ++ci) {
        const int t0 = start + ci * CH;
        const int L = min(CH, len - ci * CH);

        // ---- A1: cumulative decay per key channel (hf 0); beta * v and beta (hf 1)
        if (hf == 0) {
            float gam = 0.f;
            for (int r = 0; r < CH; ++r) {
                const float gv = (r < L) ? g[(static_cast<size_t>(t0 + r) * H + h) * KD + c] : 0.f;
                gam += gv;
                sm.rd[r * LDA + c] = gam;
            }
            sm.gc[c] = expf(gam);
        } else {
            for (int r = 0; r < CH; ++r) {
                const float bv = (r < L) ? beta[static_cast<size_t>(t0 + r) * H + h] : 0.f;
                float vv = 0.f;
                if (kind == 0 && r < L) vv = bf16_bits_to_f32(v[(static_cast<size_t>(t0 + r) * H + h) * VD + c]);
                sm.vv[r * LDA + c] = bv * vv;
                if (c == 0) sm.bt[r] = bv;
            }
        }
        __syncthreads();

        // ---- A2: decayed keys and queries
        for (int a = 0; a < 32; ++a) {
            const int r = hf + 2 * a;
            const float gam = sm.rd[r * LDA + c];
            float kv = 0.f, qv = 0.f;
            if (r < L) {
                const size_t off = (static_cast<size_t>(t0 + r) * H + h) * KD + c;
                kv = bf16_bits_to_f32(k[off]);
                qv = bf16_bits_to_f32(q[off]);
            }
            const float e = expf(gam), ei = expf(-gam);
            sm.kb[r * LDA + c] = sm.bt[r] * e * kv;
            sm.kh[r * LDH + c] = ei * kv;
            sm.qt[r * LDA + c] = scale * e * qv;
        }
        __syncthreads();

        // ---- B: M = (beta Kt) Kh^T (strictly lower), QK = Qt Kh^T (lower incl. diagonal)
        {
            const int rb = tid >> 4, ib = tid & 15;
            float am[4][4], aq[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) am[a][b] = aq[a][b] = 0.f;
            for (int kk = 0; kk < KD; ++kk) {
                float kr[4], qr[4], ki[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    kr[a] = sm.kb[(rb + 16 * a) * LDA + kk];
                    qr[a] = sm.qt[(rb + 16 * a) * LDA + kk];
                }
#pragma unroll
                for (int b = 0; b < 4; ++b) ki[b] = sm.kh[(ib + 16 * b) * LDH + kk];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        am[a][b] = fmaf(kr[a], ki[b], am[a][b]);
                        aq[a][b] = fmaf(qr[a], ki[b], aq[a][b]);
                    }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int r = rb + 16 * a, i = ib + 16 * b;
                    sm.mt[r * LDM + i] = (i < r) ? am[a][b] : 0.f;
                    sm.qk[r * LDM + i] = (i <= r) ? aq[a][b] : 0.f;
                }
        }
        __syncthreads();

        // ---- C: T = (I + M)^-1 by column-wise forward substitution (threads 0..63, one
        //      column each, no barriers); meanwhile the others turn kh into kb in place.
        if (tid < 64) {
            const int j = tid;
            float x[64];
#pragma unroll
            for (int r = 0; r < 64; ++r) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int i = 0; i + 1 < r; i += 2) {
                    a0 = fmaf(sm.mt[r * LDM + i], x[i], a0);
                    a1 = fmaf(sm.mt[r * LDM + i + 1], x[i + 1], a1);
                }
                if (r & 1) a0 = fmaf(sm.mt[r * LDM + r - 1], x[r - 1], a0);
                x[r] = (r == j) ? 1.f : ((r < j) ? 0.f : -(a0 + a1));
            }
#pragma unroll
            for (int r = 0; r < 64; ++r) sm.rd[r * LDM + j] = x[r];
        } else {
            for (int e = tid - 64; e < CH * KD; e += 192) {
                const int r = e >> 7, kk = e & 127;
                sm.kh[r * LDH + kk] *= sm.gc[kk];
            }
        }
        __syncthreads();

        // ---- D: W = T (beta Kt), Ut = T (beta V)
        {
            float w[32], u[32];
#pragma unroll
            for (int a = 0; a < 32; ++a) w[a] = u[a] = 0.f;
            for (int i = 0; i < CH; ++i) {
                const float kbv = sm.kb[i * LDA + c];
                const float vbv = sm.vv[i * LDA + c];
#pragma unroll
                for (int a = 0; a < 32; ++a) {
                    const float tv = sm.rd[(hf + 2 * a) * LDM + i];
                    w[a] = fmaf(tv, kbv, w[a]);
                    u[a] = fmaf(tv, vbv, u[a]);
                }
            }
            __syncthreads();
#pragma unroll
            for (int a = 0; a < 32; ++a) {
                sm.kb[(hf + 2 * a) * LDA + c] = w[a];
                sm.vv[(hf + 2 * a) * LDA + c] = u[a];
            }
        }
        __syncthreads();

        // ---- E: U = Ut - W S   (partial over this thread's key half, exchanged through rd)
        {
            float part[64];
#pragma unroll
            for (int r = 0; r < 64; ++r) {
                const float4 *wr = reinterpret_cast<const float4 *>(&sm.kb[r * LDA + hf * 64]);
                float acc = 0.f;
#pragma unroll
                for (int i4 = 0; i4 < 16; ++i4) {
                    const float4 w4 = wr[i4];
                    acc = fmaf(w4.x, st[4 * i4 + 0], acc);
                    acc = fmaf(w4.y, st[4 * i4 + 1], acc);
                    acc = fmaf(w4.z, st[4 * i4 + 2], acc);
                    acc = fmaf(w4.w, st[4 * i4 + 3], acc);
                }
                part[r] = acc;
            }
            if (hf == 0) {
#pragma unroll
                for (int r = 32; r < 64; ++r) sm.rd[r * LDA + c] = part[r];
            } else {
#pragma unroll
                for (int r = 0; r < 32; ++r) sm.rd[r * LDA + c] = part[r];
            }
            __syncthreads();
            if (hf == 0) {
#pragma unroll
                for (int r = 0; r < 32; ++r) sm.vv[r * LDA + c] -= part[r] + sm.rd[r * LDA + c];
            } else {
#pragma unroll
                for (int r = 32; r < 64; ++r) sm.vv[r * LDA + c] -= part[r] + sm.rd[r * LDA + c];
            }
        }
        __syncthreads();

        // ---- F: O = Qt S + (QK masked) U  -> outputs (state columns) or qhat (transition columns)
        {
            float part[64];
#pragma unroll
            for (int r = 0; r < 64; ++r) {
                const float4 *qr = reinterpret_cast<const float4 *>(&sm.qt[r * LDA + hf * 64]);
                float acc = 0.f;
#pragma unroll
                for (int i4 = 0; i4 < 16; ++i4) {
                    const float4 q4 = qr[i4];
                    acc = fmaf(q4.x, st[4 * i4 + 0], acc);
                    acc = fmaf(q4.y, st[4 * i4 + 1], acc);
                    acc = fmaf(q4.z, st[4 * i4 + 2], acc);
                    acc = fmaf(q4.w, st[4 * i4 + 3], acc);
                }
                part[r] = acc;
            }
            if (hf == 0) {
#pragma unroll
                for (int r = 32; r < 64; ++r) sm.rd[r * LDA + c] = part[r];
            } else {
#pragma unroll
                for (int r = 0; r < 32; ++r) sm.rd[r * LDA + c] = part[r];
            }
            __syncthreads();
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
                const int r = hf * 32 + rr;
                float acc = (hf == 0 ? part[rr] : part[32 + rr]) + sm.rd[r * LDA + c];
                for (int i = 0; i <= r; ++i) acc = fmaf(sm.qk[r * LDM + i], sm.vv[i * LDA + c], acc);
                if (r < L) {
                    if (kind == 0)
                        o[(static_cast<size_t>(t0 + r) * H + h) * VD + c] = f32_to_bf16_bits(acc);
                    else
                        qhat[(static_cast<size_t>(h) * T_cont + row0 + ci * CH + r) * KD + c] = acc;
                }
            }
        }

        // ---- G: S' = Diag(exp Gamma_C) S + Kb^T U
        {
#pragma unroll
            for (int i = 0; i < 64; ++i) st[i] *= sm.gc[hf * 64 + i];
            for (int r = 0; r < L; ++r) {
                const float ur = sm.vv[r * LDA + c];
                const float *kbr = &sm.kh[r * LDH + hf * 64];
#pragma unroll
                for (int i = 0; i < 64; ++i) st[i] = fmaf(kbr[i], ur, st[i]);
            }
        }
        __syncthreads();
    }

    // ---- piece end: summaries and final states
    const size_t mat = static_cast<size_t>(KD) * VD;
    const bool seg_last = flags & KDA_PIECE_SEG_LAST, seq_end = flags & KDA_PIECE_SEQ_END;
    if (kind == 0) {
        if (seg_last) {
            float *dst = B + (static_cast<size_t>(seg) * H + h) * mat;
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[(hf * 64 + i) * VD + c] = st[i];
            if (pv.seg(seg)[1] & KDA_SEG_HAS_RESET) {
                float *za = A + (static_cast<size_t>(seg) * H + h) * KD * KD;
#pragma unroll
                for (int i = 0; i < 64; ++i) za[(hf * 64 + i) * KD + c] = 0.f;
            }
        }
        if (seq_end) {
            float *dst = fin_state + (static_cast<size_t>(seq) * H + h) * mat;
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[(hf * 64 + i) * VD + c] = st[i];
        }
    } else {
        if (seg_last) {
            float *dst = A + (static_cast<size_t>(seg) * H + h) * KD * KD;
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[(hf * 64 + i) * KD + c] = st[i];
        }
        if (seq_end) {
            float *dst = afin + (static_cast<size_t>(fin) * H + h) * KD * KD;
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[(hf * 64 + i) * KD + c] = st[i];
        }
    }
}

}  // namespace

cudaError_t launch_chunk_forward(const int32_t *plan_host, const int32_t *plan_dev, int H,
                                 const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const float *g, const float *beta, const float *h0, float scale,
                                 uint16_t *o, float *A, float *B, float *final_state,
                                 float *qhat, float *afin, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    const size_t smem = sizeof(SmemV0);
    cudaError_t err = cudaFuncSetAttribute(chunk_forward_v0, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const long long blocks = static_cast<long long>(pv.n_items()) * H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    chunk_forward_v0<<<static_cast<unsigned>(blocks), 256, smem, stream>>>(
        plan_dev, H, q, k, v, g, beta, h0, scale, o, A, B, final_state, qhat, afin);
    return cudaGetLastError();
}

}  // namespace kda
