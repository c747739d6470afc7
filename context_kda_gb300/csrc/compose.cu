// Composition of the segment summaries into each segment's incoming state.
//
// cuLA PR #136 ("feat(kda): add cuDNN concatenated-summary Kimi CP", §Summary):
// affine summary composition in FP32.  With the seed (0, h0) in front of the
// first segment, the prefix composition (A_{j-1},B_{j-1}) o ... o (0, h0) always
// has a zero transition, so the incoming state is its state part:
//     S_in[0] = h0[first sequence],
//     S_in[j] = h0[s]                            if sequence s starts at b_j,
//             = B[j-1]                           if a sequence starts inside j-1,
//             = A[j-1] S_in[j-1] + B[j-1]        otherwise.
// The value columns are independent, so each CTA carries a 128 x 16 column
// slice of one head's state through all segments (FP32 CUDA cores).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int NCOL = 16;        // value columns per CTA
constexpr int LDS_A = KD + 4;   // padded row stride of the staged transition

__global__ void __launch_bounds__(256)
compose_v0(const int32_t *__restrict__ plan, int H, const float *__restrict__ A,
           const float *__restrict__ B, const float *__restrict__ h0, float *__restrict__ S_in)
{
    extern __shared__ float4 smem_raw[];
    float *sA = reinterpret_cast<float *>(smem_raw);   // [KD][LDS_A]
    float *sS = sA + KD * LDS_A;                        // [KD][NCOL]
    const PlanView pv{plan};
    const int tid = threadIdx.x;
    const int ncb = VD / NCOL;
    const int h = blockIdx.x / ncb, cb = blockIdx.x % ncb;
    const int col0 = cb * NCOL;
    const int S = pv.S();
    const size_t mat = static_cast<size_t>(KD) * VD;
    // this thread's outputs: rows rg + 32 m (m < 4), columns 2 cp, 2 cp + 1
    const int cp = tid & 7, rg = tid >> 3;

    for (int j = 0; j < S; ++j) {
        const int32_t *sg = pv.seg(j);
        float *dst = S_in + (static_cast<size_t>(j) * H + h) * mat;
        const bool reset = (j == 0) || (sg[1] & KDA_SEG_STARTS_SEQ);
        if (reset) {
            const float *src = h0 ? h0 + (static_cast<size_t>(sg[0]) * H + h) * mat : nullptr;
            for (int e = tid; e < KD * NCOL; e += 256) {
                const int r = e / NCOL, cc = e % NCOL;
                sS[e] = src ? src[r * VD + col0 + cc] : 0.f;
            }
        } else {
            const bool prev_reset = pv.seg(j - 1)[1] & KDA_SEG_HAS_RESET;
            const float *Bp = B + (static_cast<size_t>(j - 1) * H + h) * mat;
            if (prev_reset) {
                for (int e = tid; e < KD * NCOL; e += 256) sS[e] = Bp[(e / NCOL) * VD + col0 + e % NCOL];
            } else {
                const float *Ap = A + (static_cast<size_t>(j - 1) * H + h) * KD * KD;
                for (int e = tid; e < KD * KD / 4; e += 256) {
                    const int r = e / (KD / 4), c4 = e % (KD / 4);
                    const float4 a4 = reinterpret_cast<const float4 *>(Ap + r * KD)[c4];
                    *reinterpret_cast<float4 *>(&sA[r * LDS_A + 4 * c4]) = a4;
                }
                __syncthreads();
                float acc[4][2];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int r = rg + 32 * m;
                    acc[m][0] = Bp[r * VD + col0 + 2 * cp];
                    acc[m][1] = Bp[r * VD + col0 + 2 * cp + 1];
                }
                for (int i = 0; i < KD; ++i) {
                    const float2 s2 = *reinterpret_cast<const float2 *>(&sS[i * NCOL + 2 * cp]);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float a = sA[(rg + 32 * m) * LDS_A + i];
                        acc[m][0] = fmaf(a, s2.x, acc[m][0]);
                        acc[m][1] = fmaf(a, s2.y, acc[m][1]);
                    }
                }
                __syncthreads();
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int r = rg + 32 * m;
                    sS[r * NCOL + 2 * cp] = acc[m][0];
                    sS[r * NCOL + 2 * cp + 1] = acc[m][1];
                }
            }
        }
        __syncthreads();
        for (int e = tid; e < KD * NCOL; e += 256) dst[(e / NCOL) * VD + col0 + e % NCOL] = sS[e];
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_compose(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *A,
                           const float *B, const float *h0, float *S_in, cudaStream_t stream)
{
    const size_t smem = sizeof(float) * (KD * LDS_A + KD * NCOL);
    cudaError_t err = cudaFuncSetAttribute(compose_v0, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    (void)plan_host;
    compose_v0<<<H * (VD / NCOL), 256, smem, stream>>>(plan_dev, H, A, B, h0, S_in);
    return cudaGetLastError();
}

}  // namespace kda
