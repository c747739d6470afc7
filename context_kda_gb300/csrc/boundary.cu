// Boundary fix-up: completes the continuing pieces from their incoming state.
//
// For a token t of the piece that continues a sequence into segment j,
//     o_t = o_local,t + S_in[j]^T qhat_t,
// and a sequence that ends in such a piece gets
//     final = P_end S_in[j] + final_local,
// i.e. the same product with the K rows of P_end playing the role of qhat
// (cuLA PR #110, "feat(cp): add opt-in NVSHMEM CP state handoff", §Motivation:
// consumers assemble the final state from the producers' affine states).
//
// Work is cut into 64-row tiles: ceil(len / 64) tiles per continuing piece and
// two tiles (128 transition rows) per final-state record; one CTA per
// (tile, head), S_in[j] staged once per CTA in shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int TR = 64;        // rows per tile
constexpr int LDS_S = VD;     // stride of the staged S_in (column reads are consecutive)
constexpr int LDS_Q = KD + 4; // stride of the staged qhat tile

__global__ void __launch_bounds__(256)
boundary_v0(const int32_t *__restrict__ plan, int H, const float *__restrict__ S_in,
            const float *__restrict__ qhat, const float *__restrict__ afin,
            uint16_t *__restrict__ o, float *__restrict__ final_state)
{
    extern __shared__ float4 smem_raw[];
    float *sS = reinterpret_cast<float *>(smem_raw);   // [KD][VD]
    float *sQ = sS + KD * LDS_S;                        // [TR][LDS_Q]
    const PlanView pv{plan};
    const int tid = threadIdx.x;
    const int tile = blockIdx.x / H, h = blockIdx.x % H;
    const int64_t T_cont = pv.T_cont();

    // locate the record this tile belongs to
    int seg = -1, rows = 0, t_first = 0, seq = -1, fin_row = 0;
    const float *src = nullptr;
    {
        int rem = tile;
        const int nc = pv.n_cont();
        for (int ci = 0; ci < nc && seg < 0; ++ci) {
            const int32_t *cr = pv.cont(ci);
            const int nt = (cr[3] + TR - 1) / TR;
            if (rem < nt) {
                seg = cr[1];
                rows = min(TR, cr[3] - rem * TR);
                t_first = pv.piece(cr[0])[PC_START] + rem * TR;
                src = qhat + (static_cast<size_t>(h) * T_cont + cr[2] + rem * TR) * KD;
            } else {
                rem -= nt;
            }
        }
        if (seg < 0) {
            const int f = rem / 2, half = rem % 2;
            const int32_t *fr = pv.fin(f);
            seg = fr[2];
            seq = fr[1];
            fin_row = half * TR;
            rows = TR;
            src = afin + ((static_cast<size_t>(f) * H + h) * KD + half * TR) * KD;
        }
    }

    const float *Sj = S_in + (static_cast<size_t>(seg) * H + h) * KD * VD;
    for (int e = tid; e < KD * VD / 4; e += 256)
        reinterpret_cast<float4 *>(sS)[e] = reinterpret_cast<const float4 *>(Sj)[e];
    for (int e = tid; e < TR * KD / 4; e += 256) {
        const int r = e / (KD / 4), c4 = e % (KD / 4);
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < rows) v4 = reinterpret_cast<const float4 *>(src + static_cast<size_t>(r) * KD)[c4];
        *reinterpret_cast<float4 *>(&sQ[r * LDS_Q + 4 * c4]) = v4;
    }
    __syncthreads();

    const int c = tid & 127, hf = tid >> 7;
    float acc[32];
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) acc[rr] = 0.f;
    for (int k4 = 0; k4 < KD / 4; ++k4) {
        const float s0 = sS[(4 * k4 + 0) * LDS_S + c], s1 = sS[(4 * k4 + 1) * LDS_S + c];
        const float s2 = sS[(4 * k4 + 2) * LDS_S + c], s3 = sS[(4 * k4 + 3) * LDS_S + c];
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
            const float4 q4 = *reinterpret_cast<const float4 *>(&sQ[(hf * 32 + rr) * LDS_Q + 4 * k4]);
            acc[rr] = fmaf(q4.x, s0, acc[rr]);
            acc[rr] = fmaf(q4.y, s1, acc[rr]);
            acc[rr] = fmaf(q4.z, s2, acc[rr]);
            acc[rr] = fmaf(q4.w, s3, acc[rr]);
        }
    }
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) {
        const int r = hf * 32 + rr;
        if (r >= rows) continue;
        if (seq < 0) {
            uint16_t *dst = o + (static_cast<size_t>(t_first + r) * H + h) * VD + c;
            *dst = f32_to_bf16_bits(bf16_bits_to_f32(*dst) + acc[rr]);
        } else {
            float *dst = final_state + ((static_cast<size_t>(seq) * H + h) * KD + fin_row + r) * VD + c;
            *dst += acc[rr];
        }
    }
}

}  // namespace

cudaError_t launch_boundary(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *S_in,
                            const float *qhat, const float *afin, uint16_t *o, float *final_state,
                            cudaStream_t stream)
{
    const PlanView pv{plan_host};
    long long tiles = 0;
    for (int i = 0; i < pv.n_cont(); ++i) tiles += (pv.cont(i)[3] + TR - 1) / TR;
    tiles += 2LL * pv.n_fin();
    if (tiles == 0) return cudaSuccess;
    const long long blocks = tiles * H;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t smem = sizeof(float) * (KD * LDS_S + TR * LDS_Q);
    cudaError_t err = cudaFuncSetAttribute(boundary_v0, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    boundary_v0<<<static_cast<unsigned>(blocks), 256, smem, stream>>>(plan_dev, H, S_in, qhat, afin, o,
                                                                      final_state);
    return cudaGetLastError();
}

}  // namespace kda
