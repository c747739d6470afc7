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
// Each CTA takes one 128-row tile (128 continuing tokens, or the 128 rows of a
// final-state transition) of one head: D = Qhat S_in on the tcgen05 tensor
// cores (M = 128 rows, N = 128 value columns, K = 128), with both operands
// split into bf16 hi/lo and three products accumulated in FP32 in TMEM; the
// epilogue reads D back and updates the bf16 outputs (or FP32 final states)
// with 16-byte loads and stores.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int TR = 128;                     // rows per tile
constexpr uint32_t LBO = 2048;              // 128-row bf16 tiles written row by row
constexpr uint32_t TILE = 32768;            // 128 x 128 bf16
constexpr uint32_t OFF_B = 0;               // S_in^T hi | lo: rows c, cols k
constexpr uint32_t OFF_A = 2 * TILE;        // Qhat hi | lo: rows r, cols k
constexpr uint32_t SMEM_BYTES = 4 * TILE;
constexpr uint32_t TM_COLS = 128;

__device__ int g_boundary_status;

__device__ __forceinline__ void split_store8(unsigned char *base, uint32_t off_hi, uint32_t off_lo, const float *x)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) split_bf16x2(x[2 * p], x[2 * p + 1], h[p], l[p]);
    *reinterpret_cast<uint4 *>(base + off_hi) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(base + off_lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

__global__ void __launch_bounds__(256, 1)
boundary_tc(const int32_t *__restrict__ plan, int H, const float *__restrict__ S_in,
            const float *__restrict__ qhat, const float *__restrict__ afin,
            uint16_t *__restrict__ o, float *__restrict__ final_state)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) uint64_t s_mbar;
    __shared__ uint32_t s_tmem;
    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;
    const int tile = blockIdx.x / H, h = blockIdx.x % H;
    const int64_t T_cont = pv.T_cont();
    const uint32_t sbase = smem_u32(smem);
    const uint32_t mbar = smem_u32(&s_mbar);

    // locate the record this tile belongs to
    int seg = -1, rows = 0, t_first = 0, seq = -1;
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
            const int32_t *fr = pv.fin(rem);
            seg = fr[2];
            seq = fr[1];
            rows = TR;
            src = afin + (static_cast<size_t>(rem) * H + h) * KD * KD;
        }
    }

    if (tid == 0) mbar_init(mbar, 1);
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);

    // S_in^T (rows c, cols k) and the qhat tile (rows r, cols k), both split into bf16 hi/lo
    {
        const float *Sj = S_in + (static_cast<size_t>(seg) * H + h) * KD * VD;
        const int c = tid & 127, kh = tid >> 7;
        float sv[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) sv[j] = Sj[(kh * 64 + j) * VD + c];
        float4 qv[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int id = tid + 256 * i, r = id & 127, kc = id >> 7;   // lanes: consecutive rows
            const float4 *p4 = reinterpret_cast<const float4 *>(src + static_cast<size_t>(r) * KD + kc * 8);
            const bool ok = r < rows;
            qv[2 * i] = ok ? p4[0] : make_float4(0.f, 0.f, 0.f, 0.f);
            qv[2 * i + 1] = ok ? p4[1] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const uint32_t off = cm_off(c, kh * 64 + 8 * m, LBO);
            split_store8(smem, OFF_B + off, OFF_B + TILE + off, sv + 8 * m);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int id = tid + 256 * i, r = id & 127, kc = id >> 7;
            const uint32_t off = cm_off(r, kc * 8, LBO);
            split_store8(smem, OFF_A + off, OFF_A + TILE + off, reinterpret_cast<const float *>(&qv[2 * i]));
        }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    if (tid == 0) {
        const uint32_t id = idesc_bf16(128, 128);
        const uint32_t aoff[3] = {0, 0, TILE}, boff[3] = {0, TILE, 0};
#pragma unroll
        for (int ps = 0; ps < 3; ++ps)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tbase, sdesc(sbase + OFF_A + aoff[ps] + kk * 2 * LBO, LBO),
                         sdesc(sbase + OFF_B + boff[ps] + kk * 2 * LBO, LBO), id, (ps | kk) != 0);
        commit(mbar);
    }
    const bool ok = mbar_wait(mbar, 0);
    fence_after();
    if (ok) {
        const int r = quad * 32 + lane;
        float d[64];
        {
            float d0[32], d1[32];
            const uint32_t ta = tbase + (static_cast<uint32_t>(quad * 32) << 16) + hw * 64;
            tmem_ld32(ta, d0);
            tmem_ld32(ta + 32, d1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                d[j] = d0[j];
                d[32 + j] = d1[j];
            }
        }
        if (r < rows) {
            if (seq < 0) {
                uint4 *dst = reinterpret_cast<uint4 *>(o + (static_cast<size_t>(t_first + r) * H + h) * VD + hw * 64);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    uint4 w = dst[m];
                    uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const float a0 = __uint_as_float(ww[p] << 16) + d[8 * m + 2 * p];
                        const float a1 = __uint_as_float(ww[p] & 0xFFFF0000u) + d[8 * m + 2 * p + 1];
                        ww[p] = bf16x2_bits(a0, a1);
                    }
                    dst[m] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
                }
            } else {
                float4 *dst = reinterpret_cast<float4 *>(final_state + ((static_cast<size_t>(seq) * H + h) * KD + r) * VD +
                                                         hw * 64);
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    float4 f = dst[m];
                    f.x += d[4 * m];
                    f.y += d[4 * m + 1];
                    f.z += d[4 * m + 2];
                    f.w += d[4 * m + 3];
                    dst[m] = f;
                }
            }
        }
    } else if (tid == 0) {
        atomicExch(&g_boundary_status, KDA_ERR_TIMEOUT);
    }
    fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(s_tmem, TM_COLS);
}

}  // namespace

cudaError_t launch_boundary(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *S_in,
                            const float *qhat, const float *afin, uint16_t *o, float *final_state,
                            cudaStream_t stream)
{
    const PlanView pv{plan_host};
    long long tiles = 0;
    for (int i = 0; i < pv.n_cont(); ++i) tiles += (pv.cont(i)[3] + TR - 1) / TR;
    tiles += pv.n_fin();
    if (tiles == 0) return cudaSuccess;
    const long long blocks = tiles * H;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaError_t err = cudaFuncSetAttribute(boundary_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(SMEM_BYTES));
    if (err != cudaSuccess) return err;
    boundary_tc<<<static_cast<unsigned>(blocks), 256, SMEM_BYTES, stream>>>(plan_dev, H, S_in, qhat, afin, o,
                                                                           final_state);
    return cudaGetLastError();
}

}  // namespace kda
