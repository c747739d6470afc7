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
// Work units are 128-row tiles (128 continuing tokens, or the 128 rows of a
// final-state transition) of one head, numbered head-major so that consecutive
// units share S_in[j].  The kernel is persistent: one CTA per SM takes a
// contiguous run of units.  S_in[j] arrives by bulk copy and is split into a
// bf16 hi/lo operand only when the run reaches a new (head, segment); each
// qhat tile arrives by bulk copy into a staging buffer, is split likewise, and
// D = Qhat S_in is formed on the tcgen05 tensor cores (M = N = K = 128, three
// products accumulated in FP32 in TMEM).  The copy of the next item is issued
// as soon as the staging buffer has been read, and the output rows are fetched
// while the tensor core runs.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int TR = 128;                   // rows per tile
constexpr uint32_t LBO_B = 2048;          // S_in^T operand: rows c, cols k
constexpr uint32_t LBO_A = 2064;          // Qhat operand: rows r, cols k (chunk stride padded off the bank period)
constexpr uint32_t TILE_B = 32768, TILE_A = 16 * LBO_A;
constexpr uint32_t OFF_B = 0;                      // S_in^T hi | lo
constexpr uint32_t OFF_A = 2 * TILE_B;             // Qhat hi | lo
constexpr uint32_t OFF_STG = OFF_A + 2 * TILE_A;   // fp32 staging: 128 rows x 512 bytes
constexpr uint32_t SMEM_BYTES = OFF_STG + 65536;
constexpr uint32_t TM_COLS = 128;

__device__ int g_boundary_status;

// Position in the unit order: head h, record rec (continuing pieces first, then
// final-state transitions), tile within the record.
struct Cursor {
    int h, rec, tile;
};

struct Rec {
    int seg, seq, nt, rows_total, t_first;   // seq >= 0: final-state record
    size_t src;                              // float offset of row 0 in qhat (or afin) for head h
};

__device__ __forceinline__ Rec rec_info(const PlanView &pv, int H, int h, int rec)
{
    Rec r;
    if (rec < pv.n_cont()) {
        const int32_t *cr = pv.cont(rec);
        r.seg = cr[1];
        r.seq = -1;
        r.rows_total = cr[3];
        r.nt = (cr[3] + TR - 1) / TR;
        r.t_first = pv.piece(cr[0])[PC_START];
        r.src = (static_cast<size_t>(h) * pv.T_cont() + cr[2]) * KD;
    } else {
        const int f = rec - pv.n_cont();
        const int32_t *fr = pv.fin(f);
        r.seg = fr[2];
        r.seq = fr[1];
        r.rows_total = TR;
        r.nt = 1;
        r.t_first = 0;
        r.src = (static_cast<size_t>(f) * H + h) * KD * KD;
    }
    return r;
}

__device__ __forceinline__ void split_store4(unsigned char *base, uint32_t off_hi, uint32_t off_lo, float4 x)
{
    uint32_t h0, h1, l0, l1;
    split_bf16x2(x.x, x.y, h0, l0);
    split_bf16x2(x.z, x.w, h1, l1);
    *reinterpret_cast<uint2 *>(base + off_hi) = make_uint2(h0, h1);
    *reinterpret_cast<uint2 *>(base + off_lo) = make_uint2(l0, l1);
}

__global__ void __launch_bounds__(256, 1)
boundary_tc(const int32_t *__restrict__ plan, int H, int units_per_head, long long n_units,
            const float *__restrict__ S_in, const float *__restrict__ qhat, const float *__restrict__ afin,
            uint16_t *__restrict__ o, float *__restrict__ final_state)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) uint64_t s_mbar;
    __shared__ __align__(8) uint64_t s_ldbar;
    __shared__ uint32_t s_tmem;
    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;
    const int n_rec = pv.n_cont() + pv.n_fin();
    const long long u_begin = n_units * blockIdx.x / gridDim.x;
    const long long u_end = n_units * (blockIdx.x + 1) / gridDim.x;
    if (u_begin >= u_end) return;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t mbar = smem_u32(&s_mbar), ldbar = smem_u32(&s_ldbar);
    const float *stg = reinterpret_cast<const float *>(smem + OFF_STG);

    // cursor of the first unit
    Cursor c{static_cast<int>(u_begin / units_per_head), 0, 0};
    {
        int rem = static_cast<int>(u_begin % units_per_head);
        while (true) {
            const int nt = rec_info(pv, H, c.h, c.rec).nt;
            if (rem < nt) break;
            rem -= nt;
            ++c.rec;
        }
        c.tile = rem;
    }
    Rec ri = rec_info(pv, H, c.h, c.rec);

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(ldbar, 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    uint32_t ld_phase = 0, mma_phase = 0;
    bool ok = true, pending = false;

    auto fetch_S = [&](int h, int seg) {
        mbar_arrive_expect_tx(ldbar, 65536u);
        bulk_g2s(sbase + OFF_STG, S_in + (static_cast<size_t>(seg) * H + h) * KD * VD, 65536u, ldbar);
    };
    auto fetch_tile = [&](const Rec &r, int tile) {
        const uint32_t rows = static_cast<uint32_t>(min(TR, r.rows_total - tile * TR));
        const float *base = (r.seq < 0 ? qhat : afin) + r.src + static_cast<size_t>(tile) * TR * KD;
        mbar_arrive_expect_tx(ldbar, rows * KD * 4);
        bulk_g2s(sbase + OFF_STG, base, rows * KD * 4, ldbar);
    };

    int key_h = -1, key_seg = -1;
    if (tid == 0) fetch_S(c.h, ri.seg);
    pending = true;

    for (long long u = u_begin; u < u_end; ++u) {
        if (c.h != key_h || ri.seg != key_seg) {
            // S_in[j] (rows k, cols c) -> S_in^T operand (rows c, cols k) as bf16 hi/lo
            ok &= mbar_wait(ldbar, ld_phase++ & 1);
            pending = false;
            const int cc = tid & 127, kh = tid >> 7;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = stg[(kh * 64 + 8 * m + e) * VD + cc];
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) split_bf16x2(x[2 * p], x[2 * p + 1], hi[p], lo[p]);
                const uint32_t off = cm_off(cc, kh * 64 + 8 * m, LBO_B);
                *reinterpret_cast<uint4 *>(smem + OFF_B + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(smem + OFF_B + TILE_B + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_async_smem();
            __syncthreads();
            if (tid == 0) fetch_tile(ri, c.tile);
            pending = true;
            key_h = c.h;
            key_seg = ri.seg;
        }
        const int rows = min(TR, ri.rows_total - c.tile * TR);
        ok &= mbar_wait(ldbar, ld_phase++ & 1);
        pending = false;
        // qhat tile (fp32 rows) -> operand (rows r, cols k) as bf16 hi/lo; rows past the record are zero
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int id = tid + 256 * i, r = id >> 5, c4 = id & 31;   // lanes: consecutive 4-column pieces
            const float4 x = r < rows ? *reinterpret_cast<const float4 *>(stg + r * KD + c4 * 4)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            const uint32_t off = cm_off(r, c4 * 4, LBO_A);
            split_store4(smem, OFF_A + off, OFF_A + TILE_A + off, x);
        }
        fence_async_smem();
        fence_before();
        __syncthreads();   // staging read, operands written, previous epilogue done with TMEM

        // the next unit, and the copy it needs first
        Cursor nc = c;
        if (++nc.tile == ri.nt) {
            nc.tile = 0;
            if (++nc.rec == n_rec) {
                nc.rec = 0;
                ++nc.h;
            }
        }
        const bool more = u + 1 < u_end;
        Rec nri = ri;
        if (more) nri = rec_info(pv, H, nc.h, nc.rec);
        if (tid == 0) {
            fence_after();
            if (more) {
                if (nc.h != key_h || nri.seg != key_seg)
                    fetch_S(nc.h, nri.seg);
                else
                    fetch_tile(nri, nc.tile);
            }
            const uint32_t id = idesc_bf16(128, 128);
            const uint32_t aoff[3] = {0, 0, TILE_A}, boff[3] = {0, TILE_B, 0};
#pragma unroll
            for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase, sdesc(sbase + OFF_A + aoff[ps] + kk * 2 * LBO_A, LBO_A),
                             sdesc(sbase + OFF_B + boff[ps] + kk * 2 * LBO_B, LBO_B), id, (ps | kk) != 0);
            commit(mbar);
        }
        pending = more;

        // fetch this thread's destination row piece while the tensor core works
        const int r = quad * 32 + lane;
        const bool live = r < rows;
        uint4 ow[8];
        float4 fw[16];
        uint4 *odst = nullptr;
        float4 *fdst = nullptr;
        if (ri.seq < 0)
            odst = reinterpret_cast<uint4 *>(o + (static_cast<size_t>(ri.t_first + c.tile * TR + r) * H + c.h) * VD +
                                             hw * 64);
        else
            fdst = reinterpret_cast<float4 *>(final_state + ((static_cast<size_t>(ri.seq) * H + c.h) * KD + r) * VD +
                                              hw * 64);
        if (live) {
            if (odst) {
#pragma unroll
                for (int m = 0; m < 8; ++m) ow[m] = odst[m];
            } else {
#pragma unroll
                for (int m = 0; m < 16; ++m) fw[m] = fdst[m];
            }
        }
        ok &= mbar_wait(mbar, mma_phase++ & 1);
        fence_after();
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
        if (live && ok) {
            if (odst) {
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const uint32_t ww[4] = {ow[m].x, ow[m].y, ow[m].z, ow[m].w};
                    uint32_t nw[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        nw[p] = bf16x2_bits(__uint_as_float(ww[p] << 16) + d[8 * m + 2 * p],
                                            __uint_as_float(ww[p] & 0xFFFF0000u) + d[8 * m + 2 * p + 1]);
                    odst[m] = make_uint4(nw[0], nw[1], nw[2], nw[3]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    fdst[m] = make_float4(fw[m].x + d[4 * m], fw[m].y + d[4 * m + 1], fw[m].z + d[4 * m + 2],
                                          fw[m].w + d[4 * m + 3]);
            }
        }
        fence_before();
        if (!__syncthreads_and(ok)) break;
        c = nc;
        ri = nri;
    }
    if (!__syncthreads_and(ok)) {
        // a wait gave up: record it, and let any copy still in flight land before the CTA exits
        if (tid == 0) {
            atomicExch(&g_boundary_status, KDA_ERR_TIMEOUT);
            if (pending) mbar_wait(ldbar, ld_phase & 1);
            mbar_wait(mbar, mma_phase & 1);
        }
        __syncthreads();
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

cudaError_t launch_boundary(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *S_in,
                            const float *qhat, const float *afin, uint16_t *o, float *final_state,
                            cudaStream_t stream)
{
    const PlanView pv{plan_host};
    long long per_head = pv.n_fin();
    for (int i = 0; i < pv.n_cont(); ++i) per_head += (pv.cont(i)[3] + TR - 1) / TR;
    if (per_head == 0) return cudaSuccess;
    if (per_head > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const long long n_units = per_head * H;
    const long long grid = n_units < sm_count() ? n_units : sm_count();
    cudaError_t err = cudaFuncSetAttribute(boundary_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(SMEM_BYTES));
    if (err != cudaSuccess) return err;
    boundary_tc<<<static_cast<unsigned>(grid), 256, SMEM_BYTES, stream>>>(
        plan_dev, H, static_cast<int>(per_head), n_units, S_in, qhat, afin, o, final_state);
    return cudaGetLastError();
}

}  // namespace kda
