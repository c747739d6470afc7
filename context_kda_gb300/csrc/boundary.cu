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
// qhat tile (bf16) arrives by bulk copy into a staging buffer and is laid out
// as the A operand, and D = Qhat S_in is formed on the tcgen05 tensor cores
// (M = N = K = 128; qhat hi * S hi + qhat hi * S lo, FP32 in TMEM).  A final-
// state transition (fp32) is split into hi/lo and takes the third product too.  The copy of the next item is issued
// as soon as the staging buffer has been read.  A full 128-row output tile
// moves through a shared-memory buffer by tiled TMA (128-byte swizzle): loaded
// one unit ahead, updated in place by the epilogue, written back with one TMA
// store.  Ragged tail tiles and final states are read and written by the
// threads directly, so nothing outside a record is ever stored.
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
constexpr uint32_t OFF_OB = 197632;                // bf16 output tile: two swizzled 64-column boxes
constexpr uint32_t SMEM_BYTES = OFF_OB + 32768;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;   // room to align the base to 1024 bytes
static_assert(OFF_STG + 65536 <= OFF_OB && OFF_OB % 1024 == 0, "output tile buffer");
constexpr uint32_t TM_COLS = 128;

__device__ int g_boundary_status;

// Position in the unit order: head h, record rec (continuing pieces first, then
// final-state transitions), tile within the record.
struct Cursor {
    int h, rec, tile;
};

struct Rec {
    int seg, seq, nt, rows_total, t_first;   // seq >= 0: final-state record
    size_t src;                              // element offset of row 0 in qhat (bf16) or afin (fp32), head h
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
            const float *__restrict__ S_in, const uint16_t *__restrict__ qhat, const float *__restrict__ afin,
            uint16_t *__restrict__ o, float *__restrict__ final_state, const __grid_constant__ CUtensorMap tm_o)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_mbar;
    __shared__ __align__(8) uint64_t s_ldbar;
    __shared__ __align__(8) uint64_t s_obar;   // output tile landed
    __shared__ uint32_t s_tmem;
    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;
    const int n_rec = pv.n_cont() + pv.n_fin();
    const long long u_begin = n_units * blockIdx.x / gridDim.x;
    const long long u_end = n_units * (blockIdx.x + 1) / gridDim.x;
    if (u_begin >= u_end) return;
    unsigned char *const smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t mbar = smem_u32(&s_mbar), ldbar = smem_u32(&s_ldbar), obar = smem_u32(&s_obar);
    const float *stg = reinterpret_cast<const float *>(smem + OFF_STG);

    // cursor of the first unit: each warp scans the records' tile counts 32 at a time (inclusive
    // prefix sums over the lanes) and takes the first record whose running count passes the unit
    Cursor c{static_cast<int>(u_begin / units_per_head), 0, 0};
    {
        int rem = static_cast<int>(u_begin % units_per_head);
        for (int b = 0; b < n_rec; b += 32) {
            const int i = b + lane;
            const int nt = i >= n_rec ? 0 : (i < pv.n_cont() ? (pv.cont(i)[3] + TR - 1) / TR : 1);
            int incl = nt;
#pragma unroll
            for (int sh = 1; sh < 32; sh <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, sh);
                if (lane >= sh) incl += y;
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            if (rem < total) {
                const int l = __ffs(__ballot_sync(0xffffffffu, incl > rem)) - 1;
                c.rec = b + l;
                c.tile = rem - __shfl_sync(0xffffffffu, incl - nt, l);
                break;
            }
            rem -= total;
        }
    }
    Rec ri = rec_info(pv, H, c.h, c.rec);

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(ldbar, 1);
        mbar_init(obar, 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    uint32_t ld_phase = 0, mma_phase = 0, o_phase = 0;
    bool ok = true, pending = false, o_pending = false;

    auto fetch_S = [&](int h, int seg) {
        mbar_arrive_expect_tx(ldbar, 65536u);
        bulk_g2s(sbase + OFF_STG, S_in + (static_cast<size_t>(seg) * H + h) * KD * VD, 65536u, ldbar);
    };
    // a unit whose output tile goes through the buffer: 128 continuing tokens
    auto tiled = [&](const Rec &r, int tile) { return r.seq < 0 && r.rows_total - tile * TR >= TR; };
    auto fetch_o = [&](const Rec &r, int tile, int h) {   // thread 0
        mbar_arrive_expect_tx(obar, 32768u);
        const int z = r.t_first + tile * TR;
        tma_load_3d(sbase + OFF_OB, &tm_o, 0, h, z, obar);
        tma_load_3d(sbase + OFF_OB + 16384, &tm_o, 64, h, z, obar);
    };
    auto fetch_tile = [&](const Rec &r, int tile) {
        const uint32_t rows = static_cast<uint32_t>(min(TR, r.rows_total - tile * TR));
        const size_t e0 = r.src + static_cast<size_t>(tile) * TR * KD;
        const void *base = r.seq < 0 ? static_cast<const void *>(qhat + e0) : static_cast<const void *>(afin + e0);
        const uint32_t bytes = rows * KD * (r.seq < 0 ? 2u : 4u);
        mbar_arrive_expect_tx(ldbar, bytes);
        bulk_g2s(sbase + OFF_STG, base, bytes, ldbar);
    };

    int key_h = -1, key_seg = -1;
    if (tid == 0) fetch_S(c.h, ri.seg);
    pending = true;
    if (tiled(ri, c.tile)) {
        if (tid == 0) fetch_o(ri, c.tile, c.h);
        o_pending = true;
    }

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
        if (ri.seq < 0) {
            // qhat tile (bf16 rows) -> operand (rows r, cols k); rows past the record are zero.  Lanes
            // take consecutive 8-column pieces of a row.
            const unsigned char *sb = smem + OFF_STG;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int id = tid + 256 * i, r = id >> 4, c8 = id & 15;
                const uint4 x = r < rows ? *reinterpret_cast<const uint4 *>(sb + r * 256 + c8 * 16)
                                         : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(smem + OFF_A + cm_off(r, c8 * 8, LBO_A)) = x;
            }
        } else {
            // transition tile (fp32 rows) -> operand as bf16 hi/lo; lanes take consecutive 4-column pieces
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int id = tid + 256 * i, r = id >> 5, c4 = id & 31;
                const float4 x = *reinterpret_cast<const float4 *>(stg + r * KD + c4 * 4);
                const uint32_t off = cm_off(r, c4 * 4, LBO_A);
                split_store4(smem, OFF_A + off, OFF_A + TILE_A + off, x);
            }
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
            const int terms = ri.seq < 0 ? 2 : 3;   // qhat is exact in bf16: no lo * hi product
            for (int ps = 0; ps < terms; ++ps)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tbase, sdesc(sbase + OFF_A + aoff[ps] + kk * 2 * LBO_A, LBO_A),
                             sdesc(sbase + OFF_B + boff[ps] + kk * 2 * LBO_B, LBO_B), id, (ps | kk) != 0);
            commit(mbar);
        }
        pending = more;

        // fetch this thread's destination row piece while the tensor core works (units whose
        // output tile is not in the buffer)
        const bool tl_unit = tiled(ri, c.tile);
        const int r = quad * 32 + lane;
        const bool live = r < rows && !tl_unit;
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
        if (tl_unit) {   // output tile in the buffer: update in place (row r, this half's box)
            ok &= mbar_wait(obar, o_phase++ & 1);
            o_pending = false;
            unsigned char *box = smem + OFF_OB + hw * 16384;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                uint4 *p = reinterpret_cast<uint4 *>(box + sw128(r, m));
                const uint4 w4 = *p;
                const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
                uint32_t nw[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    nw[q] = bf16x2_bits(__uint_as_float(ww[q] << 16) + d[8 * m + 2 * q],
                                        __uint_as_float(ww[q] & 0xFFFF0000u) + d[8 * m + 2 * q + 1]);
                *p = make_uint4(nw[0], nw[1], nw[2], nw[3]);
            }
            fence_async_smem();
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
        if (tid == 0 && (tl_unit || (more && tiled(nri, nc.tile)))) {
            if (tl_unit) {   // write the tile back; the buffer is free once the store has read it
                const int z = ri.t_first + c.tile * TR;
                tma_store_3d(&tm_o, 0, c.h, z, sbase + OFF_OB);
                tma_store_3d(&tm_o, 64, c.h, z, sbase + OFF_OB + 16384);
                bulk_commit_group();
                bulk_wait_read_all();
            }
            if (more && tiled(nri, nc.tile)) fetch_o(nri, nc.tile, nc.h);
        }
        if (more && tiled(nri, nc.tile)) o_pending = true;
        c = nc;
        ri = nri;
    }
    if (tid == 0) bulk_wait_all();   // output tiles stored before the CTA exits
    if (!__syncthreads_and(ok)) {
        // a wait gave up: record it, and let any copy still in flight land before the CTA exits
        if (tid == 0) {
            atomicExch(&g_boundary_status, KDA_ERR_TIMEOUT);
            if (pending) mbar_wait(ldbar, ld_phase & 1);
            if (o_pending) mbar_wait(obar, o_phase & 1);
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
                            const uint16_t *qhat, const float *afin, uint16_t *o, float *final_state,
                            cudaStream_t stream)
{
    const PlanView pv{plan_host};
    long long per_head = pv.n_fin();
    for (int i = 0; i < pv.n_cont(); ++i) per_head += (pv.cont(i)[3] + TR - 1) / TR;
    if (per_head == 0) return cudaSuccess;
    if (per_head > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const long long n_units = per_head * H;
    const long long grid = n_units < sm_count() ? n_units : sm_count();
    CUtensorMap to{};   // only full 128-row tiles use it, so T < 128 never reads it
    if (pv.T() >= TR && !encode_rows_3d(&to, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, pv.T(), 64, TR))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(boundary_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(SMEM_ALLOC));
    if (err != cudaSuccess) return err;
    boundary_tc<<<static_cast<unsigned>(grid), 256, SMEM_ALLOC, stream>>>(
        plan_dev, H, static_cast<int>(per_head), n_units, S_in, qhat, afin, o, final_state, to);
    return cudaGetLastError();
}

}  // namespace kda
