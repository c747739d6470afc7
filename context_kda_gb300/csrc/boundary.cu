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
// Work units are 128-row tiles (128 continuing tokens, or the 128 rows of a final-state transition)
// of one head, numbered head-major so that consecutive units share S_in[j]; a transition follows the
// tiles of the continuing piece that ends its sequence, whose S_in[j] it needs.  The kernel is
// persistent: one CTA per SM takes a contiguous run of units as a software pipeline.  The runs are
// cut by cost, not by count (the host computes each CTA's first unit): a transition moves twice a
// tile's bytes through the threads and takes three products, and each new S_in is split once more.
// - S_in[j] is read straight into registers and split into a bf16 hi/lo operand only when the run
//   reaches a new (head, segment).
// - A qhat tile (bf16) lands by two plain bulk copies directly in the layout the tensor core reads
//   (two 64-column boxes, 128-byte swizzle): the state pass wrote it as that image, box b of a tile of
//   R rows holding row r at (b R + r) 128 bytes from the tile's start.  A ring of three buffers,
//   requested three units ahead.
// - D = Qhat S_in is formed on the tcgen05 tensor cores (M = N = K = 128; qhat * S hi + qhat * S lo,
//   FP32 in one of two TMEM accumulators).  The next unit's products are issued before this unit's
//   epilogue whenever they share S_in and their qhat tile comes by copy, so the epilogue of one unit
//   overlaps the products of the next.  A final-state transition (fp32) is split into hi/lo by the
//   threads and takes the third product too.
// - A full 128-row tile's correction D is rounded to bf16 into one of two shared-memory buffers and
//   added into the outputs in memory by a tiled TMA reduce-add (bf16): the outputs never pass through
//   the SM, so a tile costs the tensor-copy unit 512 rows of 128 bytes (qhat in, D out) instead of 768
//   (the copy unit's row rate bounds this kernel).  Ragged tail tiles are read and written by the
//   threads directly (o + D rounded once), so nothing outside a record is ever touched.  A final
//   state's D (fp32) is staged in both correction buffers and added one 512-byte row per warp
//   instruction.
#include <algorithm>
#include <vector>

#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int TR = 128;                    // rows per tile
constexpr uint32_t LBO_B = 2048;           // S_in^T operand: rows c, cols k (no swizzle)
constexpr uint32_t TILE_B = 32768;
constexpr uint32_t BOX = 16384;            // 128 rows x 128 bytes, 128-byte swizzle
constexpr uint32_t OFF_B = 0;              // S_in^T hi | lo
constexpr uint32_t OFF_A = 2 * TILE_B;     // three qhat tiles (ring), two boxes each
constexpr uint32_t OFF_OB = OFF_A + 6 * BOX;   // two bf16 correction tiles, two boxes each
constexpr uint32_t SMEM_BYTES = OFF_OB + 4 * BOX;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;   // room to align the base to 1024 bytes
static_assert(OFF_A % 1024 == 0 && OFF_OB % 1024 == 0, "swizzled buffers");
constexpr uint32_t TM_COLS = 256;          // two 128-column accumulators

// Relative costs of the run partition, fitted to the global-timer end of every CTA on a packed
// 64-segment launch (65536 tokens, 32 heads), where the stream runs at the HBM roof: a tile about
// 1.45 us, a final-state transition about 11.6 us, the load and split of a new S_in about 5.9 us.
// On shorter launches, whose data stay in L2, the last two weigh less; these weights are the
// compromise that keeps the slowest CTA nearest the mean on both.
constexpr long long COST_TILE = 8, COST_TRANSITION = 64, COST_NEW_STATE = 24;
constexpr int MAX_RUNS = 192;              // CTAs of one launch (one per SM)

// Each CTA's run: the cursor of its first unit (head, record, unit within the record) and its length.
struct Runs {
    int4 c[MAX_RUNS];
};

__device__ int g_boundary_status;

// D (bf16, a 64-column box in the 128-byte swizzled layout of the map) added element-wise into the
// outputs at (x, y, z) of the map by the memory system; completes in this thread's bulk group.
__device__ __forceinline__ void tma_reduce_add_3d(const void *tmap, int x, int y, int z, uint32_t src_smem)
{
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(tmap), "r"(x), "r"(y), "r"(z), "r"(src_smem)
                 : "memory");
}

// Position in the unit order: head h, continuing record rec, unit within the record.  A record's
// units are its 128-row qhat tiles, then, when its piece ends the sequence, the final-state
// transition (which needs the same S_in[j]): transitions spread over the run with their records.
struct Cursor {
    int h, rec, tile;
};

// One unit: segment, sequence (>= 0: a final-state transition), units in its record, rows, first
// token and first qhat row (qhat tiles), element offset of its first row in qhat (bf16) or afin (fp32)
struct Rec {
    int seg, seq, units, rows, tok, qrow;
    size_t src;
};

__device__ __forceinline__ Rec rec_info(const PlanView &pv, int H, int h, int rec, int tile)
{
    Rec r;
    const int32_t *cr = pv.cont(rec);
    const int32_t *pc = pv.piece(cr[0]);
    const int nt = (cr[3] + TR - 1) / TR;
    r.seg = cr[1];
    r.units = nt + ((pc[PC_FLAGS] & KDA_PIECE_SEQ_END) ? 1 : 0);
    if (tile < nt) {
        r.seq = -1;
        r.rows = min(TR, cr[3] - tile * TR);
        r.tok = pc[PC_START] + tile * TR;
        r.qrow = h * pv.T_cont() + cr[2] + tile * TR;
        r.src = static_cast<size_t>(r.qrow) * KD;
    } else {
        const int f = pc[PC_FIN];
        r.seq = pv.fin(f)[1];
        r.rows = TR;
        r.tok = 0;
        r.qrow = 0;
        r.src = (static_cast<size_t>(f) * H + h) * KD * KD;
    }
    return r;
}

__device__ __forceinline__ void advance(Cursor &c, const Rec &r, int n_cont)
{
    if (++c.tile == r.units) {
        c.tile = 0;
        if (++c.rec == n_cont) {
            c.rec = 0;
            ++c.h;
        }
    }
}

__global__ void __launch_bounds__(256, 1)
boundary_tc(const int32_t *__restrict__ plan, PlanSig sig, int H, const __grid_constant__ Runs runs,
            const float *__restrict__ S_in, const uint16_t *__restrict__ qhat, const float *__restrict__ afin,
            uint16_t *__restrict__ o, float *__restrict__ final_state, const __grid_constant__ CUtensorMap tm_o)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_mbar[2];   // products of a unit done, per TMEM accumulator
    __shared__ __align__(8) uint64_t s_abar[3];   // qhat tile landed, per ring slot
    __shared__ uint32_t s_tmem;
    if (!plan_matches(plan, sig)) {   // not the plan the launch was sized from: touch nothing
        if (threadIdx.x == 0) record_status(&g_boundary_status, KDA_ERR_INVALID_ARG);
        return;
    }
    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;
    const int n_cont = pv.n_cont();
    const int4 run = runs.c[blockIdx.x];
    const long long n_run = run.w;
    if (n_run <= 0) return;
    unsigned char *const smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&s_mbar[i]), 1);
        for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&s_abar[i]), 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    uint32_t mph = 0, aph = 0;   // bit i: parity of the next wait on barrier i of each kind
    bool ok = true;
    bool a_pend[3] = {false, false, false};   // thread 0's copies in flight
    uint32_t m_pend = 0;   // thread 0: bit t, products issued into accumulator t and not yet waited for

    // a continuing unit's qhat tile arrives by bulk copy
    auto by_copy = [&](const Rec &r) { return r.seq < 0; };
    // a unit whose correction goes out by TMA reduce-add: 128 continuing tokens
    auto tiled = [&](const Rec &r) { return r.seq < 0 && r.rows == TR; };
    auto fetch_q = [&](const Rec &r, int sl) {   // thread 0: the tile's two box images, r.rows rows each
        const uint32_t bar = smem_u32(&s_abar[sl]), bytes = static_cast<uint32_t>(r.rows) * 128u;
        mbar_arrive_expect_tx(bar, 2 * bytes);
        const unsigned char *src = reinterpret_cast<const unsigned char *>(qhat + r.src);
        bulk_g2s(sbase + OFF_A + sl * 2 * BOX, src, bytes, bar);
        bulk_g2s(sbase + OFF_A + sl * 2 * BOX + BOX, src + bytes, bytes, bar);
        a_pend[sl] = true;
    };
    // a unit's products into accumulator t (thread 0): qhat in ring slot sl, or a transition with its
    // hi part in slot sl and its lo part in output buffer t
    auto issue_mma = [&](const Rec &r, int sl, int t) {
        if (by_copy(r)) {
            ok &= mbar_wait(smem_u32(&s_abar[sl]), (aph >> sl) & 1u);
            aph ^= 1u << sl;
            a_pend[sl] = false;
        }
        fence_after();
        const uint32_t id = idesc_bf16(128, 128);
        const uint32_t a_hi = sbase + OFF_A + sl * 2 * BOX, a_lo = sbase + OFF_OB + t * 2 * BOX;
        const uint32_t boff[3] = {0, TILE_B, 0};
        const int terms = r.seq < 0 ? 2 : 3;   // qhat is exact in bf16: no lo * hi product
        for (int ps = 0; ps < terms; ++ps) {
            const uint32_t a = ps < 2 ? a_hi : a_lo;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tbase + t * 128, sdesc_sw128(a + (kk >> 2) * BOX + (kk & 3) * 32),
                         sdesc(sbase + OFF_B + boff[ps] + kk * 2 * LBO_B, LBO_B), id, (ps | kk) != 0);
        }
        commit(smem_u32(&s_mbar[t]));
        m_pend |= 1u << t;
    };

    // Units n .. n + 3 of the run (cursor and record; valid while inside the run).  qhat comes from
    // the state pass, which completed before the composition (this kernel's prerequisite) passed its
    // own wait and let this kernel's CTAs start: each of the first tiles is requested as soon as its
    // unit's record is known, while the composition still runs; S_in, the composition's result, only
    // after the wait.  The local outputs, also the state pass's, are only read and written after it.
    Cursor c0{run.x, run.y, run.z};
    Rec r0 = rec_info(pv, H, c0.h, c0.rec, c0.tile);
    if (tid == 0 && by_copy(r0)) fetch_q(r0, 0);
    Cursor c1 = c0, c2, c3;
    Rec r1 = r0, r2 = r0, r3 = r0;
    if (n_run > 1) {
        advance(c1, r0, n_cont);
        r1 = rec_info(pv, H, c1.h, c1.rec, c1.tile);
        if (tid == 0 && by_copy(r1)) fetch_q(r1, 1);
    }
    c2 = c1;
    if (n_run > 2) {
        advance(c2, r1, n_cont);
        r2 = rec_info(pv, H, c2.h, c2.rec, c2.tile);
        if (tid == 0 && by_copy(r2)) fetch_q(r2, 2);
    }
    c3 = c2;
    if (n_run > 3) {
        advance(c3, r2, n_cont);
        r3 = rec_info(pv, H, c3.h, c3.rec, c3.tile);
    }
    grid_dep_wait();   // S_in comes from the composition

    int key_h = -1, key_seg = -1;   // the S_in whose split is in the B operand
    bool issued = false;            // unit n's products were issued during the previous unit
    int sl = 0;                     // ring slot of unit n (n mod 3)
    for (long long n = 0; n < n_run; ++n, sl = sl == 2 ? 0 : sl + 1) {
        const int t = static_cast<int>(n & 1);
        const int sl1 = sl == 2 ? 0 : sl + 1;
        const int rows = r0.rows;
        if (!issued) {
            // operands of unit n by the threads; the previous unit's products have completed
            if (c0.h != key_h || r0.seg != key_seg) {
                // S_in[j] (rows k, cols c), read straight from HBM -> S_in^T operand (rows c, cols k)
                // (all 64 loads of a thread in flight at once)
                const float *src = S_in + (static_cast<size_t>(r0.seg) * H + c0.h) * KD * VD;
                const int cc = tid & 127, kh = tid >> 7;
                float xs[64];
#pragma unroll
                for (int e = 0; e < 64; ++e) xs[e] = src[(kh * 64 + e) * VD + cc];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float *x = xs + 8 * m;
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) split_bf16x2(x[2 * p], x[2 * p + 1], hi[p], lo[p]);
                    const uint32_t off = cm_off(cc, kh * 64 + 8 * m, LBO_B);
                    *reinterpret_cast<uint4 *>(smem + OFF_B + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(smem + OFF_B + TILE_B + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
                key_h = c0.h;
                key_seg = r0.seg;
            }
            if (r0.seq >= 0) {
                // transition rows (fp32, rows r, cols k) -> hi in ring slot sl, lo in output buffer t
                // (128-byte swizzle), once that buffer's last store has read it
                if (tid == 0) bulk_wait_read_all();
                __syncthreads();
                const float *src = afin + r0.src;
                float4 xa[16];   // all loads of a thread in flight at once
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int id = tid + 256 * i, r = id >> 5, k = (id & 31) * 4;
                    xa[i] = *reinterpret_cast<const float4 *>(src + r * KD + k);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int id = tid + 256 * i, r = id >> 5, k = (id & 31) * 4;
                    const float4 x = xa[i];
                    uint32_t h0, h1, l0, l1;
                    split_bf16x2(x.x, x.y, h0, l0);
                    split_bf16x2(x.z, x.w, h1, l1);
                    const uint32_t off = (k >> 6) * BOX + sw128(r, (k & 63) >> 3) + (k & 7) * 2;
                    *reinterpret_cast<uint2 *>(smem + OFF_A + sl * 2 * BOX + off) = make_uint2(h0, h1);
                    *reinterpret_cast<uint2 *>(smem + OFF_OB + t * 2 * BOX + off) = make_uint2(l0, l1);
                }
            }
            fence_async_smem();
            fence_before();
            __syncthreads();   // operands written
            if (tid == 0) issue_mma(r0, sl, t);
        }
        // the next unit: its products now when they need nothing from the threads (same S_in, qhat
        // tile by copy)
        const bool more1 = n + 1 < n_run;
        const bool early = more1 && by_copy(r1) && c1.h == key_h && r1.seg == key_seg;
        if (tid == 0 && early) issue_mma(r1, sl1, t ^ 1);

        // epilogue of unit n: a ragged tile fetches this thread's destination row piece while the tensor
        // core works
        const bool tl_unit = tiled(r0), fin_unit = r0.seq >= 0;
        const int r = quad * 32 + lane;
        const bool live = r < rows && !tl_unit && !fin_unit;
        uint4 ow[8];
        uint4 *const odst = reinterpret_cast<uint4 *>(o + (static_cast<size_t>(r0.tok + r) * H + c0.h) * VD + hw * 64);
        if (live) {
#pragma unroll
            for (int m = 0; m < 8; ++m) ow[m] = odst[m];
        }
        ok &= mbar_wait(smem_u32(&s_mbar[t]), (mph >> t) & 1u);
        mph ^= 1u << t;
        m_pend &= ~(1u << t);
        fence_after();
        // ring slot sl is free again: the qhat tile three units on
        if (tid == 0 && n + 3 < n_run && by_copy(r3)) fetch_q(r3, sl);
        float d[64];
        {
            float d0[32], d1[32];
            const uint32_t ta = tbase + t * 128 + (static_cast<uint32_t>(quad * 32) << 16) + hw * 64;
            tmem_ld32(ta, d0);
            tmem_ld32(ta + 32, d1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                d[j] = d0[j];
                d[32 + j] = d1[j];
            }
        }
        if (tl_unit) {   // D as bf16 into buffer t (row r, this half's box), free since the unit before last
            unsigned char *box = smem + OFF_OB + t * 2 * BOX + hw * BOX;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                uint32_t nw[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) nw[q] = bf16x2_bits(d[8 * m + 2 * q], d[8 * m + 2 * q + 1]);
                *reinterpret_cast<uint4 *>(box + sw128(r, m)) = make_uint4(nw[0], nw[1], nw[2], nw[3]);
            }
            fence_async_smem();
        }
        if (live && ok) {
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
        }
        if (fin_unit) {
            // D (fp32, rows r, cols c) into both correction buffers as four 32-column boxes with the
            // 128-byte swizzle: both are free (every reduce had read its buffer before this unit's split,
            // and the lo operand in buffer t has been read by the products)
#pragma unroll
            for (int qb = 0; qb < 2; ++qb) {
                unsigned char *box = smem + OFF_OB + (2 * hw + qb) * BOX;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float *x = d + qb * 32 + 4 * j;
                    *reinterpret_cast<float4 *>(box + sw128(r, j)) = make_float4(x[0], x[1], x[2], x[3]);
                }
            }
            __syncthreads();
            // final += D, one 512-byte row per warp instruction: warp w takes rows 16 w .. 16 w + 15, lane l
            // the 16 bytes of columns 32 (l / 8) + 4 (l % 8) ..
            const int qb = lane >> 3, j = lane & 7;
            float4 *const frow = reinterpret_cast<float4 *>(final_state + (static_cast<size_t>(r0.seq) * H + c0.h) * KD * VD) +
                                 (qb * 32 + 4 * j) / 4;
            float4 fw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) fw[i] = frow[(warp * 16 + i) * (VD / 4)];
            if (ok) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int rr = warp * 16 + i;
                    const float4 x = *reinterpret_cast<const float4 *>(smem + OFF_OB + qb * BOX + sw128(rr, j));
                    frow[rr * (VD / 4)] = make_float4(fw[i].x + x.x, fw[i].y + x.y, fw[i].z + x.z, fw[i].w + x.w);
                }
            }
        }
        // the previous unit's reduce has read its buffer, which the next unit fills
        if (tid == 0) bulk_wait_read_all();
        fence_before();
        if (!__syncthreads_and(ok)) break;
        if (tid == 0 && tl_unit) {   // o += D for the tile's 128 tokens of head h, in memory
            const int z = r0.tok;
            tma_reduce_add_3d(&tm_o, 0, c0.h, z, sbase + OFF_OB + t * 2 * BOX);
            tma_reduce_add_3d(&tm_o, 64, c0.h, z, sbase + OFF_OB + t * 2 * BOX + BOX);
            bulk_commit_group();
        }
        issued = early;
        c0 = c1;
        r0 = r1;
        c1 = c2;
        r1 = r2;
        c2 = c3;
        r2 = r3;
        if (n + 4 < n_run) {
            advance(c3, r3, n_cont);
            r3 = rec_info(pv, H, c3.h, c3.rec, c3.tile);
        }
    }
    if (tid == 0) bulk_wait_all();   // corrections added before the CTA exits
    if (!__syncthreads_and(ok)) {
        // a wait gave up: record it, and let any copy or product still in flight land (bounded waits)
        if (tid == 0) {
            record_status(&g_boundary_status, KDA_ERR_TIMEOUT);
            for (int i = 0; i < 3; ++i)
                if (a_pend[i]) mbar_wait(smem_u32(&s_abar[i]), (aph >> i) & 1u);
            for (int i = 0; i < 2; ++i)
                if ((m_pend >> i) & 1u) mbar_wait(smem_u32(&s_mbar[i]), (mph >> i) & 1u);
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
    // one head's units in order with their cumulative cost (every head has the same sequence)
    std::vector<long long> pre(1, 0);
    std::vector<long long> rec_first;
    for (int i = 0; i < pv.n_cont(); ++i) {
        const int32_t *cr = pv.cont(i);
        const long long nt = (cr[3] + TR - 1) / TR;
        const long long nu = nt + ((pv.piece(cr[0])[PC_FLAGS] & KDA_PIECE_SEQ_END) ? 1 : 0);
        rec_first.push_back(static_cast<long long>(pre.size()) - 1);
        for (long long t = 0; t < nu; ++t)
            pre.push_back(pre.back() + (t < nt ? COST_TILE : COST_TRANSITION) + (t == 0 ? COST_NEW_STATE : 0));
    }
    const long long per_head = static_cast<long long>(pre.size()) - 1;
    if (per_head == 0) return cudaSuccess;
    if (per_head > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const long long n_units = per_head * H;
    const long long grid = std::min<long long>({n_units, static_cast<long long>(sm_count()), MAX_RUNS});
    // CTA b starts at the unit boundary whose preceding cost is nearest to b/grid of the total: the
    // head from one division, the unit within it from a search of the head's cumulative costs
    const unsigned long long w_head = static_cast<unsigned long long>(pre.back());
    const unsigned long long total = w_head * static_cast<unsigned long long>(H);
    if (total / static_cast<unsigned long long>(H) != w_head || total > (1ull << 54)) return cudaErrorInvalidConfiguration;
    Runs runs{};
    long long prev = 0;
    for (long long b = 0; b < grid; ++b) {
        long long next = n_units;
        if (b + 1 < grid) {
            const unsigned long long target = total * static_cast<unsigned long long>(b + 1) / static_cast<unsigned long long>(grid);
            const long long h = static_cast<long long>(target / w_head);
            const long long rem = static_cast<long long>(target - static_cast<unsigned long long>(h) * w_head);
            // first unit boundary within head h at or past rem, or the nearer one before it
            const long long i = std::lower_bound(pre.begin(), pre.end(), rem) - pre.begin();
            next = std::min(n_units, h * per_head + i);
            if (i > 0 && rem - pre[i - 1] < pre[i] - rem && next - 1 > prev) --next;
            next = std::max(prev, next);
        }
        if (next - prev > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        const long long w = prev % per_head;
        const long long rec = std::upper_bound(rec_first.begin(), rec_first.end(), w) - rec_first.begin() - 1;
        runs.c[b] = make_int4(static_cast<int>(prev / per_head), static_cast<int>(rec),
                              static_cast<int>(w - rec_first[rec]), static_cast<int>(next - prev));
        prev = next;
    }
    // full 128-row tiles add their corrections by tiled TMA; a tensor shorter than one tile never
    // uses the map
    CUtensorMap to{};
    if (pv.T() >= TR && !encode_rows_3d(&to, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, pv.T(), 64, TR))
        return cudaErrorInvalidValue;
    cudaError_t err = set_dynamic_smem(reinterpret_cast<const void *>(boundary_tc),
                                       static_cast<int>(SMEM_ALLOC));
    if (err != cudaSuccess) return err;
    return launch_dependent(boundary_tc, dim3(static_cast<unsigned>(grid)), dim3(256), SMEM_ALLOC, stream, plan_dev,
                            plan_sig(plan_host), H, runs, S_in, qhat, afin, o, final_state, to);
}

// Self-test of the expiry path: one thread waits, bounded, on an mbarrier that nothing arrives on,
// and records the expiry in this file's status word as any kernel of the library would.
__global__ void wait_expiry_probe_tc()
{
    __shared__ __align__(8) uint64_t s_bar;
    if (threadIdx.x == 0) mbar_init(smem_u32(&s_bar), 1);
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&s_bar), 0)) record_status(&g_boundary_status, KDA_ERR_TIMEOUT);
}

cudaError_t launch_wait_expiry_probe(cudaStream_t stream)
{
    wait_expiry_probe_tc<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

// The status word of this file's kernel: read and cleared (the caller has synchronised the device).
int take_boundary_status()
{
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_boundary_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_boundary_status, &z, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return v;
}

}  // namespace kda
