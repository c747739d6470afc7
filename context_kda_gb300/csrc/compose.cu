// Composition of the segment summaries into each segment's incoming state.
//
// cuLA PR #136 ("feat(kda): add cuDNN concatenated-summary Kimi CP", §Summary):
// affine summary composition in FP32, (A2,B2) o (A1,B1) = (A2 A1, A2 B1 + B2).
// Written as maps of the state, S_in[j] = F_j(S_in[j-1]) with
//     F_j = (0, h0[s])              if sequence s starts at b_j (and F_0 = (0, h0 of the first
//                                   sequence)): a seed,
//         = (0, B[j-1])             if a sequence starts inside segment j-1: an update,
//         = (A[j-1], B[j-1])        otherwise: a step,
// so S_in[j] = (F_j o ... o F_0)(anything): a prefix scan of the maps under o.
//
// Two schedules compute it.
// - The chain: S_in[j] = F_j(S_in[j-1]) in order, one product per step.
// - The two-level (blocked) scan, log-depth across groups of about sqrt(S)
//   segments: (1) every group's total map C_g = F_last o ... o F_first, all
//   groups in parallel, as the state [Ã | B̃] (K x (K + V)) carried from the
//   identity [I | 0] through the group's maps; (2) the chain over the group
//   totals, E_{g+1} = C_g(E_g), giving each group's incoming state; (3) every
//   group in parallel from E_g through its own maps, giving S_in.  Its depth
//   is about 3 sqrt(S) steps instead of S, for about three times the products.
//
// All four are one kernel: each CTA carries a 32-column slice of one head's
// state (or of [Ã | B̃]) through a list of iterations.  An iteration is a
// product X <- M X (tcgen05, M = 128, N = 32, K = 128, three bf16 hi/lo
// products accumulated in FP32 in TMEM) or a constant, plus an added slice
// (B, h0, B̃, E, the identity or nothing), and may store the result.
// The pipeline hides memory latency behind the products:
// - Transitions arrive by tiled TMA (four 32-column boxes, 128-byte swizzle)
//   into two staging buffers, two products ahead (the L2 is warmed one
//   further), and the worker warps split each into bf16 hi/lo straight into
//   TMEM, the A operand of its product, one product ahead while the previous
//   one runs; two TMEM operand buffers alternate.
// - The slice an iteration adds arrives by TMA into one of two buffers, two
//   iterations ahead; results leave through two output buffers by TMA stores.
// - An issuer warp issues the products and the transition copies; an I/O warp
//   the stores and the slice copies.  Every mbarrier has one waiting role that
//   can fall at most one phase behind its arrivals, so parity waits never
//   alias: the issuer waits once per product, the I/O warp once per iteration
//   on the barrier of that iteration's parity.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int NS = 32;                     // value columns per CTA
constexpr int NC = NS / 2;                 // columns per epilogue thread
constexpr uint32_t CS_S = 2048;            // state operand (rows k, cols c), read MN-major
constexpr uint32_t SOP = NS / 8 * CS_S;    // one bf16 part of the state operand (8 KiB)
constexpr uint32_t STG = 65536;            // one fp32 transition, 4 swizzled boxes of 32 columns
constexpr uint32_t SLICE = 16384;          // one fp32 slice box (128 rows x 32 columns, swizzled)
constexpr uint32_t OFF_STG = 0;                       // two transition staging buffers
constexpr uint32_t OFF_VAL = OFF_STG + 2 * STG;       // two incoming slices
constexpr uint32_t OFF_OUT = OFF_VAL + 2 * SLICE;     // two result slices on their way out
constexpr uint32_t OFF_SOP = OFF_OUT + 2 * SLICE;     // state operand hi | lo
constexpr uint32_t SMEM_BYTES = OFF_SOP + 2 * SOP;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;    // room to align the base to 1024 bytes
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");

// TMEM columns: the accumulator, then two transition operands (hi: k pairs in 64 columns, lo after)
constexpr uint32_t TM_D = 0;
constexpr uint32_t TM_A = 128;             // operand buffer b at TM_A + 128 b: hi [0, 64), lo [64, 128)
constexpr uint32_t TM_COLS = 512;

__device__ int g_compose_status;

enum { IN_SEED = 0, IN_UPDATE = 1, IN_STEP = 2 };

__device__ __forceinline__ int in_kind(const PlanView &pv, int j)
{
    if (j == 0 || (pv.seg(j)[1] & KDA_SEG_STARTS_SEQ)) return IN_SEED;
    return (pv.seg(j - 1)[1] & KDA_SEG_HAS_RESET) ? IN_UPDATE : IN_STEP;
}

enum { MODE_CHAIN = 0, MODE_TOTALS = 1, MODE_GROUPS = 2, MODE_APPLY = 3 };
enum { SRC_NONE = 0, SRC_IDENT, SRC_H0, SRC_B, SRC_T, SRC_E, SRC_S };   // slice sources / result targets

// One iteration of a CTA's list.
struct Iter {
    bool step;      // a product with the transition at row a_row (of A, or of the totals' Ã part)
    int a_row;
    int vsrc, vx, vrow;   // the added slice: source, column, row (in units of K rows)
    int osrc, ox, orow;   // the stored result: target, column, row
};

// What a CTA does: head h, slice s (32 columns), group g (blocked scan).
struct Job {
    int h, s, g, m, G, S, H, has_h0;
};

__device__ __forceinline__ int group_len(const Job &b) { return min((b.g + 1) * b.m, b.S) - b.g * b.m; }

template <int MODE>
__device__ __forceinline__ int n_iters(const Job &b)
{
    if (MODE == MODE_CHAIN) return b.S;
    if (MODE == MODE_GROUPS) return b.G;
    if (MODE == MODE_APPLY) return group_len(b) + (b.g > 0 ? 1 : 0);
    return group_len(b) + 1;   // MODE_TOTALS: the identity, then the group's maps
}

// Iteration j of the chain (segment j): its map F_j and the result S_in[j].
__device__ __forceinline__ Iter chain_iter(const PlanView &pv, const Job &b, int j, int col0)
{
    Iter it{};
    const int kind = in_kind(pv, j);
    it.step = kind == IN_STEP;
    it.a_row = (j - 1) * b.H + b.h;
    if (kind == IN_SEED) {
        if (b.has_h0) {
            it.vsrc = SRC_H0;
            it.vx = col0;
            it.vrow = pv.seg(j)[0] * b.H + b.h;
        }
    } else {
        it.vsrc = SRC_B;
        it.vx = col0;
        it.vrow = (j - 1) * b.H + b.h;
    }
    it.osrc = SRC_S;
    it.ox = col0;
    it.orow = j * b.H + b.h;
    return it;
}

template <int MODE>
__device__ __forceinline__ Iter iter_info(const PlanView &pv, const Job &b, int v)
{
    const int col0 = (b.s & 3) * NS;
    if (MODE == MODE_CHAIN) return chain_iter(pv, b, v, col0);
    if (MODE == MODE_APPLY) {
        if (b.g > 0 && v == 0) {   // the group's incoming state E_g
            Iter it{};
            it.vsrc = SRC_E;
            it.vx = col0;
            it.vrow = b.g * b.H + b.h;
            return it;
        }
        return chain_iter(pv, b, b.g * b.m + v - (b.g > 0 ? 1 : 0), col0);
    }
    if (MODE == MODE_GROUPS) {   // E_v = C_{v-1}(E_{v-1}), E_0 = 0
        Iter it{};
        if (v == 0) return it;
        it.step = true;
        it.a_row = (v - 1) * b.H + b.h;
        it.vsrc = SRC_T;
        it.vx = KD + col0;
        it.vrow = (v - 1) * b.H + b.h;
        it.osrc = SRC_E;
        it.ox = col0;
        it.orow = v * b.H + b.h;
        return it;
    }
    // MODE_TOTALS: slice s < 4 carries columns of Ã (from the identity, adding nothing), s >= 4
    // columns of B̃ (from zero, adding the maps' constant slices)
    Iter it{};
    const bool bpart = b.s >= 4;
    const int len = group_len(b);
    if (v == 0) {
        it.vsrc = bpart ? SRC_NONE : SRC_IDENT;
    } else {
        const int j = b.g * b.m + v - 1;
        const Iter c = chain_iter(pv, b, j, col0);
        it.step = c.step;
        it.a_row = c.a_row;
        if (bpart) {
            it.vsrc = c.vsrc;
            it.vx = c.vx;
            it.vrow = c.vrow;
        }
    }
    if (v == len) {
        it.osrc = SRC_T;
        it.ox = b.s * NS;
        it.orow = b.g * b.H + b.h;
    }
    return it;
}

constexpr int NWORK = 256;                 // 8 worker warps
constexpr int NT = NWORK + 64;             // + issuer warp + I/O warp
constexpr int MMA_TID = NWORK, IO_TID = NWORK + 32;

template <int MODE>
__global__ void __launch_bounds__(NT, 1)
compose_tc(const int32_t *__restrict__ plan, PlanSig sig, int H, int has_h0, int m, const float *__restrict__ A_raw,
           const __grid_constant__ CUtensorMap tm_A, const __grid_constant__ CUtensorMap tm_B,
           const __grid_constant__ CUtensorMap tm_h0, const __grid_constant__ CUtensorMap tm_S,
           const __grid_constant__ CUtensorMap tm_T, const __grid_constant__ CUtensorMap tm_E)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_mbar;      // a product is done (one arrival per product)
    __shared__ __align__(8) uint64_t s_mready;    // workers -> issuer: a product's operands are in place
    __shared__ __align__(8) uint64_t s_abar[2];   // transition staged, per staging buffer
    __shared__ __align__(8) uint64_t s_vbar[2];   // incoming slice staged, per buffer
    __shared__ __align__(8) uint64_t s_oready[2]; // workers -> I/O: iteration done, per parity
    __shared__ __align__(8) uint64_t s_ofree[2];  // I/O -> workers: output buffer read by its store
    __shared__ uint32_t s_tmem;
    if (!plan_matches(plan, sig)) {   // not the plan the launch was sized from: touch nothing
        if (threadIdx.x == 0) record_status(&g_compose_status, KDA_ERR_INVALID_ARG);
        return;
    }
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = (warp >> 2) & 1;
    Job job{};
    job.S = pv.S();
    job.H = H;
    job.has_h0 = has_h0;
    job.m = m;
    job.G = (job.S + m - 1) / m;
    {
        const int nsl = MODE == MODE_TOTALS ? 8 : 4;   // slices per head
        int bid = blockIdx.x;
        job.s = bid % nsl;
        bid /= nsl;
        job.h = bid % H;
        job.g = (MODE == MODE_TOTALS || MODE == MODE_APPLY) ? bid / H : 0;
    }
    const int NIT = n_iters<MODE>(job);
    const int r = quad * 32 + lane;   // state row (and TMEM lane) of this worker
    const int cl = half * NC;         // its first column within the slice
    const uint32_t sbase = smem_u32(smem);
    const uint32_t mbar = smem_u32(&s_mbar), mready = smem_u32(&s_mready);
    const bool worker = tid < NWORK, issuer = tid == MMA_TID, io = tid == IO_TID;

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(mready, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_abar[i]), 1);
            mbar_init(smem_u32(&s_vbar[i]), 1);
            mbar_init(smem_u32(&s_oready[i]), 1);
            mbar_init(smem_u32(&s_ofree[i]), 1);
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    grid_dep_wait();     // the summaries (or the previous phase) come from the previous kernel
    grid_dep_launch();   // the next kernel may be scheduled on SMs this one leaves

    auto it_of = [&](int v) { return iter_info<MODE>(pv, job, v); };
    auto is_step = [&](int v) { return v < NIT && it_of(v).step; };
    auto next_step = [&](int v) {
        while (v < NIT && !it_of(v).step) ++v;
        return v;
    };
    auto loads = [&](const Iter &it) { return it.vsrc != SRC_NONE && it.vsrc != SRC_IDENT; };
    // issuer: the transition of the product at iteration v into staging buffer b
    auto fetch_A = [&](int v, int b) {
        const uint32_t bar = smem_u32(&s_abar[b]);
        const int y = it_of(v).a_row * KD;
        const CUtensorMap *map = MODE == MODE_GROUPS ? &tm_T : &tm_A;
        mbar_arrive_expect_tx(bar, STG);
#pragma unroll
        for (int bx = 0; bx < 4; ++bx) tma_load_2d(sbase + OFF_STG + b * STG + bx * SLICE, map, 32 * bx, y, bar);
    };
    auto map_of = [&](int src) -> const CUtensorMap * {
        switch (src) {
        case SRC_H0: return &tm_h0;
        case SRC_B: return &tm_B;
        case SRC_T: return &tm_T;
        case SRC_E: return &tm_E;
        default: return &tm_S;
        }
    };
    // I/O thread: the slice iteration v adds, into buffer v & 1
    auto fetch_vals = [&](int v) {
        const Iter it = it_of(v);
        const uint32_t bar = smem_u32(&s_vbar[v & 1]);
        mbar_arrive_expect_tx(bar, SLICE);
        tma_load_2d(sbase + OFF_VAL + (v & 1) * SLICE, map_of(it.vsrc), it.vx, it.vrow * KD, bar);
    };

    bool ok = true;
    if (worker) {
        bool bad = false;
        uint32_t n_step = 0;                       // products whose result this thread has consumed
        uint32_t n_conv = 0;                       // transitions split into TMEM so far
        uint32_t v_count[2] = {0, 0};              // slices consumed per buffer
        for (int v = 0; v < NIT; ++v) {
            const Iter it = it_of(v);
            const bool next_is_step = is_step(v + 1);
            // (a) the next product's transition: staging -> TMEM operand (bf16 hi | lo); lane = row r,
            //     this thread's half of the columns k
            if (next_is_step) {
                const int b = n_conv & 1;
                if (!mbar_wait_warp(smem_u32(&s_abar[b]), (n_conv >> 1) & 1)) bad = true;
                ++n_conv;
                const unsigned char *stg = smem + OFF_STG + b * STG;
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int bx = 0; bx < 2; ++bx) {
                    const unsigned char *box = stg + (2 * half + bx) * SLICE;
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const float4 x = *reinterpret_cast<const float4 *>(box + sw128(r, ch));
                        split_bf16x2(x.x, x.y, hi[bx * 16 + 2 * ch], lo[bx * 16 + 2 * ch]);
                        split_bf16x2(x.z, x.w, hi[bx * 16 + 2 * ch + 1], lo[bx * 16 + 2 * ch + 1]);
                    }
                }
                const uint32_t ta = tbase + (static_cast<uint32_t>(quad * 32) << 16) + TM_A + b * 128 + half * 32;
                tmem_st32_nowait(ta, hi);
                tmem_st32_nowait(ta + 64, lo);
                tmem_wait_st();
            }
            // (b) this iteration's product
            float st[NC];
            if (it.step) {
                if (!mbar_wait_warp(mbar, n_step & 1)) bad = true;
                ++n_step;
                fence_after();
                tmem_ld16(tbase + (static_cast<uint32_t>(quad * 32) << 16) + TM_D + cl, st);
            } else {
#pragma unroll
                for (int e = 0; e < NC; ++e) st[e] = 0.f;
            }
            // (c) + the iteration's slice
            if (it.vsrc == SRC_IDENT) {
                const int c0 = (job.s & 3) * NS + cl;
#pragma unroll
                for (int e = 0; e < NC; ++e) st[e] += (r == c0 + e) ? 1.f : 0.f;
            } else if (loads(it)) {
                const int b = v & 1;
                if (!mbar_wait_warp(smem_u32(&s_vbar[b]), v_count[b]++ & 1)) bad = true;
                const unsigned char *vb = smem + OFF_VAL + b * SLICE;
#pragma unroll
                for (int mm = 0; mm < NC / 4; ++mm) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(vb + sw128(r, cl / 4 + mm));
                    st[4 * mm] += b4.x;
                    st[4 * mm + 1] += b4.y;
                    st[4 * mm + 2] += b4.z;
                    st[4 * mm + 3] += b4.w;
                }
            }
            // (d) the result into output buffer v & 1, once the store of iteration v - 2 has read it
            {
                const int b = v & 1;
                if (v >= 2 && !mbar_wait_warp(smem_u32(&s_ofree[b]), ((v - 2) >> 1) & 1)) bad = true;
                if (it.osrc != SRC_NONE) {
                    unsigned char *ob = smem + OFF_OUT + b * SLICE;
#pragma unroll
                    for (int mm = 0; mm < NC / 4; ++mm)
                        *reinterpret_cast<float4 *>(ob + sw128(r, cl / 4 + mm)) =
                            make_float4(st[4 * mm], st[4 * mm + 1], st[4 * mm + 2], st[4 * mm + 3]);
                }
            }
            // (e) the result as the next product's operand (rows k = r, cols c), bf16 hi | lo
            if (next_is_step) {
#pragma unroll
                for (int mm = 0; mm < NC / 8; ++mm) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) split_bf16x2(st[8 * mm + 2 * p], st[8 * mm + 2 * p + 1], hi[p], lo[p]);
                    const uint32_t off = static_cast<uint32_t>((cl / 8 + mm) * CS_S + (r >> 3) * 128 + (r & 7) * 16);
                    *reinterpret_cast<uint4 *>(smem + OFF_SOP + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(smem + OFF_SOP + SOP + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
            // (f) hand the iteration over: the next product's operands to the issuer, the output
            //     buffer and the consumed slice buffer to the I/O warp
            fence_async_smem();
            fence_before();
            if (bar_or1(NWORK, bad)) {
                ok = false;
                break;
            }
            if (tid == 0) {
                if (next_is_step) mbar_arrive(mready);
                mbar_arrive(smem_u32(&s_oready[v & 1]));
            }
        }
        if (bad) ok = false;
    } else if (issuer) {
        // per product n (in order): once its operands are in place, the product; then the transition
        // of product n + 2 into the staging buffer product n's transition was split from
        int v_cur = next_step(0);
        int v_ahead = v_cur < NIT ? next_step(v_cur + 1) : NIT;
        uint32_t n = 0, n_fetch[2] = {0, 0};
        if (v_cur < NIT) {
            fetch_A(v_cur, 0);
            n_fetch[0] = 1;
        }
        if (v_ahead < NIT) {
            fetch_A(v_ahead, 1);
            n_fetch[1] = 1;
        }
        while (v_cur < NIT) {
            if (!(ok = mbar_wait(mready, n & 1))) break;
            fence_after();
            {
                const uint32_t id = idesc_bf16(128, NS, 0, 1);
                const uint32_t ta = tbase + TM_A + (n & 1) * 128;
                const uint32_t s_hi = sbase + OFF_SOP;
                const uint32_t aop[3] = {ta, ta, ta + 64}, sop[3] = {s_hi, s_hi + SOP, s_hi};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ta(tbase + TM_D, aop[ps] + kk * 8, sdesc(sop[ps] + kk * 256, 128, CS_S), id,
                                    (ps | kk) != 0);
                commit(mbar);
            }
            // staging buffer n & 1 was split before this product's handoff: it takes product n + 2
            const int v_next = v_ahead < NIT ? next_step(v_ahead + 1) : NIT;
            if (v_next < NIT) {
                fetch_A(v_next, n & 1);
                ++n_fetch[n & 1];
                const int v_warm = next_step(v_next + 1);   // and the L2 warms the one after
                if (MODE != MODE_GROUPS && v_warm < NIT) {
                    const float *pa = A_raw + static_cast<size_t>(it_of(v_warm).a_row) * KD * KD;
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(pa), "r"(STG) : "memory");
                }
            }
            ++n;
            v_cur = v_ahead;
            v_ahead = v_next;
        }
        if (!ok) record_status(&g_compose_status, KDA_ERR_TIMEOUT);
        // whatever happened elsewhere, the products and copies this role issued land before the CTA
        // frees its tensor memory (bounded waits; immediate when the workers consumed them)
        if (n) mbar_wait(mbar, (n - 1) & 1);
        for (int b = 0; b < 2; ++b)
            if (n_fetch[b]) mbar_wait(smem_u32(&s_abar[b]), (n_fetch[b] - 1) & 1);
    } else if (io) {
        // per iteration v: once the workers hand it over, the store of its result and the copy of the
        // slice iteration v + 2 adds (into the buffer iteration v read)
        uint32_t n_fetch[2] = {0, 0};
        for (int v = 0; v < 2 && v < NIT; ++v)
            if (loads(it_of(v))) {
                fetch_vals(v);
                ++n_fetch[v];
            }
        for (int v = 0; v < NIT; ++v) {
            if (!(ok = mbar_wait(smem_u32(&s_oready[v & 1]), (v >> 1) & 1))) break;
            const Iter it = it_of(v);
            if (it.osrc != SRC_NONE) {
                tma_store_2d(map_of(it.osrc), it.ox, it.orow * KD, sbase + OFF_OUT + (v & 1) * SLICE);
                bulk_commit_group();
            }
            if (v + 2 < NIT && loads(it_of(v + 2))) {
                fetch_vals(v + 2);
                ++n_fetch[v & 1];
            }
            bulk_wait_read_all();                      // output buffer v & 1 has been read
            mbar_arrive(smem_u32(&s_ofree[v & 1]));
        }
        if (!ok) record_status(&g_compose_status, KDA_ERR_TIMEOUT);
        bulk_wait_all();
        for (int b = 0; b < 2; ++b)
            if (n_fetch[b]) mbar_wait(smem_u32(&s_vbar[b]), (n_fetch[b] - 1) & 1);
    }
    // A role whose wait gave up has recorded it; every role has let its own copies and products land
    // above, so the tensor memory can be freed.
    if (!__syncthreads_and(ok) && tid == 0) record_status(&g_compose_status, KDA_ERR_TIMEOUT);
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

struct Maps {
    CUtensorMap A, B, H0, S, T, E;
};

bool encode_maps(Maps &mp, const PlanView &pv, int H, const float *A, const float *B, const float *h0, float *S_in,
                 float *T, float *E, int G)
{
    const uint64_t rows = static_cast<uint64_t>(pv.S()) * H * KD;
    if (!encode_f32_rows128(&mp.A, A, rows, KD) || !encode_f32_rows128(&mp.B, B, rows, KD) ||
        !encode_f32_rows128(&mp.S, S_in, rows, KD))
        return false;
    if (h0) {
        if (!encode_f32_rows128(&mp.H0, h0, static_cast<uint64_t>(pv.N()) * H * KD, KD)) return false;
    } else {
        mp.H0 = mp.B;   // never read: no iteration takes a seed from h0
    }
    if (T) {
        const uint64_t grows = static_cast<uint64_t>(G) * H * KD;
        if (!encode_f32_rows(&mp.T, T, grows, KD + VD, KD) || !encode_f32_rows128(&mp.E, E, grows, KD)) return false;
    } else {
        mp.T = mp.S;    // never used by the chain
        mp.E = mp.S;
    }
    return true;
}

template <int MODE>
cudaError_t launch_mode(const int32_t *plan_host, const int32_t *plan_dev, int H, int has_h0, int m, int G,
                        const float *A, const Maps &mp, cudaStream_t stream)
{
    cudaError_t err = set_dynamic_smem(reinterpret_cast<const void *>(compose_tc<MODE>),
                                       static_cast<int>(SMEM_ALLOC));
    if (err != cudaSuccess) return err;
    const int per_head = MODE == MODE_TOTALS ? 8 * G : MODE == MODE_APPLY ? 4 * G : 4;
    return launch_dependent(compose_tc<MODE>, dim3(static_cast<unsigned>(H * per_head)), dim3(NT), SMEM_ALLOC,
                            stream, plan_dev, plan_sig(plan_host), H, has_h0, m, A, mp.A, mp.B, mp.H0, mp.S, mp.T,
                            mp.E);
}

}  // namespace

int scan_group_size(int S)
{
    int m = 1;
    while (m * m < S) ++m;
    return m;
}

size_t scan_scratch_bytes(const int32_t *plan_host, int H)
{
    const int S = PlanView{plan_host}.S();
    const int m = scan_group_size(S), G = (S + m - 1) / m;
    const size_t totals = static_cast<size_t>(G) * H * KD * (KD + VD) * 4;
    return ((totals + 255) & ~static_cast<size_t>(255)) + static_cast<size_t>(G) * H * KD * VD * 4;
}

cudaError_t launch_compose(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *A,
                           const float *B, const float *h0, float *S_in, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    if (pv.S() <= 0) return cudaSuccess;
    Maps mp;
    if (!encode_maps(mp, pv, H, A, B, h0, S_in, nullptr, nullptr, 0)) return cudaErrorInvalidValue;
    return launch_mode<MODE_CHAIN>(plan_host, plan_dev, H, h0 ? 1 : 0, 1, 1, A, mp, stream);
}

cudaError_t launch_compose_blocked(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *A,
                                   const float *B, const float *h0, float *S_in, void *scratch, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    const int S = pv.S();
    if (S <= 0) return cudaSuccess;
    const int m = scan_group_size(S), G = (S + m - 1) / m;
    const size_t totals = static_cast<size_t>(G) * H * KD * (KD + VD) * 4;
    float *T = static_cast<float *>(scratch);
    float *E = reinterpret_cast<float *>(static_cast<char *>(scratch) + ((totals + 255) & ~static_cast<size_t>(255)));
    Maps mp;
    if (!encode_maps(mp, pv, H, A, B, h0, S_in, T, E, G)) return cudaErrorInvalidValue;
    const int has_h0 = h0 ? 1 : 0;
    cudaError_t err = launch_mode<MODE_TOTALS>(plan_host, plan_dev, H, has_h0, m, G, A, mp, stream);
    if (err == cudaSuccess && G > 1) err = launch_mode<MODE_GROUPS>(plan_host, plan_dev, H, has_h0, m, G, A, mp, stream);
    if (err == cudaSuccess) err = launch_mode<MODE_APPLY>(plan_host, plan_dev, H, has_h0, m, G, A, mp, stream);
    return err;
}

// The status word of this file's kernels: read and cleared (the caller has synchronised the device).
int take_compose_status()
{
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_compose_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_compose_status, &z, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return v;
}

}  // namespace kda
