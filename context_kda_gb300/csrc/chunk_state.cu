// Serial state pass of the chunkwise KDA forward over one piece (segment x sequence), with the
// segment summaries: state columns (outputs, state update B, final states) and transition
// columns (qhat, transition A).
//
// Per chunk, from the package the preparation kernel wrote (W, Qt, masked QK, Kh, exp(Gamma_C),
// Ut) and the chunk-start state X:
//   U = Ut - W X,   O = Qt X + QK U,   X' = Diag(exp Gamma_C) (X + Kh^T U)
// (the KDA gated delta rule unrolled over a chunk; cuLA PR #110, "feat(cp): add opt-in NVSHMEM
// CP state handoff", §Supported configuration: BF16 inputs, FP32 state).  The transition
// columns run the same recurrence on P (K x K) with zero values from P = I at the piece start,
// so their 'outputs' are qhat_t = scale P_t^T q_t and their end state is the piece's transition
// (cuLA PR #136, "feat(kda): add cuDNN concatenated-summary Kimi CP", §Summary:
// preceding_transition).
//
// Mapping.  One CTA per (work item, head): 8 worker warps, an issuer warp (tcgen05 MMAs) and a
// producer warp (package copies: a TMA unit busy with earlier copies stalls the thread that issues
// the next one, which must not be the MMA issuer).  The state lives
// transposed in TMEM (lane c, column k) twice: as an FP32 accumulator, and split into bf16 hi/lo
// pairs as the A operand of W X and Qt X, which the tensor core reads from TMEM.  Per chunk the
// chain is: (W X)^T = X^T W^T (3-term) -> workers form U^T = Ut^T - (W X)^T and split it into
// TMEM -> O^T += U^T QK^T (1-term), X^T += U^T Kh (3-term) -> workers decay X and split it for
// the next chunk, then stage O in shared memory for a tiled TMA store.  Qt X (1-term) runs right
// after W X.  Both package parts are double-buffered and arrive by bulk copies issued one chunk
// ahead; Ut goes straight into registers, also one chunk ahead.  Keeping both A operands in TMEM
// leaves shared-memory bandwidth to the B operands and the copies.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

// ---- shared-memory map (bytes from the dynamic base; bf16 tiles, hi then lo where split) ------
constexpr uint32_t P1_BYTES = PK_P1_END;          // package bytes [PK_W, PK_P1_END): W hi | lo, Qt hi
constexpr uint32_t OFF_P1 = 0;                     // two buffers of P1_BYTES
constexpr uint32_t P2_BYTES = PK_P2_END - PK_QK;   // QK, Kh hi | lo, exp(Gamma_C)          41472
constexpr uint32_t OFF_P2 = OFF_P1 + 2 * P1_BYTES;  // two buffers of P2_BYTES
constexpr uint32_t OFF_OB = OFF_P2 + 2 * P2_BYTES;  // O tile: rows r (64), two 64-column boxes of
                                                    // 128-byte rows, 128-byte swizzle     2 x 8192
constexpr uint32_t SMEM_BYTES = OFF_OB + 16384;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // the base is rounded up to 1024 bytes
constexpr uint32_t T64 = 16384;
// offsets inside a P2 buffer
constexpr uint32_t P2_QK = 0, P2_KH = PK_KH - PK_QK, P2_GC = PK_GC - PK_QK;

// ---- TMEM columns --------------------------------------------------------------------------
constexpr uint32_t TM_WX = 0;     // (W X)^T (64 cols)
constexpr uint32_t TM_O0 = 64;    // O^T of even chunks (64 cols)
constexpr uint32_t TM_X = 128;    // X^T (128 cols)
constexpr uint32_t TM_XH = 256;   // X^T bf16 hi as packed pairs: column k/2 holds k, k + 1 (64 cols)
constexpr uint32_t TM_XL = 320;   // X^T bf16 lo, the same way (64 cols)
constexpr uint32_t TM_UH = 384;   // U^T bf16 hi as packed pairs: column r/2 holds r, r + 1 (32 cols)
constexpr uint32_t TM_UL = 416;   // U^T bf16 lo (32 cols)
constexpr uint32_t TM_O1 = 448;   // O^T of odd chunks (64 cols): a chunk's Qt X may start before the
                                  // previous chunk's outputs have been read
constexpr uint32_t TM_COLS = 512;

constexpr int NWORK = 256;             // worker threads
constexpr int NTHREADS = NWORK + 64;   // plus the issuer and producer warps
constexpr int ISSUER = NWORK;
constexpr int PRODUCER = NWORK + 32;
// worker -> issuer handoffs of a chunk, each in two halves so that a product can start on the first:
// the state split (XA: k in [0, 32) and [64, 96); XB: the rest) and U (UA: r in [0, 16) and [32, 48);
// UB: the rest)
enum { HO_XA = 0, HO_XB = 1, HO_UA = 2, HO_UB = 3 };

__device__ int g_state_status;   // set to KDA_ERR_TIMEOUT when a bounded wait expires

// Splits 32 consecutive values (k0 .. k0 + 31 of this thread's TMEM lane) into packed bf16 hi / lo
// pairs and stores them at columns k0 / 2 .. k0 / 2 + 15 of the hi and lo operand copies.
__device__ __forceinline__ void tmem_st_split32(uint32_t t_hi, uint32_t t_lo, const float (&x)[32])
{
    uint32_t h[16], l[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) split_bf16x2(x[2 * p], x[2 * p + 1], h[p], l[p]);
    tmem_st16_nowait(t_hi, h);
    tmem_st16_nowait(t_lo, l);
}

// What a launch of the state pass produces.
enum StateMode {
    STATE_LOCAL = 0,     // every item: local outputs, qhat, summaries, local final states
    STATE_SUMMARY = 1,   // only the last piece of each segment, only its summary (A, B)
    STATE_OUTPUT = 2,    // the state-column item of every piece from its true incoming state (h0 or
                         // S_in of its segment): exact outputs and final states, no summaries
};

template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
chunk_state_tc(const int32_t *__restrict__ plan, PlanSig sig, int H, const float *__restrict__ h0,
               const float *__restrict__ s_in, const unsigned char *__restrict__ pkg, uint16_t *__restrict__ o,
               float *__restrict__ A, float *__restrict__ B, float *__restrict__ fin_state,
               uint16_t *__restrict__ qhat, float *__restrict__ afin, const __grid_constant__ CUtensorMap tm_o,
               int withhold, float *__restrict__ xs)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_mbar;      // W X, then the state product
    __shared__ __align__(8) uint64_t s_mbar_o;    // the output products of a chunk
    __shared__ __align__(8) uint64_t s_pbar1[2];  // package part 1 landed, per buffer
    __shared__ __align__(8) uint64_t s_pbar2[2];  // package part 2 landed, per buffer
    __shared__ __align__(8) uint64_t s_hbar[4];   // worker -> issuer handoffs
    __shared__ __align__(8) uint64_t s_free[2];   // issuer -> producer: package buffer free
    __shared__ uint32_t s_tmem;
    if (!plan_matches(plan, sig)) {   // not the plan the launch was sized from: touch nothing
        if (threadIdx.x == 0) record_status(&g_state_status, KDA_ERR_INVALID_ARG);
        return;
    }
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;   // 128-byte swizzle atoms
    unsigned char *const base = smem_raw + (sbase - smem_u32(smem_raw));

    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;          // TMEM lane quadrant, column half
    const bool worker = tid < NWORK, issuer = tid == ISSUER, producer = tid == PRODUCER;
    const int item = blockIdx.x / H, h = blockIdx.x % H;
    const int32_t *it = pv.item(item);
    const int p = it[0], kind = it[1];
    const int32_t *pc = pv.piece(p);
    const int start = pc[PC_START], len = pc[PC_LEN], seq = pc[PC_SEQ], seg = pc[PC_SEG];
    const int flags = pc[PC_FLAGS], row0 = pc[PC_ROW], fin = pc[PC_FIN];
    if constexpr (MODE == STATE_SUMMARY) {
        if (!(flags & KDA_PIECE_SEG_LAST)) return;   // no part in a segment summary
    }
    if constexpr (MODE == STATE_OUTPUT) {
        if (kind != 0) return;   // transitions are summaries
    }
    const int64_t T_cont = pv.T_cont();
    const int nch = (len + CH - 1) / CH;
    // global index of the piece's first chunk (chunks are numbered piece by piece): each warp sums
    // the earlier pieces' chunk counts, its lanes taking every 32nd piece
    int c0 = 0;
    for (int i = lane; i < p; i += 32) c0 += (pv.piece(i)[PC_LEN] + CH - 1) / CH;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) c0 += __shfl_xor_sync(0xffffffffu, c0, sh);
    const unsigned char *const pk0 = pkg + (static_cast<size_t>(h) * pv.n_chunks() + c0) * KDA_PACKAGE_BYTES;
    auto pk_of = [&](int ci) { return pk0 + static_cast<size_t>(ci) * KDA_PACKAGE_BYTES; };
    const uint32_t mbar = smem_u32(&s_mbar), mbar_o = smem_u32(&s_mbar_o);

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(mbar_o, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_pbar1[i]), 1);
            mbar_init(smem_u32(&s_pbar2[i]), 1);
            mbar_init(smem_u32(&s_free[i]), 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&s_hbar[i]), 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);  // this warp's lane quadrant
    const int c_lane = quad * 32 + lane;                                     // state column of this thread
    // (STATE_OUTPUT with xs) the start state of the piece's chunk ci: this thread's row c of X^T, columns
    // k0 .. k0 + 31, into xs[h][chunk] as the bf16 hi/lo image of X^T as it lies (rows c, cols k: 8-column
    // chunks of 128 rows x 16 bytes, chunk stride 2048; lo 32 KiB after hi), the backward's operand; a
    // warp's 16-byte stores cover 512 contiguous bytes
    auto record_x = [&](int ci, int k0, const float (&x)[32]) {
        if constexpr (MODE == STATE_OUTPUT) {
            if (!xs) return;
            unsigned char *const dst = reinterpret_cast<unsigned char *>(
                                           xs + (static_cast<size_t>(h) * pv.n_chunks() + c0 + ci) * KD * VD) +
                                       cm_off(c_lane, k0, 2048);
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int p2 = 0; p2 < 16; ++p2) split_bf16x2(x[2 * p2], x[2 * p2 + 1], hi[p2], lo[p2]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                *reinterpret_cast<uint4 *>(dst + q * 2048) = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
                *reinterpret_cast<uint4 *>(dst + 32768 + q * 2048) =
                    make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
            }
        }
    };

    // package parts by bulk copy (producer thread)
    auto load_p1 = [&](int ci) {
        const uint32_t bar = smem_u32(&s_pbar1[ci & 1]);
        mbar_arrive_expect_tx(bar, P1_BYTES);
        bulk_g2s(sbase + OFF_P1 + (ci & 1) * P1_BYTES, pk_of(ci) + PK_W, P1_BYTES, bar);
    };
    auto load_p2 = [&](int ci) {
        const uint32_t bar = smem_u32(&s_pbar2[ci & 1]);
        mbar_arrive_expect_tx(bar, P2_BYTES);
        bulk_g2s(sbase + OFF_P2 + (ci & 1) * P2_BYTES, pk_of(ci) + PK_QK, P2_BYTES, bar);
    };
    if (producer && nch > 0) {
        grid_dep_wait();   // the packages come from the preparation kernel
        load_p1(0);
        load_p2(0);
    }

    bool aborted = false;   // all workers agree on it (OR-reduced at barriers)
    bool bad = false;       // a bounded wait of this thread gave up
    uint32_t phase = 0;
    auto wait_mma = [&]() {
        if (!mbar_wait_warp(mbar, phase & 1)) bad = true;
        ++phase;
        fence_after();
    };
    // Workers hand a set of TMEM operands over to the issuer: every writer has waited for its TMEM
    // stores and fences them, the workers meet on named barrier 1 (OR-reducing their wait failures,
    // so all of them take the same abort decision), and one of them arrives.
    auto handoff = [&](int which) -> bool {
        fence_before();
        const bool ab = bar_or1(NWORK, bad);
        if (!ab && tid == 0) mbar_arrive(smem_u32(&s_hbar[which]));
        return ab;
    };
    // Ut^T row c_lane, columns hw*32 .. +32 of chunk ci, into registers (state columns only); the
    // package holds it as [hw][m][c] float4 groups, so each load of a warp reads 512 contiguous bytes
    float4 ut[8];
    auto load_ut = [&](int ci) {
        if (kind != 0 || ci >= nch) return;
        const float4 *src = reinterpret_cast<const float4 *>(pk_of(ci) + PK_U) + hw * 8 * 128 + c_lane;
#pragma unroll
        for (int m = 0; m < 8; ++m) ut[m] = src[m * 128];
    };

    if (worker) {
        // ---- piece start: X^T into TMEM, fp32 and as its bf16 split
        {
            bool from_h0 = kind == 0 && (flags & KDA_PIECE_FIRST) && h0 != nullptr;
            const float *src = h0 + (static_cast<size_t>(seq) * H + h) * KD * VD;
            if constexpr (MODE == STATE_OUTPUT) {
                grid_dep_wait();   // S_in comes from the composition
                if (flags & KDA_PIECE_CONT) {   // the true state entering the segment
                    from_h0 = true;
                    src = s_in + (static_cast<size_t>(seg) * H + h) * KD * VD;
                }
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float x[32];
                const int k0 = hw * 64 + half * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int kk = k0 + j;
                    x[j] = kind == 1 ? (kk == c_lane ? 1.f : 0.f) : (from_h0 ? src[kk * VD + c_lane] : 0.f);
                }
                tmem_st32(tl + TM_X + k0, x);
                tmem_st_split32(tl + TM_XH + k0 / 2, tl + TM_XL + k0 / 2, x);
                if (nch > 0) record_x(0, k0, x);
            }
            tmem_wait_st();
            grid_dep_wait();   // the packages come from the preparation kernel; every output write follows
            load_ut(0);
            aborted = handoff(HO_XA);  // -> W X, Qt X
            if (!aborted) aborted = handoff(HO_XB);
        }
        for (int ci = 0; ci < nch && !aborted; ++ci) {
            const int t0 = start + ci * CH;
            const int L = min(CH, len - ci * CH);

            // ================= U^T = Ut^T - (W X)^T, split into the A operand of the next products ===
            // in two rounds of 16 rows r each (hw*32 + [0, 16), then + [16, 32)): the state product
            // starts on the first
            wait_mma();
#pragma unroll
            for (int rd = 0; rd < 2; ++rd) {
                if (aborted) continue;   // (no break: the loop must unroll, ut is indexed by rd)
                float d[16];
                tmem_ld16(tl + TM_WX + hw * 32 + rd * 16, d);   // (W X)^T[c = c_lane][r = hw*32 + rd*16 + j]
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 u4 = kind == 0 ? ut[rd * 4 + m] : make_float4(0.f, 0.f, 0.f, 0.f);
                    d[4 * m] = u4.x - d[4 * m];
                    d[4 * m + 1] = u4.y - d[4 * m + 1];
                    d[4 * m + 2] = u4.z - d[4 * m + 2];
                    d[4 * m + 3] = u4.w - d[4 * m + 3];
                }
                uint32_t uh[8], ul[8];
#pragma unroll
                for (int p2 = 0; p2 < 8; ++p2) split_bf16x2(d[2 * p2], d[2 * p2 + 1], uh[p2], ul[p2]);
                tmem_st8_nowait(tl + TM_UH + hw * 16 + rd * 8, uh);
                tmem_st8_nowait(tl + TM_UL + hw * 16 + rd * 8, ul);
                tmem_wait_st();
                if (rd == 0 && tid == 0) bulk_wait_read_all();   // the previous O tile has left shared memory
                aborted = handoff(rd == 0 ? HO_UA : HO_UB);   // -> X^T += U^T Kh (then O^T += U^T QK^T)
            }
            if (aborted) break;
            load_ut(ci + 1);

            // ================= new X^T and its split into TMEM; outputs (or qhat) to HBM ==============
            // in two rounds of 32 columns k each (hw*64 + [0, 32), then + [32, 64)): the next chunk's
            // W X starts on the first
            wait_mma();
            {
                // this thread's half of X^T (X + Kh^T U) in one batch of TMEM reads
                uint32_t xa[32], xb[32];
                tmem_ld32_nowait(tl + TM_X + hw * 64, xa);
                tmem_ld32_nowait(tl + TM_X + hw * 64 + 32, xb);
                tmem_wait_ld();
                reg_fence32(xa);
                reg_fence32(xb);
                const float *gc = reinterpret_cast<const float *>(base + OFF_P2 + (ci & 1) * P2_BYTES + P2_GC);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int k0 = hw * 64 + half * 32;
                    float x[32];   // Diag(exp Gamma_C) (X + Kh^T U)
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(half ? xb[j] : xa[j]) * gc[k0 + j];
                    tmem_st32_nowait(tl + TM_X + k0, reinterpret_cast<const uint32_t (&)[32]>(x));
                    tmem_st_split32(tl + TM_XH + k0 / 2, tl + TM_XL + k0 / 2, x);
                    tmem_wait_st();
                    aborted = handoff(half == 0 ? HO_XA : HO_XB);   // -> next chunk's W X, Qt X
                    if (aborted) break;
                    if (ci + 1 < nch) record_x(ci + 1, k0, x);
                }
                if (aborted) break;
                if constexpr (MODE != STATE_SUMMARY) {
                    // O^T[c][r] -> bf16 tile of rows r in the TMA store layout (128-byte swizzle; the
                    // previous tile was read before the U^T handoff), then outputs (state columns) go out
                    // by tiled TMA stores, a ragged last chunk by 16-byte stores of its rows; qhat
                    // (transition columns) leaves as the two boxes lie, into the piece's qhat image
                    if (!mbar_wait_warp(mbar_o, ci & 1)) bad = true;
                    fence_after();
                    {
                        uint32_t od[32];
                        tmem_ld32_nowait(tl + ((ci & 1) ? TM_O1 : TM_O0) + hw * 32, od);   // O^T[c][r = hw*32 + j]
                        tmem_wait_ld();
                        reg_fence32(od);
                        unsigned char *ob = base + OFF_OB + (c_lane >> 6) * 8192 + (c_lane & 7) * 2;
                        const int ch = (c_lane & 63) >> 3;
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {   // one conversion per pair of rows
                            const uint32_t w = bf16x2_bits(__uint_as_float(od[j]), __uint_as_float(od[j + 1]));
                            *reinterpret_cast<uint16_t *>(ob + sw128(hw * 32 + j, ch)) = static_cast<uint16_t>(w);
                            *reinterpret_cast<uint16_t *>(ob + sw128(hw * 32 + j + 1, ch)) = static_cast<uint16_t>(w >> 16);
                        }
                    }
                    fence_async_smem();
                    bar_sync1(NWORK);
                    if (kind != 0) {
                        // qhat image of the piece: its rows in tiles of 2 CH (the last one R_t < 2 CH rows);
                        // box b (columns 64 b ..) of a tile holds its rows r at (b R_t + r) 128 bytes from the
                        // tile's start, each row's 16-byte groups in the swizzled order of the box, so that
                        // the fix-up brings a tile in with two plain bulk copies
                        const int tq = ci >> 1, r_in = (ci & 1) * CH;
                        const int R_t = min(2 * CH, len - tq * 2 * CH);
                        unsigned char *const tile = reinterpret_cast<unsigned char *>(
                            qhat + (static_cast<size_t>(h) * T_cont + row0 + tq * 2 * CH) * KD);
                        if (L == CH) {
                            if (tid == 0) {
                                bulk_s2g(tile + static_cast<size_t>(r_in) * 128, sbase + OFF_OB, 8192);
                                bulk_s2g(tile + static_cast<size_t>(R_t + r_in) * 128, sbase + OFF_OB + 8192, 8192);
                                bulk_commit_group();
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int id = tid + 256 * i, r = id >> 4, c16 = id & 15, b = c16 >> 3;
                                if (r < L)
                                    *reinterpret_cast<uint4 *>(tile + static_cast<size_t>(b * R_t + r_in + r) * 128 +
                                                               (c16 & 7) * 16) =
                                        *reinterpret_cast<const uint4 *>(base + OFF_OB + b * 8192 + r * 128 + (c16 & 7) * 16);
                            }
                        }
                    } else if (L == CH) {
                        if (tid == 0) {
                            tma_store_3d(&tm_o, 0, h, t0, sbase + OFF_OB);
                            tma_store_3d(&tm_o, 64, h, t0, sbase + OFF_OB + 8192);
                            bulk_commit_group();
                        }
                    } else {
                        uint16_t *const dst_row0 = o + (static_cast<size_t>(t0) * H + h) * VD;
                        const size_t row_stride = static_cast<size_t>(H) * VD;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int id = tid + 256 * i, r = id >> 4, c16 = id & 15;
                            if (r < L)
                                *reinterpret_cast<uint4 *>(dst_row0 + r * row_stride + c16 * 8) =
                                    *reinterpret_cast<const uint4 *>(base + OFF_OB + (c16 >> 3) * 8192 + sw128(r, c16 & 7));
                        }
                    }
                }
            }
        }
    } else if (issuer) {
        // Issuer: per chunk, W X and Qt X once the state split is in, the output / state products
        // once U^T is.  Chunk ci's state handoff means every product of chunk ci - 1 has completed,
        // so the producer may refill that chunk's package buffers with chunk ci + 1.
        // The package waits sit where the issuer idles anyway (while the workers run U and J).
        bool ok = nch == 0 || mbar_wait(smem_u32(&s_pbar1[0]), 0);
        for (int ci = 0; ci < nch && ok; ++ci) {
            const uint32_t par = ci & 1;
            const uint32_t t_o = tbase + ((ci & 1) ? TM_O1 : TM_O0);
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_XA]), par))) break;
            if (ci + 1 < nch) mbar_arrive(smem_u32(&s_free[(ci + 1) & 1]));
            fence_after();
            {
                const uint32_t p1 = sbase + OFF_P1 + (ci & 1) * P1_BYTES;
                // (W X)^T = X^T W^T (3-term; X^T from TMEM, W read MN-major): the K steps of the first
                // half of the state split (k in [0, 32) and [64, 96)), then, once it is in, the rest
                const uint32_t idw = idesc_bf16(128, 64, 0, 1);
                const uint32_t aoff[3] = {TM_XH, TM_XH, TM_XL}, boff[3] = {0, T64, 0};
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    if (hf == 1) {
                        if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_XB]), par))) break;
                        fence_after();
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int kk = (q4 & 1) + 2 * hf + 4 * (q4 >> 1);   // hf 0: 0, 1, 4, 5; hf 1: 2, 3, 6, 7
#pragma unroll
                        for (int ps = 0; ps < 3; ++ps)
                            mma_bf16_ta(tbase + TM_WX, tbase + aoff[ps] + kk * 8,
                                        sdesc(p1 + PK_W + boff[ps] + kk * 256, 128, 2048), idw,
                                        (hf | q4 | ps) != 0);
                    }
                }
                if (!ok) break;
                commit(mbar);
                if constexpr (MODE != STATE_SUMMARY) {   // O^T = X^T Qt^T (1-term)
                    const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ta(t_o, tbase + TM_XH + kk * 8, sdesc(p1 + PK_Q + kk * 2 * 1024, 1024), id, kk != 0);
                }
            }
            if (!(ok = mbar_wait(smem_u32(&s_pbar2[ci & 1]), (ci >> 1) & 1))) break;
            if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_UA]), par))) break;
            fence_after();
            {
                const unsigned char *p2 = base + OFF_P2 + (ci & 1) * P2_BYTES;
                const uint32_t s2 = smem_u32(p2);
                const uint32_t id64 = idesc_bf16(128, 64), id128 = idesc_bf16(128, 128, 0, 1);
                // X^T += U^T Kh (3-term; U^T from TMEM, Kh read MN-major): the next chunk waits on it.  The
                // K steps of U's first half (r in [0, 16) and [32, 48)), then, once it is in, the rest
                const uint32_t aoff[3] = {TM_UH, TM_UH, TM_UL}, boff[3] = {0, T64, 0};
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    if (hf == 1) {
                        if (!(ok = mbar_wait(smem_u32(&s_hbar[HO_UB]), par))) break;
                        fence_after();
                    }
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const int kk = hf + 2 * q2;   // hf 0: 0, 2; hf 1: 1, 3
#pragma unroll
                        for (int ps = 0; ps < 3; ++ps)
                            mma_bf16_ta(tbase + TM_X, tbase + aoff[ps] + kk * 8,
                                        sdesc(s2 + P2_KH + boff[ps] + kk * 256, 128, 1024), id128, 1);
                    }
                }
                if (!ok) break;
                commit(mbar);
                if constexpr (MODE != STATE_SUMMARY) {   // O^T += U^T QK^T (1-term)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ta(t_o, tbase + TM_UH + kk * 8, sdesc(s2 + P2_QK + kk * 2 * 1024, 1024), id64, 1);
                    commit(mbar_o);
                }
            }
            // the next chunk's W and Qt (issued when this chunk began)
            if (ci + 1 < nch && !(ok = mbar_wait(smem_u32(&s_pbar1[(ci + 1) & 1]), ((ci + 1) >> 1) & 1))) break;
        }
        if (!ok) record_status(&g_state_status, KDA_ERR_TIMEOUT);
    } else if (producer) {
        // Producer: chunk j's package parts once the issuer has freed their buffers (the free signal
        // of buffer j & 1 cannot run a phase ahead: the next one needs chunk j's products).
        bool ok = true;
        int n_p1[2] = {nch > 0 ? 1 : 0, 0}, n_p2[2] = {nch > 0 ? 1 : 0, 0};
        for (int j = 1; j < nch && ok; ++j) {
            if (!(ok = mbar_wait(smem_u32(&s_free[j & 1]), ((j - 1) >> 1) & 1))) break;
            if (j == withhold) continue;   // the abort-path self-test: this chunk's copies never come
            load_p1(j);
            load_p2(j);
            ++n_p1[j & 1];
            ++n_p2[j & 1];
        }
        if (!ok) record_status(&g_state_status, KDA_ERR_TIMEOUT);
        // every staged copy lands before the CTA exits (bounded waits)
        for (int b = 0; b < 2; ++b) {
            if (n_p1[b]) mbar_wait(smem_u32(&s_pbar1[b]), (n_p1[b] - 1) & 1);
            if (n_p2[b]) mbar_wait(smem_u32(&s_pbar2[b]), (n_p2[b] - 1) & 1);
        }
    }

    // ---- piece end: summaries and final states (X[k][c] from TMEM lane c, column k)
    if (worker && !aborted) {
        const size_t mat = static_cast<size_t>(KD) * VD;
        const bool seg_last = flags & KDA_PIECE_SEG_LAST, seq_end = flags & KDA_PIECE_SEQ_END;
        float *dst0 = nullptr, *dst1 = nullptr;
        if (kind == 0) {
            if (MODE != STATE_OUTPUT && seg_last) dst0 = B + (static_cast<size_t>(seg) * H + h) * mat;
            if (MODE != STATE_SUMMARY && seq_end) dst1 = fin_state + (static_cast<size_t>(seq) * H + h) * mat;
            if (MODE != STATE_OUTPUT && seg_last && (pv.seg(seg)[1] & KDA_SEG_HAS_RESET)) {
                float *za = A + (static_cast<size_t>(seg) * H + h) * KD * KD;
                for (int e = tid; e < KD * KD / 4; e += NWORK)
                    reinterpret_cast<float4 *>(za)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        } else {
            if (seg_last) dst0 = A + (static_cast<size_t>(seg) * H + h) * KD * KD;
            if (MODE == STATE_LOCAL && seq_end) dst1 = afin + (static_cast<size_t>(fin) * H + h) * KD * KD;
        }
        if (dst0 || dst1) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int k0 = hw * 64 + half * 32;
                float x[32];
                tmem_ld32(tl + TM_X + k0, x);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (dst0) dst0[(k0 + j) * VD + c_lane] = x[j];
                    if (dst1) dst1[(k0 + j) * VD + c_lane] = x[j];
                }
            }
        }
    } else if (worker && tid == 0) {
        record_status(&g_state_status, KDA_ERR_TIMEOUT);
    }
    if (tid == 0) bulk_wait_all();   // the last O tiles are written before shared memory goes away
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

// The state pass in one of its modes, as a programmatic dependent of the kernel before it.
template <int MODE>
cudaError_t launch_state(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *h0, const float *s_in,
                         const unsigned char *pkg, uint16_t *o, float *A, float *B, float *final_state,
                         uint16_t *qhat, float *afin, cudaStream_t stream, int withhold = -1, float *xs = nullptr)
{
    const PlanView pv{plan_host};
    const long long blocks = static_cast<long long>(pv.n_items()) * H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // full 64-row output chunks leave by tiled TMA stores ([T][H][V]); a tensor shorter than one chunk
    // has no full chunk, so its map stays unused
    CUtensorMap to{};
    if (MODE != STATE_SUMMARY && pv.T() >= CH &&
        !encode_rows_3d(&to, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, pv.T(), 64, CH))
        return cudaErrorInvalidValue;
    cudaError_t err = set_dynamic_smem(reinterpret_cast<const void *>(chunk_state_tc<MODE>),
                                       static_cast<int>(SMEM_ALLOC));
    if (err != cudaSuccess) return err;
    return launch_dependent(chunk_state_tc<MODE>, dim3(static_cast<unsigned>(blocks)), dim3(NTHREADS), SMEM_ALLOC,
                            stream, plan_dev, plan_sig(plan_host), H, h0, s_in, pkg, o, A, B, final_state, qhat, afin, to,
                            withhold, xs);
}

}  // namespace

cudaError_t launch_chunk_state(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *h0,
                               const unsigned char *pkg, uint16_t *o, float *A, float *B, float *final_state,
                               uint16_t *qhat, float *afin, cudaStream_t stream)
{
    return launch_state<STATE_LOCAL>(plan_host, plan_dev, H, h0, nullptr, pkg, o, A, B, final_state, qhat, afin,
                                     stream);
}

// The local chunkwise forward: the chunk-parallel preparation (in its backward mode when bimg and bterms
// are given), then the serial state pass.
cudaError_t launch_chunk_forward(const int32_t *plan_host, const int32_t *plan_dev, int H,
                                 const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const float *g, const float *beta, const float *h0, float scale,
                                 uint16_t *o, float *A, float *B, float *final_state,
                                 uint16_t *qhat, float *afin, unsigned char *pkg, cudaStream_t stream,
                                 unsigned char *bimg, float *bterms)
{
    cudaError_t err = launch_chunk_prep(plan_host, plan_dev, H, q, k, v, g, beta, scale, pkg, stream, bimg, bterms);
    if (err != cudaSuccess) return err;
    return launch_chunk_state(plan_host, plan_dev, H, h0, pkg, o, A, B, final_state, qhat, afin, stream);
}

// The forward from preceding summaries: the preparation; the segment summaries alone (the last piece of
// each segment); their composition into S_in; then every piece's chain again from its true incoming
// state, reading the same packages, which gives the outputs and final states directly.
cudaError_t launch_two_pass(const int32_t *plan_host, const int32_t *plan_dev, int H,
                            const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *g, const float *beta, const float *h0, float scale,
                            uint16_t *o, float *A, float *B, float *S_in, float *final_state,
                            unsigned char *pkg, cudaStream_t stream)
{
    cudaError_t err = launch_chunk_prep(plan_host, plan_dev, H, q, k, v, g, beta, scale, pkg, stream);
    if (err != cudaSuccess) return err;
    err = launch_state<STATE_SUMMARY>(plan_host, plan_dev, H, h0, nullptr, pkg, o, A, B, final_state, nullptr,
                                      nullptr, stream);
    if (err != cudaSuccess) return err;
    err = launch_compose(plan_host, plan_dev, H, A, B, h0, S_in, stream);
    if (err != cudaSuccess) return err;
    return launch_state<STATE_OUTPUT>(plan_host, plan_dev, H, h0, S_in, pkg, o, A, B, final_state, nullptr, nullptr,
                                      stream);
}

// Every piece's state chain from its true incoming state (h0, or S_in of its segment), recording the
// start state X of each chunk into xs[h][chunk] as the bf16 hi/lo image of X^T (K x V x 4 bytes); the
// outputs and final states go to o and final_state.  The packages and S_in come from the kernels before
// it on the stream.
cudaError_t launch_state_record(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *h0,
                                const float *S_in, const unsigned char *pkg, uint16_t *o, float *final_state,
                                float *xs, cudaStream_t stream)
{
    return launch_state<STATE_OUTPUT>(plan_host, plan_dev, H, h0, S_in, pkg, o, nullptr, nullptr, final_state,
                                      nullptr, nullptr, stream, -1, xs);
}

// Self-test of the state pass's abort path: the preparation, then the state pass with the package copies
// of every piece's second chunk withheld, so that its waits run out.
cudaError_t launch_state_abort_selftest(const int32_t *plan_host, const int32_t *plan_dev, int H,
                                        const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                                        const float *beta, const float *h0, float scale, uint16_t *o, float *A,
                                        float *B, float *final_state, uint16_t *qhat, float *afin,
                                        unsigned char *pkg, cudaStream_t stream)
{
    cudaError_t err = launch_chunk_prep(plan_host, plan_dev, H, q, k, v, g, beta, scale, pkg, stream);
    if (err != cudaSuccess) return err;
    return launch_state<STATE_LOCAL>(plan_host, plan_dev, H, h0, nullptr, pkg, o, A, B, final_state, qhat, afin,
                                     stream, 1);
}

// The status word of this file's kernel: read and cleared (the caller has synchronised the device).
int take_state_status()
{
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_state_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_state_status, &z, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return v;
}

}  // namespace kda
