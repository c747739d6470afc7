// Reverse chains of the segment-parallel KDA backward on the tensor cores.
//
// For a chunk with the forward's terms (W, Kh, Qt, masked QK, Dc = Diag(exp Gamma_C)) and the gradient G
// of the state after the chunk, the gradient of the state before it is
//     DG = Dc G,   dU = Kh DG + QK^T dO,   G' = DG + Qt^T dO - W^T dU
// (the reverse of U = Ut - W X, O = Qt X + QK U, X' = Dc (X + Kh^T U)).  A chain runs this backwards
// over a piece's chunks; the local pass starts from a zero gradient at the end of every piece that
// continues a sequence and gives the gradient of its incoming state through its own outputs (the
// backward summary Qd of the segment), the true pass starts from dfinal or from the segment's
// end-state gradient, records DG = Dc G for every chunk (as the gradient pass's bf16 operand image) and
// gives dh0 at a sequence start (cuLA PR #136,
// "feat(kda): add cuDNN concatenated-summary Kimi CP", §Summary: the following summaries are
// gathered during the backward).
//
// Mapping: one CTA per (piece, head), like the forward's state pass.  G lives transposed in TMEM
// (lane v, column k) as an FP32 accumulator, and DG next to it split into bf16 hi/lo pairs, the A
// operand of the first product.  Per chunk:
//   workers: DG = Dc G (FP32 back into the accumulator, and split)   -> issuer:
//   dU^T = dO^T QK (2-term, issued while the workers form DG) + DG^T Kh^T (3-term) -> workers:
//   -dU^T split into TMEM (meanwhile the issuer adds G^T += dO^T Qt, 2-term)       -> issuer:
//   G^T -= dU^T W (3-term)
// The operands come as ready bf16 images (written once per chunk by the forward's preparation in its
// backward mode, dO's by a small kernel) by bulk copies: the part the first product reads is
// double-buffered and arrives a chunk ahead, the part the second reads is single-buffered and arrives
// once the previous chunk's second product is done.
#include "kda_internal.cuh"
#include "tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr uint32_t A_STRIDE = 67584;                      // one buffer of the first part (66 KiB)
constexpr uint32_t OFF_A = 0;                             // two buffers
constexpr uint32_t OFF_B = 2 * A_STRIDE;                  // the second part
constexpr uint32_t SMEM_BYTES = OFF_B + RIMG_B_BYTES;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;        // the base is rounded up to 1024 bytes
static_assert(RIMG_A_BYTES <= A_STRIDE && SMEM_ALLOC <= 227 * 1024, "shared memory");

// TMEM columns
constexpr uint32_t TG = 0;      // G^T, FP32 (128 columns k)
constexpr uint32_t TDGH = 128;  // DG^T bf16 hi as packed pairs (64 columns: k / 2)
constexpr uint32_t TDGL = 192;  // DG^T bf16 lo
constexpr uint32_t TU = 256;    // dU^T, FP32 (64 columns r)
constexpr uint32_t TUH = 320;   // -dU^T bf16 hi as packed pairs (32 columns: r / 2)
constexpr uint32_t TUL = 352;   // -dU^T bf16 lo
constexpr uint32_t TM_COLS = 512;

constexpr int NWORK = 256;
constexpr int NTHREADS = NWORK + 64;   // plus the issuer and producer warps
constexpr int ISSUER = NWORK, PRODUCER = NWORK + 32;

__device__ int g_rev_status;

__device__ __forceinline__ void split_pairs32(const float (&x)[32], uint32_t (&h)[16], uint32_t (&l)[16])
{
#pragma unroll
    for (int p = 0; p < 16; ++p) split_bf16x2(x[2 * p], x[2 * p + 1], h[p], l[p]);
}

template <bool TRUE_PASS>
__global__ void __launch_bounds__(NTHREADS, 1)
reverse_tc(const int32_t *__restrict__ plan, PlanSig sig, int H, const unsigned char *__restrict__ img,
           const float *__restrict__ dfinal, const float *__restrict__ G_end, float *__restrict__ Qd,
           float *__restrict__ gs, float *__restrict__ dh0)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_pa[2];   // first part of a chunk landed, per buffer
    __shared__ __align__(8) uint64_t s_pb;      // second part landed
    __shared__ __align__(8) uint64_t s_hdg;     // workers -> issuer: DG in TMEM
    __shared__ __align__(8) uint64_t s_hu;      // workers -> issuer: -dU in TMEM
    __shared__ __align__(8) uint64_t s_m1;      // first product done
    __shared__ __align__(8) uint64_t s_m2;      // second product done
    __shared__ uint32_t s_tmem;
    if (!plan_matches(plan, sig)) {   // not the plan the launch was sized from: touch nothing
        if (threadIdx.x == 0) record_status(&g_rev_status, KDA_ERR_INVALID_ARG);
        return;
    }
    const PlanView pv{plan};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hw = warp >> 2;
    const int p = blockIdx.x / H, h = blockIdx.x % H;
    const int32_t *pc = pv.piece(p);
    const int len = pc[PC_LEN], seq = pc[PC_SEQ], seg = pc[PC_SEG], flags = pc[PC_FLAGS];
    if (!TRUE_PASS && !(flags & KDA_PIECE_CONT)) return;   // no incoming state to differentiate
    const int nch = (len + CH - 1) / CH;
    // global index of the piece's first chunk: each warp sums the earlier pieces' chunk counts
    int c0 = 0;
    for (int i = lane; i < p; i += 32) c0 += (pv.piece(i)[PC_LEN] + CH - 1) / CH;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) c0 += __shfl_xor_sync(0xffffffffu, c0, sh);
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    unsigned char *const base = smem_raw + (sbase - smem_u32(smem_raw));
    auto image = [&](int ci) {
        return img + (static_cast<size_t>(h) * pv.n_chunks() + c0 + ci) * RIMG_UNIT;
    };
    const uint32_t m1 = smem_u32(&s_m1), m2 = smem_u32(&s_m2);

    if (tid == 0) {
        mbar_init(smem_u32(&s_pa[0]), 1);
        mbar_init(smem_u32(&s_pa[1]), 1);
        mbar_init(smem_u32(&s_pb), 1);
        mbar_init(smem_u32(&s_hdg), 1);
        mbar_init(smem_u32(&s_hu), 1);
        mbar_init(m1, 1);
        mbar_init(m2, 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), TM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = s_tmem;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);   // this warp's lane quadrant
    const int v = quad * 32 + lane;                                         // value column of this thread

    if (tid < NWORK) {
        bool bad = false, aborted = false;
        // a set of TMEM operands handed to the issuer: every writer waited for its stores and fences them,
        // the workers meet on named barrier 1 (OR-reducing their wait failures), one of them arrives
        auto handoff = [&](uint64_t *bar) -> bool {
            fence_before();
            const bool ab = bar_or1(NWORK, bad);
            if (!ab && tid == 0) mbar_arrive(smem_u32(bar));
            return ab;
        };
        // ---- piece end: G^T from its source (rows k of this thread's half, column v)
        {
            const float *src = nullptr;
            if (TRUE_PASS) {
                if (flags & KDA_PIECE_SEQ_END) {
                    if (dfinal) src = dfinal + (static_cast<size_t>(seq) * H + h) * KD * VD;
                } else {
                    src = G_end + (static_cast<size_t>(seg) * H + h) * KD * VD;
                }
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int k0 = hw * 64 + half * 32;
                float x[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = src ? src[(k0 + j) * VD + v] : 0.f;
                tmem_st32(tl + TG + k0, x);
            }
            tmem_wait_st();
        }
        for (int i = 0; i < nch && !aborted; ++i) {
            const int ci = nch - 1 - i, b = i & 1;
            if (i > 0) {   // the previous chunk's second product has completed G
                if (!mbar_wait_warp(m2, (i - 1) & 1)) bad = true;
                fence_after();
            }
            if (!mbar_wait_warp(smem_u32(&s_pa[b]), (i >> 1) & 1)) bad = true;   // exp(Gamma_C) of the chunk
            const float *gc = reinterpret_cast<const float *>(base + OFF_A + b * A_STRIDE + RIMG_GC);
            // ---- G of the chunk's end, then DG = Dc G: FP32 into the accumulator (the second product adds
            //      onto it) and split into the A operand (and, in the true pass, recorded as an image)
            {
                uint32_t ga[32], gb[32];
                tmem_ld32_nowait(tl + TG + hw * 64, ga);
                tmem_ld32_nowait(tl + TG + hw * 64 + 32, gb);
                tmem_wait_ld();
                reg_fence32(ga);
                reg_fence32(gb);
                // (true pass) DG's record: this thread's row v of DG^T as the bf16 hi/lo image of DG^T as it lies
                // (rows v, cols k: 8-column chunks of 128 rows x 16 bytes, chunk stride 2048; lo 32 KiB after
                // hi), the words of its split into TMEM; a warp's 16-byte stores cover 512 contiguous bytes
                unsigned char *const rec =
                    TRUE_PASS ? reinterpret_cast<unsigned char *>(gs + (static_cast<size_t>(h) * pv.n_chunks() + c0 + ci) * KD * VD)
                              : nullptr;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int k0 = hw * 64 + half * 32;
                    float x[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(half ? gb[j] : ga[j]) * gc[k0 + j];
                    tmem_st32(tl + TG + k0, x);
                    uint32_t hi[16], lo[16];
                    split_pairs32(x, hi, lo);
                    tmem_st16_nowait(tl + TDGH + k0 / 2, hi);
                    tmem_st16_nowait(tl + TDGL + k0 / 2, lo);
                    if (TRUE_PASS) {
                        unsigned char *const dst = rec + cm_off(v, k0, 2048);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            *reinterpret_cast<uint4 *>(dst + q * 2048) =
                                make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
                            *reinterpret_cast<uint4 *>(dst + 32768 + q * 2048) =
                                make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
                        }
                    }
                }
                tmem_wait_st();
            }
            aborted = handoff(&s_hdg);   // -> dU^T = DG^T Kh^T + dO^T QK
            if (aborted) break;
            // ---- -dU^T split (rows r of this thread's half), the A operand of the second product
            if (!mbar_wait_warp(m1, i & 1)) bad = true;
            fence_after();
            {
                float d[32];
                tmem_ld32(tl + TU + hw * 32, d);
#pragma unroll
                for (int j = 0; j < 32; ++j) d[j] = -d[j];
                uint32_t hi[16], lo[16];
                split_pairs32(d, hi, lo);
                tmem_st16_nowait(tl + TUH + hw * 16, hi);
                tmem_st16_nowait(tl + TUL + hw * 16, lo);
                tmem_wait_st();
            }
            aborted = handoff(&s_hu);   // -> G^T += dO^T Qt - dU^T W
        }
        // ---- piece start: the gradient of the incoming state
        if (!aborted) {
            if (nch > 0) {
                if (!mbar_wait_warp(m2, (nch - 1) & 1)) bad = true;
                fence_after();
            }
            float *dst = nullptr;
            if (!TRUE_PASS) dst = Qd + (static_cast<size_t>(seg) * H + h) * KD * VD;
            else if ((flags & KDA_PIECE_FIRST) && dh0) dst = dh0 + (static_cast<size_t>(seq) * H + h) * KD * VD;
            if (dst && !bad) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int k0 = hw * 64 + half * 32;
                    float x[32];
                    tmem_ld32(tl + TG + k0, x);
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst[(k0 + j) * VD + v] = x[j];
                }
            }
        }
        if (bad || aborted) {
            if (tid == 0) record_status(&g_rev_status, KDA_ERR_TIMEOUT);
        }
    } else if (tid == ISSUER) {
        bool ok = true;
        uint32_t n1 = 0, n2 = 0;   // products committed
        for (int i = 0; i < nch && ok; ++i) {
            const int b = i & 1;
            const uint32_t pa = sbase + OFF_A + b * A_STRIDE, pb = sbase + OFF_B;
            if (!(ok = mbar_wait(smem_u32(&s_pa[b]), (i >> 1) & 1))) break;
            fence_after();
            // dU^T = dO^T QK + DG^T Kh^T.  The first term needs only the chunk's images: it goes in while the
            // workers form DG (the accumulator is free: the workers read the previous chunk's dU before
            // handing its split over, and that chunk's second product was issued after it).
            {
                // dO^T QK: A = dO^T (rows r, cols v, read MN-major), B(r, r') = QK[r'][r] (rows r', read MN-major)
                const uint32_t id2 = idesc_bf16(128, 64, 1, 1);
#pragma unroll
                for (int ps = 0; ps < 2; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tbase + TU, sdesc(pa + RIMG_DO + kk * 256, 128, RIMG_CS),
                                 sdesc(pa + RIMG_QK + ps * 8192 + kk * 256, 128, RIMG_CS), id2, (ps | kk) != 0);
            }
            if (!(ok = mbar_wait(smem_u32(&s_hdg), i & 1))) {
                commit(m1);   // the first term is in flight: it lands before the CTA frees its tensor memory
                ++n1;
                break;
            }
            fence_after();
            {
                // + DG^T Kh^T: A = DG^T from TMEM (K = k), B = Kh read K-major (rows r, cols k)
                const uint32_t id = idesc_bf16(128, 64);
                const uint32_t aof[3] = {TDGH, TDGH, TDGL}, bof[3] = {0, 16384, 0};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ta(tbase + TU, tbase + aof[ps] + kk * 8,
                                    sdesc(pa + RIMG_KH + bof[ps] + kk * 2 * RIMG_CS, RIMG_CS), id, 1u);
                commit(m1);
                ++n1;
            }
            if (!(ok = mbar_wait(smem_u32(&s_pb), i & 1))) break;
            fence_after();
            {
                // G^T += dO^T Qt: B(k, r) = Qt[r][k] (rows r, read MN-major).  DG is in the accumulator: this
                // term goes in while the workers split -dU.
                const uint32_t id3 = idesc_bf16(128, 128, 1, 1);
#pragma unroll
                for (int ps = 0; ps < 2; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tbase + TG, sdesc(pa + RIMG_DO + kk * 256, 128, RIMG_CS),
                                 sdesc(pb + ps * 16384 + kk * 256, 128, RIMG_CS), id3, 1u);
            }
            if (!(ok = mbar_wait(smem_u32(&s_hu), i & 1))) {
                commit(m2);   // the term in flight lands before the CTA frees its tensor memory
                ++n2;
                break;
            }
            fence_after();
            {
                // G^T += (-dU^T) W: A from TMEM (K = r), B(k, r) = W^T[k][r] (the image of W^T: rows k,
                // chunk stride 2048, read K-major)
                const uint32_t id4 = idesc_bf16(128, 128, 0, 0);
                const uint32_t aof[3] = {TUH, TUH, TUL}, bof[3] = {0, 16384, 0};
#pragma unroll
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ta(tbase + TG, tbase + aof[ps] + kk * 8,
                                    sdesc(pb + (RIMG_W - RIMG_QT) + bof[ps] + kk * 2 * 2048, 2048), id4, 1u);
                commit(m2);
                ++n2;
            }
        }
        if (!ok) record_status(&g_rev_status, KDA_ERR_TIMEOUT);
        // every committed product lands before the CTA frees its tensor memory (bounded waits)
        if (n1) mbar_wait(m1, (n1 - 1) & 1);
        if (n2) mbar_wait(m2, (n2 - 1) & 1);
    } else if (tid == PRODUCER) {
        bool ok = true;
        uint32_t na[2] = {0, 0}, nb = 0;   // copies issued per buffer
        auto copy_a = [&](int i) {   // step i's first part into buffer i & 1
            const int b = i & 1;
            const uint32_t bar = smem_u32(&s_pa[b]);
            mbar_arrive_expect_tx(bar, RIMG_A_BYTES);
            bulk_g2s(sbase + OFF_A + b * A_STRIDE, image(nch - 1 - i), RIMG_A_BYTES, bar);
            ++na[b];
        };
        auto copy_b = [&](int i) {
            const uint32_t bar = smem_u32(&s_pb);
            mbar_arrive_expect_tx(bar, RIMG_B_BYTES);
            bulk_g2s(sbase + OFF_B, image(nch - 1 - i) + RIMG_QT, RIMG_B_BYTES, bar);
            ++nb;
        };
        if (nch > 0) {
            copy_a(0);
            copy_b(0);
        }
        if (nch > 1) copy_a(1);
        for (int i = 0; i < nch && ok; ++i) {
            // step i's second product has read buffer B and buffer A of step i
            if (!(ok = mbar_wait(m2, i & 1))) break;
            if (i + 1 < nch) copy_b(i + 1);
            if (i + 2 < nch) copy_a(i + 2);
        }
        if (!ok) record_status(&g_rev_status, KDA_ERR_TIMEOUT);
        // every issued copy lands before the CTA exits (bounded waits)
        for (int b = 0; b < 2; ++b)
            if (na[b]) mbar_wait(smem_u32(&s_pa[b]), (na[b] - 1) & 1);
        if (nb) mbar_wait(smem_u32(&s_pb), (nb - 1) & 1);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

cudaError_t launch_reverse_tc(const int32_t *plan_host, const int32_t *plan_dev, int H, bool true_pass,
                              const unsigned char *img, const float *dfinal, const float *G_end, float *Qd,
                              float *gs, float *dh0, cudaStream_t stream)
{
    const PlanView pv{plan_host};
    const long long blocks = static_cast<long long>(pv.n_pieces()) * H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const void *fn = true_pass ? reinterpret_cast<const void *>(reverse_tc<true>)
                               : reinterpret_cast<const void *>(reverse_tc<false>);
    cudaError_t err = set_dynamic_smem(fn, static_cast<int>(SMEM_ALLOC));
    if (err != cudaSuccess) return err;
    const PlanSig sig = plan_sig(plan_host);
    if (true_pass)
        reverse_tc<true><<<static_cast<unsigned>(blocks), NTHREADS, SMEM_ALLOC, stream>>>(plan_dev, sig, H, img, dfinal,
                                                                                         G_end, Qd, gs, dh0);
    else
        reverse_tc<false><<<static_cast<unsigned>(blocks), NTHREADS, SMEM_ALLOC, stream>>>(plan_dev, sig, H, img, dfinal,
                                                                                          G_end, Qd, gs, dh0);
    return cudaGetLastError();
}

// The status word of this file's kernels: read and cleared (the caller has synchronised the device).
int take_reverse_status()
{
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_rev_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_rev_status, &z, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    return v;
}

}  // namespace kda
