// Internal definitions shared by the libkda translation units (not installed).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int KD = KDA_HEAD_DIM_K;  // key dimension
constexpr int VD = KDA_HEAD_DIM_V;  // value dimension
constexpr int CH = KDA_CHUNK;       // chunk length

// Plan-word accessors (valid on host and device; 'w' points at plan word 0).
struct PlanView {
    const int32_t *w;
    __host__ __device__ int32_t T() const { return w[KDA_PH_T]; }
    __host__ __device__ int32_t N() const { return w[KDA_PH_N]; }
    __host__ __device__ int32_t S() const { return w[KDA_PH_S]; }
    __host__ __device__ int32_t n_pieces() const { return w[KDA_PH_NPIECES]; }
    __host__ __device__ int32_t n_cont() const { return w[KDA_PH_NCONT]; }
    __host__ __device__ int32_t T_cont() const { return w[KDA_PH_TCONT]; }
    __host__ __device__ int32_t n_fin() const { return w[KDA_PH_NFIN]; }
    __host__ __device__ int32_t n_items() const { return w[KDA_PH_NITEMS]; }
    __host__ __device__ const int32_t *bounds() const { return w + w[KDA_PH_OFF_BOUNDS]; }
    __host__ __device__ const int32_t *cu() const { return w + w[KDA_PH_OFF_CU]; }
    __host__ __device__ const int32_t *seg(int j) const { return w + w[KDA_PH_OFF_SEGS] + 4 * j; }
    __host__ __device__ const int32_t *piece(int i) const { return w + w[KDA_PH_OFF_PIECES] + 8 * i; }
    __host__ __device__ const int32_t *item(int i) const { return w + w[KDA_PH_OFF_ITEMS] + 2 * i; }
    __host__ __device__ const int32_t *cont(int i) const { return w + w[KDA_PH_OFF_CONT] + 4 * i; }
    __host__ __device__ const int32_t *fin(int i) const { return w + w[KDA_PH_OFF_FIN] + 4 * i; }
    __host__ __device__ int32_t n_chunks() const { return w[KDA_PH_NCHUNKS]; }
    // chunk records: piece, start token, rows, index within the piece (pieces in order)
    __host__ __device__ const int32_t *chunk(int i) const { return w + w[KDA_PH_OFF_CHUNKS] + 4 * i; }
};

// Identity of the host plan a launch was sized from: its length and checksum words.  Every kernel
// compares them with its device plan before it reads anything else from it.
struct PlanSig {
    int32_t total, checksum;
};
inline PlanSig plan_sig(const int32_t *plan_host) { return PlanSig{plan_host[KDA_PH_TOTAL], plan_host[KDA_PH_CHECKSUM]}; }
__device__ __forceinline__ bool plan_matches(const int32_t *plan_dev, PlanSig s)
{
    return plan_dev[KDA_PH_TOTAL] == s.total && plan_dev[KDA_PH_CHECKSUM] == s.checksum;
}

// Records an error code in a kernel's device status word unless an earlier one is there.
__device__ __forceinline__ void record_status(int *word, int code) { atomicCAS(word, 0, code); }

// Chunk package: the operands one (chunk, head) hands from the preparation kernel to the state
// pass, each tile in the shared-memory layout its MMA reads (byte offsets; bf16 tiles in the
// no-swizzle core-matrix layout, hi then lo where split).
enum : uint32_t {
    PK_W = 0,          // W = T' Kt, read MN-major: rows k (128), cols r (64), CS 2048, hi | lo
    PK_Q = 32768,      // Qt (scaled) hi, K-major: rows r (64), cols k (128), CS 1024
    PK_P1_END = 49152,
    PK_QK = 49152,     // masked Qt Kh^T, K-major: rows r (64), cols i (64), CS 1024
    PK_KH = 57344,     // Kh, read MN-major: rows i (64), cols k (128), CS 1024, hi | lo
    PK_GC = 90112,     // exp(Gamma_C), 128 fp32
    PK_P2_END = 90624,
    PK_U = 90624,      // Ut^T = (T' V)^T, fp32 (128 x 64) as float4 groups [r / 32][(r % 32) / 4][c]
    PK_END = 123392
};
static_assert(static_cast<uint32_t>(PK_END) == static_cast<uint32_t>(KDA_PACKAGE_BYTES), "package size");

// Piece record fields.
enum { PC_START = 0, PC_LEN = 1, PC_SEQ = 2, PC_SEG = 3, PC_FLAGS = 4, PC_CONT = 5, PC_ROW = 6, PC_FIN = 7 };

// Workspace regions resolved to typed device pointers.
struct Workspace {
    uint16_t *qhat;       // H * T_cont * K bf16: per continuing piece, 128-row tile images
    float *afin;          // [n_fin][H][K][K]
    unsigned char *pkg;   // [H][n_chunks][KDA_PACKAGE_BYTES]
    float *A;             // [S][H][K][K]
    float *B;      // [S][H][K][V]
    float *S_in;   // [S][H][K][V]
};

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// Checksum of a plan's words by the rule of kda.h (the checksum word taken as 0).
uint32_t plan_checksum_words(const int32_t *plan, size_t total);

// Records a cudaError_t for kda_last_cuda_error() on the calling thread.
void record_cuda_error(int err);

// Number of SMs of the current device (cached per device).
int sm_count();
cudaError_t current_context_id(unsigned long long *id);   // unique id of the current context
cudaError_t set_dynamic_smem(const void *fn, int bytes);   // once per (kernel, context)

// Each kernel file's device status word (KDA_ERR_TIMEOUT once a bounded wait of its kernel expired),
// read and cleared; the device must be synchronised first.
int take_prep_status();
int take_state_status();
int take_compose_status();
int take_boundary_status();
int take_backward_status();
cudaError_t launch_wait_expiry_probe(cudaStream_t stream);
cudaError_t launch_state_record(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *h0,
                                const float *S_in, const unsigned char *pkg, uint16_t *o, float *final_state,
                                float *xs, cudaStream_t stream);
cudaError_t launch_state_abort_selftest(const int32_t *plan_host, const int32_t *plan_dev, int H,
                                        const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                                        const float *beta, const float *h0, float scale, uint16_t *o, float *A,
                                        float *B, float *final_state, uint16_t *qhat, float *afin,
                                        unsigned char *pkg, cudaStream_t stream);

// Launches a kernel that may begin while the previous kernel on the stream finishes (programmatic
// dependent launch): its CTAs can be scheduled once every CTA of that kernel has signalled (or
// exited), and the kernel itself waits (griddepcontrol.wait) before it touches anything the previous
// kernel writes.  For kernels whose inputs come from the library's own previous kernel only.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// cuTensorMapEncodeTiled from the driver (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn();

// Tensor map of a row-major [rows][128] fp32 matrix with a box of 32 columns x box_rows
// rows and the 128-byte swizzle (16-byte chunk c of box row r lands at chunk c ^ (r % 8)).
bool encode_f32_rows128(CUtensorMap *m, const void *ptr, uint64_t rows, uint32_t box_rows);
// The same for a row-major [rows][cols] fp32 matrix (cols a multiple of 32).
bool encode_f32_rows(CUtensorMap *m, const void *ptr, uint64_t rows, uint32_t cols, uint32_t box_rows);

// Tensor map of a [T][H][128] tensor (inner dimension first) with a box of 'inner' columns x 1
// head x box_rows rows and the 128-byte swizzle; elem = element bytes.
bool encode_rows_3d(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, uint32_t elem, int H, int T,
                    uint32_t inner, uint32_t box_rows = 64);

// Launchers (return cudaError_t of the launch).
cudaError_t launch_chunk_forward(const int32_t *plan_host, const int32_t *plan_dev, int H,
                                 const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const float *g, const float *beta, const float *h0, float scale,
                                 uint16_t *o, float *A, float *B, float *final_state,
                                 uint16_t *qhat, float *afin, unsigned char *pkg, cudaStream_t stream,
                                 unsigned char *bimg = nullptr, float *bterms = nullptr);
// With bimg and bterms (the backward's per-unit images and FP32 terms), the preparation also writes
// those: its backward mode.
cudaError_t launch_chunk_prep(const int32_t *plan_host, const int32_t *plan_dev, int H, const uint16_t *q,
                              const uint16_t *k, const uint16_t *v, const float *g, const float *beta, float scale,
                              unsigned char *pkg, cudaStream_t stream, unsigned char *bimg = nullptr,
                              float *bterms = nullptr);
cudaError_t launch_chunk_state(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *h0,
                               const unsigned char *pkg, uint16_t *o, float *A, float *B, float *final_state,
                               uint16_t *qhat, float *afin, cudaStream_t stream);
cudaError_t launch_compose(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *A,
                           const float *B, const float *h0, float *S_in, cudaStream_t stream);
// The two-level (blocked) scan: group totals, a chain over the groups, then every group from its
// incoming state; 'scratch' holds scan_scratch_bytes(plan_host, H) bytes.
cudaError_t launch_compose_blocked(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *A,
                                   const float *B, const float *h0, float *S_in, void *scratch, cudaStream_t stream);
size_t scan_scratch_bytes(const int32_t *plan_host, int H);
// The backward (FP32 matrices, products on tcgen05): see backward.cu.  'scratch' holds grid x
// backward_scratch_floats() floats; xs and gs hold, per (head, chunk), K x V x 4 bytes: the bf16 hi/lo
// images (rows v, cols k, 8-column chunks of 128 rows x 16 bytes, lo 32 KiB after hi) of X^T (the chunk's
// start state) and of DG^T (DG = Dc G, G its end-state gradient); G_end and Qd are [S][H][K][V] floats.
size_t backward_scratch_floats();
// The FP32 chunk terms the backward's gradient pass reads element-wise or as an accumulated input, per
// (head, chunk) (floats, row-major): Ut (64 x 128) and S = strictly_lower(Kt Kh^T) (64 x 64).  The
// preparation kernel writes them in its backward mode.
constexpr int BT_UT = 0, BT_S = 64 * 128, BT_FLOATS = BT_S + 64 * 64;
// Per-(chunk, head) operand images of the backward (bytes), written by the preparation kernel's
// backward mode (dO by its own small kernel): bf16 tiles in the no-swizzle canonical layout (8-column
// chunks of the tile's rows x 16 bytes), hi then lo where split.  The part the first product of a
// reverse chain step reads (Kh rows r x cols k, QK rows r' x cols r, dO rows r x cols v, each with
// chunk stride RIMG_CS, and exp(Gamma_C) as 128 fp32) comes first, then the part the second reads (Qt
// rows r x cols k, chunk stride RIMG_CS; W as its transpose, rows k x cols r, chunk stride 2048), then
// what only the gradient pass reads: Diag(beta) Kt (rows r x cols k), Diag(beta) V (rows r x cols v) and
// T (rows r x cols i), chunk stride RIMG_CS.
constexpr uint32_t RIMG_CS = 1024;
constexpr uint32_t RIMG_KH = 0, RIMG_QK = 32768, RIMG_DO = 49152, RIMG_GC = 65536, RIMG_A_BYTES = 66048;
constexpr uint32_t RIMG_QT = 66560, RIMG_W = RIMG_QT + 32768, RIMG_B_BYTES = 65536;
constexpr uint32_t RIMG_BKT = RIMG_QT + RIMG_B_BYTES, RIMG_BV = RIMG_BKT + 32768, RIMG_T = RIMG_BV + 32768;
constexpr uint32_t RIMG_UNIT = RIMG_T + 16384;
static_assert(RIMG_UNIT % 1024 == 0 && RIMG_QT % 1024 == 0 && RIMG_A_BYTES % 16 == 0, "image layout");
cudaError_t launch_reverse_tc(const int32_t *plan_host, const int32_t *plan_dev, int H, bool true_pass,
                              const unsigned char *img, const float *dfinal, const float *G_end, float *Qd,
                              float *gs, float *dh0, cudaStream_t stream);
int take_reverse_status();
cudaError_t launch_backward(const int32_t *plan_host, const int32_t *plan_dev, int H, const uint16_t *q,
                            const uint16_t *k, const uint16_t *v, const float *g, const float *beta, float scale,
                            const uint16_t *dout, const float *dfinal, const float *A, const float *afin,
                            const float *xs, float *gs, float *G_end, float *Qd, const float *S_in,
                            const float *fin_out, float *terms, unsigned char *img, float *scratch, int grid, float *dq,
                            float *dk, float *dv, float *dg, float *dbeta, float *dh0, cudaStream_t stream);
// Segments per group of the blocked scan (about sqrt(S)) and the number of groups.
int scan_group_size(int S);
cudaError_t launch_boundary(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *S_in,
                            const uint16_t *qhat, const float *afin, uint16_t *o, float *final_state,
                            cudaStream_t stream);
cudaError_t launch_two_pass(const int32_t *plan_host, const int32_t *plan_dev, int H,
                            const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const float *g, const float *beta, const float *h0, float scale,
                            uint16_t *o, float *A, float *B, float *S_in, float *final_state,
                            unsigned char *pkg, cudaStream_t stream);

}  // namespace kda
