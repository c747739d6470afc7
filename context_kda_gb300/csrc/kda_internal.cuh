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
};

// Piece record fields.
enum { PC_START = 0, PC_LEN = 1, PC_SEQ = 2, PC_SEG = 3, PC_FLAGS = 4, PC_CONT = 5, PC_ROW = 6, PC_FIN = 7 };

// Workspace regions resolved to typed device pointers.
struct Workspace {
    float *qhat;   // [H][T_cont][K]
    float *afin;   // [n_fin][H][K][K]
    float *A;      // [S][H][K][K]
    float *B;      // [S][H][K][V]
    float *S_in;   // [S][H][K][V]
};

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// Records a cudaError_t for kda_last_cuda_error() on the calling thread.
void record_cuda_error(int err);

// Number of SMs of the current device (cached per device).
int sm_count();

// cuTensorMapEncodeTiled from the driver (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn();

// Tensor map of a row-major [rows][128] fp32 matrix with a box of 32 columns x box_rows
// rows and the 128-byte swizzle (16-byte chunk c of box row r lands at chunk c ^ (r % 8)).
bool encode_f32_rows128(CUtensorMap *m, const void *ptr, uint64_t rows, uint32_t box_rows);

// Launchers (return cudaError_t of the launch).
cudaError_t launch_chunk_forward(const int32_t *plan_host, const int32_t *plan_dev, int H,
                                 const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const float *g, const float *beta, const float *h0, float scale,
                                 uint16_t *o, float *A, float *B, float *final_state,
                                 float *qhat, float *afin, cudaStream_t stream);
cudaError_t launch_compose(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *A,
                           const float *B, const float *h0, float *S_in, cudaStream_t stream);
cudaError_t launch_boundary(const int32_t *plan_host, const int32_t *plan_dev, int H, const float *S_in,
                            const float *qhat, const float *afin, uint16_t *o, float *final_state,
                            cudaStream_t stream);

}  // namespace kda
