// Internal interface between the host API (dsa_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsa {

constexpr int kD = 512;             // latent row width
constexpr int kTileKeys = 128;      // keys per tensor-core tile (MMA M)
constexpr int kHeadsPad = 64;       // heads per tensor-core tile (MMA N)
// Decode rows are split into key chunks of this size so that a small batch
// still spreads over many SMs; each chunk leaves (m, l, O) partials that a
// second kernel merges in chunk order.  It depends only on the call's shape,
// so a row's result does not depend on the rest of the batch.
constexpr int kDecodeChunkKeys = 128;
// Floats of one chunk's partial result: O [64][512] plus (m, l) [2][64].
constexpr size_t kPartialFloats = static_cast<size_t>(kHeadsPad) * kD + 2 * kHeadsPad;

// One launch of the tensor-core kernel.  A unit is (row, key chunk): keys
// [chunk * chunk_keys, min((chunk + 1) * chunk_keys, n_sel)) of one row.
// launch_tc() fills tmap_q from q, R and H.
struct TcParams {
    CUtensorMap tmap_q;       // [R*H][512] bf16, box 64 x H, 128-byte swizzle
    const uint16_t* q;        // [R][H][512] bf16
    const uint16_t* kv;       // [N][512] or [R][N][512] bf16
    const int32_t* idx;       // [R][k_max]
    const int32_t* n_sel;     // [R]
    const float* sink;        // [H]
    void* out;                // final mode: [R][H][512], fp32 or (out_bf16) bf16
    int out_bf16;
    float* part;              // partial mode: O [units][64][512] then (m, l) [units][2][64]
    uint32_t* err;            // device error word
    int* queue;               // null: units round-robin over the grid; else the launch's unit
                              // queue [next ticket, CTAs finished], zero at launch, left zero
    float scale_log2;         // scale * log2(e)
    int R, H, N, k_max;
    int decode;               // 0: prefill (one cache); T >= 1: row r reads slot r / T
    int chunk_keys;           // keys per unit (multiple of 16)
    int chunks;               // units per row
    int units;                // R * chunks
    int partial;              // 1: write partials instead of final outputs
};

struct SimtParams {
    const float* q;
    const float* kv;
    const int32_t* idx;
    const int32_t* n_sel;
    const float* sink;
    void* out;                // [R][H][512], fp32 or (out_bf16) bf16
    int out_bf16;
    uint32_t* err;
    float scale;
    int R, H, N, k_max;
    int decode;               // as TcParams::decode
};

struct CombineParams {
    const float* part;        // as TcParams::part
    const float* sink;
    void* out;                // [R][H][512], fp32 or (out_bf16) bf16
    int out_bf16;
    int R, H, chunks, units;
};

// One launch of the top-k selection kernel (dsa_topk.cu).
struct TopkParams {
    const float* scores;      // [R][ld] (ld a multiple of 4, rows 16-byte aligned)
    const int32_t* n_valid;   // [R]: row r's candidates are positions [0, n_valid[r])
    int32_t* idx;             // [R][k_max]
    int32_t* n_sel;           // [R]
    uint32_t* err;            // device error word
    int R, ld, k, k_max;
    // rows longer than one share (4096 positions) are selected in two steps
    // through a scratch of [R][cand_ld] keys and positions: the picks of the
    // row's `shares` shares, k each, share after share
    int shares;               // topk_shares(ld)
    int cand_ld;              // >= shares * k, a multiple of 4
    uint32_t* cand_key;
    int32_t* cand_pos;
};

// Largest k and row length the top-k kernel takes.
constexpr int kTopkMaxK = 2048;
constexpr int kTopkMaxLd = 32768;
int topk_shares(int ld);
cudaError_t launch_topk(const TopkParams& p, int grid, cudaStream_t s);

// Shared memory of the tensor-core kernel (bytes, dynamic).
size_t tc_smem_bytes();

cudaError_t launch_tc(const TcParams& p, int grid, cudaStream_t s);
cudaError_t launch_simt(const SimtParams& p, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* err, cudaStream_t s);
// out [M][N] fp32 = a [M][K] bf16 . b [K][N] bf16 on the tensor cores
// (dsa_gemm.cu); K and N multiples of 8, pointers 16-byte aligned.
cudaError_t launch_gemm(const void* a, const void* b, float* out, int M, int K, int N, uint32_t* err, int sms,
                        cudaStream_t s);

// Drops the cached device addresses of the no-allocation decode's static
// array (dsa_noalloc.cu), so that the next call looks them up again: after
// dsa_shutdown() the caller may reset the device, which reloads the module
// and can move the array.
void noalloc_forget();

}  // namespace dsa
