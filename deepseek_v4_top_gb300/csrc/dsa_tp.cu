// Head-sharded tensor parallelism around the attention calls (TensorFold
// PR #1206, "What changes": the 64 heads are split over the ranks, 16 a rank
// at world 4; heads added to fill the last rank get zero sinks; the output
// groups are gathered before the output projections).
//
// A rank runs the ordinary attention call over its own heads.  Around it
// this file gives the host-side plan (which heads a rank owns), a kernel
// that cuts a rank's heads out of full q and sink arrays (zero q and zero
// sink for padding heads), and a kernel that lays the ranks' gathered
// outputs, [world][R][heads a rank][512] as a collective all-gather leaves
// them, out as [R][H][512] with the padding heads dropped.  Both kernels
// only move bytes: a head's values are copied bit for bit.
#include <stdint.h>

#include "../../include/dsa.h"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kCopyThreads = 256;

// q_local [R][hpr][512] from q [R][H][512]: head j of the rank is global
// head first + j, zero when that is a padding head (>= H).  One 16-byte
// vector a thread-step; row bytes = 512 * esz, a multiple of 16.
__global__ void __launch_bounds__(kCopyThreads)
    dsa_shard_heads_kernel(const uint4* __restrict__ q, uint4* __restrict__ q_local, const float* sink,
                           float* sink_local, long long R, int H, int hpr, int first, int vec_per_row) {
    const long long n = R * hpr * vec_per_row;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int v = static_cast<int>(i % vec_per_row);
        const long long rj = i / vec_per_row;
        const int j = static_cast<int>(rj % hpr);
        const long long r = rj / hpr;
        const int h = first + j;
        q_local[i] = h < H ? q[(r * H + h) * vec_per_row + v] : make_uint4(0u, 0u, 0u, 0u);
    }
    if (blockIdx.x == 0)
        for (int j = threadIdx.x; j < hpr; j += blockDim.x) sink_local[j] = first + j < H ? sink[first + j] : 0.0f;
}

// out [R][H][512] from gathered [world][R][hpr][512]: head h comes from rank
// h / hpr, its head h % hpr.
__global__ void __launch_bounds__(kCopyThreads)
    dsa_unshard_heads_kernel(const uint4* __restrict__ gathered, uint4* __restrict__ out, long long R, int H,
                             int hpr, int vec_per_row) {
    const long long n = R * H * vec_per_row;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int v = static_cast<int>(i % vec_per_row);
        const long long rh = i / vec_per_row;
        const int h = static_cast<int>(rh % H);
        const long long r = rh / H;
        const int w = h / hpr, j = h - w * hpr;
        out[i] = gathered[((static_cast<long long>(w) * R + r) * hpr + j) * vec_per_row + v];
    }
}

int copy_grid(long long vectors) {
    const long long b = (vectors + kCopyThreads - 1) / kCopyThreads;
    return static_cast<int>(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

size_t esize(dsa_dtype dt) { return dt == DSA_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dsa

extern "C" {

dsa_status dsa_head_shard(int H, int world, int rank, dsa_head_shard_plan* plan) {
    if (!plan || H < 1 || world < 1 || rank < 0 || rank >= world) return DSA_ERR_INVALID_ARG;
    const int hpr = (H + world - 1) / world;
    if (hpr > 64) return DSA_ERR_UNSUPPORTED;   // one attention call takes at most 64 heads
    plan->heads_per_rank = hpr;
    plan->padded_heads = hpr * world;
    plan->first_head = hpr * rank;
    const int real = H - plan->first_head;
    plan->real_heads = real < 0 ? 0 : (real > hpr ? hpr : real);
    return DSA_OK;
}

dsa_status dsa_shard_heads(const void* q, const float* sink, void* q_local, float* sink_local, int R, int H,
                           int world, int rank, dsa_dtype dtype, void* stream) {
    dsa_head_shard_plan plan;
    dsa_status st = dsa_head_shard(H, world, rank, &plan);
    if (st != DSA_OK) return st;
    if (R < 0) return DSA_ERR_INVALID_ARG;
    if (dtype != DSA_F32 && dtype != DSA_BF16) return DSA_ERR_UNSUPPORTED;
    if (R == 0) return DSA_OK;
    if (!q || !sink || !q_local || !sink_local) return DSA_ERR_INVALID_ARG;
    if (!dsa::aligned16(q) || !dsa::aligned16(q_local)) return DSA_ERR_INVALID_ARG;
    const int vec = static_cast<int>(dsa::kD * dsa::esize(dtype) / 16);
    const long long n = static_cast<long long>(R) * plan.heads_per_rank * vec;
    dsa::dsa_shard_heads_kernel<<<dsa::copy_grid(n), dsa::kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(q), static_cast<uint4*>(q_local), sink, sink_local, R, H, plan.heads_per_rank,
        plan.first_head, vec);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_unshard_heads(const void* gathered, void* out, int R, int H, int world, dsa_dtype dtype,
                             void* stream) {
    dsa_head_shard_plan plan;
    dsa_status st = dsa_head_shard(H, world, 0, &plan);
    if (st != DSA_OK) return st;
    if (R < 0) return DSA_ERR_INVALID_ARG;
    if (dtype != DSA_F32 && dtype != DSA_BF16) return DSA_ERR_UNSUPPORTED;
    if (R == 0) return DSA_OK;
    if (!gathered || !out || !dsa::aligned16(gathered) || !dsa::aligned16(out)) return DSA_ERR_INVALID_ARG;
    const int vec = static_cast<int>(dsa::kD * dsa::esize(dtype) / 16);
    const long long n = static_cast<long long>(R) * H * vec;
    dsa::dsa_unshard_heads_kernel<<<dsa::copy_grid(n), dsa::kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(gathered), static_cast<uint4*>(out), R, H, plan.heads_per_rank, vec);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // extern "C"
