// fp32 top-k sparse attention on CUDA cores, and the combine step that merges
// the per-chunk partial results of a split decode row.
//
// fp32 inputs need fp32 products to hold a 1e-5 relative error, which the
// tf32 tensor-core path cannot give, so this kernel uses FFMA.  One CTA per
// (head, row); 16-key tiles of gathered rows in shared memory; an exact
// running maximum per tile (akol1 TensorFold PR #4, first commit message:
// running maximum, tile sum, value sum), precise expf, the sink folded in at
// the end (TensorFold PR #1206, "What changes").
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "dsa_internal.h"
#include "dsa_merge.cuh"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kSimtThreads = 128;
constexpr int kSimtTile = 16;

#define DSA_R8(x) x, x, x, x, x, x, x, x
#define DSA_R64(x) DSA_R8(DSA_R8(x))
// Source row for an out-of-range selection: NaN everywhere.
__device__ __align__(16) uint32_t kNanRowF32[512] = {
    DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u),
    DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u)};

__global__ void __launch_bounds__(kSimtThreads) dsa_simt_kernel(const SimtParams p) {
    __shared__ __align__(16) float qs[kD];
    __shared__ __align__(16) float kvs[kSimtTile][kD];
    __shared__ float sc[kSimtTile];
    __shared__ float ps[kSimtTile];

    const int h = blockIdx.x, r = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const float* qrow = p.q + (static_cast<size_t>(r) * p.H + h) * kD;
    reinterpret_cast<float4*>(qs)[tid] = reinterpret_cast<const float4*>(qrow)[tid];

    const int ns = p.n_sel[r];
    const bool bad_n = ns < 0 || ns > p.k_max;
    if (bad_n && h == 0 && tid == 0) atomicOr(p.err, DSA_DEVERR_NSEL_RANGE);
    const int eff = bad_n ? 1 : ns;
    const float* cache = p.kv + (p.decode ? static_cast<size_t>(r / p.decode) * p.N * kD : 0);
    const float* nan_row = reinterpret_cast<const float*>(kNanRowF32);

    float m = -INFINITY, l = 0.0f;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};

    for (int t0 = 0; t0 < eff; t0 += kSimtTile) {
        const int nk = min(kSimtTile, eff - t0);
        // gather: nk rows, thread tid copies float4 number tid of each row
        for (int j = 0; j < nk; ++j) {
            const float* src = nan_row;
            if (!bad_n) {
                const int id = p.idx[static_cast<size_t>(r) * p.k_max + t0 + j];
                if (id >= 0 && id < p.N) {
                    src = cache + static_cast<size_t>(id) * kD;
                } else if (h == 0 && tid == 0) {
                    atomicOr(p.err, DSA_DEVERR_IDX_RANGE);
                }
            }
            reinterpret_cast<float4*>(kvs[j])[tid] = reinterpret_cast<const float4*>(src)[tid];
        }
        __syncthreads();
        // scores: warp w takes keys 4w .. 4w+3; lane sums d = lane + 32 i in order
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int j = warp * 4 + jj;
            if (j < nk) {
                float part = 0.0f;
#pragma unroll
                for (int i = 0; i < kD / 32; ++i) part = fmaf(qs[lane + 32 * i], kvs[j][lane + 32 * i], part);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (lane == 0) sc[j] = part * p.scale;
            }
        }
        __syncthreads();
        float tm = -INFINITY;
        for (int j = 0; j < nk; ++j) tm = fmaxf(tm, sc[j]);
        const float mn = (m == -INFINITY) ? tm : fmaxf(m, tm);
        const float mu_new = (mn == -INFINITY) ? 0.0f : mn;
        const float al = (m == -INFINITY) ? 1.0f : expf(m - mu_new);
        if (tid < nk) ps[tid] = expf(sc[tid] - mu_new);
        __syncthreads();
        float ls = 0.0f;
        for (int j = 0; j < nk; ++j) ls += ps[j];
        l = l * al + ls;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int d = tid + 128 * i;
            float a = acc[i] * al;
            for (int j = 0; j < nk; ++j) a = fmaf(ps[j], kvs[j][d], a);
            acc[i] = a;
        }
        m = mn;
        __syncthreads();
    }

    // sink fold: out = acc * e^{mu - m*} / (l e^{mu - m*} + e^{sink - m*})
    const float mu = (m == -INFINITY) ? 0.0f : m;
    const float sk = p.sink[h];
    const float mstar = isfinite(sk) ? fmaxf(mu, sk) : mu;
    const float e1 = expf(mu - mstar);
    const float e2 = expf(sk - mstar);
    const float f = e1 / (l * e1 + e2);
    const size_t o0 = (static_cast<size_t>(r) * p.H + h) * kD;
    if (p.out_bf16) {
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + o0;
#pragma unroll
        for (int i = 0; i < 4; ++i) orow[tid + 128 * i] = __float2bfloat16_rn(acc[i] * f);
    } else {
        float* orow = static_cast<float*>(p.out) + o0;
#pragma unroll
        for (int i = 0; i < 4; ++i) orow[tid + 128 * i] = acc[i] * f;
    }
}

// One CTA per (row, head); thread t owns columns 4t .. 4t+3.  Partials of
// one row are merged in chunk order (dsa_merge.cuh), so the result is
// deterministic and the same as the merge inside the tensor-core kernel.
__global__ void __launch_bounds__(128) dsa_combine_kernel(const CombineParams p) {
    grid_launch_dependents();
    grid_dependency_wait();          // the split kernel's partials are complete
    merge_row_head(p.part, p.units, p.chunks, p.H, blockIdx.x, blockIdx.y, threadIdx.x, p.sink[blockIdx.y],
                   p.out, p.out_bf16);
}

}  // namespace

cudaError_t launch_simt(const SimtParams& p, cudaStream_t s) {
    dim3 grid(p.H, p.R);
    dsa_simt_kernel<<<grid, kSimtThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
    // launched while the split kernel still runs; it waits for that kernel
    // before it reads the partials
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.R), static_cast<unsigned>(p.H));
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dsa_combine_kernel, p);
}

}  // namespace dsa
