// fp32 top-k sparse attention on CUDA cores, and the combine step that merges
// the per-chunk partial results of a split decode row.
//
// fp32 inputs need fp32 products to hold a 1e-5 relative error, which the
// tf32 tensor-core path cannot give, so this kernel uses FFMA.  One CTA per
// (row, group of 8 heads), one warp per head: each 16-key tile of gathered
// rows is staged in shared memory once and serves the group's 8 heads.  An
// exact running maximum per tile (akol1 TensorFold PR #4, first commit
// message: running maximum, tile sum, value sum), precise expf, the sink
// folded in at the end (TensorFold PR #1206, "What changes").
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "dsa_internal.h"
#include "dsa_merge.cuh"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kSimtHeads = 8;                 // heads (warps) a CTA
constexpr int kSimtThreads = 32 * kSimtHeads;
constexpr int kSimtTile = 16;
constexpr size_t kSimtSmem = (static_cast<size_t>(kSimtHeads) + kSimtTile) * kD * sizeof(float);

#define DSA_R8(x) x, x, x, x, x, x, x, x
#define DSA_R64(x) DSA_R8(DSA_R8(x))
// Source row for an out-of-range selection: NaN everywhere.
__device__ __align__(16) uint32_t kNanRowF32[512] = {
    DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u),
    DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u), DSA_R64(0x7FC00000u)};

// Warp w handles head 8 blockIdx.x + w of row blockIdx.y; lane l owns the
// output columns l + 32 i.  A key's score is the lane's in-order FFMA sum
// over its 16 columns, then a fixed butterfly over the lanes.
__global__ void __launch_bounds__(kSimtThreads) dsa_simt_kernel(const SimtParams p) {
    extern __shared__ __align__(16) float simt_smem[];
    float* qs = simt_smem;                                // [8][512]
    float* kvs = simt_smem + kSimtHeads * kD;             // [16][512]

    const int r = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = kSimtHeads * blockIdx.x + warp;
    const bool live = h < p.H;

    if (live) {
        const float4* qrow = reinterpret_cast<const float4*>(p.q + (static_cast<size_t>(r) * p.H + h) * kD);
#pragma unroll
        for (int i = 0; i < 4; ++i) reinterpret_cast<float4*>(qs + warp * kD)[lane + 32 * i] = qrow[lane + 32 * i];
    }

    const int ns = p.n_sel[r];
    const bool bad_n = ns < 0 || ns > p.k_max;
    if (bad_n && blockIdx.x == 0 && tid == 0) atomicOr(p.err, DSA_DEVERR_NSEL_RANGE);
    const int eff = bad_n ? 1 : ns;
    const float* cache = p.kv + (p.decode ? static_cast<size_t>(r / p.decode) * p.N * kD : 0);
    const float* nan_row = reinterpret_cast<const float*>(kNanRowF32);

    float m = -INFINITY, l = 0.0f;
    float acc[kD / 32];
#pragma unroll
    for (int i = 0; i < kD / 32; ++i) acc[i] = 0.0f;

    for (int t0 = 0; t0 < eff; t0 += kSimtTile) {
        const int nk = min(kSimtTile, eff - t0);
        __syncthreads();             // the previous tile's rows have been read
        // gather: row j = e / 128 of the tile, float4 e % 128 of the row
        for (int e = tid; e < nk * (kD / 4); e += kSimtThreads) {
            const int j = e / (kD / 4), c4 = e - j * (kD / 4);
            const float* src = nan_row;
            if (!bad_n) {
                const int id = p.idx[static_cast<size_t>(r) * p.k_max + t0 + j];
                if (id >= 0 && id < p.N) {
                    src = cache + static_cast<size_t>(id) * kD;
                } else if (blockIdx.x == 0 && c4 == 0) {
                    atomicOr(p.err, DSA_DEVERR_IDX_RANGE);
                }
            }
            reinterpret_cast<float4*>(kvs + j * kD)[c4] = reinterpret_cast<const float4*>(src)[c4];
        }
        __syncthreads();
        if (!live) continue;
        // scores of the tile's keys for this warp's head (every lane ends with all)
        float sc[kSimtTile];
#pragma unroll
        for (int j = 0; j < kSimtTile; ++j) {
            float part = 0.0f;
            if (j < nk) {
#pragma unroll
                for (int i = 0; i < kD / 32; ++i)
                    part = fmaf(qs[warp * kD + lane + 32 * i], kvs[j * kD + lane + 32 * i], part);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            }
            sc[j] = part * p.scale;
        }
        float tm = -INFINITY;
#pragma unroll
        for (int j = 0; j < kSimtTile; ++j)
            if (j < nk) tm = fmaxf(tm, sc[j]);
        const float mn = (m == -INFINITY) ? tm : fmaxf(m, tm);
        const float mu_new = (mn == -INFINITY) ? 0.0f : mn;
        const float al = (m == -INFINITY) ? 1.0f : expf(m - mu_new);
        float ps[kSimtTile];
        float ls = 0.0f;
#pragma unroll
        for (int j = 0; j < kSimtTile; ++j) {
            ps[j] = j < nk ? expf(sc[j] - mu_new) : 0.0f;
            if (j < nk) ls += ps[j];
        }
        l = l * al + ls;
#pragma unroll
        for (int i = 0; i < kD / 32; ++i) {
            float a = acc[i] * al;
#pragma unroll
            for (int j = 0; j < kSimtTile; ++j)
                if (j < nk) a = fmaf(ps[j], kvs[j * kD + lane + 32 * i], a);
            acc[i] = a;
        }
        m = mn;
    }
    if (!live) return;

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
        for (int i = 0; i < kD / 32; ++i) orow[lane + 32 * i] = __float2bfloat16_rn(acc[i] * f);
    } else {
        float* orow = static_cast<float*>(p.out) + o0;
#pragma unroll
        for (int i = 0; i < kD / 32; ++i) orow[lane + 32 * i] = acc[i] * f;
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
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(dsa_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSimtSmem));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    dim3 grid((p.H + kSimtHeads - 1) / kSimtHeads, p.R);
    dsa_simt_kernel<<<grid, kSimtThreads, kSimtSmem, s>>>(p);
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
