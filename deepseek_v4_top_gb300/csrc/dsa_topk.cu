// Top-k selection of an indexer's scores: the step that turns a row's index
// scores into the selection the sparse attention reads (DeepSeek V4.1
// indexer PR #2, title: the indexer's merge and finish on a threadgroup a
// row, the same picks).  The order is: larger score first, NaN after every
// number, -0 equal to +0, equal scores by smaller position first; a row
// keeps min(k, n_valid) positions in that order and pads with -1.
//
// One CTA a row (256 threads for rows of up to 4096 candidates, 1024 up to
// 32768), the row's keys held in registers: warp w owns a contiguous share
// of the positions, lane l positions share_w + l + 32 i.
//   1. the scores become 32-bit keys whose unsigned order is the selection
//      order of the values (NaN lowest);
//   2. a 3-pass radix select (11, 11 and 10 bits, most significant first;
//      2048-bin shared histograms, a block scan to find the bin) finds the
//      key T of the k-th pick and how many keys equal to T it takes (the
//      first ones by position);
//   3. each warp counts the picks of its share, one prefix over the warps
//      gives every share its output offset, and each warp writes its picks'
//      positions in ascending order.
// The picks depend only on the row, never on the launch.
#include <stdint.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTopkBins = 2048;

// Order-preserving key of a score: NaN -> 0, -0 -> the key of +0, negative
// values bit-inverted, positive values with the sign bit set.
__device__ __forceinline__ uint32_t score_key(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int kThreads>
struct TopkSmem {
    static constexpr int kWarps = kThreads / 32;
    uint32_t hist[kTopkBins];
    uint32_t warp_sum[kWarps];      // bin-scan totals, then per-share counts above T
    uint32_t warp_eq[kWarps];       // per share: keys equal to T
    uint32_t prefix, need;          // radix select state: key bits fixed so far, picks left
};

// The digit passes: bits [21, 32), [10, 21), [0, 10).
__device__ __forceinline__ int digit_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t digit_bins(int pass) { return pass == 2 ? 1024u : 2048u; }

// Short rows run six CTAs an SM (40 registers), long rows one.
template <int kThreads, int kPerThread>
__global__ void __launch_bounds__(kThreads, kThreads == 256 ? 6 : 1) dsa_topk_kernel(const TopkParams p) {
    using Smem = TopkSmem<kThreads>;
    constexpr int kWarps = Smem::kWarps;
    constexpr int kBinsPerThread = kTopkBins / kThreads;
    __shared__ Smem sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    grid_launch_dependents();
    grid_dependency_wait();          // the scores may come from the grid before this one

    for (int r = blockIdx.x; r < p.R; r += gridDim.x) {
        const int n = __ldg(p.n_valid + r);
        int32_t* out = p.idx + static_cast<size_t>(r) * p.k_max;
        if (n < 0 || n > p.ld) {
            if (tid == 0) {
                atomicOr(p.err, DSA_DEVERR_NVALID_RANGE);
                p.n_sel[r] = 0;
            }
            for (int j = tid; j < p.k_max; j += kThreads) out[j] = -1;
            continue;
        }
        const int m = n < p.k ? n : p.k;
        // 1. keys of this thread's positions (coalesced per warp)
        const int share = (n + kWarps * 32 - 1) / (kWarps * 32) * 32;
        const int j_lo = warp * share, j_hi = min(n, j_lo + share);
        const float* row = p.scores + static_cast<size_t>(r) * p.ld;
        uint32_t key[kPerThread];
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
            const int j = j_lo + lane + 32 * i;
            key[i] = j < j_hi ? score_key(__ldg(row + j)) : 0u;
        }
        if (tid == 0) {
            sm.prefix = 0u;
            sm.need = static_cast<uint32_t>(m);
        }

        // 2. radix select of the m-th largest key (unless every candidate is a pick)
        uint32_t thr = 0u, need = 0u;     // picks: keys > thr, and the first `need` keys == thr
        const bool all = m == n;
        if (!all) {
            uint32_t mask = 0u;
            for (int pass = 0; pass < 3; ++pass) {
                const int shift = digit_shift(pass);
                const uint32_t nb = digit_bins(pass);
#pragma unroll
                for (int b = 0; b < kBinsPerThread; ++b) sm.hist[tid * kBinsPerThread + b] = 0u;
                __syncthreads();
                const uint32_t prefix = sm.prefix;
#pragma unroll
                for (int i = 0; i < kPerThread; ++i) {
                    const int j = j_lo + lane + 32 * i;
                    if (j < j_hi && (key[i] & mask) == prefix) atomicAdd(&sm.hist[(key[i] >> shift) & (nb - 1)], 1u);
                }
                __syncthreads();
                // thread t holds bins counted from the top: nb-1-t*B .. nb-B-t*B
                uint32_t c[kBinsPerThread], s = 0u;
#pragma unroll
                for (int b = 0; b < kBinsPerThread; ++b) {
                    const int bin = static_cast<int>(nb) - 1 - tid * kBinsPerThread - b;
                    c[b] = bin >= 0 ? sm.hist[bin] : 0u;
                    s += c[b];
                }
                uint32_t incl = s;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += v;
                }
                if (lane == 31) sm.warp_sum[warp] = incl;
                const uint32_t want = sm.need;
                __syncthreads();
                uint32_t before = 0u;
                for (int w = 0; w < warp; ++w) before += sm.warp_sum[w];
                const uint32_t excl = before + incl - s;
                if (excl < want && want <= excl + s) {
                    uint32_t above = excl;
#pragma unroll
                    for (int b = 0; b < kBinsPerThread; ++b) {
                        if (above + c[b] >= want) {
                            const uint32_t bin = nb - 1u - tid * kBinsPerThread - b;
                            sm.prefix = prefix | (bin << shift);
                            sm.need = want - above;
                            break;
                        }
                        above += c[b];
                    }
                }
                mask |= (nb - 1u) << shift;
                __syncthreads();
            }
            thr = sm.prefix;
            need = sm.need;
        }

        // 3. count the picks of this warp's share, prefix over the warps,
        //    then write them in position order
        uint32_t c_gt = 0u, c_eq = 0u;
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
            const int j = j_lo + lane + 32 * i;
            c_gt += __popc(__ballot_sync(0xFFFFFFFFu, j < j_hi && (all || key[i] > thr)));
            c_eq += __popc(__ballot_sync(0xFFFFFFFFu, j < j_hi && !all && key[i] == thr));
        }
        if (lane == 0) {
            sm.warp_sum[warp] = c_gt;
            sm.warp_eq[warp] = c_eq;
        }
        __syncthreads();
        uint32_t eq_before = 0u, out_at = 0u;     // over the shares before this one
        for (int w = 0; w < warp; ++w) {
            const uint32_t eq_w = sm.warp_eq[w];
            const uint32_t taken = eq_before >= need ? 0u : min(eq_w, need - eq_before);
            out_at += sm.warp_sum[w] + taken;
            eq_before += eq_w;
        }
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
            const int j = j_lo + lane + 32 * i;
            const bool gt = j < j_hi && (all || key[i] > thr);
            const bool eq = j < j_hi && !all && key[i] == thr;
            const uint32_t be = __ballot_sync(0xFFFFFFFFu, eq);
            const bool pick = gt || (eq && eq_before + __popc(be & lt_mask) < need);
            const uint32_t bp = __ballot_sync(0xFFFFFFFFu, pick);
            if (pick) out[out_at + __popc(bp & lt_mask)] = j;
            out_at += __popc(bp);
            eq_before += __popc(be);
        }
        for (int j = m + tid; j < p.k_max; j += kThreads) out[j] = -1;
        if (tid == 0) p.n_sel[r] = m;
        __syncthreads();             // the shared state is rewritten by the next row
    }
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.ld <= 256 * 16) {
        cfg.blockDim = dim3(256);
        return cudaLaunchKernelEx(&cfg, dsa_topk_kernel<256, 16>, p);
    }
    if (p.ld > kTopkMaxLd) return cudaErrorInvalidValue;
    cfg.blockDim = dim3(1024);
    return cudaLaunchKernelEx(&cfg, dsa_topk_kernel<1024, 32>, p);
}

}  // namespace dsa
