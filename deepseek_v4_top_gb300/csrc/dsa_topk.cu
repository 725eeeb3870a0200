// Top-k selection of an indexer's scores: the step that turns a row's index
// scores into the selection the sparse attention reads (DeepSeek V4.1
// indexer PR #2, title: the indexer's merge and finish on a threadgroup a
// row, the same picks).  The order is: larger score first, NaN after every
// number, -0 equal to +0, equal scores by smaller position first; a row
// keeps min(k, n_valid) positions in that order and pads with -1.
//
// A CTA selects over one segment of up to 16 keys a thread, held in
// registers; thread t owns the segment's contiguous entries [16 t, 16 t + 16).
// A row of up to 4096 positions is one segment of a 256-thread CTA, and one
// of up to 8192 a segment of a 512-thread CTA, read as float4 (rows are
// 16-byte aligned with a stride of a multiple of 4 scores).  A longer row is
// selected in two steps: each 8192-position share of it selects its own top
// k (one 512-thread CTA a share, all the row's shares at once), and one CTA
// then selects the row's top k among the shares' picks.  That is exact: a pick of the row
// has fewer than k entries above it in the row, so fewer in its share.  The
// shares' picks are stored share after share, each in position order, so the
// second step sees them in position order too.
// For a segment:
//   1. the scores become 32-bit keys whose unsigned order is the selection
//      order of the values (NaN lowest); entries past the segment get key 0;
//   2. a radix select (11, 11 and 10 bits, most significant first) finds the
//      key T of the k-th pick and how many keys equal to T it takes (the
//      first ones by position).  Each pass counts into a 2048-bin shared
//      histogram whose bins, counted from the top, are owned B to a thread
//      (their addresses padded so that a warp reading the b-th bin of each
//      thread hits 32 banks); a scan of the owners' sums finds the bin that
//      holds the k-th pick.  A pass whose bin is taken whole ends the select
//      early (a row of N(0,1) scores usually ends after two passes);
//   3. one block scan of packed per-thread counts (keys above T in the high
//      16 bits, keys equal to T in the low) gives every thread its output
//      offset, the keys above T before it plus min(keys equal to T before
//      it, need), and each thread writes its own picks in position order.
// Entries past the segment hold key 0, the key of NaN, and come after every
// candidate: they can only fall in the lowest bin of a pass, whose count then
// exceeds the candidates' but never changes which bin is chosen, and they are
// never among the first `need` keys equal to T.  The picks depend only on the
// row, never on the launch.
#include <stdint.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTopkBins = 2048;
constexpr int kTopkPerThread = 16;
constexpr int kTopkShortRow = 256 * kTopkPerThread;  // rows up to this long: one 256-thread CTA
constexpr int kTopkShare = 512 * kTopkPerThread;     // positions a share of a long row (and a one-step
                                                     // row of 512 threads) holds

// What a launch selects over and where it writes.
enum TopkMode {
    kRowsToIdx = 0,      // rows of up to 4096 scores -> idx, n_sel
    kSharesToCand = 1,   // a share of a long row -> its picks' keys and positions
    kCandToIdx = 2,      // a long row's shares' picks -> idx, n_sel
};

// Order-preserving key of a score: NaN -> 0; otherwise positive values with
// the sign bit set and negative values negated (two's complement), which
// sends -0 and +0 to the same key 0x80000000.
__device__ __forceinline__ uint32_t score_key(float x) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t s = static_cast<uint32_t>(static_cast<int32_t>(u) >> 31);
    const uint32_t k = (u ^ (s | 0x80000000u)) - s;
    return x == x ? k : 0u;
}

template <int kThreads>
struct TopkSmem {
    static constexpr int kWarps = kThreads / 32;
    static constexpr int kBinsPerThread = kTopkBins / kThreads;
    // one padding word after every kBinsPerThread bins
    static constexpr int kSlots = kTopkBins + kTopkBins / kBinsPerThread;
    uint32_t hist[kSlots];
    uint32_t warp_sum[kWarps];
    uint32_t prefix, need, done;    // select state: key bits fixed so far, picks left, bin taken whole
};

template <int kBinsPerThread>
__device__ __forceinline__ int bin_slot(uint32_t d) { return static_cast<int>(d + d / kBinsPerThread); }

// The sum of the totals of the warps before this one (warp_sum holds one a
// warp): lane w < warp reads warp w's, and the warp adds them up at once.
__device__ __forceinline__ uint32_t earlier_warps(const uint32_t* warp_sum, int warp, int lane) {
    return __reduce_add_sync(0xFFFFFFFFu, lane < warp ? warp_sum[lane] : 0u);
}

// The digit passes: bits [21, 32), [10, 21), [0, 10).
__device__ __forceinline__ int digit_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__device__ __forceinline__ int digit_bins(int pass) { return pass == 2 ? 1024 : 2048; }

// Picks a long row's shares hold before share c: k for every earlier share
// (a share that holds candidates has only full shares before it).
__device__ __forceinline__ int share_len(int n, int c) {
    const int len = n - c * kTopkShare;
    return len < 0 ? 0 : (len > kTopkShare ? kTopkShare : len);
}

template <int kThreads, int kMode>
__global__ void __launch_bounds__(kThreads, kMode == kCandToIdx ? 1 : (kThreads == 256 ? 4 : 2))
    dsa_topk_kernel(const TopkParams p) {
    using Smem = TopkSmem<kThreads>;
    constexpr int kWarps = Smem::kWarps;
    constexpr int kB = Smem::kBinsPerThread;
    static_assert(kB >= 2 && kThreads * kB == kTopkBins, "bin ownership");
    static_assert(kMode != kSharesToCand || kThreads * kTopkPerThread == kTopkShare, "a share a CTA");
    // rows of up to 4096 (four CTAs an SM): a thread wholly past its row's
    // candidates holds only padding and skips the counting and compaction
    constexpr bool kSkipPadding = kMode == kRowsToIdx && kThreads == 256;
    static_assert(kTopkMaxLd / kTopkShare * kTopkMaxK <= 512 * kTopkPerThread, "a long row's picks fit 512 threads");
    __shared__ Smem sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_launch_dependents();
    grid_dependency_wait();          // the scores may come from the grid before this one
#pragma unroll
    for (int b = 0; b < kB; ++b) sm.hist[bin_slot<kB>(tid * kB + b)] = 0u;

    const int segments = kMode == kSharesToCand ? p.R * p.shares : p.R;
    for (int sg = blockIdx.x; sg < segments; sg += gridDim.x) {
        const int r = kMode == kSharesToCand ? sg / p.shares : sg;
        const int c = kMode == kSharesToCand ? sg - r * p.shares : 0;
        const int n = __ldg(p.n_valid + r);
        const bool bad = n < 0 || n > p.ld;
        int32_t* out = p.idx + static_cast<size_t>(r) * p.k_max;
        uint32_t* cand_key = p.cand_key + static_cast<size_t>(r) * p.cand_ld;
        int32_t* cand_pos = p.cand_pos + static_cast<size_t>(r) * p.cand_ld;
        if (kMode == kSharesToCand && bad) continue;       // (the second step reports the row)
        if (kMode != kSharesToCand && bad) {
            if (tid == 0) {
                atomicOr(p.err, DSA_DEVERR_NVALID_RANGE);
                p.n_sel[r] = 0;
            }
            for (int j = tid; j < p.k_max; j += kThreads) out[j] = -1;
            continue;
        }
        // the segment: n_seg entries; its picks, m, go to offset `at0` of the output
        int n_seg, m;
        if (kMode == kRowsToIdx) {
            n_seg = n;
            m = n < p.k ? n : p.k;
        } else if (kMode == kSharesToCand) {
            n_seg = share_len(n, c);
            m = n_seg < p.k ? n_seg : p.k;
            if (n_seg == 0) continue;
        } else {
            const int full = n / kTopkShare, part = n - full * kTopkShare;
            n_seg = full * p.k + (part < p.k ? part : p.k);
            m = n < p.k ? n : p.k;
        }
        const int share0 = c * kTopkShare;                  // first position of the share
        const int at0 = c * p.k;                            // its picks' offset among the row's
        if (kMode != kSharesToCand && m == n_seg) {
            // every entry is a pick, in position order
            for (int j = tid; j < p.k_max; j += kThreads)
                out[j] = j < n_seg ? (kMode == kCandToIdx ? cand_pos[j] : j) : -1;
            if (tid == 0) p.n_sel[r] = m;
            continue;
        }

        // 1. keys of this thread's entries (and, for the shares' picks, their
        //    positions, loaded with them rather than one by one as picks are written)
        const int j0 = tid * kTopkPerThread;
        const int rem = n_seg - j0;  // this thread's entries: the first min(max(rem, 0), 16)
        uint32_t key[kTopkPerThread];
        int32_t cpos[kMode == kCandToIdx ? kTopkPerThread : 1];
        if (kMode == kCandToIdx) {
            const uint4* src4 = reinterpret_cast<const uint4*>(cand_key) + j0 / 4;
            const int4* pos4 = reinterpret_cast<const int4*>(cand_pos) + j0 / 4;
#pragma unroll
            for (int i = 0; i < kTopkPerThread / 4; ++i) {
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                int4 w = make_int4(0, 0, 0, 0);
                if (4 * i < rem) {
                    v = src4[i];
                    w = pos4[i];
                }
                key[4 * i] = 4 * i < rem ? v.x : 0u;
                key[4 * i + 1] = 4 * i + 1 < rem ? v.y : 0u;
                key[4 * i + 2] = 4 * i + 2 < rem ? v.z : 0u;
                key[4 * i + 3] = 4 * i + 3 < rem ? v.w : 0u;
                cpos[(4 * i) % (kMode == kCandToIdx ? kTopkPerThread : 1)] = w.x;
                cpos[(4 * i + 1) % (kMode == kCandToIdx ? kTopkPerThread : 1)] = w.y;
                cpos[(4 * i + 2) % (kMode == kCandToIdx ? kTopkPerThread : 1)] = w.z;
                cpos[(4 * i + 3) % (kMode == kCandToIdx ? kTopkPerThread : 1)] = w.w;
            }
        } else {
            const float4* src4 =
                reinterpret_cast<const float4*>(p.scores + static_cast<size_t>(r) * p.ld + share0) + j0 / 4;
#pragma unroll
            for (int i = 0; i < kTopkPerThread / 4; ++i) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (4 * i < rem) v = __ldg(src4 + i);
                key[4 * i] = 4 * i < rem ? score_key(v.x) : 0u;
                key[4 * i + 1] = 4 * i + 1 < rem ? score_key(v.y) : 0u;
                key[4 * i + 2] = 4 * i + 2 < rem ? score_key(v.z) : 0u;
                key[4 * i + 3] = 4 * i + 3 < rem ? score_key(v.w) : 0u;
            }
        }
        if (kMode == kSharesToCand && m == n_seg) {
            // a short share: all of it, in position order
#pragma unroll
            for (int i = 0; i < kTopkPerThread; ++i) {
                if (i < rem) {
                    cand_key[at0 + j0 + i] = key[i];
                    cand_pos[at0 + j0 + i] = share0 + j0 + i;
                }
            }
            continue;
        }
        if (tid == 0) {
            sm.prefix = 0u;
            sm.need = static_cast<uint32_t>(m);
            sm.done = 0u;
        }
        __syncthreads();             // (the histogram is clear: each pass clears it)

        // 2. radix select of the m-th largest key
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = digit_shift(pass), nb = digit_bins(pass);
            const int hi = shift + (pass == 2 ? 10 : 11);      // bits fixed before this pass: [hi, 32)
            const uint32_t prefix = sm.prefix;
            if (!kSkipPadding || rem > 0) {
#pragma unroll
                for (int i = 0; i < kTopkPerThread; ++i) {
                    if (pass == 0 || (key[i] >> hi) == (prefix >> hi))
                        atomicAdd(&sm.hist[bin_slot<kB>((key[i] >> shift) & static_cast<uint32_t>(nb - 1))], 1u);
                }
            }
            __syncthreads();
            // thread t: bins nb-1-t*B-b, b = 0 .. B-1, counted from the top
            uint32_t cnt[kB], sum = 0u;
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int d = nb - 1 - tid * kB - b;
                cnt[b] = d >= 0 ? sm.hist[bin_slot<kB>(static_cast<uint32_t>(d))] : 0u;
                sum += cnt[b];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            if (lane == 31) sm.warp_sum[warp] = incl;
            const uint32_t want = sm.need;
            __syncthreads();
#pragma unroll
            for (int b = 0; b < kB; ++b) sm.hist[bin_slot<kB>(tid * kB + b)] = 0u;
            const uint32_t before = earlier_warps(sm.warp_sum, warp, lane);
            const uint32_t excl = before + incl - sum;
            if (excl < want && want <= excl + sum) {
                uint32_t above = excl;
#pragma unroll
                for (int b = 0; b < kB; ++b) {
                    if (above + cnt[b] >= want) {
                        const uint32_t d = static_cast<uint32_t>(nb - 1 - tid * kB - b);
                        sm.prefix = prefix | (d << shift);
                        sm.need = want - above;
                        sm.done = above + cnt[b] == want ? 1u : 0u;
                        break;
                    }
                    above += cnt[b];
                }
            }
            __syncthreads();
            if (sm.done) break;
        }
        // picks: the keys > thr, and the first `need` keys == thr
        uint32_t thr = sm.prefix, need = sm.need;
        if (sm.done) {
            // every key of the chosen bin is a pick: the picks are the keys >=
            // prefix (never 0 here: that bin would hold every candidate)
            need = thr == 0u ? 0xFFFFFFFFu : 0u;
            thr = thr == 0u ? 0u : thr - 1u;
        }

        // 3. this thread's keys above thr and equal to thr, packed; block scan
        uint32_t packed = 0u;
        if (kSkipPadding && rem <= 0) {
            // only padding: no picks
        } else if (need == 0u) {
#pragma unroll
            for (int i = 0; i < kTopkPerThread; ++i) packed += key[i] > thr ? 0x10000u : 0u;
        } else {
#pragma unroll
            for (int i = 0; i < kTopkPerThread; ++i) packed += key[i] > thr ? 0x10000u : (key[i] == thr ? 1u : 0u);
        }
        uint32_t incl = packed;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) sm.warp_sum[warp] = incl;
        __syncthreads();
        const uint32_t before = incl - packed + earlier_warps(sm.warp_sum, warp, lane);
        const uint32_t eq_before = before & 0xFFFFu;
        int at = static_cast<int>((before >> 16) + (eq_before < need ? eq_before : need));
        // writes pick i at output entry `at`
        auto put = [&](int i, int a) {
            if (kMode == kRowsToIdx) {
                out[a] = j0 + i;
            } else if (kMode == kSharesToCand) {
                cand_key[at0 + a] = key[i];
                cand_pos[at0 + a] = share0 + j0 + i;
            } else {
                out[a] = cpos[i % (kMode == kCandToIdx ? kTopkPerThread : 1)];
            }
        };
        if (kSkipPadding && rem <= 0) {
            // only padding: no picks
        } else if (need == 0u) {
#pragma unroll
            for (int i = 0; i < kTopkPerThread; ++i) {
                if (key[i] > thr) put(i, at++);
            }
        } else {
            uint32_t eq_seen = eq_before;
#pragma unroll
            for (int i = 0; i < kTopkPerThread; ++i) {
                const bool eq = key[i] == thr;
                if (key[i] > thr || (eq && eq_seen < need)) put(i, at++);
                eq_seen += eq ? 1u : 0u;
            }
        }
        if (kMode != kSharesToCand) {
            for (int j = m + tid; j < p.k_max; j += kThreads) out[j] = -1;
            if (tid == 0) p.n_sel[r] = m;
        }
        __syncthreads();             // warp_sum and the select state are rewritten by the next segment
    }
}

template <int kThreads, int kMode>
cudaError_t launch_mode(const TopkParams& p, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dsa_topk_kernel<kThreads, kMode>, p);
}

}  // namespace

int topk_shares(int ld) { return ld <= kTopkShare ? 1 : (ld + kTopkShare - 1) / kTopkShare; }

cudaError_t launch_topk(const TopkParams& p, int grid, cudaStream_t s) {
    if (p.ld % 4 != 0 || reinterpret_cast<uintptr_t>(p.scores) % 16 != 0 || p.ld > kTopkMaxLd)
        return cudaErrorInvalidValue;
    if (p.shares == 1)
        return p.ld <= kTopkShortRow ? launch_mode<256, kRowsToIdx>(p, grid, s) : launch_mode<512, kRowsToIdx>(p, grid, s);
    // long rows: the shares' selections, then one over their picks
    if (p.cand_ld % 4 != 0 || p.cand_ld < p.shares * p.k || p.shares * p.k > 512 * kTopkPerThread)
        return cudaErrorInvalidValue;
    const long long share_grid = static_cast<long long>(grid) * p.shares;
    cudaError_t e = launch_mode<512, kSharesToCand>(p, static_cast<int>(share_grid), s);
    if (e != cudaSuccess) return e;
    const int cap = p.shares * p.k;
    // (at most 32768 / 8192 = 4 shares of 2048 picks: 8192 candidates)
    if (cap <= 256 * kTopkPerThread) return launch_mode<256, kCandToIdx>(p, grid, s);
    return launch_mode<512, kCandToIdx>(p, grid, s);
}

}  // namespace dsa
