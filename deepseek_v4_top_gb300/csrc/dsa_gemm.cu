// The output projection on the sm_103a tensor cores: out [M][N] fp32 =
// A [M][K] bf16 . B [K][N] bf16, accumulated in fp32 (TensorFold PR #1206,
// "What changes": the attention's output groups go on to the output
// projections; the pages give the step, not its shape).
//
// How: a persistent kernel, one CTA per SM, over 128 x 256 output tiles
// (M-block fastest, so the CTAs running at one time share their B columns
// and all of A in L2).  Warp-specialised:
//   * warp 0 (one thread) streams 64-deep K slices of A (one 128 x 64 box)
//     and B (four 64 x 64 boxes) by TMA into a ring of four 48 KB stages,
//     128-byte swizzled;
//   * warp 1 (one thread) issues tcgen05.mma (M = 128, N = 256, K = 16, A
//     K-major, B N-major) into one of two TMEM accumulators of 256 columns,
//     and frees each stage with tcgen05.commit;
//   * warps 2-5 read a finished accumulator back (one TMEM lane quadrant
//     each) and store it while the next tile accumulates in the other one.
// There is no split of K, so every output is one fp32 sum in a fixed order
// and repeated calls give the same bits.  Every wait is bounded: on a
// timeout the kernel raises DSA_DEVERR_TIMEOUT, frees its TMEM and returns.
#include <stdint.h>

#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;            // 16 KB: 128 rows x 128 B
constexpr uint32_t kBBoxBytes = kBK * 64 * 2;          // 8 KB: 64 K-rows x 64 columns
constexpr uint32_t kBBytes = 4 * kBBoxBytes;           // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;    // 48 KB
constexpr int kGemmThreads = 192;
constexpr uint32_t kGemmTmemCols = 512;                // two accumulators of 256 columns

struct GemmBars {
    uint64_t full[kStages];     // TMA -> MMA: the stage's A and B landed
    uint64_t empty[kStages];    // MMA -> TMA: the stage's MMAs completed
    uint64_t acc_full[2];       // MMA -> epilogue: the accumulator's tile is complete
    uint64_t acc_empty[2];      // epilogue -> MMA: the accumulator has been read
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kGemmSmem = kStages * kStageBytes + sizeof(GemmBars) + 1024;   // + alignment slack

struct GemmParams {
    CUtensorMap tmap_a;         // A [M][K] bf16: box 64 (K) x 128 (M), 128-byte swizzle
    CUtensorMap tmap_b;         // B [K][N] bf16: box 64 (N) x 64 (K), 128-byte swizzle
    float* out;                 // [M][N] fp32
    uint32_t* err;
    int M, N, K;
    int tiles_m, tiles_n, kblocks;
};

__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mb, int& nb) {
    mb = t % p.tiles_m;
    nb = t / p.tiles_m;
}

__device__ void producer(const GemmParams& p, uint8_t* stages, GemmBars& b) {
    volatile int* ab = &b.abort_flag;
    int stage = 0;
    uint32_t phase = 0;
    const int tiles = p.tiles_m * p.tiles_n;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            // a fresh barrier's preceding phase counts as complete
            if (!mbar_wait(smem_addr(&b.empty[stage]), phase ^ 1u, ab, p.err)) return;
            const uint32_t full = smem_addr(&b.full[stage]);
            const uint32_t sA = smem_addr(stages + stage * kStageBytes);
            mbar_arrive_expect_tx(full, kStageBytes);
            tma_load_2d(sA, &p.tmap_a, kb * kBK, mb * kBM, full);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                tma_load_2d(sA + kABytes + j * kBBoxBytes, &p.tmap_b, nb * kBN + 64 * j, kb * kBK, full);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// One K slice: four MMAs of K = 16.  A K-major: +32 bytes a step inside the
// 128-byte swizzled row; B N-major: +16 K-rows (2 KB) a step.
template <int k>
__device__ __forceinline__ void gemm_kstep(uint32_t d, uint64_t dA, uint64_t dB, uint32_t acc0) {
    constexpr uint32_t idesc = idesc_bf16(kBM, kBN, false, true);
    constexpr uint32_t aoff = (k * 32) / 16, boff = (k * 2048) / 16;
    umma_bf16_at<aoff, boff>(d, dA, dB, idesc, acc0 | (k != 0 ? 1u : 0u));
    if constexpr (k + 1 < 4) gemm_kstep<k + 1>(d, dA, dB, acc0);
}

__device__ void mma_issuer(const GemmParams& p, uint8_t* stages, GemmBars& b, uint32_t tmem) {
    volatile int* ab = &b.abort_flag;
    int stage = 0;
    uint32_t phase = 0;
    const int tiles = p.tiles_m * p.tiles_n;
    int lt = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++lt) {
        const int buf = lt & 1;
        if (!mbar_wait(smem_addr(&b.acc_empty[buf]), ((lt >> 1) & 1) ^ 1u, ab, p.err)) return;
        tc_fence_after();
        const uint32_t d = tmem + buf * kBN;
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!mbar_wait(smem_addr(&b.full[stage]), phase, ab, p.err)) return;
            tc_fence_after();
            const uint32_t sA = smem_addr(stages + stage * kStageBytes);
            const uint64_t dA = sdesc_sw128(sA, 16, 1024);
            const uint64_t dB = sdesc_sw128(sA + kABytes, kBBoxBytes, 1024);
            gemm_kstep<0>(d, dA, dB, kb > 0 ? 1u : 0u);
            umma_commit(smem_addr(&b.empty[stage]));
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        umma_commit(smem_addr(&b.acc_full[buf]));
    }
}

// Warp w (2..5) reads TMEM lane quadrant w % 4: rows 32 (w % 4) .. + 31 of
// the tile, 32 columns at a time, and stores each row's 128 contiguous bytes.
__device__ void epilogue(const GemmParams& p, GemmBars& b, uint32_t tmem, int warp, int lane) {
    volatile int* ab = &b.abort_flag;
    const int q = warp & 3;
    const int tiles = p.tiles_m * p.tiles_n;
    int lt = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++lt) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const int buf = lt & 1;
        if (!mbar_wait(smem_addr(&b.acc_full[buf]), (lt >> 1) & 1, ab, p.err)) return;
        tc_fence_after();
        const int row = mb * kBM + 32 * q + lane;
        float* orow = p.out + static_cast<size_t>(row) * p.N;
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * kBN + c0, v);
            const int col = nb * kBN + c0;
            if (row < p.M) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    if (col + j < p.N)       // N is a multiple of 8: a float4 is wholly in or out
                        *reinterpret_cast<float4*>(orow + col + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&b.acc_empty[buf]));
    }
}

__global__ void __launch_bounds__(kGemmThreads, 1) dsa_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle needs 1024-byte aligned stages (the launch adds 1 KB of slack)
    uint8_t* stages = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    GemmBars& b = *reinterpret_cast<GemmBars*>(stages + kStages * kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_addr(&b.full[i]), 1);
            mbar_init(smem_addr(&b.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&b.acc_full[i]), 1);
            mbar_init(smem_addr(&b.acc_empty[i]), 4);
        }
        b.abort_flag = 0;
        mbar_fence_init();
        prefetch_tmap(&p.tmap_a);
        prefetch_tmap(&p.tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&b.tmem_base), kGemmTmemCols);
        tmem_relinquish();
    }
    // A and B may be written by the grid before this one in the stream
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem_base;
    if (warp == 0) {
        if (lane == 0) producer(p, stages, b);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) mma_issuer(p, stages, b, tmem);
        __syncwarp();
    } else {
        epilogue(p, b, tmem, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kGemmTmemCols);
    }
}

// ------------------------------------------------------------------------
// The same product on SM pairs (tcgen05 cta_group::2): a cluster of two CTAs
// computes 256 x 256 tiles.  Each CTA stages its own 128 rows of A and its
// own 128 columns of B (32 KB a K slice instead of 48 KB), so an SM takes in
// a third less data per MMA; the even CTA issues M = 256 MMAs that read both
// CTAs' halves and write each CTA's 128 accumulator rows into its own TMEM.
// Seven 32 KB stages.  The stage-full barriers live in the even CTA (both
// CTAs' TMA loads complete their bytes there), the stage-empty and
// accumulator-full barriers in each CTA (the even CTA's commits arrive on
// both), the accumulator-empty barriers in the even CTA (both CTAs'
// epilogue warps arrive).
constexpr int kPairStages = 7;
constexpr uint32_t kPairBBytes = 2 * kBBoxBytes;                 // 16 KB: 64 K-rows x 128 columns
constexpr uint32_t kPairStageBytes = kABytes + kPairBBytes;      // 32 KB
constexpr int kPairBM = 256;

struct PairBars {
    uint64_t full[kPairStages];     // even CTA: both halves of the stage landed
    uint64_t empty[kPairStages];    // each CTA: the stage's MMAs completed
    uint64_t acc_full[2];           // each CTA: the accumulator's tile is complete
    uint64_t acc_empty[2];          // even CTA: all eight epilogue warps read the accumulator
    uint32_t tmem_base;
    int abort_flag;
};

constexpr size_t kPairSmem = kPairStages * kPairStageBytes + sizeof(PairBars) + 1024;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of `a` (a shared::cta address of this CTA's
// layout) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bounded wait with cluster-scope acquire (arrivals come from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint32_t* err) {
    const unsigned long long t0 = global_ns();
    uint32_t n = 0;
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((++n & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(err, DSA_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// One box into this CTA's shared memory, its bytes completed on a barrier
// that may be in the peer CTA (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int col, int row, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(col), "r"(row), "r"(bar)
        : "memory");
}

template <uint32_t kAOff, uint32_t kBOff>
__device__ __forceinline__ void umma_pair_at(uint32_t d_tmem, uint64_t a_base, uint64_t b_base, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 a, b;\n\t"
        "add.u64 a, %1, %5;\n\t"
        "add.u64 b, %2, %6;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_base), "l"(b_base), "r"(idesc), "r"(accumulate), "n"(kAOff), "n"(kBOff)
        : "memory");
}

// Arrive once on the barrier at `bar`'s offset in both CTAs of the pair when
// every MMA this thread issued has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

template <int k>
__device__ __forceinline__ void pair_kstep(uint32_t d, uint64_t dA, uint64_t dB, uint32_t acc0) {
    constexpr uint32_t idesc = idesc_bf16(kPairBM, kBN, false, true);
    constexpr uint32_t aoff = (k * 32) / 16, boff = (k * 2048) / 16;
    umma_pair_at<aoff, boff>(d, dA, dB, idesc, acc0 | (k != 0 ? 1u : 0u));
    if constexpr (k + 1 < 4) pair_kstep<k + 1>(d, dA, dB, acc0);
}

__device__ void pair_producer(const GemmParams& p, uint8_t* stages, PairBars& b, uint32_t rank) {
    volatile int* ab = &b.abort_flag;
    int stage = 0;
    uint32_t phase = 0;
    const int tiles = p.tiles_m * p.tiles_n;
    const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
    for (int t = pair; t < tiles; t += pairs) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!mbar_wait(smem_addr(&b.empty[stage]), phase ^ 1u, ab, p.err)) return;
            const uint32_t full = cluster_addr(smem_addr(&b.full[stage]), 0);
            const uint32_t sA = smem_addr(stages + stage * kPairStageBytes);
            // the even CTA expects both CTAs' bytes of the stage
            if (rank == 0) mbar_arrive_expect_tx(smem_addr(&b.full[stage]), 2 * kPairStageBytes);
            tma_load_2d_pair(sA, &p.tmap_a, kb * kBK, mb * kPairBM + static_cast<int>(rank) * kBM, full);
#pragma unroll
            for (int j = 0; j < 2; ++j)
                tma_load_2d_pair(sA + kABytes + j * kBBoxBytes, &p.tmap_b,
                                 nb * kBN + static_cast<int>(rank) * 128 + 64 * j, kb * kBK, full);
            if (++stage == kPairStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

__device__ void pair_mma(const GemmParams& p, uint8_t* stages, PairBars& b, uint32_t tmem) {
    volatile int* ab = &b.abort_flag;
    int stage = 0;
    uint32_t phase = 0;
    const int tiles = p.tiles_m * p.tiles_n;
    const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
    int lt = 0;
    for (int t = pair; t < tiles; t += pairs, ++lt) {
        const int buf = lt & 1;
        if (!mbar_wait_cluster(smem_addr(&b.acc_empty[buf]), ((lt >> 1) & 1) ^ 1u, ab, p.err)) return;
        tc_fence_after();
        const uint32_t d = tmem + buf * kBN;
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!mbar_wait_cluster(smem_addr(&b.full[stage]), phase, ab, p.err)) return;
            tc_fence_after();
            const uint32_t sA = smem_addr(stages + stage * kPairStageBytes);
            const uint64_t dA = sdesc_sw128(sA, 16, 1024);
            const uint64_t dB = sdesc_sw128(sA + kABytes, kBBoxBytes, 1024);
            pair_kstep<0>(d, dA, dB, kb > 0 ? 1u : 0u);
            umma_commit_pair(smem_addr(&b.empty[stage]));
            if (++stage == kPairStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        umma_commit_pair(smem_addr(&b.acc_full[buf]));
    }
}

__device__ void pair_epilogue(const GemmParams& p, PairBars& b, uint32_t tmem, uint32_t rank, int warp, int lane) {
    volatile int* ab = &b.abort_flag;
    const int q = warp & 3;
    const int tiles = p.tiles_m * p.tiles_n;
    const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
    int lt = 0;
    for (int t = pair; t < tiles; t += pairs, ++lt) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const int buf = lt & 1;
        if (!mbar_wait(smem_addr(&b.acc_full[buf]), (lt >> 1) & 1, ab, p.err)) return;
        tc_fence_after();
        const int row = mb * kPairBM + static_cast<int>(rank) * kBM + 32 * q + lane;
        float* orow = p.out + static_cast<size_t>(row) * p.N;
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * kBN + c0, v);
            const int col = nb * kBN + c0;
            if (row < p.M) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    if (col + j < p.N)
                        *reinterpret_cast<float4*>(orow + col + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            const uint32_t bar = cluster_addr(smem_addr(&b.acc_empty[buf]), 0);
            asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
        }
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    dsa_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* stages = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    PairBars& b = *reinterpret_cast<PairBars*>(stages + kPairStages * kPairStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    grid_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < kPairStages; ++i) {
            mbar_init(smem_addr(&b.full[i]), 1);
            mbar_init(smem_addr(&b.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&b.acc_full[i]), 1);
            mbar_init(smem_addr(&b.acc_empty[i]), 8);
        }
        b.abort_flag = 0;
        mbar_fence_init();
        prefetch_tmap(&p.tmap_a);
        prefetch_tmap(&p.tmap_b);
    }
    if (warp == 1) {
        // one warp of each CTA allocates the pair's columns together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&b.tmem_base)),
                     "r"(kGemmTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    cluster_sync();                  // both CTAs' barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem = b.tmem_base;
    if (warp == 0) {
        if (lane == 0) pair_producer(p, stages, b, rank);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) pair_mma(p, stages, b, tmem);
        __syncwarp();
    } else {
        pair_epilogue(p, b, tmem, rank, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                  // neither CTA leaves while the other may still use its memory
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kGemmTmemCols)
                     : "memory");
    }
}

std::mutex g_gemm_mu;

PFN_cuTensorMapEncodeTiled_v12000 gemm_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    std::lock_guard<std::mutex> lock(g_gemm_mu);
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// A row-major bf16 matrix [rows][cols], read in boxes of 64 columns x box_rows
// rows with the 128-byte swizzle; reads past the edges return zeros.
bool encode_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = gemm_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(const void* a, const void* b, float* out, int M, int K, int N, uint32_t* err, int sms,
                        cudaStream_t s) {
    static bool attr_set[64] = {false};
    static int pair_clusters[64] = {0};     // co-resident SM pairs of the pair kernel (0: none)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_gemm_mu);
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(dsa_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kGemmSmem));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(dsa_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kPairSmem));
            if (e != cudaSuccess) return e;
            cudaLaunchConfig_t occ = {};
            occ.gridDim = dim3(2);
            occ.blockDim = dim3(kGemmThreads);
            occ.dynamicSmemBytes = kPairSmem;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, dsa_gemm_pair_kernel, &occ) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            pair_clusters[dev] = n;
            attr_set[dev] = true;
        }
    }
    GemmParams p;
    if (!encode_bf16(&p.tmap_a, a, static_cast<uint64_t>(M), static_cast<uint64_t>(K), kBM) ||
        !encode_bf16(&p.tmap_b, b, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kBK))
        return cudaErrorInvalidValue;
    p.out = out;
    p.err = err;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_n = (N + kBN - 1) / kBN;
    p.kblocks = (K + kBK - 1) / kBK;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kGemmThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pair_clusters[dev] > 0) {
        // SM pairs over 256 x 256 tiles
        p.tiles_m = (M + kPairBM - 1) / kPairBM;
        const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n;
        const int pairs = static_cast<int>(tiles < pair_clusters[dev] ? tiles : pair_clusters[dev]);
        cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
        cfg.dynamicSmemBytes = kPairSmem;
        return cudaLaunchKernelEx(&cfg, dsa_gemm_pair_kernel, p);
    }
    p.tiles_m = (M + kBM - 1) / kBM;
    const long long tiles = static_cast<long long>(p.tiles_m) * p.tiles_n;
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.dynamicSmemBytes = kGemmSmem;
    return cudaLaunchKernelEx(&cfg, dsa_gemm_kernel, p);
}

}  // namespace dsa
