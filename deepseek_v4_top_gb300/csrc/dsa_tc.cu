// Top-k sparse attention on the sm_103a tensor cores (bf16 inputs).
//
// What it computes: for one query row and all of its heads, the softmax over
// the row's selected latent KV rows plus one sink logit per head, weighted
// sum of the same rows (akol1 TensorFold PR #4, first commit message: score a
// tile of keys, keep a running maximum, a tile sum and a value sum;
// TensorFold PR #1206, "What changes": per-head sinks).
//
// How (one CTA per SM, persistent over work units; a unit is one row, or one
// key chunk of a row when a decode batch is split across SMs).  Per 128-key
// tile the work is a chain: gather -> scores -> softmax -> P.V, and the one
// shared-memory KV tile (128 KiB) is busy from its gather to the end of its
// P.V.  Eight worker warps therefore do every CUDA-core step in turn, so that
// each step runs on all of them:
//
//   * gather: 16-byte cp.async of whole 1 KiB rows (each thread copies 16
//     bytes of each 128-byte column segment, back to back) straight into a
//     128-byte-swizzled tile of 8 segments x 128 keys x 64 columns.  The tile
//     is read once from global memory and serves every head, as keys and as
//     values.  Q arrives by tiled TMA.  Keys past n_sel are zero-filled;
//     an out-of-range selection gathers a NaN row.
//   * MMA warp 8 (one thread) issues tcgen05.mma:
//       S^T[key][head]  = KV_tile (K-major, M=128) x Q^T (K-major, N=64)
//       O^T[col][head] += V^T (MN-major, M=128 per 128 columns) x P^T
//     P^T is one N=128 operand [P_hi | P_lo] for three of the four 128-column
//     chunks (the tensor core runs N=128 at full rate and N=64 at two
//     thirds) and two N=64 operands for the fourth, so the accumulators fit
//     TMEM: S^T columns [0,64), O^T chunks 0-2 at [64,192), [192,320),
//     [320,448) (hi | lo halves), chunk 3 at [448,512).
//   * softmax: worker w reads TMEM lane quadrant w%4 (32 keys) and heads
//     32*(w/4) .. +31.  A per-head reference maximum moves only when a score
//     exceeds it by more than 2^8 (then the running sums and O^T are
//     rescaled); only then are the tile maxima reduced (warp-shuffle
//     transpose reduction).  Weights are written as two bf16 terms
//     (P = hi + lo) so the value sum keeps ~16 bits; each thread keeps its
//     key lane's running sums, reduced over the 128 lanes once per unit.
//   * epilogue: sink fold and fp32 store, overlapped with the next tile's
//     gather and scores.
//
// Every wait is bounded (see dsa_ptx.cuh); on a timeout the kernel raises an
// error bit, lets its copies land, frees its TMEM and returns.
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kWorkerWarps = 8;
constexpr int kWorkers = 32 * kWorkerWarps;
constexpr int kMmaWarp = kWorkerWarps;
constexpr int kThreads = kWorkers + 32;
constexpr float kTau = 8.0f;            // log2 units
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kSegBytes = 128 * 128;          // 128 keys x 128 B
constexpr uint32_t kKvBytes = 8 * kSegBytes;       // 128 KiB
constexpr uint32_t kQSegBytes = 64 * 128;          // 64 heads x 128 B
constexpr uint32_t kQBytes = 8 * kQSegBytes;       // 64 KiB
constexpr uint32_t kPBytes = 128 * 128;            // 128 keys x 64 heads bf16
constexpr uint32_t kOffKv = 0;
constexpr uint32_t kOffQ = kOffKv + kKvBytes;
constexpr uint32_t kOffPhi = kOffQ + kQBytes;
constexpr uint32_t kOffPlo = kOffPhi + kPBytes;
constexpr uint32_t kOffMisc = kOffPlo + kPBytes;   // 229376

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;                     // S^T: 64 columns
// O^T chunk i (128 output columns): chunks 0-2 hold [hi | lo] halves of 64
// columns each, chunk 3 one 64-column accumulator for both terms.
__host__ __device__ constexpr uint32_t tmem_o(int i) { return 64u + 128u * static_cast<uint32_t>(i); }

struct Misc {
    uint64_t kv_full;       // workers' cp.async -> MMA: the KV tile landed
    uint64_t kv_free;       // MMA -> workers: P.V of the tile done (buffer and O^T free)
    uint64_t s_full;        // MMA -> workers: scores of the tile ready
    uint64_t p_full;        // workers -> MMA: P written (and O^T rescaled)
    uint64_t q_full;        // Q TMA -> MMA: Q of the unit landed
    uint64_t q_free;        // MMA -> worker 0: last score MMA of the unit done
    uint64_t grp[3];        // worker-group syncs
    uint64_t drain;         // MMA thread: everything it issued completed
    // the arrays below are read as float2 / float4: keep them 16-byte aligned
    alignas(16) float red_max[4][64];   // [TMEM lane quadrant][head]
    alignas(16) float red_sum[4][64];
    alignas(16) float m_ref[64];        // per-head reference maximum (log2 units)
    alignas(16) float alpha[64];        // per-head rescale factor; epilogue: output factor
    int ovf[kWorkerWarps];              // per worker warp: a score passed its reference max
    uint32_t tmem_base;
    int abort_flag;
    int rescale_flag;
};

static_assert(offsetof(Misc, red_max) % 16 == 0 && offsetof(Misc, red_sum) % 16 == 0 &&
                  offsetof(Misc, m_ref) % 16 == 0 && offsetof(Misc, alpha) % 16 == 0,
              "vector-accessed arrays must be 16-byte aligned");
static_assert(kOffMisc % 16 == 0, "Misc must start 16-byte aligned");
constexpr size_t kSmemBytes = kOffMisc + ((sizeof(Misc) + 15) / 16) * 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

#define DSA_R8(x) x, x, x, x, x, x, x, x
#define DSA_R64(x) DSA_R8(DSA_R8(x))
// Source row used for a selection that is out of range: every element NaN,
// so the whole output row of that query becomes NaN.
__device__ __align__(16) uint32_t kNanRowBf16[256] = {DSA_R64(0x7FC07FC0u), DSA_R64(0x7FC07FC0u),
                                                      DSA_R64(0x7FC07FC0u), DSA_R64(0x7FC07FC0u)};

struct Unit {
    int r, c, n_valid, tiles, bad_n;
};

__device__ __forceinline__ Unit unit_from(const TcParams& p, int u, int ns) {
    Unit x;
    x.r = u / p.chunks;
    x.c = u - x.r * p.chunks;
    x.bad_n = (ns < 0 || ns > p.k_max);
    const int eff = x.bad_n ? 1 : ns;                 // bad row: one NaN key
    int nv = eff - x.c * p.chunk_keys;
    nv = nv < 0 ? 0 : (nv > p.chunk_keys ? p.chunk_keys : nv);
    x.n_valid = nv;
    x.tiles = nv == 0 ? 1 : (nv + 127) / 128;         // an empty unit runs one masked tile
    return x;
}

__device__ __forceinline__ Unit unit_info(const TcParams& p, int u) {
    return unit_from(p, u, __ldg(p.n_sel + u / p.chunks));
}

__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t& phase, volatile int* ab,
                                           uint32_t* err) {
    mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, ab, err);
    phase ^= 1u;
    return ok;
}

// One halving step of the warp transpose reduction: lanes whose bit `O` is
// set keep the upper half of their W live values, the others the lower half,
// and each combines its kept half with the partner's sent half.
template <int W, int O, bool kMax>
__device__ __forceinline__ void tr_step(float* v, int lane) {
    const bool up = (lane & O) != 0;
#pragma unroll
    for (int i = 0; i < W / 2; ++i) {
        const float send = up ? v[i] : v[i + W / 2];
        const float keep = up ? v[i + W / 2] : v[i];
        const float recv = __shfl_xor_sync(0xffffffffu, send, O);
        v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
}

// Reduce 32 per-lane values over the 32 lanes of the warp, in place (v is
// clobbered): lane l ends with the result for value index l.  Fixed order:
// deterministic.
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce32(float* v, int lane) {
    tr_step<32, 16, kMax>(v, lane);
    tr_step<16, 8, kMax>(v, lane);
    tr_step<8, 4, kMax>(v, lane);
    tr_step<4, 2, kMax>(v, lane);
    tr_step<2, 1, kMax>(v, lane);
    return v[0];
}

// ------------------------------------------------------------------ gather
// The indices of this worker thread's four rows of a tile, loaded ahead
// without being looked at (so the loads do not stall the thread), and the
// n_sel of the tile's row.  Worker thread (warp w, lane l) copies 16 bytes
// (column chunk l%8) of each 128-byte segment of rows j = 4*(w + 8q) + l/8.
struct Prefetch {
    int raw[4];
    int nsel;
};

__device__ __forceinline__ Prefetch prefetch_rows(const TcParams& p, int u, int t, int wt) {
    const int w = wt >> 5, lane = wt & 31;
    const int r = u / p.chunks, c = u - r * p.chunks;
    Prefetch f;
    f.nsel = __ldg(p.n_sel + r);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int kk = c * p.chunk_keys + t * 128 + 4 * (w + 8 * q) + (lane >> 3);
        f.raw[q] = kk < p.k_max ? __ldg(p.idx + static_cast<size_t>(r) * p.k_max + kk) : 0;
    }
    return f;
}

// Validate the prefetched indices against the unit and copy the rows: keys
// past n_valid are zero-filled, an out-of-range selection copies a NaN row.
__device__ __forceinline__ void issue_rows(const TcParams& p, const Prefetch& f, const Unit& un, int t,
                                          uint32_t sKv, int wt) {
    const int w = wt >> 5, lane = wt & 31, cc = lane & 7;
    const uint16_t* cache = p.kv + (p.decode ? static_cast<size_t>(un.r) * p.N * kD : 0);
    const uint16_t* nan_row = reinterpret_cast<const uint16_t*>(kNanRowBf16);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int j = 4 * (w + 8 * q) + (lane >> 3);
        const bool valid = t * 128 + j < un.n_valid;
        const int id = f.raw[q];
        const bool in_range = !un.bad_n && id >= 0 && id < p.N;
        if (valid && !un.bad_n && !in_range && cc == 0) atomicOr(p.err, DSA_DEVERR_IDX_RANGE);
        const uint16_t* sp = (in_range ? cache + static_cast<size_t>(id) * kD : nan_row) + cc * 8;
        const uint32_t nb = valid ? 16u : 0u;
        const uint32_t dst = sKv + j * 128 + ((cc ^ (j & 7)) << 4);
#pragma unroll
        for (int s = 0; s < 8; ++s) cp_async16(dst + s * kSegBytes, sp + s * 64, nb);
    }
}

// --------------------------------------------------------------------- MMA
// S^T = KV x Q^T: 32 MMAs of K = 16 columns (segment s = k / 4, 32 bytes a step).
template <int k>
__device__ __forceinline__ void score_mma_step(uint32_t d, uint64_t dKv, uint64_t dQ) {
    constexpr uint32_t idS = idesc_bf16(128, 64, false, false);
    constexpr uint32_t aoff = ((k >> 2) * kSegBytes + (k & 3) * 32) >> 4;
    constexpr uint32_t boff = ((k >> 2) * kQSegBytes + (k & 3) * 32) >> 4;
    umma_bf16_at<aoff, boff>(d, dKv, dQ, idS, k != 0);
    if constexpr (k + 1 < 32) score_mma_step<k + 1>(d, dKv, dQ);
}

__device__ __forceinline__ void score_mmas(uint32_t d, uint64_t dKv, uint64_t dQ) {
    score_mma_step<0>(d, dKv, dQ);
}

// O^T += V^T x P^T for one 128-column chunk with the stacked N=128 operand.
template <int i, int kk>
__device__ __forceinline__ void pv128_step(uint32_t tmem, uint64_t dV, uint64_t dPst, uint32_t acc0) {
    constexpr uint32_t idPV128 = idesc_bf16(128, 128, true, true);
    constexpr uint32_t aoff = (2 * i * kSegBytes + kk * 2048) >> 4;
    constexpr uint32_t boff = (kk * 2048) >> 4;
    umma_bf16_at<aoff, boff>(tmem + tmem_o(i), dV, dPst, idPV128, acc0 | kk);
    if constexpr (kk + 1 < 8) pv128_step<i, kk + 1>(tmem, dV, dPst, acc0);
}

// Chunk 3: two N=64 operands (P_hi, P_lo) into one 64-column accumulator.
template <int kk>
__device__ __forceinline__ void pv64_step(uint32_t tmem, uint64_t dV, uint64_t dPhi, uint64_t dPlo,
                                          uint32_t acc0) {
    constexpr uint32_t idPV64 = idesc_bf16(128, 64, true, true);
    constexpr uint32_t aoff = (6 * kSegBytes + kk * 2048) >> 4;
    constexpr uint32_t boff = (kk * 2048) >> 4;
    umma_bf16_at<aoff, boff>(tmem + tmem_o(3), dV, dPhi, idPV64, acc0 | kk);
    umma_bf16_at<aoff, boff>(tmem + tmem_o(3), dV, dPlo, idPV64, 1u);
    if constexpr (kk + 1 < 8) pv64_step<kk + 1>(tmem, dV, dPhi, dPlo, acc0);
}

__device__ __forceinline__ void pv_mmas(uint32_t tmem, uint64_t dV, uint64_t dPst, uint64_t dPhi,
                                        uint64_t dPlo, uint32_t acc0) {
    pv128_step<0, 0>(tmem, dV, dPst, acc0);
    pv128_step<1, 0>(tmem, dV, dPst, acc0);
    pv128_step<2, 0>(tmem, dV, dPst, acc0);
    pv64_step<0>(tmem, dV, dPhi, dPlo, acc0);
}

__device__ void mma_role(const TcParams& p, uint8_t* smem, Misc& ms, uint32_t tmem) {
    const uint32_t sKv = smem_addr(smem + kOffKv);
    const uint32_t sQ = smem_addr(smem + kOffQ);
    const uint32_t sPhi = smem_addr(smem + kOffPhi);
    const uint32_t sPlo = smem_addr(smem + kOffPlo);
    volatile int* ab = &ms.abort_flag;
    // descriptor bases; steps are added to the start-address field (16-byte units)
    const uint64_t dKv = sdesc_sw128(sKv, 16, 1024);
    const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dV = sdesc_sw128(sKv, kSegBytes, 1024);     // MN-major: 64-column blocks 16 KiB apart
    const uint64_t dPst = sdesc_sw128(sPhi, kPBytes, 1024);    // N=128: block 0 = P_hi, block 1 = P_lo
    const uint64_t dPhi = sdesc_sw128(sPhi, 1024, 1024);
    const uint64_t dPlo = sdesc_sw128(sPlo, 1024, 1024);
    int g = 0, nu = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++nu) {
        const Unit un = unit_info(p, u);
        if (!mbar_wait(smem_addr(&ms.q_full), nu & 1, ab, p.err)) return;
        for (int t = 0; t < un.tiles; ++t, ++g) {
            // scores: S^T[key][head] over the 512 columns, 16 at a time
            if (!mbar_wait(smem_addr(&ms.kv_full), g & 1, ab, p.err)) return;
            fence_proxy_async();
            tc_fence_after();
            score_mmas(tmem + kTmemS, dKv, dQ);
            umma_commit(smem_addr(&ms.s_full));
            if (t == un.tiles - 1) umma_commit(smem_addr(&ms.q_free));

            // values: O^T[col][head] += V^T x (P_hi + P_lo)^T, 128 columns at a time
            if (!mbar_wait(smem_addr(&ms.p_full), g & 1, ab, p.err)) return;
            tc_fence_after();
            pv_mmas(tmem, dV, dPst, dPhi, dPlo, t > 0 ? 1u : 0u);
            umma_commit(smem_addr(&ms.kv_free));
        }
    }
}

// ----------------------------------------------------------------- workers
struct WorkerCtx {
    int wt, w, lane, qd, hf, key;   // thread, warp, lane, TMEM lane quadrant, head half, key in tile
    uint32_t lane_off;
    uint32_t ph[3];
};

// Per-head sums over the 128 key lanes, sink fold, store of one finished unit.
__device__ __forceinline__ bool epilogue(const TcParams& p, Misc& ms, WorkerCtx& c, uint32_t tmem, int u,
                                         int r, float* lacc /* clobbered */) {
    volatile int* ab = &ms.abort_flag;
    ms.red_sum[c.qd][32 * c.hf + c.lane] = warp_transpose_reduce32<false>(lacc, c.lane);
    if (!group_sync(smem_addr(&ms.grp[1]), c.ph[1], ab, p.err)) return false;
    if (c.w == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * c.lane + e;
            const float l = (ms.red_sum[0][h] + ms.red_sum[1][h]) + (ms.red_sum[2][h] + ms.red_sum[3][h]);
            const float m = ms.m_ref[h];
            float f = 1.0f;
            if (!p.partial) {
                const float mu = m == -INFINITY ? 0.0f : m;
                const float s2 = h < p.H ? __ldg(p.sink + h) * kLog2e : 0.0f;
                const float mstar = isfinite(s2) ? fmaxf(mu, s2) : mu;
                const float e1 = exp2f(mu - mstar);
                const float e2 = exp2f(s2 - mstar);
                f = e1 / (l * e1 + e2);
            } else {
                float* ml = p.part + static_cast<size_t>(p.units) * kHeadsPad * kD +
                            static_cast<size_t>(u) * 2 * kHeadsPad;
                ml[h] = m;
                ml[kHeadsPad + h] = l;
            }
            ms.alpha[h] = f;
            ms.m_ref[h] = -INFINITY;          // the next unit starts afresh
        }
    }
    if (!group_sync(smem_addr(&ms.grp[0]), c.ph[0], ab, p.err)) return false;
    tc_fence_after();
    float* dst = p.partial ? p.part + static_cast<size_t>(u) * kHeadsPad * kD
                           : p.out + static_cast<size_t>(r) * p.H * kD;
    // four chunks of this thread's column x its 32 heads; chunks 0-2 add the lo half
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
        const uint32_t ta = tmem + c.lane_off + tmem_o(i) + 32 * c.hf;
        float o[32];
        tmem_ld32(ta, o);
        if (i < 3) {
            float lo[32];
            tmem_ld32(ta + 64, lo);
#pragma unroll
            for (int h = 0; h < 32; ++h) o[h] += lo[h];
        }
        const int d = i * 128 + c.key;
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
            const float4 f = *reinterpret_cast<const float4*>(&ms.alpha[32 * c.hf + 4 * h4]);
            const float ff[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = 32 * c.hf + 4 * h4 + e;
                if (h < p.H) dst[static_cast<size_t>(h) * kD + d] = o[4 * h4 + e] * ff[e];
            }
        }
    }
    return true;
}

// Softmax of one tile: weights into P (hi, lo), running sums into lacc.
__device__ bool softmax_tile(const TcParams& p, uint8_t* smem, Misc& ms, WorkerCtx& c, uint32_t tmem,
                             const Unit& un, int t, float* lacc) {
    volatile int* ab = &ms.abort_flag;
    const uint32_t ts = tmem + c.lane_off + kTmemS + 32 * c.hf;
    const bool valid = t * 128 + c.key < un.n_valid;
    const float sc = p.scale_log2;
    const float* mref = &ms.m_ref[32 * c.hf];

    float x[32];
    tmem_ld32(ts, x);
#pragma unroll
    for (int h = 0; h < 32; ++h) x[h] = valid ? x[h] * sc : -INFINITY;

    // Does any score exceed its head's reference maximum by more than 2^8?
    // (The reference is -inf at the start of a unit, so any finite score
    // does.)  Only then are the tile maxima reduced.
    bool ovf = false;
#pragma unroll
    for (int h4 = 0; h4 < 8; ++h4) {
        const float4 m4 = *reinterpret_cast<const float4*>(&mref[4 * h4]);
        ovf |= (x[4 * h4] > m4.x + kTau) | (x[4 * h4 + 1] > m4.y + kTau) | (x[4 * h4 + 2] > m4.z + kTau) |
               (x[4 * h4 + 3] > m4.w + kTau);
    }
    ovf = __any_sync(0xffffffffu, ovf);
    if (c.lane == 0) ms.ovf[c.w] = ovf ? 1 : 0;
    if (!group_sync(smem_addr(&ms.grp[0]), c.ph[0], ab, p.err)) return false;
    int any_ovf = 0;
#pragma unroll
    for (int w = 0; w < kWorkerWarps; ++w) any_ovf |= ms.ovf[w];
    if (any_ovf) {
        ms.red_max[c.qd][32 * c.hf + c.lane] = warp_transpose_reduce32<true>(x, c.lane);
        // the reduction clobbered x: read the scores again
        tmem_ld32(ts, x);
#pragma unroll
        for (int h = 0; h < 32; ++h) x[h] = valid ? x[h] * sc : -INFINITY;
        if (!group_sync(smem_addr(&ms.grp[1]), c.ph[1], ab, p.err)) return false;
        if (c.w == 0) {
            bool resc = false;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = 2 * c.lane + e;
                const float tm = fmaxf(fmaxf(ms.red_max[0][h], ms.red_max[1][h]),
                                       fmaxf(ms.red_max[2][h], ms.red_max[3][h]));
                const float mo = ms.m_ref[h];
                float mn = mo, al = 1.0f;
                if (mo == -INFINITY) {
                    mn = tm;                       // nothing weighted yet
                } else if (tm > mo + kTau) {
                    mn = tm;
                    al = exp2f(mo - mn);
                    resc = true;
                }
                ms.m_ref[h] = mn;
                ms.alpha[h] = al;
            }
            const bool any = __any_sync(0xffffffffu, resc);
            if (c.lane == 0) ms.rescale_flag = any ? 1 : 0;
        }
        if (!group_sync(smem_addr(&ms.grp[2]), c.ph[2], ab, p.err)) return false;
        if (ms.rescale_flag) {
            // a moved reference maximum rescales the running sums (O^T below)
            const float* al = &ms.alpha[32 * c.hf];
#pragma unroll
            for (int h = 0; h < 32; ++h) lacc[h] *= al[h];
        }
    }

    // weights relative to the reference maximum (0 when it is -inf)
#pragma unroll
    for (int h4 = 0; h4 < 8; ++h4) {
        const float4 m4 = *reinterpret_cast<const float4*>(&mref[4 * h4]);
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float mu = mm[e] == -INFINITY ? 0.0f : mm[e];
            const float pe = ex2_approx(x[4 * h4 + e] - mu);
            x[4 * h4 + e] = pe;
            lacc[4 * h4 + e] += pe;
        }
    }
    // P = hi + lo, both bf16: this key's row, this thread's 4 chunks of 8 heads
    uint8_t* prow_hi = smem + kOffPhi + c.key * 128;
    uint8_t* prow_lo = smem + kOffPlo + c.key * 128;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = x[8 * c4 + 2 * e], b = x[8 * c4 + 2 * e + 1];
            const __nv_bfloat162 hv = __floats2bfloat162_rn(a, b);
            const float2 hf = __bfloat1622float2(hv);
            const __nv_bfloat162 lv = __floats2bfloat162_rn(a - hf.x, b - hf.y);
            hw[e] = *reinterpret_cast<const uint32_t*>(&hv);
            lw[e] = *reinterpret_cast<const uint32_t*>(&lv);
        }
        const int pc = ((4 * c.hf + c4) ^ (c.key & 7)) << 4;
        *reinterpret_cast<uint4*>(prow_hi + pc) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(prow_lo + pc) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    if (any_ovf && ms.rescale_flag) {
        // ... and what P.V accumulated so far (that P.V finished before this
        // tile's gather was issued); before P_full, so before this tile's P.V
        const float* al = &ms.alpha[32 * c.hf];
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < 7; ++i) {     // chunks 0-2: hi and lo halves; chunk 3
            const uint32_t ta = tmem + c.lane_off + tmem_o(i >> 1) + 64 * (i & 1) + 32 * c.hf;
            float o[32];
            tmem_ld32(ta, o);
#pragma unroll
            for (int h = 0; h < 32; ++h) o[h] *= al[h];
            tmem_st32(ta, o);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    mbar_arrive(smem_addr(&ms.p_full));
    return true;
}

__device__ void worker_role(const TcParams& p, uint8_t* smem, Misc& ms, uint32_t tmem, int& q_armed) {
    WorkerCtx c;
    c.wt = threadIdx.x;
    c.w = c.wt >> 5;
    c.lane = c.wt & 31;
    c.qd = c.w & 3;
    c.hf = c.w >> 2;
    c.key = 32 * c.qd + c.lane;
    c.lane_off = static_cast<uint32_t>(32 * c.qd) << 16;
    c.ph[0] = c.ph[1] = c.ph[2] = 0u;
    volatile int* ab = &ms.abort_flag;
    const uint32_t sKv = smem_addr(smem + kOffKv);
    const uint32_t sQ = smem_addr(smem + kOffQ);
    const uint32_t q_bytes = 8u * static_cast<uint32_t>(p.H) * 128u;
    const bool q_thread = c.wt == 0;

    int u = blockIdx.x;
    if (u >= p.units) return;
    Prefetch cur = prefetch_rows(p, u, 0, c.wt);
    Unit un = unit_from(p, u, cur.nsel);
    if (q_thread) {
        const uint32_t bar = smem_addr(&ms.q_full);
        mbar_arrive_expect_tx(bar, q_bytes);
        for (int s = 0; s < 8; ++s) tma_load_2d(sQ + s * kQSegBytes, &p.tmap_q, s * 64, un.r * p.H, bar);
        ++q_armed;
    }
    float lacc[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) lacc[h] = 0.0f;
    int t = 0, g = 0, nu = 0;
    int prev_u = -1, prev_r = 0;
    bool have_tile = true;
    while (true) {
        // 1. the previous tile's P.V is done with the KV buffer (and O^T)
        if (g > 0 && !mbar_wait(smem_addr(&ms.kv_free), (g - 1) & 1, ab, p.err)) return;
        bool last_tile = false, more = false;
        int u_next = u;
        if (have_tile) {
            // 2. gather this tile
            if (t == 0 && un.bad_n && un.c == 0 && c.wt == 0) atomicOr(p.err, DSA_DEVERR_NSEL_RANGE);
            issue_rows(p, cur, un, t, sKv, c.wt);
            cp_async_arrive(smem_addr(&ms.kv_full));
            last_tile = t + 1 == un.tiles;
            u_next = last_tile ? u + static_cast<int>(gridDim.x) : u;
            more = u_next < p.units;
        }
        // 3. finish the previous unit (its last P.V is done) while the gather
        //    of this tile runs
        if ((t == 0 || !have_tile) && prev_u >= 0) {
            if (!epilogue(p, ms, c, tmem, prev_u, prev_r, lacc)) return;
#pragma unroll
            for (int h = 0; h < 32; ++h) lacc[h] = 0.0f;
        }
        if (!have_tile) break;
        // 4. scores of this tile
        if (!mbar_wait(smem_addr(&ms.s_full), g & 1, ab, p.err)) return;
        tc_fence_after();
        // 5. indices of the next tile, loaded while the weights are computed
        //    (global loads running beside the score MMAs slow them down)
        if (more) cur = prefetch_rows(p, u_next, last_tile ? 0 : t + 1, c.wt);
        // 6. weights
        if (last_tile && more && q_thread) {
            // the unit's last score MMA has read Q: load the next unit's
            if (!mbar_wait(smem_addr(&ms.q_free), nu & 1, ab, p.err)) return;
            const uint32_t bar = smem_addr(&ms.q_full);
            mbar_arrive_expect_tx(bar, q_bytes);
            for (int s = 0; s < 8; ++s)
                tma_load_2d(sQ + s * kQSegBytes, &p.tmap_q, s * 64, (u_next / p.chunks) * p.H, bar);
            ++q_armed;
        }
        if (!softmax_tile(p, smem, ms, c, tmem, un, t, lacc)) return;
        ++g;
        if (last_tile) {
            prev_u = u;
            prev_r = un.r;
            ++nu;
            have_tile = more;
            u = u_next;
            if (more) un = unit_from(p, u, cur.nsel);
            t = 0;
        } else {
            ++t;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) dsa_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
    const int warp = threadIdx.x >> 5;
    if (smem_addr(smem) & 1023u) {   // the swizzle needs 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(p.err, DSA_DEVERR_LAYOUT);
        return;
    }
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&ms.kv_full), kWorkers);
        mbar_init(smem_addr(&ms.kv_free), 1);
        mbar_init(smem_addr(&ms.s_full), 1);
        mbar_init(smem_addr(&ms.p_full), kWorkers);
        mbar_init(smem_addr(&ms.q_full), 1);
        mbar_init(smem_addr(&ms.q_free), 1);
        for (int i = 0; i < 3; ++i) mbar_init(smem_addr(&ms.grp[i]), kWorkers);
        mbar_init(smem_addr(&ms.drain), 1);
        for (int h = 0; h < 64; ++h) ms.m_ref[h] = -INFINITY;
        ms.abort_flag = 0;
        ms.rescale_flag = 0;
        mbar_fence_init();
        prefetch_tmap(&p.tmap_q);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&ms.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (p.H < 64) {
        // rows of Q beyond H are never loaded and stay zero for the launch
        for (int e = threadIdx.x; e < (64 - p.H) * 64; e += kThreads) {
            const int h = p.H + e / 64, s = (e % 64) / 8, c = e % 8;
            *reinterpret_cast<uint4*>(smem + kOffQ + s * kQSegBytes + h * 128 + (c << 4)) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;

    if (warp < kWorkerWarps) {
        int q_armed = 0;
        worker_role(p, smem, ms, tmem, q_armed);
        cp_async_wait_all();
        if (q_armed > 0) {
            // the Q copies this thread armed have landed before the CTA can exit
            int dummy = 0;
            mbar_wait(smem_addr(&ms.q_full), (q_armed - 1) & 1, &dummy, p.err);
        }
        __syncwarp();
    } else {
        if ((threadIdx.x & 31) == 0) {
            mma_role(p, smem, ms, tmem);
            // every MMA this thread issued has completed before TMEM is freed
            umma_commit(smem_addr(&ms.drain));
            int dummy = 0;
            mbar_wait(smem_addr(&ms.drain), 0, &dummy, p.err);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t tc_smem_bytes() { return kSmemBytes; }

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// A 2-D bf16 tensor of `rows` rows of 512 values (1024-byte pitch), read in
// boxes of 64 columns x box_rows rows with the 128-byte swizzle (the layout
// the MMA descriptors expect).
bool encode_rows(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc(const TcParams& params, int grid, cudaStream_t s) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(dsa_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    TcParams p = params;
    if (!encode_rows(&p.tmap_q, p.q, static_cast<uint64_t>(p.R) * p.H, static_cast<uint32_t>(p.H)))
        return cudaErrorInvalidValue;
    dsa_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
