// Top-k sparse attention on the sm_103a tensor cores (bf16 inputs).
//
// What it computes: for one query row and all of its heads, the softmax over
// the row's selected latent KV rows plus one sink logit per head, weighted
// sum of the same rows (akol1 TensorFold PR #4, first commit message: score a
// tile of keys, keep a running maximum, a tile sum and a value sum;
// TensorFold PR #1206, "What changes": per-head sinks).
//
// How (one CTA per SM, persistent over work units; a unit is one row, or one
// key chunk of a row when a decode batch is split across SMs).  A prefill
// launch with more rows than CTAs hands rows out from a queue in device
// memory (warp 14 takes them, one unit ahead), since SMs run at slightly
// different speeds; otherwise units go round-robin over the grid.  Per 128-key
// tile the work is a chain: gather -> scores -> softmax -> P.V, and the one
// shared-memory KV tile (128 KiB) is busy from its gather to the end of its
// P.V.  Sixteen warps in four warpgroups:
//
//   * worker warps 0-7 (176 registers each, by setmaxnreg):
//     gather: 16-byte cp.async of whole 1 KiB rows (each thread copies 16
//     bytes of each 128-byte column segment, back to back) straight into a
//     128-byte-swizzled tile of 8 segments x 128 keys x 64 columns, 32 keys
//     at a time as the previous tile's P.V releases them.  The tile is read
//     once from global memory and serves every head, as keys and as values.
//     The tile's indices arrive one tile ahead by cp.async (warp 14), Q by
//     tiled TMA (warp 13).
//     Keys past n_sel are zero-filled; an out-of-range selection gathers a
//     NaN row.
//     softmax: worker w reads TMEM lane quadrant w%4 (32 keys) and heads
//     32*(w/4) .. +31.  With finite sinks a unit starts from per-head
//     reference maxima equal to the sink logits; otherwise its first tile
//     sets them to the tile's maxima (warp transpose reduction, one sync).
//     The references are used optimistically: a score more than 2^32 above
//     its reference, or a sink-seeded first tile that leaves a head without
//     a weight of at least 2^-100, flags the tile and the MMA warp has it
//     redone with moved references (running sums and O^T rescaled; a
//     flagged first tile takes its exact maxima).  Weights are written as two bf16 terms
//     (P = hi + lo) so the value sum keeps ~14 bits; each thread keeps its
//     key lane's running sums, reduced over the 128 lanes once per unit.
//   * warp 13 (one thread) loads each unit's Q by TMA once the workers have
//     written P for the last tile of the unit before (its score MMAs, the
//     last reads of Q, are done by then).
//   * MMA warp 12 (one thread) issues tcgen05.mma:
//       S^T[key][head]  = KV_tile (K-major, M=128) x Q^T (K-major, N=64)
//       O^T[col][head] += V^T (MN-major, M=128 per 128 columns) x P^T
//     P^T is one N=128 operand [P_hi | P_lo] for three of the four 128-column
//     chunks (the tensor core runs N=128 at full rate and N=64 at two
//     thirds) and two N=64 operands for the fourth, so the accumulators fit
//     TMEM: S^T columns [0,64), O^T chunks 0-2 at [64,192), [192,320),
//     [320,448) (hi | lo halves), chunk 3 at [448,512).
//   * output warps 8-11 (one per TMEM lane quadrant): sink fold and fp32
//     store of a finished unit while the workers run the next one; the next
//     unit's first P.V waits until they have read O^T.
//
// Every wait is bounded (see dsa_ptx.cuh); on a timeout the kernel raises an
// error bit, lets its copies land, frees its TMEM and returns.
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

// Four warpgroups: two of worker warps, one of output warps (one per TMEM
// lane quadrant), one holding the MMA warp.  The launch gives every thread
// 128 registers; the workers take 176 and the others keep 80.
constexpr int kWorkerWarps = 8;
constexpr int kWorkers = 32 * kWorkerWarps;
constexpr int kOutWarp0 = 8;
constexpr int kOutWarps = 4;
constexpr int kMmaWarp = 12;
constexpr int kThreads = 512;
constexpr int kQWarp = kMmaWarp + 1;         // loads each unit's Q
constexpr int kIdxWarp = kMmaWarp + 2;       // copies each tile's indices ahead
constexpr uint32_t kRegsWorker = 176;
constexpr uint32_t kRegsOther = 80;
// two warpgroups at kRegsWorker and two at kRegsOther use exactly the
// 65536 registers that 512 threads x 128 bring
static_assert((2 * kRegsWorker + 2 * kRegsOther) * 128 == 65536 && 65536 / kThreads == 128,
              "the register split must add up to what the launch provides");
// A reference maximum may lag the scores by up to 2^kTau (log2 units): the
// weights stay below 2^32 and a unit's sums below 2^42.
constexpr float kTau = 32.0f;
// A unit whose first tile is weighed against the sinks must give every head
// with a selected key a weight of at least 2^kLowest (log2 units); else the
// tile is redone with its exact maxima.
constexpr float kLowest = -100.0f;
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
    uint64_t kv_free[5];    // MMA -> workers: P.V is done with keys [0, 32(i+1)) of the
                            // tile for i < 3, [0, 112) for [3], all of them for [4]
    uint64_t s_full;        // MMA -> workers: scores of the tile ready
    uint64_t p_full;        // worker warps -> MMA: P written (and O^T rescaled)
    uint64_t q_full;        // Q TMA -> MMA: Q of the unit landed
    uint64_t q_free;        // MMA -> Q warp: P of the unit's last tile written (its scores, the
                            // last reads of Q, are done), so Q may be reloaded
    uint64_t p_ack;         // MMA -> workers: P accepted, or ms.redo set
    uint64_t red_sync;      // worker-warp sync of the tile-maxima reduction (one arrival per warp)
    uint64_t drain;         // MMA thread: everything it issued completed
    uint64_t idx_full;      // index warp's cp.async -> workers: idx[] holds the next tile's
    uint64_t o_full;        // MMA -> output warps: the unit's last P.V is done
    uint64_t o_free;        // output warps -> MMA: the unit's O^T has been read
    uint64_t l_ready;       // worker warps -> output warps: red_l, m_ref hold the unit's sums, maxima
    uint64_t l_free;        // output warps -> workers: red_l, m_ref of the unit have been read
    // the arrays below are read as float4: keep them 16-byte aligned
    alignas(16) float red[4][64];       // [TMEM lane quadrant][head]: tile maxima
    alignas(16) float red_l[4][64];     // [TMEM lane quadrant][head]: a finished unit's sums
    alignas(16) float m_ref[64];        // per-head reference maximum (log2 units)
    uint64_t unit_full[4];  // index warp -> all roles: unit_ring[nu % 4] holds the CTA's nu-th unit
    int unit_ring[4];       // units taken from the launch's queue, in the CTA's order
    int ovf;                            // a worker warp saw a score pass its reference max
    uint32_t seen[2];       // per head half, a unit's first tile weighed against the sinks: bit h
                            // set if head 32*half+h has a weight >= 2^kLowest
    uint32_t tmem_base;
    int abort_flag;
    int redo;                           // the flagged tile is to be redone
    int idx[128];                       // the selected rows of the tile being gathered
    int idx_nsel;                       // n_sel of that tile's query row
};

static_assert(offsetof(Misc, red) % 16 == 0 && offsetof(Misc, red_l) % 16 == 0 &&
                  offsetof(Misc, m_ref) % 16 == 0,
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

// Whether every sink of the launch is finite (the same answer in every lane).
__device__ __forceinline__ bool sinks_finite(const TcParams& p, int lane) {
    const bool a = lane >= p.H || isfinite(__ldg(p.sink + lane));
    const bool b = lane + 32 >= p.H || isfinite(__ldg(p.sink + lane + 32));
    return __all_sync(0xffffffffu, a && b);
}

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

// The CTA's nu-th unit, or p.units when it has no more: round-robin over
// the grid, or, with a launch queue (p.queue), the units the index warp has
// taken from it in turn.  A row's result does not depend on which CTA runs it.
__device__ __forceinline__ int unit_at(const TcParams& p, Misc& ms, int nu) {
    if (!p.queue) return blockIdx.x + nu * static_cast<int>(gridDim.x);
    if (!mbar_wait(smem_addr(&ms.unit_full[nu & 3]), (nu >> 2) & 1, &ms.abort_flag, p.err)) return p.units;
    return *reinterpret_cast<volatile int*>(&ms.unit_ring[nu & 3]);
}

// Index warp: takes the next unit of the launch queue as the CTA's nu-th
// and publishes it in the ring (p.units once the queue is empty).  It runs
// one unit ahead of the CTA, and a unit's slot is reused four units later,
// when every role has long read it: the slowest reader, the output warps,
// read the CTA's unit nu - 2 before any P.V of unit nu - 1 can start (that
// waits for them), and the ring is filled for unit nu + 1 only once the
// scores of unit nu - 1's last tile are done.
__device__ __forceinline__ int take_unit(const TcParams& p, Misc& ms, int nu, int lane) {
    int u = 0;
    if (lane == 0) {
        const int ticket = atomicAdd(p.queue, 1);
        u = ticket < p.units ? ticket : p.units;
        ms.unit_ring[nu & 3] = u;
        mbar_arrive(smem_addr(&ms.unit_full[nu & 3]));
    }
    return __shfl_sync(0xffffffffu, u, 0);
}

// Sync of the worker warps: one arrival per warp (after __syncwarp, which
// orders the lanes' shared-memory writes before lane 0's release).
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t& phase, volatile int* ab,
                                           uint32_t* err) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
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
// The index warp copies the 128 selected rows of a tile (and its row's
// n_sel) into shared memory with cp.async while the previous tile is being
// computed, so that no thread holds them in registers meanwhile.  Entries at
// or past k_max are never read.
__device__ __forceinline__ void prefetch_idx(const TcParams& p, int u, int t, Misc& ms, int lane) {
    const int r = u / p.chunks, c = u - r * p.chunks;
    const int* row = p.idx + static_cast<size_t>(r) * p.k_max;
    const int k0 = c * p.chunk_keys + t * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int kk = k0 + lane + 32 * i;
        const bool in = kk < p.k_max;
        cp_async4(smem_addr(&ms.idx[lane + 32 * i]), in ? row + kk : row, in ? 4u : 0u);
    }
    if (lane == 0) cp_async4(smem_addr(&ms.idx_nsel), p.n_sel + r, 4u);
    cp_async_arrive(smem_addr(&ms.idx_full));
}

// Validate the prefetched indices against the unit and copy rows [32q,
// 32q + 32) of the tile: worker thread (warp w, lane l) copies 16 bytes
// (column chunk l%8) of each 128-byte segment of row 4*(w + 8q) + l/8.  Keys
// past n_valid are zero-filled, an out-of-range selection copies a NaN row.
// kShared: several decode rows share a slot (row r reads slot r / p.decode);
// a separate kernel instance, so that the common one keeps its plain address.
template <int q, bool kShared>
__device__ __forceinline__ void issue_rows(const TcParams& p, const Misc& ms, const Unit& un, int t,
                                          uint32_t sKv, int wt) {
    const int w = wt >> 5, lane = wt & 31, cc = lane & 7;
    const size_t slot = kShared ? static_cast<size_t>(un.r / p.decode) : static_cast<size_t>(un.r);
    const uint16_t* cache = p.kv + (p.decode ? slot * p.N * kD : 0);
    const uint16_t* nan_row = reinterpret_cast<const uint16_t*>(kNanRowBf16);
    {
        const int j = 4 * (w + 8 * q) + (lane >> 3);
        const bool valid = t * 128 + j < un.n_valid;
        const int id = ms.idx[j];
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

// O^T += V^T x P^T for 16 keys (k-step kk) of every 128-column chunk: the
// stacked N=128 operand for chunks 0-2, two N=64 operands for chunk 3.
template <int kk>
__device__ __forceinline__ void pv_kstep(uint32_t tmem, uint64_t dV, uint64_t dPst, uint64_t dPhi, uint64_t dPlo,
                                         uint32_t acc0) {
    constexpr uint32_t idPV128 = idesc_bf16(128, 128, true, true);
    constexpr uint32_t idPV64 = idesc_bf16(128, 64, true, true);
    constexpr uint32_t boff = (kk * 2048) >> 4;
    constexpr uint32_t a0 = (0 * kSegBytes + kk * 2048) >> 4, a1 = (2 * kSegBytes + kk * 2048) >> 4;
    constexpr uint32_t a2 = (4 * kSegBytes + kk * 2048) >> 4, a3 = (6 * kSegBytes + kk * 2048) >> 4;
    umma_bf16_at<a0, boff>(tmem + tmem_o(0), dV, dPst, idPV128, acc0 | kk);
    umma_bf16_at<a1, boff>(tmem + tmem_o(1), dV, dPst, idPV128, acc0 | kk);
    umma_bf16_at<a2, boff>(tmem + tmem_o(2), dV, dPst, idPV128, acc0 | kk);
    umma_bf16_at<a3, boff>(tmem + tmem_o(3), dV, dPhi, idPV64, acc0 | kk);
    umma_bf16_at<a3, boff>(tmem + tmem_o(3), dV, dPlo, idPV64, 1u);
}

// Keys [32q, 32q + 32) of the tile, then a commit that frees those rows of
// the KV buffer for the next tile's gather.
// The last quarter is released in two halves, so only 16 rows are left to
// gather once the P.V is over.
template <int q>
__device__ __forceinline__ void pv_quarter(uint32_t tmem, uint64_t dV, uint64_t dPst, uint64_t dPhi,
                                           uint64_t dPlo, uint32_t acc0, Misc& ms) {
    pv_kstep<2 * q>(tmem, dV, dPst, dPhi, dPlo, acc0);
    if (q == 3) umma_commit(smem_addr(&ms.kv_free[3]));
    pv_kstep<2 * q + 1>(tmem, dV, dPst, dPhi, dPlo, acc0);
    umma_commit(smem_addr(&ms.kv_free[q == 3 ? 4 : q]));
}

__device__ void mma_role(const TcParams& p, uint8_t* smem, Misc& ms, uint32_t tmem, bool sinks) {
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
    uint32_t ph_p = 0;
    // heads of the launch, per head half
    const uint32_t need0 = p.H >= 32 ? 0xFFFFFFFFu : (1u << p.H) - 1u;
    const uint32_t need1 = p.H >= 64 ? 0xFFFFFFFFu : (p.H > 32 ? (1u << (p.H - 32)) - 1u : 0u);
    for (;; ++nu) {
        const int u = unit_at(p, ms, nu);
        if (u >= p.units) break;
        const Unit un = unit_info(p, u);
        if (!mbar_wait(smem_addr(&ms.q_full), nu & 1, ab, p.err)) return;
        for (int t = 0; t < un.tiles; ++t, ++g) {
            // scores: S^T[key][head] over the 512 columns, 16 at a time
            if (!mbar_wait(smem_addr(&ms.kv_full), g & 1, ab, p.err)) return;
            fence_proxy_async();
            tc_fence_after();
            score_mmas(tmem + kTmemS, dKv, dQ);
            umma_commit(smem_addr(&ms.s_full));

            // values: O^T[col][head] += V^T x (P_hi + P_lo)^T, 128 columns at a time
            if (!mbar_wait(smem_addr(&ms.p_full), ph_p, ab, p.err)) return;
            ph_p ^= 1u;
            // a tile that a worker warp flagged is redone with new reference maxima
            volatile int* ovf = &ms.ovf;
            int flagged = *ovf;
            if (t == 0 && sinks) {
                // a sink-seeded first tile must leave every head a weight >= 2^kLowest
                volatile uint32_t* seen = ms.seen;
                if (un.n_valid > 0 && ((seen[0] & need0) != need0 || (seen[1] & need1) != need1)) flagged = 1;
                seen[0] = 0;
                seen[1] = 0;
            }
            if (flagged) {
                *ovf = 0;
                *reinterpret_cast<volatile int*>(&ms.redo) = 1;
                mbar_arrive(smem_addr(&ms.p_ack));
                if (!mbar_wait(smem_addr(&ms.p_full), ph_p, ab, p.err)) return;
                ph_p ^= 1u;
                *reinterpret_cast<volatile int*>(&ms.redo) = 0;
            }
            // the workers saw the unit's last score MMAs complete before they
            // wrote P: the Q warp may load the next unit's Q (not earlier, so
            // that its copy does not run beside this tile's softmax)
            if (t == un.tiles - 1) mbar_arrive(smem_addr(&ms.q_free));
            mbar_arrive(smem_addr(&ms.p_ack));
            // a unit's first P.V overwrites O^T: the output warps must have read the last one
            if (t == 0 && nu > 0 && !mbar_wait(smem_addr(&ms.o_free), (nu - 1) & 1, ab, p.err)) return;
            tc_fence_after();
            const uint32_t acc0 = t > 0 ? 1u : 0u;
            pv_quarter<0>(tmem, dV, dPst, dPhi, dPlo, acc0, ms);
            pv_quarter<1>(tmem, dV, dPst, dPhi, dPlo, acc0, ms);
            pv_quarter<2>(tmem, dV, dPst, dPhi, dPlo, acc0, ms);
            pv_quarter<3>(tmem, dV, dPst, dPhi, dPlo, acc0, ms);
            if (t == un.tiles - 1) umma_commit(smem_addr(&ms.o_full));
        }
    }
}

// ----------------------------------------------------------------- workers
struct WorkerCtx {
    int wt, w, lane, qd, hf, key;   // thread, warp, lane, TMEM lane quadrant, head half, key in tile
    bool sinks;                     // every sink is finite: units start from sink references
    float sink_mine;                // the sink reference of head 32 hf + lane (quadrant 0 publishes it)
    uint32_t lane_off;
    uint32_t ph_red, ph_ack;        // phases of red_sync and p_ack
};

// Scores of this thread's key for its 32 heads, in log2 units; -inf for a
// key past n_valid.
__device__ __forceinline__ void load_scores(uint32_t ts, bool valid, float sc, float* x) {
    tmem_ld32(ts, x);
#pragma unroll
    for (int h = 0; h < 32; ++h) x[h] = valid ? x[h] * sc : -INFINITY;
}

// New reference maxima for this thread's 32 heads from the tile maxima of
// all four key quadrants (one sync of the worker warps).  On a unit's first
// tile the references are set; later a reference moves only when the tile
// maximum passes it by more than 2^kTau, and then this thread's running sums
// and its block of O^T are rescaled.  The quadrant-0 warps publish the new
// references for later tiles and for the output warps.  x is clobbered.
template <bool kFirst>
__device__ bool new_reference(const TcParams& p, Misc& ms, WorkerCtx& c, uint32_t tmem, float* x,
                              float* mref, int nu, float* lacc) {
    volatile int* ab = &ms.abort_flag;
    // lane l: head l's maximum over this warp's 32 keys
    ms.red[c.qd][32 * c.hf + c.lane] = warp_transpose_reduce32<true>(x, c.lane);
    if (!group_sync(smem_addr(&ms.red_sync), c.ph_red, ab, p.err)) return false;
    if (c.qd == 0) {
        // lane l publishes head l's reference (read by later tiles and the
        // output warps, which may still be reading the previous unit's)
        if (kFirst && nu > 0 && !mbar_wait(smem_addr(&ms.l_free), (nu - 1) & 1, ab, p.err)) return false;
        const int h = 32 * c.hf + c.lane;
        const float tm = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
        if (kFirst) {
            ms.m_ref[h] = tm;
        } else {
            const float mo = ms.m_ref[h];
            if (mo == -INFINITY || tm > mo + kTau) ms.m_ref[h] = tm;
        }
    }
    bool resc = false;           // the same in every lane: the warp's lanes share their heads
    float alpha[32];
#pragma unroll
    for (int h4 = 0; h4 < 8; ++h4) {
        const float4 q0 = *reinterpret_cast<const float4*>(&ms.red[0][32 * c.hf + 4 * h4]);
        const float4 q1 = *reinterpret_cast<const float4*>(&ms.red[1][32 * c.hf + 4 * h4]);
        const float4 q2 = *reinterpret_cast<const float4*>(&ms.red[2][32 * c.hf + 4 * h4]);
        const float4 q3 = *reinterpret_cast<const float4*>(&ms.red[3][32 * c.hf + 4 * h4]);
        const float tm[4] = {fmaxf(fmaxf(q0.x, q1.x), fmaxf(q2.x, q3.x)), fmaxf(fmaxf(q0.y, q1.y), fmaxf(q2.y, q3.y)),
                             fmaxf(fmaxf(q0.z, q1.z), fmaxf(q2.z, q3.z)), fmaxf(fmaxf(q0.w, q1.w), fmaxf(q2.w, q3.w))};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int h = 4 * h4 + e;
            if (kFirst) {
                mref[h] = tm[e];
                continue;
            }
            const float mo = mref[h];
            float mn = mo, al = 1.0f;
            if (mo == -INFINITY) {
                mn = tm[e];                    // nothing weighted yet
            } else if (tm[e] > mo + kTau) {
                mn = tm[e];
                al = exp2f(mo - mn);
                resc = true;
            }
            mref[h] = mn;
            alpha[h] = al;
        }
    }
    if (!kFirst && resc) {
#pragma unroll
        for (int h = 0; h < 32; ++h) lacc[h] *= alpha[h];
        // O^T of the earlier tiles (their P.V is complete: this tile's gather
        // waited for it), before this tile's P.V
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < 7; ++i) {     // chunks 0-2: hi and lo halves; chunk 3
            const uint32_t ta = tmem + c.lane_off + tmem_o(i >> 1) + 64 * (i & 1) + 32 * c.hf;
            float o[32];
            tmem_ld32(ta, o);
#pragma unroll
            for (int h = 0; h < 32; ++h) o[h] *= alpha[h];
            tmem_st32(ta, o);
        }
    }
    return true;
}

// Weights of this thread's key for its 32 heads, in place over the raw
// scores in x: 2^(s*sc - m_h), one FFMA and one ex2 each (the reference's
// negation is an operand modifier); 0 for a key past n_valid.  A head whose
// reference is still -inf (no finite score yet) weighs against 0 instead,
// on a separate path that the warp takes as a whole (its lanes share their
// heads).  Returns whether a valid score passes its reference by more than
// 2^kTau (the largest exponent against kTau: a NaN exponent passes nothing).
// kFull: every key of the tile is valid, so no weight needs masking.
template <bool kSeen = false, bool kFull = false>
__device__ __forceinline__ bool tile_weights(float* x, bool valid, float sc, const float* mref, bool ninf,
                                             uint32_t* seen = nullptr) {
    bool ovf = false;
    if (kSeen) {
        // references from the sinks (all finite); bit h of *seen: this key
        // gives head h a weight of at least 2^kLowest
        uint32_t m = 0;
        float dmax = -INFINITY;
#pragma unroll
        for (int h = 0; h < 32; ++h) {
            const float d = fmaf(x[h], sc, -mref[h]);
            dmax = fmaxf(dmax, d);
            m |= (d >= kLowest) ? (1u << h) : 0u;
            x[h] = (kFull || valid) ? ex2_approx_ftz(d) : 0.0f;
        }
        ovf = dmax > kTau;
        *seen = valid ? m : 0u;
    } else if (!ninf) {
        float dmax = -INFINITY;
#pragma unroll
        for (int h = 0; h < 32; ++h) {
            const float d = fmaf(x[h], sc, -mref[h]);
            dmax = fmaxf(dmax, d);
            x[h] = (kFull || valid) ? ex2_approx_ftz(d) : 0.0f;
        }
        ovf = dmax > kTau;
    } else {
#pragma unroll
        for (int h = 0; h < 32; ++h) {
            const float s = x[h] * sc;
            ovf |= s > mref[h] + kTau;
            const float mu = mref[h] == -INFINITY ? 0.0f : mref[h];
            x[h] = valid ? ex2_approx_ftz(s - mu) : 0.0f;
        }
    }
    return valid && ovf;
}

// Whether any of this thread's 32 references is -inf.
__device__ __forceinline__ bool any_ninf(const float* mref) {
    bool any = false;
#pragma unroll
    for (int h = 0; h < 32; ++h) any |= mref[h] == -INFINITY;
    return any;
}

// Writes the weights in x to P as two bf16 terms: hi is the top 16 bits of
// the fp32 weight, lo the top 16 bits of the exact remainder, so hi + lo is
// within 2^-14 of the weight (relative) and the split takes no conversion
// instructions.  This key's row, this thread's 4 chunks of 8 heads.
__device__ __forceinline__ void store_p(uint8_t* smem, const WorkerCtx& c, const float* x) {
    uint8_t* prow_hi = smem + kOffPhi + c.key * 128;
    uint8_t* prow_lo = smem + kOffPlo + c.key * 128;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t ua = __float_as_uint(x[8 * c4 + 2 * e]);
            const uint32_t ub = __float_as_uint(x[8 * c4 + 2 * e + 1]);
            const float la = x[8 * c4 + 2 * e] - __uint_as_float(ua & 0xFFFF0000u);
            const float lb = x[8 * c4 + 2 * e + 1] - __uint_as_float(ub & 0xFFFF0000u);
            hw[e] = __byte_perm(ua, ub, 0x7632);     // head 2e in the low half, 2e+1 in the high
            lw[e] = __byte_perm(__float_as_uint(la), __float_as_uint(lb), 0x7632);
        }
        const int pc = ((4 * c.hf + c4) ^ (c.key & 7)) << 4;
        *reinterpret_cast<uint4*>(prow_hi + pc) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(prow_lo + pc) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
}

// P (and any O^T rescale) done: hand the tile to the MMA warp and wait for its
// answer, which says whether a flagged tile has to be redone.
__device__ __forceinline__ bool publish_p(const TcParams& p, Misc& ms, WorkerCtx& c) {
    fence_proxy_async();
    tc_fence_before();
    __syncwarp();
    if (c.lane == 0) mbar_arrive(smem_addr(&ms.p_full));
    if (!mbar_wait(smem_addr(&ms.p_ack), c.ph_ack, &ms.abort_flag, p.err)) return false;
    c.ph_ack ^= 1u;
    return true;
}

// Sink logit of head h in log2 units, the reference a unit's first tile
// starts from when every sink is finite (0 for a padding head).
__device__ __forceinline__ float sink_ref(const TcParams& p, int h) {
    return h < p.H ? __ldg(p.sink + h) * kLog2e : 0.0f;
}

// Softmax of one tile: weights into P, running sums into lacc.  mref holds
// this thread's references across tiles (ninf: one of them is -inf).
// With finite sinks (c.sinks) a unit starts from references equal to the
// sink logits, loaded into mref during the gather; otherwise its first tile
// sets them to the tile's exact maxima (a reduction over the worker warps).
// The references are used optimistically: a warp that sees a score more
// than 2^kTau above its reference flags the tile (and so does the MMA warp
// when a sink-seeded first tile leaves a head without a weight of at least
// 2^kLowest); every worker then redoes the tile with new references before
// any P.V reads P.
__device__ __forceinline__ bool softmax_tile(const TcParams& p, uint8_t* smem, Misc& ms, WorkerCtx& c, uint32_t tmem,
                             const Unit& un, int t, int nu, float* lacc, float* mref, bool& ninf) {
    const uint32_t ts = tmem + c.lane_off + kTmemS + 32 * c.hf;
    const bool valid = t * 128 + c.key < un.n_valid;
    const bool seeded = t == 0 && c.sinks;
    float x[32];
    if (t == 0) {
        if (seeded) {
            // publish the sink references for the output warps, once they
            // have read the previous unit's
            ninf = false;
            if (c.qd == 0) {
                if (nu > 0 && !mbar_wait(smem_addr(&ms.l_free), (nu - 1) & 1, &ms.abort_flag, p.err)) return false;
                ms.m_ref[32 * c.hf + c.lane] = c.sink_mine;
            }
        } else {
            load_scores(ts, valid, p.scale_log2, x);
            if (!new_reference<true>(p, ms, c, tmem, x, mref, nu, lacc)) return false;
            ninf = any_ninf(mref);
        }
    }
    tmem_ld32(ts, x);
    bool ovf;
    const bool full = (t + 1) * 128 <= un.n_valid;      // the same in every thread
    if (seeded) {
        uint32_t seen;
        ovf = full ? tile_weights<true, true>(x, valid, p.scale_log2, mref, false, &seen)
                   : tile_weights<true>(x, valid, p.scale_log2, mref, false, &seen);
        seen = __reduce_or_sync(0xffffffffu, seen);
        if (c.lane == 0 && seen) atomicOr(&ms.seen[c.hf], seen);
    } else {
        // an exact first tile's references are its maxima: nothing can pass them
        ovf = (full ? tile_weights<false, true>(x, valid, p.scale_log2, mref, ninf)
                    : tile_weights(x, valid, p.scale_log2, mref, ninf)) &&
              t > 0;
    }
    ovf = __any_sync(0xffffffffu, ovf);
    store_p(smem, c, x);
    if (ovf && c.lane == 0) ms.ovf = 1;
    if (!publish_p(p, ms, c)) return false;
    if (ms.redo) {
        if (seeded) {
            // a sink-seeded first tile is redone with its exact maxima: from
            // references of -inf they move to the tile's maxima, and nothing
            // weighted so far needs rescaling
#pragma unroll
            for (int h = 0; h < 32; ++h) mref[h] = -INFINITY;
            if (c.qd == 0) ms.m_ref[32 * c.hf + c.lane] = -INFINITY;
        }
        load_scores(ts, valid, p.scale_log2, x);
        if (!new_reference<false>(p, ms, c, tmem, x, mref, nu, lacc)) return false;
        ninf = any_ninf(mref);
        tmem_ld32(ts, x);
        tile_weights(x, valid, p.scale_log2, mref, ninf);
        store_p(smem, c, x);
        if (!publish_p(p, ms, c)) return false;
    }
#pragma unroll
    for (int h = 0; h < 32; ++h) lacc[h] += x[h];
    return true;
}

template <bool kShared>
__device__ void worker_role(const TcParams& p, uint8_t* smem, Misc& ms, uint32_t tmem) {
    WorkerCtx c;
    c.wt = threadIdx.x;
    c.w = c.wt >> 5;
    c.lane = c.wt & 31;
    c.qd = c.w & 3;
    c.hf = c.w >> 2;
    c.key = 32 * c.qd + c.lane;
    c.lane_off = static_cast<uint32_t>(32 * c.qd) << 16;
    c.ph_red = c.ph_ack = 0u;
    c.sinks = sinks_finite(p, c.lane);
    volatile int* ab = &ms.abort_flag;
    const uint32_t sKv = smem_addr(smem + kOffKv);

    int u = unit_at(p, ms, 0);
    if (u >= p.units) return;
    Unit un;
    float lacc[32], mref[32];   // this thread's running sums and references (set by each unit's first tile)
    bool ninf = true;
#pragma unroll
    for (int h = 0; h < 32; ++h) lacc[h] = 0.0f;
    int t = 0, g = 0, nu = 0;
    while (true) {
        // 1-2. gather this tile, 32 keys at a time, each as soon as the previous
        //      tile's P.V is done with those rows of the buffer
        if (!mbar_wait(smem_addr(&ms.idx_full), g & 1, ab, p.err)) return;
        if (t == 0) un = unit_from(p, u, ms.idx_nsel);
        if (t == 0 && un.bad_n && un.c == 0 && c.wt == 0) atomicOr(p.err, DSA_DEVERR_NSEL_RANGE);
        const uint32_t ph = (g - 1) & 1;
        if (g > 0 && !mbar_wait(smem_addr(&ms.kv_free[0]), ph, ab, p.err)) return;
        issue_rows<0, kShared>(p, ms, un, t, sKv, c.wt);
        cp_async_arrive(smem_addr(&ms.kv_full));
        if (g > 0 && !mbar_wait(smem_addr(&ms.kv_free[1]), ph, ab, p.err)) return;
        issue_rows<1, kShared>(p, ms, un, t, sKv, c.wt);
        cp_async_arrive(smem_addr(&ms.kv_full));
        if (g > 0 && !mbar_wait(smem_addr(&ms.kv_free[2]), ph, ab, p.err)) return;
        issue_rows<2, kShared>(p, ms, un, t, sKv, c.wt);
        cp_async_arrive(smem_addr(&ms.kv_full));
        // rows 96-111 (warps 0-3) are free one k-step before rows 112-127
        if (g > 0 && !mbar_wait(smem_addr(&ms.kv_free[c.w < 4 ? 3 : 4]), ph, ab, p.err)) return;
        issue_rows<3, kShared>(p, ms, un, t, sKv, c.wt);
        cp_async_arrive(smem_addr(&ms.kv_full));
        if (t == 0 && c.sinks) {
            // the unit starts from the sink references
#pragma unroll
            for (int h = 0; h < 32; ++h) mref[h] = sink_ref(p, 32 * c.hf + h);
            c.sink_mine = sink_ref(p, 32 * c.hf + c.lane);
        }
        const bool last_tile = t + 1 == un.tiles;
        const int u_next = last_tile ? unit_at(p, ms, nu + 1) : u;
        const bool more = u_next < p.units;
        // 3. scores of this tile
        if (!mbar_wait(smem_addr(&ms.s_full), g & 1, ab, p.err)) return;
        tc_fence_after();
        // 4. weights
        if (!softmax_tile(p, smem, ms, c, tmem, un, t, nu, lacc, mref, ninf)) return;
        ++g;
        if (!last_tile) {
            ++t;
            continue;
        }
        // 5. the unit is done: hand its per-head sums (reduced over this
        //    warp's 32 key lanes) and its maxima to the output warps
        if (nu > 0 && !mbar_wait(smem_addr(&ms.l_free), (nu - 1) & 1, ab, p.err)) return;
        ms.red_l[c.qd][32 * c.hf + c.lane] = warp_transpose_reduce32<false>(lacc, c.lane);
#pragma unroll
        for (int h = 0; h < 32; ++h) lacc[h] = 0.0f;
        __syncwarp();
        if (c.lane == 0) mbar_arrive(smem_addr(&ms.l_ready));
        ++nu;
        if (!more) break;
        u = u_next;
        t = 0;
    }
}

// ----------------------------------------------------------- index warp
// A spare warp walks the same tiles as the workers and copies the indices of
// tile g + 1 as soon as the scores of tile g are ready (by then every worker
// has issued tile g's gather, so idx[] is free).
__device__ void idx_role(const TcParams& p, Misc& ms, int lane) {
    volatile int* ab = &ms.abort_flag;
    // with a launch queue this warp takes the CTA's units, one unit ahead
    int u = p.queue ? take_unit(p, ms, 0, lane) : static_cast<int>(blockIdx.x);
    if (u >= p.units) return;
    int u_next = p.queue ? take_unit(p, ms, 1, lane) : u + static_cast<int>(gridDim.x);
    prefetch_idx(p, u, 0, ms, lane);
    Unit un = unit_info(p, u);
    int t = 0, g = 0, nu = 0;
    while (true) {
        int u2 = u, t2 = t + 1;
        if (t2 == un.tiles) {
            u2 = u_next;
            t2 = 0;
        }
        if (u2 >= p.units) break;
        if (!mbar_wait(smem_addr(&ms.s_full), g & 1, ab, p.err)) break;
        prefetch_idx(p, u2, t2, ms, lane);
        if (t2 == 0) {
            u = u2;
            ++nu;
            un = unit_info(p, u);
            u_next = p.queue ? take_unit(p, ms, nu + 1, lane) : u + static_cast<int>(gridDim.x);
        }
        t = t2;
        ++g;
    }
    cp_async_wait_all();    // its copies land before the CTA can exit
}

// ------------------------------------------------------------------ Q load
// One thread of a spare warp: loads each unit's Q by tiled TMA once the
// unit before has written P for its last tile, off the workers' path (a
// copy started as soon as the last score MMA is done ran beside that tile's
// softmax and slowed it).
__device__ void q_role(const TcParams& p, uint8_t* smem, Misc& ms) {
    volatile int* ab = &ms.abort_flag;
    const uint32_t sQ = smem_addr(smem + kOffQ);
    const uint32_t q_bytes = 8u * static_cast<uint32_t>(p.H) * 128u;
    const uint32_t bar = smem_addr(&ms.q_full);
    int nu = 0;
    for (;; ++nu) {
        const int u = unit_at(p, ms, nu);
        if (u >= p.units) break;
        if (nu > 0 && !mbar_wait(smem_addr(&ms.q_free), (nu - 1) & 1, ab, p.err)) break;
        mbar_arrive_expect_tx(bar, q_bytes);
        for (int s = 0; s < 8; ++s) tma_load_2d(sQ + s * kQSegBytes, &p.tmap_q, s * 64, (u / p.chunks) * p.H, bar);
    }
    if (nu > 0) {
        // the copies armed here have landed before the CTA can exit
        int dummy = 0;
        mbar_wait(bar, (nu - 1) & 1, &dummy, p.err);
    }
}

// ------------------------------------------------------------ output warps
// One warp per TMEM lane quadrant, running beside the workers' next unit:
// per-head factors of a finished unit (sink fold, or the partial's m and l),
// then O^T read back 16 heads at a time, scaled and stored.  The stores take
// about 4k cycles per unit (the SM writes ~32 bytes a clock); overlapped
// with the next unit's gather, scores and softmax they leave its chain.
__device__ void output_role(const TcParams& p, Misc& ms, uint32_t tmem, int qd, int lane) {
    volatile int* ab = &ms.abort_flag;
    const uint32_t lane_off = static_cast<uint32_t>(32 * qd) << 16;
    for (int nu = 0;; ++nu) {
        const int u = unit_at(p, ms, nu);
        if (u >= p.units) break;
        if (!mbar_wait(smem_addr(&ms.l_ready), nu & 1, ab, p.err)) return;
        float f[2];     // heads lane and lane + 32
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = lane + 32 * e;
            const float l = (ms.red_l[0][h] + ms.red_l[1][h]) + (ms.red_l[2][h] + ms.red_l[3][h]);
            const float m = ms.m_ref[h];
            f[e] = 1.0f;
            if (!p.partial) {
                const float mu = m == -INFINITY ? 0.0f : m;
                const float s2 = h < p.H ? __ldg(p.sink + h) * kLog2e : 0.0f;
                const float mstar = isfinite(s2) ? fmaxf(mu, s2) : mu;
                const float e1 = exp2f(mu - mstar);
                const float e2 = exp2f(s2 - mstar);
                f[e] = e1 / (l * e1 + e2);
            } else if (qd == 0) {
                float* ml = p.part + static_cast<size_t>(p.units) * kHeadsPad * kD +
                            static_cast<size_t>(u) * 2 * kHeadsPad;
                ml[h] = m;
                ml[kHeadsPad + h] = l;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ms.l_free));
        if (!mbar_wait(smem_addr(&ms.o_full), nu & 1, ab, p.err)) return;
        tc_fence_after();
        // fp32 (partials, or the final output) or bf16 (final output, rounded to nearest even)
        const size_t dst_off = p.partial ? static_cast<size_t>(u) * kHeadsPad * kD
                                         : static_cast<size_t>(u / p.chunks) * p.H * kD;
        float* dst = (p.partial ? p.part : static_cast<float*>(p.out)) + dst_off;
        __nv_bfloat16* dst16 = static_cast<__nv_bfloat16*>(p.out) + dst_off;
        const bool to_bf16 = !p.partial && p.out_bf16;
        const int d0 = 32 * qd + lane;
#pragma unroll 1
        for (int hg = 0; hg < 4; ++hg) {
            float fh[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) fh[j] = __shfl_sync(0xffffffffu, hg < 2 ? f[0] : f[1], 16 * (hg & 1) + j);
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                // chunks 0-2 keep the hi and lo halves 64 columns apart
                const uint32_t ta = tmem + lane_off + tmem_o(i) + 16 * hg;
                float o[16];
                tmem_ld16(ta, o);
                if (i < 3) {
                    float lo[16];
                    tmem_ld16(ta + 64, lo);
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] += lo[j];
                }
                const int d = i * 128 + d0;
                if (to_bf16) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int h = 16 * hg + j;
                        if (h < p.H) dst16[static_cast<size_t>(h) * kD + d] = __float2bfloat16_rn(o[j] * fh[j]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int h = 16 * hg + j;
                        if (h < p.H) dst[static_cast<size_t>(h) * kD + d] = o[j] * fh[j];
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ms.o_free));
    }
}

template <bool kShared>
__global__ void __launch_bounds__(kThreads, 1) dsa_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
    const int warp = threadIdx.x >> 5;
    grid_launch_dependents();        // the next grid in the stream may start its prologue
    if (smem_addr(smem) & 1023u) {   // the swizzle needs 1024-byte alignment
        grid_dependency_wait();
        if (threadIdx.x == 0) atomicOr(p.err, DSA_DEVERR_LAYOUT);
        return;
    }
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&ms.kv_full), 4 * kWorkers);   // one arrive per quarter tile and thread
        for (int i = 0; i < 5; ++i) mbar_init(smem_addr(&ms.kv_free[i]), 1);
        mbar_init(smem_addr(&ms.s_full), 1);
        mbar_init(smem_addr(&ms.p_full), kWorkerWarps);
        mbar_init(smem_addr(&ms.q_full), 1);
        mbar_init(smem_addr(&ms.q_free), 1);
        mbar_init(smem_addr(&ms.p_ack), 1);
        mbar_init(smem_addr(&ms.red_sync), kWorkerWarps);
        ms.ovf = 0;
        ms.seen[0] = ms.seen[1] = 0;
        for (int i = 0; i < 4; ++i) mbar_init(smem_addr(&ms.unit_full[i]), 1);
        ms.redo = 0;
        mbar_init(smem_addr(&ms.drain), 1);
        mbar_init(smem_addr(&ms.idx_full), 32);
        mbar_init(smem_addr(&ms.o_full), 1);
        mbar_init(smem_addr(&ms.o_free), kOutWarps);
        mbar_init(smem_addr(&ms.l_ready), kWorkerWarps);
        mbar_init(smem_addr(&ms.l_free), kOutWarps);
        for (int h = 0; h < 64; ++h) ms.m_ref[h] = -INFINITY;
        ms.abort_flag = 0;
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
    // everything above touched only shared memory and TMEM; the inputs and
    // outputs may belong to the grid before this one in the stream
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;

    if (warp < kWorkerWarps) {
        regs_inc<kRegsWorker>();
        worker_role<kShared>(p, smem, ms, tmem);
        cp_async_wait_all();
        __syncwarp();
    } else if (warp < kOutWarp0 + kOutWarps) {
        regs_dec<kRegsOther>();
        output_role(p, ms, tmem, warp & 3, threadIdx.x & 31);
        __syncwarp();
    } else {
        regs_dec<kRegsOther>();
        if (warp == kQWarp && (threadIdx.x & 31) == 0) q_role(p, smem, ms);
        if (warp == kIdxWarp) idx_role(p, ms, threadIdx.x & 31);
        // the whole warp tests the sinks, one thread issues
        const bool sinks = warp == kMmaWarp && sinks_finite(p, threadIdx.x & 31);
        if (warp == kMmaWarp && (threadIdx.x & 31) == 0) {
            mma_role(p, smem, ms, tmem, sinks);
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
    if (p.queue && threadIdx.x == 0) {
        // every CTA has taken its last ticket: the last one out (even after
        // an abort) leaves the queue at zero for the next launch
        __threadfence();
        if (atomicAdd(p.queue + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            atomicExch(p.queue, 0);
            atomicExch(p.queue + 1, 0);
        }
    }
}

}  // namespace

size_t tc_smem_bytes() { return kSmemBytes; }

namespace {

std::mutex g_launch_mu;    // guards the one-time set-up below

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    std::lock_guard<std::mutex> lock(g_launch_mu);
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
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_launch_mu);
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(dsa_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemBytes));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(dsa_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemBytes));
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    TcParams p = params;
    if (!encode_rows(&p.tmap_q, p.q, static_cast<uint64_t>(p.R) * p.H, static_cast<uint32_t>(p.H)))
        return cudaErrorInvalidValue;
    // programmatic serialisation: the kernel's prologue may overlap the tail
    // of the previous grid in the stream; it waits for that grid before it
    // reads or writes global memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return p.decode > 1 ? cudaLaunchKernelEx(&cfg, dsa_tc_kernel<true>, p)
                        : cudaLaunchKernelEx(&cfg, dsa_tc_kernel<false>, p);
}

}  // namespace dsa
