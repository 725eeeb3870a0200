// Top-k sparse attention on the sm_103a tensor cores (bf16 inputs).
//
// What it computes: for one query row and all of its heads, the softmax over
// the row's selected latent KV rows plus one sink logit per head, weighted
// sum of the same rows (akol1 TensorFold PR #4, first commit message: score a
// tile of keys, keep a running maximum, a tile sum and a value sum;
// TensorFold PR #1206, "What changes": per-head sinks).
//
// How (one CTA per SM, persistent over work units; a unit is one row, or one
// key chunk of a row when a decode batch is split across SMs):
//
//   * producer warps 4-7 gather each 128-key tile of selected rows with
//     16-byte cp.async straight into a 128-byte-swizzled shared-memory tile
//     (8 segments of 128 keys x 64 columns).  The tile is read once from
//     global memory and serves every head, as keys and as values.
//   * MMA warp 8 (one thread) issues tcgen05.mma:
//       S^T[key][head]  = KV_tile (K-major, M=128) x Q^T (K-major, N=64)
//       O^T[col][head] += V^T     (MN-major, M=128 per 128 columns) x P^T
//     S^T lives in TMEM columns [0,128) (double buffer), O^T in [128,384).
//   * softmax warps 0-3 (one TMEM lane = one key per thread) take per-head
//     tile maxima and sums with warp-shuffle transpose reductions, keep a
//     per-head reference maximum that moves only when a tile's maximum
//     exceeds it by more than 2^8 (then O^T and the sum are rescaled), write
//     P as two bf16 terms (P = hi + lo) so the value sum keeps ~16 bits, and
//     finish with the sink fold and an fp32 store.
//
// Every wait is bounded (see dsa_ptx.cuh); on a timeout the kernel raises an
// error bit, lets its copies land, frees its TMEM and returns.
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 288;
constexpr int kMmaWarp = 8;
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
constexpr uint32_t kTmemO = 128;                   // O^T chunk i at 128 + 64 i

struct Misc {
    uint64_t seg_full[8];   // producers -> MMA: segment s of the tile landed
    uint64_t seg_free[4];   // MMA -> producers/softmax: P.V chunk i done
    uint64_t s_full;        // MMA -> softmax: scores of the tile ready
    uint64_t p_full;        // softmax -> MMA: P written (and O rescaled)
    uint64_t q_full;        // producers -> MMA: Q of the unit landed
    uint64_t q_free;        // MMA -> producers: last score MMA of the unit done
    uint64_t grp[3];        // softmax-group syncs
    uint64_t drain;         // MMA thread: everything it issued completed
    float red_max[4][64];
    float red_sum[4][64];
    float m_ref[64];        // per-head reference maximum (log2 units)
    float l_run[64];        // per-head running sum
    float alpha[64];        // per-head rescale factor; epilogue: output factor
    uint32_t tmem_base;
    int abort_flag;
    int rescale_flag;
};

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

__device__ __forceinline__ Unit unit_info(const TcParams& p, int u) {
    Unit x;
    x.r = u / p.chunks;
    x.c = u - x.r * p.chunks;
    const int ns = __ldg(p.n_sel + x.r);
    x.bad_n = (ns < 0 || ns > p.k_max);
    const int eff = x.bad_n ? 1 : ns;                 // bad row: one NaN key
    int nv = eff - x.c * p.chunk_keys;
    nv = nv < 0 ? 0 : (nv > p.chunk_keys ? p.chunk_keys : nv);
    x.n_valid = nv;
    x.tiles = nv == 0 ? 1 : (nv + 127) / 128;         // an empty unit runs one masked tile
    return x;
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

// Reduce 64 per-lane values over the 32 lanes of the warp.  Lane l ends with
// the results for heads 2l (.x) and 2l+1 (.y).  Fixed order: deterministic.
template <bool kMax>
__device__ __forceinline__ float2 warp_transpose_reduce(const float* x, int lane) {
    float v[32];
    {
        const bool up = (lane & 16) != 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float send = up ? x[i] : x[i + 32];
            const float keep = up ? x[i + 32] : x[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
    tr_step<32, 8, kMax>(v, lane);
    tr_step<16, 4, kMax>(v, lane);
    tr_step<8, 2, kMax>(v, lane);
    tr_step<4, 1, kMax>(v, lane);
    return make_float2(v[0], v[1]);
}

// ------------------------------------------------------------------ roles
__device__ void producer_role(const TcParams& p, uint8_t* smem, Misc& ms) {
    const int pt = threadIdx.x - 128;
    const int pw = pt >> 5, lane = pt & 31;
    const int cc = lane & 7;
    const uint32_t sKv = smem_addr(smem + kOffKv);
    const uint32_t sQ = smem_addr(smem + kOffQ);
    volatile int* ab = &ms.abort_flag;
    const uint16_t* nan_row = reinterpret_cast<const uint16_t*>(kNanRowBf16);
    int g = 0, nu = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++nu) {
        const Unit un = unit_info(p, u);
        if (un.bad_n && un.c == 0 && pt == 0) atomicOr(p.err, DSA_DEVERR_NSEL_RANGE);
        const uint16_t* cache = p.kv + (p.decode ? static_cast<size_t>(un.r) * p.N * kD : 0);

        // Q of this row: H rows x 64 chunks of 16 B, swizzled per 8 rows
        if (nu > 0 && !mbar_wait(smem_addr(&ms.q_free), (nu - 1) & 1, ab, p.err)) return;
        const uint16_t* qrow = p.q + static_cast<size_t>(un.r) * p.H * kD;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int h = j * 16 + pw * 4 + (lane >> 3);
            if (h < p.H) {
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    cp_async16(sQ + s * kQSegBytes + h * 128 + ((cc ^ (h & 7)) << 4),
                               qrow + static_cast<size_t>(h) * kD + s * 64 + cc * 8, 16);
            }
        }
        cp_async_arrive(smem_addr(&ms.q_full));

        for (int t = 0; t < un.tiles; ++t, ++g) {
            const uint16_t* src[8];
            uint32_t nb[8];
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                const int j = q8 * 16 + pw * 4 + (lane >> 3);
                const int key = t * 128 + j;
                src[q8] = nan_row;
                nb[q8] = 0;
                if (key < un.n_valid) {
                    nb[q8] = 16;
                    if (!un.bad_n) {
                        const int id = __ldg(p.idx + static_cast<size_t>(un.r) * p.k_max +
                                             un.c * p.chunk_keys + key);
                        if (id >= 0 && id < p.N) {
                            src[q8] = cache + static_cast<size_t>(id) * kD;
                        } else if (cc == 0) {
                            atomicOr(p.err, DSA_DEVERR_IDX_RANGE);
                        }
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                if ((s & 1) == 0 && g > 0 &&
                    !mbar_wait(smem_addr(&ms.seg_free[s >> 1]), (g - 1) & 1, ab, p.err))
                    return;
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) {
                    const int j = q8 * 16 + pw * 4 + (lane >> 3);
                    cp_async16(sKv + s * kSegBytes + j * 128 + ((cc ^ (j & 7)) << 4),
                               src[q8] + s * 64 + cc * 8, nb[q8]);
                }
                cp_async_arrive(smem_addr(&ms.seg_full[s]));
            }
        }
    }
}

__device__ void mma_role(const TcParams& p, uint8_t* smem, Misc& ms, uint32_t tmem) {
    const uint32_t sKv = smem_addr(smem + kOffKv);
    const uint32_t sQ = smem_addr(smem + kOffQ);
    const uint32_t sPhi = smem_addr(smem + kOffPhi);
    const uint32_t sPlo = smem_addr(smem + kOffPlo);
    volatile int* ab = &ms.abort_flag;
    constexpr uint32_t idS = idesc_bf16(128, 64, false, false);
    constexpr uint32_t idPV = idesc_bf16(128, 64, true, true);
    int g = 0, nu = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++nu) {
        const Unit un = unit_info(p, u);
        if (!mbar_wait(smem_addr(&ms.q_full), nu & 1, ab, p.err)) return;
        for (int t = 0; t < un.tiles; ++t, ++g) {
            // scores: S^T[key][head] over the 512 columns, 16 at a time
            const uint32_t dS = tmem + static_cast<uint32_t>(g & 1) * 64;
            for (int s = 0; s < 8; ++s) {
                if (!mbar_wait(smem_addr(&ms.seg_full[s]), g & 1, ab, p.err)) return;
                fence_proxy_async();
                tc_fence_after();
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) {
                    const uint64_t a = sdesc_sw128(sKv + s * kSegBytes + sub * 32, 16, 1024);
                    const uint64_t b = sdesc_sw128(sQ + s * kQSegBytes + sub * 32, 16, 1024);
                    umma_bf16(dS, a, b, idS, (s | sub) != 0);
                }
            }
            umma_commit(smem_addr(&ms.s_full));
            if (t == un.tiles - 1) umma_commit(smem_addr(&ms.q_free));

            // values: O^T[col][head] += V^T x (P_hi + P_lo)^T, 128 columns at a time
            if (!mbar_wait(smem_addr(&ms.p_full), g & 1, ab, p.err)) return;
            tc_fence_after();
            for (int i = 0; i < 4; ++i) {
                const uint32_t dO = tmem + kTmemO + i * 64;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t a = sdesc_sw128(sKv + 2 * i * kSegBytes + kk * 2048, kSegBytes, 1024);
                    // P^T holds one 64-head block along N, so its leading
                    // offset is never stepped; 1024 keeps it inside P either way
                    const uint64_t bh = sdesc_sw128(sPhi + kk * 2048, 1024, 1024);
                    const uint64_t bl = sdesc_sw128(sPlo + kk * 2048, 1024, 1024);
                    umma_bf16(dO, a, bh, idPV, (t > 0 || kk > 0) ? 1u : 0u);
                    umma_bf16(dO, a, bl, idPV, 1u);
                }
                umma_commit(smem_addr(&ms.seg_free[i]));
            }
        }
    }
}

__device__ void softmax_role(const TcParams& p, uint8_t* smem, Misc& ms, uint32_t tmem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int key_in_tile = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    volatile int* ab = &ms.abort_flag;
    uint32_t ph[3] = {0u, 0u, 0u};
    uint8_t* prow_hi = smem + kOffPhi + key_in_tile * 128;
    uint8_t* prow_lo = smem + kOffPlo + key_in_tile * 128;
    int g = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const Unit un = unit_info(p, u);
        for (int t = 0; t < un.tiles; ++t, ++g) {
            if (!mbar_wait(smem_addr(&ms.s_full), g & 1, ab, p.err)) return;
            tc_fence_after();
            float x[64];
            const uint32_t ts = tmem + lane_off + static_cast<uint32_t>(g & 1) * 64;
            tmem_ld32(ts, x);
            tmem_ld32(ts + 32, x + 32);
            const bool valid = t * 128 + key_in_tile < un.n_valid;
#pragma unroll
            for (int h = 0; h < 64; ++h) x[h] = valid ? x[h] * p.scale_log2 : -INFINITY;

            // per-head tile maximum -> new reference maximum (warp 0 owns the state)
            {
                const float2 mx = warp_transpose_reduce<true>(x, lane);
                *reinterpret_cast<float2*>(&ms.red_max[warp][2 * lane]) = mx;
            }
            if (!group_sync(smem_addr(&ms.grp[0]), ph[0], ab, p.err)) return;
            if (warp == 0) {
                bool resc = false;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = 2 * lane + e;
                    const float tm = fmaxf(fmaxf(ms.red_max[0][h], ms.red_max[1][h]),
                                           fmaxf(ms.red_max[2][h], ms.red_max[3][h]));
                    const float mo = (t == 0) ? -INFINITY : ms.m_ref[h];
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
                if (lane == 0) ms.rescale_flag = any ? 1 : 0;
            }
            if (!group_sync(smem_addr(&ms.grp[1]), ph[1], ab, p.err)) return;

            // weights relative to the reference maximum (0 when it is -inf)
#pragma unroll
            for (int h4 = 0; h4 < 16; ++h4) {
                const float4 m4 = *reinterpret_cast<const float4*>(&ms.m_ref[4 * h4]);
                const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mu = mm[e] == -INFINITY ? 0.0f : mm[e];
                    x[4 * h4 + e] = exp2f(x[4 * h4 + e] - mu);
                }
            }
            // P = hi + lo, both bf16, row = key, 64 heads, 128-byte swizzle
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = x[8 * c + 2 * e], b = x[8 * c + 2 * e + 1];
                    const __nv_bfloat162 hv = __floats2bfloat162_rn(a, b);
                    const float2 hf = __bfloat1622float2(hv);
                    const __nv_bfloat162 lv = __floats2bfloat162_rn(a - hf.x, b - hf.y);
                    hw[e] = *reinterpret_cast<const uint32_t*>(&hv);
                    lw[e] = *reinterpret_cast<const uint32_t*>(&lv);
                }
                const int pc = (c ^ (key_in_tile & 7)) << 4;
                *reinterpret_cast<uint4*>(prow_hi + pc) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(prow_lo + pc) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            fence_proxy_async();

            // a moved reference maximum rescales what P.V accumulated so far
            if (ms.rescale_flag) {
                if (!mbar_wait(smem_addr(&ms.seg_free[3]), (g - 1) & 1, ab, p.err)) return;
                tc_fence_after();
#pragma unroll 1
                for (int i = 0; i < 8; ++i) {
                    const uint32_t ta = tmem + lane_off + kTmemO + i * 32;
                    float o[32];
                    tmem_ld32(ta, o);
                    const float* al = &ms.alpha[(i & 1) * 32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= al[j];
                    tmem_st32(ta, o);
                }
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&ms.p_full));

            // per-head tile sums -> running sums
            {
                const float2 sm = warp_transpose_reduce<false>(x, lane);
                *reinterpret_cast<float2*>(&ms.red_sum[warp][2 * lane]) = sm;
            }
            if (!group_sync(smem_addr(&ms.grp[2]), ph[2], ab, p.err)) return;
            if (warp == 0) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = 2 * lane + e;
                    const float ls = (ms.red_sum[0][h] + ms.red_sum[1][h]) +
                                     (ms.red_sum[2][h] + ms.red_sum[3][h]);
                    ms.l_run[h] = (t == 0) ? ls : ms.l_run[h] * ms.alpha[h] + ls;
                }
            }
        }

        // epilogue: wait for the last P.V, fold the sink, store
        if (!mbar_wait(smem_addr(&ms.seg_free[3]), (g - 1) & 1, ab, p.err)) return;
        tc_fence_after();
        if (warp == 0) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = 2 * lane + e;
                float f = 1.0f;
                if (!p.partial) {
                    const float m = ms.m_ref[h];
                    const float mu = m == -INFINITY ? 0.0f : m;
                    const float s2 = h < p.H ? __ldg(p.sink + h) * kLog2e : 0.0f;
                    const float mstar = isfinite(s2) ? fmaxf(mu, s2) : mu;
                    const float e1 = exp2f(mu - mstar);
                    const float e2 = exp2f(s2 - mstar);
                    f = e1 / (ms.l_run[h] * e1 + e2);
                }
                ms.alpha[h] = f;
            }
            if (p.partial) {
                float* ml = p.part + static_cast<size_t>(p.units) * kHeadsPad * kD +
                            static_cast<size_t>(u) * 2 * kHeadsPad;
                ml[2 * lane] = ms.m_ref[2 * lane];
                ml[2 * lane + 1] = ms.m_ref[2 * lane + 1];
                ml[kHeadsPad + 2 * lane] = ms.l_run[2 * lane];
                ml[kHeadsPad + 2 * lane + 1] = ms.l_run[2 * lane + 1];
            }
        }
        if (!group_sync(smem_addr(&ms.grp[0]), ph[0], ab, p.err)) return;
        float f[64];
#pragma unroll
        for (int h4 = 0; h4 < 16; ++h4) {
            const float4 v = *reinterpret_cast<const float4*>(&ms.alpha[4 * h4]);
            f[4 * h4] = v.x;
            f[4 * h4 + 1] = v.y;
            f[4 * h4 + 2] = v.z;
            f[4 * h4 + 3] = v.w;
        }
        float* dst = p.partial ? p.part + static_cast<size_t>(u) * kHeadsPad * kD
                               : p.out + static_cast<size_t>(un.r) * p.H * kD;
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
            float o[64];
            const uint32_t ta = tmem + lane_off + kTmemO + i * 64;
            tmem_ld32(ta, o);
            tmem_ld32(ta + 32, o + 32);
            const int d = i * 128 + key_in_tile;
#pragma unroll
            for (int h = 0; h < 64; ++h)
                if (h < p.H) dst[static_cast<size_t>(h) * kD + d] = o[h] * f[h];
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) dsa_tc_kernel(const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
    const int warp = threadIdx.x >> 5;
    if (smem_addr(smem) & 1023u) {   // the swizzle needs 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(p.err, DSA_DEVERR_LAYOUT);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < 8; ++s) mbar_init(smem_addr(&ms.seg_full[s]), 128);
        for (int i = 0; i < 4; ++i) mbar_init(smem_addr(&ms.seg_free[i]), 1);
        mbar_init(smem_addr(&ms.s_full), 1);
        mbar_init(smem_addr(&ms.p_full), 128);
        mbar_init(smem_addr(&ms.q_full), 128);
        mbar_init(smem_addr(&ms.q_free), 1);
        for (int i = 0; i < 3; ++i) mbar_init(smem_addr(&ms.grp[i]), 128);
        mbar_init(smem_addr(&ms.drain), 1);
        ms.abort_flag = 0;
        ms.rescale_flag = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&ms.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp >= 4 && warp < 8 && p.H < 64) {
        // rows of Q beyond H stay zero for the whole launch
        const int pt = threadIdx.x - 128;
        for (int e = pt; e < (64 - p.H) * 64; e += 128) {
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

    if (warp < 4) {
        softmax_role(p, smem, ms, tmem);
    } else if (warp < 8) {
        producer_role(p, smem, ms);
        cp_async_wait_all();
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

cudaError_t launch_tc(const TcParams& p, int grid, cudaStream_t s) {
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
    dsa_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
