// C ABI of the top-k sparse-attention library: argument checks, launch
// planning and the small per-device state (error word, decode scratch).
#include <math.h>
#include <stdint.h>

#include <mutex>

#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kMaxDevices = 64;
// Prefill launches with more rows than CTAs hand rows out from a queue in
// device memory (two ints); each stream gets its own, up to this many a device.
constexpr int kQueues = 64;

struct DeviceState {
    uint32_t* err = nullptr;       // error word, followed by the stream queues
    float* scratch = nullptr;
    size_t scratch_bytes = 0;
    void* topk_scratch = nullptr;  // two-step top-k: the shares' picks
    size_t topk_scratch_bytes = 0;
    int sm_count = 0;
    cudaStream_t queue_stream[kQueues] = {};
    int queues_used = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Lazily creates the current device's error word.
dsa_status device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_UNSUPPORTED;
    if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.err) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DSA_ERR_CUDA;
        if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED;   // built for sm_103a only
        uint32_t* e = nullptr;
        const size_t bytes = (4 + 2 * kQueues) * sizeof(uint32_t);
        if (cudaMalloc(&e, bytes) != cudaSuccess) return DSA_ERR_CUDA;
        // zeroed on the legacy stream: wait, so that a non-blocking stream
        // never sees the block before the memset ran
        if (cudaMemset(e, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
            cudaFree(e);
            return DSA_ERR_CUDA;
        }
        st.err = e;
        st.sm_count = sms;
    }
    *out = &st;
    return DSA_OK;
}

// Grows a scratch buffer to `bytes` and returns it (under the lock, so a
// concurrent grow cannot free it between the check and the use).
dsa_status ensure_buffer(void** buf, size_t* have, size_t bytes, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (*have >= bytes) {
        *out = *buf;
        return DSA_OK;
    }
    if (*buf) {
        // the old buffer may still be read by queued work
        if (cudaDeviceSynchronize() != cudaSuccess) return DSA_ERR_CUDA;
        cudaFree(*buf);
        *buf = nullptr;
        *have = 0;
    }
    if (cudaMalloc(buf, bytes) != cudaSuccess) return DSA_ERR_CUDA;
    *have = bytes;
    *out = *buf;
    return DSA_OK;
}

// The decode scratch.
dsa_status ensure_scratch(DeviceState* st, size_t bytes, float** out) {
    void* v = nullptr;
    const dsa_status r = ensure_buffer(reinterpret_cast<void**>(&st->scratch), &st->scratch_bytes, bytes, &v);
    *out = static_cast<float*>(v);
    return r;
}

// The row queue of stream s, or null (round-robin rows) when s may run on
// several threads' behalf at once (the per-thread default stream), while s
// is being captured into a graph (a replay could overlap other work that
// uses the same queue), or when every queue is taken.  Calls on one stream
// run in order, so they never use a queue at the same time.
int* stream_queue(DeviceState* st, cudaStream_t s) {
    if (s == cudaStreamPerThread) return nullptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    int slot = -1;
    for (int i = 0; i < st->queues_used; ++i)
        if (st->queue_stream[i] == s) slot = i;
    if (slot < 0) {
        if (st->queues_used == kQueues) return nullptr;
        slot = st->queues_used++;
        st->queue_stream[slot] = s;
    }
    return reinterpret_cast<int*>(st->err) + 4 + 2 * slot;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dsa_status check_args(const void* q, const void* kv, const int32_t* idx, const int32_t* n_sel,
                      const float* sink, const void* out, int R, int H, int N, int k_max,
                      dsa_dtype dtype, int decode) {
    if (R < 0 || N <= 0 || k_max <= 0 || H <= 0) return DSA_ERR_INVALID_ARG;
    if (dtype != DSA_F32 && dtype != DSA_BF16) return DSA_ERR_UNSUPPORTED;
    if (H > kHeadsPad) return DSA_ERR_UNSUPPORTED;   // heads are padded to 64 on chip
    if (R == 0) return DSA_OK;
    if (!q || !kv || !idx || !n_sel || !sink || !out) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
    // 32-bit unit counts and grid limits
    if (static_cast<long long>(R) * ((k_max + kDecodeChunkKeys - 1) / kDecodeChunkKeys) > (1LL << 30))
        return DSA_ERR_INVALID_ARG;
    if (dtype == DSA_F32 && R > 65535) return DSA_ERR_UNSUPPORTED;
    // the TMA map of q counts its rows (R * H) in int32; a decode batch's
    // cache holds R / T slots of N rows (decode = T rows a slot)
    if ((decode && static_cast<long long>(R / decode) * N >= (1LL << 31)) ||
        static_cast<long long>(R) * H >= (1LL << 31))
        return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

// decode: 0 for prefill (one cache shared by every row), T >= 1 for decode
// with T query rows a slot (row r reads slot r / T).  split: a decode row's
// keys run as 128-key chunks on several SMs and are merged; otherwise each
// row runs whole in one CTA, as a prefill row does.
dsa_status run(const void* q, const void* kv, const int32_t* idx, const int32_t* n_sel,
               const float* sink, float scale, void* out, int R, int H, int N, int k_max,
               dsa_dtype dtype, void* stream, int decode, dsa_dtype out_dtype = DSA_F32,
               bool split = true) {
    if (out_dtype != DSA_F32 && out_dtype != DSA_BF16) return DSA_ERR_UNSUPPORTED;
    dsa_status st = check_args(q, kv, idx, n_sel, sink, out, R, H, N, k_max, dtype, decode);
    if (st != DSA_OK || R == 0) return st;
    const int out_bf16 = out_dtype == DSA_BF16 ? 1 : 0;
    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != DSA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (dtype == DSA_F32) {
        SimtParams p;
        p.q = static_cast<const float*>(q);
        p.kv = static_cast<const float*>(kv);
        p.idx = idx;
        p.n_sel = n_sel;
        p.sink = sink;
        p.out = out;
        p.out_bf16 = out_bf16;
        p.err = ds->err;
        p.scale = scale;
        p.R = R;
        p.H = H;
        p.N = N;
        p.k_max = k_max;
        p.decode = decode;
        return launch_simt(p, s) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
    }

    TcParams p;
    p.q = static_cast<const uint16_t*>(q);
    p.kv = static_cast<const uint16_t*>(kv);
    p.idx = idx;
    p.n_sel = n_sel;
    p.sink = sink;
    p.out = out;
    p.out_bf16 = out_bf16;
    p.part = nullptr;
    p.err = ds->err;
    p.queue = nullptr;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.R = R;
    p.H = H;
    p.N = N;
    p.k_max = k_max;
    p.decode = decode;
    const int chunks = decode && split ? (k_max + kDecodeChunkKeys - 1) / kDecodeChunkKeys : 1;
    p.chunk_keys = chunks > 1 ? kDecodeChunkKeys : k_max;
    p.chunks = chunks;
    p.units = R * chunks;
    p.partial = chunks > 1 ? 1 : 0;
    if (p.partial) {
        const size_t bytes =
            static_cast<size_t>(p.units) * kPartialFloats * sizeof(float);
        st = ensure_scratch(ds, bytes, &p.part);
        if (st != DSA_OK) return st;
    }
    const int grid = p.units < ds->sm_count ? p.units : ds->sm_count;
    // rows of unequal speed (SMs differ by a few percent) balance through a
    // queue when there are more of them than CTAs
    if (!p.partial && p.units > grid) p.queue = stream_queue(ds, s);
    if (launch_tc(p, grid, s) != cudaSuccess) return DSA_ERR_CUDA;
    if (p.partial) {
        CombineParams c;
        c.part = p.part;
        c.sink = sink;
        c.out = out;
        c.out_bf16 = out_bf16;
        c.R = R;
        c.H = H;
        c.chunks = chunks;
        c.units = p.units;
        if (launch_combine(c, s) != cudaSuccess) return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" {

dsa_status dsa_sparse_attn_decode(const void* q, const void* kv_cache, const int32_t* idx,
                                  const int32_t* n_sel, const float* sink, float scale, float* out,
                                  int B, int H, int N, int k_max, dsa_dtype dtype, void* stream) {
    return dsa::run(q, kv_cache, idx, n_sel, sink, scale, out, B, H, N, k_max, dtype, stream, 1);
}

dsa_status dsa_sparse_attn_decode_rows(const void* q, const void* kv_cache, const int32_t* idx,
                                       const int32_t* n_sel, const float* sink, float scale, float* out,
                                       int B, int T, int H, int N, int k_max, dsa_dtype dtype,
                                       void* stream) {
    if (B < 0 || T < 1 || static_cast<long long>(B) * T > 0x7FFFFFFFLL) return DSA_ERR_INVALID_ARG;
    return dsa::run(q, kv_cache, idx, n_sel, sink, scale, out, B * T, H, N, k_max, dtype, stream, T);
}

dsa_status dsa_sparse_attn_prefill(const void* q, const void* kv_cache, const int32_t* idx,
                                   const int32_t* n_sel, const float* sink, float scale, float* out,
                                   int R, int H, int N, int k_max, dsa_dtype dtype, void* stream) {
    return dsa::run(q, kv_cache, idx, n_sel, sink, scale, out, R, H, N, k_max, dtype, stream, 0);
}

dsa_status dsa_sparse_attn(const void* q, const void* kv_cache, const int32_t* idx, const int32_t* n_sel,
                           const float* sink, float scale, void* out, int R, int rows_per_slot, int H,
                           int N, int k_max, dsa_dtype dtype, dsa_dtype out_dtype, void* stream) {
    if (R < 0 || rows_per_slot < 0 || (rows_per_slot > 0 && R % rows_per_slot != 0)) return DSA_ERR_INVALID_ARG;
    return dsa::run(q, kv_cache, idx, n_sel, sink, scale, out, R, H, N, k_max, dtype, stream, rows_per_slot,
                    out_dtype);
}

dsa_status dsa_sparse_attn_decode_whole_rows(const void* q, const void* kv_cache, const int32_t* idx,
                                             const int32_t* n_sel, const float* sink, float scale, void* out,
                                             int R, int rows_per_slot, int H, int N, int k_max, dsa_dtype dtype,
                                             dsa_dtype out_dtype, void* stream) {
    if (R < 0 || rows_per_slot < 1 || R % rows_per_slot != 0) return DSA_ERR_INVALID_ARG;
    return dsa::run(q, kv_cache, idx, n_sel, sink, scale, out, R, H, N, k_max, dtype, stream, rows_per_slot,
                    out_dtype, false);
}

dsa_status dsa_oproj(const void* attn, const void* w_o, float* out, int R, int K, int d_out, void* stream) {
    if (R < 0 || K <= 0 || d_out <= 0) return DSA_ERR_INVALID_ARG;
    if (R == 0) return DSA_OK;
    if (!attn || !w_o || !out) return DSA_ERR_INVALID_ARG;
    if (!dsa::aligned16(attn) || !dsa::aligned16(w_o) || !dsa::aligned16(out) || K % 8 != 0 || d_out % 8 != 0)
        return DSA_ERR_INVALID_ARG;
    dsa::DeviceState* ds = nullptr;
    dsa_status st = dsa::device_state(&ds);
    if (st != DSA_OK) return st;
    return dsa::launch_gemm(attn, w_o, out, R, K, d_out, ds->err, ds->sm_count, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? DSA_OK
               : DSA_ERR_CUDA;
}

dsa_status dsa_sparse_attn_prefill_oproj(const void* q, const void* kv_cache, const int32_t* idx,
                                         const int32_t* n_sel, const float* sink, float scale,
                                         const void* w_o, void* attn, float* out, int R, int H, int N,
                                         int k_max, int d_out, void* stream) {
    if (R < 0 || H <= 0 || d_out <= 0) return DSA_ERR_INVALID_ARG;
    if (R == 0) return DSA_OK;
    if (!w_o || !attn || !out) return DSA_ERR_INVALID_ARG;
    if (!dsa::aligned16(w_o) || !dsa::aligned16(out) || d_out % 8 != 0) return DSA_ERR_INVALID_ARG;
    dsa_status st = dsa::run(q, kv_cache, idx, n_sel, sink, scale, attn, R, H, N, k_max, DSA_BF16, stream, 0,
                             DSA_BF16);
    if (st != DSA_OK) return st;
    return dsa_oproj(attn, w_o, out, R, H * dsa::kD, d_out, stream);
}

dsa_status dsa_topk_select(const float* scores, int ld, const int32_t* n_valid, int R, int k,
                           int32_t* idx, int k_max, int32_t* n_sel, void* stream) {
    if (R < 0 || k < 1 || k_max < k || ld < 1 || (ld & 3) != 0) return DSA_ERR_INVALID_ARG;
    if (k > dsa::kTopkMaxK || ld > dsa::kTopkMaxLd) return DSA_ERR_UNSUPPORTED;
    if (R == 0) return DSA_OK;
    if (!scores || !n_valid || !idx || !n_sel) return DSA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(scores) & 15u) != 0) return DSA_ERR_INVALID_ARG;
    dsa::DeviceState* ds = nullptr;
    dsa_status st = dsa::device_state(&ds);
    if (st != DSA_OK) return st;
    dsa::TopkParams p;
    p.scores = scores;
    p.n_valid = n_valid;
    p.idx = idx;
    p.n_sel = n_sel;
    p.err = ds->err;
    p.R = R;
    p.ld = ld;
    p.k = k;
    p.k_max = k_max;
    p.shares = dsa::topk_shares(ld);
    p.cand_ld = (p.shares * k + 3) & ~3;
    p.cand_key = nullptr;
    p.cand_pos = nullptr;
    // long rows go in two steps through a scratch of at most 256 MB: as many
    // rows at a time as fit
    int rows = R;
    if (p.shares > 1) {
        const size_t row_bytes = static_cast<size_t>(p.cand_ld) * 8;
        const size_t fit = (static_cast<size_t>(256) << 20) / row_bytes;
        rows = fit < static_cast<size_t>(R) ? static_cast<int>(fit) : R;
        rows = rows < (1 << 24) ? rows : (1 << 24);      // (rows x shares stays an int)
        const size_t per = static_cast<size_t>(rows) * static_cast<size_t>(p.cand_ld);
        void* buf = nullptr;
        st = dsa::ensure_buffer(&ds->topk_scratch, &ds->topk_scratch_bytes, per * 8, &buf);
        if (st != DSA_OK) return st;
        p.cand_key = static_cast<uint32_t*>(buf);
        p.cand_pos = reinterpret_cast<int32_t*>(p.cand_key + per);
    }
    for (int r0 = 0; r0 < R; r0 += rows) {
        dsa::TopkParams q = p;
        q.R = R - r0 < rows ? R - r0 : rows;
        q.scores = scores + static_cast<size_t>(r0) * ld;
        q.n_valid = n_valid + r0;
        q.idx = idx + static_cast<size_t>(r0) * k_max;
        q.n_sel = n_sel + r0;
        const int grid = q.R < (1 << 20) ? q.R : (1 << 20);
        if (dsa::launch_topk(q, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

dsa_status dsa_selftest_wait_limit(void* stream) {
    dsa::DeviceState* ds = nullptr;
    dsa_status st = dsa::device_state(&ds);
    if (st != DSA_OK) return st;
    return dsa::launch_wait_selftest(ds->err, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DSA_OK
                                                                                            : DSA_ERR_CUDA;
}

dsa_status dsa_get_device_error(void* stream, uint32_t* code) {
    if (!code) return DSA_ERR_INVALID_ARG;
    dsa::DeviceState* ds = nullptr;
    dsa_status st = dsa::device_state(&ds);
    if (st != DSA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, ds->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return DSA_ERR_CUDA;
    if (cudaMemset(ds->err, 0, sizeof v) != cudaSuccess) return DSA_ERR_CUDA;
    *code = v;
    return DSA_OK;
}

const char* dsa_status_string(dsa_status status) {
    switch (status) {
        case DSA_OK: return "DSA_OK";
        case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
        case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
        case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
        case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
    }
    return "DSA_UNKNOWN_STATUS";
}

dsa_status dsa_shutdown(void) {
    std::lock_guard<std::mutex> lock(dsa::g_mu);
    int cur = 0;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    dsa_status st = DSA_OK;
    for (int d = 0; d < dsa::kMaxDevices; ++d) {
        dsa::DeviceState& ds = dsa::g_dev[d];
        if (!ds.err && !ds.scratch && !ds.topk_scratch) continue;
        if (cudaSetDevice(d) != cudaSuccess) {
            st = DSA_ERR_CUDA;
            continue;
        }
        if (ds.err) cudaFree(ds.err);
        if (ds.scratch) cudaFree(ds.scratch);
        if (ds.topk_scratch) cudaFree(ds.topk_scratch);
        ds = dsa::DeviceState();
    }
    if (have_cur) cudaSetDevice(cur);
    dsa::noalloc_forget();
    return st;
}

}  // extern "C"
