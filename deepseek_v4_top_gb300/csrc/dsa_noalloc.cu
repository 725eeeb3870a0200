// Decode entry point for callers that must not allocate device memory.
//
// dsa_sparse_attn_decode() allocates its error word and its split-partial
// scratch with cudaMalloc the first time a device needs them (and grows the
// scratch for larger batches).  Some callers cannot allow that: engines that
// reserve all device memory when they start and forbid allocation afterwards,
// and callers on a latency-critical path where cudaMalloc / cudaFree would
// synchronise the device.  This file gives them dsa_sparse_attn_decode_noalloc(),
// which runs the same bf16 split kernel and combine kernel, with the same key
// chunking, but keeps the partials and the error word in one fixed-size
// static __device__ array instead.
//
// Host code must not pass g_noalloc_scratch itself to a kernel: in host code
// that name is only a host-side stand-in for the device symbol.  The device
// address comes from cudaGetSymbolAddress(), once per device, on that
// device's first call.
#include <stdint.h>

#include <mutex>

#include <cuda_runtime.h>

#include "../../include/dsa.h"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kNoAllocMaxDevices = 64;
constexpr size_t kHeaderFloats = 64;   // 256 bytes; the first word is the error word

// Every GPU that loads the library holds this array until the process exits:
// 256 bytes of header plus DSA_NOALLOC_MAX_UNITS chunk partials (8,421,632 bytes).
static __device__ __align__(256) float
    g_noalloc_scratch[kHeaderFloats + static_cast<size_t>(DSA_NOALLOC_MAX_UNITS) * kPartialFloats];

struct NoAllocDevice {
    float* base = nullptr;     // device address of g_noalloc_scratch
    int sm_count = 0;
};

std::mutex g_na_mu;
NoAllocDevice g_na[kNoAllocMaxDevices];

// Resolves the array's device address (and the SM count) for the current
// device.  Runs once per device; allocates nothing.
dsa_status noalloc_setup(NoAllocDevice** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_UNSUPPORTED;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return DSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_na_mu);
    NoAllocDevice& d = g_na[dev];
    if (!d.base) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DSA_ERR_CUDA;
        if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED;
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return DSA_ERR_CUDA;
        d.base = static_cast<float*>(ptr);
        d.sm_count = sms;
    }
    *out = &d;
    return DSA_OK;
}

}  // namespace

void noalloc_forget() {
    std::lock_guard<std::mutex> lock(g_na_mu);
    for (int d = 0; d < kNoAllocMaxDevices; ++d) g_na[d] = NoAllocDevice();
}

}  // namespace dsa

extern "C" dsa_status dsa_sparse_attn_decode_noalloc(const void* q, const void* kv_cache,
                                                     const int32_t* idx, const int32_t* n_sel,
                                                     const float* sink, float scale, float* out,
                                                     int B, int H, int N, int k_max, dsa_dtype dtype,
                                                     void* stream) {
    using namespace dsa;
    if (B < 0 || N <= 0 || k_max <= 0 || H <= 0) return DSA_ERR_INVALID_ARG;
    if (dtype != DSA_BF16 || H > kHeadsPad) return DSA_ERR_UNSUPPORTED;
    if (B == 0) return DSA_OK;
    if (!q || !kv_cache || !idx || !n_sel || !sink || !out) return DSA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_cache) |
         reinterpret_cast<uintptr_t>(out)) & 15u)
        return DSA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * N >= (1LL << 31)) return DSA_ERR_INVALID_ARG;
    const long long chunks = (static_cast<long long>(k_max) + kDecodeChunkKeys - 1) / kDecodeChunkKeys;
    if (static_cast<long long>(B) * chunks > DSA_NOALLOC_MAX_UNITS) return DSA_ERR_UNSUPPORTED;

    NoAllocDevice* d = nullptr;
    dsa_status st = noalloc_setup(&d);
    if (st != DSA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // The error word accumulates bits with atomicOr, so it starts each call at
    // zero.  Every partial the combine kernel reads is written earlier in the
    // same call, so nothing else needs clearing.
    uint32_t* err = reinterpret_cast<uint32_t*>(d->base);
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return DSA_ERR_CUDA;

    TcParams p;
    p.q = static_cast<const uint16_t*>(q);
    p.kv = static_cast<const uint16_t*>(kv_cache);
    p.idx = idx;
    p.n_sel = n_sel;
    p.sink = sink;
    p.out = out;
    p.out_bf16 = 0;
    p.part = d->base + kHeaderFloats;
    p.err = err;
    p.queue = nullptr;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.R = B;
    p.H = H;
    p.N = N;
    p.k_max = k_max;
    p.decode = 1;
    p.chunks = static_cast<int>(chunks);
    p.chunk_keys = chunks > 1 ? kDecodeChunkKeys : k_max;
    p.units = B * p.chunks;
    p.partial = chunks > 1 ? 1 : 0;
    const int grid = p.units < d->sm_count ? p.units : d->sm_count;
    if (launch_tc(p, grid, s) != cudaSuccess) return DSA_ERR_CUDA;
    if (p.partial) {
        CombineParams c;
        c.part = p.part;
        c.sink = sink;
        c.out = out;
        c.out_bf16 = 0;
        c.R = B;
        c.H = H;
        c.chunks = p.chunks;
        c.units = p.units;
        if (launch_combine(c, s) != cudaSuccess) return DSA_ERR_CUDA;
    }
    return DSA_OK;
}
