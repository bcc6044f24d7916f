// accept_noalloc.cu -- sv_accept_sample_noalloc: the sampled acceptance for
// callers that cannot allocate device memory.
//
// Some callers only ever hold the buffers they were handed: a plugin invoked
// by a host framework that owns all device memory and exposes no allocator,
// or a latency-critical loop that must not call cudaMalloc (or any routine
// that allocates) while it runs.  For them this entry point takes the same
// inputs and outputs as sv_accept_sample but no workspace: its scratch (one
// float2 of row statistics per verify row) lives in the fixed device array
// below, so the library itself allocates nothing either.
//
// Properties of the fixed array (documented in include/sv.h as well):
//   * it is kNoAllocMaxRows float2 (64 KiB) and every GPU that loads the
//     library keeps it until the process exits;
//   * calls with B*R above kNoAllocMaxRows are rejected with SV_ERR_SHAPE;
//   * all calls on a device share it and it keeps the last call's contents;
//     nothing in it needs to start at zero (every row is written before it is
//     read), but two calls that overlap on the GPU (different streams, no
//     ordering between them) race on it;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress with that device current) and caches it; that
//     first call should come before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "sv.h"
#include "sv_internal.h"

namespace {

constexpr int kNoAllocMaxRows = 8192;
using sv::kMaxDevices;

static __device__ __align__(256) float2 g_noalloc_stats[kNoAllocMaxRows];

sv::PerDeviceOnce g_noalloc_once;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_stats on the current device, looked up once per
// device and again if the device's context has been replaced (after
// cudaDeviceReset the module is loaded anew and the array may move); nullptr
// if the lookup fails.
void* noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const cudaError_t e = g_noalloc_once.run([dev]() {
        void* p = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&p, g_noalloc_stats);
        g_noalloc_addr[dev] = r == cudaSuccess ? p : nullptr;
        return r;
    });
    return e == cudaSuccess ? g_noalloc_addr[dev] : nullptr;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" sv_status sv_accept_sample_noalloc(const float* logits, const float* q, int32_t Vq, const int32_t* tok,
                                              const int32_t* parent, int32_t B, int32_t R, int32_t V,
                                              float temperature, uint64_t seed, uint64_t step,
                                              const float* uniforms, int32_t* n_acc, int32_t* out_tok,
                                              int32_t* path, void* stream) {
    if (!logits || !tok || !n_acc || !out_tok || !path) return SV_ERR_ARG;
    if (R > 1 || parent) {
        if (!q || !aligned16(q)) return SV_ERR_ARG;
    }
    if (!aligned16(logits)) return SV_ERR_ARG;
    if (!(temperature > 0.0f) || !(temperature < 1e30f)) return SV_ERR_ARG;
    if (B < 1 || R < 1 || R > 128 || V < 4 || V > (1 << 18) || V % 4) return SV_ERR_SHAPE;
    if (Vq < 4 || Vq > V || Vq % 4) return SV_ERR_SHAPE;
    if (static_cast<int64_t>(B) * R > kNoAllocMaxRows) return SV_ERR_SHAPE;
    void* scratch = noalloc_scratch();
    if (!scratch) return SV_ERR_CUDA;
    // Only the statistics' bytes are offered, so chains and trees alike take
    // the one-cluster-per-sequence walk, which needs no other scratch.
    const size_t stats = (static_cast<size_t>(B) * R * sizeof(float2) + 255) / 256 * 256;
    const cudaError_t e = sv::launch_accept_sample(logits, q, Vq, tok, parent, B, R, V, temperature, seed, step,
                                                   uniforms, n_acc, out_tok, path, scratch, stats,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
