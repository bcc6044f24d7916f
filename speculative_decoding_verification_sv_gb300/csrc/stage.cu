// stage.cu -- device-initiated copies between device memory and pinned host
// memory (or within either).
//
// [SpecDec-Context-Scaling guide, sec. 7.1] puts the control plane of a verify
// round first: fewer synchronisations per round and no host-to-device token
// copies between the round's kernels.  Here the SMs themselves load and store
// across the host link, so a round's inputs come in, and its accepted tokens go
// out, as kernels in the round's own programmatic launch chain rather than as
// copy-engine operations between kernels (each of those measured ~8.5 us of
// node latency per round in a CUDA graph on GB300, for 589 KB in and 28 B out).
// On GB300 the host link is NVLink-C2C and coherent: once the kernel has
// completed (stream order or an event), the host reads the stored bytes with
// no further copy.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;   // 16-byte loads in flight per thread before its stores

__global__ void __launch_bounds__(kThreads) stage_copy_kernel(uint8_t* __restrict__ dst,
                                                              const uint8_t* __restrict__ src, size_t bytes,
                                                              int vec) {
    // the next kernel waits for this one to complete before it reads dst
    pdl_launch_dependents();
    pdl_wait();   // src may be the preceding kernel's output
    const size_t tid = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;
    const size_t nthreads = static_cast<size_t>(gridDim.x) * kThreads;
    size_t head = 0;
    if (vec) {
        const size_t n16 = bytes >> 4;
        const uint4* s = reinterpret_cast<const uint4*>(src);
        uint4* d = reinterpret_cast<uint4*>(dst);
        for (size_t base = tid; base < n16; base += nthreads * kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const size_t i = base + static_cast<size_t>(u) * nthreads;
                if (i < n16) v[u] = s[i];
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const size_t i = base + static_cast<size_t>(u) * nthreads;
                if (i < n16) d[i] = v[u];
            }
        }
        head = n16 << 4;
    }
    for (size_t i = head + tid; i < bytes; i += nthreads) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, cudaStream_t st) {
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
    const size_t items = vec ? (bytes >> 4) + (bytes & 15u) : bytes;
    // every item's load in flight at once where the SMs allow (the host link is
    // latency-bound at these sizes), at most two CTAs per SM
    size_t grid = (items + static_cast<size_t>(kThreads) * kUnroll - 1) / (static_cast<size_t>(kThreads) * kUnroll);
    const size_t cap = static_cast<size_t>(device_sm_count()) * 2;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch_pdl(stage_copy_kernel, dim3(static_cast<unsigned int>(grid)), dim3(kThreads), 0, st,
                      static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), bytes, vec ? 1 : 0);
}

}  // namespace sv
