// Relaxed, lossy acceptance: the Delta-logit relaxation of "SpecDec-Context-
// Scaling project guide" sec. 7.2.  A draft passes when the target's top-1
// logit exceeds the draft token's logit by at most delta; the walk (the
// longest passing prefix of the chain, or from the root the first passing
// child in index order), the output token (the top-1 of the row the walk
// stops at: replacement or bonus) and the path are those of greedy
// acceptance (sec. 3).  The output no longer follows the target model
// exactly, so this is an entry point of its own beside the exact ones.
//
// Two launches: the row maxima and their lowest indices per vocab chunk
// (every row in parallel), then one CTA per sequence reduces them and walks.
// The gap is one float32 subtraction, fsub_rn(top1, logit[draft]), compared
// with delta; delta = 0 with a unique maximum is greedy acceptance.

#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kRelaxChunk = 8192;   // vocab columns per partial CTA
constexpr int kRelaxThreads = 256;
constexpr int kRelaxMaxR = 128;

struct Top {
    float v;
    int i;
};

// larger value, then lower index
__device__ __forceinline__ Top better(Top a, Top b) { return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a; }

__device__ __forceinline__ Top warp_best(Top a) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Top o;
        o.v = __shfl_xor_sync(0xffffffffu, a.v, off);
        o.i = __shfl_xor_sync(0xffffffffu, a.i, off);
        a = better(a, o);
    }
    return a;
}

// part[row][chunk] = (bits of the chunk's maximum, its lowest index); NaN
// entries are skipped and flagged.
__global__ void __launch_bounds__(kRelaxThreads) relaxed_partial_kernel(const float* __restrict__ logits, int V,
                                                                        int nchunk, int2* __restrict__ part,
                                                                        unsigned int* err) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    const int row = blockIdx.y;
    const int c0 = blockIdx.x * kRelaxChunk;
    const int c1 = min(c0 + kRelaxChunk, V);
    const float* L = logits + static_cast<size_t>(row) * V;
    Top best{-INFINITY, INT_MAX};
    bool bad = false;
    for (int i = c0 + threadIdx.x; i < c1; i += kRelaxThreads) {
        const float x = __ldg(L + i);
        if (x != x) {
            bad = true;
            continue;
        }
        best = better(best, Top{x, i});
    }
    if (bad) raise_error(err, SV_DEVERR_NONFINITE);
    best = warp_best(best);
    __shared__ Top red[kRelaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < kRelaxThreads / 32 ? red[lane] : Top{-INFINITY, INT_MAX};
        best = warp_best(best);
        if (lane == 0) part[static_cast<size_t>(row) * nchunk + blockIdx.x] = make_int2(__float_as_int(best.v), best.i);
    }
}

// One CTA per sequence: each row's top-1 (value and lowest index) from the
// partials, then the walk by thread 0.
__global__ void __launch_bounds__(128) relaxed_finish_kernel(const int2* __restrict__ part, int nchunk,
                                                             const float* __restrict__ logits,
                                                             const int32_t* __restrict__ tok,
                                                             const int32_t* __restrict__ parent, int R, int V,
                                                             float delta, int32_t* n_acc, int32_t* out_tok,
                                                             int32_t* path, unsigned int* err) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    __shared__ int top_i[kRelaxMaxR];
    __shared__ float top_v[kRelaxMaxR];
    __shared__ int par_s[kRelaxMaxR];
    __shared__ int tree_bad;
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < R; j += 4) {
        Top best{-INFINITY, INT_MAX};
        const int2* pr = part + (static_cast<size_t>(b) * R + j) * nchunk;
        for (int c = lane; c < nchunk; c += 32) {
            const int2 x = pr[c];
            best = better(best, Top{__int_as_float(x.x), x.y});
        }
        best = warp_best(best);
        if (lane == 0) {
            top_i[j] = best.i == INT_MAX ? 0 : best.i;
            top_v[j] = best.v;
        }
    }
    if (threadIdx.x == 0) tree_bad = 0;
    __syncthreads();
    if (parent) {
        for (int j = threadIdx.x; j < R; j += blockDim.x) {
            const int p = parent[static_cast<size_t>(b) * R + j];
            par_s[j] = p;
            if ((j == 0 && p != -1) || (j > 0 && (p < 0 || p >= j))) tree_bad = 1;
        }
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    const bool tree_ok = tree_bad == 0;
    if (!tree_ok) raise_error(err, SV_DEVERR_TREE);
    const int32_t* tk = tok + static_cast<size_t>(b) * R;
    const float* L = logits + static_cast<size_t>(b) * R * V;
    int32_t* pth = path + static_cast<size_t>(b) * R;
    for (int j = 1; j < R; ++j)
        if (tk[j] < 0 || tk[j] >= V) raise_error(err, SV_DEVERR_TOKEN);
    int u = 0, depth = 0;
    pth[0] = 0;
    if (tree_ok) {
        for (int guard = 0; guard < R; ++guard) {
            int next = -1;
            for (int c = u + 1; c < R; ++c) {
                const bool child = parent ? par_s[c] == u : c == u + 1;
                if (!child) continue;
                const int d = tk[c];
                if (d < 0 || d >= V) continue;
                const float gap = __fsub_rn(top_v[u], __ldg(L + static_cast<size_t>(u) * V + d));
                if (gap <= delta) {
                    next = c;
                    break;
                }
            }
            if (next < 0) break;
            u = next;
            pth[++depth] = u;
        }
    }
    for (int j = depth + 1; j < R; ++j) pth[j] = -1;
    n_acc[b] = depth;
    out_tok[b] = top_i[u];
}

}  // namespace

size_t relaxed_workspace(int B, int R, int V) {
    const int nchunk = (V + kRelaxChunk - 1) / kRelaxChunk;
    return static_cast<size_t>(B) * R * nchunk * sizeof(int2);
}

cudaError_t launch_accept_relaxed(const float* logits, const int32_t* tok, const int32_t* parent, int B, int R, int V,
                                  float delta, int32_t* n_acc, int32_t* out_tok, int32_t* path, void* ws,
                                  cudaStream_t st) {
    const int nchunk = (V + kRelaxChunk - 1) / kRelaxChunk;
    int2* part = static_cast<int2*>(ws);
    unsigned int* err = device_error_word();
    cudaError_t e = launch_pdl(relaxed_partial_kernel, dim3(nchunk, B * R), dim3(kRelaxThreads), 0, st, logits, V,
                               nchunk, part, err);
    if (e != cudaSuccess) return e;
    e = launch_pdl(relaxed_finish_kernel, dim3(B), dim3(128), 0, st, static_cast<const int2*>(part), nchunk, logits,
                   tok, parent, R, V, delta, n_acc, out_tok, path, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sv
