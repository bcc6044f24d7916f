// kv_commit.cu -- commit of the accepted verify rows into the KV cache.
//
// [SpecDec-Context-Scaling guide, sec. 3.2]: the cache length must equal the
// number of committed tokens; after m accepted drafts the pending token, the
// m drafts and nothing else are in the cache, whose length becomes t+m+1.
// [mini-infer Phase 11, hidden KV position bug and "v2"]: the committed
// tokens' KV comes from the verify forward itself (no second forward).
// [SubSpec summary, sec. 4.2]: for a token tree the accepted root-to-node
// path is compacted into consecutive slots t..t+m.
//
// One 8-CTA cluster per sequence: every CTA reads len[b] and stages the path,
// copies its share of the layers' accepted rows with 16-byte vector moves
// (eight in flight per thread), and after
// a cluster barrier (all reads of len[b] done) rank 0 advances len[b].  The
// block rows live in a separate staging buffer, so rejected rows never enter
// the cache and nothing has to be rolled back.
//
// Paged caches ([mini-infer Phase 11], implementation architecture: the KV
// lives in a block tensor addressed through each request's block table):
// position p of sequence b is row p % 64 of page pages[b][p / 64] of every
// layer's pool; the pages of the rows to write are staged and checked first.
#include <cooperative_groups.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kCluster = 8;
constexpr int kThreads = 256;
constexpr int kMaxR = 128;         // block rows (the ABI's bound)
constexpr int kPage = 64;          // positions per page of a paged cache

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    kv_commit_kernel(uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache,
                     const uint16_t* __restrict__ k_blk, const uint16_t* __restrict__ v_blk, int L, int B, int Hkv,
                     int D, int T_cap, int R, const int32_t* __restrict__ path, const int32_t* __restrict__ n_acc,
                     int32_t* len, const int32_t* __restrict__ pages, int max_pages, int num_pages,
                     unsigned int* err) {
    pdl_wait();   // path, n_acc and the block rows come from the kernels before this one
    pdl_launch_dependents();
    __shared__ int path_s[kMaxR];
    __shared__ int page_s[kMaxR];   // paged: the page of slot t + i
    __shared__ int ok_s, page_ok_s;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.x / kCluster;
    const int t = len[b];
    const int m = n_acc[b];
    const bool shape_ok = t >= 0 && m >= 0 && m < R && t + m + 1 <= T_cap;
    const int32_t* pb = path + static_cast<size_t>(b) * R;
    if (threadIdx.x == 0) {
        ok_s = shape_ok ? 1 : 0;
        page_ok_s = 1;
    }
    __syncthreads();
    if (shape_ok && threadIdx.x <= m) {   // the path (and the pages), staged once
        const int p = pb[threadIdx.x];
        path_s[threadIdx.x] = p;
        if (p < 0 || p >= R) ok_s = 0;
        if (pages) {
            const int pg = pages[static_cast<size_t>(b) * max_pages + (t + threadIdx.x) / kPage];
            page_s[threadIdx.x] = pg;
            if (pg < 0 || pg >= num_pages) page_ok_s = 0;
        }
    }
    __syncthreads();
    if (!ok_s || !page_ok_s) {   // uniform across the cluster: nobody copies, nobody waits
        if (rank == 0 && threadIdx.x == 0)
            raise_error(err, !ok_s ? ((t >= 0 && m >= 0 && m < R && t + m + 1 > T_cap) || t < 0 ? SV_DEVERR_LENGTH
                                                                                             : SV_DEVERR_PATH)
                                   : SV_DEVERR_PAGE);
        return;
    }
    const int vec = D / 8;                    // 16-byte pieces per row
    const int rows = m + 1;
    const int per_layer = 2 * Hkv * rows * vec;
    const int nl = rank < L ? (L - 1 - rank) / kCluster + 1 : 0;   // layers rank, rank + 8, ...
    const int total = nl * per_layer;
    // eight pieces per thread in flight: all loads, then all stores
    constexpr int kBatch = 8;
    for (int w0 = threadIdx.x; w0 < total; w0 += kBatch * kThreads) {
        uint4 v[kBatch];
        uint4* dst[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int w = w0 + u * kThreads;
            dst[u] = nullptr;
            if (w >= total) continue;
            int x = w % per_layer;
            const int l = rank + (w / per_layer) * kCluster;
            const int c = x % vec;
            x /= vec;
            const int i = x % rows;
            x /= rows;
            const int g = x % Hkv;
            const int is_v = x / Hkv;
            const size_t lbg = (static_cast<size_t>(l) * B + b) * Hkv + g;
            const uint4* src = reinterpret_cast<const uint4*>((is_v ? v_blk : k_blk) +
                                                              (lbg * R + static_cast<size_t>(path_s[i])) * D) + c;
            const size_t drow =
                pages ? ((static_cast<size_t>(l) * num_pages + page_s[i]) * Hkv + g) * kPage + (t + i) % kPage
                      : lbg * T_cap + static_cast<size_t>(t + i);
            dst[u] = reinterpret_cast<uint4*>((is_v ? v_cache : k_cache) + drow * D) + c;
            v[u] = __ldg(src);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (dst[u]) *dst[u] = v[u];
    }
    cluster.sync();   // every CTA has read len[b]
    if (rank == 0 && threadIdx.x == 0) len[b] = t + m + 1;
}

}  // namespace

cudaError_t launch_kv_commit(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk,
                             int L, int B, int Hkv, int D, int T_cap, int R, const int32_t* path,
                             const int32_t* n_acc, int32_t* len, const int32_t* pages, int max_pages,
                             int num_pages, cudaStream_t st) {
    return launch_pdl(kv_commit_kernel, dim3(B * kCluster), dim3(kThreads), 0, st, k_cache, v_cache, k_blk, v_blk, L,
                      B, Hkv, D, T_cap, R, path, n_acc, len, pages, max_pages, num_pages, device_error_word());
}

}  // namespace sv
