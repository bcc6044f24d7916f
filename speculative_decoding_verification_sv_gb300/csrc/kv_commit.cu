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
// One 8-CTA cluster per sequence: every CTA reads len[b] and the path, copies
// its share of the layers' accepted rows with 16-byte vector moves, and after
// a cluster barrier (all reads of len[b] done) rank 0 advances len[b].  The
// block rows live in a separate staging buffer, so rejected rows never enter
// the cache and nothing has to be rolled back.
#include <cooperative_groups.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kCluster = 8;
constexpr int kThreads = 256;

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    kv_commit_kernel(uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache,
                     const uint16_t* __restrict__ k_blk, const uint16_t* __restrict__ v_blk, int L, int B, int Hkv,
                     int D, int T_cap, int R, const int32_t* __restrict__ path, const int32_t* __restrict__ n_acc,
                     int32_t* len, unsigned int* err) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.x / kCluster;
    const int t = len[b];
    const int m = n_acc[b];
    bool ok = t >= 0 && m >= 0 && m < R && t + m + 1 <= T_cap;
    const int32_t* pb = path + static_cast<size_t>(b) * R;
    if (ok)
        for (int i = 0; i <= m; ++i)
            if (pb[i] < 0 || pb[i] >= R) ok = false;
    if (!ok) {   // uniform across the cluster: nobody copies, nobody waits
        if (rank == 0 && threadIdx.x == 0)
            raise_error(err, (t >= 0 && m >= 0 && m < R && t + m + 1 > T_cap) || t < 0 ? SV_DEVERR_LENGTH
                                                                                     : SV_DEVERR_PATH);
        return;
    }
    const int vec = D / 8;                    // 16-byte pieces per row
    const int rows = m + 1;
    const int per_layer = 2 * Hkv * rows * vec;
    for (int l = rank; l < L; l += kCluster) {
        for (int w = threadIdx.x; w < per_layer; w += kThreads) {
            int x = w;
            const int c = x % vec;
            x /= vec;
            const int i = x % rows;
            x /= rows;
            const int g = x % Hkv;
            const int is_v = x / Hkv;
            const size_t lbg = (static_cast<size_t>(l) * B + b) * Hkv + g;
            const uint4* src = reinterpret_cast<const uint4*>((is_v ? v_blk : k_blk) +
                                                              (lbg * R + static_cast<size_t>(pb[i])) * D) + c;
            uint4* dst = reinterpret_cast<uint4*>((is_v ? v_cache : k_cache) +
                                                  (lbg * T_cap + static_cast<size_t>(t + i)) * D) + c;
            *dst = __ldg(src);
        }
    }
    cluster.sync();   // every CTA has read len[b]
    if (rank == 0 && threadIdx.x == 0) len[b] = t + m + 1;
}

}  // namespace

cudaError_t launch_kv_commit(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk,
                             int L, int B, int Hkv, int D, int T_cap, int R, const int32_t* path,
                             const int32_t* n_acc, int32_t* len, cudaStream_t st) {
    kv_commit_kernel<<<B * kCluster, kThreads, 0, st>>>(k_cache, v_cache, k_blk, v_blk, L, B, Hkv, D, T_cap, R, path,
                                                        n_acc, len, device_error_word());
    return cudaGetLastError();
}

}  // namespace sv
