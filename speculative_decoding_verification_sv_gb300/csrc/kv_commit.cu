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

// Copies this CTA's share of the accepted rows (layers rank, rank + 8, ...)
// of sequence b: block row path_s[i] -> cache slot t + i, for K and V, in
// 16-byte pieces, eight loads in flight per thread before their stores.
__device__ __forceinline__ void copy_accepted_rows(uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache,
                                                   const uint16_t* __restrict__ k_blk,
                                                   const uint16_t* __restrict__ v_blk, int L, int B, int Hkv, int D,
                                                   int T_cap, int R, int b, int t, int m, int rank,
                                                   const int* path_s, const int* page_s, bool paged, int num_pages) {
    const int vec = D / 8;                    // 16-byte pieces per row
    const int rows = m + 1;
    const int per_layer = 2 * Hkv * rows * vec;
    const int nl = rank < L ? (L - 1 - rank) / kCluster + 1 : 0;   // layers rank, rank + 8, ...
    const int total = nl * per_layer;
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
                paged ? ((static_cast<size_t>(l) * num_pages + page_s[i]) * Hkv + g) * kPage + (t + i) % kPage
                      : lbg * T_cap + static_cast<size_t>(t + i);
            dst[u] = reinterpret_cast<uint4*>((is_v ? v_cache : k_cache) + drow * D) + c;
            v[u] = __ldg(src);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (dst[u]) *dst[u] = v[u];
    }
}

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
    copy_accepted_rows(k_cache, v_cache, k_blk, v_blk, L, B, Hkv, D, T_cap, R, b, t, m, rank, path_s, page_s,
                       pages != nullptr, num_pages);
    cluster.sync();   // every CTA has read len[b]
    if (rank == 0 && threadIdx.x == 0) len[b] = t + m + 1;
}

// Greedy acceptance from the LM head's argmax keys, then the commit, in one
// launch: one 8-CTA cluster per sequence.
//   1. The R rows' keys (nslab per row) are split into pieces over the
//      cluster's 64 warps; each warp reduces its piece and pushes the result
//      into every CTA's shared memory; after a cluster barrier each CTA
//      holds every row's greedy token g_j.
//   2. Draft c matches when tok[c] == g_parent(c); the first matching child
//      of each node (lowest index) comes from one shared-memory atomicMin
//      per matching draft, and the walk from the root follows those links --
//      the same walk in every CTA, so every CTA knows the path.
//   3. The commit as in kv_commit_kernel: each CTA copies its layers' share
//      of the accepted rows (into page pools through the page table when
//      pages != nullptr); after a second cluster barrier rank 0 advances
//      len[b] (rank 0 also writes n_acc, out_tok and path).
// Without caches (k_cache == nullptr) it is greedy acceptance alone.
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    greedy_commit_kernel(const uint64_t* __restrict__ amax, int nslab, const int32_t* __restrict__ tok,
                         const int32_t* __restrict__ parent, int R, int V, int32_t* n_acc, int32_t* out_tok,
                         int32_t* path, uint16_t* __restrict__ k_cache, uint16_t* __restrict__ v_cache,
                         const uint16_t* __restrict__ k_blk, const uint16_t* __restrict__ v_blk, int L, int B,
                         int Hkv, int D, int T_cap, int32_t* len, const int32_t* __restrict__ pages, int max_pages,
                         int num_pages, unsigned int* err) {
    constexpr int kWarpsPerCta = kThreads / 32;
    constexpr int kClusterWarps = kCluster * kWarpsPerCta;
    constexpr int kPieces = 2 * kClusterWarps;   // (row, piece) items: at most two per warp
    static_assert(kPieces >= kMaxR, "every row gets at least one piece");
    __shared__ uint64_t piece_s[kPieces];
    __shared__ int g_s[kMaxR];
    __shared__ int tok_s[kMaxR];
    __shared__ int par_s[kMaxR];
    __shared__ int fmc_s[kMaxR];    // first matching child of each node (R: none)
    __shared__ int path_s[kMaxR];
    __shared__ int page_s[kMaxR];   // paged: the page of slot t + i
    __shared__ int m_s, t_s, bad_s, page_ok_s;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.x / kCluster;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    cluster_arrive_relaxed();   // this CTA has started (remote stores below wait for all)
    pdl_wait();                 // the keys, tokens and block rows come from the kernels before this one
    pdl_launch_dependents();

    // the sequence's tokens, tree and length, loaded in parallel
    if (threadIdx.x == 0) {
        bad_s = 0;
        t_s = k_cache ? len[b] : 0;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < R; j += kThreads) {
        const int tk = tok[static_cast<size_t>(b) * R + j];
        const int p = parent ? parent[static_cast<size_t>(b) * R + j] : j - 1;
        tok_s[j] = tk;
        par_s[j] = p;
        fmc_s[j] = R;
        if (j > 0 && (tk < 0 || tk >= V)) atomicOr(&bad_s, 1);
        if ((j == 0 && p != -1) || (j > 0 && (p < 0 || p >= j))) atomicOr(&bad_s, 2);
    }

    // 1. row argmax: P pieces per row, items (row, piece) over the cluster's warps
    const int P = kPieces / R;
    const int items = R * P;
    const int gw = rank * kWarpsPerCta + warp;
    // both of a warp's items at once, up to 8 keys per lane and item in
    // flight per round (one dependent round trip per 256 keys of both items,
    // not per 256 keys of each item in turn)
    // keys [p, p + n) of item `it` of this sequence (n = 0 past the last item)
    auto item_keys = [&](int it, const uint64_t*& p_out, int& n_out) {
        p_out = amax;
        n_out = 0;
        if (it < items) {
            const int j = it / P, p = it % P;
            // p < P <= 128, so nslab * (p + 1) <= ceil(V / 128) * 128 < 2^32
            const int s0 = static_cast<int>(static_cast<uint32_t>(nslab) * p / static_cast<uint32_t>(P));
            const int s1 = static_cast<int>(static_cast<uint32_t>(nslab) * (p + 1) / static_cast<uint32_t>(P));
            p_out = amax + (static_cast<size_t>(b) * R + j) * nslab + s0;
            n_out = s1 - s0;
        }
    };
    const uint64_t *kp0, *kp1;
    int kn0, kn1;
    item_keys(gw, kp0, kn0);
    item_keys(gw + kClusterWarps, kp1, kn1);
    uint64_t best0 = 0, best1 = 0;
    constexpr int kKeysInFlight = 8;
    for (int base = lane; base < max(kn0, kn1); base += 32 * kKeysInFlight) {
        uint64_t k0[kKeysInFlight], k1[kKeysInFlight];
#pragma unroll
        for (int u = 0; u < kKeysInFlight; ++u) {
            const int s = base + 32 * u;
            k0[u] = s < kn0 ? __ldg(kp0 + s) : 0ull;
            k1[u] = s < kn1 ? __ldg(kp1 + s) : 0ull;
        }
#pragma unroll
        for (int u = 0; u < kKeysInFlight; ++u) {
            best0 = k0[u] > best0 ? k0[u] : best0;
            best1 = k1[u] > best1 ? k1[u] : best1;
        }
    }
    const uint64_t res0 = warp_max_key(best0), res1 = warp_max_key(best1);
    cluster_wait();   // every CTA of the cluster has started
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int it = gw + r * kClusterWarps;
            if (it >= items) break;
            for (int dst = 0; dst < kCluster; ++dst)
                *cluster.map_shared_rank(&piece_s[it], dst) = r == 0 ? res0 : res1;
        }
    }
    cluster.sync();   // every piece pushed into every CTA (and tok_s, par_s, t_s visible in the CTA)
    for (int j = threadIdx.x; j < R; j += kThreads) {
        uint64_t k = 0;
        for (int p = 0; p < P; ++p) k = piece_s[j * P + p] > k ? piece_s[j * P + p] : k;
        g_s[j] = argmax_col(k);
    }
    __syncthreads();

    // 2. first matching child of every node, then the walk
    const bool tree_ok = (bad_s & 2) == 0;
    if (tree_ok)
        for (int c = 1 + threadIdx.x; c < R; c += kThreads)
            if (tok_s[c] == g_s[par_s[c]]) atomicMin(&fmc_s[par_s[c]], c);
    __syncthreads();
    if (threadIdx.x == 0) {
        if (rank == 0) {
            if (bad_s & 1) raise_error(err, SV_DEVERR_TOKEN);
            if (parent && !tree_ok) raise_error(err, SV_DEVERR_TREE);
        }
        int u = 0, depth = 0;
        path_s[0] = 0;
        for (int guard = 0; tree_ok && guard < R && fmc_s[u] < R; ++guard) {
            u = fmc_s[u];
            path_s[++depth] = u;
        }
        m_s = depth;
        if (rank == 0) {
            n_acc[b] = depth;
            out_tok[b] = g_s[u];
        }
    }
    __syncthreads();
    const int m = m_s;
    if (rank == 0)
        for (int j = threadIdx.x; j < R; j += kThreads) path[static_cast<size_t>(b) * R + j] = j <= m ? path_s[j] : -1;
    if (k_cache == nullptr) return;

    // 3. the commit
    const int t = t_s;
    if (t < 0 || t + m + 1 > T_cap) {   // uniform across the cluster: nobody copies, nobody waits
        if (rank == 0 && threadIdx.x == 0) raise_error(err, SV_DEVERR_LENGTH);
        return;
    }
    if (pages) {   // the pages of slots t..t+m, staged and checked first
        if (threadIdx.x == 0) page_ok_s = 1;
        __syncthreads();
        if (threadIdx.x <= m) {
            const int pg = pages[static_cast<size_t>(b) * max_pages + (t + threadIdx.x) / kPage];
            page_s[threadIdx.x] = pg;
            if (pg < 0 || pg >= num_pages) page_ok_s = 0;
        }
        __syncthreads();
        if (!page_ok_s) {   // uniform across the cluster
            if (rank == 0 && threadIdx.x == 0) raise_error(err, SV_DEVERR_PAGE);
            return;
        }
    }
    copy_accepted_rows(k_cache, v_cache, k_blk, v_blk, L, B, Hkv, D, T_cap, R, b, t, m, rank, path_s, page_s,
                       pages != nullptr, num_pages);
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

cudaError_t launch_accept_greedy_commit(const uint64_t* amax, const int32_t* tok, const int32_t* parent, int B, int R,
                                        int V, int32_t* n_acc, int32_t* out_tok, int32_t* path, uint16_t* k_cache,
                                        uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk, int L,
                                        int Hkv, int D, int T_cap, int32_t* len, const int32_t* pages, int max_pages,
                                        int num_pages, cudaStream_t st) {
    const int nslab = (V + kArgmaxSlab - 1) / kArgmaxSlab;
    return launch_pdl(greedy_commit_kernel, dim3(B * kCluster), dim3(kThreads), 0, st, amax, nslab, tok, parent, R,
                      V, n_acc, out_tok, path, k_cache, v_cache, k_blk, v_blk, L, B, Hkv, D, T_cap, len, pages,
                      max_pages, num_pages, device_error_word());
}

}  // namespace sv
