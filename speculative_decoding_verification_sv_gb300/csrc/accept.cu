// accept.cu -- greedy and sampled acceptance of one verify round.
//
// Greedy ([SpecDec-Context-Scaling guide, sec. 3 and 3.1]): a vocab-parallel
// argmax of every verify row, then a per-sequence walk that compares draft j
// with the argmax of row j-1 (row 0 is saved_next), or walks a draft tree.
//
// Sampled ([wmrh.cn tutorial, sec. 2.2]; [mini-infer Phase 11, "Modified
// Rejection Sampling"]; trees: [SubSpec summary, sec. 4.2]):
//   1. sample_stats_kernel: one 8-CTA cluster per verify row pulls the row
//      into shared memory with bulk copies, reduces the max of l/T across the
//      cluster through distributed shared memory, and forms the canonical
//      sum Z of exp(l/T - max).  The row is read from HBM exactly once.
//   2. sample_finish_kernel: one cluster per sequence (16 CTAs for a few
//      sequences, else 8) runs the acceptance walk (element-wise ratio tests
//      from the row statistics),
//      and the full-vocab passes it needs: the residual max(0, w - q) and its
//      canonical sum, then inverse-CDF sampling by descending the summation
//      tree (block level across the cluster, chunk level in shared memory,
//      leaf level in one warp).
// The summation tree: leaves = vocab entries zero-padded to 2^18; 4 leaves per
// lane (level 2), 32 lanes per 128-leaf chunk (level 7), 32 chunks per
// 4096-leaf block (level 12), 64 blocks (level 18).  Every level pairs
// contiguous siblings, so the value of every node does not depend on the
// launch shape.
#include <cooperative_groups.h>
#include <float.h>
#include <limits.h>
#include <stdlib.h>

#include <mutex>
#include <type_traits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kBlk = 4096;            // leaves per block
constexpr int kChunk = 128;           // leaves per chunk
constexpr int kChunksPerBlk = kBlk / kChunk;
constexpr int kMaxBlocks = 64;        // 2^18 / 4096
constexpr int kCluster = 8;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxLocalBlocks = kMaxBlocks / kCluster;
constexpr int kMaxR = 128;
#ifndef SV_ROW_STATS_MIN_ROWS
#define SV_ROW_STATS_MIN_ROWS 128
#endif
constexpr int kRowStatsMinRows = SV_ROW_STATS_MIN_ROWS;   // B*R from which statistics use one CTA per row

// With SV_SYNC_EACH_KERNEL=1 in the environment the launchers synchronise
// after every kernel so a failing kernel is reported by name.
bool debug_sync() {
    static const bool on = [] {
        const char* e = getenv("SV_SYNC_EACH_KERNEL");
        return e && e[0] == '1';
    }();
    return on;
}

// ==========================================================================
// greedy
// ==========================================================================

#ifndef SV_GREEDY_CHUNK
#define SV_GREEDY_CHUNK 8192
#endif
constexpr int kGreedyChunk = SV_GREEDY_CHUNK;   // vocab columns per argmax CTA
constexpr int kGreedyThreads = 256;

struct ArgMax {
    float v;
    int i;
};

__device__ __forceinline__ ArgMax pick(ArgMax a, ArgMax b) {
    return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__device__ __forceinline__ ArgMax warp_pick(ArgMax a) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ArgMax o;
        o.v = __shfl_xor_sync(0xffffffffu, a.v, off);
        o.i = __shfl_xor_sync(0xffffffffu, a.i, off);
        a = pick(a, o);
    }
    return a;
}

__global__ void __launch_bounds__(kGreedyThreads) greedy_partial_kernel(const float* __restrict__ logits, int V,
                                                                         int nchunk, int2* __restrict__ part,
                                                                         unsigned int* err) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    const int row = blockIdx.y;
    const int c0 = blockIdx.x * kGreedyChunk;
    const int c1 = min(c0 + kGreedyChunk, V);
    const float* L = logits + static_cast<size_t>(row) * V;
    ArgMax best{-INFINITY, INT_MAX};
    bool bad = false;
    if ((V & 3) == 0) {
        // all of a thread's loads of the chunk in flight at once (8 float4)
        constexpr int kPer = kGreedyChunk / (4 * kGreedyThreads);
        float4 xv[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int i = c0 + 4 * (threadIdx.x + u * kGreedyThreads);
            xv[u] = i < c1 ? __ldg(reinterpret_cast<const float4*>(L + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int i = c0 + 4 * (threadIdx.x + u * kGreedyThreads);
            if (i >= c1) continue;
            const float xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (xs[e] != xs[e]) { bad = true; continue; }
                if (xs[e] > best.v || (xs[e] == best.v && i + e < best.i)) best = ArgMax{xs[e], i + e};
            }
        }
    } else {
        for (int i = c0 + threadIdx.x; i < c1; i += kGreedyThreads) {
            const float x = __ldg(L + i);
            if (x != x) { bad = true; continue; }
            if (x > best.v || (x == best.v && i < best.i)) best = ArgMax{x, i};
        }
    }
    if (bad) raise_error(err, SV_DEVERR_NONFINITE);
    best = warp_pick(best);
    __shared__ ArgMax red[kGreedyThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < kGreedyThreads / 32 ? red[lane] : ArgMax{-INFINITY, INT_MAX};
        best = warp_pick(best);
        if (lane == 0) part[static_cast<size_t>(row) * nchunk + blockIdx.x] = make_int2(__float_as_int(best.v), best.i);
    }
}

__global__ void __launch_bounds__(128) greedy_finish_kernel(const int2* __restrict__ part, int nchunk,
                                                             const int32_t* __restrict__ tok,
                                                             const int32_t* __restrict__ parent, int R, int V,
                                                             int32_t* n_acc, int32_t* out_tok, int32_t* path,
                                                             unsigned int* err) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    __shared__ int g[kMaxR];
    __shared__ int par_s[kMaxR];
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < R; j += 4) {
        ArgMax best{-INFINITY, INT_MAX};
        const int2* pr = part + (static_cast<size_t>(b) * R + j) * nchunk;
        for (int c = lane; c < nchunk; c += 32) {
            const int2 x = pr[c];
            best = pick(best, ArgMax{__int_as_float(x.x), x.y});
        }
        best = warp_pick(best);
        if (lane == 0) g[j] = (best.i == INT_MAX) ? 0 : best.i;
    }
    bool tree_ok = true;
    if (parent) tree_ok = load_tree(parent, b, R, par_s, err);
    __syncthreads();
    if (threadIdx.x != 0) return;
    const int32_t* tk = tok + static_cast<size_t>(b) * R;
    int32_t* pth = path + static_cast<size_t>(b) * R;
    for (int j = 1; j < R; ++j)
        if (tk[j] < 0 || tk[j] >= V) raise_error(err, SV_DEVERR_TOKEN);
    const int* par = parent ? par_s : nullptr;
    int u = 0, depth = 0;
    pth[0] = 0;
    if (tree_ok) {
        for (int guard = 0; guard < R; ++guard) {
            int next = -1;
            for (int c = next_child(par, R, u, -1); c >= 0; c = next_child(par, R, u, c))
                if (tk[c] == g[u]) { next = c; break; }
            if (next < 0) break;
            u = next;
            pth[++depth] = u;
        }
    }
    for (int j = depth + 1; j < R; ++j) pth[j] = -1;
    n_acc[b] = depth;
    out_tok[b] = g[u];
}

// ==========================================================================
// sampled: row statistics
// ==========================================================================

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    sample_stats_kernel(const float* __restrict__ logits, int V, float T, int nblk, int smem_blocks,
                        float2* __restrict__ stats, unsigned int* err) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    extern __shared__ __align__(128) float srow[];   // [local blocks][4096]
    __shared__ float cmax[kCluster];
    __shared__ float bsum[kMaxBlocks];
    __shared__ float csum[kMaxLocalBlocks * kChunksPerBlk];
    __shared__ __align__(8) uint64_t bar;
    __shared__ float wred[kWarps];

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int row = blockIdx.x / kCluster;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float* L = logits + static_cast<size_t>(row) * V;
    const int nlocal = rank < nblk ? (nblk - rank + kCluster - 1) / kCluster : 0;

    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (tid < kMaxBlocks) bsum[tid] = 0.0f;
    __syncthreads();
    cluster_arrive_relaxed();   // paired with cluster_wait() before the first remote store
    if (tid == 0 && nlocal > 0) {
        uint32_t total = 0;
        for (int lb = 0; lb < nlocal; ++lb) {
            const int gb = rank + lb * kCluster;
            total += static_cast<uint32_t>(min(kBlk, V - gb * kBlk)) * 4u;
        }
        mbar_arrive_expect_tx(&bar, total);
        for (int lb = 0; lb < nlocal; ++lb) {
            const int gb = rank + lb * kCluster;
            const int n = min(kBlk, V - gb * kBlk);
            if (!SV_CHECK(n > 0 && (n & 3) == 0 && lb < smem_blocks, err, 3)) continue;
            bulk_g2s(srow + lb * kBlk, L + static_cast<size_t>(gb) * kBlk, static_cast<uint32_t>(n) * 4u, &bar);
        }
    }
    if (nlocal > 0) mbar_wait(&bar, 0, err);

    // local max of z = l / T (z stored back when T != 1)
    float m = -INFINITY;
    float nf = 0.0f;   // stays 0 unless some z is NaN or infinite (z * 0 is then NaN)
    for (int lb = 0; lb < nlocal; ++lb) {
        const int gb = rank + lb * kCluster;
        const int n = min(kBlk, V - gb * kBlk);
        float* s = srow + lb * kBlk;
        for (int i = 4 * tid; i < n; i += 4 * kThreads) {
            float4 x = *reinterpret_cast<float4*>(s + i);
            if (T != 1.0f) {
                x = make_float4(__fdiv_rn(x.x, T), __fdiv_rn(x.y, T), __fdiv_rn(x.z, T), __fdiv_rn(x.w, T));
                *reinterpret_cast<float4*>(s + i) = x;
            }
            nf = __fmaf_rn(x.x, 0.0f, __fmaf_rn(x.y, 0.0f, __fmaf_rn(x.z, 0.0f, __fmaf_rn(x.w, 0.0f, nf))));
            m = fmaxf(fmaxf(m, fmaxf(x.x, x.y)), fmaxf(x.z, x.w));
        }
    }
    if (nf != 0.0f) raise_error(err, SV_DEVERR_NONFINITE);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) wred[warp] = m;
    __syncthreads();
    cluster_wait();             // every CTA of the cluster has started
    if (tid < kCluster) {
        float mm = -INFINITY;
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, wred[w]);
        *cluster.map_shared_rank(&cmax[rank], tid) = mm;
    }
    cluster.sync();
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) M = fmaxf(M, cmax[r]);

    // chunk sums (level 7) of e = exp(z - M), zero beyond V
    for (int cid = warp; cid < nlocal * kChunksPerBlk; cid += kWarps) {
        const int lb = cid / kChunksPerBlk, c = cid % kChunksPerBlk;
        const int gb = rank + lb * kCluster;
        const int v = gb * kBlk + c * kChunk + 4 * lane;
        float4 e = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < V) {
            const float4 z = *reinterpret_cast<const float4*>(srow + lb * kBlk + c * kChunk + 4 * lane);
            e = make_float4(sv_exp_nb(__fsub_rn(z.x, M)), sv_exp_nb(__fsub_rn(z.y, M)), sv_exp_nb(__fsub_rn(z.z, M)),
                            sv_exp_nb(__fsub_rn(z.w, M)));
        }
        const float cs = warp_tree_sum(quad_sum(e));
        if (lane == 0) csum[cid] = cs;
    }
    __syncthreads();
    // block sums (level 12), pushed to rank 0
    if (warp < nlocal) {
        const float bs = warp_tree_sum(csum[warp * kChunksPerBlk + lane]);
        if (lane == 0 && SV_CHECK(rank + warp * kCluster < kMaxBlocks, err, 4))
            *cluster.map_shared_rank(&bsum[rank + warp * kCluster], 0) = bs;
    }
    cluster.sync();
    if (rank == 0 && warp == 0) {
        const float Z = warp_tree_sum(__fadd_rn(bsum[2 * lane], bsum[2 * lane + 1]));   // level 13 -> 18
        if (lane == 0) {
            if (!(Z > 0.0f) || !isfinite(Z)) raise_error(err, SV_DEVERR_NONFINITE);
            stats[row] = make_float2(M, Z);
        }
    }
}

// Many rows (B*R large): persistent pairs of CTAs (2-CTA clusters), each pair
// taking whole rows (row = cluster, + clusters, ...), each CTA one half of the
// row's 4096-leaf blocks.  A row needs two passes: the exact maximum of
// z = l / T, then the canonical tree over exp(z - M) -- chunk sums over 128
// leaves (4 per lane), block sums over 32 chunks, then the 64 zero-padded
// block sums.  The two are software pipelined across the pair's rows: one
// loop over the chunks re-reads row i (from L2, where its own max pass left
// it) for the exponential sums and reads row i + 1 from HBM for its maximum,
// so the DRAM stream of the next row runs under the issue-bound
// exponentials of the current one.  Splitting each row over two SMs halves
// the rows in flight (about 2 x 76 x 600 KB), so the re-read stays in L2; the
// halves' block sums and maxima meet through distributed shared memory, one
// cluster barrier per row.  The re-read carries an evict-first L2 policy (a
// summed chunk is dead).
#ifndef SV_ROW_THREADS
#define SV_ROW_THREADS 768
#endif
#ifndef SV_ROW_FUSE
#define SV_ROW_FUSE 4
#endif
constexpr int kRowThreads = SV_ROW_THREADS;       // one CTA of 24 warps per SM (80 registers)
constexpr int kRowCtasPerSm = kRowThreads >= 512 ? 1 : 512 / kRowThreads;
constexpr int kRowWarps = kRowThreads / 32;
static_assert(kRowWarps <= 32, "one warp's lanes reduce the CTA's warps");
constexpr int kRowFuse = SV_ROW_FUSE;             // chunks in flight per warp and row
static_assert(kRowFuse == 2 || kRowFuse == 4, "two or four chunks per warp and row");
constexpr int kRowPair = 2;                       // CTAs per row

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ float4 ldg_policy(const float* p, uint64_t pol) {
    float4 v;
    asm("ld.global.nc.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p), "l"(pol));
    return v;
}

// z = l / T of four leaves (kUnitT: T = 1, the logits themselves)
template <bool kUnitT>
__device__ __forceinline__ float4 scaled(float4 z, float T) {
    if constexpr (!kUnitT)
        z = make_float4(__fdiv_rn(z.x, T), __fdiv_rn(z.y, T), __fdiv_rn(z.z, T), __fdiv_rn(z.w, T));
    return z;
}

// Running maximum of four z values (NaN-ignoring: the row's M is the largest
// number), and a running NaN-propagating minimum: the row holds a non-finite
// z iff that minimum ends NaN or -inf, or the maximum +inf.
__device__ __forceinline__ void max_leaves(float4 z, float& m, float& mn) {
    m = fmax3(m, fmax3(z.x, z.y, z.z), z.w);
    mn = fmin3_nan(mn, fmin3_nan(z.x, z.y, z.z), z.w);
}

template <bool kUnitT>
__global__ void __cluster_dims__(kRowPair, 1, 1) __launch_bounds__(kRowThreads, kRowCtasPerSm)
    sample_stats_row_kernel(const float* __restrict__ logits, int V, float T, int nblk, int nrows,
                            float2* __restrict__ stats, unsigned int* err) {
    cluster_arrive_relaxed();   // the partner's shared memory is written only after it has started
    pdl_wait();                 // inputs come from the kernels before this one
    pdl_launch_dependents();
    __shared__ float csum[kMaxBlocks * kChunksPerBlk];
    __shared__ float bsum[2][kMaxBlocks];    // rank 0: the row's block sums, by row parity
    __shared__ float2 xch[2][kRowPair];      // (max, NaN-propagating min) of each half, by parity
    __shared__ float wred[kRowWarps];
    __shared__ float wmin[kRowWarps];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's blocks [b0, b1) and chunks [cb0, cb1); chunks below cfull
    // have all 128 leaves below V
    const int hb = (nblk + 1) / 2;
    const int b0 = min(nblk, rank * hb), b1 = min(nblk, b0 + hb);
    const int cb0 = b0 * kChunksPerBlk, cb1 = b1 * kChunksPerBlk;
    const int cfull = min(cb1, V / kChunk);
    const float4 ninf4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (rank == 0)
        for (int i = tid; i < 2 * kMaxBlocks; i += kRowThreads) bsum[i / kMaxBlocks][i % kMaxBlocks] = 0.0f;
    // the warp's chunks c0 + u * kRowWarps; lane holds leaves 4 lane .. of each
    auto leaf = [&](int c) { return c * kChunk + 4 * lane; };
    // the CTA's (max, min) of the next row by warp 0 and lane 0 of each warp
    // (after the barrier that follows), then into both CTAs' slot `rank`
    auto warp_minmax = [&](float m, float mn) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            mn = fmin_nan(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        }
        if (lane == 0) {
            wred[warp] = m;
            wmin[warp] = mn;
        }
    };
    auto publish_minmax = [&](int p) {   // warp 0, after a barrier over the warps' values
        float m = lane < kRowWarps ? wred[lane] : -INFINITY;
        float mn = lane < kRowWarps ? wmin[lane] : INFINITY;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            mn = fmin_nan(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        }
        if (lane < kRowPair) *cluster.map_shared_rank(&xch[p][rank], lane) = make_float2(m, mn);
    };
    // the row's M after the cluster barrier; flags non-finite z; nrm: every
    // z - M of the row lies where sv_exp_nrm applies
    auto take_max = [&](int p, bool& nrm) {
        const float2 h0 = xch[p][0], h1 = xch[p][1];
        const float M = fmaxf(h0.x, h1.x), zmin = fmin_nan(h0.y, h1.y);
        if (tid == 0 && rank == 0 && (M == INFINITY || !(zmin > -INFINITY))) raise_error(err, SV_DEVERR_NONFINITE);
        // z - M >= zmin - M for every z (rounding is monotonic); false for NaN
        nrm = __fsub_rn(zmin, M) > kExpNormalMin;
        return M;
    };

    const int ncl = static_cast<int>(gridDim.x) / kRowPair;
    int row = static_cast<int>(blockIdx.x) / kRowPair;
    cluster_wait();
    if (row >= nrows) return;   // both CTAs of the pair
    float M;
    bool nrm;
    {
        // prologue: the first row's maximum alone, twice the loads in flight
        const float* L = logits + static_cast<size_t>(row) * V;
        float m = -INFINITY, mn = INFINITY;
        for (int c0 = cb0 + warp; c0 < cb1; c0 += 2 * kRowFuse * kRowWarps) {
            float4 y[2 * kRowFuse];
#pragma unroll
            for (int u = 0; u < 2 * kRowFuse; ++u) {
                const int c = c0 + u * kRowWarps, v = leaf(c);
                y[u] = (c < cb1 && v < V) ? __ldg(reinterpret_cast<const float4*>(L + v)) : ninf4;
            }
#pragma unroll
            for (int u = 0; u < 2 * kRowFuse; ++u)
                if (c0 + u * kRowWarps < cb1 && leaf(c0 + u * kRowWarps) < V)
                    max_leaves(scaled<kUnitT>(y[u], T), m, mn);
        }
        warp_minmax(m, mn);
        __syncthreads();
        if (warp == 0) publish_minmax(1);
        cluster.sync();
        M = take_max(1, nrm);
    }
    const uint64_t pol = l2_evict_first_policy();
    for (int it = 0; row < nrows; row += ncl, ++it) {
        const int p = it & 1;
        const int nxt = row + ncl;
        const bool more = nxt < nrows;   // uniform over the pair
        const float* L = logits + static_cast<size_t>(row) * V;
        const float* Ln = logits + static_cast<size_t>(more ? nxt : row) * V;
        float m = -INFINITY, mn = INFINITY;
        // chunks c0 + u * kRowWarps, u < kRowFuse: row i's leaves (x) and row
        // i + 1's (y); kFull: all of them lie below V (no per-leaf test)
        auto load = [&](auto full, int c0, float4 (&x)[kRowFuse], float4 (&y)[kRowFuse]) {
            constexpr bool kFull = decltype(full)::value;
#pragma unroll
            for (int u = 0; u < kRowFuse; ++u) {
                const int c = c0 + u * kRowWarps, v = leaf(c);
                x[u] = (kFull || (c < cb1 && v < V)) ? ldg_policy(L + v, pol) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (more) {
#pragma unroll
                for (int u = 0; u < kRowFuse; ++u) {
                    const int c = c0 + u * kRowWarps, v = leaf(c);
                    y[u] = (kFull || (c < cb1 && v < V)) ? __ldg(reinterpret_cast<const float4*>(Ln + v)) : ninf4;
                }
            }
        };
        auto work = [&](auto full, const float4 (&x)[kRowFuse], const float4 (&y)[kRowFuse], int c0) {
            constexpr bool kFull = decltype(full)::value;
            // row i: chunk sums (level 7) of e = exp(z - M), zero beyond V.
            // Lane l's node over its 4 leaves of each chunk, then the 32
            // lanes' tree for all the chunks at once: at each of the first
            // levels a lane keeps half of its chunks and trades the other
            // half with its partner, so every lane ends with one chunk's sum
            // (chunk l % kRowFuse).  Each node is still its two children's
            // sum, so the values are those of the plain per-chunk tree.
            float q[kRowFuse];
#pragma unroll
            for (int u = 0; u < kRowFuse; ++u) {
                const int c = c0 + u * kRowWarps, v = leaf(c);
                float4 e = make_float4(0.f, 0.f, 0.f, 0.f);
                if (kFull || (c < cb1 && v < V)) {
                    const float4 z = scaled<kUnitT>(x[u], T);
                    const float4 d = make_float4(__fsub_rn(z.x, M), __fsub_rn(z.y, M), __fsub_rn(z.z, M),
                                                 __fsub_rn(z.w, M));
                    if (nrm)   // uniform: the row's exponentials are all normal
                        e = make_float4(sv_exp_nrm(d.x), sv_exp_nrm(d.y), sv_exp_nrm(d.z), sv_exp_nrm(d.w));
                    else
                        e = make_float4(sv_exp_nb(d.x), sv_exp_nb(d.y), sv_exp_nb(d.z), sv_exp_nb(d.w));
                }
                q[u] = quad_sum(e);
            }
            float w;
            const bool hi1 = (lane & 1) != 0;
            if constexpr (kRowFuse == 4) {
                const bool hi2 = (lane & 2) != 0;
                const float s0 = __shfl_xor_sync(0xffffffffu, hi1 ? q[0] : q[1], 1);
                const float s1 = __shfl_xor_sync(0xffffffffu, hi1 ? q[2] : q[3], 1);
                const float v0 = __fadd_rn(hi1 ? q[1] : q[0], s0);   // chunk (lane & 1)
                const float v1 = __fadd_rn(hi1 ? q[3] : q[2], s1);   // chunk 2 + (lane & 1)
                w = __fadd_rn(hi2 ? v1 : v0, __shfl_xor_sync(0xffffffffu, hi2 ? v0 : v1, 2));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) w = __fadd_rn(w, __shfl_xor_sync(0xffffffffu, w, off));
            } else {
                w = __fadd_rn(hi1 ? q[1] : q[0], __shfl_xor_sync(0xffffffffu, hi1 ? q[0] : q[1], 1));
#pragma unroll
                for (int off = 2; off < 32; off <<= 1) w = __fadd_rn(w, __shfl_xor_sync(0xffffffffu, w, off));
            }
            {
                const int c = c0 + (lane % kRowFuse) * kRowWarps;
                if (lane < kRowFuse && (kFull || c < cb1)) csum[c] = w;
            }
            // row i + 1: its maximum
            if (more) {
#pragma unroll
                for (int u = 0; u < kRowFuse; ++u)
                    if (kFull || (c0 + u * kRowWarps < cb1 && leaf(c0 + u * kRowWarps) < V))
                        max_leaves(scaled<kUnitT>(y[u], T), m, mn);
            }
        };
        constexpr int kStep = kRowFuse * kRowWarps;
        using Full = std::true_type;
        using Edge = std::false_type;
        int c0 = cb0 + warp;
        for (; c0 + (kRowFuse - 1) * kRowWarps < cfull; c0 += kStep) {
            float4 x[kRowFuse], y[kRowFuse];
            load(Full{}, c0, x, y);
            work(Full{}, x, y, c0);
        }
        for (; c0 < cb1; c0 += kStep) {
            float4 x[kRowFuse], y[kRowFuse];
            load(Edge{}, c0, x, y);
            work(Edge{}, x, y, c0);
        }
        if (more) warp_minmax(m, mn);
        __syncthreads();   // csum, wred and wmin complete
        // this half's block sums (level 12) into rank 0's; blocks beyond the
        // vocab stay zero
        for (int bk = b0 + warp; bk < b1; bk += kRowWarps) {
            const float bs = warp_tree_sum(csum[bk * kChunksPerBlk + lane]);
            if (lane == 0) *cluster.map_shared_rank(&bsum[p][bk], 0) = bs;   // rank 0's
        }
        if (more && warp == 0) publish_minmax(p);
        cluster.sync();    // both halves' block sums and next-row maxima are in place
        if (rank == 0 && warp == 0) {
            const float Z = warp_tree_sum(__fadd_rn(bsum[p][2 * lane], bsum[p][2 * lane + 1]));   // level 13 -> 18
            if (lane == 0) {
                if (!(Z > 0.0f) || !isfinite(Z)) raise_error(err, SV_DEVERR_NONFINITE);
                stats[row] = make_float2(M, Z);
            }
        }
        if (more) M = take_max(p, nrm);
    }
}

// ==========================================================================
// sampled: acceptance walk and full-vocab passes
// ==========================================================================

struct SampleArgs {
    const float* logits;
    const float* q;
    const int32_t* tok;
    const int32_t* parent;
    const float2* stats;
    const float* uniforms;
    int32_t* n_acc;
    int32_t* out_tok;
    int32_t* path;
    unsigned int* err;
    uint64_t seed, step;
    int R, Rq, V, Vq, nblk;
    float T;
};

// The working distribution at node u after `nsteps` rejected children:
// w_0 = p_u;  w_i = max(0, w_{i-1} - q_u) / S_i if S_i > 0, else w_{i-1}.
struct RowValues {
    const float* L;     // logits row u
    const float* Q;     // q row u (Vq entries); nullptr when no q row exists (a leaf)
    int Vq;
    float T, M, Z;
    float rZ;           // 1 / Z rounded to nearest (the divisions by Z through div_rn_by)
    const float* S;     // S_1..S_nsteps
    const float* rS;    // 1 / S_s rounded to nearest, where S_s > 0
    int nsteps;
    bool residual;      // value = max(0, w_nsteps - q) instead of w_nsteps
    int V;
    unsigned int* err;

    __device__ __forceinline__ float one(float l, float qv) const {
        const float z = (T == 1.0f) ? l : __fdiv_rn(l, T);
        float w = div_rn_by(sv_exp_nb(__fsub_rn(z, M)), Z, rZ);
        for (int s = 0; s < nsteps; ++s) {
            const float d = __fsub_rn(w, qv);
            const float rho = d > 0.0f ? d : 0.0f;
            w = S[s] > 0.0f ? div_rn_by(rho, S[s], rS[s]) : w;
        }
        if (residual) {
            const float d = __fsub_rn(w, qv);
            return d > 0.0f ? d : 0.0f;
        }
        return w;
    }
    __device__ __forceinline__ float at(int v) const {
        if (!SV_CHECK(v >= 0 && v < V, err, 5)) return 0.0f;
        const float qv = (Q != nullptr && v < Vq) ? __ldg(Q + v) : 0.0f;
        return one(__ldg(L + v), qv);
    }
    // 4 consecutive entries starting at v (v % 4 == 0, v < V, V % 4 == 0),
    // as a load (raw) and an evaluation, so callers can batch the loads
    struct Raw {
        float4 l, q;
    };
    __device__ __forceinline__ Raw load4(int v) const {
        Raw r{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
        if (!SV_CHECK(v >= 0 && v + 3 < V && (v & 3) == 0, err, 6)) return r;
        r.l = __ldg(reinterpret_cast<const float4*>(L + v));
        if (Q != nullptr && v < Vq) r.q = __ldg(reinterpret_cast<const float4*>(Q + v));
        return r;
    }
    __device__ __forceinline__ float4 eval4(const Raw& r) const {
        return make_float4(one(r.l.x, r.q.x), one(r.l.y, r.q.y), one(r.l.z, r.q.z), one(r.l.w, r.q.w));
    }
    __device__ __forceinline__ float4 at4(int v) const { return eval4(load4(v)); }
};

// Raw values of a float array (diagnostic path).
struct ArrayValues {
    const float* x;
    using Raw = float4;
    __device__ __forceinline__ Raw load4(int v) const { return __ldg(reinterpret_cast<const float4*>(x + v)); }
    __device__ __forceinline__ float4 eval4(const Raw& r) const { return r; }
    __device__ __forceinline__ float4 at4(int v) const { return load4(v); }
};

// Shared state of one cluster's full-vocab pass.
struct PassSmem {
    float csum[kMaxLocalBlocks * kChunksPerBlk];
    float bsum[kMaxBlocks];
    float tree[2 * kMaxBlocks];   // upper levels of the summation tree during a descent
    int token;
    int node;
    float acc;
    float total;   // canonical sum of the last full pass
};

// Builds the levels above `n` leaves (n a power of two <= 64) in sm.tree by
// warp 0: tree[0..n) = leaves, then each level follows the previous one.
__device__ __forceinline__ void build_levels(const float* leaves, int n, float* tree) {
    const int lane = threadIdx.x & 31;
    for (int i = lane; i < n; i += 32) tree[i] = leaves[i];
    __syncwarp();
    int in = 0, out = n;
    for (int m = n >> 1; m >= 1; m >>= 1) {
        for (int i = lane; i < m; i += 32) tree[out + i] = __fadd_rn(tree[in + 2 * i], tree[in + 2 * i + 1]);
        __syncwarp();
        in = out;
        out += m;
    }
}

// Descends from the root of a tree built by build_levels over n leaves;
// returns the leaf index and updates acc.
__device__ __forceinline__ int descend_levels(const float* tree, int n, float tau, float& acc) {
    // level offsets: leaves at 0, parents at n, ... ; root at 2n-2
    int offs[8];
    int lv = 0, off = 0;
    for (int m = n; m >= 1; m >>= 1) { offs[lv++] = off; off += m; }
    int node = 0;
    for (int l = lv - 1; l >= 1; --l) {   // node at level l, children at level l-1
        const float sl = tree[offs[l - 1] + 2 * node], sr = tree[offs[l - 1] + 2 * node + 1];
        if (tau < __fadd_rn(acc, sl) || sr == 0.0f) {
            node = 2 * node;
        } else {
            acc = __fadd_rn(acc, sl);
            node = 2 * node + 1;
        }
    }
    return node;
}

// Full pass over the vocab: chunk sums into csum (this CTA's blocks), block
// sums into every CTA's bsum; returns the canonical total (identical in every
// CTA).  All threads of all CTAs of the cluster must call it.
template <int kC, int kW, class Vals>
__device__ float full_pass(const Vals& vals, int V, int nblk, PassSmem& sm, cg::cluster_group& cluster) {
    static_assert(kC <= 32 && kMaxBlocks / kC <= kMaxLocalBlocks && kW >= kMaxBlocks / kC, "cluster shape");
    const int rank = static_cast<int>(cluster.block_rank());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nlocal = rank < nblk ? (nblk - rank + kC - 1) / kC : 0;
    cluster.sync();   // all CTAs started (first pass) / previous pass fully consumed everywhere
    const int nch = nlocal * kChunksPerBlk;
    constexpr int kBatch = 2;   // chunks whose loads a warp keeps in flight
    for (int cid0 = warp; cid0 < nch; cid0 += kBatch * kW) {
        typename Vals::Raw raw[kBatch];
        bool live[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int cid = cid0 + u * kW;
            const int lb = cid / kChunksPerBlk, c = cid % kChunksPerBlk;
            const int v = (rank + lb * kC) * kBlk + c * kChunk + 4 * lane;
            live[u] = cid < nch && v < V;
            if (live[u]) raw[u] = vals.load4(v);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int cid = cid0 + u * kW;
            const float4 x = live[u] ? vals.eval4(raw[u]) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float cs = warp_tree_sum(quad_sum(x));
            if (lane == 0 && cid < nch) sm.csum[cid] = cs;
        }
    }
    __syncthreads();
    if (warp < nlocal) {
        const float bs = warp_tree_sum(sm.csum[warp * kChunksPerBlk + lane]);
        if (lane < kC) *cluster.map_shared_rank(&sm.bsum[rank + warp * kC], lane) = bs;
    }
    cluster.sync();
    // levels 13 -> 18 over the 64 block sums (lane i: blocks 2i, 2i+1)
    if (warp == 0) {
        const float tot = warp_tree_sum(__fadd_rn(sm.bsum[2 * lane], sm.bsum[2 * lane + 1]));
        if (lane == 0) sm.total = tot;
    }
    __syncthreads();
    return sm.total;
}

// One descent step: children sums sl, sr of the current node.
__device__ __forceinline__ bool go_left(float tau, float acc, float sl, float sr) {
    return tau < __fadd_rn(acc, sl) || sr == 0.0f;
}

// Levels 7 -> 0 of the summation tree inside one 128-leaf chunk starting at
// v0, by one full warp that recomputes the chunk's leaves; acc is the prefix
// sum before the chunk and tau the target.  Returns the token (every lane).
template <class Vals>
__device__ __forceinline__ int descend_chunk(const Vals& vals, int v0, int V, float tau, float acc) {
    const int lane = threadIdx.x & 31;
    const int v = v0 + 4 * lane;
    const float4 x = v < V ? vals.at4(v) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float n1a = __fadd_rn(x.x, x.y), n1b = __fadd_rn(x.z, x.w);
    float lvl[6];                      // lvl[k]: node at level k+2 containing this lane
    lvl[0] = __fadd_rn(n1a, n1b);
#pragma unroll
    for (int k = 1; k < 6; ++k) lvl[k] = __fadd_rn(lvl[k - 1], __shfl_xor_sync(0xffffffffu, lvl[k - 1], 1 << (k - 1)));
    int base = 0;                       // first lane of the current node
#pragma unroll
    for (int k = 5; k >= 1; --k) {      // node at level k+2 -> children at level k+1
        const int half = 1 << (k - 1);
        const float sl = __shfl_sync(0xffffffffu, lvl[k - 1], base);
        const float sr = __shfl_sync(0xffffffffu, lvl[k - 1], base + half);
        if (!go_left(tau, acc, sl, sr)) {
            acc = __fadd_rn(acc, sl);
            base += half;
        }
    }
    // level 2 -> 1 -> 0 inside lane `base`
    const float a = __shfl_sync(0xffffffffu, x.x, base), bb = __shfl_sync(0xffffffffu, x.y, base);
    const float c = __shfl_sync(0xffffffffu, x.z, base), d = __shfl_sync(0xffffffffu, x.w, base);
    const float s01 = __fadd_rn(a, bb), s23 = __fadd_rn(c, d);
    int leaf;
    if (go_left(tau, acc, s01, s23)) {
        leaf = go_left(tau, acc, a, bb) ? 0 : 1;
    } else {
        acc = __fadd_rn(acc, s01);
        leaf = go_left(tau, acc, c, d) ? 2 : 3;
    }
    return min(v0 + 4 * base + leaf, V - 1);
}

// Inverse-CDF draw after full_pass(vals): returns the token in the CTA that
// owns the chosen block (and -1 elsewhere).  All threads of all CTAs call it.
template <int kC, class Vals>
__device__ int tree_descent(const Vals& vals, int V, float total, float u, PassSmem& sm,
                            cg::cluster_group& cluster, unsigned int* err) {
    const int rank = static_cast<int>(cluster.block_rank());
    const float tau = __fmul_rn(u, total);
    // levels 18 -> 12 over the 64 block sums (every CTA reaches the same block)
    if ((threadIdx.x >> 5) == 0) build_levels(sm.bsum, kMaxBlocks, sm.tree);
    __syncthreads();
    if (threadIdx.x == 0) {
        float acc = 0.0f;
        sm.node = descend_levels(sm.tree, kMaxBlocks, tau, acc);
        sm.acc = acc;
    }
    __syncthreads();
    const int blk = sm.node;
    if (!SV_CHECK(blk >= 0 && blk < kMaxBlocks, err, 1)) return -1;
    if (blk % kC != rank) return -1;
    const int lb = blk / kC;
    __syncthreads();
    // levels 12 -> 7 over the block's 32 chunk sums
    if ((threadIdx.x >> 5) == 0) build_levels(sm.csum + lb * kChunksPerBlk, kChunksPerBlk, sm.tree);
    __syncthreads();
    if (threadIdx.x == 0) {
        float acc = sm.acc;
        sm.node = descend_levels(sm.tree, kChunksPerBlk, tau, acc);
        sm.acc = acc;
    }
    __syncthreads();
    const int chunk = sm.node;
    float acc = sm.acc;
    if (!SV_CHECK(chunk >= 0 && chunk < kChunksPerBlk, err, 2)) return -1;
    // levels 7 -> 0 inside the chunk: warp 0 recomputes its 128 leaves
    if ((threadIdx.x >> 5) == 0) {
        const int tokn = descend_chunk(vals, blk * kBlk + chunk * kChunk, V, tau, acc);
        if ((threadIdx.x & 31) == 0) sm.token = tokn;
    }
    __syncthreads();
    return sm.token;
}

template <int kC, int kW>
__global__ void __launch_bounds__(kW * 32, 1) sample_finish_kernel(SampleArgs a) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    __shared__ PassSmem sm;
    __shared__ int par_s[kMaxR];
    __shared__ float Schain[kMaxR];
    __shared__ float rSchain[kMaxR];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int b = blockIdx.x / kC;
    const int R = a.R, V = a.V, Vq = a.Vq;
    if (threadIdx.x < kMaxBlocks) sm.bsum[threadIdx.x] = 0.0f;
    bool tree_ok = true;
    if (a.parent) tree_ok = load_tree(a.parent, b, R, par_s, a.err);
    __syncthreads();
    const int* par = a.parent ? par_s : nullptr;
    const int32_t* tk = a.tok + static_cast<size_t>(b) * R;
    const float* Lb = a.logits + static_cast<size_t>(b) * R * V;
    const float* Qb = a.q + static_cast<size_t>(b) * a.Rq * Vq;
    const float2* st = a.stats + static_cast<size_t>(b) * R;

    int u = 0, depth = 0, token = -1;
    int32_t* pth = a.path + static_cast<size_t>(b) * R;
    for (int guard = 0; guard <= R && token < 0; ++guard) {
        if (!SV_CHECK(u >= 0 && u < R, a.err, 7)) break;
        const float2 ms = st[u];
        RowValues rv{Lb + static_cast<size_t>(u) * V, Qb + static_cast<size_t>(u) * Vq, Vq, a.T, ms.x, ms.y,
                     __frcp_rn(ms.y), Schain, rSchain, 0, false, V, a.err};
        int first = tree_ok ? next_child(par, R, u, -1) : -1;
        if (first < 0) {   // leaf: bonus token from p_u
            rv.Q = nullptr;
            const float tot = full_pass<kC, kW>(rv, V, a.nblk, sm, cluster);
            token = tree_descent<kC>(rv, V, tot, node_uniforms(a.seed, a.step, b, u, a.uniforms, R).y, sm, cluster,
                                     a.err);
            break;
        }
        int accepted = -1, nsteps = 0;
        for (int c = first; c >= 0; c = next_child(par, R, u, c)) {
            const int d = tk[c];
            const bool tok_ok = d >= 0 && d < V;
            if (!tok_ok && threadIdx.x == 0 && rank == 0) raise_error(a.err, SV_DEVERR_TOKEN);
            bool accept = false;
            if (tok_ok) {
                const float qd = d < Vq ? __ldg(rv.Q + d) : 0.0f;
                if (!(qd >= 0.0f) && threadIdx.x == 0 && rank == 0) raise_error(a.err, SV_DEVERR_QPROB);
                rv.nsteps = nsteps;
                rv.residual = false;
                const float wd = rv.at(d);
                const float ua = node_uniforms(a.seed, a.step, b, c, a.uniforms, R).x;
                accept = (qd == 0.0f) || (ua < __fdiv_rn(wd, qd));
            }
            if (accept) { accepted = c; break; }
            const bool last = next_child(par, R, u, c) < 0;
            rv.nsteps = nsteps;
            rv.residual = true;
            const float S = full_pass<kC, kW>(rv, V, a.nblk, sm, cluster);
            if (last) {
                const float ur = node_uniforms(a.seed, a.step, b, u, a.uniforms, R).y;
                if (S > 0.0f) {
                    token = tree_descent<kC>(rv, V, S, ur, sm, cluster, a.err);
                } else {
                    rv.residual = false;
                    const float tot = full_pass<kC, kW>(rv, V, a.nblk, sm, cluster);
                    token = tree_descent<kC>(rv, V, tot, ur, sm, cluster, a.err);
                }
                break;
            }
            if (threadIdx.x == 0 && SV_CHECK(nsteps < kMaxR, a.err, 8)) {
                Schain[nsteps] = S;
                rSchain[nsteps] = S > 0.0f ? __frcp_rn(S) : 0.0f;
            }
            __syncthreads();
            ++nsteps;
        }
        if (token >= 0 || accepted < 0) break;
        u = accepted;
        ++depth;
        if (rank == 0 && threadIdx.x == 0 && SV_CHECK(depth < R, a.err, 9)) pth[depth] = u;
    }
    // The owner of the sampled block writes the token; rank 0 the walk.
    if (token >= 0 && threadIdx.x == 0) a.out_tok[b] = token;
    if (rank == 0 && threadIdx.x == 0) {
        pth[0] = 0;
        for (int j = depth + 1; j < R; ++j) pth[j] = -1;
        a.n_acc[b] = depth;
    }
}

// ==========================================================================
// sampled, chain drafts: three launches instead of one walk per cluster
// ==========================================================================
//
// In a chain every ratio test depends only on its own row's statistics, so
// all k tests run at once (one thread per draft) and the first rejection is
// found by a reduction; the one full-vocab pass the round then needs (the
// residual max(0, p - q) of the rejection row, or p of the last row for the
// bonus) is spread over one CTA per (sequence, 4096-block); one warp per
// sequence finally descends the summation tree.  Values, sums, uniforms and
// the descent are those of the cluster walk, term for term.

constexpr int kChainResidual = 0, kChainBonus = 1;
constexpr int kSumFloats = kMaxBlocks * kChunksPerBlk + kMaxBlocks;   // chunk sums then block sums

struct ChainWs {
    int4* rec;       // [B]: row u, mode, -, -
    float* sums;     // [B][2][kSumFloats]: set 0 = residual, set 1 = p
};

__host__ __device__ constexpr size_t chain_ws_bytes(int B) {
    return ((static_cast<size_t>(B) * sizeof(int4) + 255) / 256) * 256 +
           static_cast<size_t>(B) * 2 * kSumFloats * sizeof(float);
}

__global__ void __launch_bounds__(kMaxR) chain_walk_kernel(SampleArgs a, ChainWs w) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    __shared__ int first_rej;
    const int b = blockIdx.x, t = threadIdx.x;
    const int R = a.R, V = a.V, Vq = a.Vq;
    if (t == 0) first_rej = R - 1;
    __syncthreads();
    bool accept = true, tok_bad = false, q_bad = false;
    if (t < R - 1) {   // draft j = t + 1 against row u = t
        const int u = t, d = a.tok[static_cast<size_t>(b) * R + t + 1];
        const float2 ms = a.stats[static_cast<size_t>(b) * R + u];
        RowValues rv{a.logits + (static_cast<size_t>(b) * R + u) * V, a.q + (static_cast<size_t>(b) * (R - 1) + u) * Vq,
                     Vq, a.T, ms.x, ms.y, __frcp_rn(ms.y), nullptr, nullptr, 0, false, V, a.err};
        tok_bad = !(d >= 0 && d < V);
        accept = false;
        if (!tok_bad) {
            const float qd = d < Vq ? __ldg(rv.Q + d) : 0.0f;
            q_bad = !(qd >= 0.0f);
            const float wd = rv.at(d);
            const float ua = node_uniforms(a.seed, a.step, b, t + 1, a.uniforms, R).x;
            accept = (qd == 0.0f) || (ua < __fdiv_rn(wd, qd));
        }
        if (!accept) atomicMin(&first_rej, t);
    }
    __syncthreads();
    const int depth = first_rej;   // drafts 1..depth accepted
    // flags only for the drafts the sequential walk reaches
    if (t < R - 1 && t <= depth) {
        if (tok_bad) raise_error(a.err, SV_DEVERR_TOKEN);
        if (q_bad) raise_error(a.err, SV_DEVERR_QPROB);
    }
    int32_t* pth = a.path + static_cast<size_t>(b) * R;
    for (int j = t; j < R; j += blockDim.x) pth[j] = j <= depth ? j : -1;
    if (t == 0) {
        const bool rejected = depth < R - 1;
        a.n_acc[b] = depth;
        w.rec[b] = make_int4(depth, rejected ? kChainResidual : kChainBonus, 0, 0);
    }
}

// One CTA per (4096-block, sequence): chunk and block sums of the residual and
// of p over the row the walk stopped at.
__global__ void __launch_bounds__(kThreads) chain_sums_kernel(SampleArgs a, ChainWs w) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    const int blk = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int V = a.V, Vq = a.Vq, R = a.R;
    const int4 rc = w.rec[b];
    const int u = rc.x;
    const float2 ms = a.stats[static_cast<size_t>(b) * R + u];
    const float* Qrow = rc.y == kChainResidual ? a.q + (static_cast<size_t>(b) * (R - 1) + u) * Vq : nullptr;
    RowValues rv{a.logits + (static_cast<size_t>(b) * R + u) * V, Qrow, Vq, a.T, ms.x, ms.y, __frcp_rn(ms.y), nullptr,
                 nullptr, 0, false, V, a.err};
    float* sr = w.sums + static_cast<size_t>(b) * 2 * kSumFloats;
    float* sp = sr + kSumFloats;
    __shared__ float cr[kChunksPerBlk], cp[kChunksPerBlk];
    constexpr int kPer = kChunksPerBlk / kWarps;   // chunks per warp
    static_assert(kPer == 4, "four chunks per warp: eight sums per lane");
    typename RowValues::Raw raw[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int v = blk * kBlk + (warp * kPer + i) * kChunk + 4 * lane;
        raw[i] = v < V ? rv.load4(v)
                       : typename RowValues::Raw{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    }
    // d = z - M of the warp's 16 leaves per lane; the normal-range form of the
    // exponential when all of them allow it (uniform over the warp; NaN: no)
    float4 d[kPer];
    float dmin = INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int v = blk * kBlk + (warp * kPer + i) * kChunk + 4 * lane;
        const float4 l = raw[i].l;
        const float4 z = a.T == 1.0f ? l : make_float4(__fdiv_rn(l.x, a.T), __fdiv_rn(l.y, a.T), __fdiv_rn(l.z, a.T),
                                                         __fdiv_rn(l.w, a.T));
        d[i] = make_float4(__fsub_rn(z.x, ms.x), __fsub_rn(z.y, ms.x), __fsub_rn(z.z, ms.x), __fsub_rn(z.w, ms.x));
        if (v < V) dmin = fmin_nan(dmin, fmin3_nan(d[i].x, d[i].y, fmin_nan(d[i].z, d[i].w)));
    }
    const bool nrm = __all_sync(0xffffffffu, dmin > kExpNormalMin);
    // p = exp(z - M) / Z and the residual max(0, p - q) (the same operations
    // as RowValues::one without sibling steps), then each lane's node over its
    // 4 leaves of each chunk: sums 0-3 the residual's chunks, 4-7 p's
    float sv8[2 * kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int v = blk * kBlk + (warp * kPer + i) * kChunk + 4 * lane;
        float4 p = make_float4(0.f, 0.f, 0.f, 0.f), r = p;
        if (v < V) {
            auto ex = [&](float x) { return nrm ? sv_exp_nrm(x) : sv_exp_nb(x); };
            p = make_float4(div_rn_by(ex(d[i].x), ms.y, rv.rZ), div_rn_by(ex(d[i].y), ms.y, rv.rZ),
                            div_rn_by(ex(d[i].z), ms.y, rv.rZ), div_rn_by(ex(d[i].w), ms.y, rv.rZ));
            auto res = [](float w, float qv) {   // RowValues::one with residual: max(0, w - q)
                const float dd = __fsub_rn(w, qv);
                return dd > 0.0f ? dd : 0.0f;
            };
            r = make_float4(res(p.x, raw[i].q.x), res(p.y, raw[i].q.y), res(p.z, raw[i].q.z), res(p.w, raw[i].q.w));
        }
        sv8[i] = quad_sum(r);
        sv8[kPer + i] = quad_sum(p);
    }
    // the 32 lanes' trees of all eight sums at once: at each of the first
    // three levels a lane keeps half of its sums and trades the other half
    // with its partner (lanes l ^ 1, l ^ 2, l ^ 4), so lane l ends with sum
    // l % 8; every node is still its two children's sum
    const bool h1 = (lane & 1) != 0, h2 = (lane & 2) != 0, h4 = (lane & 4) != 0;
    float w4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w4[j] = __fadd_rn(h1 ? sv8[2 * j + 1] : sv8[2 * j],
                          __shfl_xor_sync(0xffffffffu, h1 ? sv8[2 * j] : sv8[2 * j + 1], 1));
    float w2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
        w2[j] = __fadd_rn(h2 ? w4[2 * j + 1] : w4[2 * j],
                          __shfl_xor_sync(0xffffffffu, h2 ? w4[2 * j] : w4[2 * j + 1], 2));
    float t = __fadd_rn(h4 ? w2[1] : w2[0], __shfl_xor_sync(0xffffffffu, h4 ? w2[0] : w2[1], 4));
    t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 8));
    t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 16));
    if (lane < kPer) cr[warp * kPer + lane] = t;
    else if (lane < 2 * kPer) cp[warp * kPer + lane - kPer] = t;
    __syncthreads();
    if (warp == 0) {
        const float br = warp_tree_sum(cr[lane]), bp = warp_tree_sum(cp[lane]);
        sr[blk * kChunksPerBlk + lane] = cr[lane];
        sp[blk * kChunksPerBlk + lane] = cp[lane];
        if (lane == 0) {
            sr[kMaxBlocks * kChunksPerBlk + blk] = br;
            sp[kMaxBlocks * kChunksPerBlk + blk] = bp;
        }
    }
}

// One warp per sequence: totals (levels 13 -> 18), the choice between the
// residual and p, and the descent.
__global__ void __launch_bounds__(32) chain_draw_kernel(SampleArgs a, ChainWs w) {
    pdl_wait();   // inputs come from the kernels before this one
    pdl_launch_dependents();
    __shared__ float bs[kMaxBlocks];
    __shared__ float tree[2 * kMaxBlocks];
    const int b = blockIdx.x, lane = threadIdx.x;
    const int V = a.V, Vq = a.Vq, R = a.R;
    const int4 rc = w.rec[b];
    const int u = rc.x;
    const float* base = w.sums + static_cast<size_t>(b) * 2 * kSumFloats;
    auto block_sum = [&](const float* set, int i) { return i < a.nblk ? set[kMaxBlocks * kChunksPerBlk + i] : 0.0f; };
    const float Sr = warp_tree_sum(__fadd_rn(block_sum(base, 2 * lane), block_sum(base, 2 * lane + 1)));
    const float Sp = warp_tree_sum(__fadd_rn(block_sum(base + kSumFloats, 2 * lane),
                                             block_sum(base + kSumFloats, 2 * lane + 1)));
    // residual when it has mass, else p (also for the bonus)
    const bool use_r = rc.y == kChainResidual && Sr > 0.0f;
    const float* set = use_r ? base : base + kSumFloats;
    const float total = use_r ? Sr : Sp;
    const float2 ms = a.stats[static_cast<size_t>(b) * R + u];
    RowValues rv{a.logits + (static_cast<size_t>(b) * R + u) * V,
                 use_r ? a.q + (static_cast<size_t>(b) * (R - 1) + u) * Vq : nullptr, Vq, a.T, ms.x, ms.y,
                 __frcp_rn(ms.y), nullptr, nullptr, 0, use_r, V, a.err};
    const float tau = __fmul_rn(node_uniforms(a.seed, a.step, b, u, a.uniforms, R).y, total);
    bs[lane] = block_sum(set, lane);
    bs[lane + 32] = block_sum(set, lane + 32);
    __syncwarp();
    build_levels(bs, kMaxBlocks, tree);
    float acc = 0.0f;
    const int blk = descend_levels(tree, kMaxBlocks, tau, acc);
    __syncwarp();
    if (!SV_CHECK(blk >= 0 && blk < a.nblk, a.err, 10)) return;
    build_levels(set + blk * kChunksPerBlk, kChunksPerBlk, tree);
    const int chunk = descend_levels(tree, kChunksPerBlk, tau, acc);
    const int tokn = descend_chunk(rv, blk * kBlk + chunk * kChunk, V, tau, acc);
    if (lane == 0) a.out_tok[b] = tokn;
}

// ==========================================================================
// diagnostics
// ==========================================================================

__global__ void diag_exp_kernel(const float* x, float* y, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    {
        // the branch-free and the normal-range forms used by the softmax
        // passes must agree bit for bit wherever each is defined; a
        // disagreement shows up as 12345
        const float e = sv_exp(x[i]);
        const bool defined = !(x[i] != x[i]) && x[i] <= 0.0f;
        const bool normal = defined && x[i] > kExpNormalMin;
        const bool bad = (defined && __float_as_uint(sv_exp_nb(x[i])) != __float_as_uint(e)) ||
                         (normal && __float_as_uint(sv_exp_nrm(x[i])) != __float_as_uint(e));
        y[i] = bad ? 12345.0f : e;
    }
}

__global__ void diag_philox_kernel(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 c = make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
        const uint4 r = philox4x32_10(c, make_uint2(key[2 * i], key[2 * i + 1]));
        out[4 * i] = r.x;
        out[4 * i + 1] = r.y;
        out[4 * i + 2] = r.z;
        out[4 * i + 3] = r.w;
    }
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    diag_canon_kernel(const float* x, int n, int nblk, const float* u, float* sums, int32_t* draws) {
    __shared__ PassSmem sm;
    cg::cluster_group cluster = cg::this_cluster();
    const int row = blockIdx.x / kCluster;
    if (threadIdx.x < kMaxBlocks) sm.bsum[threadIdx.x] = 0.0f;
    __syncthreads();
    ArrayValues vals{x + static_cast<size_t>(row) * n};
    const float tot = full_pass<kCluster, kWarps>(vals, n, nblk, sm, cluster);
    const int tok = tree_descent<kCluster>(vals, n, tot, u[row], sm, cluster, nullptr);
    if (threadIdx.x == 0 && cluster.block_rank() == 0) sums[row] = tot;
    if (threadIdx.x == 0 && tok >= 0) draws[row] = tok;
}

int blocks_for(int V) { return (V + kBlk - 1) / kBlk; }

// Pairs of statistics CTAs that can be resident at once (a cluster sits in
// one GPC); SMs / 2 when the query fails.
int row_pairs() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    const int fallback = device_sm_count() * kRowCtasPerSm / kRowPair > 0 ? device_sm_count() * kRowCtasPerSm / kRowPair
                                                                            : 1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fallback;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev]) return cache[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kRowPair, 1, 1);
    cfg.blockDim = dim3(kRowThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sample_stats_row_kernel<true>, &cfg) != cudaSuccess) n = 0;
    cudaGetLastError();
    cache[dev] = n > 0 ? n : fallback;
    return cache[dev];
}

}  // namespace

size_t greedy_workspace(int B, int R, int V) {
    const int nchunk = (V + kGreedyChunk - 1) / kGreedyChunk;
    return static_cast<size_t>(B) * R * nchunk * sizeof(int2);
}

cudaError_t launch_accept_greedy(const float* logits, const int32_t* tok, const int32_t* parent, int B, int R,
                                 int V, int32_t* n_acc, int32_t* out_tok, int32_t* path, void* ws,
                                 cudaStream_t st) {
    const int nchunk = (V + kGreedyChunk - 1) / kGreedyChunk;
    int2* part = static_cast<int2*>(ws);
    unsigned int* err = device_error_word();
    cudaError_t e = launch_pdl(greedy_partial_kernel, dim3(nchunk, B * R), dim3(kGreedyThreads), 0, st, logits, V,
                               nchunk, part, err);
    if (e != cudaSuccess) return e;
    e = launch_pdl(greedy_finish_kernel, dim3(B), dim3(128), 0, st, static_cast<const int2*>(part), nchunk, tok, parent,
                   R, V, n_acc, out_tok, path, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Row statistics (B*R float2); then, for the chain path, the per-sequence
// records and summation-tree sums.
constexpr int kWideWalkMaxB = 4;   // sequences up to which the walk takes 16-CTA clusters
#ifndef SV_WIDE_WALK_WARPS
#define SV_WIDE_WALK_WARPS 24
#endif
constexpr int kWideWalkWarps = SV_WIDE_WALK_WARPS;   // warps per CTA of those clusters

template <int kC, int kW>
cudaError_t launch_finish(const SampleArgs& a, int B, cudaStream_t st) {
    static PerDeviceOnce attr_once;
    const cudaError_t ea = attr_once.run([]() {
        return kC > 8 ? cudaFuncSetAttribute(sample_finish_kernel<kC, kW>,
                                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1)
                      : cudaSuccess;
    });
    if (ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B * kC, 1, 1);
    cfg.blockDim = dim3(kW * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = kC;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sample_finish_kernel<kC, kW>, a);
}

static size_t stats_bytes(int B, int R) { return ((static_cast<size_t>(B) * R * sizeof(float2) + 255) / 256) * 256; }
size_t sample_workspace(int B, int R, int /*V*/) { return stats_bytes(B, R) + chain_ws_bytes(B); }

cudaError_t launch_accept_sample(const float* logits, const float* q, int Vq, const int32_t* tok,
                                 const int32_t* parent, int B, int R, int V, float temperature, uint64_t seed,
                                 uint64_t step, const float* uniforms, int32_t* n_acc, int32_t* out_tok,
                                 int32_t* path, void* ws, size_t ws_bytes, cudaStream_t st) {
    unsigned int* err = device_error_word();
    const int nblk = blocks_for(V);
    const int nlocal = (nblk + kCluster - 1) / kCluster;
    const size_t smem = static_cast<size_t>(nlocal) * kBlk * sizeof(float);
    cudaError_t e = cudaSuccess;
    static PerDeviceOnce attr_once;   // per device: the largest row (2^18 entries) fits
    e = attr_once.run([]() {
        return cudaFuncSetAttribute(sample_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kMaxLocalBlocks * kBlk * static_cast<int>(sizeof(float)));
    });
    if (e != cudaSuccess) return e;
    float2* stats = static_cast<float2*>(ws);
    // Few rows: an 8-CTA cluster per row keeps each row's latency short.  Many
    // rows: one CTA per row keeps every SM busy without cluster waves.
    if (static_cast<int64_t>(B) * R >= kRowStatsMinRows)
    {
        const int slots = row_pairs();
        const int nrows = B * R, grid = kRowPair * (nrows < slots ? nrows : slots);
        e = temperature == 1.0f
                ? launch_pdl(sample_stats_row_kernel<true>, dim3(grid), dim3(kRowThreads), 0, st, logits, V, temperature,
                             nblk, nrows, stats, err)
                : launch_pdl(sample_stats_row_kernel<false>, dim3(grid), dim3(kRowThreads), 0, st, logits, V,
                             temperature, nblk, nrows, stats, err);
        if (e != cudaSuccess) return e;
    }
    else
    {
        e = launch_pdl(sample_stats_kernel, dim3(B * R * kCluster), dim3(kThreads), smem, st, logits, V, temperature, nblk,
                       nlocal, stats, err);
        if (e != cudaSuccess) return e;
    }
    if (debug_sync()) {
        e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return e;
    }
    SampleArgs a;
    a.logits = logits;
    a.q = q;
    a.tok = tok;
    a.parent = parent;
    a.stats = stats;
    a.uniforms = uniforms;
    a.n_acc = n_acc;
    a.out_tok = out_tok;
    a.path = path;
    a.err = err;
    a.seed = seed;
    a.step = step;
    a.R = R;
    a.Rq = parent ? R : R - 1;
    a.V = V;
    a.Vq = Vq;
    a.nblk = nblk;
    a.T = temperature;
    if (parent == nullptr && ws_bytes >= sample_workspace(B, R, V)) {
        // chain: parallel ratio tests, one full-vocab pass over the whole GPU
        ChainWs w;
        w.rec = reinterpret_cast<int4*>(static_cast<uint8_t*>(ws) + stats_bytes(B, R));
        w.sums = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + stats_bytes(B, R) +
                                          ((static_cast<size_t>(B) * sizeof(int4) + 255) / 256) * 256);
        e = launch_pdl(chain_walk_kernel, dim3(B), dim3(kMaxR), 0, st, a, w);
        if (e != cudaSuccess) return e;
        e = launch_pdl(chain_sums_kernel, dim3(nblk, B), dim3(kThreads), 0, st, a, w);
        if (e != cudaSuccess) return e;
        e = launch_pdl(chain_draw_kernel, dim3(B), dim3(32), 0, st, a, w);
        if (e != cudaSuccess) return e;
    } else {
        // trees (sibling residuals depend on each other), or a workspace that
        // only holds the row statistics: one cluster walks each sequence.  Its
        // passes evaluate the exponential, the division by Z and one division
        // per rejected sibling for every vocab entry on the cluster's SMs, so a
        // few sequences take 16-CTA clusters of 768 threads (the 64-node tree's
        // acceptance 167 -> 86 us against 8 x 256; 512 threads 92 us, 1024
        // spill); many sequences keep 8 x 256 (more clusters resident at once)
        e = B <= kWideWalkMaxB ? launch_finish<16, kWideWalkWarps>(a, B, st) : launch_finish<kCluster, kWarps>(a, B, st);
        if (e != cudaSuccess) return e;
    }
    if (debug_sync()) {
        e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

// the acceptance's division by a per-divisor reciprocal
__global__ void diag_div_kernel(const float* a, const float* b, float* q, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        q[i] = div_rn_by(a[i], b[i], __frcp_rn(b[i]));
}

cudaError_t launch_diag_div(const float* a, const float* b, float* q, int64_t n, cudaStream_t st) {
    const int64_t blocks = (n + 255) / 256;
    diag_div_kernel<<<static_cast<int>(blocks > 65535 ? 65535 : (blocks < 1 ? 1 : blocks)), 256, 0, st>>>(a, b, q, n);
    return cudaGetLastError();
}

cudaError_t launch_diag_exp(const float* x, float* y, int64_t n, cudaStream_t st) {
    const int64_t blocks = (n + 255) / 256;
    diag_exp_kernel<<<static_cast<int>(blocks > 65535 ? 65535 : (blocks < 1 ? 1 : blocks)), 256, 0, st>>>(x, y, n);
    return cudaGetLastError();
}

cudaError_t launch_diag_philox(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int64_t n,
                               cudaStream_t st) {
    const int64_t blocks = (n + 255) / 256;
    diag_philox_kernel<<<static_cast<int>(blocks > 65535 ? 65535 : (blocks < 1 ? 1 : blocks)), 256, 0, st>>>(
        ctr, key, out, n);
    return cudaGetLastError();
}

cudaError_t launch_diag_canon(const float* x, int n, int m, const float* u, float* sums, int32_t* draws,
                              cudaStream_t st) {
    diag_canon_kernel<<<m * kCluster, kThreads, 0, st>>>(x, n, blocks_for(n), u, sums, draws);
    return cudaGetLastError();
}

}  // namespace sv
