// verify_attn.cu -- attention of the k+1 verify rows over the committed KV
// cache and the block's own K/V.
//
// [SpecDec-Context-Scaling guide, sec. 3]: the target runs one forward over
// the block and row j sees the committed prefix plus block rows 0..j;
// [wmrh.cn tutorial, sec. 3.2]: causal attention makes that one pass give all
// positions at once; [SubSpec summary, sec. 4.2]: for a draft tree row j sees
// its ancestors instead.
//
// Decomposition.  For every (sequence b, KV head g) the R*G query rows of the
// G query heads that share g are packed together (row r = j*G + local head),
// so each K/V tile streamed from HBM serves all of them (GQA); rows are cut
// into tiles of 64.  One thread-block cluster of C CTAs (C up to 16) handles
// one (b, g, row tile): the key tiles -- ceil(t/64) context tiles followed by
// ceil(R/64) block tiles -- are split evenly over the C CTAs (split-KV over the
// context, sized so the grid fills the SMs).  Each CTA:
//   * streams 64-key K and V tiles through a TMA (cp.async.bulk.tensor, 128B
//     swizzle) ring of mbarrier-tracked stages;
//   * computes S = Q K^T and O += P V on the tensor cores (mma.sync bf16,
//     fp32 accumulate; Q fragments stay in registers);
//   * keeps an online softmax per row in registers (quad shuffles);
//   * leaves its unnormalised partial (max, sum, o[128]) in shared memory.
// The cluster then merges the C partials of every row through distributed
// shared memory (each CTA merges every C-th row) and writes bf16 rows.  No
// partial goes through global memory and there is no second kernel.
//
// Launch: programmatic dependent launch -- the CTA prologue (barrier set-up,
// descriptor prefetch) overlaps the previous kernel; everything the previous
// kernels may have written (lengths, cache rows, Q, block K/V, tree) is read
// only after griddepcontrol.wait.
#include <cooperative_groups.h>
#include <math.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kD = 128;
constexpr int kKT = 64;                  // keys per tile
constexpr int kStages = 3;
constexpr int kTileBytes = kKT * kD * 2; // 16 KB: two 64x64 swizzled boxes
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kRec = kD + 4;             // partial record: m, l, 2 pad, o[128] (16-byte aligned)
constexpr int kMaxR = 128;
constexpr int kMaxCluster = 16;
constexpr int kSmemBytes = kStages * kStageBytes + kStages * 8 + kMaxR * 16 + 1024;
static_assert(64 * kRec * 4 <= kStages * kStageBytes, "partials reuse the stage ring");

struct AttnArgs {
    const uint16_t* q;
    const int32_t* len;
    const int32_t* parent;
    uint16_t* out;
    unsigned int* err;
    int B, R, Hq, Hkv, G, T_cap, rows, row_tiles;
    float scale_log2;
};

__global__ void __launch_bounds__(128) attn_cluster_kernel(const __grid_constant__ CUtensorMap tmK,
                                                          const __grid_constant__ CUtensorMap tmV,
                                                          const __grid_constant__ CUtensorMap tmKb,
                                                          const __grid_constant__ CUtensorMap tmVb, AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* anc = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kStages * 8);   // [kMaxR][2]
    float* part = reinterpret_cast<float*>(smem);                                              // [64][kRec] after the loop

    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwarps = blockDim.x >> 5;
    const int hg = blockIdx.y, rt = blockIdx.z;
    const int b = hg / a.Hkv, g = hg % a.Hkv;

    if (tid == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmKb);
        prefetch_tmap(&tmVb);
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    // Inputs may come from the kernels before this one.
    pdl_wait();
    pdl_launch_dependents();

    int t = a.len[b];
    if (t < 0 || t > a.T_cap) {
        if (tid == 0 && rank == 0 && rt == 0) raise_error(a.err, SV_DEVERR_LENGTH);
        t = t < 0 ? 0 : a.T_cap;
    }
    const int n_ctx = (t + kKT - 1) / kKT;
    const int n_blk = (a.R + kKT - 1) / kKT;
    const int n_all = n_ctx + n_blk;
    const int first = static_cast<int>((static_cast<int64_t>(n_all) * rank) / C);
    const int last = static_cast<int>((static_cast<int64_t>(n_all) * (rank + 1)) / C);
    const int ntiles = last - first;

    // tree ancestor masks: bit i of anc[j] set iff block row i is j or one of
    // its ancestors (only CTAs that own a block tile need them)
    const bool has_block = last > n_ctx;
    if (has_block && a.parent) {
        const int32_t* par = a.parent + static_cast<size_t>(b) * a.R;
        for (int j = tid; j < a.R; j += blockDim.x) {
            uint64_t m0 = 0, m1 = 0;
            int i = j;
            bool bad = false;
            for (int steps = 0; steps <= a.R && i >= 0; ++steps) {
                if (i < 64) m0 |= 1ull << i; else m1 |= 1ull << (i - 64);
                const int p = par[i];
                if ((i == 0 && p != -1) || (i > 0 && (p < 0 || p >= i))) { bad = true; break; }
                i = p;
            }
            if (bad) {
                raise_error(a.err, SV_DEVERR_TREE);
                m0 = j < 64 ? 1ull << j : 0;
                m1 = j >= 64 ? 1ull << (j - 64) : 0;
            }
            anc[2 * j] = m0;
            anc[2 * j + 1] = m1;
        }
    }
    __syncthreads();

    auto issue = [&](int i) {
        const int s = i % kStages;
        const int gt = first + i;
        uint8_t* st = smem + s * kStageBytes;
        const void* tk = gt < n_ctx ? static_cast<const void*>(&tmK) : static_cast<const void*>(&tmKb);
        const void* tv = gt < n_ctx ? static_cast<const void*>(&tmV) : static_cast<const void*>(&tmVb);
        const int y = gt < n_ctx ? hg * a.T_cap + gt * kKT : hg * a.R + (gt - n_ctx) * kKT;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tma_load_2d(st, tk, 0, y, &full[s]);
        tma_load_2d(st + kKT * 128, tk, 64, y, &full[s]);
        tma_load_2d(st + kTileBytes, tv, 0, y, &full[s]);
        tma_load_2d(st + kTileBytes + kKT * 128, tv, 64, y, &full[s]);
    };
    if (tid == 0)
        for (int i = 0; i < ntiles && i < kStages; ++i) issue(i);

    // rows owned by this warp: ra = rbase + lane/4 and rb = ra + 8
    const int rbase = rt * 64 + warp * 16;
    const bool active = rbase < a.rows;
    const int ra = rbase + (lane >> 2), rb = ra + 8;
    const int ja = ra / a.G, jb = rb / a.G;
    uint32_t qa[8][4];
    {
        const uint16_t* pa = nullptr;
        const uint16_t* pb = nullptr;
        if (ra < a.rows) pa = a.q + ((static_cast<size_t>(b) * a.R + ja) * a.Hq + g * a.G + ra % a.G) * kD;
        if (rb < a.rows) pb = a.q + ((static_cast<size_t>(b) * a.R + jb) * a.Hq + g * a.G + rb % a.G) * kD;
        const int c = 2 * (lane & 3);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = pa ? __ldg(reinterpret_cast<const uint32_t*>(pa + ks * 16 + c)) : 0u;
            qa[ks][1] = pb ? __ldg(reinterpret_cast<const uint32_t*>(pb + ks * 16 + c)) : 0u;
            qa[ks][2] = pa ? __ldg(reinterpret_cast<const uint32_t*>(pa + ks * 16 + 8 + c)) : 0u;
            qa[ks][3] = pb ? __ldg(reinterpret_cast<const uint32_t*>(pb + ks * 16 + 8 + c)) : 0u;
        }
    }
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][e] = 0.f;

    const bool tree = a.parent != nullptr && has_block;
    const uint64_t anc_a0 = (tree && ra < a.rows) ? anc[2 * ja] : 0;
    const uint64_t anc_a1 = (tree && ra < a.rows) ? anc[2 * ja + 1] : 0;
    const uint64_t anc_b0 = (tree && rb < a.rows) ? anc[2 * jb] : 0;
    const uint64_t anc_b1 = (tree && rb < a.rows) ? anc[2 * jb + 1] : 0;

    for (int it = 0; it < ntiles; ++it) {
        const int s = it % kStages;
        mbar_wait(&full[s], (it / kStages) & 1, a.err);
        const int gt = first + it;
        const bool is_block = gt >= n_ctx;
        const int k0 = is_block ? (gt - n_ctx) * kKT : gt * kKT;   // first key of the tile
        if (active) {
            const uint32_t kbase = smem_u32(smem + s * kStageBytes);
            const uint32_t vbase = kbase + kTileBytes;
            float sc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t box = kbase + (ks >> 2) * (kKT * 128);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    const int chunk = ((2 * ks) & 7) + ((lane >> 3) & 1);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(swz128(box, key, chunk), r0, r1, r2, r3);
                    mma_bf16(sc[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], r0, r1);
                    mma_bf16(sc[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], r2, r3);
                }
            }
            // scale, mask, tile max
            float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kl = k0 + nt * 8 + 2 * (lane & 3) + (e & 1);
                    const bool row_a = e < 2;
                    bool vis;
                    if (!is_block) {
                        vis = kl < t;
                    } else if (kl >= a.R) {
                        vis = false;
                    } else if (tree) {
                        const uint64_t w = kl < 64 ? (row_a ? anc_a0 : anc_b0) : (row_a ? anc_a1 : anc_b1);
                        vis = (w >> (kl & 63)) & 1ull;
                    } else {
                        vis = kl <= (row_a ? ja : jb);
                    }
                    const float v = vis ? sc[nt][e] * a.scale_log2 : -INFINITY;
                    sc[nt][e] = v;
                    if (row_a) mx_a = fmaxf(mx_a, v); else mx_b = fmaxf(mx_b, v);
                }
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
            const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
            const float base_a = mn_a == -INFINITY ? 0.f : mn_a;
            const float base_b = mn_b == -INFINITY ? 0.f : mn_b;
            const float corr_a = fast_exp2(m_a - base_a), corr_b = fast_exp2(m_b - base_b);
            m_a = mn_a;
            m_b = mn_b;
            float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                sc[nt][0] = fast_exp2(sc[nt][0] - base_a);
                sc[nt][1] = fast_exp2(sc[nt][1] - base_a);
                sc[nt][2] = fast_exp2(sc[nt][2] - base_b);
                sc[nt][3] = fast_exp2(sc[nt][3] - base_b);
                sum_a += sc[nt][0] + sc[nt][1];
                sum_b += sc[nt][2] + sc[nt][3];
            }
            l_a = l_a * corr_a + sum_a;
            l_b = l_b * corr_b + sum_b;
#pragma unroll
            for (int dt = 0; dt < 16; ++dt) {
                o[dt][0] *= corr_a;
                o[dt][1] *= corr_a;
                o[dt][2] *= corr_b;
                o[dt][3] *= corr_b;
            }
            // O += P V
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t p0 = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
                const uint32_t p1 = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
                const uint32_t p2 = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
                const uint32_t p3 = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
                const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                for (int dp = 0; dp < 8; ++dp) {
                    const int dchunk = 2 * dp + (lane >> 4);
                    const uint32_t box = vbase + (dchunk >> 3) * (kKT * 128);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(swz128(box, key, dchunk & 7), r0, r1, r2, r3);
                    mma_bf16(o[2 * dp], p0, p1, p2, p3, r0, r1);
                    mma_bf16(o[2 * dp + 1], p0, p1, p2, p3, r2, r3);
                }
            }
        }
        __syncthreads();   // stage s consumed by every warp
        if (tid == 0 && it + kStages < ntiles) issue(it + kStages);
    }

    // this CTA's partial -> shared memory (the stage ring is free now)
    if (active) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
        float* rec_a = part + (ra - rt * 64) * kRec;
        float* rec_b = part + (rb - rt * 64) * kRec;
        if ((lane & 3) == 0) {
            rec_a[0] = m_a;
            rec_a[1] = l_a;
            rec_b[0] = m_b;
            rec_b[1] = l_b;
        }
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            *reinterpret_cast<float2*>(rec_a + 4 + dt * 8 + 2 * (lane & 3)) = make_float2(o[dt][0], o[dt][1]);
            *reinterpret_cast<float2*>(rec_b + 4 + dt * 8 + 2 * (lane & 3)) = make_float2(o[dt][2], o[dt][3]);
        }
    }
    cluster.sync();   // all partials written (and every CTA of the cluster has started)

    // merge: this CTA finalises rows rank, rank + C, ... of the row tile
    const int nrows = min(64, a.rows - rt * 64);
    for (int lr = rank + C * warp; lr < nrows; lr += C * nwarps) {
        float ms = -INFINITY, ls = 0.f;
        const float* rec_s = nullptr;
        if (lane < C) {
            rec_s = cluster.map_shared_rank(part + lr * kRec, lane);
            ms = rec_s[0];
            ls = rec_s[1];
        }
        float M = ms;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float wgt = (lane < C && ls > 0.f && M != -INFINITY) ? exp2f(ms - M) : 0.f;
        float L = wgt * ls;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < C; ++s) {
            const float ws = __shfl_sync(0xffffffffu, wgt, s);
            if (ws == 0.f) continue;
            const float4 x = *reinterpret_cast<const float4*>(cluster.map_shared_rank(part + lr * kRec + 4, s) + 4 * lane);
            acc.x += ws * x.x;
            acc.y += ws * x.y;
            acc.z += ws * x.z;
            acc.w += ws * x.w;
        }
        const float inv = L > 0.f ? 1.0f / L : 0.f;
        const int r = rt * 64 + lr;
        const int j = r / a.G, h = g * a.G + r % a.G;
        uint16_t* dst = a.out + ((static_cast<size_t>(b) * a.R + j) * a.Hq + h) * kD + 4 * lane;
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
    cluster.sync();   // no CTA leaves while its partials may still be read
}

}  // namespace

AttnPlan attn_plan(const sv_attn_shape& s) {
    AttnPlan p;
    p.G = s.Hq / s.Hkv;
    p.rows = s.R * p.G;
    p.row_tiles = (p.rows + 63) / 64;
    p.warps = p.row_tiles > 1 ? 4 : (p.rows + 15) / 16;
    // cluster size: grow while the grid still fits in two CTAs per SM and
    // every CTA keeps at least one key tile
    const int units = s.B * s.Hkv * p.row_tiles;
    const int slots = 2 * device_sm_count();
    const int tiles = (s.T_cap + kKT - 1) / kKT + (s.R + kKT - 1) / kKT;
    int C = 1;
    while (C < kMaxCluster && units * C * 2 <= slots && C * 2 <= tiles) C *= 2;
    p.splits = C;
    return p;
}

size_t attn_workspace(const sv_attn_shape&) { return 0; }

cudaError_t launch_verify_attn(const sv_attn_shape& s, const uint16_t* q, const uint16_t* k_cache,
                               const uint16_t* v_cache, const int32_t* len, const uint16_t* k_blk,
                               const uint16_t* v_blk, const int32_t* parent, float scale, uint16_t* out,
                               void* /*ws*/, cudaStream_t st) {
    const AttnPlan p = attn_plan(s);
    alignas(64) uint8_t tK[128], tV[128], tKb[128], tVb[128];
    const uint64_t ctx_rows = static_cast<uint64_t>(s.B) * s.Hkv * s.T_cap;
    const uint64_t blk_rows = static_cast<uint64_t>(s.B) * s.Hkv * s.R;
    if (!encode_tmap_2d_bf16(tK, k_cache, kD, ctx_rows, kD * 2, 64, kKT) ||
        !encode_tmap_2d_bf16(tV, v_cache, kD, ctx_rows, kD * 2, 64, kKT) ||
        !encode_tmap_2d_bf16(tKb, k_blk, kD, blk_rows, kD * 2, 64, kKT) ||
        !encode_tmap_2d_bf16(tVb, v_blk, kD, blk_rows, kD * 2, 64, kKT))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    AttnArgs a;
    a.q = q;
    a.len = len;
    a.parent = parent;
    a.out = out;
    a.err = device_error_word();
    a.B = s.B;
    a.R = s.R;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.G = p.G;
    a.T_cap = s.T_cap;
    a.rows = p.rows;
    a.row_tiles = p.row_tiles;
    a.scale_log2 = scale * 1.4426950408889634f;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.splits, s.B * s.Hkv, p.row_tiles);
    cfg.blockDim = dim3(32 * p.warps, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = p.splits;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, attn_cluster_kernel, *reinterpret_cast<const CUtensorMap*>(tK),
                              *reinterpret_cast<const CUtensorMap*>(tV), *reinterpret_cast<const CUtensorMap*>(tKb),
                              *reinterpret_cast<const CUtensorMap*>(tVb), a);
}

}  // namespace sv
