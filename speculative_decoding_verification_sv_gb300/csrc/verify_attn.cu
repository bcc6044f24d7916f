// verify_attn.cu -- attention of the k+1 verify rows over the committed KV
// cache and the block's own K/V.
//
// [SpecDec-Context-Scaling guide, sec. 3]: the target runs one forward over
// the block and row j sees the committed prefix plus block rows 0..j;
// [wmrh.cn tutorial, sec. 3.2]: causal attention makes that one pass give all
// positions at once; [SubSpec summary, sec. 4.2]: for a draft tree row j sees
// its ancestors instead.
//
// Decomposition: for every (sequence b, KV head g) the R*G query rows of the
// G query heads that share g are packed together (row r = j*G + local head),
// so each K/V tile streamed from HBM serves all of them (GQA).  The context
// is split into `splits` equal chunks (flash-decoding style split-KV, sized
// so the grid covers the SMs); one extra split handles the R block rows with
// the chain or tree mask.  Each CTA:
//   * streams 64-key K and V tiles through a TMA (cp.async.bulk.tensor, 128B
//     swizzle) ring of mbarrier-tracked stages;
//   * computes S = Q K^T and O += P V on the tensor cores (mma.sync bf16,
//     fp32 accumulate; Q fragments stay in registers for the whole split);
//   * keeps an online softmax per row in registers (quad shuffles);
//   * writes its unnormalised partial (max, sum, o) to the workspace.
// attn_combine_kernel merges the splits of every row and rounds to bf16.
#include <math.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kD = 128;
constexpr int kKT = 64;                  // keys per tile
constexpr int kStages = 3;
constexpr int kTileBytes = kKT * kD * 2; // 16 KB: two 64x64 swizzled boxes
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kRec = kD + 4;             // partial record: m, l, 2 pad, o[128] (16-byte aligned)
constexpr int kMaxR = 128;
constexpr int kSmemBytes = kStages * kStageBytes + kStages * 8 + kMaxR * 16 + 1024;

struct AttnArgs {
    const uint16_t* q;
    const int32_t* len;
    const int32_t* parent;
    float* part;
    unsigned int* err;
    int B, R, Hq, Hkv, G, T_cap, rows, row_tiles, splits;
    float scale_log2;
};

__global__ void __launch_bounds__(128) attn_split_kernel(const __grid_constant__ CUtensorMap tmK,
                                                        const __grid_constant__ CUtensorMap tmV,
                                                        const __grid_constant__ CUtensorMap tmKb,
                                                        const __grid_constant__ CUtensorMap tmVb, AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* anc = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kStages * 8);   // [kMaxR][2]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, hg = blockIdx.y, rt = blockIdx.z;
    const int b = hg / a.Hkv, g = hg % a.Hkv;
    const bool is_block = split == a.splits;

    int t = a.len[b];
    if (t < 0 || t > a.T_cap) {
        if (tid == 0 && split == 0 && rt == 0 && g == 0) raise_error(a.err, SV_DEVERR_LENGTH);
        t = t < 0 ? 0 : a.T_cap;
    }
    int k_begin, nkeys;
    const void* tk;
    const void* tv;
    int row0;
    if (!is_block) {
        int chunk = (t + a.splits - 1) / a.splits;
        chunk = ((chunk + kKT - 1) / kKT) * kKT;
        if (chunk < kKT) chunk = kKT;
        k_begin = split * chunk;
        const int k_end = min(t, k_begin + chunk);
        nkeys = k_end > k_begin ? k_end - k_begin : 0;
        tk = &tmK;
        tv = &tmV;
        row0 = hg * a.T_cap + k_begin;
    } else {
        k_begin = 0;
        nkeys = a.R;
        tk = &tmKb;
        tv = &tmVb;
        row0 = hg * a.R;
    }
    const int ntiles = (nkeys + kKT - 1) / kKT;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    // tree ancestor masks (block split only): bit i of anc[j] set iff block
    // row i is j itself or one of its ancestors
    if (is_block && a.parent) {
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

    auto issue = [&](int it) {
        const int s = it % kStages;
        uint8_t* st = smem + s * kStageBytes;
        const int y = row0 + it * kKT;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        tma_load_2d(st, tk, 0, y, &full[s]);
        tma_load_2d(st + kKT * 128, tk, 64, y, &full[s]);
        tma_load_2d(st + kTileBytes, tv, 0, y, &full[s]);
        tma_load_2d(st + kTileBytes + kKT * 128, tv, 64, y, &full[s]);
    };
    if (tid == 0)
        for (int it = 0; it < ntiles && it < kStages; ++it) issue(it);

    // rows owned by this warp: ra = rb + lane/4 and rb_ = ra + 8
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

    const uint64_t anc_a0 = (is_block && a.parent && ra < a.rows) ? anc[2 * ja] : 0;
    const uint64_t anc_a1 = (is_block && a.parent && ra < a.rows) ? anc[2 * ja + 1] : 0;
    const uint64_t anc_b0 = (is_block && a.parent && rb < a.rows) ? anc[2 * jb] : 0;
    const uint64_t anc_b1 = (is_block && a.parent && rb < a.rows) ? anc[2 * jb + 1] : 0;

    for (int it = 0; it < ntiles; ++it) {
        const int s = it % kStages;
        mbar_wait(&full[s], (it / kStages) & 1, a.err);
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
                    const int kl = it * kKT + nt * 8 + 2 * (lane & 3) + (e & 1);
                    const bool row_a = e < 2;
                    bool vis;
                    if (!is_block) {
                        vis = kl < nkeys;
                    } else if (kl >= a.R) {
                        vis = false;
                    } else if (a.parent) {
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

    if (!active) return;
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    const int nsplit = a.splits + 1;
    const size_t rows_pad = static_cast<size_t>(a.row_tiles) * 64;
    if (ra < a.rows) {
        float* rec = a.part + ((static_cast<size_t>(hg) * rows_pad + ra) * nsplit + split) * kRec;
        if ((lane & 3) == 0) {
            rec[0] = m_a;
            rec[1] = l_a;
        }
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
            *reinterpret_cast<float2*>(rec + 4 + dt * 8 + 2 * (lane & 3)) = make_float2(o[dt][0], o[dt][1]);
    }
    if (rb < a.rows) {
        float* rec = a.part + ((static_cast<size_t>(hg) * rows_pad + rb) * nsplit + split) * kRec;
        if ((lane & 3) == 0) {
            rec[0] = m_b;
            rec[1] = l_b;
        }
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
            *reinterpret_cast<float2*>(rec + 4 + dt * 8 + 2 * (lane & 3)) = make_float2(o[dt][2], o[dt][3]);
    }
}

// One warp per (sequence, KV head, row): merge the splits, normalise, round.
__global__ void __launch_bounds__(128) attn_combine_kernel(const float* __restrict__ part, uint16_t* __restrict__ out,
                                                          int B, int R, int Hq, int Hkv, int G, int rows,
                                                          int row_tiles, int nsplit) {
    const int wid = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (wid >= B * Hkv * rows) return;
    const int hg = wid / rows, r = wid % rows;
    const int b = hg / Hkv, g = hg % Hkv;
    const float* rec0 = part + (static_cast<size_t>(hg) * row_tiles * 64 + r) * nsplit * kRec;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, rec0[s * kRec]);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
        for (int s = 0; s < nsplit; ++s) {
            const float* rec = rec0 + s * kRec;
            const float l = rec[1];
            if (l == 0.f) continue;
            const float w = exp2f(rec[0] - M);
            L += l * w;
            const float4 x = *reinterpret_cast<const float4*>(rec + 4 + 4 * lane);
            acc.x += w * x.x;
            acc.y += w * x.y;
            acc.z += w * x.z;
            acc.w += w * x.w;
        }
    }
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    const int j = r / G, h = g * G + r % G;
    uint16_t* dst = out + ((static_cast<size_t>(b) * R + j) * Hq + h) * kD + 4 * lane;
    const uint32_t lo = pack_bf16x2(acc.x * inv, acc.y * inv), hi = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
}

}  // namespace

AttnPlan attn_plan(const sv_attn_shape& s) {
    AttnPlan p;
    p.G = s.Hq / s.Hkv;
    p.rows = s.R * p.G;
    p.row_tiles = (p.rows + 63) / 64;
    p.warps = p.row_tiles > 1 ? 4 : (p.rows + 15) / 16;
    const int units = s.B * s.Hkv * p.row_tiles;
    const int target = 2 * device_sm_count();
    int splits = (target + units - 1) / units;
    const int max_splits = (s.T_cap + kKT - 1) / kKT;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    p.splits = splits;
    return p;
}

size_t attn_workspace(const sv_attn_shape& s) {
    const AttnPlan p = attn_plan(s);
    return static_cast<size_t>(s.B) * s.Hkv * p.row_tiles * 64 * (p.splits + 1) * kRec * sizeof(float);
}

cudaError_t launch_verify_attn(const sv_attn_shape& s, const uint16_t* q, const uint16_t* k_cache,
                               const uint16_t* v_cache, const int32_t* len, const uint16_t* k_blk,
                               const uint16_t* v_blk, const int32_t* parent, float scale, uint16_t* out,
                               void* ws, cudaStream_t st) {
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
        cudaError_t e = cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    AttnArgs a;
    a.q = q;
    a.len = len;
    a.parent = parent;
    a.part = static_cast<float*>(ws);
    a.err = device_error_word();
    a.B = s.B;
    a.R = s.R;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.G = p.G;
    a.T_cap = s.T_cap;
    a.rows = p.rows;
    a.row_tiles = p.row_tiles;
    a.splits = p.splits;
    a.scale_log2 = scale * 1.4426950408889634f;
    dim3 grid(p.splits + 1, s.B * s.Hkv, p.row_tiles);
    attn_split_kernel<<<grid, 32 * p.warps, kSmemBytes, st>>>(
        *reinterpret_cast<const CUtensorMap*>(tK), *reinterpret_cast<const CUtensorMap*>(tV),
        *reinterpret_cast<const CUtensorMap*>(tKb), *reinterpret_cast<const CUtensorMap*>(tVb), a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int nwarps = s.B * s.Hkv * p.rows;
    attn_combine_kernel<<<(nwarps + 3) / 4, 128, 0, st>>>(static_cast<const float*>(ws), out, s.B, s.R, s.Hq, s.Hkv,
                                                           p.G, p.rows, p.row_tiles, p.splits + 1);
    return cudaGetLastError();
}

}  // namespace sv
