// verify_attn.cu -- attention of the k+1 verify rows over the committed KV
// cache and the block's own K/V, on the 5th-generation tensor cores.
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
// into tiles of 128, the MMA's M.  One thread-block cluster of C CTAs (C up
// to 16) handles one (b, g, row tile): the 64-key tiles -- ceil(t/64) context
// tiles followed by ceil(R/64) block tiles -- are split evenly over its CTAs
// (split-KV, sized so the grid fills the SMs).  Inside a CTA, keys are
// processed one 64-key tile per step:
//   * warp 16 streams K and V tiles through a TMA ring (cp.async.bulk.tensor,
//     128-byte swizzle, full/empty mbarriers);
//   * one thread of warp 17 issues tcgen05.mma: S = Q K^T into one of two
//     64-column TMEM score buffers (A = Q K-major, B = K tile K-major), and
//     O += P V into a TMEM accumulator (A = P K-major from one of two shared
//     P buffers, B = V tile MN-major), releasing stages and buffers with
//     tcgen05.commit; S of step st+1 is issued before P V of step st, so the
//     score MMAs run under the softmax;
//   * sixteen row-owner warps: warp w reads TMEM lanes 32*(w%4).. (one query
//     row per thread) and the 16-score column group w/4 of each step; the four
//     threads of a row exchange their partial maxima through shared memory,
//     apply the chain/tree/length mask, keep the running max and sum, write P
//     (bf16) to shared memory, and rescale their part of the row of O in TMEM
//     only when the max has grown by more than 2^8 since it was last used
//     (otherwise the stale max keeps every P <= 256, exact in fp32).  Warps
//     whose 32 rows are all padding skip the arithmetic;
//   * at the end every CTA leaves its unnormalised partial (max, sum, O row)
//     in shared memory and the cluster merges the C partials of each row
//     through distributed shared memory, writing bf16 rows.
// Launch: programmatic dependent launch; everything earlier kernels may have
// written (lengths, cache rows, Q, block K/V, tree) is read after
// griddepcontrol.wait.
#include <cooperative_groups.h>
#include <math.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kD = 128;
constexpr int kNk = 64;                   // keys per TMA tile
constexpr int kStepTiles = 1;             // TMA tiles per softmax step
constexpr int kStepKeys = kStepTiles * kNk;   // keys per softmax step
constexpr int kRows = 128;                // query rows per CTA (MMA M)
constexpr int kStages = 4;                // TMA ring depth in tiles
constexpr int kQBytes = kRows * kD * 2;   // 32 KB: two 64-column halves of 128 rows
constexpr int kPBlock = kRows * kNk * 2;  // 16 KB: P for one 64-key tile
constexpr int kPStep = kStepTiles * kPBlock;   // P for one step
constexpr int kPBytes = 2 * kPStep;            // two P buffers: step st uses buffer st % 2
constexpr int kHalfBytes = kNk * 128;     // one 64-key x 64-dim swizzled box: 8 KB
constexpr int kStageBytes = 4 * kHalfBytes;   // K and V, two halves each: 32 KB
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kRec = kD + 4;              // partial record: m, l, 2 pad, o[128]
constexpr int kMaxR = 128;
constexpr int kMaxCluster = 16;
constexpr int kSoftWarps = 16;            // row-owner warps
constexpr int kGroups = 4;                // column groups of a step
constexpr int kGCols = kStepKeys / kGroups;   // scores per thread per step
constexpr int kTmaWarp = kSoftWarps, kMmaWarp = kSoftWarps + 1;
constexpr int kThreads = 32 * (kSoftWarps + 2);
constexpr uint32_t kTmemCols = 4 * kStepKeys;   // S buffers at 0 and kStepKeys, O (128 columns) after them
constexpr float kRescale = 8.0f;          // log2 of the largest tolerated P
static_assert(kRows * kRec * 4 <= kRingBytes, "partials reuse the K/V ring");
// S of step st+1 is issued before the P V of step st: both tiles stay resident
static_assert(kStages >= 2 * kStepTiles + 1, "ring too shallow for the S/PV overlap");

constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffRing = kOffP + kPBytes;
constexpr int kOffBar = kOffRing + kRingBytes;
constexpr int kOffAnc = kOffBar + 256;
constexpr int kOffRed = kOffAnc + kMaxR * 16;                 // [2][kGroups][kRows] partial row maxima
constexpr int kOffLsum = kOffRed + 2 * kGroups * kRows * 4;    // [kGroups][kRows] partial row sums
constexpr int kSmemBytes = kOffLsum + kGroups * kRows * 4 + 1024;

struct AttnArgs {
    const uint16_t* q;
    const int32_t* len;
    const int32_t* parent;
    uint16_t* out;
    unsigned int* err;
    int B, R, Hq, Hkv, G, T_cap, rows, row_tiles;
    float scale_log2;
};

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                                                             const __grid_constant__ CUtensorMap tmV,
                                                             const __grid_constant__ CUtensorMap tmKb,
                                                             const __grid_constant__ CUtensorMap tmVb, AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* kv_full = bars;                    // [kStages]
    uint64_t* kv_empty = bars + kStages;         // [kStages]
    uint64_t* s_full = bars + 2 * kStages;       // [2]
    uint64_t* s_empty = s_full + 2;              // [2]
    uint64_t* p_full = s_empty + 2;              // [2], per P buffer
    uint64_t* o_done = p_full + 2;               // [2], per P buffer
    uint64_t* q_ready = o_done + 2;
    uint32_t* tmem_s = reinterpret_cast<uint32_t*>(q_ready + 1);
    uint64_t* anc = reinterpret_cast<uint64_t*>(smem + kOffAnc);   // [kMaxR][2]
    float* part = reinterpret_cast<float*>(smem + kOffRing);        // [kRows][kRec] after the loop

    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hg = blockIdx.y, rt = blockIdx.z;
    const int b = hg / a.Hkv, g = hg % a.Hkv;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmKb);
        prefetch_tmap(&tmVb);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], kSoftWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&p_full[i], kSoftWarps);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(q_ready, kSoftWarps);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(tmem_s, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_s;
    const uint32_t tS[2] = {tmem, tmem + kStepKeys};
    const uint32_t tO = tmem + 2 * kStepKeys;

    // inputs may come from the kernels before this one
    pdl_wait();
    pdl_launch_dependents();

    int t = a.len[b];
    if (t < 0 || t > a.T_cap) {
        if (threadIdx.x == 0 && rank == 0 && rt == 0) raise_error(a.err, SV_DEVERR_LENGTH);
        t = t < 0 ? 0 : a.T_cap;
    }
    const int n_ctx = (t + kNk - 1) / kNk;
    const int n_blk = (a.R + kNk - 1) / kNk;
    const int n_all = n_ctx + n_blk;
    const int first = static_cast<int>((static_cast<int64_t>(n_all) * rank) / C);
    const int last = static_cast<int>((static_cast<int64_t>(n_all) * (rank + 1)) / C);
    const int ntiles = last - first;
    const int nsteps = (ntiles + kStepTiles - 1) / kStepTiles;
    const bool has_block = last > n_ctx;
    const bool tree = a.parent != nullptr && has_block;

    if (warp == kTmaWarp) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            for (int i = 0; i < ntiles; ++i) {
                const int s = i % kStages;
                mbar_wait(&kv_empty[s], ((i / kStages) & 1) ^ 1, a.err);
                const int gt = first + i;
                const void* tk = gt < n_ctx ? static_cast<const void*>(&tmK) : static_cast<const void*>(&tmKb);
                const void* tv = gt < n_ctx ? static_cast<const void*>(&tmV) : static_cast<const void*>(&tmVb);
                const int y = gt < n_ctx ? hg * a.T_cap + gt * kNk : hg * a.R + (gt - n_ctx) * kNk;
                uint8_t* st = smem + kOffRing + s * kStageBytes;
                mbar_arrive_expect_tx(&kv_full[s], kStageBytes);
                tma_load_2d(st, tk, 0, y, &kv_full[s]);
                tma_load_2d(st + kHalfBytes, tk, 64, y, &kv_full[s]);
                tma_load_2d(st + 2 * kHalfBytes, tv, 0, y, &kv_full[s]);
                tma_load_2d(st + 3 * kHalfBytes, tv, 64, y, &kv_full[s]);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kNk, false, false);   // S tile = Q K^T
            constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, kD, false, true);     // O += P V
            const uint32_t sq = smem_u32(smem + kOffQ);
            const uint32_t sp = smem_u32(smem + kOffP);
            // both S operands K-major; the two 64-dim halves are separate boxes
            const uint64_t qd0 = smem_desc_sw128(sq, 16, 1024);
            mbar_wait(q_ready, 0, a.err);
            auto pv = [&](int st) {
                const int pb = st & 1;
                mbar_wait(&p_full[pb], (st >> 1) & 1, a.err);
                tc_fence_after();
                const int t0 = kStepTiles * st, nt = min(kStepTiles, ntiles - t0);
                for (int h = 0; h < nt; ++h) {
                    const int s = (t0 + h) % kStages;
                    const uint32_t sv = smem_u32(smem + kOffRing + s * kStageBytes + 2 * kHalfBytes);
                    // A = P [128 rows][64 keys of tile h], K-major; B = V [64 keys][128
                    // dims], MN-major: 8-key groups 1024 B apart, the two 64-dim halves
                    // kHalfBytes apart, 16 keys = 2048 B (descriptor units of 16 B).
                    const uint64_t ad0 = smem_desc_sw128(sp + pb * kPStep + h * kPBlock, 16, 1024);
                    const uint64_t bd0 = smem_desc_sw128(sv, kHalfBytes, 1024);
#pragma unroll
                    for (int k16 = 0; k16 < kNk / 16; ++k16)
                        tc_mma(tO, ad0 + k16 * (32 >> 4), bd0 + k16 * (2048 >> 4), idesc_o,
                               (st > 0 || h > 0 || k16 > 0) ? 1u : 0u);
                }
                tc_commit(&o_done[pb]);
                for (int h = 0; h < nt; ++h) tc_commit(&kv_empty[(t0 + h) % kStages]);
            };
            for (int st = 0; st < nsteps; ++st) {
                const int sb = st & 1;
                mbar_wait(&s_empty[sb], ((st >> 1) & 1) ^ 1, a.err);
                const int t0 = kStepTiles * st, nt = min(kStepTiles, ntiles - t0);
                for (int h = 0; h < nt; ++h) {
                    const int i = t0 + h;
                    const int s = i % kStages;
                    mbar_wait(&kv_full[s], (i / kStages) & 1, a.err);
                    tc_fence_after();
                    const uint64_t kd0 = smem_desc_sw128(smem_u32(smem + kOffRing + s * kStageBytes), 16, 1024);
#pragma unroll
                    for (int k16 = 0; k16 < kD / 16; ++k16) {
                        const uint32_t half = k16 >> 2, kin = (k16 & 3) * 32;
                        tc_mma(tS[sb] + h * kNk, qd0 + ((half * (kRows * 128) + kin) >> 4),
                               kd0 + ((half * kHalfBytes + kin) >> 4), idesc_s, k16 > 0 ? 1u : 0u);
                    }
                }
                tc_commit(&s_full[sb]);
                if (st > 0) pv(st - 1);
            }
            pv(nsteps - 1);
        }
    } else {
        // ---------------- row-owner warps: row r, column group cgp ----------------
        const int cgp = warp / 4;                         // 16-column group of each step
        const int r = (warp & 3) * 32 + lane;             // row inside the tile (TMEM lane)
        const int gr = rt * kRows + r;                    // row inside (b, g)
        const bool valid = gr < a.rows;
        const int j = valid ? gr / a.G : 0;
        // rows of this warp's TMEM quarter that exist (the rest of a 128-row
        // tile is padding whose P and O are never read)
        const bool quarter_live = rt * kRows + (warp & 3) * 32 < a.rows;
        float* red = reinterpret_cast<float*>(smem + kOffRed);
        float* lsx = reinterpret_cast<float*>(smem + kOffLsum);
        // tree ancestor masks: bit i of anc[jj] set iff block row i is jj or an ancestor
        if (tree) {
            const int32_t* par = a.parent + static_cast<size_t>(b) * a.R;
            for (int jj = threadIdx.x; jj < a.R; jj += 32 * kSoftWarps) {
                uint64_t m0 = 0, m1 = 0;
                int i = jj;
                bool bad = false;
                for (int steps = 0; steps <= a.R && i >= 0; ++steps) {
                    if (i < 64) m0 |= 1ull << i; else m1 |= 1ull << (i - 64);
                    const int p = par[i];
                    if ((i == 0 && p != -1) || (i > 0 && (p < 0 || p >= i))) { bad = true; break; }
                    i = p;
                }
                if (bad) {
                    raise_error(a.err, SV_DEVERR_TREE);
                    m0 = jj < 64 ? 1ull << jj : 0;
                    m1 = jj >= 64 ? 1ull << (jj - 64) : 0;
                }
                anc[2 * jj] = m0;
                anc[2 * jj + 1] = m1;
            }
        }
        // gather the Q tile (zero rows beyond the group) into the K-major
        // 128-byte-swizzled layout the MMA reads
        {
            uint8_t* q_s = smem + kOffQ;
            for (int x = threadIdx.x; x < kRows * 16; x += 32 * kSoftWarps) {
                const int row = x >> 4, c = x & 15;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                const int grow = rt * kRows + row;
                if (grow < a.rows) {
                    const int jr = grow / a.G, hl = grow % a.G;
                    const uint16_t* src = a.q + ((static_cast<size_t>(b) * a.R + jr) * a.Hq + g * a.G + hl) * kD;
                    v = __ldg(reinterpret_cast<const uint4*>(src) + c);
                }
                const int half = c >> 3, cc = c & 7;
                *reinterpret_cast<uint4*>(q_s + half * (kRows * 128) + row * 128 + ((cc ^ (row & 7)) << 4)) = v;
            }
        }
        fence_proxy_async_smem();
        named_barrier(1, 32 * kSoftWarps);   // anc and Q written by every row-owner warp
        if (lane == 0) mbar_arrive(q_ready);
        const uint64_t anc0 = (tree && valid) ? anc[2 * j] : 0, anc1 = (tree && valid) ? anc[2 * j + 1] : 0;

        float m_ref = -INFINITY, lsum = 0.f;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        for (int st = 0; st < nsteps; ++st) {
            const int sb = st & 1;
            mbar_wait(&s_full[sb], (st >> 1) & 1, a.err);
            tc_fence_after();
            // this thread's scores: columns kGCols*cgp.. of the step, all in tile ti
            const int ti = kStepTiles * st + (cgp * kGCols) / kNk;
            const int col_in_tile = (cgp * kGCols) % kNk;
            const bool work = quarter_live && ti < ntiles;
            uint32_t ra[16], rb[16];
            if (work) {
                tmem_ld16_sync(tS[sb] + lane_off + cgp * kGCols, ra);
                if (kGCols > 16) tmem_ld16_sync(tS[sb] + lane_off + cgp * kGCols + 16, rb);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[sb]);
            const int gt = first + ti;
            const bool is_block = gt >= n_ctx;
            const int kb = (is_block ? (gt - n_ctx) * kNk : gt * kNk) + col_in_tile;
            float sc[kGCols];
            float mpart = -INFINITY;
            if (work) {
#pragma unroll
                for (int e = 0; e < 16; ++e) sc[e] = __uint_as_float(ra[e]) * a.scale_log2;
#pragma unroll
                for (int e = 16; e < kGCols; ++e) sc[e] = __uint_as_float(rb[e - 16]) * a.scale_log2;
                if (is_block || kb + kGCols > t) {
#pragma unroll
                    for (int e = 0; e < kGCols; ++e) {
                        const int kl = kb + e;
                        bool vis;
                        if (!is_block) {
                            vis = kl < t;
                        } else if (kl >= a.R) {
                            vis = false;
                        } else if (tree) {
                            vis = ((kl < 64 ? anc0 : anc1) >> (kl & 63)) & 1ull;
                        } else {
                            vis = kl <= j;
                        }
                        if (!vis) sc[e] = -INFINITY;
                    }
                }
                float mx[kGCols / 2];
#pragma unroll
                for (int e = 0; e < kGCols / 2; ++e) mx[e] = fmaxf(sc[e], sc[e + kGCols / 2]);
#pragma unroll
                for (int w2 = kGCols / 4; w2 >= 1; w2 >>= 1)
#pragma unroll
                    for (int e = 0; e < w2; ++e) mx[e] = fmaxf(mx[e], mx[e + w2]);
                mpart = mx[0];
            }
            red[(sb * kGroups + cgp) * kRows + r] = mpart;
            named_barrier(2, 32 * kSoftWarps);
            float mt = red[(sb * kGroups + 0) * kRows + r];
#pragma unroll
            for (int c2 = 1; c2 < kGroups; ++c2) mt = fmaxf(mt, red[(sb * kGroups + c2) * kRows + r]);
            float m_new = m_ref, corr = 1.f;
            if (mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescale)) {
                m_new = mt;
                corr = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - m_new);
            }
            // P (bf16) and this thread's share of its sum
            uint32_t pk[kGCols / 2];
            float ps0 = 0.f, ps1 = 0.f;
            if (work) {
#pragma unroll
                for (int e = 0; e < kGCols; e += 2) {
                    const float p0 = (m_new == -INFINITY) ? 0.f : fast_exp2(sc[e] - m_new);
                    const float p1 = (m_new == -INFINITY) ? 0.f : fast_exp2(sc[e + 1] - m_new);
                    const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                    ps0 += __bfloat162float(pb.x);
                    ps1 += __bfloat162float(pb.y);
                    pk[e / 2] = *reinterpret_cast<const uint32_t*>(&pb);
                }
            }
            lsum = lsum * corr + (ps0 + ps1);
            m_ref = m_new;
            // P buffer sb is free once the P V of step st-2 is done
            if (st >= 2) {
                mbar_wait(&o_done[sb], ((st - 2) >> 1) & 1, a.err);
                tc_fence_after();
            }
            if (quarter_live && st >= 1 && __any_sync(0xffffffffu, corr != 1.f)) {
                // rescale O: wait for the P V of step st-1 to settle it
                mbar_wait(&o_done[sb ^ 1], ((st - 1) >> 1) & 1, a.err);
                tc_fence_after();
                {
#pragma unroll
                    for (int c0 = 0; c0 < kD / kGroups; c0 += 16) {
                        const uint32_t ta = tO + lane_off + cgp * (kD / kGroups) + c0;
                        uint32_t o16[16];
                        tmem_ld16_sync(ta, o16);
#pragma unroll
                        for (int e = 0; e < 16; ++e) o16[e] = __float_as_uint(__uint_as_float(o16[e]) * corr);
                        tmem_st16(ta, o16);
                    }
                    tmem_st_wait();
                }
            }
            if (work) {
                uint8_t* p_row = smem + kOffP + sb * kPStep + ((cgp * kGCols) / kNk) * kPBlock + r * 128;
#pragma unroll
                for (int h = 0; h < kGCols / 8; ++h) {
                    const int cc = col_in_tile / 8 + h;
                    *reinterpret_cast<uint4*>(p_row + ((cc ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
        }
        if (nsteps > 0) {
            mbar_wait(&o_done[(nsteps - 1) & 1], ((nsteps - 1) >> 1) & 1, a.err);
            tc_fence_after();
        }
        // row sum across the four column groups -> this CTA's partial
        lsx[cgp * kRows + r] = lsum;
        named_barrier(2, 32 * kSoftWarps);
        float lt = 0.f;
#pragma unroll
        for (int c2 = 0; c2 < kGroups; ++c2) lt += lsx[c2 * kRows + r];
        const bool use = nsteps >= 1 && lt > 0.f;
        float* rec = part + r * kRec;
        if (cgp == 0) {
            rec[0] = use ? m_ref : -INFINITY;
            rec[1] = use ? lt : 0.f;
        }
#pragma unroll
        for (int c0 = 0; c0 < kD / kGroups; c0 += 16) {
            const uint32_t col = cgp * (kD / kGroups) + c0;
            uint32_t o16[16] = {};
            if (nsteps >= 1) tmem_ld16_sync(tO + lane_off + col, o16);
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<uint4*>(rec + 4 + col + e) =
                    use ? make_uint4(o16[e], o16[e + 1], o16[e + 2], o16[e + 3]) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster.sync();   // all partials written (and every CTA of the cluster has started)

    // merge: this CTA finalises rows rank, rank + C, ... of the row tile (all warps)
    const int nrows = min(kRows, a.rows - rt * kRows);
    for (int lr = rank + C * warp; lr < nrows; lr += C * (kThreads / 32)) {
        float ms = -INFINITY, ls = 0.f;
        if (lane < C) {
            const float* rec_s = cluster.map_shared_rank(part + lr * kRec, lane);
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
            const float4 x =
                *reinterpret_cast<const float4*>(cluster.map_shared_rank(part + lr * kRec + 4, s) + 4 * lane);
            acc.x += ws * x.x;
            acc.y += ws * x.y;
            acc.z += ws * x.z;
            acc.w += ws * x.w;
        }
        const float inv = L > 0.f ? 1.0f / L : 0.f;
        const int row = rt * kRows + lr;
        const int jr = row / a.G, h = g * a.G + row % a.G;
        uint16_t* dst = a.out + ((static_cast<size_t>(b) * a.R + jr) * a.Hq + h) * kD + 4 * lane;
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
    cluster.sync();   // no CTA leaves while its partials may still be read
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

AttnPlan attn_plan(const sv_attn_shape& s) {
    AttnPlan p;
    p.G = s.Hq / s.Hkv;
    p.rows = s.R * p.G;
    p.row_tiles = (p.rows + kRows - 1) / kRows;
    p.warps = kThreads / 32;
    // cluster size: grow while the grid still fits in one CTA per SM and every
    // CTA keeps at least one step of key tiles
    const int units = s.B * s.Hkv * p.row_tiles;
    const int slots = device_sm_count();
    const int tiles = (s.T_cap + kNk - 1) / kNk + (s.R + kNk - 1) / kNk;
    int C = 1;
    while (C < kMaxCluster && units * C * 2 <= slots && C * 4 <= tiles) C *= 2;
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
    if (!encode_tmap_2d_bf16(tK, k_cache, kD, ctx_rows, kD * 2, 64, kNk) ||
        !encode_tmap_2d_bf16(tV, v_cache, kD, ctx_rows, kD * 2, 64, kNk) ||
        !encode_tmap_2d_bf16(tKb, k_blk, kD, blk_rows, kD * 2, 64, kNk) ||
        !encode_tmap_2d_bf16(tVb, v_blk, kD, blk_rows, kD * 2, 64, kNk))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
    cfg.blockDim = dim3(kThreads, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel, *reinterpret_cast<const CUtensorMap*>(tK),
                              *reinterpret_cast<const CUtensorMap*>(tV), *reinterpret_cast<const CUtensorMap*>(tKb),
                              *reinterpret_cast<const CUtensorMap*>(tVb), a);
}

}  // namespace sv
