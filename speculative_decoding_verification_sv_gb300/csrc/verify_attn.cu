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
// so each K/V tile streamed from HBM serves all of them (GQA).  Rows are cut
// into row tiles: half tiles of 64 rows (M = 64 MMAs) or full tiles of 128
// (M = 128), whichever the plan costs lower.  One thread-block cluster of C
// CTAs (1 <= C <= 16) handles one (b, g, row tile), a unit: its 64-key tiles
// -- ceil(t/64) context tiles followed by ceil(R/64) block tiles -- are split
// evenly over the CTAs (split-KV, sized so the grid fills the SMs; several
// clusters per unit meet in a workspace).  Inside a CTA, keys are processed
// two 64-key tiles per step:
//   * one warp streams K and V tiles through a TMA ring (cp.async.bulk.tensor,
//     128-byte swizzle, full/empty mbarriers; K and V regions on barriers of
//     their own where the loop outgrows the ring);
//   * one thread of another warp issues tcgen05.mma: S = Q K^T (N = 128, both
//     tiles) into one of two TMEM score buffers, and O += P V into a TMEM
//     accumulator with P read from TMEM, releasing stages and buffers with
//     tcgen05.commit; S of step st+1 is issued before P V of step st, so the
//     score MMAs run under the softmax;
//   * row-owner warps read the scores of their TMEM quadrant, exchange partial
//     maxima through shared memory, apply the chain/tree/length mask, keep the
//     running max and sum, write P (bf16) back to TMEM, and rescale their part
//     of the row of O only when the max has grown by more than 2^8 since it was
//     last used (otherwise the stale max keeps every P <= 256, exact in fp32).
//     Warps whose rows are all padding skip the arithmetic;
//   * at the end each CTA's unnormalised partial (max, sum, O row) of every
//     row reaches the row's owner CTA (pushed into its shared memory, or with
//     128-row tiles through an L2 exchange area), which writes the bf16 rows.
// Launch: programmatic dependent launch; everything earlier kernels may have
// written (lengths, cache rows, Q, block K/V, tree) is read after
// griddepcontrol.wait.
#include <cooperative_groups.h>
#include <math.h>

#include <mutex>
#include <type_traits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kD = 128;
constexpr int kNk = 64;                   // keys per TMA tile
constexpr int kRows = 128;                // query rows per full row tile
constexpr int kHalfBytes = kNk * 128;     // one 64-key x 64-dim swizzled box: 8 KB
constexpr int kTileBytes = 4 * kHalfBytes;   // K and V of one tile, two halves each: 32 KB
constexpr int kRec = kD + 4;              // partial record: m, l, 2 pad, o[128]
constexpr int kMaxR = 128;
constexpr int kMaxCluster = 16;
#ifndef SV_ATTN_MERGE_COST
#define SV_ATTN_MERGE_COST 7
#endif
constexpr int kMergeCost = SV_ATTN_MERGE_COST;   // workspace merge, in key-tile times
constexpr int kWsMergeBatch = 12;         // workspace partials per unit merged in one round of loads
constexpr int kXchMaxCluster = 6;         // largest cluster whose partials meet through the L2 exchange
constexpr int kGroups = 4;                // full tiles: column groups of a step
#ifndef SV_ATTN_HALF_MAX_ROWS
#define SV_ATTN_HALF_MAX_ROWS 64
#endif
// Row tiles: (b, g) groups of at most kHalfMaxRows rows use one half tile;
// larger groups use half or full tiles as the plan's cost decides (full tiles
// serve twice the rows with the same MMAs per key, half tiles make more units
// for the SMs)
constexpr int kHalfMaxRows = SV_ATTN_HALF_MAX_ROWS;

// Full tiles (128 rows): 16 row-owner warps, warp w on TMEM quadrant w % 4
// and the 32-column group w / 4 of each step.  Half tiles (64 rows): kHW = 2 or 4 row-owner warps
// per quadrant (= per SM sub-partition, so one hides another's latency), the
// rows spread over the first 16 lanes of every quadrant, 2 kHW threads per row
// (two per warp via the 16x32bx2 access, one warp per column slice).
#ifndef SV_ATTN_HW4_MIN_TILES
#define SV_ATTN_HW4_MIN_TILES 16
#endif
// half tiles: four row-owner warps per quadrant when every CTA streams at least
// this many key tiles (long loops: more latency hiding pays), else two (a few
// steps: the smaller cross-warp exchange wins)
constexpr int kHw4MinTiles = SV_ATTN_HW4_MIN_TILES;
// kHW: row-owner warps per TMEM quadrant with half tiles (2 or 4)
template <bool kHalf, int kHW = 2>
struct Roles {
    static_assert(kHW == 2 || kHW == 4, "two or four warps per quadrant");
    static constexpr int kSoft = kHalf ? 4 * kHW : 16;
    static constexpr int kTma = kSoft, kMma = kSoft + 1;
    static constexpr int kThreads = 32 * (kSoft + 2);
};
constexpr uint32_t kTmemCols = 512;
constexpr float kRescale = 8.0f;          // log2 of the largest tolerated P

// Shared-memory and TMEM layout.  Both modes take two key tiles per step
// (S = Q K^T as one N = 128 MMA chain over both: fewer, larger MMAs per key).
// Full tiles: M = 128 MMAs, 32 KB of Q, 2 ring stages of two tiles (always
// on split K/V barriers: with two stages the K loads must run ahead of the
// P V reads).  Half tiles: M = 64 MMAs (row m of the tile in TMEM lane
// 32 * (m / 16) + m % 16), 16 KB of Q, 3 stages; an M = 64 MMA issues as
// slowly as an M = 128 one, so full tiles do twice the work per MMA.
// A stage holds its tiles' boxes region by region: K dims 0-63 of every tile,
// K dims 64-127, V dims 0-63, V dims 64-127, so keys are contiguous per region.
template <bool kHalf>
struct Lay {
    static constexpr int kM = kHalf ? 64 : 128;            // MMA M (rows of the Q tile)
    static constexpr int kT = 2;                            // key tiles per softmax step
    static constexpr int kStepKeys = kT * kNk;
    static constexpr int kStageBytes = kT * kTileBytes;
    static constexpr int kRegion = kT * kHalfBytes;        // one region of a stage
    static constexpr int kStages = kHalf ? 3 : 2;           // ring depth in steps
    static constexpr int kQBytes = kM * kD * 2;             // two 64-dim halves of kM rows
    static constexpr int kRingBytes = kStages * kStageBytes;
    // TMEM columns: two S buffers, O (128 columns), two P buffers (two bf16 per column)
    static constexpr uint32_t kColS = 0, kColO = 2 * kStepKeys, kColP = kColO + kD;
    static constexpr int kPCols = kStepKeys / 2;
    static_assert(kColP + 2 * kPCols <= kTmemCols, "TMEM budget");
    static constexpr int kOffQ = 0;
    static constexpr int kOffRing = kOffQ + kQBytes;
    static constexpr int kOffBar = kOffRing + kRingBytes;
    static constexpr int kOffAnc = kOffBar + 256;
    static constexpr int kOffRed = kOffAnc + kMaxR * 16;               // [2][kGroups][kRows] partial row maxima
    static constexpr int kOffLsum = kOffRed + 2 * kGroups * kRows * 4;  // [kGroups][kRows] partial row sums
    static constexpr int kSmemBytes = kOffLsum + kGroups * kRows * 4 + 1024;
    static_assert((kRows + kMaxCluster - 1) * kRec * 4 <= kRingBytes, "pushed partials reuse the K/V ring");
    // a CTA's block of the L2 exchange: (max, sum) of each row, then O as
    // [kD / 4 column chunks][kM rows] float4, so that a warp's 32 rows of one
    // chunk are one contiguous 512-byte store or load
    static constexpr int kXchFloats = kM * (2 + kD);
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
    static_assert((4 * kStages + 9) * 8 + 4 <= 248, "barrier area (the word at +248 is the ticket flag)");
};

struct AttnArgs {
    const uint16_t* q;
    const uint16_t* k_blk;   // [B][Hkv][R][D] (read through tmKb / tmVb; raw for the L2 prefetch)
    const uint16_t* v_blk;
    const int32_t* len;
    const int32_t* parent;
    uint16_t* out;
    unsigned int* err;
    float* ws_part;          // [unit][cluster][part_rows][kRec] cluster partials (clusters > 1)
    float* xch;              // [grid CTA][Lay::kXchFloats] partial rows exchanged through L2 (nullptr:
                             // pushed into the owners' shared memory)
    unsigned int* ws_cnt;    // [unit] tickets of clusters done; zero between launches
    int B, R, Hq, Hkv, G, T_cap, rows, row_tiles;
    int clusters;            // clusters per (b, g, row tile); their partials meet in ws_part
    int part_rows;           // rows of a partial record block: min(rows, rows per row tile)
    float scale_log2;
    int cache_ready;         // len and the cache are final before the preceding kernel runs
    const int32_t* pages;    // paged cache: [B][max_pages] page of each 64-position tile (nullptr: contiguous)
    int max_pages, num_pages;
};

// floor(n * i / k), the first key tile of split i of k: unsigned 32-bit
// arithmetic whenever n * i cannot overflow (every realistic cache), instead of
// the long out-of-line 64-bit division routine.
__device__ __forceinline__ int split_bound(int n, int i, int k) {
    if (n <= 65535 && i <= 65535) return static_cast<int>(static_cast<uint32_t>(n) * static_cast<uint32_t>(i) /
                                                          static_cast<uint32_t>(k));
    return static_cast<int>((static_cast<int64_t>(n) * i) / k);
}

// TMEM lane that holds row gr of (b, g): full tiles lane = gr - 128 * rt;
// half tiles put row gr in lane 32 * (gr % 4) + gr / 4, so every quadrant
// (SM sub-partition) carries a quarter of the rows.

// kTree: the launch carries a draft tree (parent != NULL).  Chains compile
// without any ancestor-mask code: the speculatively evaluated 64-bit window
// of the tree mask stalled the chain's block-tile step by ~2500 cycles.
// kSplit: the K and V halves of a ring stage land and are released on
// barriers of their own (long loops over tiles no other row tile shares).
template <bool kHalf, bool kTree, int kHW, bool kSplit>
__global__ void __launch_bounds__(Roles<kHalf, kHW>::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmKb, const __grid_constant__ CUtensorMap tmVb, AttnArgs a) {
    using Ro = Roles<kHalf, kHW>;
    constexpr int kHalfWarps = kHW;
    using Ly = Lay<kHalf>;
    constexpr int kSoftWarps = Ro::kSoft, kTmaWarp = Ro::kTma, kMmaWarp = Ro::kMma, kThreads = Ro::kThreads;
    constexpr int kStages = Ly::kStages, kM = Ly::kM, kT = Ly::kT, kStepKeys = Ly::kStepKeys;
    constexpr int kStageBytes = Ly::kStageBytes, kRegion = Ly::kRegion;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::kOffBar);
    // kSplit: the K and V halves of a ring stage land and are released on
    // barriers of their own; otherwise v_full / v_empty are k_full / k_empty
    // (one barrier per stage for both halves)
    uint64_t* k_full = bars;                                     // [kStages]
    uint64_t* v_full = kSplit ? bars + kStages : k_full;         // [kStages]
    uint64_t* k_empty = bars + 2 * kStages;                      // [kStages]
    uint64_t* v_empty = kSplit ? bars + 3 * kStages : k_empty;   // [kStages]
    uint64_t* s_full = bars + 4 * kStages;       // [2]
    uint64_t* s_empty = s_full + 2;              // [2]
    uint64_t* p_full = s_empty + 2;              // [2], per P buffer
    uint64_t* o_done = p_full + 2;               // [2], per P buffer
    uint64_t* q_ready = o_done + 2;
    uint32_t* tmem_s = reinterpret_cast<uint32_t*>(q_ready + 1);
    uint64_t* anc = reinterpret_cast<uint64_t*>(smem + Ly::kOffAnc);   // [kMaxR][2]
    // after the loop: partial records pushed to this CTA, [row / C][source rank][kRec]
    float* part = reinterpret_cast<float*>(smem + Ly::kOffRing);
    // the L2 exchange (128-row tiles only: half-tile kernels compile without it)
    float* const xch = kHalf ? nullptr : a.xch;

    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // (sequence, KV head) and row tile: the row tiles of one KV head are
    // adjacent in launch order, so their CTAs share its K/V tiles through L2
    const int hg = blockIdx.y / a.row_tiles, rt = blockIdx.y % a.row_tiles;
    constexpr int kTileRows = Lay<kHalf>::kM;   // query rows per row tile
    const int b = hg / a.Hkv, g = hg % a.Hkv;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmKb);
        prefetch_tmap(&tmVb);
        for (int s = 0; s < 4 * kStages; ++s) mbar_init(&bars[s], 1);   // the ring's full / empty barriers
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
    // this CTA has started (and initialised its barriers): waited for by every
    // thread before the first store into another CTA's shared memory
    cluster_arrive_relaxed();
    const uint32_t tmem = *tmem_s;
    // TMEM addresses of score buffer / P buffer `i` (arithmetic, not arrays: a
    // runtime-indexed array would live in local memory)
    auto tS = [tmem](int i) { return tmem + Ly::kColS + static_cast<uint32_t>(i) * Ly::kStepKeys; };
    const uint32_t tO = tmem + Ly::kColO;
    auto tP = [tmem](int i) { return tmem + Ly::kColP + static_cast<uint32_t>(i) * Ly::kPCols; };

    // Inputs may come from the kernel before this one: every thread waits for
    // it before touching them.  The next kernel is let start only once this
    // CTA's loop is over (pdl_launch_dependents before the merge): started at
    // once, the next layer's early cache loads competed with this layer's
    // own, 1.5B layer 8.34 -> 8.20 us measured.  With
    // cache_ready the length and the committed cache rows were final before that
    // kernel started, so they are read first, and the producer issues its
    // context loads before waiting.
    // Warm L2 with this unit's Q rows (and, in the CTAs that take the block
    // tiles, the block's K/V rows) while the preceding kernel may still run.
    // A prefetch only fills L2, the point of coherence, so rows that kernel is
    // still writing are read fresh by the loads after the wait below; it saves
    // the DRAM round trip of the Q gather that follows the wait.
    if (warp == kMmaWarp && lane == 0) {
        const int gr0 = rt * kTileRows, gr1 = min(a.rows, gr0 + kTileRows) - 1;
        for (int jq = gr0 / a.G; jq <= gr1 / a.G; ++jq)
            prefetch_l2(a.q + ((static_cast<size_t>(b) * a.R + jq) * a.Hq + g * a.G) * kD,
                        static_cast<uint32_t>(a.G * kD * 2));
        if (static_cast<int>(blockIdx.x) >= static_cast<int>(gridDim.x) - 2) {
            const size_t off = static_cast<size_t>(hg) * a.R * kD;
            prefetch_l2(a.k_blk + off, static_cast<uint32_t>(a.R * kD * 2));
            prefetch_l2(a.v_blk + off, static_cast<uint32_t>(a.R * kD * 2));
        }
    }
    // Without cache_ready the length may come from the kernel before: every
    // thread waits first.  With it, the plan below (split bounds, fold, merge
    // plan) is computed while that kernel drains, and each warp waits only
    // before its first read of that kernel's outputs (Q, the block K/V, the
    // tree) or its first global store: reading the parameter block and doing
    // this set-up after the wait put ~1 us on every batch-1 layer's critical
    // path.
    const bool early = a.cache_ready != 0;
    if (!early) pdl_wait();
    int t = a.len[b];
    const bool bad_len = t < 0 || t > a.T_cap;
    if (bad_len) t = t < 0 ? 0 : a.T_cap;
    const int n_ctx = (t + kNk - 1) / kNk;
    const int n_blk = (a.R + kNk - 1) / kNk;
    const int n_all = n_ctx + n_blk;
    // this CTA's share of the key tiles: split blockIdx.x of the gridDim.x
    // CTAs (a.clusters clusters of C) working on (b, g, row tile)
    const int split = blockIdx.x, nsplit = gridDim.x;
    const int first = split_bound(n_all, split, nsplit);
    const int last = split_bound(n_all, split + 1, nsplit);
    const int ntiles = last - first;
    const int nsteps = (ntiles + kT - 1) / kT;   // ring steps (stages of up to kT tiles)
    // Fold (half tiles, two warps per quadrant): an odd last tile joins the step
    // before it as a third tile -- its scores in the first 64 columns of the
    // other score buffer, its P in the other P buffer -- instead of a step of
    // its own; softmax steps are then one fewer than ring steps
    const bool fold = kHalf && kHW == 2 && (ntiles & 1) != 0 && ntiles >= 3;
    const int nsoft = nsteps - (fold ? 1 : 0);
    const bool has_block = last > n_ctx;
    const bool tree = kTree && has_block;
    const int nrows = min(kTileRows, a.rows - rt * kTileRows);

    // Receive plan of the cluster merge (computed by each warp, lane r for CTA
    // r of the cluster).  A CTA whose steps never reach the last `need` ring
    // stages is "light": those stages can take pushed partial records from the
    // start.  When the light CTAs can hold every row, they own the rows and each
    // CTA pushes as soon as its own loop ends; otherwise (need = 0) every CTA
    // owns rows prow % C, received at the front of the ring once all CTAs of
    // the cluster have drained theirs.
    auto merge_plan = [&](int& need_o, uint32_t& light_o) {
        int st_r = 1 << 30;
        if (lane < C) {
            const int sr = split - rank + lane;
            const int f = split_bound(n_all, sr, nsplit);
            const int l = split_bound(n_all, sr + 1, nsplit);
            st_r = (l - f + kT - 1) / kT;
        }
        need_o = 0;
        light_o = 0u;
        for (int nd = 1; nd < kStages; ++nd) {
            const uint32_t m = __ballot_sync(0xffffffffu, st_r <= kStages - nd);
            const int nl = __popc(m);
            if (nl > 0 && ((nrows + nl - 1) / nl) * C * kRec * 4 <= nd * kStageBytes) {
                need_o = nd;
                light_o = m;
                break;
            }
        }
    };
    int need = 0;
    uint32_t light = 0u;

    if (warp == kTmaWarp) {
        // ---------------- TMA producer ----------------
        // first row of context tile gt in the K/V tensor maps: the contiguous
        // cache [B][Hkv][T_cap][D], or the tile's page of a [pages][Hkv][64][D]
        // pool (a page outside the pool reads as zeros and is flagged)
        auto ctx_row = [&](int gt) {
            if (a.pages == nullptr) return hg * a.T_cap + gt * kNk;
            int pg = __ldg(a.pages + static_cast<size_t>(b) * a.max_pages + gt);
            if (pg < 0 || pg >= a.num_pages) {
                raise_error(a.err, SV_DEVERR_PAGE);
                pg = a.num_pages;
            }
            return (pg * a.Hkv + g) * kNk;
        };
        // kSplit: lane 0 streams the K half of every ring step and lane 1 the
        // V half, each on its own barriers, so a stage's K region is reloaded
        // as soon as the step's score MMAs have read it, its V region once the
        // P V MMAs have; in long loops over tiles no other CTA shares, the K
        // loads then run ahead of the P V MMAs (7B batch-16 layer 57.3 -> 53.5
        // us in a probe chain).  Otherwise lane 0 loads whole stages on one
        // barrier each: where several row tiles share each tile through L2
        // (the tree) or the loop fits the ring (batch 1) the split measured
        // slower (27.4 -> 28.4 us, 8.17 -> 8.30 us).
        auto load_step = [&](int i, bool vp) {
            const int s = i % kStages;
            uint64_t* ful = vp ? &v_full[s] : &k_full[s];
            mbar_wait(vp ? &v_empty[s] : &k_empty[s], ((i / kStages) & 1) ^ 1, a.err);
            const int t0 = first + i * kT, nt = min(kT, last - t0);
            uint8_t* st = smem + Ly::kOffRing + s * kStageBytes;
            mbar_arrive_expect_tx(ful, static_cast<uint32_t>(nt * (kSplit ? kTileBytes / 2 : kTileBytes)));
            for (int h = 0; h < nt; ++h) {
                const int gt = t0 + h;
                const void* tk = gt < n_ctx ? static_cast<const void*>(&tmK) : static_cast<const void*>(&tmKb);
                const void* tv = gt < n_ctx ? static_cast<const void*>(&tmV) : static_cast<const void*>(&tmVb);
                const int y = gt < n_ctx ? ctx_row(gt) : hg * a.R + (gt - n_ctx) * kNk;
                if (!kSplit || !vp) {
                    tma_load_2d(st + h * kHalfBytes, tk, 0, y, ful);
                    tma_load_2d(st + kRegion + h * kHalfBytes, tk, 64, y, ful);
                }
                if (!kSplit || vp) {
                    tma_load_2d(st + 2 * kRegion + h * kHalfBytes, tv, 0, y, ful);
                    tma_load_2d(st + 3 * kRegion + h * kHalfBytes, tv, 64, y, ful);
                }
            }
        };
        if (kSplit ? lane < 2 : lane == 0) {
            const bool vp = kSplit && lane == 1;
            int i = 0;
            if (early) {
                // the first ring pass of context-only steps, while the preceding
                // kernel drains (committed rows: no kernel writes them now)
                for (; i < nsteps && i < kStages && min(first + (i + 1) * kT, last) <= n_ctx; ++i) load_step(i, vp);
            }
            if (early) pdl_wait();
            for (; i < nsteps; ++i) load_step(i, vp);
        } else if (early) {
            pdl_wait();
        }
        __syncwarp();
        merge_plan(need, light);
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        merge_plan(need, light);   // before the wait (cache_ready) or while the Q tile is on its way
        if (early) pdl_wait();
        if (lane == 0 && ntiles > 0) {
            // S = Q K^T over the step's tiles (N = 64 per tile), O += P V
            constexpr uint32_t idesc_s = idesc_bf16_f32(kM, kStepKeys, false, false);
            constexpr uint32_t idesc_s1 = idesc_bf16_f32(kM, kNk, false, false);      // a last, single tile
            constexpr uint32_t idesc_o = idesc_bf16_f32(kM, kD, false, true);
            const uint32_t sq = smem_u32(smem + Ly::kOffQ);
            // both S operands K-major; the two 64-dim halves are separate boxes
            const uint64_t qd0 = smem_desc_sw128(sq, 16, 1024);
            mbar_wait(q_ready, 0, a.err);
            if constexpr (!(kHalf && kHW == 2)) {
                // Long loops (four row-owner warps per quadrant, or full tiles): every
                // step but the last takes kT tiles, so its MMA chains are issued with
                // compile-time trip counts (a run-time count cost the single issuing
                // thread ~12-40 cycles per MMA in a probe, against ~65 for the MMA
                // itself; the tree layer 24.7 -> 23.8 us).  The last step picks its
                // variant once.  Short loops (batch 1: two or three steps, two warps
                // per quadrant, the only ones that fold an odd tile) keep the single
                // loop below: there the separate variants' code, run once per CTA,
                // cost more than the chains saved (1.5B layer 8.12 -> 8.34 us).
                using NtFull = std::integral_constant<int, kT>;
                using NtOne = std::integral_constant<int, 1>;
                using NoFold = std::false_type;
                using Fold = std::true_type;
                auto pv = [&](int st, auto nt_c, auto fold_c) {
                    constexpr int NT = decltype(nt_c)::value;
                    constexpr bool FOLD = decltype(fold_c)::value;
                    const int pb = st & 1, s = st % kStages;
                    mbar_wait(&p_full[pb], (st >> 1) & 1, a.err);
                    // (one barrier per stage: S already waited for the whole stage)
                    if constexpr (kSplit) mbar_wait(&v_full[s], (st / kStages) & 1, a.err);
                    tc_fence_after();
                    // A = P [M lanes][keys] in TMEM (8 columns per 16 keys); B = V
                    // [keys][128 dims], MN-major: 8-key groups 1024 B apart (keys run
                    // on across the step's tiles), the two 64-dim halves one region
                    // apart, 16 keys = 2048 B (descriptor units of 16 B)
                    const uint32_t sv = smem_u32(smem + Ly::kOffRing + s * kStageBytes + 2 * kRegion);
                    const uint64_t bd0 = smem_desc_sw128(sv, kRegion, 1024);
                    const uint32_t acc0 = st > 0 ? 1u : 0u;
    #pragma unroll
                    for (int kc = 0; kc < NT * (kNk / 16); ++kc)
                        tc_mma_ts(tO, tP(pb) + kc * 8, bd0 + kc * (2048 >> 4), idesc_o, kc > 0 ? 1u : acc0);
                    if constexpr (FOLD) {
                        // the folded tile: P in the other P buffer, V in ring step st + 1
                        const int sx = (st + 1) % kStages;
                        if constexpr (kSplit) mbar_wait(&v_full[sx], ((st + 1) / kStages) & 1, a.err);
                        tc_fence_after();
                        const uint64_t bdx =
                            smem_desc_sw128(smem_u32(smem + Ly::kOffRing + sx * kStageBytes + 2 * kRegion), kRegion, 1024);
    #pragma unroll
                        for (int kc = 0; kc < kNk / 16; ++kc)
                            tc_mma_ts(tO, tP(pb ^ 1) + kc * 8, bdx + kc * (2048 >> 4), idesc_o, 1u);
                        tc_commit(&v_empty[sx]);
                    }
                    tc_commit(&o_done[pb]);
                    tc_commit(&v_empty[s]);
                };
                auto scores = [&](int st, auto nt_c, auto fold_c) {
                    constexpr int NT = decltype(nt_c)::value;
                    constexpr bool FOLD = decltype(fold_c)::value;
                    const int sb = st & 1, s = st % kStages;
                    mbar_wait(&s_empty[sb], ((st >> 1) & 1) ^ 1, a.err);
                    mbar_wait(&k_full[s], (st / kStages) & 1, a.err);
                    tc_fence_after();
                    const uint64_t kd0 = smem_desc_sw128(smem_u32(smem + Ly::kOffRing + s * kStageBytes), 16, 1024);
                    constexpr uint32_t id = NT == kT ? idesc_s : idesc_s1;
    #pragma unroll
                    for (int k16 = 0; k16 < kD / 16; ++k16) {
                        const uint32_t half = k16 >> 2, kin = (k16 & 3) * 32;
                        tc_mma(tS(sb), qd0 + ((half * (kM * 128) + kin) >> 4), kd0 + ((half * kRegion + kin) >> 4), id,
                               k16 > 0 ? 1u : 0u);
                    }
                    if constexpr (FOLD) {
                        // the folded tile (ring step st + 1): scores into the first 64
                        // columns of the other buffer, once step st - 1 has read it
                        const int sx = (st + 1) % kStages;
                        if (st >= 1) mbar_wait(&s_empty[sb ^ 1], ((st - 1) >> 1) & 1, a.err);
                        mbar_wait(&k_full[sx], ((st + 1) / kStages) & 1, a.err);
                        tc_fence_after();
                        const uint64_t kdx = smem_desc_sw128(smem_u32(smem + Ly::kOffRing + sx * kStageBytes), 16, 1024);
    #pragma unroll
                        for (int k16 = 0; k16 < kD / 16; ++k16) {
                            const uint32_t half = k16 >> 2, kin = (k16 & 3) * 32;
                            tc_mma(tS(sb ^ 1), qd0 + ((half * (kM * 128) + kin) >> 4),
                                   kdx + ((half * kRegion + kin) >> 4), idesc_s1, k16 > 0 ? 1u : 0u);
                        }
                        if constexpr (kSplit) tc_commit(&k_empty[sx]);
                    }
                    if constexpr (kSplit) tc_commit(&k_empty[s]);   // K of this step read once these MMAs are done
                    tc_commit(&s_full[sb]);
                };
                const int last = nsoft - 1;
                for (int st = 0; st < last; ++st) {
                    scores(st, NtFull{}, NoFold{});
                    if (st > 0) pv(st - 1, NtFull{}, NoFold{});
                }
                // the last step: kT tiles or one tile
                if (ntiles - last * kT >= kT) {
                    scores(last, NtFull{}, NoFold{});
                    if (last > 0) pv(last - 1, NtFull{}, NoFold{});
                    pv(last, NtFull{}, NoFold{});
                } else {
                    scores(last, NtOne{}, NoFold{});
                    if (last > 0) pv(last - 1, NtFull{}, NoFold{});
                    pv(last, NtOne{}, NoFold{});
                }
            } else {
                auto pv = [&](int st) {
                    const int pb = st & 1, s = st % kStages;
                    const int nt = min(kT, ntiles - st * kT);
                    mbar_wait(&p_full[pb], (st >> 1) & 1, a.err);
                    // (one barrier per stage: S already waited for the whole stage)
                    if constexpr (kSplit) mbar_wait(&v_full[s], (st / kStages) & 1, a.err);
                    tc_fence_after();
                    // A = P [M lanes][keys] in TMEM (8 columns per 16 keys); B = V
                    // [keys][128 dims], MN-major: 8-key groups 1024 B apart (keys run
                    // on across the step's tiles), the two 64-dim halves one region
                    // apart, 16 keys = 2048 B (descriptor units of 16 B)
                    const uint32_t sv = smem_u32(smem + Ly::kOffRing + s * kStageBytes + 2 * kRegion);
                    const uint64_t bd0 = smem_desc_sw128(sv, kRegion, 1024);
                    for (int kc = 0; kc < nt * (kNk / 16); ++kc)
                        tc_mma_ts(tO, tP(pb) + kc * 8, bd0 + kc * (2048 >> 4), idesc_o, (st > 0 || kc > 0) ? 1u : 0u);
                    if (fold && st == nsoft - 1) {
                        // the folded tile: P in the other P buffer, V in ring step st + 1
                        const int sx = (st + 1) % kStages;
                        if constexpr (kSplit) mbar_wait(&v_full[sx], ((st + 1) / kStages) & 1, a.err);
                        tc_fence_after();
                        const uint64_t bdx =
                            smem_desc_sw128(smem_u32(smem + Ly::kOffRing + sx * kStageBytes + 2 * kRegion), kRegion, 1024);
                        for (int kc = 0; kc < kNk / 16; ++kc)
                            tc_mma_ts(tO, tP(pb ^ 1) + kc * 8, bdx + kc * (2048 >> 4), idesc_o, 1u);
                        tc_commit(&v_empty[sx]);
                    }
                    tc_commit(&o_done[pb]);
                    tc_commit(&v_empty[s]);
                };
                for (int st = 0; st < nsoft; ++st) {
                    const int sb = st & 1, s = st % kStages;
                    const int nt = min(kT, ntiles - st * kT);
                    mbar_wait(&s_empty[sb], ((st >> 1) & 1) ^ 1, a.err);
                    mbar_wait(&k_full[s], (st / kStages) & 1, a.err);
                    tc_fence_after();
                    const uint64_t kd0 = smem_desc_sw128(smem_u32(smem + Ly::kOffRing + s * kStageBytes), 16, 1024);
                    const uint32_t id = nt == kT ? idesc_s : idesc_s1;
    #pragma unroll
                    for (int k16 = 0; k16 < kD / 16; ++k16) {
                        const uint32_t half = k16 >> 2, kin = (k16 & 3) * 32;
                        tc_mma(tS(sb), qd0 + ((half * (kM * 128) + kin) >> 4), kd0 + ((half * kRegion + kin) >> 4), id,
                               k16 > 0 ? 1u : 0u);
                    }
                    if (fold && st == nsoft - 1) {
                        // the folded tile (ring step st + 1): scores into the first 64
                        // columns of the other buffer, once step st - 1 has read it
                        const int sx = (st + 1) % kStages;
                        if (st >= 1) mbar_wait(&s_empty[sb ^ 1], ((st - 1) >> 1) & 1, a.err);
                        mbar_wait(&k_full[sx], ((st + 1) / kStages) & 1, a.err);
                        tc_fence_after();
                        const uint64_t kdx = smem_desc_sw128(smem_u32(smem + Ly::kOffRing + sx * kStageBytes), 16, 1024);
    #pragma unroll
                        for (int k16 = 0; k16 < kD / 16; ++k16) {
                            const uint32_t half = k16 >> 2, kin = (k16 & 3) * 32;
                            tc_mma(tS(sb ^ 1), qd0 + ((half * (kM * 128) + kin) >> 4),
                                   kdx + ((half * kRegion + kin) >> 4), idesc_s1, k16 > 0 ? 1u : 0u);
                        }
                        if constexpr (kSplit) tc_commit(&k_empty[sx]);
                    }
                    if constexpr (kSplit) tc_commit(&k_empty[s]);   // K of this step read once these MMAs are done
                    tc_commit(&s_full[sb]);
                    if (st > 0) pv(st - 1);
                }
                pv(nsoft - 1);
            }
        }
    } else {
        // ---------------- row-owner warps ----------------
        if (early) {
            merge_plan(need, light);
            pdl_wait();
        }
        if (bad_len && threadIdx.x == 0 && rank == 0 && rt == 0) raise_error(a.err, SV_DEVERR_LENGTH);
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
        // gather the Q tile (zero rows for padding lanes) into the K-major
        // 128-byte-swizzled layout the MMA reads
        {
            uint8_t* q_s = smem + Ly::kOffQ;
            for (int x = threadIdx.x; x < kM * 16; x += 32 * kSoftWarps) {
                const int row = x >> 4, c = x & 15;   // row of the MMA's A operand
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                // half tiles: A row m sits in TMEM lane 32 * (m / 16) + m % 16 and
                // carries row 4 * (m % 16) + m / 16 of (b, g)
                const int grow = rt * kTileRows + (kHalf ? 4 * (row & 15) + (row >> 4) : row);
                const int half = c >> 3, cc = c & 7;
                uint8_t* dst = q_s + half * (kM * 128) + row * 128 + ((cc ^ (row & 7)) << 4);
                if (grow < a.rows) {
                    // all of a thread's copies in flight at once
                    const int jr = grow / a.G, hl = grow % a.G;
                    const uint16_t* src = a.q + ((static_cast<size_t>(b) * a.R + jr) * a.Hq + g * a.G + hl) * kD;
                    cp_async16(dst, reinterpret_cast<const uint4*>(src) + c);
                } else {
                    *reinterpret_cast<uint4*>(dst) = v;
                }
            }
            if (!early) merge_plan(need, light);   // while the Q copies are in flight
            cp_async_wait_all();
        }
        fence_proxy_async_smem();
        named_barrier(1, 32 * kSoftWarps);   // anc and Q written by every row-owner warp
        if (lane == 0) mbar_arrive(q_ready);

        // this thread's row: TMEM lane r (also its P row), row gr of (b, g)
        const int q4 = warp & 3;   // TMEM quadrant = SM sub-partition
        const int r = kHalf ? (q4 * 32 + (lane & 15)) : (q4 * 32 + lane);
        const int gr = rt * kTileRows + (kHalf ? 4 * (lane & 15) + q4 : r);
        const bool valid = gr < a.rows;
        const int j = valid ? gr / a.G : 0;
        // the warp's quadrant holds at least one real row (padding lanes' P and
        // O are never read, so a warp with none skips the arithmetic)
        const bool quarter_live = rt * kTileRows + (kHalf ? q4 : q4 * 32) < a.rows;
        const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
        // full tiles: 16 consecutive columns of the one-tile step (group cgp);
        // half tiles: 32 columns -- key tile `sub` of the step (thread half of
        // the warp), its column half `cgp` (the quadrant's warp)
        constexpr int kCols = kHalf ? kStepKeys / (2 * kHalfWarps) : kStepKeys / kGroups;
        const int cgp = warp / 4;
        const int sub = kHalf ? (lane >> 4) : 0;
        const int col0 = kHalf ? sub * (kStepKeys / 2) + cgp * kCols : cgp * kCols;   // S columns of the step
        const int tsub = col0 / kNk, ctile = col0 % kNk;     // tile within the step, first key in it
        // tree: this thread's windows of the row's ancestor mask, one per block
        // tile (block keys ctile.. of tile 0 and of tile 1)
        using Win = typename std::conditional<(kCols > 32), uint64_t, uint32_t>::type;
        Win win_t0 = 0, win_t1 = 0;
        if (tree && valid) {
            win_t0 = static_cast<Win>(anc[2 * j] >> ctile);
            win_t1 = static_cast<Win>(anc[2 * j + 1] >> ctile);
        }
        float* red = reinterpret_cast<float*>(smem + Ly::kOffRed);
        float* lsx = reinterpret_cast<float*>(smem + Ly::kOffLsum);
        // the folded tile (the CTA's last): this thread's 16 of its 64 columns,
        // 32 sub + 16 cgp .., and for a tree block tile the ancestor window there
        constexpr int kCX = kNk / 4;
        const int cx0 = sub * (kNk / 2) + cgp * kCX;
        uint32_t winx = 0;
        if (kTree && fold && valid && last - 1 >= n_ctx)
            winx = static_cast<uint32_t>(anc[2 * j + (last - 1 - n_ctx)] >> cx0) & 0xFFFFu;

        float m_ref = -INFINITY, lsum = 0.f;
        for (int st = 0; st < nsoft; ++st) {
            const int sb = st & 1;
            const bool fx = fold && st == nsoft - 1;   // this step also takes the folded tile
            mbar_wait(&s_full[sb], (st >> 1) & 1, a.err);
            tc_fence_after();
            const bool work = quarter_live;
            if constexpr (!kHalf) {
                // Full tiles: 32 columns per thread.  The max pass and the
                // exponent pass each read them from TMEM in one 32-column load
                // (one round trip each); P goes back in two 16-column stores, so
                // the exponent pass holds 32 scores and 8 packed P words at most
                // (holding all 16 P words besides spilled at the 96 registers an
                // 18-warp CTA leaves each thread)
                const int ti = st * kT + tsub;
                const bool tile_live = ti < ntiles;
                const int gt = first + ti;
                const bool is_block = gt >= n_ctx;
                const int kb = (is_block ? (gt - n_ctx) * kNk : gt * kNk) + ctile;
                // visibility of this thread's 32 keys as one bit mask, formed once
                // per step (context: kl < t; chain block: kl <= j and kl < R; no
                // tile: none; tree block: the ancestor window, read from shared
                // memory), so that chains and trees run the same per-key code and
                // unmasked steps skip it; a per-key choice between the tree and the
                // length test, kept by the compiler in every step, doubled the
                // tree variant's step time
                const bool masked = is_block || kb + kCols > t || !tile_live;
                uint32_t vmask = ~0u;
                if (masked) {
                    const int lim = !tile_live ? 0 : !is_block ? t - kb : (j + 1 < a.R ? j + 1 : a.R) - kb;
                    vmask = lim >= 32 ? ~0u : lim <= 0 ? 0u : (1u << lim) - 1u;
                    if (kTree && is_block && tile_live) vmask = static_cast<uint32_t>(anc[2 * j + (gt - n_ctx)] >> ctile);
                }
                // all 32 columns in one TMEM round trip per pass
                auto load_all = [&](uint32_t (&v)[32]) {
                    tmem_ld32_sync(tS(sb) + lane_off + col0, v);
                    if (vmask != ~0u) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = ((vmask >> e) & 1u) != 0u ? v[e] : __float_as_uint(-INFINITY);
                    }
                };
                float mpart = -INFINITY;
                if (work) {
                    uint32_t v[32];
                    load_all(v);
                    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            mq[u] = fmax3(mq[u], __uint_as_float(v[e + 2 * u]), __uint_as_float(v[e + 2 * u + 1]));
                    mpart = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * a.scale_log2;
                }
                // a row's four column groups are the quadrant's four warps:
                // one 128-thread barrier per quadrant
                red[(sb * kGroups + cgp) * kRows + r] = mpart;
                named_barrier(3 + q4, 128);
                float mt = red[(sb * kGroups + 0) * kRows + r];
#pragma unroll
                for (int c2 = 1; c2 < kGroups; ++c2) mt = fmaxf(mt, red[(sb * kGroups + c2) * kRows + r]);
                float m_new = m_ref, corr = 1.f;
                if (mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescale)) {
                    m_new = mt;
                    corr = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - m_new);
                }
                // P buffer sb is free once the P V of step st-2 is done; O is
                // rescaled once the P V of step st-1 has settled it
                if (st >= 2) {
                    mbar_wait(&o_done[sb], ((st - 2) >> 1) & 1, a.err);
                    tc_fence_after();
                }
                if (quarter_live && st >= 1 && __any_sync(0xffffffffu, corr != 1.f)) {
                    mbar_wait(&o_done[sb ^ 1], ((st - 1) >> 1) & 1, a.err);
                    tc_fence_after();
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
                float ps0 = 0.f, ps1 = 0.f;
                if (work) {
                    const float nm = m_new == -INFINITY ? 0.f : -m_new;
                    uint32_t v[32];
                    load_all(v);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float p0 = fast_exp2(fmaf(__uint_as_float(v[16 * h + e]), a.scale_log2, nm));
                            const float p1 = fast_exp2(fmaf(__uint_as_float(v[16 * h + e + 1]), a.scale_log2, nm));
                            ps0 += p0;
                            ps1 += p1;
                            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                            pk[e / 2] = *reinterpret_cast<const uint32_t*>(&pb);
                        }
                        tmem_st8(tP(sb) + lane_off + (col0 + 16 * h) / 2, pk);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                lsum = lsum * corr + (ps0 + ps1);
                m_ref = m_new;
            } else {
            uint32_t rs[kCols];
            uint32_t rx[kCX];
            if constexpr (kHalf && kHW == 2) {
                if (work && fx) tmem_ld16_h_sync<kNk / 2>(tS(sb ^ 1) + lane_off + cgp * kCX, rx);
            }
            if (work) {
                // columns 32 cgp .. of the step's first tile (threads 0-15)
                // and of its second tile (threads 16-31)
                if constexpr (kCols == 32) tmem_ld32_h_sync<kStepKeys / 2>(tS(sb) + lane_off + cgp * kCols, rs);
                else tmem_ld16_h_sync<kStepKeys / 2>(tS(sb) + lane_off + cgp * kCols, rs);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[sb]);
            const int ti = st * kT + tsub;            // this thread's tile of the CTA's range
            const bool tile_live = ti < ntiles;       // a last, odd step has one tile
            const int gt = first + ti;
            const bool is_block = gt >= n_ctx;
            const int kb = (is_block ? (gt - n_ctx) * kNk : gt * kNk) + ctile;
            // rs holds the raw q.k bits (scaled in the exponent), masked in place
            float mpart = -INFINITY;
            if (work) {
                if (is_block || kb + kCols > t || !tile_live) {
                    // branch-free mask: key kb + e is visible iff e < lim (context:
                    // kl < t; chain block: kl <= j and kl < R; no tile: none) or,
                    // for a tree block, iff bit e of the ancestor window is set
                    const bool tree_blk = kTree && is_block && tile_live;
                    const int lim = !tile_live ? 0 : !is_block ? t - kb : (j + 1 < a.R ? j + 1 : a.R) - kb;
                    const Win win = tree_blk ? (gt - n_ctx == 0 ? win_t0 : win_t1) : Win(0);
#pragma unroll
                    for (int e = 0; e < kCols; ++e) {
                        const bool vis = tree_blk ? ((win >> e) & Win(1)) != Win(0) : e < lim;
                        rs[e] = vis ? rs[e] : __float_as_uint(-INFINITY);
                    }
                }
                // four running maxima of three-input max.f32 (short chains)
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kCols; e += 8)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        mq[u] = fmax3(mq[u], __uint_as_float(rs[e + 2 * u]), __uint_as_float(rs[e + 2 * u + 1]));
                mpart = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * a.scale_log2;   // the scale is positive
                if (fx) {
                    // the folded tile's columns: the same mask, its own key base
                    const int gtx = last - 1;
                    const bool blk_x = gtx >= n_ctx;
                    const int kbx = (blk_x ? (gtx - n_ctx) * kNk : gtx * kNk) + cx0;
                    if (blk_x || kbx + kCX > t) {
                        const bool tree_x = kTree && blk_x;
                        const int limx = !blk_x ? t - kbx : (j + 1 < a.R ? j + 1 : a.R) - kbx;
#pragma unroll
                        for (int e = 0; e < kCX; ++e) {
                            const bool vis = tree_x ? ((winx >> e) & 1u) != 0u : e < limx;
                            rx[e] = vis ? rx[e] : __float_as_uint(-INFINITY);
                        }
                    }
                    float mxx = -INFINITY;
#pragma unroll
                    for (int e = 0; e < kCX; e += 2)
                        mxx = fmax3(mxx, __uint_as_float(rx[e]), __uint_as_float(rx[e + 1]));
                    mpart = fmaxf(mpart, mxx * a.scale_log2);
                }
            }
            // the row's other tile sits 16 lanes away in the same warp, its
            // other column half in the quadrant's other warp
            float mt = fmaxf(mpart, __shfl_xor_sync(0xffffffffu, mpart, 16));
            red[(sb * kGroups + cgp) * kRows + r] = mt;
            named_barrier(3 + q4, 32 * kHalfWarps);
#pragma unroll
            for (int c2 = 0; c2 < kHalfWarps; ++c2) mt = fmaxf(mt, red[(sb * kGroups + c2) * kRows + r]);
            float m_new = m_ref, corr = 1.f;
            if (mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescale)) {
                m_new = mt;
                corr = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - m_new);
            }
            // P (bf16, rounded to nearest even) and this thread's share of the
            // row sum (of the fp32 values).  exp2(scale * s - m) is one FMA and
            // one ex2; a row with no visible key yet (m = -inf) has every score
            // -inf, and exp2(-inf - 0) = 0.
            uint32_t pk[kCols / 2];
            uint32_t pkx[kCX / 2];
            float ps0 = 0.f, ps1 = 0.f;
            if (work) {
                const float nm = m_new == -INFINITY ? 0.f : -m_new;
#pragma unroll
                for (int e = 0; e < kCols; e += 2) {
                    const float p0 = fast_exp2(fmaf(__uint_as_float(rs[e]), a.scale_log2, nm));
                    const float p1 = fast_exp2(fmaf(__uint_as_float(rs[e + 1]), a.scale_log2, nm));
                    ps0 += p0;
                    ps1 += p1;
                    const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                    pk[e / 2] = *reinterpret_cast<const uint32_t*>(&pb);
                }
                if (fx) {
#pragma unroll
                    for (int e = 0; e < kCX; e += 2) {
                        const float p0 = fast_exp2(fmaf(__uint_as_float(rx[e]), a.scale_log2, nm));
                        const float p1 = fast_exp2(fmaf(__uint_as_float(rx[e + 1]), a.scale_log2, nm));
                        ps0 += p0;
                        ps1 += p1;
                        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                        pkx[e / 2] = *reinterpret_cast<const uint32_t*>(&pb);
                    }
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
                // O columns 64 sub + (64 / kHalfWarps) cgp .. of the row
#pragma unroll
                for (int c0 = 0; c0 < kD / (2 * kHalfWarps); c0 += 16) {
                    const uint32_t ta = tO + lane_off + cgp * (kD / (2 * kHalfWarps)) + c0;
                    uint32_t o16[16];
                    tmem_ld16_h_sync<kD / 2>(ta, o16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) o16[e] = __float_as_uint(__uint_as_float(o16[e]) * corr);
                    tmem_st16_h<kD / 2>(ta, o16);
                }
                tmem_st_wait();
            }
            if (work) {
                // P of this thread's columns into TMEM buffer sb, two keys per column
                if constexpr (kCols == 32) tmem_st16_h<kStepKeys / 4>(tP(sb) + lane_off + cgp * (kCols / 2), pk);
                else tmem_st8_h<kStepKeys / 4>(tP(sb) + lane_off + cgp * (kCols / 2), pk);
                tmem_st_wait();
            }
            if constexpr (kHalf && kHW == 2) {
                if (fx) {
                    // the folded tile's P into the other P buffer once the P V of
                    // step st - 1 has read it: P columns 16 sub + 8 cgp ..
                    if (st >= 1) {
                        mbar_wait(&o_done[sb ^ 1], ((st - 1) >> 1) & 1, a.err);
                        tc_fence_after();
                    }
                    if (work) {
                        tmem_st8_h<kNk / 4>(tP(sb ^ 1) + lane_off + cgp * (kCX / 2), pkx);
                        tmem_st_wait();
                    }
                }
            }
            }
            {
                // V rows of cache positions >= t in the last, partial context
                // tile: P is 0 there, but 0 * a non-finite cache entry is NaN in
                // P V, so they are zeroed before the P V of this step
                const int tl = n_ctx - 1 - first - st * kT;   // that tile within this step
                if ((t & (kNk - 1)) != 0 && tl >= 0 && tl < kT && tl < ntiles - st * kT) {
                    // with split barriers V lands on its own: wait for it before
                    // zeroing rows (otherwise the score MMAs waited for the stage)
                    if constexpr (kSplit) mbar_wait(&v_full[st % kStages], (st / kStages) & 1, a.err);
                    uint8_t* vt = smem + Ly::kOffRing + (st % kStages) * kStageBytes + 2 * kRegion + tl * kHalfBytes;
                    const int r0 = t & (kNk - 1);
                    for (int x = threadIdx.x; x < (kNk - r0) * 16; x += 32 * kSoftWarps) {
                        const int row = r0 + (x >> 4), c = x & 15;   // a whole 128-byte row of each half
                        *reinterpret_cast<uint4*>(vt + (c >> 3) * kRegion + row * 128 + (c & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                if (fx && (t & (kNk - 1)) != 0 && last - 1 == n_ctx - 1) {
                    // ... and the folded tile when it is that tile (ring step st + 1)
                    if constexpr (kSplit) mbar_wait(&v_full[(st + 1) % kStages], ((st + 1) / kStages) & 1, a.err);
                    uint8_t* vt = smem + Ly::kOffRing + ((st + 1) % kStages) * kStageBytes + 2 * kRegion;
                    const int r0 = t & (kNk - 1);
                    for (int x = threadIdx.x; x < (kNk - r0) * 16; x += 32 * kSoftWarps) {
                        const int row = r0 + (x >> 4), c = x & 15;
                        *reinterpret_cast<uint4*>(vt + (c >> 3) * kRegion + row * 128 + (c & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
        }
        if (nsoft > 0) {
            mbar_wait(&o_done[(nsoft - 1) & 1], ((nsoft - 1) >> 1) & 1, a.err);
            tc_fence_after();
        }
        // row sum across the row's threads -> this CTA's partial record, kept
        // by row of (b, g) relative to the tile
        float lt;
        if constexpr (kHalf) {
            lt = lsum + __shfl_xor_sync(0xffffffffu, lsum, 16);
            lsx[cgp * kRows + r] = lt;
            named_barrier(3 + q4, 32 * kHalfWarps);
            lt = 0.f;
#pragma unroll
            for (int c2 = 0; c2 < kHalfWarps; ++c2) lt += lsx[c2 * kRows + r];
        } else {
            lsx[cgp * kRows + r] = lsum;
            named_barrier(3 + q4, 128);   // the row's four column groups: the quadrant's warps
            lt = 0.f;
#pragma unroll
            for (int c2 = 0; c2 < kGroups; ++c2) lt += lsx[c2 * kRows + r];
        }
        const bool use = nsteps >= 1 && lt > 0.f;
        // O of this thread's columns, held in registers across the barrier
        constexpr int kOCols = kHalf ? kD / (2 * kHalfWarps) : kD / kGroups;   // O columns per thread
        const int ocol0 = kHalf ? sub * (kD / 2) + cgp * kOCols : cgp * (kD / kGroups);
        uint32_t ov[kOCols];
#pragma unroll
        for (int c0 = 0; c0 < kOCols; c0 += 16) {
            uint32_t(&o16)[16] = *reinterpret_cast<uint32_t(*)[16]>(ov + c0);
            // the condition of a warp-collective TMEM load must be warp-uniform
            // (nsteps is; `use` is per row)
            if (nsteps >= 1) {
                if constexpr (kHalf) tmem_ld16_h_sync<kD / 2>(tO + lane_off + cgp * kOCols + c0, o16);
                else tmem_ld16_sync(tO + lane_off + ocol0 + c0, o16);
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) o16[e] = (nsteps >= 1 && use) ? o16[e] : 0u;
        }
        tc_fence_before();
        __syncwarp();
        pdl_launch_dependents();             // see the note at the programmatic-launch wait
        cluster_wait();                      // every CTA of the cluster has started
        if (need == 0 && xch == nullptr) cluster_sync_warp();  // (1) and has drained its ring
        if (valid && xch != nullptr) {
            // the partial row into this CTA's block of the L2 exchange (a warp's
            // 32 rows of one column chunk are one contiguous 512-byte store)
            const int prow = gr - rt * kTileRows;
            float* xmine = xch + static_cast<size_t>(blockIdx.y * gridDim.x + blockIdx.x) * Ly::kXchFloats;
            if (cgp == 0 && sub == 0)
                __stcg(reinterpret_cast<float2*>(xmine) + prow, make_float2(use ? m_ref : -INFINITY, use ? lt : 0.f));
            uint4* xo = reinterpret_cast<uint4*>(xmine + 2 * kTileRows);
#pragma unroll
            for (int e = 0; e < kOCols; e += 4)
                __stcg(xo + ((ocol0 + e) >> 2) * kTileRows + prow, make_uint4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]));
        } else if (valid) {
            // push the partial record of row prow into slot `rank` of the row's
            // owner: slots [(prow / n_owners) * C + src] of its receive area
            const int prow = gr - rt * kTileRows;      // < kTileRows for every real row
            int owner, li;
            if (need > 0) {
                const int nl = __popc(light);
                uint32_t m = light;
                for (int k = prow % nl; k > 0; --k) m &= m - 1u;   // the (prow % nl)-th light CTA
                owner = __ffs(m) - 1;
                li = prow / nl;
            } else {
                owner = prow % C;
                li = prow / C;
            }
            float* recv = need > 0 ? reinterpret_cast<float*>(smem + Ly::kOffRing + (kStages - need) * kStageBytes)
                                   : part;
            float* rec = cluster.map_shared_rank(recv + (li * C + rank) * kRec, owner);
            if (cgp == 0 && sub == 0)
                *reinterpret_cast<float2*>(rec) = make_float2(use ? m_ref : -INFINITY, use ? lt : 0.f);
#pragma unroll
            for (int e = 0; e < kOCols; e += 4)
                *reinterpret_cast<uint4*>(rec + 4 + ocol0 + e) = make_uint4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
        }
    }
    if (warp >= kSoftWarps) {   // producer and MMA warps, once their lane 0 is done
        __syncwarp();
        pdl_launch_dependents();
        cluster_wait();
        if (need == 0 && xch == nullptr) cluster_sync_warp();   // (1)
    }
    __syncwarp();
    cluster_sync_warp();   // (2) every record pushed (or stored) and visible to its owner

    // merge: this CTA finalises rows rank, rank + C, ... of the row tile (all
    // warps) from the records pushed to it; with one cluster per (b, g, row
    // tile) it writes the bf16 rows, otherwise the cluster's merged partial
    // (max, sum, unnormalised O)
    const int unit = hg * a.row_tiles + rt;
    const int ci = blockIdx.x / C;
    auto store_row = [&](int lr, float4 acc, float L) {
        const float inv = L > 0.f ? 1.0f / L : 0.f;
        const int row = rt * kTileRows + lr;
        const int jr = row / a.G, h = g * a.G + row % a.G;
        uint16_t* dst = a.out + ((static_cast<size_t>(b) * a.R + jr) * a.Hq + h) * kD + 4 * lane;
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    };
    // the rows this CTA owns: k0, k0 + n_owners, ...
    const bool owns = need == 0 || ((light >> rank) & 1u) != 0u;
    const int k0 = need > 0 ? __popc(light & ((1u << rank) - 1u)) : rank;
    const int n_owners = need > 0 ? __popc(light) : C;
    const float* recv = need > 0 ? reinterpret_cast<const float*>(smem + Ly::kOffRing + (kStages - need) * kStageBytes)
                                 : part;
    if (xch != nullptr) {
        // merge from the L2 exchange: units of (32-row group, 4-column chunk)
        // split evenly over the cluster's CTAs, up to two per warp at a time;
        // lane l takes row 32 * group + l, so each load of a source's partial
        // is one contiguous 512-byte (O) or 256-byte (max, sum) piece.  The
        // rows' weights are formed once per CTA (a warp per row group) while
        // the first O pieces are in flight, and shared through shared memory
        // (the drained ring): one round of loads for the whole merge
        constexpr int kCh = kD / 4, kNW = kThreads / 32, kX = kXchMaxCluster;
        const int nunits = ((nrows + 31) / 32) * kCh;
        const int per = (nunits + C - 1) / C;
        const int u0 = min(nunits, rank * per), u1 = min(nunits, u0 + per);
        const int g0 = u0 / kCh, ng = u1 > u0 ? (u1 - 1) / kCh - g0 + 1 : 0;
        const float* xb = xch + static_cast<size_t>(blockIdx.y * gridDim.x + blockIdx.x - rank) * Ly::kXchFloats;
        float* wsm = reinterpret_cast<float*>(smem + Ly::kOffRing);   // [group][kX weights, M, L][32 rows]
        auto load_unit = [&](int u, float4 (&x)[kX]) {
            const int lr = (u / kCh) * 32 + lane, ch = u % kCh;
#pragma unroll
            for (int sr = 0; sr < kX; ++sr) {
                x[sr] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (u < u1 && lr < nrows && sr < C)
                    x[sr] = __ldcg(reinterpret_cast<const float4*>(xb + sr * Ly::kXchFloats + 2 * kTileRows) +
                                   ch * kTileRows + lr);
            }
        };
        auto finish_unit = [&](int u, const float4 (&x)[kX]) {
            const int lr = (u / kCh) * 32 + lane, ch = u % kCh;
            if (u >= u1 || lr >= nrows) return;
            const float* wr = wsm + (u / kCh - g0) * (kX + 2) * 32 + lane;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int sr = 0; sr < kX; ++sr) {
                const float w = sr < C ? wr[sr * 32] : 0.f;
                acc.x += w * x[sr].x;
                acc.y += w * x[sr].y;
                acc.z += w * x[sr].z;
                acc.w += w * x[sr].w;
            }
            const float M = wr[kX * 32], L = wr[(kX + 1) * 32];
            if (a.clusters == 1) {
                const float inv = L > 0.f ? 1.0f / L : 0.f;
                const int row = rt * kTileRows + lr;
                const int jr = row / a.G, h = g * a.G + row % a.G;
                uint16_t* dst = a.out + ((static_cast<size_t>(b) * a.R + jr) * a.Hq + h) * kD + 4 * ch;
                *reinterpret_cast<uint2*>(dst) =
                    make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
            } else {
                float* rec_g = a.ws_part + ((static_cast<size_t>(unit) * a.clusters + ci) * a.part_rows + lr) * kRec;
                if (ch == 0) {
                    rec_g[0] = L > 0.f ? M : -INFINITY;
                    rec_g[1] = L;
                }
                *reinterpret_cast<float4*>(rec_g + 4 + 4 * ch) = acc;
            }
        };
        for (int base = u0; base < u1; base += 2 * kNW) {   // CTA-uniform trip count
            float4 xa[kX], xc[kX];
            load_unit(base + warp, xa);
            load_unit(base + kNW + warp, xc);
            if (base == u0) {
                if (warp < ng) {
                    // weights of row 32 (g0 + warp) + lane: exp2(m_s - M) over
                    // the sources with a non-empty partial, and the merged sum
                    const int lr = (g0 + warp) * 32 + lane;
                    float2 ml[kX];
#pragma unroll
                    for (int sr = 0; sr < kX; ++sr)
                        ml[sr] = (lr < nrows && sr < C)
                                     ? __ldcg(reinterpret_cast<const float2*>(xb + sr * Ly::kXchFloats) + lr)
                                     : make_float2(-INFINITY, 0.f);
                    float M = -INFINITY;
#pragma unroll
                    for (int sr = 0; sr < kX; ++sr) M = fmaxf(M, ml[sr].x);
                    float L = 0.f;
                    float* wr = wsm + warp * (kX + 2) * 32 + lane;
#pragma unroll
                    for (int sr = 0; sr < kX; ++sr) {
                        // an empty partial (-inf, 0) and its zero O row weigh nothing
                        const float w = (ml[sr].y > 0.f && M != -INFINITY) ? exp2f(ml[sr].x - M) : 0.f;
                        L += w * ml[sr].y;
                        wr[sr * 32] = w;
                    }
                    wr[kX * 32] = M;
                    wr[(kX + 1) * 32] = L;
                }
                __syncthreads();
            }
            finish_unit(base + warp, xa);
            finish_unit(base + kNW + warp, xc);
        }
    }
    for (int li = warp; xch == nullptr && owns && k0 + n_owners * li < nrows; li += kThreads / 32) {
        const int lr = k0 + n_owners * li;
        const float* slots = recv + li * C * kRec;
        float ms = -INFINITY, ls = 0.f;
        if (lane < C) {
            const float2 ml = *reinterpret_cast<const float2*>(slots + lane * kRec);
            ms = ml.x;
            ls = ml.y;
        }
        float M = ms;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float wgt = (lane < C && ls > 0.f && M != -INFINITY) ? exp2f(ms - M) : 0.f;
        float L = wgt * ls;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        // O: branch-free, eight slots at a time (an empty partial has weight 0
        // and an all-zero record)
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < C; s0 += 8) {
            float4 x[8];
            float wv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int sr = s0 + u < C ? s0 + u : 0;
                wv[u] = __shfl_sync(0xffffffffu, wgt, sr);
                x[u] = *reinterpret_cast<const float4*>(slots + sr * kRec + 4 + 4 * lane);
                if (s0 + u >= C) wv[u] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                acc.x += wv[u] * x[u].x;
                acc.y += wv[u] * x[u].y;
                acc.z += wv[u] * x[u].z;
                acc.w += wv[u] * x[u].w;
            }
        }
        if (a.clusters == 1) {
            store_row(lr, acc, L);
        } else {
            float* rec_g = a.ws_part + ((static_cast<size_t>(unit) * a.clusters + ci) * a.part_rows + lr) * kRec;
            if (lane == 0) {
                rec_g[0] = L > 0.f ? M : -INFINITY;
                rec_g[1] = L;
            }
            *reinterpret_cast<float4*>(rec_g + 4 + 4 * lane) = acc;
        }
    }
    if (a.clusters > 1) {
        // ticket: the last cluster of (b, g, row tile) to finish merges all the
        // cluster partials (written above, made visible by the fence) and
        // resets the ticket for the next launch
        uint32_t* last_flag = reinterpret_cast<uint32_t*>(smem + Ly::kOffBar + 248);
        __threadfence();
        cluster.sync();
        if (rank == 0 && threadIdx.x == 0) {
            const unsigned int done = atomicAdd(a.ws_cnt + unit, 1u);
            const bool is_last = done == static_cast<unsigned int>(a.clusters - 1);
            if (is_last) a.ws_cnt[unit] = 0u;
            // the verdict goes to every CTA's own flag, so that no CTA reads
            // another's shared memory after the barrier below (and none waits
            // for the others before it exits)
            for (int r = 0; r < C; ++r) *cluster.map_shared_rank(last_flag, r) = is_last ? 1u : 0u;
        }
        cluster.sync();
        if (*last_flag != 0u) {
            __threadfence();
            const float* base = a.ws_part + static_cast<size_t>(unit) * a.clusters * a.part_rows * kRec;
            const int nc = a.clusters;
            const size_t pstride = static_cast<size_t>(a.part_rows) * kRec;
            if (nc <= kWsMergeBatch) {
                // one work item per (row, 4 output dims) over every thread of the
                // cluster; each item's partials are all loaded in one round
                const int nitems = nrows * 32;
                for (int it = rank * kThreads + threadIdx.x; it < nitems; it += C * kThreads) {
                    const int lr = it >> 5, l4 = it & 31;
                    float2 ml[kWsMergeBatch];
                    float4 ox[kWsMergeBatch];
#pragma unroll
                    for (int c = 0; c < kWsMergeBatch; ++c) {
                        if (c < nc) {
                            const float* rc = base + c * pstride + static_cast<size_t>(lr) * kRec;
                            ml[c] = __ldcg(reinterpret_cast<const float2*>(rc));
                            ox[c] = __ldcg(reinterpret_cast<const float4*>(rc + 4) + l4);
                        } else {
                            ml[c] = make_float2(-INFINITY, 0.f);
                            ox[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    float M = -INFINITY;
#pragma unroll
                    for (int c = 0; c < kWsMergeBatch; ++c)
                        if (ml[c].y > 0.f) M = fmaxf(M, ml[c].x);
                    float L = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (M != -INFINITY) {
#pragma unroll
                        for (int c = 0; c < kWsMergeBatch; ++c) {
                            const float w = ml[c].y > 0.f ? exp2f(ml[c].x - M) : 0.f;
                            L += w * ml[c].y;
                            acc.x += w * ox[c].x;
                            acc.y += w * ox[c].y;
                            acc.z += w * ox[c].z;
                            acc.w += w * ox[c].w;
                        }
                    }
                    const float inv = L > 0.f ? 1.0f / L : 0.f;
                    const int row = rt * kTileRows + lr;
                    const int jr = row / a.G, h = g * a.G + row % a.G;
                    uint16_t* dst = a.out + ((static_cast<size_t>(b) * a.R + jr) * a.Hq + h) * kD + 4 * l4;
                    *reinterpret_cast<uint2*>(dst) =
                        make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
                }
            } else
            for (int lr = rank + C * warp; lr < nrows; lr += C * (kThreads / 32)) {
                // lane c holds partial c's (max, sum) (nc <= 32), then the O
                // records are read eight at a time, branch-free
                float mc = -INFINITY, lc = 0.f;
                if (lane < nc) {
                    const float2 ml = __ldcg(reinterpret_cast<const float2*>(
                        base + (static_cast<size_t>(lane) * a.part_rows + lr) * kRec));
                    mc = ml.x;
                    lc = ml.y;
                }
                float M = lc > 0.f ? mc : -INFINITY;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                const float wc = (lc > 0.f && M != -INFINITY) ? exp2f(mc - M) : 0.f;
                float L = wc * lc;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c0 = 0; c0 < nc; c0 += 8) {
                    float4 x[8];
                    float wv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int c = c0 + u < nc ? c0 + u : 0;
                        wv[u] = __shfl_sync(0xffffffffu, wc, c);
                        x[u] = __ldcg(reinterpret_cast<const float4*>(
                                          base + (static_cast<size_t>(c) * a.part_rows + lr) * kRec + 4) +
                                      lane);
                        if (c0 + u >= nc) wv[u] = 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        acc.x += wv[u] * x[u].x;
                        acc.y += wv[u] * x[u].y;
                        acc.z += wv[u] * x[u].z;
                        acc.w += wv[u] * x[u].w;
                    }
                }
                store_row(lr, acc, L);
            }
        }
    }
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kHalf, bool kTree, int kHW, bool kSplit>
cudaError_t prepare_kernel() {
    static PerDeviceOnce attr_once;
    return attr_once.run([]() {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<kHalf, kTree, kHW, kSplit>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<kHalf>::kSmemBytes);
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(attn_tc_kernel<kHalf, kTree, kHW, kSplit>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                    1);
    });
}

// Clusters of C CTAs that can be resident at once (a cluster must fit in one
// GPC, so large clusters leave SMs idle); SMs / C when the query fails.
template <bool kHalf>
int active_clusters(int C) {
    static std::mutex mu;
    static int cache[64][17] = {};
    int dev = 0;
    const int fallback = device_sm_count() / C > 0 ? device_sm_count() / C : 1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return fallback;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev][C]) return cache[dev][C];
    int n = 0;
    if (prepare_kernel<kHalf, false, 2, !kHalf>() == cudaSuccess) {   // every variant uses the same resources
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C, 1, 1);
        cfg.blockDim = dim3(Roles<kHalf, 2>::kThreads, 1, 1);
        cfg.dynamicSmemBytes = Lay<kHalf>::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<kHalf, false, 2, !kHalf>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    if (n <= 0) n = fallback;
    cache[dev][C] = n;
    return n;
}

template <bool kHalf, bool kTree, int kHW, bool kSplit>
cudaError_t launch_mode(const AttnPlan& p, const sv_attn_shape& s, const uint8_t* tK, const uint8_t* tV,
                        const uint8_t* tKb, const uint8_t* tVb, const AttnArgs& a, cudaStream_t st) {
    constexpr int kThreads = Roles<kHalf, kHW>::kThreads;
    cudaError_t e = prepare_kernel<kHalf, kTree, kHW, kSplit>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.splits * p.clusters, s.B * s.Hkv * p.row_tiles, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Lay<kHalf>::kSmemBytes;
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
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<kHalf, kTree, kHW, kSplit>, *reinterpret_cast<const CUtensorMap*>(tK),
                              *reinterpret_cast<const CUtensorMap*>(tV), *reinterpret_cast<const CUtensorMap*>(tKb),
                              *reinterpret_cast<const CUtensorMap*>(tVb), a);
}

}  // namespace

// Split-KV plan.  Every (sequence, KV head, row tile) -- a unit -- gets
// `clusters` clusters of `splits` CTAs; its key tiles are divided evenly over
// those CTAs.  For each row-tile mode (half tiles; full tiles when a (b, g)
// group has more than 64 rows) and each cluster size C = 16 .. 1, one cluster
// per unit or as many as fit in one wave of resident clusters (at most 32, at
// least one key tile per CTA) are costed: the key tiles of the busiest CTA
// plus a fixed start-up of three tiles per wave, and a merge through the
// workspace as seven tiles (its partials cross the L2 in a few dependent round
// trips: at 7B batch 1 two clusters per KV head measured 17.4 -> 22.9 us, and
// on the draft tree's shape 4 x 2 CTAs took 27.6 us against 25.6-26.1 us for
// one cluster of 6) plus the partial bytes each merging SM reads (one SM
// pulls about 40 KB per tile time).  A full-tile step takes
// 9/8 of a half-tile step (measured on the draft tree's shape: ~2650 against
// ~2360 cycles per two-tile step).  Resident clusters come from the occupancy
// query, so sizes that leave a unit for a second wave (7, 8 and 9 CTAs fit 15
// times on the GB300) are costed as such.  Ties keep the larger cluster.
AttnPlan attn_plan(const sv_attn_shape& s) {
    AttnPlan p;
    p.G = s.Hq / s.Hkv;
    p.rows = s.R * p.G;
    const int64_t tiles = (s.T_cap + kNk - 1) / kNk + (s.R + kNk - 1) / kNk;
    int64_t best = -1;
    p.half = true;
    p.row_tiles = (p.rows + Lay<true>::kM - 1) / Lay<true>::kM;
    p.splits = 1;
    p.clusters = 1;
    for (int mode = 0; mode < 2; ++mode) {
        const bool half = mode == 0;
        if (!half && p.rows <= kHalfMaxRows) continue;
        const int tile_rows = half ? Lay<true>::kM : Lay<false>::kM;
        const int step_cost = half ? 8 : 9;   // eighths of a half-tile step per tile
        const int row_tiles = (p.rows + tile_rows - 1) / tile_rows;
        const int64_t units = static_cast<int64_t>(s.B) * s.Hkv * row_tiles;
        for (int C = kMaxCluster; C >= 1; --C) {
            if (C > tiles && C > 1) continue;
            const int64_t cap = half ? active_clusters<true>(C) : active_clusters<false>(C);
            int64_t nc_max = cap / units;
            if (nc_max > 32) nc_max = 32;
            if (nc_max > tiles / C) nc_max = tiles / C;
            if (nc_max < 1) nc_max = 1;
            for (int64_t nc = 1; nc <= nc_max; nc = nc < nc_max ? nc_max : nc_max + 1) {   // one cluster, or the most
                const int64_t waves = (units * nc + cap - 1) / cap;
                const int64_t per_cta = (tiles + C * nc - 1) / (C * nc);
                const int64_t part_rows = p.rows < tile_rows ? p.rows : tile_rows;
                const int64_t merge_bytes = nc * part_rows * kRec * 4 / C;   // per SM of the merging cluster
                const int64_t cost = waves * (3 * 8 + step_cost * per_cta) +
                                     (nc > 1 ? 8 * (kMergeCost + merge_bytes / (40 * 1024)) : 0);
                if (best < 0 || cost < best) {
                    best = cost;
                    p.half = half;
                    p.row_tiles = row_tiles;
                    p.splits = C;
                    p.clusters = static_cast<int>(nc);
                }
            }
        }
    }
    p.hw4 = p.half && (tiles + p.splits * p.clusters - 1) / (p.splits * p.clusters) >= kHw4MinTiles;
    // separate K and V barriers: always with full tiles (two ring stages), and
    // for chains in half tiles whose loops are longer than the ring over tiles
    // no other row tile of the unit shares
    p.split_kv = !p.half ||
                 (p.row_tiles == 1 &&
                  ((tiles + p.splits * p.clusters - 1) / (p.splits * p.clusters) + Lay<true>::kT - 1) / Lay<true>::kT >
                      Lay<true>::kStages);
    p.warps = !p.half ? Roles<false>::kThreads / 32 : p.hw4 ? Roles<true, 4>::kThreads / 32 : Roles<true, 2>::kThreads / 32;
    // Clusters of 128-row tiles meet through L2: each CTA stores its partial
    // rows in coalesced pieces and the owners load them after one cluster
    // barrier.  Pushed into the owners' shared memory instead, the records
    // (66 KB per CTA) cross the cluster at the ~20 GB/s per SM that distributed
    // shared memory gives an all-to-all, after a barrier for every ring to
    // drain: the draft tree's layer (6-CTA clusters) 23.4 -> 21.6 us.  Half
    // tiles keep the push: with 2-CTA clusters of 63 rows (7B batch 16) half
    // of a CTA's records stay in its own shared memory, and the exchange
    // measured 48.1 -> 50.3 us
    p.xch = !p.half && p.splits >= 2 && p.splits <= kXchMaxCluster;
    return p;
}

// Ticket words (one per unit, 256-byte aligned block) then the partial records.
static size_t attn_ticket_bytes(const AttnPlan& p, const sv_attn_shape& s) {
    const size_t units = static_cast<size_t>(s.B) * s.Hkv * p.row_tiles;
    return (units * 4 + 255) / 256 * 256;
}

// Bytes of the tickets and cluster partials (0 with one cluster per unit).
static size_t attn_part_bytes(const AttnPlan& p, const sv_attn_shape& s) {
    if (p.clusters <= 1) return 0;
    const size_t units = static_cast<size_t>(s.B) * s.Hkv * p.row_tiles;
    const int tile_rows = p.half ? Lay<true>::kM : Lay<false>::kM;
    const size_t part_rows = p.rows < tile_rows ? p.rows : tile_rows;
    return attn_ticket_bytes(p, s) + units * p.clusters * part_rows * kRec * sizeof(float);
}

// Offset and bytes of the L2 exchange area (one block per CTA of the grid).
static size_t attn_xch_offset(const AttnPlan& p, const sv_attn_shape& s) {
    return (attn_part_bytes(p, s) + 255) / 256 * 256;
}
static size_t attn_xch_bytes(const AttnPlan& p, const sv_attn_shape& s) {
    if (!p.xch) return 0;
    const size_t ctas = static_cast<size_t>(p.splits) * p.clusters * s.B * s.Hkv * p.row_tiles;
    return ctas * (p.half ? Lay<true>::kXchFloats : Lay<false>::kXchFloats) * sizeof(float);
}

size_t attn_workspace(const sv_attn_shape& s) {
    const AttnPlan p = attn_plan(s);
    return p.xch ? attn_xch_offset(p, s) + attn_xch_bytes(p, s) : attn_part_bytes(p, s);
}

cudaError_t launch_verify_attn(const sv_attn_shape& s, const uint16_t* q, const uint16_t* k_cache,
                               const uint16_t* v_cache, const int32_t* len, const uint16_t* k_blk,
                               const uint16_t* v_blk, const int32_t* parent, float scale, uint16_t* out,
                               void* ws, bool cache_ready, const int32_t* pages, int max_pages, int num_pages,
                               cudaStream_t st) {
    const AttnPlan p = attn_plan(s);
    if ((p.clusters > 1 || p.xch) && ws == nullptr) return cudaErrorInvalidValue;
    alignas(64) uint8_t tK[128], tV[128], tKb[128], tVb[128];
    // rows of the context tensor maps: the caches, or the page pool
    const uint64_t ctx_rows = pages ? static_cast<uint64_t>(num_pages) * s.Hkv * kNk
                                    : static_cast<uint64_t>(s.B) * s.Hkv * s.T_cap;
    const uint64_t blk_rows = static_cast<uint64_t>(s.B) * s.Hkv * s.R;
    if (!encode_tmap_2d_bf16(tK, k_cache, kD, ctx_rows, kD * 2, 64, kNk) ||
        !encode_tmap_2d_bf16(tV, v_cache, kD, ctx_rows, kD * 2, 64, kNk) ||
        !encode_tmap_2d_bf16(tKb, k_blk, kD, blk_rows, kD * 2, 64, kNk) ||
        !encode_tmap_2d_bf16(tVb, v_blk, kD, blk_rows, kD * 2, 64, kNk))
        return cudaErrorInvalidValue;
    AttnArgs a;
    a.q = q;
    a.k_blk = k_blk;
    a.v_blk = v_blk;
    a.len = len;
    a.parent = parent;
    a.out = out;
    a.err = device_error_word();
    a.ws_cnt = p.clusters > 1 ? static_cast<unsigned int*>(ws) : nullptr;
    a.ws_part = p.clusters > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + attn_ticket_bytes(p, s))
                               : nullptr;
    a.xch = p.xch ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + attn_xch_offset(p, s)) : nullptr;
    a.B = s.B;
    a.R = s.R;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.G = p.G;
    a.T_cap = s.T_cap;
    a.rows = p.rows;
    a.row_tiles = p.row_tiles;
    a.clusters = p.clusters;
    const int tile_rows = p.half ? Lay<true>::kM : Lay<false>::kM;
    a.part_rows = p.rows < tile_rows ? p.rows : tile_rows;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.cache_ready = cache_ready ? 1 : 0;
    a.pages = pages;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    if (parent != nullptr)
        return !p.half ? launch_mode<false, true, 2, true>(p, s, tK, tV, tKb, tVb, a, st)
               : p.hw4 ? launch_mode<true, true, 4, false>(p, s, tK, tV, tKb, tVb, a, st)
                       : launch_mode<true, true, 2, false>(p, s, tK, tV, tKb, tVb, a, st);
    if (!p.half) return launch_mode<false, false, 2, true>(p, s, tK, tV, tKb, tVb, a, st);   // always split
    if (p.split_kv)
        return p.hw4 ? launch_mode<true, false, 4, true>(p, s, tK, tV, tKb, tVb, a, st)
                     : launch_mode<true, false, 2, true>(p, s, tK, tV, tKb, tVb, a, st);
    return p.hw4 ? launch_mode<true, false, 4, false>(p, s, tK, tV, tKb, tVb, a, st)
                 : launch_mode<true, false, 2, false>(p, s, tK, tV, tKb, tVb, a, st);
}

}  // namespace sv
