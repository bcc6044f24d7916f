/*
 * sv.h -- C ABI of the GB300 (sm_103a) speculative-decoding block-verification
 * library (libsv.so).
 *
 * One verify round of speculative decoding, as the pages on the subject
 * define it, in five calls:
 *   sv_verify_attn    k+1-row causal (or tree-masked) GQA attention over the
 *                     committed KV cache plus the block's own K/V;
 *   sv_lm_head        projection of the verified rows to vocab logits;
 *   sv_accept_greedy  longest-prefix acceptance against the target argmax;
 *   sv_accept_sample  modified rejection sampling with residual resample and
 *                     bonus token;
 *   sv_kv_commit      copy of the committed rows into the cache and the length
 *                     update (cache length == committed-token count).
 *
 * Sources, cited by page title and section:
 *   [SCS]  "SpecDec-Context-Scaling project guide", sec. 3, 3.1, 3.2, 7.1
 *   [TUT]  wmrh.cn speculative-decoding tutorial, sec. 2.2, 3.2, 3.3
 *   [MINI] "mini-infer Phase 11: Speculative Decoding", sections "Modified
 *          Rejection Sampling", cross-device tensor alignment, hidden KV
 *          position bug, "v2"
 *   [SUB]  "SubSpec (NeurIPS'25)" summary, sec. 4.1 (shared KV cache), 4.2
 *          (draft token trees)
 *
 * The verify block.  A round verifies R = k+1 tokens per sequence: block row 0
 * is the pending token c (committed last round, KV not yet in the cache, see
 * [MINI] hidden KV position bug), rows 1..k are the drafts d_1..d_k (chain) or
 * the draft-tree nodes in topological order (tree, parent[j] < j).  The cache
 * holds t = len[b] committed positions.  Query row j attends to the cache and
 * to block rows i <= j (chain) or to j's ancestors and j itself (tree).  Row
 * j's logits are the target's next-token prediction after row j, so row 0 is
 * [SCS] sec. 3.1's saved_next and verifies d_1, row j verifies the children of
 * node j, and row k (chain) supplies only the bonus token.
 *
 * Conventions for every call.
 *   - All array pointers are DEVICE pointers to caller-owned memory, 16-byte
 *     aligned; bf16 tensors are passed as raw 16-bit patterns (uint16_t).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work: no call allocates, frees or synchronises, except
 *     sv_get_device_error (which synchronises the stream).
 *   - Workspace: calls that need scratch take (ws, ws_bytes), caller-owned
 *     device memory of at least the size the matching *_workspace query
 *     returns.  Contents need not be initialised and are not preserved.
 *   - Host-detectable problems (NULL pointer, bad shape, unsupported size,
 *     short workspace) return an error code before anything is enqueued.
 *     Problems only the device can see (non-finite logits, token id out of
 *     range, negative q, length over capacity, malformed tree) set a bit in
 *     the library's device error word and produce defined outputs (the
 *     offending sequence is left unchanged or given clamped values); nothing
 *     traps.  Read and clear the word with sv_get_device_error.
 *   - Calls on different streams may run concurrently if their buffers do
 *     not overlap; the only shared state is the error word.
 */
#ifndef SV_H
#define SV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SV_API __attribute__((visibility("default")))
#else
#define SV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sv_status {
    SV_OK = 0,
    SV_ERR_ARG = 1,          /* NULL pointer, misaligned pointer, bad scalar */
    SV_ERR_SHAPE = 2,        /* inconsistent or out-of-range sizes */
    SV_ERR_UNSUPPORTED = 3,  /* valid but not implemented (e.g. head dim != 128) */
    SV_ERR_WORKSPACE = 4,    /* ws_bytes below the *_workspace query */
    SV_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch, query) */
    SV_ERR_DEVICE = 6        /* sv_get_device_error found a device-side error bit */
} sv_status;

/* Device error word bits (sv_get_device_error). */
#define SV_DEVERR_NONFINITE   0x01u  /* NaN/Inf logit or temperature-scaled logit */
#define SV_DEVERR_TOKEN       0x02u  /* draft token id outside [0, V) */
#define SV_DEVERR_LENGTH      0x04u  /* len[b] < 0, or len[b] + (committed rows) > T_cap */
#define SV_DEVERR_QPROB       0x08u  /* negative or NaN draft probability */
#define SV_DEVERR_TREE        0x10u  /* parent[b][0] != -1 or parent[b][j] not in [0, j) */
#define SV_DEVERR_PATH        0x20u  /* commit: n_acc outside [0, R) or path entry outside [0, R) */
#define SV_DEVERR_TIMEOUT     0x40u  /* an internal bounded wait gave up (should never happen) */
#define SV_DEVERR_PAGE        0x80u  /* paged KV: a page-table entry outside [0, num_pages) */
/* (A library built with -DSV_DEBUG also reports failed internal self-checks,
 * as bit 31 plus a check code in bits 8..23.) */

/* Library version, e.g. 100 for 0.1.0. */
SV_API int sv_version(void);

/* Human-readable name of a status code (static string). */
SV_API const char* sv_status_string(sv_status s);

/* Reads and clears the device error word of the current device.  Synchronises
 * `stream` first.  Returns SV_OK if the word was zero, SV_ERR_DEVICE if any bit
 * was set (the bits are stored in *word in both cases; word may be NULL). */
SV_API sv_status sv_get_device_error(uint32_t* word, void* stream);

/* ------------------------------------------------------------------------ */
/* Verify attention ([SCS] sec. 3; [TUT] sec. 3.2; [SUB] sec. 4.2).          */
/* ------------------------------------------------------------------------ */

typedef struct sv_attn_shape {
    int32_t B;      /* sequences */
    int32_t R;      /* block rows = k+1 (chain) or tree nodes incl. root; 1..128 */
    int32_t Hq;     /* query heads */
    int32_t Hkv;    /* KV heads; Hq % Hkv == 0, Hq/Hkv <= 16 */
    int32_t D;      /* head dim; must be 128 */
    int32_t T_cap;  /* cache capacity per (sequence, KV head) */
} sv_attn_shape;

/* Workspace bytes sv_verify_attn needs for this shape (device-dependent: the
 * split-KV plan follows the SM count and how many thread-block clusters fit at
 * once).  0 when every (sequence, KV head) is handled by one cluster whose
 * split partials merge on chip; ws may then be NULL.  Otherwise it holds, in
 * this order and as the plan needs them:
 *   - when several clusters share a (sequence, KV head): one ticket word per
 *     (sequence, KV head, row tile of 64 or 128 rows, as the plan picks), then
 *     the clusters' fp32 partials;
 *   - when the plan takes 128-row tiles (more than 64 query rows per
 *     (sequence, KV head), e.g. a draft tree) in clusters of 2 to 6 CTAs: an
 *     exchange area, one fp32 block of partial rows per CTA, through which
 *     the cluster's CTAs merge (any contents before a call).
 * The ticket words must be zero before the first call on a workspace (e.g.
 * cudaMemset to 0 once); every call that completes leaves them zero again, so
 * one workspace serves any number of calls in stream order.  Calls running
 * concurrently need separate workspaces. */
SV_API size_t sv_verify_attn_workspace(const sv_attn_shape* shape);

/* For sequence b, query head h (KV head g = h / (Hq/Hkv), heads grouped
 * contiguously) and block row j:
 *     out[b][j][h] = sum_i softmax_i(scale * q[b][j][h] . k_i) v_i
 * over the visible keys i: cache positions 0..len[b]-1 of KV head g, and the
 * block rows visible to j (chain: 0..j; tree: j and its ancestors).
 *   q       [B][R][Hq][D]       bf16, already projected and rotated
 *   k_cache [B][Hkv][T_cap][D]  bf16, this layer's cache (positions >= len ignored)
 *   v_cache [B][Hkv][T_cap][D]  bf16
 *   len     [B]                 int32, 0 <= len[b] <= T_cap (else SV_DEVERR_LENGTH
 *                               and the length is clamped into [0, T_cap])
 *   k_blk   [B][Hkv][R][D]      bf16, K of the block rows
 *   v_blk   [B][Hkv][R][D]      bf16
 *   parent  NULL (chain) or [B][R] int32 tree (parent[b][0] = -1, parent[b][j] in [0, j))
 *   scale   softmax scale, > 0 (typically 1/sqrt(D))
 *   out     [B][R][Hq][D]       bf16 (fp32 accumulation, rounded to nearest even)
 * Numerics: bf16 inputs, fp32 products and softmax, P rounded to bf16 for the
 * P.V product; max|err| <= 1e-2 max|exact|. */
SV_API sv_status sv_verify_attn(const sv_attn_shape* shape, const uint16_t* q, const uint16_t* k_cache,
                         const uint16_t* v_cache, const int32_t* len, const uint16_t* k_blk,
                         const uint16_t* v_blk, const int32_t* parent, float scale, uint16_t* out,
                         void* ws, size_t ws_bytes, void* stream);

/* sv_verify_attn with launch flags (sv_verify_attn is flags = 0).
 *   SV_ATTN_CACHE_READY  the caller promises that the kernel enqueued on
 *       `stream` just before this call writes neither len nor k_cache /
 *       v_cache (e.g. the previous layer's attention within one verify round;
 *       NOT the first layer after sv_kv_commit).  The kernel then reads len
 *       and starts loading the committed cache rows while that kernel is
 *       still finishing (programmatic dependent launch); q, the block K/V,
 *       parent and every output are still touched only after it completes.
 * Unknown flag bits return SV_ERR_ARG. */
#define SV_ATTN_CACHE_READY 1u
SV_API sv_status sv_verify_attn_ex(const sv_attn_shape* shape, const uint16_t* q, const uint16_t* k_cache,
                                   const uint16_t* v_cache, const int32_t* len, const uint16_t* k_blk,
                                   const uint16_t* v_blk, const int32_t* parent, float scale, uint16_t* out,
                                   void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* Paged KV cache ([MINI] implementation architecture: the committed KV lives
 * in a block tensor addressed through each request's block table, and only
 * accepted tokens are written into it).  The cache of one layer is a pool of
 * pages of SV_KV_PAGE (64) positions,
 *     k_pool, v_pool  [num_pages][Hkv][64][D] bf16,
 * and position p of sequence b lives in page page_table[b][p / 64], row
 * p % 64.  page_table [B][max_pages] int32, caller-owned; the pool's pages
 * are the caller's to allocate (several sequences may not share a page they
 * both commit into).  shape->T_cap must equal max_pages * 64.
 * Otherwise as sv_verify_attn_ex (same flags, workspace, numerics); with
 * SV_ATTN_CACHE_READY the promise covers page_table too (it is read, like
 * len, before the preceding kernel has finished).  A page entry the
 * attention reaches that lies outside [0, num_pages) sets SV_DEVERR_PAGE and
 * reads as zeros. */
#define SV_KV_PAGE 64
SV_API sv_status sv_verify_attn_paged(const sv_attn_shape* shape, const uint16_t* q, const uint16_t* k_pool,
                                      const uint16_t* v_pool, int32_t num_pages, const int32_t* page_table,
                                      int32_t max_pages, const int32_t* len, const uint16_t* k_blk,
                                      const uint16_t* v_blk, const int32_t* parent, float scale, uint16_t* out,
                                      void* ws, size_t ws_bytes, uint32_t flags, void* stream);

/* ------------------------------------------------------------------------ */
/* LM head ([SCS] sec. 3: the target's block forward yields one logits row   */
/* per block row; [TUT] sec. 1.1: the weights are read once per forward).    */
/* ------------------------------------------------------------------------ */

/* logits[n][v] = sum_h hid[n][h] * W[h][v], fp32 accumulation.
 *   hid    [N][H] bf16 (N = B*R verified rows), 1 <= N <= 4096
 *   W      [H][V] bf16 row-major; H % 8 == 0, V % 8 == 0
 *   logits [N][V] fp32
 * No workspace. */
SV_API sv_status sv_lm_head(const uint16_t* hid, const uint16_t* W, float* logits, int32_t N, int32_t H,
                     int32_t V, void* stream);

/* sv_lm_head with launch flags (sv_lm_head is flags = 0).
 *   SV_LM_WEIGHTS_READY  the caller promises that the kernel enqueued on
 *       `stream` just before this call does not write W (model weights: true
 *       unless, e.g., a dequantisation kernel produces W right before).  The
 *       kernel then starts loading W while that kernel is still finishing
 *       (programmatic dependent launch); hid and logits are touched only after
 *       it completes.
 * Unknown flag bits return SV_ERR_ARG. */
#define SV_LM_WEIGHTS_READY 1u
SV_API sv_status sv_lm_head_ex(const uint16_t* hid, const uint16_t* W, float* logits, int32_t N, int32_t H,
                               int32_t V, uint32_t flags, void* stream);

/* The LM head with the greedy argmax folded into its epilogue ([SCS] sec. 3:
 * greedy verification needs only each row's top-1 token; [SCS] sec. 7.1:
 * the round's control plane -- syncs, token movement, launches after the
 * target forward -- is worth trimming).  As sv_lm_head_ex, and in addition,
 * for every row n and 128-column slab s (S = ceil(V / 128) slabs):
 *     argmax[n][s] = the largest key(logits[n][v]) over v in slab s,
 *     key(x, v) = (okey(x) << 32) | (~v & 0xffffffff)  (uint64),
 * where okey(NaN) = 0 and, for every other x, okey(x) is x's bit pattern
 * (with -0 taken as +0) mapped to an unsigned word in the order of the floats
 * (sign bit set: all bits flipped; else the sign bit set).  The row's greedy
 * token -- largest logit, NaN skipped, lowest column on ties, as
 * sv_accept_greedy takes it -- is the complement of the low word of the
 * row's largest key (column 0 when that key's high word is 0: only NaN).
 *   logits  [N][V] fp32, or NULL: the logits are then not written (a greedy
 *           round that needs only the tokens)
 *   argmax  [N][S] uint64, caller-owned, at least sv_lm_head_argmax_bytes
 *           (N, V) bytes (else SV_ERR_WORKSPACE)
 * NaN logits set SV_DEVERR_NONFINITE.  Other arguments, flags and errors as
 * for sv_lm_head_ex. */
#define SV_ARGMAX_SLAB 128
SV_API size_t sv_lm_head_argmax_bytes(int32_t N, int32_t V);
SV_API sv_status sv_lm_head_argmax(const uint16_t* hid, const uint16_t* W, float* logits, int32_t N, int32_t H,
                                   int32_t V, uint64_t* argmax, size_t argmax_bytes, uint32_t flags, void* stream);

/* ------------------------------------------------------------------------ */
/* Greedy acceptance ([SCS] sec. 3 and 3.1).                                 */
/* ------------------------------------------------------------------------ */

/* g_j = argmax_v logits[b][j][v] (ties: lowest id).  Chain: m is the largest
 * m <= R-1 with tok[b][i] == g_{i-1} for all 1 <= i <= m.  Tree: from the root,
 * repeatedly move to the first child (in index order) whose token equals the
 * current node's argmax.  Outputs: n_acc[b] = m, out_tok[b] = argmax of the
 * last accepted node's row (replacement if a draft failed, bonus if all
 * passed), path[b][0..m] = accepted node indices (path[b][0] = 0), -1 after.
 *   logits [B][R][V] fp32;  tok [B][R] int32 (tok[b][0] is the pending token,
 *   not tested);  parent NULL or [B][R] as for sv_verify_attn.
 * Token ids outside [0, V) set SV_DEVERR_TOKEN (the draft is rejected); NaN
 * logits set SV_DEVERR_NONFINITE and are skipped by the argmax. */
SV_API size_t sv_accept_greedy_workspace(int32_t B, int32_t R, int32_t V);
SV_API sv_status sv_accept_greedy(const float* logits, const int32_t* tok, const int32_t* parent, int32_t B,
                           int32_t R, int32_t V, int32_t* n_acc, int32_t* out_tok, int32_t* path,
                           void* ws, size_t ws_bytes, void* stream);

/* Greedy acceptance and the KV commit in one launch, from the argmax keys
 * of sv_lm_head_argmax ([SCS] sec. 3 and 3.1 for the acceptance; [SCS] sec.
 * 3.2, [TUT] sec. 3.2 and [SUB] sec. 4.2 for the commit; [SCS] sec. 7.1: one
 * launch instead of three after the target forward).  The result is that of
 * sv_accept_greedy on the same logits followed by sv_kv_commit:
 *   argmax [B*R][ceil(V/128)] uint64 keys (row b*R + j is sequence b's block
 *          row j), as written by sv_lm_head_argmax;
 *   tok, parent, n_acc, out_tok, path as for sv_accept_greedy;
 *   k_cache, v_cache, k_blk, v_blk, L, Hkv, D, T_cap, len as for
 *          sv_kv_commit (len updated in place).
 * k_cache == NULL (with v_cache, k_blk, v_blk NULL; L, Hkv, D, T_cap, len
 * ignored) gives greedy acceptance alone.  Errors: those of the two calls
 * (a sequence whose commit would pass T_cap still gets its acceptance
 * outputs, and its cache and length are left untouched, SV_DEVERR_LENGTH). */
SV_API sv_status sv_accept_greedy_commit(const uint64_t* argmax, const int32_t* tok, const int32_t* parent,
                                         int32_t B, int32_t R, int32_t V, int32_t* n_acc, int32_t* out_tok,
                                         int32_t* path, uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_blk,
                                         const uint16_t* v_blk, int32_t L, int32_t Hkv, int32_t D, int32_t T_cap,
                                         int32_t* len, void* stream);

/* sv_accept_greedy_commit into paged caches: the acceptance as above, the
 * commit as sv_kv_commit_paged (pools [L][num_pages][Hkv][64][D], page_table
 * [B][max_pages], capacity max_pages * 64).  A sequence whose new rows would
 * reach a page entry outside [0, num_pages) keeps its pages and length and
 * sets SV_DEVERR_PAGE; it still gets its acceptance outputs. */
SV_API sv_status sv_accept_greedy_commit_paged(const uint64_t* argmax, const int32_t* tok, const int32_t* parent,
                                               int32_t B, int32_t R, int32_t V, int32_t* n_acc, int32_t* out_tok,
                                               int32_t* path, uint16_t* k_pool, uint16_t* v_pool, int32_t num_pages,
                                               const int32_t* page_table, int32_t max_pages, const uint16_t* k_blk,
                                               const uint16_t* v_blk, int32_t L, int32_t Hkv, int32_t D, int32_t* len,
                                               void* stream);

/* ------------------------------------------------------------------------ */
/* Relaxed, lossy acceptance ([SCS] sec. 7.2: the Delta-logit relaxation).   */
/* ------------------------------------------------------------------------ */

/* As sv_accept_greedy, but a draft passes when the gap between its parent
 * row's top-1 logit and its own logit, one float32 subtraction
 * fsub_rn(top1, logits[b][u][d]), is <= delta.  The walk, out_tok (the top-1
 * of the row the walk stops at, lowest index on ties) and path are those of
 * sv_accept_greedy; delta = 0 with a unique row maximum is greedy acceptance.
 * LOSSY: the tokens no longer follow the target model exactly ([SCS] sec.
 * 7.2 measured higher acceptance rates at that cost).
 *   delta >= 0 (NaN or negative: SV_ERR_ARG); other arguments, the workspace
 *   (from sv_accept_greedy_relaxed_workspace, caller-owned, any contents) and
 *   the error flags as for sv_accept_greedy. */
SV_API size_t sv_accept_greedy_relaxed_workspace(int32_t B, int32_t R, int32_t V);
SV_API sv_status sv_accept_greedy_relaxed(const float* logits, const int32_t* tok, const int32_t* parent, int32_t B,
                                   int32_t R, int32_t V, float delta, int32_t* n_acc, int32_t* out_tok,
                                   int32_t* path, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Modified rejection sampling ([TUT] sec. 2.2; [MINI] "Modified Rejection   */
/* Sampling"; trees: [SUB] sec. 4.2).                                        */
/* ------------------------------------------------------------------------ */

/* p_j = softmax(logits[b][j] / T).  Chain: for j = 1..k, accept d_j = tok[b][j]
 * iff u_acc(j) < p_{j-1}(d_j) / q_{j-1}(d_j) (q == 0 accepts); at the first
 * rejection draw the replacement from max(0, p_{j-1} - q_{j-1}) (from p_{j-1}
 * if that is all zero) with u_res(j-1) and stop; if all k pass, draw the bonus
 * token from p_k with u_res(k).  Tree: at node u try its children in index
 * order against the working distribution w (initially p_u); a rejected child
 * turns w into norm(max(0, w - q_u)); after the last rejected child sample its
 * residual with u_res(u); at a leaf sample the bonus from p_u with u_res(u).
 *
 * Arithmetic (fixed so two implementations agree bit for bit): float32; the
 * softmax uses the max shift, a Cody-Waite/degree-7-Taylor exponential and a
 * canonical pairwise summation (balanced binary tree over the zero-padded
 * vocab, contiguous pairs); sampling descends that summation tree
 * (inverse CDF with target u_res * total).
 *
 * Uniforms: u_acc(u) and u_res(u) are words 0 and 1 of
 * Philox4x32-10(key = (seed lo, seed hi), counter = (b, u, step lo, step hi)),
 * each mapped to (w >> 8) * 2^-24; or, if `uniforms` is not NULL, read from
 * uniforms[b][u][0] and uniforms[b][u][1].
 *   logits   [B][R][V] fp32
 *   q        chain: [B][R-1][Vq] (row u = distribution of d_{u+1});
 *            tree:  [B][R][Vq]   (row u = distribution node u's children were
 *            drawn from).  Vq <= V; ids >= Vq have q = 0 ([MINI] cross-device
 *            alignment: the draft vocab is zero-padded to the target's).
 *   tok, parent as for sv_accept_greedy;  temperature > 0
 *   outputs as for sv_accept_greedy. */
/* Workspace: the (M, Z) statistics of every row (B*R float2, padded to 256
 * bytes), then for chain drafts one record per sequence and the summation-tree
 * sums of the one full-vocab pass it needs (B * 16 bytes padded to 256, then
 * B * 2 * (64*32 + 64) floats).  Chains then run three short launches (all
 * ratio tests at once, the residual or bonus pass spread over the GPU, one
 * warp per sequence for the draw); trees walk each sequence with one cluster.
 * Both give the same result bit for bit. */
SV_API size_t sv_accept_sample_workspace(int32_t B, int32_t R, int32_t V);
SV_API sv_status sv_accept_sample(const float* logits, const float* q, int32_t Vq, const int32_t* tok,
                           const int32_t* parent, int32_t B, int32_t R, int32_t V, float temperature,
                           uint64_t seed, uint64_t step, const float* uniforms, int32_t* n_acc,
                           int32_t* out_tok, int32_t* path, void* ws, size_t ws_bytes, void* stream);

/* sv_accept_sample without a workspace argument, for callers that cannot
 * allocate device memory (for example a plugin that is handed only its input
 * and output buffers by a host framework owning all device memory, or a loop
 * that must not call an allocating routine while it runs).  The pages have no
 * counterpart for this entry point; it exists for those callers only.
 * Behaviour and outputs are those of sv_accept_sample.  Its scratch is a
 * fixed 64 KiB device array (8192 rows of statistics) inside the library:
 *   - B*R above 8192 returns SV_ERR_SHAPE before anything is enqueued;
 *   - every GPU that loads the library holds the array until the process exits;
 *   - all calls share the array and it keeps the last call's contents (no
 *     entry needs to start at zero); calls that overlap on the GPU race on it,
 *     so order them on one stream or with events;
 *   - the first call on a device looks up the array's device address and
 *     caches it; make that first call before any stream capture.  A device
 *     reset (cudaDeviceReset) loads the library's device code anew, so the
 *     first call after it looks the address up again (make that call, too,
 *     outside any capture);
 *   - chains and trees alike are walked by one thread-block cluster per
 *     sequence (the path sv_accept_sample takes for trees), since the array
 *     holds only the row statistics; the results are those of
 *     sv_accept_sample bit for bit.
 * No cudaMalloc, cudaFree or other allocating call is made. */
SV_API sv_status sv_accept_sample_noalloc(const float* logits, const float* q, int32_t Vq, const int32_t* tok,
                                          const int32_t* parent, int32_t B, int32_t R, int32_t V,
                                          float temperature, uint64_t seed, uint64_t step, const float* uniforms,
                                          int32_t* n_acc, int32_t* out_tok, int32_t* path, void* stream);

/* ------------------------------------------------------------------------ */
/* KV commit ([SCS] sec. 3.2; [TUT] sec. 3.2; [MINI] hidden KV position bug, */
/* "v2"; [SUB] sec. 4.1).                                                    */
/* ------------------------------------------------------------------------ */

/* For every layer l, sequence b, KV head g and i = 0..n_acc[b]:
 *     cache[l][b][g][len[b] + i] = blk[l][b][g][path[b][i]]   (K and V)
 * then len[b] += n_acc[b] + 1.  Only the pending token and the accepted
 * drafts enter the cache; tree paths are compacted to consecutive slots.
 * Rows at or beyond the new length are not touched.
 *   k_cache, v_cache [L][B][Hkv][T_cap][D] bf16 (the per-layer caches of
 *                    sv_verify_attn, stacked)
 *   k_blk, v_blk     [L][B][Hkv][R][D] bf16
 *   path [B][R], n_acc [B] int32 (as produced by the accept calls)
 *   len  [B] int32, updated in place
 * A sequence with len + n_acc + 1 > T_cap or a bad path is left untouched and
 * sets SV_DEVERR_LENGTH / SV_DEVERR_PATH.  D % 8 == 0. */
SV_API sv_status sv_kv_commit(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk,
                       int32_t L, int32_t B, int32_t Hkv, int32_t D, int32_t T_cap, int32_t R,
                       const int32_t* path, const int32_t* n_acc, int32_t* len, void* stream);

/* sv_kv_commit into paged caches (see sv_verify_attn_paged): position
 * len[b] + i goes to page page_table[b][(len[b] + i) / 64], row
 * (len[b] + i) % 64, of every layer's pool.
 *   k_pool, v_pool [L][num_pages][Hkv][64][D] bf16 (the layers' pools, stacked)
 *   page_table [B][max_pages] int32 (shared by the layers); capacity max_pages * 64
 * A sequence whose new rows would reach a page entry outside [0, num_pages)
 * is left untouched and sets SV_DEVERR_PAGE; length and path errors as for
 * sv_kv_commit. */
SV_API sv_status sv_kv_commit_paged(uint16_t* k_pool, uint16_t* v_pool, int32_t num_pages, const int32_t* page_table,
                                    int32_t max_pages, const uint16_t* k_blk, const uint16_t* v_blk, int32_t L,
                                    int32_t B, int32_t Hkv, int32_t D, int32_t R, const int32_t* path,
                                    const int32_t* n_acc, int32_t* len, void* stream);

/* Moving a round's inputs in and its results out ([SCS] sec. 7.1: the control
 * plane of a round first -- fewer synchronisations and no host-to-device
 * copies between its kernels).  dst[0..bytes) = src[0..bytes), copied by a
 * kernel on `stream` (programmatic dependent launch, like every kernel here)
 * whose SMs load and store the bytes themselves: either side may be device
 * memory or page-locked host memory (cudaHostAlloc / cudaHostRegister;
 * reached through unified addressing -- on GB300 over the coherent
 * NVLink-C2C link), so a round's inputs and outputs cross the host link inside
 * the round's own kernel chain instead of as copy-engine operations.  The host
 * may read host-side dst once the copy has completed in stream order (an
 * event or a stream synchronisation).
 *   dst, src: non-NULL when bytes > 0, each device or page-locked host memory
 *             (checked with cudaPointerGetAttributes: anything else, e.g.
 *             pageable host memory, returns SV_ERR_ARG before any launch); both
 *             ranges [p, p + bytes) must lie inside their allocations and must
 *             not overlap.  Any alignment; 16-byte aligned pointers move 16
 *             bytes per access.
 *   bytes == 0: SV_OK, nothing launched.
 * Ownership: the caller's; the library keeps nothing. */
SV_API sv_status sv_copy(void* dst, const void* src, size_t bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics: the device building blocks of sv_accept_sample, exposed so    */
/* they can be compared element by element with an independent host         */
/* implementation.  Not part of the verify round.                            */
/* ------------------------------------------------------------------------ */

/* y[i] = the device exponential used by sv_accept_sample, for n inputs; where
 * one of the two faster forms of it used by the softmax passes -- the
 * branch-free one (defined for x <= 0) and the normal-range one (defined for
 * -86.5 < x <= 0) -- differs from it in any bit, y[i] = 12345 instead. */
SV_API sv_status sv_diag_exp(const float* x, float* y, int64_t n, void* stream);

/* q[i] = a[i] / b[i] as sv_accept_sample divides by a row's sum Z or a
 * sibling residual sum S: from the reciprocal 1/b rounded to nearest by one
 * Markstein correction step where a and b lie in [2^-60, 2^60], the
 * correctly rounded division elsewhere.  Either way the result must be the
 * IEEE quotient rounded to nearest even, bit for bit. */
SV_API sv_status sv_diag_div(const float* a, const float* b, float* q, int64_t n, void* stream);

/* out[i][0..3] = Philox4x32-10(counter = ctr[i][0..3], key = key[i][0..1]). */
SV_API sv_status sv_diag_philox(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int64_t n, void* stream);

/* sums[i] = canonical sum of x[i][0..n) (float32, pairwise tree), for m rows;
 * draws[i] = tree-descent sample of row i with uniform u[i]. */
SV_API sv_status sv_diag_canon(const float* x, int32_t n, int32_t m, const float* u, float* sums, int32_t* draws,
                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SV_H */
