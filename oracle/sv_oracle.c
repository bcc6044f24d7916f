/*
 * sv_oracle.c -- plain, slow, CPU reference for the speculative-decoding
 * block-verification step.  TEST INFRASTRUCTURE ONLY: nothing in the product
 * path may link, load or call this file.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg use it.
 *
 * It shares no source with the CUDA library: its own bf16 widening, its own
 * Philox4x32-10, its own exponential, its own canonical summation.
 *
 * Sources (web pages on the subject, cited by title and section):
 *   [SCS]  "SpecDec-Context-Scaling project guide" (richardf123.github.io):
 *          sec. 3 (block verification, longest accepted prefix, replacement and
 *          bonus token), sec. 3.1 (logits-row alignment), sec. 3.2 (cache length
 *          equals committed-token count), sec. 7.2 (the lossy Delta-logit
 *          relaxation of the acceptance test).
 *   [TUT]  wmrh.cn speculative-decoding tutorial: sec. 2.2 (accept with
 *          min(1, p/q), otherwise resample from norm(max(0, p - q))), sec. 3.2
 *          (one target forward over the gamma drafts, drop rejected KV),
 *          sec. 3.3 (accept/reject on the untruncated, temperature-scaled
 *          distribution), sec. 8 (draft and target temperatures match).
 *   [MINI] "mini-infer Phase 11: Speculative Decoding" (smarter.xin): section
 *          "Modified Rejection Sampling" (test, resample, stop, bonus from the
 *          last verify row), section on cross-device tensor alignment (draft
 *          probabilities zero-padded from 151936 to 152064), section on the
 *          hidden KV position bug (the pending token's KV must be committed),
 *          implementation architecture (the KV in a block tensor behind a
 *          block table: the paged cache, which the tests gather into the
 *          contiguous one this oracle takes).
 *   [SUB]  "SubSpec (NeurIPS'25)" summary: sec. 4.2 (draft token trees verified
 *          by the target in one pass).
 *
 * Readings adopted where the pages are silent:
 *   - the verify block has R = k+1 rows: row 0 is the pending committed token
 *     c, rows 1..k the drafts; row j is [SCS] sec. 3.1's rows[j-1] and row 0 is
 *     its saved_next;
 *   - argmax ties go to the lowest token id;
 *   - accept iff u < p(d)/q(d) (strict, as [MINI] writes it); q(d) == 0 accepts;
 *   - softmax arithmetic is fixed to single precision with a canonical
 *     summation order and a specified exponential so that a second
 *     implementation can reproduce every decision bit for bit;
 *   - residual sampling is inverse-CDF sampling by descent of the canonical
 *     summation tree; an all-zero residual falls back to the current
 *     distribution (the threshold fallback of [MINI], with the threshold at 0);
 *   - token trees: children are tried in index order; after a rejected child
 *     the working distribution becomes norm(max(0, w - q)) (recursive
 *     rejection sampling); after the last rejected child the residual is
 *     sampled directly, which makes a one-child-per-node tree identical to the
 *     chain.
 *
 * Floating point: built with -ffp-contract=off and no fast-math, so every
 * a*b+c below is two roundings unless written as fmaf().  Attention and the
 * LM head accumulate in double (more exact than the fp32 the kernels use);
 * the sampled acceptance runs in float because float decides its integers on
 * both sides.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR (-1)

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> float                                                           */
/* ------------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of a binary32; widening is exact. */
static float bf16_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As   */
/* Easy as 1, 2, 3", SC'11): a 10-round counter-based generator.  Each round */
/* multiplies words 0 and 2 by fixed odd constants, swaps and xors the high  */
/* halves with the other words and the key; the key is bumped by two Weyl    */
/* constants between rounds.                                                 */
/* ------------------------------------------------------------------------ */

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint32_t MUL_A = 0xD2511F53u, MUL_B = 0xCD9E8D57u;
    const uint32_t WEYL_A = 0x9E3779B9u, WEYL_B = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += WEYL_A;
            k1 += WEYL_B;
        }
        uint64_t prod_a = (uint64_t)MUL_A * (uint64_t)c0;
        uint64_t prod_b = (uint64_t)MUL_B * (uint64_t)c2;
        uint32_t hi_a = (uint32_t)(prod_a >> 32), lo_a = (uint32_t)prod_a;
        uint32_t hi_b = (uint32_t)(prod_b >> 32), lo_b = (uint32_t)prod_b;
        uint32_t n0 = hi_b ^ c1 ^ k0;
        uint32_t n1 = lo_b;
        uint32_t n2 = hi_a ^ c3 ^ k1;
        uint32_t n3 = lo_a;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* A 32-bit word becomes a uniform in [0, 1) on the 2^-24 grid: its top 24
 * bits times 2^-24 (exact in float). */
float orc_uniform24(uint32_t w) {
    return (float)(w >> 8) * (1.0f / 16777216.0f);
}

/* The two uniforms attached to tree node u of sequence b at round `step`:
 * key = seed, counter = (b, u, step_lo, step_hi); word 0 is the acceptance
 * uniform of node u's draft, word 1 the sampling uniform used when the round
 * stops at node u. */
static void node_uniforms(uint64_t seed, uint64_t step, int b, int u, float* u_acc, float* u_res) {
    uint32_t ctr[4] = {(uint32_t)b, (uint32_t)u, (uint32_t)(step & 0xffffffffu), (uint32_t)(step >> 32)};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    *u_acc = orc_uniform24(w[0]);
    *u_res = orc_uniform24(w[1]);
}

/* ------------------------------------------------------------------------ */
/* Exponential: Cody-Waite argument reduction (W. J. Cody and W. Waite,      */
/* "Software Manual for the Elementary Functions", 1980) followed by the     */
/* degree-7 Taylor polynomial of e^r, evaluated by Horner's rule with fused  */
/* multiply-adds, and an exact scaling by 2^n.                               */
/*   x = n ln2 + r,  n = rint(x / ln2),  |r| <= ln2/2 (about 0.347)          */
/*   ln2 is split into a head with 12 significant bits (so n*head is exact   */
/*   for |n| < 2^12) and a float tail.                                       */
/*   Taylor truncation: r^8/8! < 6e-9, below 0.07 ulp of e^r.                */
/* ------------------------------------------------------------------------ */

float orc_exp(float x) {
    if (x != x) return x;                      /* NaN */
    if (x < -104.0f) return 0.0f;              /* e^x < 2^-150: rounds to zero */
    if (x > 88.0f) return INFINITY;            /* domain limit; the method only evaluates x <= 0 */
    const float inv_ln2 = 1.44269504088896340736f;
    const float ln2_head = 0.693145751953125f;      /* 0x3F317000 */
    const float ln2_tail = 1.428606820309417232e-06f;
    float n = rintf(x * inv_ln2);
    float r = fmaf(-n, ln2_head, x);
    r = fmaf(-n, ln2_tail, r);
    float poly = 1.0f / 5040.0f;               /* 1/7! */
    poly = fmaf(poly, r, 1.0f / 720.0f);       /* 1/6! */
    poly = fmaf(poly, r, 1.0f / 120.0f);
    poly = fmaf(poly, r, 1.0f / 24.0f);
    poly = fmaf(poly, r, 1.0f / 6.0f);
    poly = fmaf(poly, r, 0.5f);
    poly = fmaf(poly, r, 1.0f);
    poly = fmaf(poly, r, 1.0f);
    int ni = (int)n;
    if (ni >= -126) {
        uint32_t bits = (uint32_t)(ni + 127) << 23;
        float scale;
        memcpy(&scale, &bits, 4);
        return poly * scale;                   /* exact, or one rounding into subnormals */
    }
    /* 2^n is subnormal: scale in two steps; the first is exact, the second
     * rounds once. */
    uint32_t bits_a = (uint32_t)(ni + 64 + 127) << 23;
    uint32_t bits_b = (uint32_t)(-64 + 127) << 23;
    float sa, sb;
    memcpy(&sa, &bits_a, 4);
    memcpy(&sb, &bits_b, 4);
    return (poly * sa) * sb;
}

/* orc_exp over an array (used by the oracle's own pins). */
void orc_exp_array(const float* x, float* y, long n) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) y[i] = orc_exp(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Canonical summation: the n values, zero-padded to the next power of two,  */
/* are the leaves of a balanced binary tree whose node covering             */
/* [lo, lo + size) is the float sum of its two halves.  Zero padding does    */
/* not change the result (x + 0 == x), so the same value comes out for any   */
/* padded length >= n.                                                       */
/* ------------------------------------------------------------------------ */

static int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

static float tree_node_sum(const float* x, int n, int lo, int size) {
    if (lo >= n) return 0.0f;
    if (size == 1) return x[lo];
    int half = size >> 1;
    float left = tree_node_sum(x, n, lo, half);
    float right = tree_node_sum(x, n, lo + half, half);
    return left + right;
}

float orc_canon_sum(const float* x, int n) {
    if (n <= 0) return 0.0f;
    return tree_node_sum(x, n, 0, next_pow2(n));
}

/* Inverse-CDF draw from the unnormalised weights x[0..n) with uniform u in
 * [0, 1): target tau = u * S with S the canonical sum; descend from the root,
 * going left while tau < acc + S(left) or the right half weighs nothing,
 * otherwise adding S(left) to acc and going right.  A zero-weight leaf is
 * never returned when S > 0. */
int orc_tree_sample(const float* x, int n, float u) {
    int size = next_pow2(n);
    float total = tree_node_sum(x, n, 0, size);
    float tau = u * total;
    float acc = 0.0f;
    int lo = 0;
    while (size > 1) {
        int half = size >> 1;
        float s_left = tree_node_sum(x, n, lo, half);
        float s_right = tree_node_sum(x, n, lo + half, half);
        if (tau < acc + s_left || s_right == 0.0f) {
            size = half;
        } else {
            acc = acc + s_left;
            lo = lo + half;
            size = half;
        }
    }
    return lo;
}

/* orc_tree_sample for many uniforms over the same weights (oracle pins). */
void orc_tree_sample_batch(const float* x, int n, const float* us, long m, int32_t* out) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < m; ++i) out[i] = orc_tree_sample(x, n, us[i]);
}

/* Target distribution of one verify row: p = softmax(l / T) in float with a
 * max shift, orc_exp and the canonical sum.  T > 0 ([TUT] sec. 3.3: the
 * accept/reject runs on the full temperature-scaled distribution). */
void orc_softmax(const float* l, int V, float T, float* p) {
    float m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        float z = l[v] / T;
        p[v] = z;
        if (z > m) m = z;
    }
    for (int v = 0; v < V; ++v) p[v] = orc_exp(p[v] - m);
    float Z = orc_canon_sum(p, V);
    for (int v = 0; v < V; ++v) p[v] = p[v] / Z;
}

/* ------------------------------------------------------------------------ */
/* Greedy acceptance ([SCS] sec. 3 and 3.1).                                */
/* ------------------------------------------------------------------------ */

static int argmax_lowest(const float* row, int V) {
    int best = 0;
    float bv = row[0];
    for (int v = 1; v < V; ++v) {
        if (row[v] > bv) { bv = row[v]; best = v; }
    }
    return best;
}

static int check_tree(const int32_t* parent, int R) {
    if (parent[0] != -1) return ORC_ERR;
    for (int j = 1; j < R; ++j)
        if (parent[j] < 0 || parent[j] >= j) return ORC_ERR;
    return ORC_OK;
}

/* logits [B, R, V] float; tok [B, R] (tok[b][0] is the pending token, tok[b][j]
 * the j-th draft or tree node); parent NULL for a chain, else [B, R].
 * Outputs: n_acc[b] accepted drafts, out_tok[b] the replacement (if a draft
 * was rejected) or bonus token (if all were accepted), path[b][0..n_acc] the
 * accepted node indices starting with 0, -1 after. */
int orc_accept_greedy(const float* logits, const int32_t* tok, const int32_t* parent,
                      int B, int R, int V, int32_t* n_acc, int32_t* out_tok, int32_t* path) {
    if (B < 0 || R < 1 || V < 1) return ORC_ERR;
    for (int b = 0; b < B; ++b) {
        const float* L = logits + (size_t)b * R * V;
        const int32_t* tk = tok + (size_t)b * R;
        int32_t* pth = path + (size_t)b * R;
        for (int j = 0; j < R; ++j) pth[j] = -1;
        for (int j = 1; j < R; ++j)
            if (tk[j] < 0 || tk[j] >= V) return ORC_ERR;
        if (parent == NULL) {
            /* Row j is the target's next-token prediction after the block's
             * first j+1 tokens, so row j-1 verifies draft j: row 0
             * (saved_next) verifies d_1, row k-1 verifies d_k, and row k is
             * only the bonus row. */
            int m = 0;
            while (m < R - 1 && tk[m + 1] == argmax_lowest(L + (size_t)m * V, V)) ++m;
            for (int i = 0; i <= m; ++i) pth[i] = i;
            n_acc[b] = m;
            out_tok[b] = argmax_lowest(L + (size_t)m * V, V);
        } else {
            const int32_t* par = parent + (size_t)b * R;
            if (check_tree(par, R) != ORC_OK) return ORC_ERR;
            int u = 0, depth = 0;
            pth[0] = 0;
            for (;;) {
                int g = argmax_lowest(L + (size_t)u * V, V);
                int next = -1;
                for (int c = u + 1; c < R; ++c)
                    if (par[c] == u && tk[c] == g) { next = c; break; }
                if (next < 0) break;
                u = next;
                pth[++depth] = u;
            }
            n_acc[b] = depth;
            out_tok[b] = argmax_lowest(L + (size_t)u * V, V);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Relaxed, lossy acceptance ([SCS] sec. 7.2, the Delta-logit relaxation): a */
/* draft passes when the target's top-1 logit exceeds the draft token's      */
/* logit by at most delta.  The walk, the output token (the top-1 of the     */
/* row the walk stops at) and the path are those of greedy acceptance; the   */
/* output no longer follows the target model exactly.  The gap is one        */
/* float32 subtraction.                                                      */
/* ------------------------------------------------------------------------ */

static int within_delta(const float* row, int top, int d, float delta) {
    float gap = row[top] - row[d];
    return gap <= delta;
}

int orc_accept_greedy_relaxed(const float* logits, const int32_t* tok, const int32_t* parent,
                              int B, int R, int V, float delta, int32_t* n_acc, int32_t* out_tok,
                              int32_t* path) {
    if (B < 0 || R < 1 || V < 1 || !(delta >= 0.0f)) return ORC_ERR;
    for (int b = 0; b < B; ++b) {
        const float* L = logits + (size_t)b * R * V;
        const int32_t* tk = tok + (size_t)b * R;
        int32_t* pth = path + (size_t)b * R;
        for (int j = 0; j < R; ++j) pth[j] = -1;
        for (int j = 1; j < R; ++j)
            if (tk[j] < 0 || tk[j] >= V) return ORC_ERR;
        if (parent != NULL && check_tree(parent + (size_t)b * R, R) != ORC_OK) return ORC_ERR;
        /* from the root (row 0), into the first child in index order that
         * passes the test against its parent's row */
        int u = 0, depth = 0;
        pth[0] = 0;
        for (;;) {
            const float* row = L + (size_t)u * V;
            int top = argmax_lowest(row, V);
            int next = -1;
            for (int c = u + 1; c < R; ++c) {
                int child = parent == NULL ? (c == u + 1) : (parent[(size_t)b * R + c] == u);
                if (child && within_delta(row, top, tk[c], delta)) { next = c; break; }
            }
            if (next < 0) break;
            u = next;
            pth[++depth] = u;
        }
        n_acc[b] = depth;
        out_tok[b] = argmax_lowest(L + (size_t)u * V, V);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Modified rejection sampling ([TUT] sec. 2.2; [MINI] "Modified Rejection   */
/* Sampling").                                                               */
/* ------------------------------------------------------------------------ */

/* Acceptance test of draft token d against target probabilities w and draft
 * probabilities qrow (qrow has Vq entries; ids >= Vq have q = 0, the zero
 * padding of [MINI]'s vocab alignment). */
static int ratio_accept(const float* w, const float* qrow, int Vq, int d, float u) {
    float qd = (d < Vq) ? qrow[d] : 0.0f;
    if (qd == 0.0f) return 1;
    float r = w[d] / qd;
    return u < r;
}

/* rho = max(0, w - q) over the target vocab (q zero-padded beyond Vq). */
static void residual(const float* w, const float* qrow, int Vq, int V, float* rho) {
    for (int v = 0; v < V; ++v) {
        float qv = (v < Vq) ? qrow[v] : 0.0f;
        float d = w[v] - qv;
        rho[v] = d > 0.0f ? d : 0.0f;
    }
}

static void get_uniforms(const float* uniforms, uint64_t seed, uint64_t step, int b, int R, int u,
                         float* u_acc, float* u_res) {
    if (uniforms) {
        *u_acc = uniforms[((size_t)b * R + u) * 2 + 0];
        *u_res = uniforms[((size_t)b * R + u) * 2 + 1];
    } else {
        node_uniforms(seed, step, b, u, u_acc, u_res);
    }
}

/* logits [B, R, V]; q [B, Rq, Vq] with Rq = R-1 (chain: row u is the draft
 * distribution d_{u+1} was drawn from) or Rq = R (tree: row u is the
 * distribution node u's children were drawn from); uniforms NULL (Philox)
 * or [B, R, 2]. */
int orc_accept_sample(const float* logits, const float* q, int Vq, const int32_t* tok,
                      const int32_t* parent, int B, int R, int V, float T, uint64_t seed,
                      uint64_t step, const float* uniforms, int32_t* n_acc, int32_t* out_tok,
                      int32_t* path) {
    if (B < 0 || R < 1 || V < 1 || Vq < 1 || Vq > V || !(T > 0.0f)) return ORC_ERR;
    int Rq = parent ? R : R - 1;
    int err = 0;
#pragma omp parallel reduction(| : err)
    {
    /* per-thread scratch rows */
    float* w = (float*)malloc(sizeof(float) * (size_t)V);
    float* rho = (float*)malloc(sizeof(float) * (size_t)V);
#pragma omp for schedule(dynamic, 64)
    for (int b = 0; b < B; ++b) {
        const float* L = logits + (size_t)b * R * V;
        const float* Q = q + (size_t)b * Rq * Vq;
        const int32_t* tk = tok + (size_t)b * R;
        int32_t* pth = path + (size_t)b * R;
        for (int j = 0; j < R; ++j) pth[j] = -1;
        pth[0] = 0;
        int bad = 0;
        for (int j = 1; j < R; ++j)
            if (tk[j] < 0 || tk[j] >= V) bad = 1;
        if (parent && check_tree(parent + (size_t)b * R, R) != ORC_OK) bad = 1;
        if (bad) { err |= 1; continue; }
        float u_acc, u_res;
        if (parent == NULL) {
            /* Chain: d_j is tested against row j-1; the first rejection
             * resamples from the residual of that row and ends the round; if
             * every draft passes, the bonus token is drawn from row k. */
            int m = 0;
            int done = 0;
            for (int j = 1; j < R && !done; ++j) {
                int u = j - 1;
                orc_softmax(L + (size_t)u * V, V, T, w);
                get_uniforms(uniforms, seed, step, b, R, j, &u_acc, &u_res);
                if (ratio_accept(w, Q + (size_t)u * Vq, Vq, tk[j], u_acc)) {
                    m = j;
                    pth[j] = j;
                    continue;
                }
                residual(w, Q + (size_t)u * Vq, Vq, V, rho);
                float S = orc_canon_sum(rho, V);
                get_uniforms(uniforms, seed, step, b, R, u, &u_acc, &u_res);
                out_tok[b] = (S > 0.0f) ? orc_tree_sample(rho, V, u_res) : orc_tree_sample(w, V, u_res);
                done = 1;
            }
            if (!done) {
                orc_softmax(L + (size_t)(R - 1) * V, V, T, w);
                get_uniforms(uniforms, seed, step, b, R, R - 1, &u_acc, &u_res);
                out_tok[b] = orc_tree_sample(w, V, u_res);
            }
            n_acc[b] = m;
        } else {
            /* Tree: at node u try its children in index order; a rejected
             * child turns the working distribution into norm(max(0, w - q_u));
             * when every child is rejected, sample the last residual (or w
             * if it is all zero); at a leaf, sample the bonus from p_u. */
            const int32_t* par = parent + (size_t)b * R;
            int u = 0, depth = 0;
            for (;;) {
                orc_softmax(L + (size_t)u * V, V, T, w);
                const float* qrow = Q + (size_t)u * Vq;
                int n_child = 0, last_child = -1;
                for (int c = u + 1; c < R; ++c)
                    if (par[c] == u) { ++n_child; last_child = c; }
                if (n_child == 0) {
                    get_uniforms(uniforms, seed, step, b, R, u, &u_acc, &u_res);
                    out_tok[b] = orc_tree_sample(w, V, u_res);
                    break;
                }
                int next = -1, finished = 0;
                for (int c = u + 1; c < R && next < 0 && !finished; ++c) {
                    if (par[c] != u) continue;
                    get_uniforms(uniforms, seed, step, b, R, c, &u_acc, &u_res);
                    if (ratio_accept(w, qrow, Vq, tk[c], u_acc)) { next = c; break; }
                    residual(w, qrow, Vq, V, rho);
                    float S = orc_canon_sum(rho, V);
                    if (c == last_child) {
                        get_uniforms(uniforms, seed, step, b, R, u, &u_acc, &u_res);
                        out_tok[b] = (S > 0.0f) ? orc_tree_sample(rho, V, u_res) : orc_tree_sample(w, V, u_res);
                        finished = 1;
                    } else if (S > 0.0f) {
                        for (int v = 0; v < V; ++v) w[v] = rho[v] / S;
                    }
                }
                if (finished) break;
                u = next;
                pth[++depth] = u;
            }
            n_acc[b] = depth;
        }
    }
    free(w);
    free(rho);
    }
    return err ? ORC_ERR : ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* KV commit ([SCS] sec. 3.2; [TUT] sec. 3.2; [MINI] hidden KV position bug): */
/* the pending token and the accepted drafts enter the cache at positions    */
/* t..t+m, no rejected row does, and the length becomes t+m+1.               */
/* cache [L, B, Hkv, T_cap, D] bf16; block [L, B, Hkv, R, D] bf16.           */
/* ------------------------------------------------------------------------ */

int orc_kv_commit(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk,
                  int L, int B, int Hkv, int D, int T_cap, int R, const int32_t* path,
                  const int32_t* n_acc, int32_t* len) {
    int err = 0;
    for (int b = 0; b < B; ++b) {
        int t = len[b], m = n_acc[b];
        if (t < 0 || m < 0 || m >= R || t + m + 1 > T_cap) { err = 1; continue; }
        int bad = 0;
        for (int i = 0; i <= m; ++i)
            if (path[(size_t)b * R + i] < 0 || path[(size_t)b * R + i] >= R) bad = 1;
        if (bad) { err = 1; continue; }
        for (int l = 0; l < L; ++l)
            for (int g = 0; g < Hkv; ++g)
                for (int i = 0; i <= m; ++i) {
                    int src = path[(size_t)b * R + i];
                    size_t dst_off = ((((size_t)l * B + b) * Hkv + g) * T_cap + (size_t)(t + i)) * D;
                    size_t src_off = ((((size_t)l * B + b) * Hkv + g) * R + (size_t)src) * D;
                    memcpy(k_cache + dst_off, k_blk + src_off, sizeof(uint16_t) * (size_t)D);
                    memcpy(v_cache + dst_off, v_blk + src_off, sizeof(uint16_t) * (size_t)D);
                }
        len[b] = t + m + 1;
    }
    return err ? ORC_ERR : ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Verify attention ([SCS] sec. 3, [TUT] sec. 3.2, [SUB] sec. 4.2): for      */
/* query row j of sequence b and Q head h (KV head g = h / (Hq/Hkv)), the    */
/* visible keys are the t = len[b] cached positions plus the block rows i    */
/* with i <= j (chain) or i an ancestor of j or j itself (tree);             */
/* o = sum_i softmax_i(scale * q.k_i) v_i, all in double.                    */
/* q, out [B, R, Hq, D]; cache [B, Hkv, T_cap, D]; block [B, Hkv, R, D].      */
/* ------------------------------------------------------------------------ */

int orc_verify_attn(int B, int R, int Hq, int Hkv, int D, int T_cap, const uint16_t* q,
                    const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* len,
                    const uint16_t* k_blk, const uint16_t* v_blk, const int32_t* parent,
                    double scale, double* out) {
    if (B < 0 || R < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1) return ORC_ERR;
    for (int b = 0; b < B; ++b) {
        if (len[b] < 0 || len[b] > T_cap) return ORC_ERR;
        if (parent && check_tree(parent + (size_t)b * R, R) != ORC_OK) return ORC_ERR;
    }
    int G = Hq / Hkv;
    long total = (long)B * R * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (long idx = 0; idx < total; ++idx) {
        int h = (int)(idx % Hq);
        int j = (int)((idx / Hq) % R);
        int b = (int)(idx / ((long)Hq * R));
        int g = h / G;
        int t = len[b];
        const uint16_t* qv = q + (((size_t)b * R + j) * Hq + h) * D;
        /* visible block rows */
        char* vis = (char*)calloc((size_t)R, 1);
        if (parent == NULL) {
            for (int i = 0; i <= j; ++i) vis[i] = 1;
        } else {
            const int32_t* par = parent + (size_t)b * R;
            for (int i = j; i >= 0; i = par[i]) vis[i] = 1;
        }
        int nkeys = t + R;
        double* s = (double*)malloc(sizeof(double) * (size_t)nkeys);
        double mx = -INFINITY;
        for (int i = 0; i < nkeys; ++i) {
            const uint16_t* kv;
            if (i < t) {
                kv = k_cache + (((size_t)b * Hkv + g) * T_cap + i) * D;
            } else {
                if (!vis[i - t]) { s[i] = -INFINITY; continue; }
                kv = k_blk + (((size_t)b * Hkv + g) * R + (i - t)) * D;
            }
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += (double)bf16_to_float(qv[d]) * (double)bf16_to_float(kv[d]);
            s[i] = dot * scale;
            if (s[i] > mx) mx = s[i];
        }
        double denom = 0.0;
        for (int i = 0; i < nkeys; ++i) {
            s[i] = (s[i] == -INFINITY) ? 0.0 : exp(s[i] - mx);
            denom += s[i];
        }
        double* o = out + (((size_t)b * R + j) * Hq + h) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int i = 0; i < nkeys; ++i) {
            if (s[i] == 0.0) continue;
            const uint16_t* vv = (i < t) ? v_cache + (((size_t)b * Hkv + g) * T_cap + i) * D
                                         : v_blk + (((size_t)b * Hkv + g) * R + (i - t)) * D;
            double wgt = s[i] / denom;
            for (int d = 0; d < D; ++d) o[d] += wgt * (double)bf16_to_float(vv[d]);
        }
        free(s);
        free(vis);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* LM head: logits[r][v] = sum_h hid[r][h] * W[h][v] in double, for the      */
/* vocab columns [v0, v1).  hid [N, H] bf16; W [H, V] bf16 row-major;        */
/* out [N, v1 - v0] double.                                                  */
/* ------------------------------------------------------------------------ */

int orc_lm_head(const uint16_t* hid, const uint16_t* W, int N, int H, int V, int v0, int v1, double* out) {
    if (N < 0 || H < 1 || V < 1 || v0 < 0 || v1 > V || v0 > v1) return ORC_ERR;
    int width = v1 - v0;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < N; ++r) {
        double* o = out + (size_t)r * width;
        for (int v = 0; v < width; ++v) o[v] = 0.0;
        for (int h = 0; h < H; ++h) {
            double x = (double)bf16_to_float(hid[(size_t)r * H + h]);
            const uint16_t* wrow = W + (size_t)h * V + v0;
            for (int v = 0; v < width; ++v) o[v] += x * (double)bf16_to_float(wrow[v]);
        }
    }
    return ORC_OK;
}
