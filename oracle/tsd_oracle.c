/*
 * tsd_oracle.c -- float64 CPU oracle for bounded-tree speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously-correct
 * restatement of what the CUDA library computes, used to check it.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library, and the
 * product path never calls it.
 *
 * Sources (page title, section / equation):
 *   [EXIT]  "Where Draft Trees Lose Target Mass: Exit-Guided Speculative
 *           Decoding" -- Sec. 3 Eq. 1-2 (p_v, P), Sec. 3.1 Eq. 4 (rho, w),
 *           Eq. 6 (target coverage), Eq. 7 (residual law), App. A.4.1
 *           (predraw-and-follow), Sec. 3.1 Lemma 1 (the canonical exit
 *           law that Tree Exit Verification samples).
 *   [CAST]  "CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters"
 *           -- Sec. 2 Eq. 1 (plug-in score), Thm. 1 (tie order), App. C
 *           "Candidate construction" (top-K heap, push all K children) and
 *           "Packed verification" (ancestor mask, position ids), App. B.1
 *           Thm. 3 (recursive speculative sampling without replacement),
 *           Sec. 3.3 Thm. 2 and App. B.3-B.4 Prop. 2-3 (cost-aware width,
 *           shared budget under load).
 *           Sec. 5 Eq. 14 and App. C.2 Eq. 66 (the exit-guided loss), App.
 *           A.4.2 Eq. 45-53 (exact sequential residual verification).
 *   [MFD]   "Multi-Future Drafting: Mixture Block Drafters for Tree-Verified
 *           Speculative Decoding" -- Sec. 3.4 Eq. 2 (best-mode score),
 *           App. B "Merged heap" and Prop. 6 (sibling / first-child pushes,
 *           node reuse across modes), App. B "Max or log-sum-exp" Eq. 6
 *           (mixture-probability score over the modes' per-depth lists).
 *   [PHILOX] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 *           as 1, 2, 3", SC'11 -- the Philox4x64-10 counter-based generator.
 *
 * Readings where the pages are open:
 *   - Uniforms: u = (x0 >> 40) * 2^-24 from Philox4x64-10 with
 *     counter (tree, node, stream, sub) and key (seed, 0); stream 0 = TEV exit
 *     draw, 1 = TEV bonus draw, 2 = predraw at node `node` (sub 0); 3 =
 *     sequential-residual test of the node's child number `sub`, 4 = its
 *     bonus draw; 5 / 6 = proposal-aware candidate draw / acceptance test at
 *     step `sub`, 7 = its final residual draw.
 *   - The sequential-residual and proposal-aware verifiers take a node's
 *     children in ascending token order; their decisions compare without
 *     dividing (u (1 - M) < p, u q~ < mu).
 *   - The pages leave the two draws of TEV (exit node, bonus token)
 *     unspecified beyond their laws; both are inverse-CDF sampling: nodes in index
 *     (build) order for the exit, token ids ascending (skipping the drafted
 *     children) for the bonus; strict '>' so zero-mass items are never drawn;
 *     the normaliser is the computed total, not 1.
 *   - rho(v) is evaluated as the residual sum over non-child tokens (the
 *     equality of Eq. 4 and Eq. 13 of [EXIT]); the test suite checks it
 *     against 1 - sum of child probabilities.
 *   - T = 0 is the greedy limit: p_v is one-hot at the arg-max (lowest id on
 *     ties).
 *   - Builder tie order: score desc, depth asc, mode asc, rank sequence
 *     lexicographic asc; top-k per position ordered by (logit desc, id asc).
 *   - Prefixes of zero drafter probability (score -inf) never become nodes.
 *   - Log-sum-exp tree: a mode's depth-d list is its B most probable
 *     length-d prefixes in the capped universe, built depth by depth and
 *     ordered by (path sum desc, parent's place asc, token rank asc); a
 *     distinct prefix is known by its first (depth, mode, place); the ranking
 *     key is s_lse clamped to the parent's key, ties by (depth, mode, place).
 *
 * Parity status: every function here is pinned by tests/test_oracle_pins.py
 * (brute force, closed forms, library routines, hand-computed fixtures).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_NONFINITE 5
#define ORC_ERR_BAD_TREE 4
#define ORC_MAX_DEPTH 64

/* ------------------------------------------------------------------------ */
/* Philox4x64-10 [PHILOX]: ten rounds of two 64x64->128 multiplies, with a  */
/* Weyl-sequence key schedule.                                               */
/* ------------------------------------------------------------------------ */
static const uint64_t PHILOX_M0 = 0xD2E7470EE14C6C93ULL;
static const uint64_t PHILOX_M1 = 0xCA5A826395121157ULL;
static const uint64_t PHILOX_W0 = 0x9E3779B97F4A7C15ULL;
static const uint64_t PHILOX_W1 = 0xBB67AE8584CAA73BULL;

void orc_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4])
{
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        unsigned __int128 p0 = (unsigned __int128)PHILOX_M0 * c0;
        unsigned __int128 p1 = (unsigned __int128)PHILOX_M1 * c2;
        uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        uint64_t n0 = hi1 ^ c1 ^ k0;
        uint64_t n1 = lo1;
        uint64_t n2 = hi0 ^ c3 ^ k1;
        uint64_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* One uniform in [0, 1) on a 2^-24 grid, for (seed; tree, node, stream, sub). */
double orc_uniform_sub(uint64_t seed, uint64_t tree, uint64_t node, uint64_t stream,
                       uint64_t sub)
{
    uint64_t ctr[4] = {tree, node, stream, sub};
    uint64_t key[2] = {seed, 0};
    uint64_t out[4];
    orc_philox4x64_10(ctr, key, out);
    return (double)(out[0] >> 40) * (1.0 / 16777216.0);
}

double orc_uniform(uint64_t seed, uint64_t tree, uint64_t node, uint64_t stream)
{
    return orc_uniform_sub(seed, tree, node, stream, 0);
}

/* ------------------------------------------------------------------------ */
/* Drafter statistics [CAST Sec. 2 Eq. 1, App. C]: for each row j,           */
/*   LSE_j = log sum_a exp(z_j(a)/T),  log q_j(a) = z_j(a)/T - LSE_j,       */
/* and the top-k tokens ordered by (logit desc, id asc), with their log q    */
/* and their scaled logits z/T (top_zt, nullable).                           */
/* ------------------------------------------------------------------------ */
int orc_drafter_stats(const double *z, int64_t rows, int64_t V, double temp, int k,
                      double *lse, int32_t *top_id, double *top_logq, double *top_zt)
{
    if (!(temp > 0.0) || k < 1 || k > V || V < 1) return ORC_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        const double *row = z + r * V;
        double m = -INFINITY;
        for (int64_t a = 0; a < V; ++a) {
            if (isnan(row[a]) || row[a] == INFINITY) return ORC_ERR_NONFINITE;
            if (row[a] > m) m = row[a];
        }
        if (m == -INFINITY) return ORC_ERR_NONFINITE;
        double s = 0.0;
        for (int64_t a = 0; a < V; ++a) s += exp((row[a] - m) / temp);
        lse[r] = m / temp + log(s);
        /* top-k by repeated selection: rank i is the best token that comes
         * after rank i-1 in the order (logit desc, id asc) */
        for (int i = 0; i < k; ++i) {
            int64_t best = -1;
            int64_t prev = i > 0 ? top_id[r * k + i - 1] : -1;
            for (int64_t a = 0; a < V; ++a) {
                if (prev >= 0 && !(row[a] < row[prev] || (row[a] == row[prev] && a > prev)))
                    continue; /* a is rank i-1 or ranked before it */
                if (best < 0 || row[a] > row[best]) best = a;  /* ties keep the lower id */
            }
            top_id[r * k + i] = (int32_t)best;
            top_logq[r * k + i] = row[best] / temp - lse[r];
            if (top_zt) top_zt[r * k + i] = row[best] / temp;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Best-first tree builder.                                                  */
/*                                                                           */
/* Universe: for each mode m (K modes; K = 1 is DDTree / CAST) and drafter   */
/* position j = 1..L, the k retained tokens of that mode's row.  A heap      */
/* entry (m, v) is a prefix v scored under mode m by its unrenormalised      */
/* log-probability s_m(v) = sum_j log q_{m,j}(v_j) [CAST Eq. 1; MFD Eq. 2    */
/* with a uniform prior, whose constant log(1/K) is dropped from the         */
/* ranking], evaluated as                                                    */
/*   s_m(v) = (sum_j z_{m,j}(v_j)/T) - C_m(|v|),  C_m(d) = sum_{j<=d} LSE_{m,j} */
/* with the path sum taken left to right: equal in exact arithmetic to the  */
/* sum of log q, and two prefixes of one depth and mode whose scaled logits  */
/* sum to the same value tie exactly, so the tie order decides them.         */
/*                                                                           */
/* push_rule 0 [MFD App. B]: seed with each mode's rank-0 first token; a pop */
/*   pushes its next sibling (rank r+1) and its first child (rank 0 at the   */
/*   next position).                                                         */
/* push_rule 1 [CAST App. C]: seed with each mode's k first tokens; a pop    */
/*   pushes all k children at the next position.                             */
/* A popped prefix already in the tree reuses its node and spends no budget; */
/* its successors are pushed either way [MFD App. B].                        */
/* ------------------------------------------------------------------------ */
typedef struct {
    double score;        /* s_m(v) = zsum - C_m(depth) */
    double zsum;         /* sum of z/T along v */
    double pzsum;        /* the same sum along v's parent */
    double pscore;       /* the score of v's parent (the root's is 0) */
    int32_t mode;
    int32_t depth;       /* |v| >= 1 */
    int32_t rank;        /* rank of v's last token in mode m's list */
    int32_t pnode;       /* tree node of v's parent */
    uint8_t ranks[ORC_MAX_DEPTH]; /* rank sequence r_1..r_depth */
} orc_entry;

/* 1 if a comes before b in the total order. */
static int orc_before(const orc_entry *a, const orc_entry *b)
{
    if (a->score != b->score) return a->score > b->score;
    if (a->depth != b->depth) return a->depth < b->depth;
    if (a->mode != b->mode) return a->mode < b->mode;
    for (int i = 0; i < a->depth; ++i)
        if (a->ranks[i] != b->ranks[i]) return a->ranks[i] < b->ranks[i];
    return 0;
}

typedef struct {
    orc_entry *e;
    int64_t n, cap;
} orc_heap;

static void heap_push(orc_heap *h, const orc_entry *x)
{
    int64_t i = h->n++;
    h->e[i] = *x;
    while (i > 0) {
        int64_t p = (i - 1) / 2;
        if (!orc_before(&h->e[i], &h->e[p])) break;
        orc_entry t = h->e[i]; h->e[i] = h->e[p]; h->e[p] = t;
        i = p;
    }
}

static orc_entry heap_pop(orc_heap *h)
{
    orc_entry top = h->e[0];
    h->e[0] = h->e[--h->n];
    int64_t i = 0;
    for (;;) {
        int64_t l = 2 * i + 1, r = l + 1, b = i;
        if (l < h->n && orc_before(&h->e[l], &h->e[b])) b = l;
        if (r < h->n && orc_before(&h->e[r], &h->e[b])) b = r;
        if (b == i) break;
        orc_entry t = h->e[i]; h->e[i] = h->e[b]; h->e[b] = t;
        i = b;
    }
    return top;
}

/*
 * top_id, top_zt: [K][L][k] (mode-major, then position, then rank): the
 * retained tokens and their scaled logits z/T; lse: [K][L] the rows'
 * log-normalisers.
 * Outputs have B+1 slots; node 0 is the root (parent -1, token -1, depth 0,
 * score 0).  Slots past n_nodes are filled with -1 and score -inf.
 */
int orc_build_tree(const int32_t *top_id, const double *top_zt, const double *lse, int K, int L,
                   int k, int B, int push_rule, int32_t *parent, int32_t *token,
                   int32_t *depth, double *score, int32_t *rank, int32_t *mode,
                   int32_t *n_nodes_out)
{
    if (K < 1 || L < 1 || L > ORC_MAX_DEPTH || k < 1 || k > 255 || B < 0) return ORC_ERR_ARG;
    for (int i = 0; i <= B; ++i) {
        parent[i] = token[i] = depth[i] = rank[i] = mode[i] = -1;
        score[i] = -INFINITY;
    }
    parent[0] = -1; token[0] = -1; depth[0] = 0; score[0] = 0.0;
    int32_t *first_child = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B + 1));
    int32_t *next_sib = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B + 1));
    for (int i = 0; i <= B; ++i) first_child[i] = next_sib[i] = -1;

    orc_heap h;
    h.cap = (int64_t)K * k + (int64_t)(k + 2) * K * (B + 1) + 16;
    h.n = 0;
    h.e = (orc_entry *)malloc(sizeof(orc_entry) * (size_t)h.cap);

#define ZT(m, j, r) top_zt[((int64_t)(m) * L + (j)) * k + (r)]
#define TK(m, j, r) top_id[((int64_t)(m) * L + (j)) * k + (r)]
    /* C_m(d): cumulative log-normaliser of mode m over positions 1..d */
    double *cum = (double *)malloc(sizeof(double) * (size_t)K * (size_t)(L + 1));
    for (int m = 0; m < K; ++m) {
        cum[m * (L + 1)] = 0.0;
        for (int d = 1; d <= L; ++d) cum[m * (L + 1) + d] = cum[m * (L + 1) + d - 1] + lse[m * L + d - 1];
    }
#define CUM(m, d) cum[(m) * (L + 1) + (d)]
    for (int m = 0; m < K; ++m) {
        int nseed = (push_rule == 0) ? 1 : k;
        for (int r = 0; r < nseed; ++r) {
            orc_entry x;
            memset(&x, 0, sizeof x);
            x.mode = m; x.depth = 1; x.rank = r; x.pnode = 0;
            x.pzsum = 0.0; x.zsum = 0.0 + ZT(m, 0, r);
            x.score = x.zsum - CUM(m, 1);
            x.pscore = 0.0;
            x.ranks[0] = (uint8_t)r;
            heap_push(&h, &x);
        }
    }
    int n = 1;
    int status = ORC_OK;
    while (n <= B && h.n > 0) {
        orc_entry e = heap_pop(&h);
        if (isnan(e.score)) { status = ORC_ERR_NONFINITE; break; }
        if (e.score == -INFINITY) break; /* only zero-probability prefixes remain */
        int32_t t = TK(e.mode, e.depth - 1, e.rank);
        /* find the node (pnode, t) if some mode already created it */
        int node = -1;
        for (int c = first_child[e.pnode]; c >= 0; c = next_sib[c])
            if (token[c] == t) { node = c; break; }
        if (node < 0) {
            node = n++;
            parent[node] = e.pnode; token[node] = t; depth[node] = e.depth;
            score[node] = e.score; rank[node] = e.rank; mode[node] = e.mode;
            /* append to the parent's child list */
            if (first_child[e.pnode] < 0) first_child[e.pnode] = node;
            else {
                int c = first_child[e.pnode];
                while (next_sib[c] >= 0) c = next_sib[c];
                next_sib[c] = node;
            }
        }
        if (push_rule == 0) {
            if (e.rank + 1 < k) { /* next sibling: same parent, rank + 1 */
                orc_entry s = e;
                s.rank = e.rank + 1;
                s.ranks[e.depth - 1] = (uint8_t)(e.rank + 1);
                s.zsum = e.pzsum + ZT(e.mode, e.depth - 1, e.rank + 1);
                s.score = s.zsum - CUM(e.mode, e.depth);
                /* A child's sum of log q cannot exceed its parent's (each
                 * log q <= 0, [CAST] Sec. 2 Eq. 1); where the rounding of the
                 * two path sums would put it above, it takes the parent's
                 * score, so that a parent always precedes its children in the
                 * (score desc, depth asc, ...) order.  Depth 1 is below the
                 * root's 0 already (z/T <= LSE). */
                if (e.depth > 1 && s.score > s.pscore) s.score = s.pscore;
                heap_push(&h, &s);
            }
            if (e.depth < L) { /* first child: rank 0 at the next position */
                orc_entry c = e;
                c.depth = e.depth + 1; c.rank = 0; c.pnode = node;
                c.pzsum = e.zsum; c.zsum = e.zsum + ZT(e.mode, e.depth, 0);
                c.score = c.zsum - CUM(e.mode, e.depth + 1);
                c.pscore = e.score;
                if (c.score > e.score) c.score = e.score;  /* as for siblings */
                c.ranks[e.depth] = 0;
                heap_push(&h, &c);
            }
        } else {
            if (e.depth < L) {
                for (int r = 0; r < k; ++r) {
                    orc_entry c = e;
                    c.depth = e.depth + 1; c.rank = r; c.pnode = node;
                    c.pzsum = e.zsum; c.zsum = e.zsum + ZT(e.mode, e.depth, r);
                    c.score = c.zsum - CUM(e.mode, e.depth + 1);
                    c.pscore = e.score;  /* clamped as for siblings */
                    if (c.score > e.score) c.score = e.score;
                    c.ranks[e.depth] = (uint8_t)r;
                    heap_push(&h, &c);
                }
            }
        }
    }
#undef ZT
#undef TK
#undef CUM
    free(cum);
    *n_nodes_out = n;
    free(h.e);
    free(first_child);
    free(next_sib);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Ancestor mask and position ids [CAST App. C "Packed verification";       */
/* Lemma 1]: row v sees the P prefix entries, its ancestors and itself;      */
/* pos(root) = P, pos(v) = P + depth(v).  Rows past n_nodes are padding:     */
/* they see the prefix and themselves only, at position P.                   */
/* bits: [B+1][W] u32 with W = ceil((B+1)/32), bit u of row v = column u.    */
/* addmask (nullable): [B+1][ld], 0 where visible and -inf elsewhere, over   */
/* columns [0, P + B + 1).                                                   */
/* ------------------------------------------------------------------------ */
int orc_tree_mask(const int32_t *parent, int n_nodes, int B, int prefix_len,
                  uint32_t *bits, int32_t *pos, double *addmask, int64_t ld)
{
    if (n_nodes < 1 || n_nodes > B + 1 || prefix_len < 0) return ORC_ERR_ARG;
    int W = (B + 1 + 31) / 32;
    memset(bits, 0, sizeof(uint32_t) * (size_t)(B + 1) * (size_t)W);
    for (int v = 0; v <= B; ++v) {
        int d = 0;
        if (v < n_nodes) {
            int u = v, steps = 0;
            while (u >= 0) {
                if (u >= n_nodes || steps > n_nodes) return ORC_ERR_BAD_TREE;
                bits[(int64_t)v * W + u / 32] |= 1u << (u % 32);
                u = parent[u];
                ++steps;
            }
            d = steps - 1;
        } else {
            bits[(int64_t)v * W + v / 32] |= 1u << (v % 32);
        }
        pos[v] = prefix_len + d;
        if (addmask) {
            double *row = addmask + (int64_t)v * ld;
            for (int c = 0; c < prefix_len; ++c) row[c] = 0.0;
            for (int u = 0; u <= B; ++u)
                row[prefix_len + u] = ((bits[(int64_t)v * W + u / 32] >> (u % 32)) & 1u) ? 0.0 : -INFINITY;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Target distributions at one node [EXIT Eq. 1]: p(a) = softmax(z/T)(a),    */
/* or one-hot at the arg-max (lowest id on ties) when T == 0.                */
/* ------------------------------------------------------------------------ */
int orc_row_probs(const double *z, int64_t V, double T, double *p)
{
    double m = -INFINITY;
    int64_t am = -1;
    for (int64_t a = 0; a < V; ++a) {
        if (isnan(z[a]) || z[a] == INFINITY) return ORC_ERR_NONFINITE;
        if (am < 0 || z[a] > m) { m = z[a]; am = a; }
    }
    if (m == -INFINITY) return ORC_ERR_NONFINITE;
    if (T == 0.0) {
        for (int64_t a = 0; a < V; ++a) p[a] = (a == am) ? 1.0 : 0.0;
        return ORC_OK;
    }
    double s = 0.0;
    for (int64_t a = 0; a < V; ++a) s += exp((z[a] - m) / T);
    for (int64_t a = 0; a < V; ++a) p[a] = exp((z[a] - m) / T) / s;
    return ORC_OK;
}

/* Check the tree: node 0 is the root, parents precede children, tokens lie in
 * [0, V), sibling tokens are distinct.  Fills depth[]. */
static int orc_check_tree(const int32_t *parent, const int32_t *token, int n, int64_t V,
                          int32_t *depth)
{
    if (n < 1 || parent[0] != -1) return ORC_ERR_BAD_TREE;
    depth[0] = 0;
    for (int u = 1; u < n; ++u) {
        if (parent[u] < 0 || parent[u] >= u) return ORC_ERR_BAD_TREE;
        if (token[u] < 0 || token[u] >= V) return ORC_ERR_BAD_TREE;
        depth[u] = depth[parent[u]] + 1;
        for (int s = 1; s < u; ++s)
            if (parent[s] == parent[u] && token[s] == token[u]) return ORC_ERR_BAD_TREE;
    }
    return ORC_OK;
}

/* Mark the drafted-child tokens of node v: mark[a] = child node index (>= 1)
 * for a in A(v), 0 otherwise.  The caller clears the marks with
 * orc_unmark_children. */
static void orc_mark_children(const int32_t *parent, const int32_t *token, int n, int v,
                              int32_t *mark)
{
    for (int u = 1; u < n; ++u)
        if (parent[u] == v) mark[token[u]] = u;
}

static void orc_unmark_children(const int32_t *parent, const int32_t *token, int n, int v,
                                int32_t *mark)
{
    for (int u = 1; u < n; ++u)
        if (parent[u] == v) mark[token[u]] = 0;
}

/* ------------------------------------------------------------------------ */
/* Tree Exit Verification on one tree: one draw from the canonical exit     */
/* law [EXIT Sec. 3.1 Lemma 1] -- exit at node v with probability w(v) =     */
/* P(v) rho(v) (Eq. 2, Eq. 4) -- then the bonus token from the residual law  */
/* of the exit node (Eq. 7).                                                 */
/*   z: [n][V] target logits, row v = node v.                                */
/* Outputs (length n unless noted):                                          */
/*   P      prefix probability, P(root) = 1, P(u) = P(pa u) p_pa(u)(x_u)     */
/*   rho    local exit probability (residual mass of non-child tokens)       */
/*   w      exit mass w = P rho                                              */
/*   pedge  p_pa(u)(x_u) for u >= 1 (pedge[0] = 1)                           */
/*   *coverage = C_p = sum_{u != root} P(u)                  [EXIT Eq. 6]    */
/*   *exit_node, *bonus, *accept_len = depth(exit) + 1                       */
/*   *u_exit, *u_bonus: the two uniforms used                                */
/* ------------------------------------------------------------------------ */
int orc_tev(const double *z, const int32_t *parent, const int32_t *token, int n, int64_t V,
            double T, uint64_t seed, uint64_t tree, double *P, double *rho, double *w,
            double *pedge, double *coverage, int32_t *exit_node, int32_t *bonus,
            int32_t *accept_len, double *u_exit, double *u_bonus)
{
    if (V < 1 || !(T >= 0.0)) return ORC_ERR_ARG;
    int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int st = orc_check_tree(parent, token, n, V, depth);
    if (st) { free(depth); return st; }
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    int32_t *mark = (int32_t *)calloc((size_t)V, sizeof(int32_t));

    /* The node-local quantities of Eq. 1 and Eq. 4 (p_v, rho(v)), the prefix
     * probabilities of Eq. 2 and the exit masses w = P rho.  Node indices are
     * parent-before-child, so one pass in index order visits every parent
     * before its children. */
    P[0] = 1.0;
    pedge[0] = 1.0;
    for (int v = 0; v < n; ++v) {
        st = orc_row_probs(z + (int64_t)v * V, V, T, p);
        if (st) break;
        orc_mark_children(parent, token, n, v, mark);
        double res = 0.0;
        for (int64_t a = 0; a < V; ++a)
            if (!mark[a]) res += p[a];
        orc_unmark_children(parent, token, n, v, mark);
        rho[v] = res;
        for (int u = v + 1; u < n; ++u)
            if (parent[u] == v) {
                pedge[u] = p[token[u]];
                P[u] = P[v] * pedge[u];
            }
        w[v] = P[v] * rho[v];
    }
    if (st) { free(mark); free(p); free(depth); return st; }
    double cp = 0.0;
    for (int u = 1; u < n; ++u) cp += P[u];
    *coverage = cp;

    /* The exit node: V ~ Categorical(w) [Lemma 1], inverse CDF in node order. */
    double wsum = 0.0;
    for (int v = 0; v < n; ++v) wsum += w[v];
    double u1 = orc_uniform(seed, tree, 0, 0);
    double thr = u1 * wsum, cum = 0.0;
    int ex = -1;
    for (int v = 0; v < n; ++v) {
        cum += w[v];
        if (cum > thr) { ex = v; break; }
    }
    if (ex < 0) { /* rounding left the last item short: take the last node with mass */
        for (int v = n - 1; v >= 0; --v)
            if (w[v] > 0.0) { ex = v; break; }
    }

    /* The bonus token: Y ~ p_V at a leaf, else the residual law of Eq. 7
     * (children's tokens removed, renormalised by rho(V)). */
    st = orc_row_probs(z + (int64_t)ex * V, V, T, p);
    double u2 = orc_uniform(seed, tree, 0, 1);
    double thr2 = u2 * rho[ex], cum2 = 0.0;
    int64_t y = -1, last_pos = -1;
    orc_mark_children(parent, token, n, ex, mark);
    for (int64_t a = 0; a < V; ++a) {
        if (mark[a]) continue;
        if (p[a] > 0.0) last_pos = a;
        cum2 += p[a];
        if (cum2 > thr2) { y = a; break; }
    }
    orc_unmark_children(parent, token, n, ex, mark);
    if (y < 0) y = last_pos;

    *exit_node = ex;
    *bonus = (int32_t)y;
    *accept_len = depth[ex] + 1;
    *u_exit = u1;
    *u_bonus = u2;
    free(mark);
    free(p);
    free(depth);
    return st;
}

/* ------------------------------------------------------------------------ */
/* Predraw-and-follow [EXIT Sec. 2, App. A.4.1]: draw R_v ~ p_v at every     */
/* node (inverse CDF over token ids, uniform stream 2 at node v); walk from  */
/* the root into the child whose token equals R_v; exit at the first node    */
/* with no matching child and return R_v as the bonus token.                 */
/*   draws: [n] the per-node draws R_v.                                      */
/* ------------------------------------------------------------------------ */
int orc_predraw(const double *z, const int32_t *parent, const int32_t *token, int n, int64_t V,
                double T, uint64_t seed, uint64_t tree, int32_t *draws, int32_t *exit_node,
                int32_t *bonus, int32_t *accept_len)
{
    if (V < 1 || !(T >= 0.0)) return ORC_ERR_ARG;
    int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int st = orc_check_tree(parent, token, n, V, depth);
    if (st) { free(depth); return st; }
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    int32_t *mark = (int32_t *)calloc((size_t)V, sizeof(int32_t));
    for (int v = 0; v < n && !st; ++v) {
        st = orc_row_probs(z + (int64_t)v * V, V, T, p);
        if (st) break;
        double tot = 0.0;
        for (int64_t a = 0; a < V; ++a) tot += p[a];
        double thr = orc_uniform(seed, tree, (uint64_t)v, 2) * tot, cum = 0.0;
        int64_t r = -1, last_pos = -1;
        for (int64_t a = 0; a < V; ++a) {
            if (p[a] > 0.0) last_pos = a;
            cum += p[a];
            if (cum > thr) { r = a; break; }
        }
        draws[v] = (int32_t)(r >= 0 ? r : last_pos);
    }
    if (!st) {
        int v = 0;
        for (;;) {
            orc_mark_children(parent, token, n, v, mark);
            int c = mark[draws[v]];
            orc_unmark_children(parent, token, n, v, mark);
            if (!c) break;
            v = c;
        }
        *exit_node = v;
        *bonus = draws[v];
        *accept_len = depth[v] + 1;
    }
    free(mark);
    free(p);
    free(depth);
    return st;
}

/* ------------------------------------------------------------------------ */
/* Repeated draws for the law tests: draw i uses tree index first_tree + i,  */
/* so every draw has its own uniforms on the same tree and logits.           */
/* ------------------------------------------------------------------------ */
int orc_tev_sample_many(const double *z, const int32_t *parent, const int32_t *token, int n,
                        int64_t V, double T, uint64_t seed, uint64_t first_tree, int64_t n_draws,
                        int32_t *exit_out, int32_t *bonus_out)
{
    double *P = (double *)malloc(sizeof(double) * (size_t)n * 4);
    double cov, ue, ub;
    int32_t al;
    int st = ORC_OK;
    for (int64_t i = 0; i < n_draws && !st; ++i)
        st = orc_tev(z, parent, token, n, V, T, seed, first_tree + (uint64_t)i, P, P + n, P + 2 * n,
                     P + 3 * n, &cov, exit_out + i, bonus_out + i, &al, &ue, &ub);
    free(P);
    return st;
}

int orc_predraw_sample_many(const double *z, const int32_t *parent, const int32_t *token, int n,
                            int64_t V, double T, uint64_t seed, uint64_t first_tree,
                            int64_t n_draws, int32_t *exit_out, int32_t *bonus_out)
{
    int32_t *draws = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t al;
    int st = ORC_OK;
    for (int64_t i = 0; i < n_draws && !st; ++i)
        st = orc_predraw(z, parent, token, n, V, T, seed, first_tree + (uint64_t)i, draws,
                         exit_out + i, bonus_out + i, &al);
    free(draws);
    return st;
}

/* ------------------------------------------------------------------------ */
/* Exit-guided loss [EXIT Sec. 5 Eq. 14, App. C.2 Eq. 66], one example.      */
/* The numerator of Eq. 14: the sum over non-root nodes v of                 */
/*   omega(v) * (-log q_{depth(v)}(x_v)),                                    */
/* where x_v is scored by the drafter row of future position depth(v)        */
/* (row depth(v) - 1 of z) and log q = z/T_d - logsumexp(z/T_d) over the     */
/* row.  Every node's term is formed on its own, as Eq. 66 writes it (not    */
/* through the per-row regrouping of Eq. 67).                                */
/*   z: [L][V] drafter logits; token, depth: [n] (node 0 is the root and     */
/*   is skipped); omega: [n] detached weights (the exit masses w(v)).        */
/*   *num: the numerator.  grad (nullable): [L][V] d(num)/dz, i.e.           */
/*   sum over nodes v on row m of omega(v) (softmax(z_m/T)(a) - [a = x_v])/T. */
/* ------------------------------------------------------------------------ */
int orc_exit_loss(const double *z, int L, int64_t V, double T, const int32_t *token,
                  const int32_t *depth, int n, const double *omega, double *num, double *grad)
{
    if (L < 1 || V < 1 || n < 1 || !(T > 0.0)) return ORC_ERR_ARG;
    for (int v = 1; v < n; ++v)
        if (depth[v] < 1 || depth[v] > L || token[v] < 0 || (int64_t)token[v] >= V)
            return ORC_ERR_BAD_TREE;
    if (grad) memset(grad, 0, sizeof(double) * (size_t)L * (size_t)V);
    double total = 0.0;
    for (int v = 1; v < n; ++v) {
        const double *row = z + (int64_t)(depth[v] - 1) * V;
        double m = -INFINITY;
        for (int64_t a = 0; a < V; ++a)
            if (row[a] / T > m) m = row[a] / T;
        if (!isfinite(m)) return ORC_ERR_NONFINITE;
        double s = 0.0;
        for (int64_t a = 0; a < V; ++a) s += exp(row[a] / T - m);
        const double lse = m + log(s);
        const double nlq = lse - row[token[v]] / T; /* -log q_{depth(v)}(x_v) */
        if (!isfinite(nlq)) return ORC_ERR_NONFINITE;
        total += omega[v] * nlq;
        if (grad) {
            double *g = grad + (int64_t)(depth[v] - 1) * V;
            for (int64_t a = 0; a < V; ++a) g[a] += omega[v] * exp(row[a] / T - lse) / T;
            g[token[v]] -= omega[v] / T;
        }
    }
    *num = total;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Children of v in ascending token order (the order both verifiers below    */
/* test them in); returns their count.                                       */
/* ------------------------------------------------------------------------ */
static int orc_children_by_token(const int32_t *parent, const int32_t *token, int n, int v,
                                 int32_t *kids)
{
    int k = 0;
    for (int u = 1; u < n; ++u)
        if (parent[u] == v) kids[k++] = u;
    for (int i = 1; i < k; ++i) { /* insertion sort by token (sibling tokens are distinct) */
        int x = kids[i], j = i - 1;
        while (j >= 0 && token[kids[j]] > token[x]) { kids[j + 1] = kids[j]; --j; }
        kids[j + 1] = x;
    }
    return k;
}

/* Inverse-CDF draw over token ids ascending of the masses m[0..V) with total
 * `tot` and uniform u: the first a whose running sum exceeds u * tot (strict),
 * or the last token with mass when rounding leaves the threshold past it. */
static int64_t orc_draw_tokens(const double *m, int64_t V, double tot, double u)
{
    double thr = u * tot, cum = 0.0;
    int64_t last = -1;
    for (int64_t a = 0; a < V; ++a) {
        if (m[a] > 0.0) last = a;
        cum += m[a];
        if (cum > thr) return a;
    }
    return last;
}

/* ------------------------------------------------------------------------ */
/* Exact sequential residual verification [EXIT App. A.4.2, Eq. 45-53].      */
/* At the current node v, children u_1..u_k (ascending token) are tested in  */
/* turn: with p_j = p_v(x_j) and M_{j-1} = p_1 + ... + p_{j-1}, child u_j is  */
/* followed with the conditional probability g^(j-1)(x_j) = p_j/(1-M_{j-1})  */
/* (Eq. 49), decided as u_j (1 - M_{j-1}) < p_j with u_j the uniform of      */
/* stream 3, sub j-1, at node v.  If every child is rejected the walk exits  */
/* at v and draws the bonus token from g^(k), which is p_v without the       */
/* children's tokens renormalised (Eq. 53; p_v at a leaf), by inverse CDF     */
/* over token ids with the uniform of stream 4 at v.                         */
/* ------------------------------------------------------------------------ */
int orc_seqres(const double *z, const int32_t *parent, const int32_t *token, int n, int64_t V,
               double T, uint64_t seed, uint64_t tree, int32_t *exit_node, int32_t *bonus,
               int32_t *accept_len)
{
    if (V < 1 || !(T >= 0.0)) return ORC_ERR_ARG;
    int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int st = orc_check_tree(parent, token, n, V, depth);
    if (st) { free(depth); return st; }
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    int32_t *kids = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int v = 0;
    for (;;) {
        st = orc_row_probs(z + (int64_t)v * V, V, T, p);
        if (st) break;
        const int k = orc_children_by_token(parent, token, n, v, kids);
        double M = 0.0;
        int next = -1;
        for (int j = 0; j < k; ++j) {
            const double pj = p[token[kids[j]]];
            const double u = orc_uniform_sub(seed, tree, (uint64_t)v, 3, (uint64_t)j);
            if (u * (1.0 - M) < pj) { next = kids[j]; break; }
            M += pj;
        }
        if (next >= 0) { v = next; continue; }
        /* exit at v: the residual law of Eq. 53 */
        for (int j = 0; j < k; ++j) p[token[kids[j]]] = 0.0;
        double tot = 0.0;
        for (int64_t a = 0; a < V; ++a) tot += p[a];
        const int64_t y = orc_draw_tokens(p, V, tot, orc_uniform_sub(seed, tree, (uint64_t)v, 4, 0));
        *exit_node = v;
        *bonus = (int32_t)y;
        *accept_len = depth[v] + 1;
        break;
    }
    free(kids);
    free(p);
    free(depth);
    return st;
}

/* ------------------------------------------------------------------------ */
/* Proposal-aware verification [CAST App. B.1 Thm. 3]: recursive            */
/* speculative sampling without replacement at each visited node.  The       */
/* residual mu starts at p_v.  While retained siblings remain, a candidate c */
/* is drawn from the proposal renormalised over them, q~ (inverse CDF over   */
/* the retained children in ascending token order, uniform of stream 5, sub  */
/* = step), and accepted with probability min(1, mu(c)/q~(c)), decided as    */
/* u q~(c) < mu(c) (stream 6, sub = step).  Acceptance follows the child.    */
/* Rejection sets mu <- (mu - q~)_+ / ||(mu - q~)_+||_1 (q~ is zero off the   */
/* retained siblings) and retires c.  When every sibling is retired, the     */
/* committed token is drawn from mu (stream 7) and the walk exits at v with  */
/* it as the bonus token; at a leaf mu = p_v.                                */
/*   q_child: [n] the proposal's probability of each node's token under its  */
/*   parent, q_{pa(u)}(x_u) (q_child[0] unused); positive on every child.     */
/* ------------------------------------------------------------------------ */
int orc_proposal(const double *z, const int32_t *parent, const int32_t *token, int n, int64_t V,
                 double T, const double *q_child, uint64_t seed, uint64_t tree, int32_t *exit_node,
                 int32_t *bonus, int32_t *accept_len)
{
    if (V < 1 || !(T >= 0.0)) return ORC_ERR_ARG;
    int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int st = orc_check_tree(parent, token, n, V, depth);
    if (st) { free(depth); return st; }
    for (int u = 1; u < n; ++u)
        if (!(q_child[u] > 0.0) || !isfinite(q_child[u])) { free(depth); return ORC_ERR_ARG; }
    double *mu = (double *)malloc(sizeof(double) * (size_t)V);
    int32_t *kids = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    char *avail = (char *)malloc((size_t)n);
    int v = 0;
    for (;;) {
        st = orc_row_probs(z + (int64_t)v * V, V, T, mu);
        if (st) break;
        const int k = orc_children_by_token(parent, token, n, v, kids);
        for (int j = 0; j < k; ++j) avail[j] = 1;
        int next = -1, left = k;
        for (int step = 0; left > 0; ++step) {
            double Q = 0.0;
            for (int j = 0; j < k; ++j)
                if (avail[j]) Q += q_child[kids[j]];
            const double u1 = orc_uniform_sub(seed, tree, (uint64_t)v, 5, (uint64_t)step);
            double thr = u1 * Q, cum = 0.0;
            int c = -1, lastj = -1;
            for (int j = 0; j < k; ++j) {
                if (!avail[j]) continue;
                lastj = j;
                cum += q_child[kids[j]];
                if (cum > thr) { c = j; break; }
            }
            if (c < 0) c = lastj;
            const double qc = q_child[kids[c]] / Q;
            const double u2 = orc_uniform_sub(seed, tree, (uint64_t)v, 6, (uint64_t)step);
            if (u2 * qc < mu[token[kids[c]]]) { next = kids[c]; break; }
            /* rejection: mu <- (mu - q~)_+ normalised */
            double norm = 0.0;
            for (int j = 0; j < k; ++j)
                if (avail[j]) {
                    const int64_t a = token[kids[j]];
                    const double d = mu[a] - q_child[kids[j]] / Q;
                    mu[a] = d > 0.0 ? d : 0.0;
                }
            for (int64_t a = 0; a < V; ++a) norm += mu[a];
            if (!(norm > 0.0)) { st = ORC_ERR_NONFINITE; break; }
            for (int64_t a = 0; a < V; ++a) mu[a] /= norm;
            avail[c] = 0;
            --left;
        }
        if (st) break;
        if (next >= 0) { v = next; continue; }
        double tot = 0.0;
        for (int64_t a = 0; a < V; ++a) tot += mu[a];
        const int64_t y = orc_draw_tokens(mu, V, tot, orc_uniform_sub(seed, tree, (uint64_t)v, 7, 0));
        *exit_node = v;
        *bonus = (int32_t)y;
        *accept_len = depth[v] + 1;
        break;
    }
    free(avail);
    free(kids);
    free(mu);
    free(depth);
    return st;
}

/* Repeated draws of the two verifiers above (draw i on tree index first_tree + i). */
int orc_seqres_sample_many(const double *z, const int32_t *parent, const int32_t *token, int n,
                           int64_t V, double T, uint64_t seed, uint64_t first_tree,
                           int64_t n_draws, int32_t *exit_out, int32_t *bonus_out)
{
    int32_t al;
    int st = ORC_OK;
    for (int64_t i = 0; i < n_draws && !st; ++i)
        st = orc_seqres(z, parent, token, n, V, T, seed, first_tree + (uint64_t)i, exit_out + i,
                        bonus_out + i, &al);
    return st;
}

int orc_proposal_sample_many(const double *z, const int32_t *parent, const int32_t *token, int n,
                             int64_t V, double T, const double *q_child, uint64_t seed,
                             uint64_t first_tree, int64_t n_draws, int32_t *exit_out,
                             int32_t *bonus_out)
{
    int32_t al;
    int st = ORC_OK;
    for (int64_t i = 0; i < n_draws && !st; ++i)
        st = orc_proposal(z, parent, token, n, V, T, q_child, seed, first_tree + (uint64_t)i,
                          exit_out + i, bonus_out + i, &al);
    return st;
}

/* ------------------------------------------------------------------------ */
/* Shared budget under load [CAST Sec. 3.3, App. B.4 Prop. 2-3].            */
/* Each of R requests brings its candidate prefixes in its best-first order  */
/* (the builder's pop order: scores[r][1..n_r-1] nonincreasing, node 0 the   */
/* root).  The disjoint union is ranked by prefix mass rho = exp(score)      */
/* (score desc), ties toward shorter prefixes (depth asc), then request      */
/* index, then the request's own order (node index).  With the affine round  */
/* time l(M) = l0 + c1 M, global node M+1 is added while                     */
/*   rho_(M+1) >= (G(M) + R) / l(M) * c1,   G(M) = sum of the M largest,     */
/* at most M_max nodes in all.  width[r] = how many of request r's prefixes  */
/* are among the M* selected; they are its first width[r] nodes.            */
/*   scores, depth: [R][stride] (stride >= max n_r), n_nodes: [R].          */
/* ------------------------------------------------------------------------ */
int orc_forest_select(const double *scores, const int32_t *depth, const int32_t *n_nodes, int R,
                      int stride, int M_max, double l0, double c1, int32_t *width,
                      int32_t *M_star, double *G_star)
{
    if (R < 1 || stride < 1 || M_max < 0 || !(l0 > 0.0) || !(c1 >= 0.0)) return ORC_ERR_ARG;
    int *pos = (int *)malloc(sizeof(int) * (size_t)R); /* next node of each request */
    for (int r = 0; r < R; ++r) {
        pos[r] = 1;
        width[r] = 0;
        if (n_nodes[r] < 0 || n_nodes[r] > stride) { free(pos); return ORC_ERR_ARG; }
    }
    double G = 0.0;
    int M = 0;
    while (M < M_max) {
        /* the next global node: the best head among the requests */
        int best = -1;
        for (int r = 0; r < R; ++r) {
            if (pos[r] >= n_nodes[r]) continue;
            if (best < 0) { best = r; continue; }
            const double a = scores[(int64_t)r * stride + pos[r]];
            const double b = scores[(int64_t)best * stride + pos[best]];
            const int da = depth[(int64_t)r * stride + pos[r]];
            const int db = depth[(int64_t)best * stride + pos[best]];
            if (a > b || (a == b && da < db)) best = r; /* equal: the lower index stays */
        }
        if (best < 0) break;
        const double rho = exp(scores[(int64_t)best * stride + pos[best]]);
        const double l = l0 + c1 * (double)M;
        if (!(rho >= (G + (double)R) / l * c1)) break;
        G += rho;
        ++width[best];
        ++pos[best];
        ++M;
    }
    *M_star = M;
    *G_star = G;
    free(pos);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Mixture tree under the log-sum-exp score [MFD App. B "Max or log-sum-exp", */
/* Eq. 6]: s_lse(v) = log sum_m pi_m Q_m(v), Q_m(v) = prod_j q_{m,j}(v_j).   */
/* No heap merge yields it: the pages rank by the mixture probability the     */
/* distinct prefixes of the modes' per-depth top-B lists.                    */
/*                                                                           */
/* Reading: mode m's depth-d list holds its B most probable length-d         */
/* prefixes whose tokens are among the mode's k retained tokens per position */
/* (the builder's capped universe).  Q_m factorises over positions, so the    */
/* parent of a listed prefix is listed one depth up, and the depth-d list is  */
/* the best B children of the depth-(d-1) list, ordered by (path sum of z/T   */
/* desc, parent's place asc, token rank asc); zero-probability prefixes are   */
/* left out.  Each distinct prefix is known by its first appearance in       */
/* (depth, mode, place) order.  It gets log Q_m(v) for every mode from the    */
/* full rows (the path sum of z_{m,j}(v_j)/T minus the summed row            */
/* log-normalisers, as the builder scores), and s_lse = log sum_m            */
/* exp(log pi_m + log Q_m(v)); pi is uniform when no prior is given.  The     */
/* ranking key is s_lse clamped to its parent's key (equal in exact          */
/* arithmetic: Q_m only falls along a path), and the tree takes the B best   */
/* distinct prefixes by (key desc, depth asc, mode asc, place asc), which is */
/* prefix-closed.                                                            */
/* ------------------------------------------------------------------------ */
typedef struct {
    double ps;   /* path sum of z/T along the prefix */
    int32_t par; /* place of the parent in the previous depth's list (-1: root) */
    int32_t r;   /* rank of the last token in the mode's list at this position */
} orc_beam_entry;

static int orc_beam_cmp(const void *a, const void *b)
{
    const orc_beam_entry *x = (const orc_beam_entry *)a, *y = (const orc_beam_entry *)b;
    if (x->ps != y->ps) return x->ps > y->ps ? -1 : 1;
    if (x->par != y->par) return x->par < y->par ? -1 : 1;
    return (x->r > y->r) - (x->r < y->r);
}

typedef struct {
    double key;
    int64_t flat; /* (depth, mode, place) flattened: the tie order */
} orc_lse_cand;

static int orc_lse_cmp(const void *a, const void *b)
{
    const orc_lse_cand *x = (const orc_lse_cand *)a, *y = (const orc_lse_cand *)b;
    if (x->key != y->key) return x->key > y->key ? -1 : 1;
    return (x->flat > y->flat) - (x->flat < y->flat);
}

/*
 * z: [K][L][V] drafter logits; log_prior: [K] or NULL (uniform).
 * Outputs have B+1 slots as orc_build_tree's (score = the ranking key);
 * n_cand_out: the number of distinct candidate prefixes.
 */
int orc_lse_tree(const double *z, int K, int L, int64_t V, double temp, int k, int B,
                 const double *log_prior, int32_t *parent, int32_t *token, int32_t *depth,
                 double *score, int32_t *n_nodes_out, int32_t *n_cand_out)
{
    if (K < 1 || K > 64 || L < 1 || L > ORC_MAX_DEPTH || k < 1 || k > V || B < 0 ||
        !(temp > 0.0))
        return ORC_ERR_ARG;
    for (int i = 0; i <= B; ++i) {
        parent[i] = token[i] = depth[i] = -1;
        score[i] = -INFINITY;
    }
    parent[0] = -1; token[0] = -1; depth[0] = 0; score[0] = 0.0;
    *n_nodes_out = 1;
    *n_cand_out = 0;
    const int64_t rows = (int64_t)K * L;
    double *lse = (double *)malloc(sizeof(double) * (size_t)rows);
    int32_t *top_id = (int32_t *)malloc(sizeof(int32_t) * (size_t)(rows * k));
    double *top_logq = (double *)malloc(sizeof(double) * (size_t)(rows * k));
    double *top_zt = (double *)malloc(sizeof(double) * (size_t)(rows * k));
    int st = orc_drafter_stats(z, rows, V, temp, k, lse, top_id, top_logq, top_zt);
    if (st != ORC_OK || B == 0) {
        free(lse); free(top_id); free(top_logq); free(top_zt);
        return st;
    }
    /* lists[m][d][i], sizes nb[m][d] */
    const int64_t per = (int64_t)B;
    orc_beam_entry *lists = (orc_beam_entry *)malloc(sizeof(orc_beam_entry) * (size_t)(rows * per));
    int32_t *nb = (int32_t *)calloc((size_t)rows, sizeof(int32_t));
    orc_beam_entry *kids = (orc_beam_entry *)malloc(sizeof(orc_beam_entry) * (size_t)(per * k + k));
    for (int m = 0; m < K; ++m) {
        for (int d = 0; d < L; ++d) {
            const int64_t row = (int64_t)m * L + d;
            int n = 0;
            const int np = d == 0 ? 1 : nb[row - 1];
            for (int i = 0; i < np; ++i) {
                const double base = d == 0 ? 0.0 : lists[(row - 1) * per + i].ps;
                for (int r = 0; r < k; ++r) {
                    const double ps = d == 0 ? top_zt[row * k + r] : base + top_zt[row * k + r];
                    if (ps == -INFINITY) continue;
                    kids[n].ps = ps;
                    kids[n].par = d == 0 ? -1 : i;
                    kids[n].r = r;
                    ++n;
                }
            }
            qsort(kids, (size_t)n, sizeof(orc_beam_entry), orc_beam_cmp);
            nb[row] = n < B ? n : B;
            memcpy(lists + row * per, kids, sizeof(orc_beam_entry) * (size_t)nb[row]);
        }
    }
    /* distinct prefixes: rep[flat] = flat index of the first appearance */
    const int64_t nflat = (int64_t)L * K * per;
#define FLAT(d, m, i) (((int64_t)(d) * K + (m)) * per + (i))
    int64_t *rep = (int64_t *)malloc(sizeof(int64_t) * (size_t)nflat);
    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)nflat);
    int64_t *prep = (int64_t *)malloc(sizeof(int64_t) * (size_t)nflat); /* parent's rep, -1 root */
    double *key = (double *)malloc(sizeof(double) * (size_t)nflat);
    orc_lse_cand *cand = (orc_lse_cand *)malloc(sizeof(orc_lse_cand) * (size_t)nflat);
    int32_t *path = (int32_t *)malloc(sizeof(int32_t) * (size_t)L);
    int64_t nc = 0;
    for (int d = 0; d < L; ++d) {
        for (int m = 0; m < K; ++m) {
            const int64_t row = (int64_t)m * L + d;
            for (int i = 0; i < nb[row]; ++i) {
                const orc_beam_entry *e = lists + row * per + i;
                const int64_t f = FLAT(d, m, i);
                tok[f] = top_id[row * k + e->r];
                prep[f] = d == 0 ? -1 : rep[FLAT(d - 1, m, e->par)];
                rep[f] = f;
                /* an earlier appearance of the same prefix at this depth */
                for (int m2 = 0; m2 <= m && rep[f] == f; ++m2) {
                    const int n2 = m2 < m ? nb[(int64_t)m2 * L + d] : i;
                    for (int i2 = 0; i2 < n2; ++i2) {
                        const int64_t g = FLAT(d, m2, i2);
                        if (rep[g] == g && tok[g] == tok[f] && prep[g] == prep[f]) {
                            rep[f] = g;
                            break;
                        }
                    }
                }
                if (rep[f] != f) continue;
                /* the token path, root first */
                int64_t u = f;
                for (int j = d; j >= 0; --j) {
                    path[j] = tok[u];
                    u = prep[u];
                }
                double tmax = -INFINITY;
                double t[64];
                for (int mm = 0; mm < K; ++mm) {
                    double ps = 0.0, c = 0.0;
                    for (int j = 0; j <= d; ++j) {
                        const int64_t rr = (int64_t)mm * L + j;
                        ps = ps + z[rr * V + path[j]] / temp;
                        c = c + lse[rr];
                    }
                    const double lp = log_prior ? log_prior[mm] : -log((double)K);
                    t[mm] = lp + (ps - c);
                    if (t[mm] > tmax) tmax = t[mm];
                }
                double s = -INFINITY;
                if (tmax > -INFINITY) {
                    double acc = 0.0;
                    for (int mm = 0; mm < K; ++mm) acc += exp(t[mm] - tmax);
                    s = tmax + log(acc);
                }
                const double up = d == 0 ? INFINITY : key[prep[f]];
                key[f] = s < up ? s : up;
                if (key[f] > -INFINITY) {
                    cand[nc].key = key[f];
                    cand[nc].flat = f;
                    ++nc;
                }
            }
        }
    }
    *n_cand_out = (int32_t)nc;
    qsort(cand, (size_t)nc, sizeof(orc_lse_cand), orc_lse_cmp);
    /* the B best, in order; a parent always precedes its children */
    int32_t *node_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)nflat);
    for (int64_t f = 0; f < nflat; ++f) node_of[f] = -1;
    const int64_t take = nc < B ? nc : B;
    st = ORC_OK;
    for (int64_t q = 0; q < take; ++q) {
        const int64_t f = cand[q].flat;
        const int n = (int)q + 1;
        node_of[f] = n;
        const int pn = prep[f] < 0 ? 0 : node_of[prep[f]];
        if (pn < 0) { st = ORC_ERR_BAD_TREE; break; }
        parent[n] = pn;
        token[n] = tok[f];
        depth[n] = (int32_t)(f / ((int64_t)K * per)) + 1;
        score[n] = cand[q].key;
    }
    *n_nodes_out = (int32_t)take + 1;
#undef FLAT
    free(lse); free(top_id); free(top_logq); free(top_zt); free(lists); free(nb); free(kids);
    free(rep); free(tok); free(prep); free(key); free(cand); free(path); free(node_of);
    return st;
}
