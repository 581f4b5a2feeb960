/*
 * tsd.h -- C ABI of the GB300 (sm_103a) library for the data-parallel hot path
 * of bounded-tree speculative decoding.
 *
 * Pages the operations restate:
 *   [EXIT] "Where Draft Trees Lose Target Mass: Exit-Guided Speculative
 *          Decoding": Sec. 3 Eq. 1-2, Sec. 3.1 Eq. 4, Eq. 6-7, App. A.4.1
 *          (predraw-and-follow), App. A.4.2 Eq. 45-53 (sequential residual
 *          verification), App. B Algorithm 1 (TEV), Sec. 5 Eq. 14 and App. C.2
 *          Eq. 66-67 (the exit-guided loss).
 *   [CAST] "CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters":
 *          Sec. 2 Eq. 1, Thm. 1, App. C ("Candidate construction",
 *          "Packed verification"), App. B Lemma 1, Sec. 3.3 Thm. 2 and App.
 *          B.4 Prop. 2-3 (cost-aware width, shared budget), App. B.1 Thm. 3
 *          (proposal-aware verification).
 *   [MFD]  "Multi-Future Drafting: Mixture Block Drafters for Tree-Verified
 *          Speculative Decoding": Sec. 3.4 Eq. 2, Prop. 4, Sec. 4.3,
 *          App. B "Merged heap", Prop. 6, "Max or log-sum-exp" Eq. 6.
 *
 * Conventions shared by every entry point:
 *   - Every array argument is DEVICE memory owned by the caller, contiguous and
 *     row-major in the shape given, except the logits (drafter_logits,
 *     target_logits), which may also be page-locked host memory
 *     (cudaHostAlloc / cudaMallocHost / cudaHostRegister): the kernels then
 *     read them in place over the host link, through the device address the
 *     runtime maps for them.  Each call resolves the logits pointer with
 *     cudaPointerGetAttributes; pageable host memory, or a pointer the runtime
 *     does not know, is TSD_ERR_INVALID_ARG.  The library allocates nothing
 *     and keeps no state between calls, apart from a host-side cache of each
 *     kernel's occupancy per device (thread-safe).
 *   - Calls are asynchronous on `stream`.  Argument errors are detected on the
 *     host before anything is launched and returned at once; nothing is
 *     written in that case.  TSD_ERR_CUDA reports a launch failure.
 *   - Errors in the data of one tree (a malformed tree, a NaN or +inf logit,
 *     a row without mass) are written to status[tree] on the device and can be
 *     read after the stream synchronises; that tree's outputs are then filled
 *     with -1 / 0 and the other trees are unaffected.  No kernel traps.
 *   - A tree has n_nodes[t] <= B+1 nodes.  Node 0 is the root (the pending
 *     root token of [CAST] Sec. 2); nodes are numbered parent-before-child
 *     (parent[0] = -1, 0 <= parent[u] < u), which is the builder's pop order.
 *     Sibling tokens are distinct.  Slots past n_nodes are ignored on input.
 *   - Logits rows follow node order: target_logits[t][v] is the target's
 *     next-token logits at node v.  bf16 or fp32; rows need not be aligned,
 *     but 16-byte aligned rows with V a multiple of 8 (bf16) or 4 (fp32) take
 *     the vectorised path.
 *   - `workspace` is device scratch of at least tsd_workspace_size(...) bytes,
 *     16-byte aligned.  Its contents on entry do not matter.
 *   - Randomness: the seed is the only source of the auxiliary randomness of
 *     [EXIT] Sec. 3.  Uniforms are Philox4x64-10 (Salmon et al., SC'11) with
 *     counter (tree, node, stream, 0) and key (seed, 0), u = (x0 >> 40) 2^-24;
 *     stream 0 = TEV exit draw, 1 = TEV bonus draw, 2 = predraw at `node`;
 *     streams 3-7 (with a sub-index in the counter's last word) belong to the
 *     sequential-residual and proposal-aware verifiers below.
 */
#ifndef TSD_H
#define TSD_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TSD_OK = 0,
    TSD_ERR_INVALID_ARG = 1, /* a null pointer, a size or option out of range */
    TSD_ERR_CUDA = 2,        /* a kernel launch failed */
    TSD_ERR_WORKSPACE = 3,   /* ws_bytes below tsd_workspace_size, or workspace misaligned */
    TSD_ERR_BAD_TREE = 4,    /* per tree: parent/token/n_nodes violate the conventions */
    TSD_ERR_NONFINITE = 5,   /* per tree: a NaN or +inf logit, or a row with no mass */
    TSD_ERR_TIMEOUT = 6      /* reserved: no kernel of this library waits on another */
} tsd_status;

typedef enum { TSD_BF16 = 0, TSD_F32 = 1 } tsd_dtype;

typedef enum {
    TSD_OP_BUILD_TREE = 0,
    TSD_OP_VERIFY_TEV = 1,
    TSD_OP_VERIFY_DDTREE = 2,
    TSD_OP_EXIT_LOSS = 3,
    TSD_OP_BUILD_FOREST = 4,
    TSD_OP_BUILD_LSE = 5
} tsd_op;

/* Limits checked by every entry point. */
#define TSD_MAX_B 4095      /* non-root budget */
#define TSD_MAX_TOPK 32     /* per-position top-k */
#define TSD_MAX_MODES 8     /* mixture modes */
#define TSD_MAX_L 31        /* drafter rows (= maximum depth) */

/* A static English description of a status code.  Host only; never fails. */
const char *tsd_status_string(tsd_status s);

/*
 * Bytes of workspace the operation `op` needs for these sizes (0 if the sizes
 * are out of range).  Host only.  n_modes, L, topk matter for
 * TSD_OP_BUILD_TREE; B matters for all three; V and dtype for all three.
 */
size_t tsd_workspace_size(tsd_op op, int n_trees, int n_modes, int L, int64_t V, int topk, int B,
                          tsd_dtype dtype);

/*
 * tsd_build_tree -- top-k drafter statistics and the best-first tree builder
 * ([CAST] Sec. 2 Eq. 1, App. C "Candidate construction"; mixture: [MFD]
 * Sec. 3.4 Eq. 2, Sec. 4.3, App. B "Merged heap", Prop. 6).
 *
 * drafter_logits  [n_trees][n_modes][L][V] (dtype): row (t, m, j) holds mode m's
 *                 logits for future position j+1 of tree t.  Scores use
 *                 log q = z/drafter_temp - logsumexp(z/drafter_temp) over the
 *                 full V, not renormalised over the top-k.
 * topk            tokens kept per (mode, position), ordered by (logit desc,
 *                 id asc); 1 <= topk <= min(V, TSD_MAX_TOPK), and
 *                 L * ceil(log2(topk)) <= 56.
 * V               1 <= V <= 8388608 for bf16, 4194304 for fp32.
 * B               non-root node budget, 0 <= B <= TSD_MAX_B.
 * drafter_temp    > 0.
 * Outputs, [n_trees][B+1] (node 0 = root: parent -1, token -1, depth 0,
 * score 0, rank -1, mode -1; slots >= n_nodes: -1 and score -inf):
 *   parent, token, depth   the tree in pop order (parent before child);
 *   score                  the node's best-mode score sum_j log q_{m,j}(y_j)
 *                          (float32 copy of the float64 key);
 *   rank, mode (nullable)  rank of the node's token in the creating mode's
 *                          list, and that mode.
 *   n_nodes [n_trees]      number of nodes including the root (<= B+1; fewer
 *                          when the universe has fewer finite-score prefixes).
 *   status  [n_trees]      TSD_OK or TSD_ERR_NONFINITE.
 * Ties are broken by (depth asc, mode asc, rank sequence lexicographic asc).
 * With n_modes = 1 this is DDTree's / CAST's builder.
 */
tsd_status tsd_build_tree(const void *drafter_logits, tsd_dtype dtype, int n_trees, int n_modes,
                          int L, int64_t V, int topk, int B, float drafter_temp,
                          int32_t *parent, int32_t *token, int32_t *depth, float *score,
                          int32_t *rank, int32_t *mode, int32_t *n_nodes, int32_t *status,
                          void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * tsd_tree_mask -- ancestor mask and position ids of the packed verification
 * input ([CAST] App. C "Packed verification"; App. B Lemma 1).
 *
 * parent [n_trees][B+1], n_nodes [n_trees]: trees as above.
 * prefix_len      P >= 0, the number of cached prefix tokens.
 * anc_bits        [n_trees][B+1][W] uint32, W = (B+32)/32: bit u of row v is
 *                 set iff node u is node v or one of its ancestors.
 * position_ids    [n_trees][B+1]: P + depth(v).
 * additive_mask   nullable [n_trees][B+1][mask_ld] float32, mask_ld >=
 *                 P+B+1: columns [0, P) are 0 (the prefix is visible);
 *                 column P+u is 0 if bit u of row v is set, else -inf.
 *                 Columns past P+B+1 are not written.
 * Rows v >= n_nodes are padding: only their own bit, position P.
 * status [n_trees]: TSD_OK or TSD_ERR_BAD_TREE.
 */
tsd_status tsd_tree_mask(const int32_t *parent, const int32_t *n_nodes, int n_trees, int B,
                         int prefix_len, uint32_t *anc_bits, int32_t *position_ids,
                         float *additive_mask, int64_t mask_ld, int32_t *status,
                         cudaStream_t stream);

/*
 * tsd_verify_tev -- Tree Exit Verification ([EXIT] App. B Algorithm 1).
 *
 * target_logits   [n_trees][B+1][V] (dtype); only rows v < n_nodes[t] are read.
 * parent, token   [n_trees][B+1]; n_nodes [n_trees].
 * temperature     T >= 0: p_v = softmax(z_v / T) ([EXIT] Eq. 1); T = 0 is
 *                 greedy: p_v one-hot at the arg-max (lowest id on ties).
 * seed            key of the uniforms (see the conventions above).
 * Per tree, with P(root) = 1, P(u) = P(pa u) p_pa(u)(x_u), rho(v) = mass of
 * the non-child tokens under p_v, w = P rho ([EXIT] Eq. 2, 4):
 *   exit_node [n_trees]    V ~ Categorical(w): inverse CDF over node index;
 *   bonus_token [n_trees]  Y ~ p_V restricted to tokens that are not drafted
 *                          children of V, renormalised ([EXIT] Eq. 7):
 *                          inverse CDF over token id;
 *   accept_len [n_trees]   depth(V) + 1 (accepted draft tokens + bonus).
 *   exit_mass, prefix_prob nullable [n_trees][B+1]: w and P (0 past n_nodes);
 *   coverage               nullable [n_trees]: C_p = sum_{u != root} P(u)
 *                          ([EXIT] Eq. 6);
 *   status [n_trees]       TSD_OK, TSD_ERR_BAD_TREE or TSD_ERR_NONFINITE; a
 *                          failed tree gets exit_node = bonus = -1,
 *                          accept_len = 0.
 * The accepted path is the parent chain of exit_node.
 * Two internal paths give the same results: launches with B <= 64 (and other
 * launches of at most 32768 row chunks with B <= 128), with 16-byte aligned
 * rows and V a multiple of 8 (bf16) or 4 (fp32), run as two kernels (a
 * streaming row kernel, then one block per tree); the rest run as the
 * batched chain of four kernels.
 */
tsd_status tsd_verify_tev(const void *target_logits, tsd_dtype dtype, const int32_t *parent,
                          const int32_t *token, const int32_t *n_nodes, int n_trees, int B,
                          int64_t V, float temperature, uint64_t seed, int32_t *exit_node,
                          int32_t *bonus_token, int32_t *accept_len, float *exit_mass,
                          float *prefix_prob, float *coverage, int32_t *status, void *workspace,
                          size_t ws_bytes, cudaStream_t stream);

/*
 * tsd_verify_tev_timed -- tsd_verify_tev that also records five caller-created
 * CUDA events on `stream` around its kernels, for measuring each stage with
 * cudaEventElapsedTime.  On the batched path: stage_events[0] before the tree
 * preparation, [1] before the node-row reduction (the node-local reductions
 * over the logits), [2] after it, [3] after the per-node combination, [4]
 * after the exit and bonus draws.  On the two-kernel path of small launches
 * (see tsd_verify_tev): [0] and [1] before the streaming row kernel, [2]
 * after it, [3] and [4] after the per-tree kernel.  Same arguments, outputs
 * and errors as tsd_verify_tev; TSD_ERR_INVALID_ARG if stage_events or one of
 * its five entries is null.
 */
tsd_status tsd_verify_tev_timed(const void *target_logits, tsd_dtype dtype, const int32_t *parent,
                                const int32_t *token, const int32_t *n_nodes, int n_trees, int B,
                                int64_t V, float temperature, uint64_t seed, int32_t *exit_node,
                                int32_t *bonus_token, int32_t *accept_len, float *exit_mass,
                                float *prefix_prob, float *coverage, int32_t *status,
                                void *workspace, size_t ws_bytes, cudaStream_t stream,
                                cudaEvent_t *stage_events);

/*
 * tsd_verify_ddtree -- predraw-and-follow ([EXIT] Sec. 2, App. A.4.1), the
 * verifier DDTree uses, kept as an equivalence check for TEV: it draws
 * R_v ~ p_v at every node (inverse CDF over token id, uniform stream 2 at
 * node v), walks from the root into the child whose token is R_v, and exits
 * at the first node without one, returning R_v as the bonus token.
 * Inputs as tsd_verify_tev.  Outputs: exit_node, bonus_token, accept_len
 * [n_trees]; draws nullable [n_trees][B+1] (R_v; -1 past n_nodes); status.
 * Small launches take the same two-kernel path as tsd_verify_tev (the same
 * streaming row kernel, then one block per tree drawing at every node).
 */
tsd_status tsd_verify_ddtree(const void *target_logits, tsd_dtype dtype, const int32_t *parent,
                             const int32_t *token, const int32_t *n_nodes, int n_trees, int B,
                             int64_t V, float temperature, uint64_t seed, int32_t *exit_node,
                             int32_t *bonus_token, int32_t *accept_len, int32_t *draws,
                             int32_t *status, void *workspace, size_t ws_bytes,
                             cudaStream_t stream);

/*
 * tsd_build_forest -- cost-aware tree widths under a budget shared by the
 * requests of one launch ([CAST] Sec. 3.3 Thm. 2, App. B.4 Prop. 2-3).  Each
 * request's candidate tree is built as tsd_build_tree builds it (one mode) at
 * the per-request cap B; the union of the candidates is ranked by prefix mass
 * exp(score) (ties toward shorter prefixes, then the lower request index,
 * then the request's own order), and with the affine round time
 * l(M) = l0 + c1 M the global node M+1 is added while
 *   mass_(M+1) >= c1 (G(M) + n_trees) / l(M),  G(M) = sum of the M largest,
 * up to M_max nodes in all.  Every request keeps the first width nodes of its
 * tree (a prefix-closed tree in pop order); n_nodes = width + 1.
 *
 * Inputs as tsd_build_tree with n_modes = 1, plus M_max >= 0, l0 > 0, c1 >= 0
 * (the round time's intercept and slope, in any one time unit).  The
 * candidates, n_trees * B, must not exceed 8192 (TSD_ERR_INVALID_ARG).
 * Outputs: parent, token, depth, score [n_trees][B+1] and n_nodes, status
 * [n_trees] as tsd_build_tree's (slots past n_nodes cleared); total [1]
 * int32: the selected node count M*.  Workspace:
 * tsd_workspace_size(TSD_OP_BUILD_FOREST, n_trees, 1, L, V, topk, B, dtype).
 */
#define TSD_MAX_FOREST_CANDIDATES 8192
tsd_status tsd_build_forest(const void *drafter_logits, tsd_dtype dtype, int n_trees, int L,
                            int64_t V, int topk, int B, float drafter_temp, int M_max, double l0,
                            double c1, int32_t *parent, int32_t *token, int32_t *depth,
                            float *score, int32_t *n_nodes, int32_t *status, int32_t *total,
                            void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * tsd_build_lse_tree -- the mixture tree under the log-sum-exp score ([MFD]
 * App. B "Max or log-sum-exp", Eq. 6): prefixes ranked by their mixture
 * probability s_lse(v) = log sum_m pi_m Q_m(v), Q_m(v) = prod_j q_{m,j}(v_j).
 * No merge of per-mode searches yields that ranking, so the candidates are
 * the distinct prefixes of the modes' per-depth lists.  Mode m's depth-d list
 * holds its B most probable length-d prefixes whose tokens are among its topk
 * kept tokens per position, ordered by (path sum of z/T desc, parent's place
 * in the depth-(d-1) list asc, token rank asc); zero-probability prefixes are
 * left out.  Every candidate is scored under every mode from the full rows
 * (log Q_m = path sum of z/T minus the summed row log-normalisers), also
 * where its tokens fall outside a mode's kept lists.  The ranking key is
 * s_lse clamped to its parent's key (equal in exact arithmetic), and the tree
 * takes the B best distinct candidates by (key desc, depth asc, mode asc,
 * place asc) in that order, which is prefix-closed.  A candidate reached by
 * several modes counts once, under its first (depth, mode, place).
 *
 * drafter_logits  [n_trees][n_modes][L][V] as tsd_build_tree's (device or
 *                 page-locked host memory).
 * log_prior       nullable [n_trees][n_modes] float32 log pi (finite or
 *                 -inf; need not be normalised); NULL = uniform 1/n_modes.
 * Sizes as tsd_build_tree's, and also B <= 2048, n_modes * B <= 4096,
 * n_trees <= 65535, and one mode's lists must fit in a block's shared memory:
 * 16 n_modes B + 40 B + 24 P + 2496 bytes <= 227 KB, P the power of two at or
 * above sum_{r < topk} floor(B / (r+1)) (the children that can be kept);
 * else TSD_ERR_INVALID_ARG.
 * Outputs: parent, token, depth [n_trees][B+1] int32 and score (the ranking
 * key, float32 copy of the float64 value), n_nodes, status [n_trees] as
 * tsd_build_tree's; n_cand (nullable) [n_trees]: distinct candidates with
 * non-zero mixture mass.  A tree with a non-finite row gets status
 * TSD_ERR_NONFINITE and n_nodes 0.  Workspace:
 * tsd_workspace_size(TSD_OP_BUILD_LSE, n_trees, n_modes, L, V, topk, B, dtype).
 */
tsd_status tsd_build_lse_tree(const void *drafter_logits, tsd_dtype dtype, int n_trees,
                              int n_modes, int L, int64_t V, int topk, int B, float drafter_temp,
                              const float *log_prior, int32_t *parent, int32_t *token,
                              int32_t *depth, float *score, int32_t *n_nodes, int32_t *status,
                              int32_t *n_cand, void *workspace, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * tsd_verify_seqres -- exact sequential residual verification ([EXIT] App.
 * A.4.2 Eq. 45-53), another exact verifier over the same row statistics as
 * TEV: from the root, the children of the current node are tested in
 * ascending token order; child j is followed when u (1 - M_{j-1}) < p_j
 * (Eq. 49; p_j = p_v(x_j), M the sum of the earlier p's; uniform stream 3,
 * sub-index j).  If every child is rejected the walk exits and the bonus
 * token is drawn from the residual of Eq. 53 (stream 4), as TEV draws its
 * own.  Arguments, workspace (tsd_workspace_size(TSD_OP_VERIFY_TEV, ...)) and
 * errors as tsd_verify_tev; outputs exit_node, bonus_token, accept_len,
 * status [n_trees].
 */
tsd_status tsd_verify_seqres(const void *target_logits, tsd_dtype dtype, const int32_t *parent,
                             const int32_t *token, const int32_t *n_nodes, int n_trees, int B,
                             int64_t V, float temperature, uint64_t seed, int32_t *exit_node,
                             int32_t *bonus_token, int32_t *accept_len, int32_t *status,
                             void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * tsd_verify_proposal -- proposal-aware verification ([CAST] App. B.1 Thm. 3,
 * recursive speculative sampling without replacement) at every visited
 * node: the residual mu starts at p_v; a candidate child c is drawn from the
 * proposal renormalised over the retained children, q~ (inverse CDF in
 * ascending token order, stream 5, sub-index = step), and followed when
 * u q~(c) < mu(c) (stream 6); a rejection sets mu <- (mu - q~)_+ normalised
 * and retires c.  With every child retired, the committed token is drawn
 * from mu (stream 7) and the walk exits.
 * q_child  [n_trees][B+1] fp32 (device): q_{pa(u)}(x_u), the proposal's
 *          probability of node u's token (entry 0 unused); it must be
 *          positive and finite on every child, else the tree's status is
 *          TSD_ERR_NONFINITE.  Other arguments as tsd_verify_seqres.
 */
tsd_status tsd_verify_proposal(const void *target_logits, tsd_dtype dtype, const int32_t *parent,
                               const int32_t *token, const int32_t *n_nodes, const float *q_child,
                               int n_trees, int B, int64_t V, float temperature, uint64_t seed,
                               int32_t *exit_node, int32_t *bonus_token, int32_t *accept_len,
                               int32_t *status, void *workspace, size_t ws_bytes,
                               cudaStream_t stream);

/*
 * tsd_exit_loss -- the exit-guided loss of ExitTrain ([EXIT] Sec. 5 Eq. 14),
 * evaluated as App. C.2 Eq. 67 does: one log-normaliser per drafter row,
 * weighted by the summed exit mass of the nodes the row scores, minus a
 * gather of those nodes' logits.  Node v's incoming token x_v is scored by
 * the drafter row of future position depth(v), i.e. row depth(v) - 1, with
 * log q = z/T_d - logsumexp(z/T_d).
 *   L_exit = sum over trees of sum_{v != root} w(v) (-log q_{depth(v)}(x_v))
 *            / sum over trees of (n_nodes - 1).
 *
 * drafter_logits  [n_trees][L][V] (dtype), one mode; device or page-locked
 *                 host memory.  L <= TSD_MAX_L.  drafter_temp: T_d > 0.
 * token, depth    [n_trees][B+1] int32: each node's token and depth (the
 *                 builder's outputs); node 0 is the root and is skipped.
 * n_nodes         [n_trees].
 * omega           [n_trees][B+1] fp32: the detached weights, normally the
 *                 exit masses w(v) that tsd_verify_tev returns.
 * Outputs (device): loss_tree [n_trees] float64, each tree's numerator;
 *   loss [1] float64, the scalar L_exit over the valid trees; grad
 *   (nullable) [n_trees][L][V] fp32, d L_exit / d drafter_logits (rows no
 *   node scores are zero); status [n_trees]: TSD_ERR_BAD_TREE for a depth
 *   outside [1, L] or a token outside [0, V), TSD_ERR_NONFINITE for a
 *   non-finite term; such trees count nowhere and get zero gradient.
 * workspace: tsd_workspace_size(TSD_OP_EXIT_LOSS, n_trees, 1, L, V, 1, B,
 *   dtype) bytes.
 */
tsd_status tsd_exit_loss(const void *drafter_logits, tsd_dtype dtype, int n_trees, int L,
                         int64_t V, float drafter_temp, const int32_t *token,
                         const int32_t *depth, const int32_t *n_nodes, int B,
                         const float *omega, double *loss_tree, double *loss, float *grad,
                         int32_t *status, void *workspace, size_t ws_bytes,
                         cudaStream_t stream);

/*
 * tsd_verify_tev_noalloc -- tsd_verify_tev for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is a deployment
 * variant, not a step of the method.
 *
 * Some callers own no device allocator -- a plug-in that an inference engine
 * hands only input and output pointers, or a decode loop that must not call
 * cudaMalloc because it can synchronise the device and stall queued work.
 * This entry point takes the same inputs and outputs as tsd_verify_tev and
 * computes the same results, but takes no workspace: its scratch is a static
 * device array of TSD_NOALLOC_SCRATCH_BYTES inside this library, which every
 * GPU that loads the library holds until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * - Sizes: returns TSD_ERR_WORKSPACE, before launching anything, when
 *   tsd_workspace_size(TSD_OP_VERIFY_TEV, n_trees, 1, 1, V, 1, B, dtype)
 *   exceeds TSD_NOALLOC_SCRATCH_BYTES (16 MiB: e.g. 64 trees of B = 256 at
 *   V = 151936 fit); other argument errors as tsd_verify_tev.
 * - Set-up: each call outside stream capture looks up the device address of
 *   the static array on the current device (which must own `stream` and the
 *   pointers) with cudaGetSymbolAddress and remembers it for that device; a
 *   call whose stream is being captured uses the remembered address instead.
 *   So make the first call on a device before any stream capture, and after
 *   a cudaDeviceReset (which reloads the library's device code and makes the
 *   remembered address stale) make the next call outside a capture.
 *   TSD_ERR_CUDA if the look-up fails, or if a call under capture finds no
 *   remembered address.
 * - Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents; nothing in it needs to start at zero.  Calls that overlap
 *   on the GPU (on different streams, or from several host threads without
 *   ordering) race on the array and give wrong results: serialise them.
 */
#define TSD_NOALLOC_SCRATCH_BYTES (16u << 20)
tsd_status tsd_verify_tev_noalloc(const void *target_logits, tsd_dtype dtype,
                                  const int32_t *parent, const int32_t *token,
                                  const int32_t *n_nodes, int n_trees, int B, int64_t V,
                                  float temperature, uint64_t seed, int32_t *exit_node,
                                  int32_t *bonus_token, int32_t *accept_len, float *exit_mass,
                                  float *prefix_prob, float *coverage, int32_t *status,
                                  cudaStream_t stream);

/*
 * tsd_debug_check_failures -- the bounds checks of a checked build.  A
 * debugging aid with no counterpart on the pages.
 *
 * A library compiled with -DTSD_CHECKS (the package's checked build,
 * libtsd_checks.so) tests every index that a kernel takes from memory before
 * using it: parents, CSR child offsets and child ids, tokens used as columns,
 * node ids, list, chunk and candidate positions.  A failing check sets one bit
 * per site class and skips the access; no kernel traps.  This call
 * synchronises the current device, returns the OR of the bits set since the
 * previous call (0 when every check passed) and clears them.  Bit i is site
 * class i: 0 work item of the row pass, 1 CSR child list, 2 verify
 * preparation, 3 ancestor walk, 4 exit node / chunk / bonus, 5 walk verifiers,
 * 6 predraw-and-follow, 7 builder, 8 tree mask, 9 drafter statistics,
 * 10 log-sum-exp tree, 11 shared-budget selection, 12 exit loss.
 * In the default build the checks are compiled out and the call returns 0
 * without touching the device.
 */
unsigned tsd_debug_check_failures(void);

#ifdef __cplusplus
}
#endif

#endif /* TSD_H */
