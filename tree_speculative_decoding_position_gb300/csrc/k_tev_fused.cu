// k_tev_fused.cu -- Tree Exit Verification in two kernels, for launches of
// at most a few waves of row chunks.
//
// "Where Draft Trees Lose Target Mass: Exit-Guided Speculative Decoding":
// the node-row reduction (Sec. 3 Eq. 1, Sec. 3.1 Eq. 4), prefix and exit
// masses (Eq. 2, Eq. 4) and target coverage (Eq. 6), the exit draw from the
// canonical exit law (Sec. 3.1 Lemma 1) and the bonus draw from the residual
// law of the exit node (Eq. 7) -- the same outputs as the four-kernel chain of
// k_rows.cu and k_tree.cu (tree preparation, row reduction, per-node
// combination, per-tree draws).  Small launches are bound by latency: each
// kernel of the chain waits for the previous one to drain.  Here there are
// two:
//
//   tev_stream_kernel  one warp per (node row, 8 KB chunk), as the batched row
//                      kernel, but each chunk finds its row's drafted children
//                      by a warp scan of the tree's parent array (no prepared
//                      child lists), and the lane holding a child's token
//                      copies that child's logit out (so that no later step
//                      gathers from the rows again).
//   tev_finish_kernel  one block per tree, launched early (programmatic
//                      dependent launch) and released when the streaming
//                      kernel completes: validates the tree, combines each
//                      row's chunk statistics (a warp per row), forms the edge
//                      probabilities, prefix masses, exit masses and coverage,
//                      and draws the exit node and the bonus token.
//
// Measured alternative that was not kept: one kernel whose warps count
// completed chunks and rows with atomics (the warp completing a tree finishes
// it).  Each release or acquire it needs is a memory barrier that waits for
// the warp's outstanding accesses (about 1-2 us on this GPU), paid once per
// chunk in the streaming loop and several times along the finishing chain;
// it was slower than the four-kernel chain at every size.
#include "chunk_reduce.cuh"

namespace tsd {

constexpr int kStreamThreads = 256;
constexpr int kFinishThreads = 512;
static_assert(kFusedMaxB + 1 <= kFinishThreads, "the finish kernel gives each node a thread");

// Rows of tree t the streaming kernel reads: n_nodes when it is valid, else
// the root alone (the finish kernel reports the tree as malformed).
__device__ __forceinline__ int fused_rows(int n, int B) { return (n >= 1 && n <= B + 1) ? n : 1; }

// Chunk statistics a lane holds in the row combine: chunks lane + 32 k.
constexpr int kFusedStatsPerLane = 4;  // rows of at most 128 chunks

// Marks, in the lanes' child masks, the drafted children of node v whose
// tokens fall in [c0, c0 + cn): a warp scan of the tree's parent array
// (par, tok: the tree's arrays, n live nodes).  kids: some child falls in
// the chunk; dup: two children of v carry the same token (a malformed tree).
// Both are the same in every lane.  With zdst non-null, the lane that holds
// each such child's token also copies its logit, read from the chunk at rp
// (an L2 hit: its lines are being fetched), to zdst[child].
template <typename T>
__device__ __forceinline__ void mark_tree_children(const int32_t* __restrict__ par,
                                                   const int32_t* __restrict__ tok, int n, int v,
                                                   int64_t c0, int cn, int lane, ExclMask<T>& excl,
                                                   bool& kids, bool& dup, const T* __restrict__ rp,
                                                   float* __restrict__ zdst) {
    constexpr int VEC = Lanes<T>::kVec;
#pragma unroll
    for (int w = 0; w < ExclMask<T>::kWords; ++w) excl.w[w] = 0u;
    unsigned any = 0u;
    bool again = false;
    for (int u0 = 1; u0 < n; u0 += kWarp) {
        const int u = u0 + lane;
        bool hit = false;
        int o = 0;
        if (u < n) {
            const int p = par[u];
            const int64_t x = tok[u];
            hit = p == v && x >= c0 && x < c0 + cn;
            o = (int)(x - c0);
        }
        unsigned m = __ballot_sync(0xffffffffu, hit);
        any |= m;
        while (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1;
            const int oj = __shfl_sync(0xffffffffu, o, j);
            again |= excl_mark<T>(excl, oj, lane);
            if (zdst != nullptr && ((oj / VEC) & (kWarp - 1)) == lane)
                zdst[u0 + j] = load_logit(rp + oj);
        }
    }
    kids = any != 0u;
    dup = __any_sync(0xffffffffu, again);
}

// One warp per (node row, 8 KB chunk), persistent over a grid stride: the
// next live chunk's loads are issued before the current chunk's warp
// reductions.  Only 16-byte aligned rows with V a multiple of the vector
// width come here.  A chunk in which two children of its row share a token
// is marked in its statistics: amax = -2 at T > 0, r = 1 at T = 0 (both
// fields are otherwise -1 and 0).
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kStreamThreads, 2)
tev_stream_kernel(const T* __restrict__ logits, int n_trees, int B, int64_t V, int nch, float c,
                  const int32_t* __restrict__ parent, const int32_t* __restrict__ token,
                  const int32_t* __restrict__ n_nodes, VerifyWs ws, bool capture) {
    pdl_entry_early();  // the per-tree finish blocks become resident now
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    const int lane = threadIdx.x & (kWarp - 1);
    const int wpb = blockDim.x / kWarp;
    const int R = B + 1;
    const int64_t total = (int64_t)n_trees * R * nch;
    ItemStep step;
    step.stride = (int64_t)gridDim.x * wpb;
    {
        const ItemPos d = item_pos(step.stride, R, nch);
        step.dt = d.t;
        step.dv = d.v;
        step.dch = d.ch;
    }
    ItemPos p = item_pos((int64_t)blockIdx.x * wpb + threadIdx.x / kWarp, R, nch);
    auto live = [&](const ItemPos& q) {
        return TSD_IN(q.t, n_trees, kChkRowsItem) && TSD_IN(q.ch, nch, kChkRowsItem) &&
               q.v < fused_rows(__ldg(n_nodes + q.t), B);
    };
    auto chunk_ptr = [&](const ItemPos& q, int64_t& c0, int& cn) {
        c0 = (int64_t)q.ch * CE;
        cn = (int)min((int64_t)CE, V - c0);
        return logits + ((int64_t)q.t * R + q.v) * V + c0;
    };
    while (p.item < total && !live(p)) item_advance(p, step, R, nch);
    if (p.item >= total) return;
    uint4 buf[kVecPerLane];
    int64_t c0;
    int cn;
    const T* rp = chunk_ptr(p, c0, cn);
    load_chunk<T>(buf, rp, cn, lane);
    for (;;) {
        const int t = p.t, v = p.v;
        ExclMask<T> excl;
        bool kids, dup;
        // TEV at T > 0 (capture): the children's logits go to ws.pedge,
        // where the finish kernel turns them into edge probabilities
        mark_tree_children<T>(parent + (int64_t)t * R, token + (int64_t)t * R,
                              fused_rows(__ldg(n_nodes + t), B), v, c0, cn, lane, excl, kids, dup,
                              rp, (GREEDY || !capture) ? nullptr : ws.pedge + (int64_t)t * R);
        const LanePart lp = chunk_lane_marked<T, GREEDY>(buf, cn, c, excl, kids, c0, lane);
        const int64_t done = p.item;
        do {
            item_advance(p, step, R, nch);
        } while (p.item < total && !live(p));
        if (p.item < total) {
            rp = chunk_ptr(p, c0, cn);
            load_chunk<T>(buf, rp, cn, lane);
        }
        ChunkStat st = chunk_finish<GREEDY>(lp);
        if (dup) {
            if (GREEDY) st.r = 1.0f;
            else st.amax = -2;
        }
        if (lane == 0) ws.chunk[done] = st;
        if (p.item >= total) break;
    }
}

// Exclusive prefix sum of one float per thread across the block; *total gets
// the block sum.  red: shared scratch of 33 floats.
static __device__ float fused_block_scan(float x, float* red, float* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const float inc = warp_incl_scan(x, lane);
    if (lane == 31) red[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        const float y = lane < nw ? red[lane] : 0.0f;
        const float yi = warp_incl_scan(y, lane);
        red[lane] = yi - y;  // exclusive over warps
        if (lane == 31) red[32] = yi;
    }
    __syncthreads();
    const float r = red[wid] + inc - x;
    *total = red[32];
    __syncthreads();
    return r;
}

// Shared memory of the finish kernel for a tree of R = B+1 nodes and rows of
// nch chunks: per node the parent (16-bit), token, the child's logit (then its
// edge probability), P, w, and the row's reference, sum and residual sum (or
// arg-max); per (row, chunk) the chunk's maximum and residual sum (T > 0), to
// locate the bonus draw's chunk without another round of loads.
__host__ __device__ inline size_t fused_finish_smem(int B, int nch, bool greedy) {
    const size_t R = (size_t)B + 1;
    return R * 32 + 16 + (greedy ? 0 : R * (size_t)nch * 8);
}

// Shared memory layout of a finish block (pointers into the dynamic array).
struct FinishSmem {
    float* Mc;    // [R] row reference mc (T = 0: arg-max bits)
    float* Sv;    // [R] row sum S
    float* Rv;    // [R] row residual sum (T = 0: rho)
    float* Dv;    // [R] the child's logit, then p_pa(u)(x_u)
    float* Pv;    // [R] P
    float* Wv;    // [R] w (predraw: the draws)
    int32_t* tk;  // [R] tokens
    int16_t* pa;  // [R] parents
    float2* cm;   // [R][nch] (chunk maximum, chunk residual sum; predraw: chunk sum)
};
__device__ __forceinline__ FinishSmem finish_smem_layout(void* base, int R) {
    FinishSmem f;
    f.Mc = reinterpret_cast<float*>(base);
    f.Sv = f.Mc + R;
    f.Rv = f.Sv + R;
    f.Dv = f.Rv + R;
    f.Pv = f.Dv + R;
    f.Wv = f.Pv + R;
    f.tk = reinterpret_cast<int32_t*>(f.Wv + R);
    f.pa = reinterpret_cast<int16_t*>(f.tk + R);
    f.cm = reinterpret_cast<float2*>(base) + ((size_t)R * 32 + 16) / 8;
    return f;
}

// One row's statistics from its chunk statistics xs[0..KL) (chunks lane +
// 32 k), by a warp: the maximum and the sums relative to the row's reference
// (or the arg-max at T = 0) into shared memory, each chunk's maximum and
// residual sum (PRED: its sum) beside them; flags gets bit 0 for a repeated
// child token, bit 1 for a row without mass.
template <bool GREEDY, bool PRED, int KL>
__device__ __forceinline__ void finish_row(int v, const ChunkStat (&xs)[KL], int nch, float c,
                                           const FinishSmem& f, int* flags, int lane) {
    bool bad = false, dup = false;
    if (GREEDY) {
        float bm = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int k = 0; k < KL; ++k) {
            bad |= (xs[k].s != xs[k].s);
            dup |= (xs[k].r != 0.0f);
            if (better(xs[k].m, xs[k].amax, bm, bi)) {
                bm = xs[k].m;
                bi = xs[k].amax;
            }
        }
        warp_argmax(bm, bi);
        bad |= (bm == -INFINITY);  // every token masked: no arg-max
        if (lane == 0) {
            f.Mc[v] = __int_as_float(bi);
            f.Rv[v] = 1.0f;
        }
    } else {
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < KL; ++k) m = fmaxf(m, xs[k].m);
        m = warp_max(m);
        const float mc = __fmul_rn(m, c);
        float sm = 0.0f, r = 0.0f;
#pragma unroll
        for (int k = 0; k < KL; ++k) {
            bad |= (xs[k].s != xs[k].s);
            dup |= (xs[k].amax == -2);
            if (xs[k].m != -INFINITY) {
                const float e = ex2(__fmul_rn(xs[k].m, c) - mc);
                sm += xs[k].s * e;
                r += xs[k].r * e;
            }
            const int q = lane + k * kWarp;
            if (q < nch) f.cm[(size_t)v * nch + q] = make_float2(xs[k].m, PRED ? xs[k].s : xs[k].r);
        }
        sm = warp_sum(sm);
        r = warp_sum(r);
        bad = bad || m == -INFINITY || !(sm > 0.0f);
        if (lane == 0) {
            f.Mc[v] = mc;
            f.Sv[v] = sm;
            f.Rv[v] = r;
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    dup = __any_sync(0xffffffffu, dup);
    if (lane == 0 && (bad || dup)) atomicOr(flags, (dup ? 1 : 0) | (bad ? 2 : 0));
}

// Phase 1 of a finish block: every load is issued at once, before the tree's
// size is known -- the size, each node's parent, token and (T > 0, TEV)
// logit, and the chunk statistics of the rows up to B+1 (slots past n_nodes
// are in bounds and their values are never used) -- G rows per warp and
// round, rows strided over the warps.  Then the rows below n_nodes are
// reduced (finish_row) and the tree is validated; flags gets bit 0 for a
// malformed tree, bit 1 for a row without mass.  Returns the number of live
// nodes; ends with a block barrier.
template <typename T, bool GREEDY, bool PRED, int G, int KL>
__device__ __forceinline__ int finish_stage_g(int t, int B, int64_t V, int nch, float c,
                                              const int32_t* __restrict__ parent,
                                              const int32_t* __restrict__ token,
                                              const int32_t* __restrict__ n_nodes,
                                              const VerifyWs& ws, const FinishSmem& f, int* flags) {
    const int R = B + 1;
    const int lane = threadIdx.x & (kWarp - 1), wid = threadIdx.x / kWarp;
    const int nw = blockDim.x / kWarp;
    const int u = threadIdx.x;  // R <= kFinishThreads
    const int n_raw = n_nodes[t];
    int p = -1, x = 0;
    float z = 0.0f;
    if (u < R) {
        p = parent[(int64_t)t * R + u];
        x = token[(int64_t)t * R + u];
        if (!GREEDY && !PRED && u > 0) z = ws.pedge[(int64_t)t * R + u];
    }
    ChunkStat xs[G][KL];
    auto load_round = [&](int g0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int v = g0 + wid + nw * g;
#pragma unroll
            for (int k = 0; k < KL; ++k) {
                const int q = lane + k * kWarp;
                if (v < R && q < nch) {
                    xs[g][k] = ws.chunk[((int64_t)t * R + v) * nch + q];
                } else {
                    xs[g][k].m = -INFINITY;
                    xs[g][k].s = 0.0f;
                    xs[g][k].r = 0.0f;
                    xs[g][k].amax = GREEDY ? INT_MAX : -1;
                }
            }
        }
    };
    load_round(0);
    if (threadIdx.x == 0) *flags = 0;
    __syncthreads();
    const bool n_ok = n_raw >= 1 && n_raw <= R;
    const int n = n_ok ? n_raw : 1;
    if (threadIdx.x == 0 && !n_ok) atomicOr(flags, 1);
    if (u < n) {
        bool bad;
        if (u == 0) bad = p != -1;
        else bad = p < 0 || p >= u || x < 0 || (int64_t)x >= V;
        if (bad) atomicOr(flags, 1);
        f.pa[u] = (int16_t)(u == 0 ? -1 : (p >= 0 && p < u ? p : 0));
        f.tk[u] = x;
        f.Dv[u] = z;
    }
    for (int g0 = 0;;) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int v = g0 + wid + nw * g;
            if (v < n) finish_row<GREEDY, PRED, KL>(v, xs[g], nch, c, f, flags, lane);
        }
        g0 += nw * G;
        if (g0 >= n) break;
        load_round(g0);
    }
    __syncthreads();
    return n;
}

template <typename T, bool GREEDY, bool PRED>
__device__ __forceinline__ int finish_stage(int t, int B, int64_t V, int nch, float c,
                                            const int32_t* __restrict__ parent,
                                            const int32_t* __restrict__ token,
                                            const int32_t* __restrict__ n_nodes,
                                            const VerifyWs& ws, const FinishSmem& f, int* flags) {
    if (nch <= 2 * kWarp)  // five rows of up to 64 chunks per warp and round
        return finish_stage_g<T, GREEDY, PRED, 5, 2>(t, B, V, nch, c, parent, token, n_nodes, ws,
                                                     f, flags);
    return finish_stage_g<T, GREEDY, PRED, 2, kFusedStatsPerLane>(t, B, V, nch, c, parent, token,
                                                                  n_nodes, ws, f, flags);
}

// One block per tree, in two phases.
//  1. Every load at once: thread u reads node u's parent, token and (T > 0)
//     logit; each warp reads the chunk statistics of its rows, G rows at a
//     time, and reduces each row (its maximum and sums relative to the row's
//     reference, or its arg-max at T = 0) into shared memory.
//  2. From shared memory, by the whole block: validation; p_pa(u)(x_u) from
//     the parent row's statistics and the child's logit (Eq. 1); rho (Eq. 4,
//     the residual sum over the row sum); P along the root path (Eq. 2);
//     w = P rho (Eq. 4); C_p (Eq. 6); the exit draw by inverse CDF over node
//     index; the bonus draw by inverse CDF over the exit row's residual
//     (Eq. 7): the chunk from the staged chunk sums, then that chunk alone is
//     read again, one 16-byte vector per thread.  (Done by one warp instead,
//     this phase took longer: a lone warp's chain of dependent steps cannot
//     hide its own latencies.)
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kFinishThreads)
tev_finish_kernel(const T* __restrict__ logits, int B, int64_t V, int nch, float c, uint64_t seed,
                  const int32_t* __restrict__ parent, const int32_t* __restrict__ token,
                  const int32_t* __restrict__ n_nodes, VerifyWs ws, int32_t* __restrict__ exit_node,
                  int32_t* __restrict__ bonus, int32_t* __restrict__ accept_len,
                  float* __restrict__ exit_mass, float* __restrict__ prefix_prob,
                  float* __restrict__ coverage, int32_t* __restrict__ status) {
    pdl_entry();
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    constexpr int VEC = Lanes<T>::kVec;
    extern __shared__ float4 finish_smem[];
    __shared__ int flags;  // bit 0: malformed tree, bit 1: a row without mass
    const int t = blockIdx.x;
    const int R = B + 1;
    const int lane = threadIdx.x & (kWarp - 1), wid = threadIdx.x / kWarp;
    const FinishSmem f = finish_smem_layout(finish_smem, R);
    float* Mc = f.Mc;
    float* Sv = f.Sv;
    float* Rv = f.Rv;
    float* Dv = f.Dv;
    float* Wv = f.Wv;
    int32_t* tk = f.tk;
    int16_t* pa = f.pa;
    const float2* cmr = f.cm;
    const int n = finish_stage<T, GREEDY, false>(t, B, V, nch, c, parent, token, n_nodes, ws, f,
                                                 &flags);
    // ---- phase 2: from shared memory, the whole block ----------------------
    const int fl = flags;
    const int st = (fl & 1) ? kStatBadTree : ((fl & 2) ? kStatNonFinite : kStatOk);
    if (st != kStatOk) {
        for (int u = threadIdx.x; u < R; u += blockDim.x) {
            if (exit_mass) exit_mass[(int64_t)t * R + u] = 0.0f;
            if (prefix_prob) prefix_prob[(int64_t)t * R + u] = 0.0f;
        }
        if (threadIdx.x == 0) {
            exit_node[t] = -1;
            bonus[t] = -1;
            accept_len[t] = 0;
            if (coverage) coverage[t] = 0.0f;
            status[t] = st;
        }
        return;
    }
    // edge probabilities from the parent row; at T = 0 a child holding its
    // parent's arg-max takes the edge and leaves rho(parent) = 0
    for (int u = 1 + threadIdx.x; u < n; u += blockDim.x) {
        const int p = pa[u];
        if (GREEDY) {
            const bool h = tk[u] == __float_as_int(Mc[p]);
            Dv[u] = h ? 1.0f : 0.0f;
            if (h) Rv[p] = 0.0f;
        } else {
            Dv[u] = ex2(fmaf(Dv[u], c, -Mc[p])) * (1.0f / Sv[p]);
        }
    }
    __syncthreads();
    // P(u): the product of the edge probabilities on the root path, every
    // node walking its own ancestors (parents precede children, so a walk
    // ends within u steps)
    for (int u = threadIdx.x; u < R; u += blockDim.x) {
        float P = 0.0f, wu = 0.0f;
        if (u < n) {
            P = 1.0f;
            for (int x = u; x > 0; x = pa[x]) P *= Dv[x];
            wu = GREEDY ? P * Rv[u] : P * (Rv[u] / Sv[u]);
            f.Pv[u] = P;
            Wv[u] = wu;
        }
        if (exit_mass) exit_mass[(int64_t)t * R + u] = wu;
        if (prefix_prob) prefix_prob[(int64_t)t * R + u] = P;
    }
    __shared__ float red[33];
    __shared__ int pick[2];
    __shared__ int exit_v, chunk_sel, n_kids;
    __shared__ float chunk_frac, cov_sh;
    __syncthreads();
    // C_p and the exit draw by warp 0: inverse CDF over nodes, lane l owning a
    // contiguous run of them
    if (wid == 0) {
        const int per = (n + kWarp - 1) / kWarp;
        const int nb = lane * per, ne = min(n, nb + per);
        float mine = 0.0f, pc = 0.0f;
        for (int v = nb; v < ne; ++v) {
            mine += Wv[v];
            if (v > 0) pc += f.Pv[v];
        }
        const float cov_all = warp_sum(pc);
        const float incl = warp_incl_scan(mine, lane);
        const float wsum = __shfl_sync(0xffffffffu, incl, 31);
        const float thr = uniform24(seed, t, 0, 0) * wsum;
        float run = incl - mine;
        int first = INT_MAX, last = -1;
        for (int v = nb; v < ne; ++v) {
            run += Wv[v];
            if (Wv[v] > 0.0f) {
                last = v;
                if (first == INT_MAX && run > thr) first = v;
            }
        }
        first = __reduce_min_sync(0xffffffffu, first);
        last = __reduce_max_sync(0xffffffffu, last);
        if (lane == 0) {
            exit_v = first != INT_MAX ? first : (last >= 0 ? last : 0);
            cov_sh = cov_all;
        }
    }
    __syncthreads();
    const float cov = cov_sh;
    const int V_ = exit_v;
    int y = -1;
    if (GREEDY) {
        y = __float_as_int(Mc[V_]);  // the arg-max, which is not a child of V_
    } else {
        int* kid_off = reinterpret_cast<int*>(Wv);  // w is no longer needed
        // warp 0: the chunk where the running residual first exceeds u * R_V
        // (the staged chunk sums, relative to the row's reference), then the
        // offsets in that chunk of the exit node's children
        if (wid == 0) {
            const float2* cq = cmr + (size_t)V_ * nch;
            const float mcr = Mc[V_];
            const float thr2 = uniform24(seed, t, 0, 1) * Rv[V_];
            float base = 0.0f, frac = 0.0f;
            int sel = -1, lastc = -1;
            for (int q0 = 0; q0 < nch && sel < 0; q0 += kWarp) {
                const int q = q0 + lane;
                float rq = 0.0f;
                if (q < nch) {
                    const float2 x = cq[q];
                    if (x.x != -INFINITY) rq = x.y * ex2(__fmul_rn(x.x, c) - mcr);
                }
                const float inc = warp_incl_scan(rq, lane) + base;
                const unsigned hit = __ballot_sync(0xffffffffu, inc > thr2 && rq > 0.0f);
                const unsigned pos = __ballot_sync(0xffffffffu, rq > 0.0f);
                if (pos) lastc = q0 + 31 - __clz(pos);
                if (hit) {
                    const int l = __ffs(hit) - 1;
                    sel = q0 + l;
                    const float incl = __shfl_sync(0xffffffffu, inc, l);
                    const float own = __shfl_sync(0xffffffffu, rq, l);
                    frac = (thr2 - (incl - own)) / own;
                }
                base = __shfl_sync(0xffffffffu, inc, 31);
            }
            if (sel < 0) {  // rounding left the threshold past the last chunk
                sel = lastc;
                frac = 1.0f;
            }
            int cnt = 0;
            if (sel >= 0) {
                const int64_t c0 = (int64_t)sel * CE, c1 = c0 + CE;
                for (int x0 = 1; x0 < n; x0 += kWarp) {
                    const int x = x0 + lane;
                    const bool hit = x < n && pa[x] == V_ && tk[x] >= c0 && tk[x] < c1;
                    const unsigned m = __ballot_sync(0xffffffffu, hit);
                    if (hit) kid_off[cnt + __popc(m & ((1u << lane) - 1u))] = (int)(tk[x] - c0);
                    cnt += __popc(m);
                }
            }
            if (lane == 0) {
                chunk_sel = sel;
                chunk_frac = fminf(fmaxf(frac, 0.0f), 0.99999994f);
                n_kids = cnt;
            }
        }
        __syncthreads();
        const int q = chunk_sel;
        if (q >= 0 && TSD_IN(q, nch, kChkExitNode)) {
            const int64_t c0 = (int64_t)q * CE;
            const int cn = (int)min((int64_t)CE, V - c0);
            // one 16-byte vector per thread: thread i holds tokens i*VEC ..
            // i*VEC + VEC - 1 of the chunk (a chunk is kFinishThreads vectors)
            const int i0 = threadIdx.x * VEC;
            uint4 vq = Lanes<T>::neg_inf();
            if (i0 < cn) vq = ld_stream16(logits + ((int64_t)t * R + V_) * V + c0 + i0);
            unsigned skip = 0u;  // this thread's elements that are children of V_
            for (int j = 0; j < n_kids; ++j) {
                const int o = kid_off[j] - i0;
                if (o >= 0 && o < VEC) skip |= 1u << o;
            }
            const float mcq = __fmul_rn(cmr[(size_t)V_ * nch + q].x, c);
            float e[VEC];
            float sum = 0.0f;
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                e[j] = ((skip >> j) & 1u) ? 0.0f : ex2(fmaf(Lanes<T>::get(vq, j), c, -mcq));
                sum += e[j];
            }
            float tot;
            const float before = fused_block_scan(sum, red, &tot);
            const float target = chunk_frac * tot;
            if (threadIdx.x == 0) {
                pick[0] = INT_MAX;
                pick[1] = -1;
            }
            __syncthreads();
            float r2 = before;
            int lastp = -1;
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                r2 += e[j];
                if (e[j] > 0.0f) lastp = i0 + j;
                if (r2 > target && e[j] > 0.0f) {
                    atomicMin(pick, i0 + j);
                    break;
                }
            }
            if (lastp >= 0) atomicMax(pick + 1, lastp);
            __syncthreads();
            const int o = pick[0] != INT_MAX ? pick[0] : pick[1];
            y = o >= 0 ? (int)(c0 + o) : -1;
        }
    }
    if (threadIdx.x == 0) {
        int d = 0;
        for (int x = V_; x > 0; x = pa[x]) ++d;
        exit_node[t] = V_;
        bonus[t] = y;
        accept_len[t] = d + 1;
        if (coverage) coverage[t] = cov;
        status[t] = y >= 0 ? kStatOk : kStatNonFinite;
    }
}

// Predraw-and-follow on the small-launch path ([EXIT] Sec. 2 and App. A.4.1),
// kept as the equivalence check of TEV.  After the same streaming kernel:
//   predraw_nodes_fused_kernel  a warp per node: the row's maximum and sum
//                               from its chunk statistics, then R_v ~ p_v by
//                               inverse CDF over token id (the chunk from the
//                               chunk sums, then that chunk read again; at
//                               T = 0 the arg-max).  ws.draws[v] gets R_v, or
//                               -1 for a row without mass, -2 for a row with
//                               a repeated child token.
//   predraw_walk_fused_kernel   a block per tree: validation, then warp 0
//                               follows the draws from the root into the child
//                               whose token is R_v; the first node without one
//                               is the exit and R_v its bonus token.
// (The draws run over the whole GPU, a warp per node, as in the batched chain:
// drawn inside one block per tree they took longer than the rest of the
// verifier, each warp re-reading several chunks one after another.)
constexpr int kDrawFusedThreads = 256;

template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kDrawFusedThreads)
predraw_nodes_fused_kernel(const T* __restrict__ logits, int n_trees, int B, int64_t V, int nch,
                           float c, uint64_t seed, const int32_t* __restrict__ n_nodes,
                           VerifyWs ws) {
    pdl_entry();
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    constexpr int VEC = Lanes<T>::kVec;
    const int lane = threadIdx.x & (kWarp - 1);
    const int wpb = blockDim.x / kWarp;
    const int R = B + 1;
    const int64_t rows = (int64_t)n_trees * R;
    for (int64_t row = (int64_t)blockIdx.x * wpb + threadIdx.x / kWarp; row < rows;
         row += (int64_t)gridDim.x * wpb) {
        const int t = (int)(row / R);
        const int v = (int)(row - (int64_t)t * R);
        if (v >= fused_rows(__ldg(n_nodes + t), B)) continue;
        const ChunkStat* cs = ws.chunk + row * nch;
        ChunkStat x[kFusedStatsPerLane];
#pragma unroll
        for (int k = 0; k < kFusedStatsPerLane; ++k) {
            const int q = lane + k * kWarp;
            if (q < nch) {
                x[k] = cs[q];
            } else {
                x[k].m = -INFINITY;
                x[k].s = 0.0f;
                x[k].r = 0.0f;
                x[k].amax = GREEDY ? INT_MAX : -1;
            }
        }
        bool bad = false, dup = false;
        int r = -1;
        if (GREEDY) {
            float bm = -INFINITY;
            int bi = INT_MAX;
#pragma unroll
            for (int k = 0; k < kFusedStatsPerLane; ++k) {
                bad |= (x[k].s != x[k].s);
                dup |= (x[k].r != 0.0f);
                if (better(x[k].m, x[k].amax, bm, bi)) {
                    bm = x[k].m;
                    bi = x[k].amax;
                }
            }
            warp_argmax(bm, bi);
            bad = __any_sync(0xffffffffu, bad) || bm == -INFINITY;
            r = bi;
        } else {
            float m = -INFINITY;
#pragma unroll
            for (int k = 0; k < kFusedStatsPerLane; ++k) m = fmaxf(m, x[k].m);
            m = warp_max(m);
            const float mc = __fmul_rn(m, c);
            float sum = 0.0f;
#pragma unroll
            for (int k = 0; k < kFusedStatsPerLane; ++k) {
                bad |= (x[k].s != x[k].s);
                dup |= (x[k].amax == -2);
                if (x[k].m != -INFINITY) sum += x[k].s * ex2(__fmul_rn(x[k].m, c) - mc);
            }
            sum = warp_sum(sum);
            bad = __any_sync(0xffffffffu, bad) || m == -INFINITY || !(sum > 0.0f);
            if (!bad) {
                // the chunk where the running sum first exceeds u * S
                const float thr = uniform24(seed, t, v, 2) * sum;
                float base = 0.0f, frac = 1.0f;
                int sel = -1, lastc = -1;
                for (int q0 = 0; q0 < nch && sel < 0; q0 += kWarp) {
                    const int q = q0 + lane;
                    float sq = 0.0f;
                    if (q < nch) {
                        const ChunkStat y = cs[q];
                        if (y.m != -INFINITY) sq = y.s * ex2(__fmul_rn(y.m, c) - mc);
                    }
                    const float inc = warp_incl_scan(sq, lane) + base;
                    const unsigned hit = __ballot_sync(0xffffffffu, inc > thr && sq > 0.0f);
                    const unsigned pos = __ballot_sync(0xffffffffu, sq > 0.0f);
                    if (pos) lastc = q0 + 31 - __clz(pos);
                    if (hit) {
                        const int l = __ffs(hit) - 1;
                        sel = q0 + l;
                        const float incl = __shfl_sync(0xffffffffu, inc, l);
                        const float own = __shfl_sync(0xffffffffu, sq, l);
                        frac = (thr - (incl - own)) / own;
                    }
                    base = __shfl_sync(0xffffffffu, inc, 31);
                }
                if (sel < 0) sel = lastc;
                frac = fminf(fmaxf(frac, 0.0f), 0.99999994f);
                if (sel >= 0 && TSD_IN(sel, nch, kChkPredraw)) {
                    // vector i of lane l holds tokens (i*32 + l)*VEC .. +VEC,
                    // so (i, lane, element) is token order
                    const int64_t c0 = (int64_t)sel * CE;
                    const int cn = (int)min((int64_t)CE, V - c0);
                    const float mcq = __fmul_rn(cs[sel].m, c);
                    uint4 buf[kVecPerLane];
                    load_chunk<T>(buf, logits + row * V + c0, cn, lane);
                    float vs[kVecPerLane], lsum = 0.0f;
#pragma unroll
                    for (int i = 0; i < kVecPerLane; ++i) {
                        float a = 0.0f;
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            a += ex2(fmaf(Lanes<T>::get(buf[i], j), c, -mcq));
                        vs[i] = a;
                        lsum += a;
                    }
                    const float target = frac * warp_sum(lsum);
                    float run0 = 0.0f;
                    int found = -1, last_i = -1, last_l = -1;
                    bool done = false;  // warp-uniform
#pragma unroll
                    for (int i = 0; i < kVecPerLane; ++i) {
                        if (done) continue;
                        const float inc = warp_incl_scan(vs[i], lane) + run0;
                        const unsigned pos = __ballot_sync(0xffffffffu, vs[i] > 0.0f);
                        if (pos) {
                            last_i = i;
                            last_l = 31 - __clz(pos);
                        }
                        const unsigned hit = __ballot_sync(0xffffffffu, inc > target && vs[i] > 0.0f);
                        if (hit) {
                            const int l = __ffs(hit) - 1;
                            if (lane == l) {  // the crossing is inside this lane's vector
                                float r2 = inc - vs[i];
                                int lastp = -1, fi = -1;
#pragma unroll
                                for (int j = 0; j < VEC; ++j) {
                                    const float e = ex2(fmaf(Lanes<T>::get(buf[i], j), c, -mcq));
                                    r2 += e;
                                    if (e > 0.0f) lastp = (i * kWarp + lane) * VEC + j;
                                    if (fi < 0 && r2 > target && e > 0.0f)
                                        fi = (i * kWarp + lane) * VEC + j;
                                }
                                found = fi >= 0 ? fi : lastp;
                            }
                            found = __shfl_sync(0xffffffffu, found, l);
                            done = true;
                        }
                        run0 = __shfl_sync(0xffffffffu, inc, 31);
                    }
                    if (found < 0 && last_i >= 0) {  // rounding left the target past the total
#pragma unroll
                        for (int i = 0; i < kVecPerLane; ++i) {
                            if (i != last_i) continue;
                            if (lane == last_l)
                                for (int j = 0; j < VEC; ++j)
                                    if (ex2(fmaf(Lanes<T>::get(buf[i], j), c, -mcq)) > 0.0f)
                                        found = (i * kWarp + lane) * VEC + j;
                        }
                        found = __shfl_sync(0xffffffffu, found, last_l);
                    }
                    r = found >= 0 ? (int)(c0 + found) : -1;
                }
            }
        }
        dup = __any_sync(0xffffffffu, dup);
        if (lane == 0) ws.draws[row] = dup ? -2 : (bad || r < 0 ? -1 : r);
    }
}

constexpr int kWalkFusedThreads = 256;
static_assert(kFusedMaxB + 1 <= kWalkFusedThreads, "the walk block gives each node a thread");

__global__ void __launch_bounds__(kWalkFusedThreads)
predraw_walk_fused_kernel(int B, int64_t V, const int32_t* __restrict__ parent,
                          const int32_t* __restrict__ token, const int32_t* __restrict__ n_nodes,
                          VerifyWs ws, int32_t* __restrict__ exit_node, int32_t* __restrict__ bonus,
                          int32_t* __restrict__ accept_len, int32_t* __restrict__ draws,
                          int32_t* __restrict__ status) {
    pdl_entry();
    __shared__ int16_t pa[kWalkFusedThreads];
    __shared__ int32_t tk[kWalkFusedThreads], rd[kWalkFusedThreads];
    __shared__ int flags;  // bit 0: malformed tree, bit 1: a row without mass
    const int t = blockIdx.x;
    const int R = B + 1;
    const int lane = threadIdx.x & (kWarp - 1), wid = threadIdx.x / kWarp;
    const int n_raw = n_nodes[t];
    const bool n_ok = n_raw >= 1 && n_raw <= R;
    const int n = n_ok ? n_raw : 1;
    if (threadIdx.x == 0) flags = n_ok ? 0 : 1;
    __syncthreads();
    const int u = threadIdx.x;
    if (u < n) {
        const int p = parent[(int64_t)t * R + u];
        const int x = token[(int64_t)t * R + u];
        const int r = ws.draws[(int64_t)t * R + u];
        bool bad;
        if (u == 0) bad = p != -1;
        else bad = p < 0 || p >= u || x < 0 || (int64_t)x >= V;
        if (bad || r == -2) atomicOr(&flags, 1);
        if (r == -1) atomicOr(&flags, 2);
        pa[u] = (int16_t)(u == 0 ? -1 : (p >= 0 && p < u ? p : 0));
        tk[u] = x;
        rd[u] = r;
    }
    __syncthreads();
    const int fl = flags;
    const int st = (fl & 1) ? kStatBadTree : ((fl & 2) ? kStatNonFinite : kStatOk);
    if (draws)
        for (int v = threadIdx.x; v < R; v += blockDim.x)
            draws[(int64_t)t * R + v] = (st == kStatOk && v < n) ? rd[v] : -1;
    if (wid != 0) return;
    if (st != kStatOk) {
        if (lane == 0) {
            exit_node[t] = -1;
            bonus[t] = -1;
            accept_len[t] = 0;
            status[t] = st;
        }
        return;
    }
    // follow the draws from the root: the child of v whose token is R_v
    int v = 0, d = 0;
    for (int step = 0; step < n; ++step) {
        const int r = rd[v];
        int next = -1;
        for (int x0 = 1; x0 < n && next < 0; x0 += kWarp) {
            const int x = x0 + lane;
            const unsigned m = __ballot_sync(0xffffffffu, x < n && pa[x] == v && tk[x] == r);
            if (m) next = x0 + __ffs(m) - 1;
        }
        if (next < 0) break;
        v = next;
        ++d;
    }
    if (lane == 0) {
        exit_node[t] = v;
        bonus[t] = rd[v];
        accept_len[t] = d + 1;
        status[t] = kStatOk;
    }
}

bool tev_fused_fits(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    return n_trees >= 1 && B >= 0 && B <= kFusedMaxB && ((uintptr_t)logits % 16) == 0 &&
           ((V * es) % 16) == 0 && n_chunks(V, es) <= kFusedStatsPerLane * kWarp;
}

cudaError_t launch_tev_fused(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                             float c, bool greedy, uint64_t seed, const int32_t* parent,
                             const int32_t* token, const int32_t* n_nodes, const VerifyWs& ws,
                             int32_t* exit_node, int32_t* bonus, int32_t* accept_len,
                             float* exit_mass, float* prefix_prob, float* coverage,
                             int32_t* status, cudaStream_t stream, cudaEvent_t ev_between) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t items = (int64_t)n_trees * (B + 1) * nch;
    // small launches: fewer warps per block, so that the blocks spread over
    // every SM; otherwise 8 warps
    int wpb = (int)((items + sms - 1) / (sms > 0 ? sms : 1));
    wpb = wpb < 1 ? 1 : (wpb > kStreamThreads / kWarp ? kStreamThreads / kWarp : wpb);
    const size_t fsmem = fused_finish_smem(B, nch, greedy);
    auto launch = [&](auto skernel, auto fkernel, const auto* p) {
        const int64_t want = (items + wpb - 1) / wpb;
        const int grid = resident_grid((const void*)skernel, wpb * kWarp, 0, want);
        cudaError_t e = launch_pdl(skernel, grid, wpb * kWarp, 0, stream, p, n_trees, B, V, nch, c,
                                   parent, token, n_nodes, ws, true);
        if (e != cudaSuccess) return e;
        if (ev_between && (e = cudaEventRecord(ev_between, stream)) != cudaSuccess) return e;
        if (fsmem > 48 * 1024 &&
            (e = cudaFuncSetAttribute((const void*)fkernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)fsmem)) != cudaSuccess)
            return e;
        return launch_pdl(fkernel, n_trees, kFinishThreads, fsmem, stream, p, B, V, nch, c, seed,
                          parent, token, n_nodes, ws, exit_node, bonus, accept_len, exit_mass,
                          prefix_prob, coverage, status);
    };
    cudaError_t e;
    if (dtype == TSD_BF16) {
        const auto* p = static_cast<const __nv_bfloat16*>(logits);
        e = greedy ? launch(tev_stream_kernel<__nv_bfloat16, true>,
                            tev_finish_kernel<__nv_bfloat16, true>, p)
                   : launch(tev_stream_kernel<__nv_bfloat16, false>,
                            tev_finish_kernel<__nv_bfloat16, false>, p);
    } else {
        const auto* p = static_cast<const float*>(logits);
        e = greedy ? launch(tev_stream_kernel<float, true>, tev_finish_kernel<float, true>, p)
                   : launch(tev_stream_kernel<float, false>, tev_finish_kernel<float, false>, p);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_predraw_fused(const void* logits, tsd_dtype dtype, int n_trees, int B,
                                 int64_t V, float c, bool greedy, uint64_t seed,
                                 const int32_t* parent, const int32_t* token,
                                 const int32_t* n_nodes, const VerifyWs& ws, int32_t* exit_node,
                                 int32_t* bonus, int32_t* accept_len, int32_t* draws,
                                 int32_t* status, cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t rows = (int64_t)n_trees * (B + 1);
    const int64_t items = rows * nch;
    int wpb = (int)((items + sms - 1) / (sms > 0 ? sms : 1));
    wpb = wpb < 1 ? 1 : (wpb > kStreamThreads / kWarp ? kStreamThreads / kWarp : wpb);
    auto launch = [&](auto skernel, auto dkernel, const auto* p) {
        const int64_t want = (items + wpb - 1) / wpb;
        const int grid = resident_grid((const void*)skernel, wpb * kWarp, 0, want);
        cudaError_t e = launch_pdl(skernel, grid, wpb * kWarp, 0, stream, p, n_trees, B, V, nch, c,
                                   parent, token, n_nodes, ws, false);
        if (e != cudaSuccess) return e;
        // a warp per node; few warps per block when there are few nodes, so
        // that the draws spread over the SMs
        int dw = (int)((rows + sms - 1) / (sms > 0 ? sms : 1));
        dw = dw < 1 ? 1 : (dw > kDrawFusedThreads / kWarp ? kDrawFusedThreads / kWarp : dw);
        const int64_t dwant = (rows + dw - 1) / dw;
        const int dgrid = resident_grid((const void*)dkernel, dw * kWarp, 0, dwant);
        e = launch_pdl(dkernel, dgrid, dw * kWarp, 0, stream, p, n_trees, B, V, nch, c, seed,
                       n_nodes, ws);
        if (e != cudaSuccess) return e;
        return launch_pdl(predraw_walk_fused_kernel, n_trees, kWalkFusedThreads, 0, stream, B, V,
                          parent, token, n_nodes, ws, exit_node, bonus, accept_len, draws, status);
    };
    cudaError_t e;
    if (dtype == TSD_BF16) {
        const auto* p = static_cast<const __nv_bfloat16*>(logits);
        e = greedy ? launch(tev_stream_kernel<__nv_bfloat16, true>,
                            predraw_nodes_fused_kernel<__nv_bfloat16, true>, p)
                   : launch(tev_stream_kernel<__nv_bfloat16, false>,
                            predraw_nodes_fused_kernel<__nv_bfloat16, false>, p);
    } else {
        const auto* p = static_cast<const float*>(logits);
        e = greedy ? launch(tev_stream_kernel<float, true>, predraw_nodes_fused_kernel<float, true>, p)
                   : launch(tev_stream_kernel<float, false>, predraw_nodes_fused_kernel<float, false>, p);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

TSD_CHECK_READER(checks_fused)

}  // namespace tsd
