// k_tree.cu -- the per-tree part of Tree Exit Verification and the
// predraw-and-follow check.
//
// TEV, "Where Draft Trees Lose Target Mass: Exit-Guided Speculative
// Decoding", Sec. 3.1 Lemma 1 (the canonical exit law) and App. B:
//   prefix mass  P(root) = 1, P(u) = P(pa u) p_pa(u)(x_u) (Eq. 2), rho(v) from
//                the row reduction, w(v) = P(v) rho(v) (Eq. 4), C_p (Eq. 6);
//   exit draw    V ~ Categorical(w): inverse CDF over node index;
//   bonus draw   Y ~ p_V restricted to non-child tokens and renormalised (Eq. 7;
//                p_V at a leaf), inverse CDF over token id: the chunk is found
//                from the stored per-chunk residual sums, then only that chunk
//                of row V is read again.
// Predraw-and-follow (same page, Sec. 2 and App. A.4.1): R_v ~ p_v at every
// node, then a walk from the root into the child whose token is R_v.
#include "tsd_internal.cuh"

namespace tsd {

constexpr int kTreeThreads = 512;

// Exclusive prefix sum of one float per thread across the block; *total gets
// the block sum.  `red` is shared scratch of 32 floats.
__device__ float block_excl_scan(float x, float* red, float* total) {
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

// Residual bonus draw on one chunk of one row, by the whole block: the first
// token a (ascending, skipping drafted children) whose running sum of
// exp2(z*c - mc) exceeds frac * (the chunk's total).  Returns -1 only if the
// chunk has no mass.
template <typename T>
__device__ int draw_in_chunk_block(const T* __restrict__ rp, int64_t c0, int cn, float c,
                                   float mc, float frac, const int32_t* __restrict__ ctok,
                                   int clo, int chi, float* red, int* pick) {
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    constexpr int per = CE / kTreeThreads;  // elements per thread (8 bf16, 4 fp32)
    const int beg = threadIdx.x * per;
    float e[8];
    float sum = 0.0f;
    for (int j = 0; j < per; ++j) {
        const int o = beg + j;
        float v = 0.0f;
        if (o < cn) {
            bool child = false;
            for (int q = clo; q < chi; ++q) child |= ((int64_t)ctok[q] == c0 + o);
            if (!child) v = ex2(fmaf(load_logit(rp + o), c, -mc));
        }
        e[j] = v;
        sum += v;
    }
    float total;
    const float before = block_excl_scan(sum, red, &total);
    const float target = frac * total;
    if (threadIdx.x == 0) {
        pick[0] = INT_MAX;
        pick[1] = -1;
    }
    __syncthreads();
    float run = before;
    int last = -1;
    for (int j = 0; j < per; ++j) {
        run += e[j];
        if (e[j] > 0.0f) last = beg + j;
        if (run > target && e[j] > 0.0f) {
            atomicMin(pick, beg + j);
            break;
        }
    }
    if (last >= 0) atomicMax(pick + 1, last);
    __syncthreads();
    const int r = pick[0] != INT_MAX ? pick[0] : pick[1];
    __syncthreads();
    return r;
}

// The residual draw of [EXIT] Eq. 7 at exit node V_ of tree t, by the whole
// block (every thread calls it; the result is the same in all): the token a
// (ascending, drafted children skipped) at which the running residual mass
// first exceeds u * rho(V_), from the stored per-chunk residual sums, then
// only that chunk of row V_ is read again.  At T = 0 it is the row's
// arg-max, which is not a child of V_.  Returns -1 if the row has no
// residual mass.
template <typename T>
__device__ int residual_draw_block(const T* __restrict__ logits, int t, int V_, int B, int64_t V,
                                   int nch, float c, bool greedy, float u, const VerifyWs& ws,
                                   float* red, int* pick) {
    const int stride = B + 1;
    if (!TSD_IN(V_, stride, kChkExitNode)) return -1;
    const int64_t row = (int64_t)t * stride + V_;
    const NodeStat ns = ws.node[row];
    int y;
    if (greedy) {
        y = ns.amax;  // T = 0: the arg-max, which is not a child of the exit node
    } else {
        // Residual draw (Eq. 7).  Chunk sums relative to the row reference.
        const ChunkStat* cs = ws.chunk + row * nch;
        const float thr2 = u * ns.r;
        constexpr int CE = kChunkBytes / (int)sizeof(T);
        const int32_t* ctok = ws.child_tok + (int64_t)t * (B + 1);
        __shared__ int chunk_sel, chunk_clo, chunk_chh;
        __shared__ float chunk_frac;
        if (threadIdx.x < kWarp) {
            const int lane = threadIdx.x;
            // the exit node's children (sorted by token): the first 32 tokens
            // are loaded now, beside the chunk sums, one per lane
            const int32_t* cptr = ws.child_ptr + (int64_t)t * (B + 2);
            int kids_lo = cptr[V_], kids_hi = cptr[V_ + 1];
            if (!(TSD_IN(kids_lo, B + 1, kChkChildList) && TSD_IN(kids_hi, B + 1, kChkChildList)))
                kids_lo = kids_hi = 0;
            const int32_t tk0 = kids_lo + lane < kids_hi ? ctok[kids_lo + lane] : 0;
            float base = 0.0f;
            int sel = -1, lastc = -1;
            float frac = 0.0f;
            for (int q0 = 0; q0 < nch && sel < 0; q0 += kWarp) {
                const int q = q0 + lane;
                float rq = 0.0f;
                if (q < nch && cs[q].m != -INFINITY) rq = cs[q].r * ex2(__fmul_rn(cs[q].m, c) - ns.mc);
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
            // [clo, chh): the children whose tokens fall in the chosen chunk,
            // counted 32 children per step
            int clo = kids_lo, chh = kids_lo;
            if (sel >= 0) {
                const int64_t c0 = (int64_t)sel * CE, c1 = c0 + CE;
                int32_t tk = tk0;
                for (int j0 = kids_lo; j0 < kids_hi; j0 += kWarp) {
                    const bool valid = j0 + lane < kids_hi;
                    if (j0 > kids_lo) tk = valid ? ctok[j0 + lane] : 0;
                    clo += __popc(__ballot_sync(0xffffffffu, valid && (int64_t)tk < c0));
                    chh += __popc(__ballot_sync(0xffffffffu, valid && (int64_t)tk < c1));
                }
            }
            if (lane == 0) {
                chunk_sel = sel;
                chunk_frac = fminf(fmaxf(frac, 0.0f), 0.99999994f);
                chunk_clo = clo;
                chunk_chh = chh;
            }
        }
        __syncthreads();
        const int q = chunk_sel;
        y = -1;
        if (q >= 0 && TSD_IN(q, nch, kChkExitNode)) {
            const int64_t c0 = (int64_t)q * CE;
            const int cn = (int)min((int64_t)CE, V - c0);
            const int o = draw_in_chunk_block<T>(logits + row * V + c0, c0, cn, c,
                                                 __fmul_rn(cs[q].m, c), chunk_frac, ctok,
                                                 chunk_clo, chunk_chh, red, pick);
            y = o >= 0 ? (int)(c0 + o) : -1;
        }
    }
    return y;
}

template <typename T>
__global__ void __launch_bounds__(kTreeThreads)
tev_tree_kernel(const T* __restrict__ logits, int B, int64_t V, int nch, float c, bool greedy,
                uint64_t seed, const int32_t* __restrict__ parent,
                const int32_t* __restrict__ n_nodes, VerifyWs ws, int32_t* __restrict__ exit_node,
                int32_t* __restrict__ bonus, int32_t* __restrict__ accept_len,
                float* __restrict__ exit_mass, float* __restrict__ prefix_prob,
                float* __restrict__ coverage, int32_t* __restrict__ status) {
    pdl_entry();
    extern __shared__ float sh[];  // w[B+1], pedge[B+1], and parents as int[B+1]
    __shared__ float red[33];
    __shared__ int pick[2];
    __shared__ int exit_v;
    const int t = blockIdx.x;
    const int stride = B + 1;
    const int n = n_nodes[t];
    const int st = ws.tstat[t];
    if (st != kStatOk) {
        for (int v = threadIdx.x; v < stride; v += blockDim.x) {
            if (exit_mass) exit_mass[(int64_t)t * stride + v] = 0.0f;
            if (prefix_prob) prefix_prob[(int64_t)t * stride + v] = 0.0f;
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
    const int32_t* gpar = parent + (int64_t)t * stride;
    const float* gpedge = ws.pedge + (int64_t)t * stride;
    const float* rho = ws.rho + (int64_t)t * stride;
    float* w = sh;
    float* pedge = sh + stride;
    int* par = reinterpret_cast<int*>(sh + 2 * stride);
    // the tree's parents and edge probabilities in shared memory (one
    // coalesced read) so that the ancestor walks below stay on chip
    for (int u = threadIdx.x; u < n; u += blockDim.x) {
        par[u] = gpar[u];
        pedge[u] = gpedge[u];
    }
    __syncthreads();
    // Eq. 2: P(u) as the product of the edge probabilities on the
    // root path (depth-parallel: every node walks its own ancestors).
    float cov_part = 0.0f;
    for (int u = threadIdx.x; u < stride; u += blockDim.x) {
        float P = 0.0f, wu = 0.0f;
        if (u < n) {
            const float ru = rho[u];  // issued before the walk
            P = 1.0f;
            for (int x = u; x > 0;) {
                P *= pedge[x];
                const int px = par[x];
                if (!TSD_IN(px, x, kChkAncestor)) break;
                x = px;
            }
            wu = P * ru;
            if (u > 0) cov_part += P;
        }
        w[u] = wu;
        if (exit_mass) exit_mass[(int64_t)t * stride + u] = wu;
        if (prefix_prob) prefix_prob[(int64_t)t * stride + u] = P;
    }
    float cov;
    block_excl_scan(cov_part, red, &cov);
    // Exit draw: inverse CDF over nodes.  Each thread owns a contiguous run of
    // nodes so that the block scan follows node order.
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int nb = threadIdx.x * per, ne = min(n, nb + per);
    float mine = 0.0f;
    for (int v = nb; v < ne; ++v) mine += w[v];
    float wsum;
    float run = block_excl_scan(mine, red, &wsum);
    const float thr = uniform24(seed, t, 0, 0) * wsum;
    if (threadIdx.x == 0) {
        pick[0] = INT_MAX;
        pick[1] = -1;
    }
    __syncthreads();
    int last = -1;
    for (int v = nb; v < ne; ++v) {
        run += w[v];
        if (w[v] > 0.0f) last = v;
        if (run > thr && w[v] > 0.0f) {
            atomicMin(pick, v);
            break;
        }
    }
    if (last >= 0) atomicMax(pick + 1, last);
    __syncthreads();
    if (threadIdx.x == 0) exit_v = pick[0] != INT_MAX ? pick[0] : (pick[1] >= 0 ? pick[1] : 0);
    __syncthreads();
    const int V_ = exit_v;
    const int y = residual_draw_block<T>(logits, t, V_, B, V, nch, c, greedy,
                                         uniform24(seed, t, 0, 1), ws, red, pick);
    if (threadIdx.x == 0) {
        exit_node[t] = V_;
        bonus[t] = y;
        accept_len[t] = ws.depth[(int64_t)t * stride + V_] + 1;
        if (coverage) coverage[t] = cov;
        status[t] = y >= 0 ? kStatOk : kStatNonFinite;
    }
}

cudaError_t launch_tev_tree(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                            float c, bool greedy, uint64_t seed, const int32_t* parent,
                            const int32_t* n_nodes, const VerifyWs& ws, int32_t* exit_node,
                            int32_t* bonus, int32_t* accept_len, float* exit_mass,
                            float* prefix_prob, float* coverage, int32_t* status,
                            cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    const size_t smem = 3 * sizeof(float) * (size_t)(B + 1);
    cudaError_t e = cudaFuncSetAttribute(dtype == TSD_BF16 ? (const void*)tev_tree_kernel<__nv_bfloat16>
                                                           : (const void*)tev_tree_kernel<float>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dtype == TSD_BF16) {
        if (cudaError_t e_ = launch_pdl(tev_tree_kernel<__nv_bfloat16>, n_trees, kTreeThreads, smem, stream, 
            static_cast<const __nv_bfloat16*>(logits), B, V, nch, c, greedy, seed, parent, n_nodes,
            ws, exit_node, bonus, accept_len, exit_mass, prefix_prob, coverage, status); e_ != cudaSuccess) return e_;
    } else {
        if (cudaError_t e_ = launch_pdl(tev_tree_kernel<float>, n_trees, kTreeThreads, smem, stream, 
            static_cast<const float*>(logits), B, V, nch, c, greedy, seed, parent, n_nodes, ws,
            exit_node, bonus, accept_len, exit_mass, prefix_prob, coverage, status); e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Predraw-and-follow.
// ---------------------------------------------------------------------------
constexpr int kDrawThreads = 256;

// One warp per node: R_v ~ p_v by inverse CDF over token id.
template <typename T>
__global__ void __launch_bounds__(kDrawThreads)
predraw_nodes_kernel(const T* __restrict__ logits, int n_trees, int B, int64_t V, int nch, float c,
                     bool greedy, uint64_t seed, const int32_t* __restrict__ n_nodes, bool vec_ok,
                     VerifyWs ws) {
    pdl_entry();
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    constexpr int PER = CE / kWarp;  // tokens per lane in one chunk (128 bf16, 64 fp32)
    const int lane = threadIdx.x & (kWarp - 1);
    const int wpb = blockDim.x / kWarp;
    const int64_t rows = (int64_t)n_trees * (B + 1);
    for (int64_t row = (int64_t)blockIdx.x * wpb + threadIdx.x / kWarp; row < rows;
         row += (int64_t)gridDim.x * wpb) {
        const int t = (int)(row / (B + 1));
        const int v = (int)(row - (int64_t)t * (B + 1));
        if (v >= n_nodes[t] || ws.tstat[t] != kStatOk) continue;
        const NodeStat ns = ws.node[row];
        if (greedy) {
            if (lane == 0) ws.draws[row] = ns.amax;
            continue;
        }
        const ChunkStat* cs = ws.chunk + row * nch;
        const float thr = uniform24(seed, t, v, 2) * ns.s;
        float base = 0.0f, frac = 1.0f;
        int sel = -1, lastc = -1;
        for (int q0 = 0; q0 < nch && sel < 0; q0 += kWarp) {
            const int q = q0 + lane;
            float sq = 0.0f;
            if (q < nch && cs[q].m != -INFINITY) sq = cs[q].s * ex2(__fmul_rn(cs[q].m, c) - ns.mc);
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
        int r = -1;
        if (sel >= 0 && vec_ok) {
            // the chunk in 16-byte vectors, all loads in flight: vector i of
            // lane l holds tokens (i*32 + l)*VEC .. +VEC, so (i, lane, element)
            // is token order
            constexpr int VEC = Lanes<T>::kVec;
            const int64_t c0 = (int64_t)sel * CE;
            const int cn = (int)min((int64_t)CE, V - c0);
            const float mc = __fmul_rn(cs[sel].m, c);
            const T* rp = logits + row * V + c0;
            uint4 buf[kVecPerLane];
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int e = (i * kWarp + lane) * VEC;
                buf[i] = e < cn ? ld_stream16(rp + e) : Lanes<T>::neg_inf();
            }
            float vs[kVecPerLane], mine = 0.0f;
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                float a = 0.0f;
#pragma unroll
                for (int j = 0; j < VEC; ++j) a += ex2(fmaf(Lanes<T>::get(buf[i], j), c, -mc));
                vs[i] = a;
                mine += a;
            }
            const float target = frac * warp_sum(mine);
            float base = 0.0f;
            int found = -1, last_i = -1, last_l = -1;
            bool done = false;  // warp-uniform
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                if (done) continue;
                const float inc = warp_incl_scan(vs[i], lane) + base;
                const unsigned pos = __ballot_sync(0xffffffffu, vs[i] > 0.0f);
                if (pos) {
                    last_i = i;
                    last_l = 31 - __clz(pos);
                }
                const unsigned hit = __ballot_sync(0xffffffffu, inc > target && vs[i] > 0.0f);
                if (hit) {
                    const int l = __ffs(hit) - 1;
                    if (lane == l) {  // the crossing is inside this lane's vector (re-read)
                        const uint4 q = ld_stream16(rp + (i * kWarp + lane) * VEC);
                        float run = inc - vs[i];
                        int lastp = -1, f = -1;
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            const float e = ex2(fmaf(Lanes<T>::get(q, j), c, -mc));
                            run += e;
                            if (e > 0.0f) lastp = (i * kWarp + lane) * VEC + j;
                            if (f < 0 && run > target && e > 0.0f) f = (i * kWarp + lane) * VEC + j;
                        }
                        found = f >= 0 ? f : lastp;
                    }
                    found = __shfl_sync(0xffffffffu, found, l);
                    done = true;
                }
                base = __shfl_sync(0xffffffffu, inc, 31);
            }
            if (found < 0 && last_i >= 0) {  // rounding left the target past the total
#pragma unroll
                for (int i = 0; i < kVecPerLane; ++i) {
                    if (i != last_i) continue;
                    if (lane == last_l) {
                        const uint4 q = ld_stream16(rp + (i * kWarp + lane) * VEC);
                        for (int j = 0; j < VEC; ++j)
                            if (ex2(fmaf(Lanes<T>::get(q, j), c, -mc)) > 0.0f)
                                found = (i * kWarp + lane) * VEC + j;
                    }
                }
                found = __shfl_sync(0xffffffffu, found, last_l);
            }
            r = found >= 0 ? found + (int)c0 : -1;
        } else if (sel >= 0) {
            const int64_t c0 = (int64_t)sel * CE;
            const int cn = (int)min((int64_t)CE, V - c0);
            const float mc = __fmul_rn(cs[sel].m, c);
            const T* rp = logits + row * V + c0;
            // lane l scans tokens [l*PER, (l+1)*PER) of the chunk
            float sum = 0.0f;
            for (int j = 0; j < PER; ++j) {
                const int o = lane * PER + j;
                if (o < cn) sum += ex2(fmaf(load_logit(rp + o), c, -mc));
            }
            const float inc = warp_incl_scan(sum, lane);
            const float total = __shfl_sync(0xffffffffu, inc, 31);
            const float target = frac * total;
            float run = inc - sum;
            int found = -1, lastp = -1;
            for (int j = 0; j < PER; ++j) {
                const int o = lane * PER + j;
                if (o >= cn) break;
                const float e = ex2(fmaf(load_logit(rp + o), c, -mc));
                run += e;
                if (e > 0.0f) lastp = o;
                if (run > target && e > 0.0f) {
                    found = o;
                    break;
                }
            }
            const unsigned f = __ballot_sync(0xffffffffu, found >= 0);
            if (f) {
                r = __shfl_sync(0xffffffffu, found, __ffs(f) - 1);
            } else {
                const unsigned lp = __ballot_sync(0xffffffffu, lastp >= 0);
                r = lp ? __shfl_sync(0xffffffffu, lastp, 31 - __clz(lp)) : -1;
            }
            if (r >= 0) r += (int)c0;
        }
        if (lane == 0) {
            ws.draws[row] = r;
            if (r < 0) atomicExch(ws.tstat + t, kStatNonFinite);
        }
    }
}

// One CTA per tree: the block copies the draws, thread 0 follows R_v from the
// root.
__global__ void predraw_walk_kernel(int n_trees, int B, const int32_t* __restrict__ n_nodes,
                                    VerifyWs ws, int32_t* __restrict__ exit_node,
                                    int32_t* __restrict__ bonus, int32_t* __restrict__ accept_len,
                                    int32_t* __restrict__ draws, int32_t* __restrict__ status) {
    pdl_entry();
    const int t = blockIdx.x;  // one CTA per tree: the block copies the draws, thread 0 walks
    const int stride = B + 1;
    const int n = n_nodes[t];
    const int st = ws.tstat[t];
    if (draws)
        for (int v = threadIdx.x; v < stride; v += blockDim.x)
            draws[(int64_t)t * stride + v] = (st == kStatOk && v < n) ? ws.draws[(int64_t)t * stride + v] : -1;
    if (threadIdx.x != 0) return;
    if (st != kStatOk) {
        exit_node[t] = -1;
        bonus[t] = -1;
        accept_len[t] = 0;
        status[t] = st;
        return;
    }
    const int32_t* cptr = ws.child_ptr + (int64_t)t * (B + 2);
    const int32_t* ctok = ws.child_tok + (int64_t)t * (B + 1);
    const int32_t* cnode = ws.child_node + (int64_t)t * (B + 1);
    int v = 0;
    for (int step = 0; step < n; ++step) {
        const int r = ws.draws[(int64_t)t * stride + v];
        int lo = cptr[v], hi = cptr[v + 1];
        if (!(TSD_IN(lo, stride, kChkPredraw) && TSD_IN(hi, stride, kChkPredraw))) break;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (ctok[mid] < r) lo = mid + 1;
            else hi = mid;
        }
        if (lo < cptr[v + 1] && ctok[lo] == r && TSD_IN(cnode[lo], n, kChkPredraw)) v = cnode[lo];
        else break;
    }
    exit_node[t] = v;
    bonus[t] = ws.draws[(int64_t)t * stride + v];
    accept_len[t] = ws.depth[(int64_t)t * stride + v] + 1;
    status[t] = kStatOk;
}

cudaError_t launch_predraw(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                           float c, bool greedy, uint64_t seed, const int32_t* n_nodes,
                           const VerifyWs& ws, int32_t* exit_node, int32_t* bonus,
                           int32_t* accept_len, int32_t* draws, int32_t* status,
                           cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    const bool vec_ok = ((uintptr_t)logits % 16 == 0) && ((V * es) % 16 == 0);
    const int64_t rows = (int64_t)n_trees * (B + 1);
    const int wpb = kDrawThreads / kWarp;
    const int64_t want = (rows + wpb - 1) / wpb;
    const int grid = (int)(want < 65535 * 8 ? want : 65535 * 8);
    if (dtype == TSD_BF16) {
        if (cudaError_t e_ = launch_pdl(predraw_nodes_kernel<__nv_bfloat16>, grid, kDrawThreads, 0, stream, 
            static_cast<const __nv_bfloat16*>(logits), n_trees, B, V, nch, c, greedy, seed, n_nodes, vec_ok, ws); e_ != cudaSuccess) return e_;
    } else {
        if (cudaError_t e_ = launch_pdl(predraw_nodes_kernel<float>, grid, kDrawThreads, 0, stream, 
            static_cast<const float*>(logits), n_trees, B, V, nch, c, greedy, seed, n_nodes, vec_ok, ws); e_ != cudaSuccess) return e_;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (cudaError_t e_ = launch_pdl(predraw_walk_kernel, (unsigned)n_trees, 128, 0, stream, n_trees, B, n_nodes, ws, exit_node,
                                                                 bonus, accept_len, draws, status); e_ != cudaSuccess) return e_;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Exact sequential residual verification ([EXIT] App. A.4.2) and
// proposal-aware verification ([CAST] App. B.1 Thm. 3): one CTA per tree.
// Warp 0 walks from the root on the per-node statistics of the row
// reduction (p_v(x_u) of every child, rho(v)), staged with the tree and its
// uniforms in shared memory; the whole block then draws the bonus token from
// the exit node's residual, as TEV's last step does.  At each node the
// children are taken in ascending token order (the CSR lists are sorted by
// token).
// ---------------------------------------------------------------------------
template <typename T>
__device__ void finish_walk(const T* __restrict__ logits, int t, int v, int B, int64_t V, int nch,
                            float c, bool greedy, float u_bonus, const VerifyWs& ws,
                            int32_t* exit_node, int32_t* bonus, int32_t* accept_len,
                            int32_t* status, float* red, int* pick) {
    const int y = residual_draw_block<T>(logits, t, v, B, V, nch, c, greedy, u_bonus, ws, red, pick);
    if (threadIdx.x == 0) {
        exit_node[t] = v;
        bonus[t] = y;
        accept_len[t] = ws.depth[(int64_t)t * (B + 1) + v] + 1;
        status[t] = y >= 0 ? kStatOk : kStatNonFinite;
    }
}

__device__ __forceinline__ bool tree_failed(int t, int st, int32_t* exit_node, int32_t* bonus,
                                            int32_t* accept_len, int32_t* status) {
    if (st == kStatOk) return false;
    if (threadIdx.x == 0) {
        exit_node[t] = -1;
        bonus[t] = -1;
        accept_len[t] = 0;
        status[t] = st;
    }
    return true;
}

// Children u_1..u_k of the current node are tested in turn; u_j is followed
// when u_j (1 - M_{j-1}) < p_j (Eq. 49, uniform stream 3, sub j-1), where p_j
// = p_v(x_j) and M_{j-1} sums the earlier p's.  With every child rejected the
// walk exits and the bonus is drawn from the Eq. 53 residual (stream 4).
// The walk verifiers' view of one tree, staged in shared memory by the whole
// block so that the single walking thread never waits on global memory: CSR
// child offsets and nodes, every node's edge probability, and for every CSR
// edge q = cptr[v] + j the uniforms of the walk at node v, step j (streams
// given by the caller; one uniform per edge and stream).
struct WalkTree {
    int* cptr;    // [n + 1]
    int* cnode;   // [n - 1]
    float* pedge; // [n]
    float* u0;    // [n - 1] stream s0 at (v, j)
    float* u1;    // [n - 1] stream s1 at (v, j), when s1 >= 0
};

// 4-byte words of the staging: child offsets, child nodes, edge
// probabilities and one uniform stream; a second stream adds B + 1.
static size_t walk_smem_words(int B) { return (size_t)(B + 2) + 3 * (size_t)(B + 1); }

__device__ void stage_walk_tree(const VerifyWs& ws, int t, int n, int B, uint64_t seed, int s0,
                                int s1, float* sm, WalkTree& wt) {
    wt.cptr = reinterpret_cast<int*>(sm);
    wt.cnode = wt.cptr + (B + 2);
    wt.pedge = reinterpret_cast<float*>(wt.cnode + (B + 1));
    wt.u0 = wt.pedge + (B + 1);
    wt.u1 = wt.u0 + (B + 1);
    const int m = n - 1;
    for (int i = threadIdx.x; i <= n; i += blockDim.x) {
        const int x = ws.child_ptr[(int64_t)t * (B + 2) + i];
        wt.cptr[i] = TSD_IN(x, n, kChkWalk) ? x : 0;  // offsets into the n - 1 edges
    }
    for (int i = threadIdx.x; i < m; i += blockDim.x) wt.cnode[i] = ws.child_node[(int64_t)t * (B + 1) + i];
    for (int i = threadIdx.x; i < n; i += blockDim.x) wt.pedge[i] = ws.pedge[(int64_t)t * (B + 1) + i];
    __syncthreads();
    for (int q = threadIdx.x; q < m; q += blockDim.x) {
        if (!TSD_IN(wt.cnode[q], n, kChkWalk)) wt.cnode[q] = 0;
        int lo = 0, hi = n;  // the node v with cptr[v] <= q < cptr[v+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (wt.cptr[mid] <= q) lo = mid;
            else hi = mid;
        }
        wt.u0[q] = uniform24(seed, t, lo, s0, q - wt.cptr[lo]);
        if (s1 >= 0) wt.u1[q] = uniform24(seed, t, lo, s1, q - wt.cptr[lo]);
    }
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kTreeThreads)
seqres_tree_kernel(const T* __restrict__ logits, int B, int64_t V, int nch, float c, bool greedy,
                   uint64_t seed, const int32_t* __restrict__ n_nodes, VerifyWs ws,
                   int32_t* __restrict__ exit_node, int32_t* __restrict__ bonus,
                   int32_t* __restrict__ accept_len, int32_t* __restrict__ status) {
    pdl_entry();
    extern __shared__ float shw[];
    __shared__ float red[33];
    __shared__ int pick[2];
    __shared__ int exit_v;
    const int t = blockIdx.x;
    if (tree_failed(t, ws.tstat[t], exit_node, bonus, accept_len, status)) return;
    WalkTree wt;
    stage_walk_tree(ws, t, n_nodes[t], B, seed, 3, -1, shw, wt);
    // Warp 0 walks: lane l tests the children j = l, l + 32, ... of the
    // current node against their rejected mass M_j (an exclusive warp scan),
    // and the first child that passes is followed.
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int* cptr = wt.cptr;
        const int* cnode = wt.cnode;
        int v = 0;
        for (;;) {
            const int b0 = cptr[v], k = cptr[v + 1] - b0;
            float M = 0.0f;
            int next = -1;
            for (int j0 = 0; j0 < k; j0 += 32) {
                const int q = b0 + j0 + lane;
                const float pj = j0 + lane < k ? wt.pedge[cnode[q]] : 0.0f;
                const float incl = warp_incl_scan(pj, lane);
                const float Mj = M + (incl - pj);
                const unsigned hit =
                    __ballot_sync(0xffffffffu, j0 + lane < k && wt.u0[q] * (1.0f - Mj) < pj);
                if (hit) {
                    next = cnode[b0 + j0 + __ffs(hit) - 1];
                    break;
                }
                M += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (next < 0) break;
            v = next;
        }
        if (lane == 0) exit_v = v;
    }
    __syncthreads();
    const int v = exit_v;
    finish_walk<T>(logits, t, v, B, V, nch, c, greedy, uniform24(seed, t, v, 4), ws, exit_node,
                   bonus, accept_len, status, red, pick);
}

// Recursive speculative sampling without replacement at each visited node.
// mu starts at p_v: on the children it is held explicitly (mu_c), on the
// other tokens as s * p_v (s starts at 1; their total is s * rho(v)).  Each
// step draws a candidate from q~ = q over the retained children, normalised
// (inverse CDF in token order, stream 5, sub = step), and accepts it when
// u q~(c) < mu_c (stream 6, sub = step).  A rejection sets mu <- (mu - q~)_+
// normalised and retires c.  With every child retired the committed token is
// drawn from mu, which is then zero on the children: the residual draw of
// the exit node (stream 7).  q_child[u] = q_{pa(u)}(x_u); a non-positive or
// non-finite value marks the tree TSD_ERR_NONFINITE.
template <typename T>
__global__ void __launch_bounds__(kTreeThreads)
proposal_tree_kernel(const T* __restrict__ logits, int B, int64_t V, int nch, float c,
                     bool greedy, uint64_t seed, const float* __restrict__ q_child,
                     const int32_t* __restrict__ n_nodes, VerifyWs ws,
                     int32_t* __restrict__ exit_node, int32_t* __restrict__ bonus,
                     int32_t* __restrict__ accept_len, int32_t* __restrict__ status) {
    pdl_entry();
    // the staged tree (see stage_walk_tree), then q and rho per node, then the
    // current node's children's mu and q, [2][B]
    extern __shared__ float shp[];
    __shared__ float red[33];
    __shared__ int pick[2];
    __shared__ int exit_v, bad;
    const int t = blockIdx.x;
    if (tree_failed(t, ws.tstat[t], exit_node, bonus, accept_len, status)) return;
    const int n = n_nodes[t];
    WalkTree wt;
    stage_walk_tree(ws, t, n, B, seed, 5, 6, shp, wt);
    float* qn = wt.u1 + (B + 1);      // [n] q_child per node
    float* rhon = qn + (B + 1);       // [n] rho per node
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        qn[i] = q_child[(int64_t)t * (B + 1) + i];
        rhon[i] = ws.rho[(int64_t)t * (B + 1) + i];
    }
    __syncthreads();
    // Warp 0 walks; lane l owns the children j = l, l + 32, ... of the current
    // node, so the sums over the children are shuffles and the inverse-CDF
    // pick is a warp scan with a ballot.
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int* cptr = wt.cptr;
        const int* cnode = wt.cnode;
        float* mu = rhon + (B + 1);
        float* qv = mu + B;
        int v = 0, fail = 0;
        for (;;) {
            const int b0 = cptr[v], k = cptr[v + 1] - b0;
            for (int j = lane; j < k; j += 32) {
                const int u = cnode[b0 + j];
                mu[j] = wt.pedge[u];
                qv[j] = qn[u];
                if (!(qv[j] > 0.0f) || isinf(qv[j])) fail = 1;
            }
            if (__any_sync(0xffffffffu, fail)) {
                fail = 1;
                break;
            }
            __syncwarp();
            const float rho = rhon[v];
            float s = 1.0f;  // scale of the non-child tokens
            int next = -1;
            for (int step = 0; step < k; ++step) {
                float Q = 0.0f;
                for (int j = lane; j < k; j += 32)
                    if (qv[j] > 0.0f) Q += qv[j];
                Q = warp_sum(Q);
                const float thr = wt.u0[b0 + step] * Q;
                // first live child whose running proposal mass passes thr,
                // else the last live child
                float carry = 0.0f;
                int cand = -1, lastj = -1;
                for (int j0 = 0; j0 < k && cand < 0; j0 += 32) {
                    const int j = j0 + lane;
                    const bool live = j < k && qv[j] > 0.0f;
                    const float run = carry + warp_incl_scan(live ? qv[j] : 0.0f, lane);
                    const unsigned hit = __ballot_sync(0xffffffffu, live && run > thr);
                    const unsigned alive = __ballot_sync(0xffffffffu, live);
                    if (hit) cand = j0 + __ffs(hit) - 1;
                    else if (alive) lastj = j0 + 31 - __clz(alive);
                    carry = __shfl_sync(0xffffffffu, run, 31);
                }
                if (cand < 0) cand = lastj;
                const float qt = qv[cand] / Q;
                if (wt.u1[b0 + step] * qt < mu[cand]) {
                    next = cnode[b0 + cand];
                    break;
                }
                float z = 0.0f;  // (mu - q~)_+ and its total
                for (int j = lane; j < k; j += 32) {
                    if (!(qv[j] > 0.0f)) continue;
                    mu[j] = fmaxf(mu[j] - qv[j] / Q, 0.0f);
                    z += mu[j];
                }
                z = s * rho + warp_sum(z);
                if (!(z > 0.0f)) {
                    fail = 1;
                    break;
                }
                const float inv = 1.0f / z;
                s *= inv;
                for (int j = lane; j < k; j += 32) mu[j] *= inv;
                __syncwarp();
                if (lane == (cand & 31)) {
                    mu[cand] = 0.0f;
                    qv[cand] = -1.0f;  // retired
                }
                __syncwarp();
            }
            __syncwarp();
            if (fail || next < 0) break;
            v = next;
        }
        if (lane == 0) {
            exit_v = v;
            bad = fail;
        }
    }
    __syncthreads();
    if (bad) {
        tree_failed(t, kStatNonFinite, exit_node, bonus, accept_len, status);
        return;
    }
    const int v = exit_v;
    finish_walk<T>(logits, t, v, B, V, nch, c, greedy, uniform24(seed, t, v, 7), ws, exit_node,
                   bonus, accept_len, status, red, pick);
}

cudaError_t launch_seqres_tree(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                               float c, bool greedy, uint64_t seed, const int32_t* n_nodes,
                               const VerifyWs& ws, int32_t* exit_node, int32_t* bonus,
                               int32_t* accept_len, int32_t* status, cudaStream_t stream) {
    const int nch = (int)n_chunks(V, dtype == TSD_BF16 ? 2 : 4);
    const size_t smem = sizeof(float) * walk_smem_words(B);
    cudaError_t e = cudaFuncSetAttribute(dtype == TSD_BF16
                                             ? (const void*)seqres_tree_kernel<__nv_bfloat16>
                                             : (const void*)seqres_tree_kernel<float>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dtype == TSD_BF16)
        return launch_pdl(seqres_tree_kernel<__nv_bfloat16>, (unsigned)n_trees, kTreeThreads, smem,
                          stream, static_cast<const __nv_bfloat16*>(logits), B, V, nch, c, greedy,
                          seed, n_nodes, ws, exit_node, bonus, accept_len, status);
    return launch_pdl(seqres_tree_kernel<float>, (unsigned)n_trees, kTreeThreads, smem, stream,
                      static_cast<const float*>(logits), B, V, nch, c, greedy, seed, n_nodes, ws,
                      exit_node, bonus, accept_len, status);
}
cudaError_t launch_proposal_tree(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                                 float c, bool greedy, uint64_t seed, const float* q_child,
                                 const int32_t* n_nodes, const VerifyWs& ws, int32_t* exit_node,
                                 int32_t* bonus, int32_t* accept_len, int32_t* status,
                                 cudaStream_t stream) {
    const int nch = (int)n_chunks(V, dtype == TSD_BF16 ? 2 : 4);
    // staging with two uniform streams, q and rho per node, then mu and q of
    // the current node's children
    const size_t smem =
        sizeof(float) * (walk_smem_words(B) + 3 * (size_t)(B + 1) + 2 * (size_t)(B > 0 ? B : 1));
    cudaError_t e = cudaFuncSetAttribute(dtype == TSD_BF16
                                             ? (const void*)proposal_tree_kernel<__nv_bfloat16>
                                             : (const void*)proposal_tree_kernel<float>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dtype == TSD_BF16)
        return launch_pdl(proposal_tree_kernel<__nv_bfloat16>, (unsigned)n_trees, kTreeThreads,
                          smem, stream, static_cast<const __nv_bfloat16*>(logits), B, V, nch, c,
                          greedy, seed, q_child, n_nodes, ws, exit_node, bonus, accept_len, status);
    return launch_pdl(proposal_tree_kernel<float>, (unsigned)n_trees, kTreeThreads, smem, stream,
                      static_cast<const float*>(logits), B, V, nch, c, greedy, seed, q_child,
                      n_nodes, ws, exit_node, bonus, accept_len, status);
}

TSD_CHECK_READER(checks_tree)

}  // namespace tsd
