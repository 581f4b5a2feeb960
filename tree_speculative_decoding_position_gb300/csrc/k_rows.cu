// k_rows.cu -- the node-row reduction of Tree Exit Verification.
//
// "Where Draft Trees Lose Target Mass: Exit-Guided Speculative Decoding",
// Sec. 3 Eq. 1 (p_v = softmax(z_v / T)), Sec. 3.1 Eq. 4 (rho(v): the mass of
// the tokens that are not drafted children of v) and Eq. 7 (the residual law
// the bonus token is drawn from).  App. B calls these node-local reductions;
// they read every logit of every tree node once and carry all of the path's
// HBM traffic.
//
// Three kernels:
//   verify_prep_kernel   one CTA per tree: validates the tree, computes
//                        depths and a CSR list of each node's children sorted
//                        by token (so a chunk finds its children by binary
//                        search).
//   rows_kernel          one warp per (node row, 8 KB chunk): max, sum of
//                        exp2(z*c - mc), the same sum without the drafted
//                        children, or the arg-max when T = 0.
//   node_combine_kernel  one warp per node row: combines its chunks, the
//                        child probabilities p_v(x_u) and rho(v).
#include "chunk_reduce.cuh"

#include <float.h>

namespace tsd {

// ---------------------------------------------------------------------------
// Tree preparation.
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 512;
constexpr int kPrepMaxKeys = 4096;  // next power of two >= TSD_MAX_B

// key = parent << 43 | token << 12 | node: sorting orders children by parent,
// then token; parent < 4096 (12 bits), token < 2^31, node < 4096.
__device__ __forceinline__ uint64_t child_key(int p, int tok, int u) {
    return ((uint64_t)p << 43) | ((uint64_t)(uint32_t)tok << 12) | (uint64_t)u;
}

// Bitonic sort of keys[0, n2) ascending (n2 a power of two, at least 32).
// Steps with partner distance below 32 run in registers with warp shuffles;
// only longer distances exchange through shared memory between barriers.
__device__ __forceinline__ uint64_t bitonic_lane_steps_u64(uint64_t x, int e, int lane, int k,
                                                           int jtop) {
    for (int j = jtop; j > 0; j >>= 1) {
        const uint64_t y = __shfl_xor_sync(0xffffffffu, x, j);
        const bool lower = (lane & j) == 0;
        const bool asc = (e & k) == 0;
        const uint64_t lo = x < y ? x : y, hi = x < y ? y : x;
        x = (lower == asc) ? lo : hi;
    }
    return x;
}

__device__ void block_bitonic_sort(uint64_t* keys, int n2) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nblk = n2 >> 5;
    for (int b = wid; b < nblk; b += nw) {
        const int e = (b << 5) + lane;
        uint64_t x = keys[e];
        for (int k = 2; k <= 32; k <<= 1) x = bitonic_lane_steps_u64(x, e, lane, k, k >> 1);
        keys[e] = x;
    }
    __syncthreads();
    for (int k = 64; k <= n2; k <<= 1) {
        for (int j = k >> 1; j >= 32; j >>= 1) {
            for (int i = threadIdx.x; i < n2; i += blockDim.x) {
                const int l = i ^ j;
                if (l > i) {
                    const uint64_t a = keys[i], b = keys[l];
                    const bool up = (i & k) == 0;
                    if ((a > b) == up) {
                        keys[i] = b;
                        keys[l] = a;
                    }
                }
            }
            __syncthreads();
        }
        for (int b = wid; b < nblk; b += nw) {
            const int e = (b << 5) + lane;
            keys[e] = bitonic_lane_steps_u64(keys[e], e, lane, k, 16);
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kPrepThreads)
verify_prep_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ token,
                   const int32_t* __restrict__ n_nodes, int B, int64_t V, VerifyWs ws) {
    pdl_entry();
    __shared__ uint64_t keys[kPrepMaxKeys];
    __shared__ int16_t spar[kPrepMaxKeys];  // parents, for the depth walks on chip
    __shared__ int bad;
    const int t = blockIdx.x;
    const int32_t* par = parent + (int64_t)t * (B + 1);
    const int32_t* tok = token + (int64_t)t * (B + 1);
    const int n = n_nodes[t];
    if (threadIdx.x == 0) bad = (n < 1 || n > B + 1 || par[0] != -1) ? 1 : 0;
    __syncthreads();
    const int nn = bad ? 1 : n;
    const int m = nn - 1;  // number of child edges
    int n2 = 32;
    while (n2 < m) n2 <<= 1;
    for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        uint64_t key = ~0ull;
        if (i < m) {
            const int u = i + 1, p = par[u], x = tok[u];
            if (p < 0 || p >= u || x < 0 || (int64_t)x >= V) bad = 1;
            else key = child_key(p, x, u);
            spar[u] = (int16_t)p;
        }
        keys[i] = key;
    }
    __syncthreads();
    if (!bad) {
        block_bitonic_sort(keys, n2);
        for (int i = threadIdx.x + 1; i < m; i += blockDim.x)
            if ((keys[i] >> 12) == (keys[i - 1] >> 12)) bad = 1;  // repeated sibling token
    }
    __syncthreads();
    const int stat = bad ? kStatBadTree : kStatOk;
    if (threadIdx.x == 0) ws.tstat[t] = stat;
    if (bad) return;
    int32_t* cptr = ws.child_ptr + (int64_t)t * (B + 2);
    int32_t* ctok = ws.child_tok + (int64_t)t * (B + 1);
    int32_t* cnode = ws.child_node + (int64_t)t * (B + 1);
    int32_t* dep = ws.depth + (int64_t)t * (B + 1);
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
        ctok[i] = (int32_t)((keys[i] >> 12) & 0x7fffffffu);
        const int32_t u = (int32_t)(keys[i] & 0xfffu);
        cnode[i] = TSD_IN(u, nn, kChkPrep) ? u : 0;
    }
    // child_ptr[v] = first sorted edge whose parent is >= v
    for (int v = threadIdx.x; v <= nn; v += blockDim.x) {
        int lo = 0, hi = m;
        const uint64_t probe = (uint64_t)v << 43;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (keys[mid] < probe) lo = mid + 1;
            else hi = mid;
        }
        cptr[v] = lo;
    }
    for (int u = threadIdx.x; u < nn; u += blockDim.x) {
        int d = 0, x = u;
        while (x > 0) {  // parents precede children, so this ends within u steps
            x = spar[x];
            ++d;
        }
        dep[u] = d;
    }
}

cudaError_t launch_verify_prep(const int32_t* parent, const int32_t* token, const int32_t* n_nodes,
                               int n_trees, int B, int64_t V, const VerifyWs& ws,
                               cudaStream_t stream) {
    if (cudaError_t e_ = launch_pdl(verify_prep_kernel, n_trees, kPrepThreads, 0, stream, parent, token, n_nodes, B, V, ws); e_ != cudaSuccess) return e_;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Row reduction.
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 256;

// One warp per (node row, 8 KB chunk), persistent over a grid stride.  On the
// vectorised path a warp issues the next live chunk's loads as soon as the
// current chunk's per-lane partials are done, and finishes the current
// chunk's warp reductions while they are in flight; a chunk's child lookup
// likewise runs while its own loads are in flight.
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kRowThreads)
rows_kernel(const T* __restrict__ logits, int n_trees, int B, int64_t V, int nch, float c,
            bool vec_ok, const int32_t* __restrict__ n_nodes, VerifyWs ws) {
    pdl_entry();
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
        return TSD_IN(q.t, n_trees, kChkRowsItem) && TSD_IN(q.v, R, kChkRowsItem) &&
               TSD_IN(q.ch, nch, kChkRowsItem) && __ldg(n_nodes + q.t) > q.v &&
               ws.tstat[q.t] == kStatOk;
    };
    auto children = [&](const ItemPos& q, int64_t c0, int cn, int& clo, int& chi) {
        clo = chi = 0;
        if (!GREEDY) {
            const int32_t* cptr = ws.child_ptr + (int64_t)q.t * (B + 2);
            const int32_t* ctok = ws.child_tok + (int64_t)q.t * R;
            const int b0 = cptr[q.v], b1 = cptr[q.v + 1];
            if (b1 > b0 && TSD_IN(b0, R, kChkChildList) && TSD_IN(b1, R, kChkChildList)) {
                clo = lower_bound_i32(ctok, b0, b1, c0);
                chi = lower_bound_i32(ctok, clo, b1, c0 + cn);
            }
        }
    };
    auto chunk_ptr = [&](const ItemPos& q, int64_t& c0, int& cn) {
        c0 = (int64_t)q.ch * CE;
        cn = (int)min((int64_t)CE, V - c0);
        return logits + ((int64_t)q.t * R + q.v) * V + c0;
    };

    if (!vec_ok) {
        for (; p.item < total; item_advance(p, step, R, nch)) {
            if (!live(p)) continue;
            int64_t c0;
            int cn, clo, chi;
            const T* rp = chunk_ptr(p, c0, cn);
            children(p, c0, cn, clo, chi);
            const ChunkStat st = reduce_chunk_scalar<T, GREEDY>(
                rp, cn, c, ws.child_tok + (int64_t)p.t * R, clo, chi, c0, lane);
            if (lane == 0) ws.chunk[p.item] = st;
        }
        return;
    }
    while (p.item < total && !live(p)) item_advance(p, step, R, nch);
    if (p.item >= total) return;
    uint4 buf[kVecPerLane];
    int64_t c0;
    int cn;
    load_chunk<T>(buf, chunk_ptr(p, c0, cn), cn, lane);
    for (;;) {
        int clo, chi;
        children(p, c0, cn, clo, chi);
        const LanePart lp =
            chunk_lane<T, GREEDY>(buf, cn, c, ws.child_tok + (int64_t)p.t * R, clo, chi, c0, lane);
        const int64_t done = p.item;
        do {
            item_advance(p, step, R, nch);
        } while (p.item < total && !live(p));
        if (p.item < total) load_chunk<T>(buf, chunk_ptr(p, c0, cn), cn, lane);
        const ChunkStat st = chunk_finish<GREEDY>(lp);
        if (lane == 0) ws.chunk[done] = st;
        if (p.item >= total) break;
    }
}

static int row_grid(int64_t items) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int wpb = kRowThreads / kWarp;
    const int64_t want = (items + wpb - 1) / wpb;
    const int64_t cap = (int64_t)sms * 8;  // a few resident CTAs per SM, grid-stride beyond
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_rows(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                        float c, bool greedy, const int32_t* n_nodes, const VerifyWs& ws,
                        cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    const bool vec_ok = ((uintptr_t)logits % 16 == 0) && ((V * es) % 16 == 0);
    const int64_t items = (int64_t)n_trees * (B + 1) * nch;
    // A batch that fits in about one wave of resident CTAs runs as exactly that
    // wave: the grid-stride loop takes the few extra items, with their loads
    // issued early, instead of a second wave of CTAs starting cold.  Larger
    // batches stream over a few waves of CTAs (measured slightly faster there
    // than one persistent wave).
    auto launch = [&](auto kernel, const auto* p) {
        const int64_t want = (items + kRowThreads / kWarp - 1) / (kRowThreads / kWarp);
        const int wave = resident_grid((const void*)kernel, kRowThreads, 0, INT64_MAX);
        const int grid = want <= 2 * (int64_t)wave ? (int)(want < wave ? (want > 0 ? want : 1) : wave)
                                                   : row_grid(items);
        return launch_pdl(kernel, grid, kRowThreads, 0, stream, p, n_trees, B, V, nch, c, vec_ok,
                          n_nodes, ws);
    };
    cudaError_t e;
    if (dtype == TSD_BF16) {
        const auto* p = static_cast<const __nv_bfloat16*>(logits);
        e = greedy ? launch(rows_kernel<__nv_bfloat16, true>, p)
                   : launch(rows_kernel<__nv_bfloat16, false>, p);
    } else {
        const auto* p = static_cast<const float*>(logits);
        e = greedy ? launch(rows_kernel<float, true>, p) : launch(rows_kernel<float, false>, p);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Per-node combination: row max / sums, p_v(x_u) of each child, rho(v).
// ---------------------------------------------------------------------------
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(kRowThreads)
node_combine_kernel(const T* __restrict__ logits, int n_trees, int B, int64_t V, int nch, float c,
                    const int32_t* __restrict__ n_nodes, VerifyWs ws) {
    pdl_entry();
    const int lane = threadIdx.x & (kWarp - 1);
    const int wpb = blockDim.x / kWarp;
    const int64_t rows = (int64_t)n_trees * (B + 1);
    for (int64_t row = (int64_t)blockIdx.x * wpb + threadIdx.x / kWarp; row < rows;
         row += (int64_t)gridDim.x * wpb) {
        const int t = (int)(row / (B + 1));
        const int v = (int)(row - (int64_t)t * (B + 1));
        if (v >= n_nodes[t] || ws.tstat[t] != kStatOk) continue;
        const ChunkStat* cs = ws.chunk + row * nch;
        const int32_t* cptr = ws.child_ptr + (int64_t)t * (B + 2);
        const int32_t* ctok = ws.child_tok + (int64_t)t * (B + 1);
        const int32_t* cnode = ws.child_node + (int64_t)t * (B + 1);
        float* pedge = ws.pedge + (int64_t)t * (B + 1);
        int b0 = cptr[v], b1 = cptr[v + 1];
        if (!(TSD_IN(b0, B + 1, kChkChildList) && TSD_IN(b1, B + 1, kChkChildList))) b0 = b1 = 0;
        NodeStat ns;
        bool bad = false;
        if (GREEDY) {
            float bm = -INFINITY;
            int bi = INT_MAX;
            for (int q = lane; q < nch; q += kWarp) {
                const ChunkStat s = cs[q];
                bad |= (s.s != s.s);
                if (better(s.m, s.amax, bm, bi)) {
                    bm = s.m;
                    bi = s.amax;
                }
            }
            warp_argmax(bm, bi);
            bad |= (bm == -INFINITY);  // every token masked: no arg-max
            ns.mc = bm;
            ns.s = 1.0f;
            ns.amax = bi;
            bool hit = false;  // is the arg-max a drafted child?
            for (int q = b0 + lane; q < b1; q += kWarp) {
                const bool h = (ctok[q] == bi);
                if (TSD_IN(cnode[q], B + 1, kChkChildList)) pedge[cnode[q]] = h ? 1.0f : 0.0f;
                hit |= h;
            }
            ns.r = __any_sync(0xffffffffu, hit) ? 0.0f : 1.0f;
        } else {
            float m = -INFINITY;
            for (int q = lane; q < nch; q += kWarp) m = fmaxf(m, cs[q].m);
            m = warp_max(m);
            const float mc = __fmul_rn(m, c);
            float s = 0.0f, r = 0.0f;
            for (int q = lane; q < nch; q += kWarp) {
                const ChunkStat x = cs[q];
                bad |= (x.s != x.s);
                if (x.m != -INFINITY) {
                    const float f = ex2(__fmul_rn(x.m, c) - mc);
                    s += x.s * f;
                    r += x.r * f;
                }
            }
            s = warp_sum(s);
            r = warp_sum(r);
            bad = __any_sync(0xffffffffu, bad) || m == -INFINITY || !(s > 0.0f);
            ns.mc = mc;
            ns.s = s;
            ns.r = r;
            ns.amax = -1;
            if (!bad) {
                const T* rp = logits + row * V;
                const float inv_s = 1.0f / s;
                for (int q = b0 + lane; q < b1; q += kWarp) {
                    if (!(TSD_IN(ctok[q], V, kChkChildList) && TSD_IN(cnode[q], B + 1, kChkChildList)))
                        continue;
                    const float z = load_logit(rp + ctok[q]);
                    pedge[cnode[q]] = ex2(fmaf(z, c, -mc)) * inv_s;
                }
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            ws.node[row] = ns;
            ws.rho[row] = GREEDY ? ns.r : (bad ? 0.0f : ns.r / ns.s);
            if (bad) atomicExch(ws.tstat + t, kStatNonFinite);
        }
    }
}

cudaError_t launch_node_combine(const void* logits, tsd_dtype dtype, int n_trees, int B,
                                int64_t V, float c, bool greedy, const int32_t* n_nodes,
                                const VerifyWs& ws, cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    const int grid = row_grid((int64_t)n_trees * (B + 1));
    if (dtype == TSD_BF16) {
        const auto* p = static_cast<const __nv_bfloat16*>(logits);
        if (greedy) {
            if (cudaError_t e_ = launch_pdl(node_combine_kernel<__nv_bfloat16, true>, grid, kRowThreads, 0, stream, p, n_trees, B, V, nch, c, n_nodes, ws); e_ != cudaSuccess) return e_;
        } else {
            if (cudaError_t e_ = launch_pdl(node_combine_kernel<__nv_bfloat16, false>, grid, kRowThreads, 0, stream, p, n_trees, B, V, nch, c, n_nodes, ws); e_ != cudaSuccess) return e_;
        }
    } else {
        const auto* p = static_cast<const float*>(logits);
        if (greedy) {
            if (cudaError_t e_ = launch_pdl(node_combine_kernel<float, true>, grid, kRowThreads, 0, stream, p, n_trees, B, V, nch, c, n_nodes, ws); e_ != cudaSuccess) return e_;
        } else {
            if (cudaError_t e_ = launch_pdl(node_combine_kernel<float, false>, grid, kRowThreads, 0, stream, p, n_trees, B, V, nch, c, n_nodes, ws); e_ != cudaSuccess) return e_;
        }
    }
    return cudaGetLastError();
}

TSD_CHECK_READER(checks_rows)

}  // namespace tsd
