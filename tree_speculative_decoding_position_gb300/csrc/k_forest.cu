// k_forest.cu -- cost-aware width with a budget shared across requests.
//
// "CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters",
// Sec. 3.3 Thm. 2 (marginal stopping rule) and App. B.4 Prop. 2-3: under
// load, R requests share one verification budget; the optimal allocation
// takes the globally largest prefix masses (global best-first over the
// disjoint union of the requests' candidate trees), and with the affine round
// time l(M) = l0 + c1 M the global node M+1 is added while
//   rho_(M+1) >= c1 (G(M) + R) / l(M),   G(M) = sum of the M largest masses.
// Each request's candidates are its builder tree (pop order = mass order), so
// its share is the first width nodes of that tree.
//
// Each request's candidates come out of the builder in (score desc, depth
// asc) order, and the rule is monotone: with f(j) = rho_(j) l(j) - c1 (G(j) + R),
// f(j+1) - f(j) = (rho_(j+1) - rho_(j)) l(j+1) <= 0, so once a node fails every
// later one fails.  No global sort is needed: a candidate's place in the merge
// (ties go to the lower request) is the sum over the other requests of a
// binary search in their sorted lists, and the mass ahead of it is the sum of
// their prefix sums at those points.
//
// forest_prep_kernel    one CTA per request: masses rho = exp(score) and their
//                       exclusive float64 prefix sums; resets the two
//                       counters (first failing rank, candidate count).
// forest_rank_kernel    one warp per candidate: lanes split the other
//                       requests, reduce count and mass ahead, test the rule
//                       at that rank; failing ranks reduce into the counter.
// forest_finish_kernel  one CTA per request: M* = min(first failure, M_max,
//                       candidates), its width (own candidates ranked below
//                       M*, by binary search), n_nodes = width + 1, and the
//                       slots past it cleared.
#include "tsd_internal.cuh"

namespace tsd {

constexpr int kForestThreads = 256;
constexpr int kRankWarps = kForestThreads / kWarp;

// Exclusive block scan of one double per thread; *total gets the block sum.
__device__ double block_excl_scan_d(double x, double* red, double* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    double inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) red[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        double y = lane < nw ? red[lane] : 0.0;
        double yi = y;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double z = __shfl_up_sync(0xffffffffu, yi, o);
            if (lane >= o) yi += z;
        }
        red[lane] = yi - y;
        if (lane == 31) red[32] = yi;
    }
    __syncthreads();
    const double r = red[wid] + inc - x;
    *total = red[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kForestThreads)
forest_prep_kernel(const double* __restrict__ score64, int B, int M_max,
                   const int32_t* __restrict__ n_nodes, const int32_t* __restrict__ status,
                   ForestWs ws) {
    pdl_entry();
    __shared__ double red[33];
    const int r = blockIdx.x, tid = threadIdx.x;
    const int64_t base = (int64_t)r * (B + 1);
    if (r == 0 && tid == 0) {
        ws.ctl[0] = M_max;  // first failing rank (min-reduced)
        ws.ctl[1] = 0;      // number of candidates (max-reduced rank + 1)
    }
    const int m = status[r] == kStatOk ? max(n_nodes[r] - 1, 0) : 0;
    if (tid == 0) ws.cnt[r] = m;
    double carry = 0.0;
    for (int j0 = 0; j0 < m; j0 += blockDim.x) {
        const int j = j0 + tid;
        const double sc = j < m ? score64[base + 1 + j] : -INFINITY;
        const double x = j < m ? exp(sc) : 0.0;
        double tot;
        const double ex = block_excl_scan_d(x, red, &tot);
        if (j < m) {
            ws.rho[base + j] = x;
            ws.pre[base + j] = carry + ex;
            ws.img[base + j] = order_key(sc);
        }
        carry += tot;
    }
    if (tid == 0) ws.pre[base + m] = carry;
}

__global__ void __launch_bounds__(kForestThreads)
forest_rank_kernel(const int32_t* __restrict__ depth,
                   int n_trees, int B, int M_max, double l0, double c1, ForestWs ws) {
    pdl_entry();
    __shared__ int fail_min, count_max;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int r = blockIdx.y, j = blockIdx.x * kRankWarps + w;
    const int stride = B + 1;
    if (threadIdx.x == 0) {
        fail_min = INT_MAX;
        count_max = 0;
    }
    __syncthreads();
    const int m = ws.cnt[r];
    if (j < m) {
        const int64_t me = (int64_t)r * stride + 1 + j;
        const unsigned long long sc = ws.img[(int64_t)r * stride + j];  // score order image
        const int dc = depth[me];
        int ahead = 0;
        double G = 0.0;
        for (int q = lane; q < n_trees; q += kWarp) {
            if (q == r) continue;
            // first node of request q that does not precede this candidate
            const int64_t qb = (int64_t)q * stride;
            int lo = 0, hi = ws.cnt[q];
            if (!TSD_IN(hi, stride, kChkForest)) hi = 0;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                const unsigned long long sx = ws.img[qb + mid];
                bool before = sx > sc;
                if (sx == sc) {
                    const int dx = depth[qb + 1 + mid];
                    before = dx < dc || (dx == dc && q < r);
                }
                if (before) lo = mid + 1;
                else hi = mid;
            }
            ahead += lo;
            G += ws.pre[qb + lo];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ahead += __shfl_xor_sync(0xffffffffu, ahead, o);
            G += __shfl_xor_sync(0xffffffffu, G, o);
        }
        const int rank = j + ahead;
        G += ws.pre[(int64_t)r * stride + j];
        if (lane == 0) {
            ws.rank[(int64_t)r * stride + j] = rank;
            const double l = l0 + c1 * (double)rank;
            const double rho = ws.rho[(int64_t)r * stride + j];
            if (rank < M_max && !(rho >= (G + (double)n_trees) / l * c1)) atomicMin(&fail_min, rank);
            atomicMax(&count_max, rank + 1);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (fail_min != INT_MAX) atomicMin(&ws.ctl[0], fail_min);
        if (count_max > 0) atomicMax(&ws.ctl[1], count_max);
    }
}

__global__ void __launch_bounds__(kForestThreads)
forest_finish_kernel(int B, ForestWs ws, int32_t* __restrict__ n_nodes,
                     const int32_t* __restrict__ status, int32_t* __restrict__ total,
                     int32_t* __restrict__ parent, int32_t* __restrict__ token,
                     int32_t* __restrict__ depth, float* __restrict__ score) {
    pdl_entry();
    __shared__ int keep;
    const int r = blockIdx.x;
    const int64_t stride = B + 1;
    const int M = min(ws.ctl[0], ws.ctl[1]);
    if (threadIdx.x == 0) {
        if (status[r] == kStatOk) {
            // own candidates ranked below M* (ranks increase along the list)
            const int32_t* rk = ws.rank + (int64_t)r * stride;
            int lo = 0, hi = ws.cnt[r];
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (rk[mid] < M) lo = mid + 1;
                else hi = mid;
            }
            keep = TSD_IN(lo, stride, kChkForest) ? lo + 1 : 1;
            n_nodes[r] = keep;
        } else {
            keep = n_nodes[r];
        }
        if (r == 0) *total = M;
    }
    __syncthreads();
    for (int i = keep + threadIdx.x; i <= B; i += blockDim.x) {
        const int64_t s = (int64_t)r * stride + i;
        parent[s] = -1;
        token[s] = -1;
        depth[s] = -1;
        score[s] = -INFINITY;
    }
}

cudaError_t launch_forest_select(const double* score64, int32_t* depth, int n_trees, int B,
                                 int M_max, double l0, double c1, int32_t* n_nodes,
                                 const int32_t* status, int32_t* total, int32_t* parent,
                                 int32_t* token, float* score, const ForestWs& ws,
                                 cudaStream_t stream) {
    cudaError_t e = launch_pdl(forest_prep_kernel, (unsigned)n_trees, kForestThreads, 0, stream,
                               score64, B, M_max, (const int32_t*)n_nodes, status, ws);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((B + kRankWarps - 1) / kRankWarps), (unsigned)n_trees);
    e = launch_pdl(forest_rank_kernel, grid, kForestThreads, 0, stream, (const int32_t*)depth, n_trees, B, M_max, l0, c1, ws);
    if (e != cudaSuccess) return e;
    return launch_pdl(forest_finish_kernel, (unsigned)n_trees, kForestThreads, 0, stream, B, ws,
                      n_nodes, status, total, parent, token, depth, score);
}

TSD_CHECK_READER(checks_forest)

}  // namespace tsd
