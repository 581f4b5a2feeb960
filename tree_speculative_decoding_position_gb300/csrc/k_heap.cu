// k_heap.cu -- best-first tree builder over the top-k universe.
//
// "CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters", Thm. 1
// and App. C "Candidate construction": the B prefixes with the largest
// plug-in score sum_j log q_j(y_j), expanded best-first from a heap keyed by
// cumulative log-probability; ties toward shorter prefixes, then
// lexicographic.
// "Multi-Future Drafting: Mixture Block Drafters for Tree-Verified
// Speculative Decoding", Sec. 3.4 Eq. 2, Sec. 4.3 and App. B "Merged heap"
// (Prop. 6): one heap of (mode, prefix) entries keyed by that mode's score;
// popping an entry pushes its next sibling (rank r+1) and its first child
// (rank 0 at the next position); a prefix popped again from another mode
// reuses its node and spends no budget.  With one mode this is DDTree.
//
// One warp per tree.  The heap operations are sequential, so lane 0 runs
// them on a binary heap in shared memory (global workspace when a very large
// budget does not fit); the other lanes load the lists and fill the tail.
// Scores are float64 sums like the pages' host builders; comparisons use a
// 64-bit order-preserving integer of the score plus a 64-bit tie key
// (depth << 59 | mode << 56 | rank sequence).
#include "tsd_internal.cuh"

namespace tsd {

struct __align__(16) HEntry {
    unsigned long long key;  // order-preserving image of the score
    unsigned long long tb;   // depth << 59 | mode << 56 | rank digits
    double pscore;           // the same mode's score of the parent prefix
    int32_t pnode;           // tree node of the parent prefix
    int16_t rank;            // rank of the last token in this mode's list
    int8_t mode;
    int8_t depth;
};
static_assert(sizeof(HEntry) == 32, "heap entry layout");

__device__ __forceinline__ unsigned long long order_key(double s) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(s);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double key_score(unsigned long long k) {
    const unsigned long long u = (k >> 63) ? (k & 0x7fffffffffffffffull) : ~k;
    return __longlong_as_double((long long)u);
}
__device__ __forceinline__ bool hbefore(const HEntry& a, const HEntry& b) {
    return a.key > b.key || (a.key == b.key && a.tb < b.tb);
}

__device__ __forceinline__ void heap_push(HEntry* h, int& hn, const HEntry& x) {
    int i = hn++;
    while (i > 0) {
        const int p = (i - 1) >> 1;
        if (!hbefore(x, h[p])) break;
        h[i] = h[p];
        i = p;
    }
    h[i] = x;
}

__device__ __forceinline__ HEntry heap_pop(HEntry* h, int& hn) {
    const HEntry top = h[0];
    const HEntry x = h[--hn];
    int i = 0;
    for (;;) {
        const int l = 2 * i + 1;
        if (l >= hn) break;
        const int r = l + 1;
        const int c = (r < hn && hbefore(h[r], h[l])) ? r : l;
        if (!hbefore(h[c], x)) break;
        h[i] = h[c];
        i = c;
    }
    if (hn > 0) h[i] = x;
    return top;
}

struct HeapSmem {
    size_t lists, nodes, heap, total;
    bool heap_in_smem;
};

static int digit_bits(int k) {
    int b = 0;
    while ((1 << b) < k) ++b;
    return b;
}

static HeapSmem heap_smem_plan(int n_modes, int L, int topk, int B) {
    HeapSmem p;
    p.lists = (size_t)n_modes * L * topk * (sizeof(int32_t) + sizeof(double));
    p.lists = (p.lists + 15) & ~(size_t)15;
    p.nodes = (size_t)(B + 1) * (2 * sizeof(int16_t) + sizeof(int32_t));
    p.nodes = (p.nodes + 15) & ~(size_t)15;
    p.heap = sizeof(HEntry) * ((size_t)n_modes * (B + 1) + 1);
    p.heap_in_smem = p.lists + p.nodes + p.heap <= 200 * 1024;
    p.total = p.lists + p.nodes + (p.heap_in_smem ? p.heap : 0);
    return p;
}

size_t heap_spill_bytes(int n_modes, int L, int topk, int B) {
    const HeapSmem p = heap_smem_plan(n_modes, L, topk, B);
    return p.heap_in_smem ? 0 : p.heap;
}

__global__ void __launch_bounds__(kWarp)
build_heap_kernel(BuildWs ws, int K, int L, int k, int B, int bits, size_t lists_bytes,
                  size_t nodes_bytes, bool heap_in_smem, int32_t* __restrict__ parent,
                  int32_t* __restrict__ token, int32_t* __restrict__ depth,
                  float* __restrict__ score, int32_t* __restrict__ rank,
                  int32_t* __restrict__ mode, int32_t* __restrict__ n_nodes_out,
                  int32_t* __restrict__ status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int t = blockIdx.x;
    const int lane = threadIdx.x;
    const int nl = K * L * k;
    double* lq = reinterpret_cast<double*>(smem);
    int32_t* ids = reinterpret_cast<int32_t*>(smem + (size_t)nl * sizeof(double));
    int16_t* first_child = reinterpret_cast<int16_t*>(smem + lists_bytes);
    int16_t* next_sib = first_child + (B + 1);
    int32_t* ntok = reinterpret_cast<int32_t*>(next_sib + (B + 1));
    HEntry* heap = heap_in_smem ? reinterpret_cast<HEntry*>(smem + lists_bytes + nodes_bytes)
                                : reinterpret_cast<HEntry*>(ws.heap + (size_t)t * ws.heap_stride);
    const int stride = B + 1;
    bool bad = false;
    for (int i = lane; i < nl; i += kWarp) {
        const double x = ws.top_lq[(int64_t)t * nl + i];
        lq[i] = x;
        ids[i] = ws.top_id[(int64_t)t * nl + i];
        bad |= (x != x);
    }
    for (int i = lane; i <= B; i += kWarp) first_child[i] = next_sib[i] = -1;
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    int n = 0;
    if (!bad && lane == 0) {
        int32_t* par = parent + (int64_t)t * stride;
        int32_t* tok = token + (int64_t)t * stride;
        int32_t* dep = depth + (int64_t)t * stride;
        float* sc = score + (int64_t)t * stride;
        int32_t* rk = rank ? rank + (int64_t)t * stride : nullptr;
        int32_t* md = mode ? mode + (int64_t)t * stride : nullptr;
        par[0] = -1;
        tok[0] = -1;
        dep[0] = 0;
        sc[0] = 0.0f;
        if (rk) rk[0] = -1;
        if (md) md[0] = -1;
        int hn = 0;
        const unsigned long long rs_mask = (1ull << 56) - 1;
        for (int m = 0; m < K; ++m) {  // each mode's best first token
            HEntry e;
            e.key = order_key(0.0 + lq[(m * L + 0) * k + 0]);
            e.tb = (1ull << 59) | ((unsigned long long)m << 56);
            e.pscore = 0.0;
            e.pnode = 0;
            e.rank = 0;
            e.mode = (int8_t)m;
            e.depth = 1;
            heap_push(heap, hn, e);
        }
        n = 1;
        while (n <= B && hn > 0) {
            const HEntry e = heap_pop(heap, hn);
            const double s = key_score(e.key);
            if (s == -INFINITY) break;  // only zero-probability prefixes remain
            const int m = e.mode, d = e.depth, r = e.rank;
            const int x = ids[(m * L + d - 1) * k + r];
            int node = -1;
            if (K > 1)
                for (int cch = first_child[e.pnode]; cch >= 0; cch = next_sib[cch])
                    if (ntok[cch] == x) {
                        node = cch;
                        break;
                    }
            if (node < 0) {
                node = n++;
                ntok[node] = x;
                next_sib[node] = first_child[e.pnode];  // child lists are only searched
                first_child[e.pnode] = (int16_t)node;
                par[node] = e.pnode;
                tok[node] = x;
                dep[node] = d;
                sc[node] = (float)s;
                if (rk) rk[node] = r;
                if (md) md[node] = m;
            }
            if (r + 1 < k) {  // next sibling: same parent, next rank
                HEntry sb = e;
                sb.key = order_key(e.pscore + lq[(m * L + d - 1) * k + r + 1]);
                sb.tb = e.tb + 1;
                sb.rank = (int16_t)(r + 1);
                heap_push(heap, hn, sb);
            }
            if (d < L) {  // first child: rank 0 at the next position
                HEntry ch;
                ch.key = order_key(s + lq[(m * L + d) * k + 0]);
                ch.tb = ((unsigned long long)(d + 1) << 59) | ((unsigned long long)m << 56) |
                        (((e.tb & rs_mask) << bits) & rs_mask);
                ch.pscore = s;
                ch.pnode = node;
                ch.rank = 0;
                ch.mode = (int8_t)m;
                ch.depth = (int8_t)(d + 1);
                heap_push(heap, hn, ch);
            }
        }
    }
    n = __shfl_sync(0xffffffffu, n, 0);
    __syncwarp();
    // Tail slots (and every slot of a failed tree).
    const int from = bad ? 0 : n;
    for (int i = from + lane; i <= B; i += kWarp) {
        parent[(int64_t)t * stride + i] = -1;
        token[(int64_t)t * stride + i] = -1;
        depth[(int64_t)t * stride + i] = -1;
        score[(int64_t)t * stride + i] = -INFINITY;
        if (rank) rank[(int64_t)t * stride + i] = -1;
        if (mode) mode[(int64_t)t * stride + i] = -1;
    }
    if (lane == 0) {
        n_nodes_out[t] = bad ? 0 : n;
        status[t] = bad ? kStatNonFinite : kStatOk;
    }
}

cudaError_t launch_build_heap(const BuildWs& ws, int n_trees, int n_modes, int L, int topk, int B,
                              int32_t* parent, int32_t* token, int32_t* depth, float* score,
                              int32_t* rank, int32_t* mode, int32_t* n_nodes, int32_t* status,
                              cudaStream_t stream) {
    const HeapSmem p = heap_smem_plan(n_modes, L, topk, B);
    cudaError_t e = cudaFuncSetAttribute(build_heap_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)p.total);
    if (e != cudaSuccess) return e;
    build_heap_kernel<<<n_trees, kWarp, p.total, stream>>>(
        ws, n_modes, L, topk, B, digit_bits(topk), p.lists, p.nodes, p.heap_in_smem, parent,
        token, depth, score, rank, mode, n_nodes, status);
    return cudaGetLastError();
}

}  // namespace tsd
