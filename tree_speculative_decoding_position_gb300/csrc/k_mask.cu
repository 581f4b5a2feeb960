// k_mask.cu -- ancestor mask and position ids of the packed verification
// input.
//
// "CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters", App. C
// "Packed verification": the pending root sits at position P and node z_i at
// P + depth(v_i); every packed token sees the P prefix entries and its own
// ancestor chain inside the pack, itself included (an additive mask of shape
// (1, 1, 1+N, P+1+N)).  App. B Lemma 1 shows this reproduces N+1 separate
// forwards.  The pages build it on the host from the parent pointers; here
// one CTA per tree builds it on the device.
#include "tsd_internal.cuh"

namespace tsd {

constexpr int kMaskThreads = 256;

__global__ void __launch_bounds__(kMaskThreads)
tree_mask_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ n_nodes, int B,
                 int prefix_len, uint32_t* __restrict__ anc_bits,
                 int32_t* __restrict__ position_ids, float* __restrict__ additive_mask,
                 int64_t mask_ld, int32_t* __restrict__ status) {
    pdl_entry();
    __shared__ int bad;
    const int t = blockIdx.x;
    const int stride = B + 1;
    const int W = (B + 32) / 32;
    const int32_t* par = parent + (int64_t)t * stride;
    int n = n_nodes[t];
    if (threadIdx.x == 0) bad = (n < 1 || n > stride || par[0] != -1) ? 1 : 0;
    __syncthreads();
    if (!bad)
        for (int u = 1 + threadIdx.x; u < n; u += blockDim.x)
            if (par[u] < 0 || par[u] >= u) bad = 1;
    __syncthreads();
    if (bad) n = 0;  // every row becomes a padding row
    uint32_t* bits = anc_bits + (int64_t)t * stride * W;
    for (int v = threadIdx.x; v < stride; v += blockDim.x) {
        uint32_t* row = bits + (int64_t)v * W;
        int d = 0;
        if (v < n) {
            // Ancestors come out in decreasing index order (parents precede
            // children), so the row's words are written from the last down.
            int w = W - 1;
            uint32_t acc = 0;
            for (int u = v; u >= 0;
                 u = (u > 0 && TSD_IN(par[u], u, kChkMask) ? par[u] : -1)) {
                const int wu = u >> 5;
                while (w > wu) {
                    row[w--] = acc;
                    acc = 0;
                }
                acc |= 1u << (u & 31);
                if (u > 0) ++d;
            }
            while (w >= 0) {
                row[w--] = acc;
                acc = 0;
            }
        } else {
            for (int w = 0; w < W; ++w) row[w] = (w == (v >> 5)) ? (1u << (v & 31)) : 0u;
        }
        position_ids[(int64_t)t * stride + v] = prefix_len + d;
    }
    if (threadIdx.x == 0) status[t] = bad ? kStatBadTree : kStatOk;
    if (additive_mask == nullptr) return;
    __syncthreads();  // the bit rows above are visible to the whole block
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int64_t cols = (int64_t)prefix_len + stride;
    for (int v = wid; v < stride; v += nw) {
        const uint32_t* row = bits + (int64_t)v * W;
        float* out = additive_mask + ((int64_t)t * stride + v) * mask_ld;
        for (int64_t cidx = lane; cidx < cols; cidx += 32) {
            float val = 0.0f;
            if (cidx >= prefix_len) {
                const int u = (int)(cidx - prefix_len);
                val = ((row[u >> 5] >> (u & 31)) & 1u) ? 0.0f : -INFINITY;
            }
            out[cidx] = val;
        }
    }
}

cudaError_t launch_tree_mask(const int32_t* parent, const int32_t* n_nodes, int n_trees, int B,
                             int prefix_len, uint32_t* anc_bits, int32_t* position_ids,
                             float* additive_mask, int64_t mask_ld, int32_t* status,
                             cudaStream_t stream) {
    if (cudaError_t e_ = launch_pdl(tree_mask_kernel, n_trees, kMaskThreads, 0, stream, parent, n_nodes, B, prefix_len,
                                                           anc_bits, position_ids, additive_mask,
                                                           mask_ld, status); e_ != cudaSuccess) return e_;
    return cudaGetLastError();
}

TSD_CHECK_READER(checks_mask)

}  // namespace tsd
