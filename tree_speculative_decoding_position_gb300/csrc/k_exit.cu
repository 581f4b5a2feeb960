// k_exit.cu -- the exit-guided loss of ExitTrain.
//
// "Where Draft Trees Lose Target Mass: Exit-Guided Speculative Decoding",
// Sec. 5 Eq. 14 and App. C.2 Eq. 66-67:
//   L_exit = sum_v w(v) (-log q_{depth(v)}(x_v)) / sum_i (|V_i| - 1),
// summed over the non-root nodes of every tree, evaluated as Eq. 67 does:
// each drafter row m needs one log-normaliser LSE_m, weighted by the summed
// weight W_m of the nodes it scores, minus a gather of the scored logits:
//   numerator = sum_m W_m LSE_m - sum_v w(v) z_{row(v), x_v} / T_d.
// Node v is scored by the row of future position depth(v) (row depth(v) - 1).
//
// Kernels:
//   drafter_chunk_kernel (k_drafter.cu)  the streaming pass over the rows;
//   exit_tree_kernel  one CTA per tree: its rows' LSE_m, W_m, the gather and
//                     the numerator; the last CTA to finish forms the scalar;
//   exit_grad_kernel  optional streaming pass: d loss / dz = (W_m softmax_m -
//                     sum_v w(v) [a = x_v]) / (T_d N), written as the dense
//                     part, then exit_scatter_kernel subtracts the gathers.
#include "tsd_internal.cuh"

namespace tsd {

constexpr int kExitThreads = 256;

// Statistics of two rows of z / T_d from their chunk statistics as the
// builder's row kernel forms them, by one warp (the second row at cs + off2;
// off2 < 0: none, its results unused): the scaled maximum mc and the float64
// sum S = sum over chunks of s 2^(m c - mc), so that LSE = ln 2 * (mc +
// log2 S); bad when a chunk saw a NaN or +inf or the row has no mass.  The
// two rows' loads and float64 sums are interleaved so that their latencies
// overlap.
__device__ void row_stats_pair(const ChunkStat* __restrict__ cs, int64_t off2, int nch, float c,
                               int lane, float* mc_out, double* s_out, bool* bad_out) {
    float m0 = -INFINITY, m1 = -INFINITY;
    bool b0 = false, b1 = false;
    const ChunkStat* cs1 = off2 >= 0 ? cs + off2 : cs;
    for (int q = lane; q < nch; q += kWarp) {
        const ChunkStat x0 = cs[q], x1 = cs1[q];
        m0 = fmaxf(m0, x0.m);
        b0 |= (x0.s != x0.s);
        m1 = fmaxf(m1, x1.m);
        b1 |= (x1.s != x1.s);
    }
    m0 = warp_max(m0);
    m1 = warp_max(m1);
    const float mc0 = __fmul_rn(m0, c), mc1 = __fmul_rn(m1, c);
    double s0 = 0.0, s1 = 0.0;
    for (int q = lane; q < nch; q += kWarp) {
        const ChunkStat x0 = cs[q], x1 = cs1[q];
        if (x0.m != -INFINITY) s0 += (double)x0.s * (double)ex2(__fmul_rn(x0.m, c) - mc0);
        if (x1.m != -INFINITY) s1 += (double)x1.s * (double)ex2(__fmul_rn(x1.m, c) - mc1);
    }
#pragma unroll
    for (int o = kWarp / 2; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
    }
    mc_out[0] = mc0;
    mc_out[1] = mc1;
    s_out[0] = s0;
    s_out[1] = s1;
    bad_out[0] = __any_sync(0xffffffffu, b0) || m0 == -INFINITY || !(s0 > 0.0);
    bad_out[1] = __any_sync(0xffffffffu, b1) || m1 == -INFINITY || !(s1 > 0.0);
}

// One CTA per tree.  A tree's numerator sum_v w(v) (LSE_{d(v)} - z_v / T_d)
// is sum_m LSE_m W_m - (1 / T_d) sum_v w(v) z_v, with W_m the weight on row m
// (Eq. 67).  Both W_m and sum_v w(v) z_v need only this call's inputs, so the
// kernel forms them before it waits for the chunk pass: that pass lets this
// kernel be scheduled only after its own wait, so every input is complete by
// then, and the work overlaps the pass.  After the wait: one warp per row
// forms (mc, S) from the chunk statistics, one warp takes the logarithm of
// every row at once (row m on lane m, L <= 32) and the L products.  The float64
// pipe is narrow (64 clocks a warp instruction), so each float64 step is taken
// once, on full warps where it can be.  W_m is summed by one warp per row over
// the nodes in node order (deterministic, no atomics), reading (depth, weight)
// from global memory rather than staging them in shared memory: this kernel
// launches early behind the persistent chunk pass, and a CTA that needs more
// shared memory than that pass's carveout leaves free waits for its SM to
// drain.  The last CTA to finish (a completion counter; no CTA waits for
// another) forms the scalar loss from the valid trees' numerators and
// (n_nodes - 1).  A tree is malformed when n_nodes or a node's depth or token
// is out of range, and non-finite when some w(v) z_v is, or a row holding a
// node has no finite log-normaliser.
template <typename T>
__global__ void __launch_bounds__(kExitThreads)
exit_tree_kernel(const T* __restrict__ logits, int n_trees, int L, int64_t V, int nch, float c,
                 double temp, double inv_temp, const int32_t* __restrict__ token,
                 const int32_t* __restrict__ depth, const int32_t* __restrict__ n_nodes, int B,
                 const float* __restrict__ omega, double* __restrict__ loss_tree,
                 double* __restrict__ loss, int32_t* __restrict__ status, ExitWs ws) {
    __shared__ double lse[TSD_MAX_L];
    __shared__ double wrow[TSD_MAX_L];
    __shared__ int nrow[TSD_MAX_L];
    __shared__ double srow[TSD_MAX_L];
    __shared__ float mcrow[TSD_MAX_L];
    __shared__ int badrow[TSD_MAX_L];
    __shared__ double red[kExitThreads / kWarp], red2[kExitThreads / kWarp];
    __shared__ int bad, last;
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & (kWarp - 1), wid = tid / kWarp;
    const int nw = blockDim.x / kWarp;
    const int stride = B + 1;
    // ---- before the wait: this call's inputs only ----
    const int n = n_nodes[t];
    if (tid == 0) bad = (n < 1 || n > stride) ? kStatBadTree : kStatOk;
    __syncthreads();
    const int nv = bad == kStatOk ? n : 1;
    double azp = 0.0;  // sum of w(v) z_v over this thread's nodes
    for (int v = 1 + tid; v < nv; v += blockDim.x) {
        const int d = depth[(int64_t)t * stride + v];
        const int x = token[(int64_t)t * stride + v];
        if (d < 1 || d > L || x < 0 || (int64_t)x >= V) {
            atomicExch(&bad, kStatBadTree);
            continue;
        }
        const double w = (double)omega[(int64_t)t * stride + v];
        const double az = w * (double)load_logit(logits + ((int64_t)t * L + d - 1) * V + x);
        if (!(az == az) || isinf(az)) atomicCAS(&bad, kStatOk, kStatNonFinite);
        azp += az;
    }
    azp = warp_sum_d(azp);
    if (lane == 0) red[wid] = azp;
    __syncthreads();
    const int st0 = bad;
    for (int m = wid; m < L; m += nw) {
        double a = 0.0;
        int cnt = 0;
        if (st0 != kStatBadTree)
            for (int v = 1 + lane; v < nv; v += kWarp)
                if (__ldg(depth + (int64_t)t * stride + v) == m + 1) {
                    a += (double)__ldg(omega + (int64_t)t * stride + v);
                    ++cnt;
                }
        a = warp_sum_d(a);
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        if (lane == 0) {
            wrow[m] = a;
            nrow[m] = cnt;
            ws.wrow[(int64_t)t * L + m] = st0 == kStatOk ? a : 0.0;
        }
    }
    // ---- the chunk pass's statistics ----
    pdl_entry();
    // two rows a warp at once (m and m + nw), so that their loads and float64
    // sums overlap
    for (int m = wid; m < L; m += 2 * nw) {
        float mc[2];
        double s[2];
        bool b[2];
        row_stats_pair(ws.rows.chunk + ((int64_t)t * L + m) * nch, m + nw < L ? nw * nch : -1, nch, c,
                       lane, mc, s, b);
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (lane == 0 && m + j * nw < L) {
                mcrow[m + j * nw] = mc[j];
                srow[m + j * nw] = s[j];
                badrow[m + j * nw] = b[j];
            }
    }
    __syncthreads();
    if (wid == 0) {
        double term = 0.0;
        bool nf = false;
        if (lane < L) {
            const double l = badrow[lane] ? __longlong_as_double(0x7ff8000000000000ll)
                                          : 0.6931471805599453 * ((double)mcrow[lane] + log2(srow[lane]));
            lse[lane] = l;
            ws.lse[(int64_t)t * L + lane] = l;
            if (nrow[lane] > 0) {  // a row holding a node contributes LSE_m W_m
                term = l * wrow[lane];
                nf = !(term == term) || isinf(term);
            }
        }
        term = warp_sum_d(term);
        nf = __any_sync(0xffffffffu, nf);
        if (lane == 0) {
            double az = 0.0;
            for (int i = 0; i < nw; ++i) az += red[i];
            int st = bad;
            if (st == kStatOk && nf) st = kStatNonFinite;
            const double num = term - az * inv_temp;
            loss_tree[t] = st == kStatOk ? num : 0.0;
            status[t] = st;
            ws.tstat[t] = st;
            if (st != kStatOk)
                for (int m = 0; m < L; ++m) ws.wrow[(int64_t)t * L + m] = 0.0;
        }
    }
    // completion: the last CTA reads every tree's results
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(ws.done, 1u) == (unsigned)n_trees - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    double a = 0.0, b2 = 0.0;
    for (int u = tid; u < n_trees; u += blockDim.x) {
        const int su = *(volatile const int32_t*)(ws.tstat + u);
        if (su == kStatOk) {
            a += *(volatile const double*)(loss_tree + u);
            b2 += (double)(n_nodes[u] - 1);
        }
    }
    a = warp_sum_d(a);
    b2 = warp_sum_d(b2);
    if (lane == 0) {
        red[wid] = a;
        red2[wid] = b2;
    }
    __syncthreads();
    if (tid == 0) {
        double A = 0.0, Bn = 0.0;
        for (int i = 0; i < nw; ++i) {
            A += red[i];
            Bn += red2[i];
        }
        ws.norm[0] = Bn;
        ws.norm[1] = Bn > 0.0 ? 1.0 / (temp * Bn) : 0.0;  // the gradient's factor, formed once
        *loss = Bn > 0.0 ? A / Bn : 0.0;
    }
}

template <typename T>
__global__ void __launch_bounds__(kExitThreads)
exit_grad_kernel(const T* __restrict__ logits, int64_t rows, int L, int64_t V, int nch, float c,
                 float* __restrict__ grad, ExitWs ws) {
    pdl_entry();
    constexpr int VEC = Lanes<T>::kVec;
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    const int lane = threadIdx.x & (kWarp - 1);
    const double nrm = ws.norm[0], inv = ws.norm[1];
    const bool vec = ((uintptr_t)logits % 16 == 0) && ((V * (int64_t)sizeof(T)) % 16 == 0) &&
                     ((uintptr_t)grad % 16 == 0);
    const int64_t total = rows * nch;
    const int wpb = blockDim.x / kWarp;
    for (int64_t item = (int64_t)blockIdx.x * wpb + threadIdx.x / kWarp; item < total;
         item += (int64_t)gridDim.x * wpb) {
        const int64_t row = item / nch;
        const int64_t c0 = (item - row * nch) * (int64_t)CE;
        const int cn = (int)min((int64_t)CE, V - c0);
        const int t = (int)(row / L);
        const double wr = ws.wrow[row];
        float* g = grad + row * V + c0;
        const T* z = logits + row * V + c0;
        const bool zero = ws.tstat[t] != kStatOk || wr == 0.0 || !(nrm > 0.0);
        const float scale = zero ? 0.0f : (float)(wr * inv);
        const float l2 = zero ? 0.0f : (float)(ws.lse[row] * 1.4426950408889634);
        if (vec) {
            uint4 buf[kVecPerLane];
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int e = (i * kWarp + lane) * VEC;
                buf[i] = (!zero && e < cn) ? ld_stream16(z + e) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int e = (i * kWarp + lane) * VEC;
                if (e < cn) {
#pragma unroll
                    for (int j = 0; j < VEC; j += 4) {
                        float4 o;
                        o.x = zero ? 0.0f : scale * ex2(fmaf(Lanes<T>::get(buf[i], j), c, -l2));
                        o.y = zero ? 0.0f : scale * ex2(fmaf(Lanes<T>::get(buf[i], j + 1), c, -l2));
                        o.z = zero ? 0.0f : scale * ex2(fmaf(Lanes<T>::get(buf[i], j + 2), c, -l2));
                        o.w = zero ? 0.0f : scale * ex2(fmaf(Lanes<T>::get(buf[i], j + 3), c, -l2));
                        __stcs(reinterpret_cast<float4*>(g + e + j), o);
                    }
                }
            }
        } else {
            for (int e = lane; e < cn; e += kWarp)
                g[e] = zero ? 0.0f : scale * ex2(fmaf(load_logit(z + e), c, -l2));
        }
    }
}

// The gathered part: grad[row(v)][x_v] -= w(v) / (T_d N) for every node.
__global__ void __launch_bounds__(kExitThreads)
exit_scatter_kernel(int n_trees, int L, int64_t V, const int32_t* __restrict__ token,
                    const int32_t* __restrict__ depth, const int32_t* __restrict__ n_nodes, int B,
                    const float* __restrict__ omega, float* __restrict__ grad, ExitWs ws) {
    pdl_entry();
    const double nrm = ws.norm[0], inv = ws.norm[1];
    const int64_t total = (int64_t)n_trees * (B + 1);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / (B + 1)), v = (int)(i - (int64_t)t * (B + 1));
        if (v == 0 || v >= n_nodes[t] || ws.tstat[t] != kStatOk || !(nrm > 0.0)) continue;
        const int d = depth[i], x = token[i];
        if (!(TSD_IN(d - 1, L, kChkExit) && TSD_IN(x, V, kChkExit))) continue;
        atomicAdd(grad + ((int64_t)t * L + d - 1) * V + x, (float)(-(double)omega[i] * inv));
    }
}

cudaError_t launch_exit_loss(const void* logits, tsd_dtype dtype, int n_trees, int L, int64_t V,
                             float c, double temp, const int32_t* token, const int32_t* depth,
                             const int32_t* n_nodes, int B, const float* omega, double* loss_tree,
                             double* loss, float* grad, int32_t* status, const ExitWs& ws,
                             cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    const int64_t rows = (int64_t)n_trees * L;
    // the per-tree kernel's completion counter starts at zero on every call
    if (cudaError_t e = cudaMemsetAsync(ws.done, 0, sizeof(unsigned), stream); e != cudaSuccess)
        return e;
    if (cudaError_t e = launch_drafter_chunks(logits, dtype, rows, V, c, ws.rows, stream);
        e != cudaSuccess)
        return e;
    const double inv_temp = 1.0 / temp;  // z / T_d as one multiply per node
    cudaError_t e;
    if (dtype == TSD_BF16)
        e = launch_pdl(exit_tree_kernel<__nv_bfloat16>, (unsigned)n_trees, kExitThreads, 0, stream,
                       static_cast<const __nv_bfloat16*>(logits), n_trees, L, V, nch, c, temp, inv_temp,
                       token, depth, n_nodes, B, omega, loss_tree, loss, status, ws);
    else
        e = launch_pdl(exit_tree_kernel<float>, (unsigned)n_trees, kExitThreads, 0, stream,
                       static_cast<const float*>(logits), n_trees, L, V, nch, c, temp, inv_temp, token,
                       depth, n_nodes, B, omega, loss_tree, loss, status, ws);
    if (e != cudaSuccess) return e;
    if (grad) {
        int dev = 0, sms = 152;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int wpb = kExitThreads / kWarp;
        const int64_t want = (rows * nch + wpb - 1) / wpb;
        const int64_t cap = (int64_t)sms * 8;
        const unsigned g2 = (unsigned)(want < cap ? want : cap);
        if (dtype == TSD_BF16)
            e = launch_pdl(exit_grad_kernel<__nv_bfloat16>, g2, kExitThreads, 0, stream,
                           static_cast<const __nv_bfloat16*>(logits), rows, L, V, nch, c, grad,
                           ws);
        else
            e = launch_pdl(exit_grad_kernel<float>, g2, kExitThreads, 0, stream,
                           static_cast<const float*>(logits), rows, L, V, nch, c, grad, ws);
        if (e != cudaSuccess) return e;
        const int64_t nodes = (int64_t)n_trees * (B + 1);
        const int64_t gs = (nodes + kExitThreads - 1) / kExitThreads;
        if ((e = launch_pdl(exit_scatter_kernel, (unsigned)(gs < 65535 ? (gs > 0 ? gs : 1) : 65535),
                            kExitThreads, 0, stream, n_trees, L, V, token, depth, n_nodes, B,
                            omega, grad, ws)) != cudaSuccess)
            return e;
    }
    return cudaGetLastError();
}

TSD_CHECK_READER(checks_exit)

}  // namespace tsd
