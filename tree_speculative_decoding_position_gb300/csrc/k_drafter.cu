// k_drafter.cu -- drafter row statistics for the tree builder.
//
// "CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters", Sec. 2
// Eq. 1 (prefixes ranked by the product of the drafter's per-position
// probabilities) and App. C "Candidate construction" (keep the top-K tokens of
// each future position; scores use the original q_j, not a top-K
// renormalisation).  For every row j of drafter logits this computes
//   LSE_j = log sum_a exp(z_j(a) / T_d)      (over the full vocabulary)
//   the top-k tokens by (logit desc, id asc) and log q_j = z / T_d - LSE_j.
//
// drafter_chunk_kernel  one warp per (row, 8 KB chunk): chunk max, sum of
//                       exp2(z*c - mc), and the chunk's top-k, kept as a
//                       warp-distributed sorted list (lane i holds the i-th
//                       best) that a candidate enters by one shuffle step.
// drafter_row_kernel    one warp per row: merges the chunk lists and sums.
#include "tsd_internal.cuh"

namespace tsd {

constexpr int kDThreads = 256;

// Insert (x, xi) into the warp-distributed list (ev, ei) sorted by
// (value desc, id asc) over lanes [0, k).  No-op if (x, xi) is not better
// than the k-th entry.
__device__ __forceinline__ void warp_list_insert(float& ev, int& ei, float x, int xi, int k,
                                                 int lane) {
    const float pv = __shfl_up_sync(0xffffffffu, ev, 1);
    const int pi = __shfl_up_sync(0xffffffffu, ei, 1);
    if (lane < k) {
        const bool above_prev = lane > 0 && better(x, xi, pv, pi);
        if (above_prev) {
            ev = pv;
            ei = pi;
        } else if (better(x, xi, ev, ei)) {
            ev = x;
            ei = xi;
        }
    }
}

// Offer one candidate per lane (`has` marks lanes that have one); candidates
// enter the list one at a time in lane order.  Updates the threshold (the
// k-th entry).
__device__ __forceinline__ void warp_list_offer(float& ev, int& ei, float& tv, int& ti, bool has,
                                                float x, int xi, int k, int lane) {
    unsigned m = __ballot_sync(0xffffffffu, has && better(x, xi, tv, ti));
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const float cx = __shfl_sync(0xffffffffu, x, src);
        const int ci = __shfl_sync(0xffffffffu, xi, src);
        warp_list_insert(ev, ei, cx, ci, k, lane);
        tv = __shfl_sync(0xffffffffu, ev, k - 1);
        ti = __shfl_sync(0xffffffffu, ei, k - 1);
    }
}

template <typename T>
__global__ void __launch_bounds__(kDThreads)
drafter_chunk_kernel(const T* __restrict__ logits, int64_t rows, int64_t V, int nch, int k,
                     float c, bool vec_ok, BuildWs ws) {
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    constexpr int VEC = 16 / (int)sizeof(T);
    const int lane = threadIdx.x & (kWarp - 1);
    const int wpb = blockDim.x / kWarp;
    const int64_t total = rows * nch;
    for (int64_t item = (int64_t)blockIdx.x * wpb + threadIdx.x / kWarp; item < total;
         item += (int64_t)gridDim.x * wpb) {
        const int64_t row = item / nch;
        const int ch = (int)(item - row * nch);
        const int64_t c0 = (int64_t)ch * CE;
        const int cn = (int)min((int64_t)CE, V - c0);
        const T* rp = logits + row * V + c0;
        float ev = -INFINITY, tv = -INFINITY;
        int ei = INT_MAX, ti = INT_MAX;
        float m = -INFINITY, s = 0.0f;
        if (vec_ok) {
            uint4 buf[kVecPerLane];
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int e = (i * kWarp + lane) * VEC;
                const uint32_t ninf = sizeof(T) == 2 ? 0xff80ff80u : 0xff800000u;
                buf[i] = (e < cn) ? ld_stream16(rp + e) : make_uint4(ninf, ninf, ninf, ninf);
            }
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i)
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const uint32_t w = j / (VEC / 4) == 0 ? buf[i].x : j / (VEC / 4) == 1 ? buf[i].y
                                       : j / (VEC / 4) == 2 ? buf[i].z : buf[i].w;
                    const float x = sizeof(T) == 2 ? ((j & 1) ? bf16_hi(w) : bf16_lo(w))
                                                   : __uint_as_float(w);
                    m = fmaxf(m, x);
                }
            m = warp_max(m);
            const float mc = __fmul_rn(m, c);
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int e = (i * kWarp + lane) * VEC;
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const uint32_t w = j / (VEC / 4) == 0 ? buf[i].x : j / (VEC / 4) == 1 ? buf[i].y
                                       : j / (VEC / 4) == 2 ? buf[i].z : buf[i].w;
                    const float x = sizeof(T) == 2 ? ((j & 1) ? bf16_hi(w) : bf16_lo(w))
                                                   : __uint_as_float(w);
                    if (m != -INFINITY) s += ex2(fmaf(x, c, -mc));
                    warp_list_offer(ev, ei, tv, ti, e < cn, x, (int)c0 + e + j, k, lane);
                }
            }
        } else {
            for (int e = lane; e < cn; e += kWarp) m = fmaxf(m, load_logit(rp + e));
            m = warp_max(m);
            const float mc = __fmul_rn(m, c);
            for (int e0 = 0; e0 < cn; e0 += kWarp) {
                const int e = e0 + lane;
                const float x = e < cn ? load_logit(rp + e) : -INFINITY;
                if (e < cn && m != -INFINITY) s += ex2(fmaf(x, c, -mc));
                warp_list_offer(ev, ei, tv, ti, e < cn, x, (int)c0 + e, k, lane);
            }
        }
        s = warp_sum(s);
        if (lane == 0) {
            ChunkStat st;
            st.m = m;
            st.s = s;
            st.r = 0.0f;
            st.amax = -1;
            ws.chunk[item] = st;
        }
        if (lane < k) {
            ws.cand_v[item * k + lane] = ev;
            ws.cand_i[item * k + lane] = ei;
        }
    }
}

__global__ void __launch_bounds__(kDThreads)
drafter_row_kernel(int64_t rows, int nch, int k, float c, double temp, BuildWs ws) {
    const int lane = threadIdx.x & (kWarp - 1);
    const int wpb = blockDim.x / kWarp;
    for (int64_t row = (int64_t)blockIdx.x * wpb + threadIdx.x / kWarp; row < rows;
         row += (int64_t)gridDim.x * wpb) {
        const ChunkStat* cs = ws.chunk + row * nch;
        float m = -INFINITY;
        bool bad = false;
        for (int q = lane; q < nch; q += kWarp) {
            m = fmaxf(m, cs[q].m);
            bad |= (cs[q].s != cs[q].s);
        }
        m = warp_max(m);
        const float mc = __fmul_rn(m, c);
        double s = 0.0;
        for (int q = lane; q < nch; q += kWarp)
            if (cs[q].m != -INFINITY) s += (double)cs[q].s * (double)ex2(__fmul_rn(cs[q].m, c) - mc);
        s = warp_sum_d(s);
        bad = __any_sync(0xffffffffu, bad) || m == -INFINITY || !(s > 0.0);
        // LSE_j = ln 2 * (mc + log2 S), all relative to the same reference mc.
        const double lse = bad ? __longlong_as_double(0x7ff8000000000000ll)
                               : 0.6931471805599453 * ((double)mc + log2(s));
        float ev = -INFINITY, tv = -INFINITY;
        int ei = INT_MAX, ti = INT_MAX;
        for (int q = 0; q < nch; ++q) {
            const bool has = lane < k;
            const float x = has ? ws.cand_v[(row * nch + q) * k + lane] : -INFINITY;
            const int xi = has ? ws.cand_i[(row * nch + q) * k + lane] : INT_MAX;
            warp_list_offer(ev, ei, tv, ti, has && xi != INT_MAX, x, xi, k, lane);
        }
        if (lane < k) {
            ws.top_id[row * k + lane] = ei;
            ws.top_lq[row * k + lane] = (double)ev / temp - lse;
        }
    }
}

cudaError_t launch_drafter_stats(const void* logits, tsd_dtype dtype, int64_t rows, int64_t V,
                                 int topk, float c, double temp, const BuildWs& ws,
                                 cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    const bool vec_ok = ((uintptr_t)logits % 16 == 0) && ((V * es) % 16 == 0);
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int wpb = kDThreads / kWarp;
    int64_t want = (rows * nch + wpb - 1) / wpb;
    int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    if (dtype == TSD_BF16)
        drafter_chunk_kernel<__nv_bfloat16><<<grid, kDThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(logits), rows, V, nch, topk, c, vec_ok, ws);
    else
        drafter_chunk_kernel<float><<<grid, kDThreads, 0, stream>>>(
            static_cast<const float*>(logits), rows, V, nch, topk, c, vec_ok, ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    want = (rows + wpb - 1) / wpb;
    grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    drafter_row_kernel<<<grid, kDThreads, 0, stream>>>(rows, nch, topk, c, temp, ws);
    return cudaGetLastError();
}

}  // namespace tsd
