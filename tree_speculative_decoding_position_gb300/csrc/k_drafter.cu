// k_drafter.cu -- drafter row statistics for the tree builder.
//
// "CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters", Sec. 2
// Eq. 1 (prefixes ranked by the product of the drafter's per-position
// probabilities) and App. C "Candidate construction" (keep the top-K tokens of
// each future position; scores use the original q_j, not a top-K
// renormalisation).  For every row j of drafter logits this computes
//   LSE_j = log sum_a exp(z_j(a) / T_d)      (over the full vocabulary)
//   the top-k tokens by (logit desc, id asc) with their z / T_d; the builder
//   scores a prefix as (sum of its z / T_d) - (sum of the rows' LSE), which
//   is its sum of log q_j = z / T_d - LSE_j.
//
// drafter_chunk_kernel  one warp per (row, 8 KB chunk): chunk max, sum of
//                       exp2(z*c - mc), and the chunk's top-k.
// drafter_row_kernel    one warp per row: merges the chunk lists into the
//                       row's top-k, and the chunk sums into its LSE.
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

constexpr int kCandCap = 256;  // candidates per warp before the exact fallback
constexpr int kMaxListsPerLane = kMaxDrafterChunks / kWarp;

// Exact fallback for a chunk whose candidate set overflowed (e.g. a row of
// many equal logits): offer every token to the warp list, in a plain loop.
template <typename T>
__device__ __noinline__ void chunk_topk_fallback(const T* __restrict__ rp, int cn, int64_t c0,
                                                 int k, int lane, float& ev, int& ei) {
    float tv = -INFINITY;
    int ti = INT_MAX;
    ev = -INFINITY;
    ei = INT_MAX;
    for (int e0 = 0; e0 < cn; e0 += kWarp) {
        const int e = e0 + lane;
        const float x = e < cn ? load_logit(rp + e) : -INFINITY;
        warp_list_offer(ev, ei, tv, ti, e < cn, x, (int)c0 + e, k, lane);
    }
}

// Sort one float per lane, descending, across the warp (bitonic).
__device__ __forceinline__ float warp_sort_desc(float x, int lane) {
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1) {
#pragma unroll
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            const float y = __shfl_xor_sync(0xffffffffu, x, j);
            const bool lower = (lane & j) == 0;
            const bool desc = (lane & k2) == 0;
            // keep the larger value on the lower lane of a descending block
            x = (lower == desc) ? fmaxf(x, y) : fminf(x, y);
        }
    }
    return x;
}

// Sort one (value, id) pair per lane across the warp into (value desc, id
// asc) order (bitonic; lane 0 ends with the best).
__device__ __forceinline__ void warp_sort_pairs(float& v, int& id, int lane) {
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1) {
#pragma unroll
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, j);
            const int oi = __shfl_xor_sync(0xffffffffu, id, j);
            const bool lower = (lane & j) == 0;
            const bool first = (lane & k2) == 0;  // this block ends up best-first
            const bool mine_first = better(v, id, ov, oi);
            if ((lower == first) != mine_first) {
                v = ov;
                id = oi;
            }
        }
    }
}

// One warp per (row, 8 KB chunk).  Pass 1: the chunk max, the sum of
// exp2(z*c - mc) and each vector's max.  Threshold: the k-th largest of the 32
// lane maxima -- k distinct tokens reach it, so every token of the chunk's
// top-k does too.  Pass 2: only vectors whose max reaches the threshold are
// opened; their qualifying tokens go to a per-warp shared list.  Then k rounds
// of warp arg-max pick the top-k by (logit desc, id asc).
template <typename T>
__global__ void __launch_bounds__(kDThreads)
drafter_chunk_kernel(const T* __restrict__ logits, int64_t rows, int64_t V, int nch, int k,
                     float c, bool vec_ok, BuildWs ws) {
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    constexpr int VEC = 16 / (int)sizeof(T);
    __shared__ float cand_v[kDThreads / kWarp][kCandCap];
    __shared__ int cand_i[kDThreads / kWarp][kCandCap];
    __shared__ int cand_n[kDThreads / kWarp];
    const int lane = threadIdx.x & (kWarp - 1);
    const int wid = threadIdx.x / kWarp;
    const int wpb = blockDim.x / kWarp;
    const int64_t total = rows * nch;
    for (int64_t item = (int64_t)blockIdx.x * wpb + wid; item < total;
         item += (int64_t)gridDim.x * wpb) {
        const int64_t row = item / nch;
        const int ch = (int)(item - row * nch);
        const int64_t c0 = (int64_t)ch * CE;
        const int cn = (int)min((int64_t)CE, V - c0);
        const T* rp = logits + row * V + c0;
        float m = -INFINITY, s = 0.0f, lm = -INFINITY;
        float ev = -INFINITY;
        int ei = INT_MAX;
        if (lane == 0) cand_n[wid] = 0;
        __syncwarp();
        if (vec_ok) {
            uint4 buf[kVecPerLane];
            float vmax[kVecPerLane];
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int e = (i * kWarp + lane) * VEC;
                const uint32_t ninf = sizeof(T) == 2 ? 0xff80ff80u : 0xff800000u;
                buf[i] = (e < cn) ? ld_stream16(rp + e) : make_uint4(ninf, ninf, ninf, ninf);
            }
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                if (sizeof(T) == 2) {
                    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&buf[i].x);
                    a = __hmax2(a, *reinterpret_cast<const __nv_bfloat162*>(&buf[i].y));
                    a = __hmax2(a, *reinterpret_cast<const __nv_bfloat162*>(&buf[i].z));
                    a = __hmax2(a, *reinterpret_cast<const __nv_bfloat162*>(&buf[i].w));
                    vmax[i] = fmaxf(__low2float(a), __high2float(a));
                } else {
                    vmax[i] = fmaxf(fmaxf(__uint_as_float(buf[i].x), __uint_as_float(buf[i].y)),
                                    fmaxf(__uint_as_float(buf[i].z), __uint_as_float(buf[i].w)));
                }
                lm = fmaxf(lm, vmax[i]);
            }
            m = warp_max(lm);
            const float mc = __fmul_rn(m, c);
            if (m != -INFINITY) {
                float acc[VEC];
#pragma unroll
                for (int j = 0; j < VEC; ++j) acc[j] = 0.0f;
#pragma unroll
                for (int i = 0; i < kVecPerLane; ++i)
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const uint32_t w = j / (VEC / 4) == 0 ? buf[i].x : j / (VEC / 4) == 1 ? buf[i].y
                                           : j / (VEC / 4) == 2 ? buf[i].z : buf[i].w;
                        const float x = sizeof(T) == 2 ? ((j & 1) ? bf16_hi(w) : bf16_lo(w))
                                                       : __uint_as_float(w);
                        acc[j] += ex2(fmaf(x, c, -mc));
                    }
#pragma unroll
                for (int j = 0; j < VEC; ++j) s += acc[j];
            }
            const float theta = __shfl_sync(0xffffffffu, warp_sort_desc(lm, lane), k - 1);
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int e = (i * kWarp + lane) * VEC;
                if (e < cn && vmax[i] >= theta) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        const uint32_t w = j / (VEC / 4) == 0 ? buf[i].x : j / (VEC / 4) == 1 ? buf[i].y
                                           : j / (VEC / 4) == 2 ? buf[i].z : buf[i].w;
                        const float x = sizeof(T) == 2 ? ((j & 1) ? bf16_hi(w) : bf16_lo(w))
                                                       : __uint_as_float(w);
                        if (x >= theta) {
                            const int pos = atomicAdd(&cand_n[wid], 1);
                            if (pos < kCandCap) {
                                cand_v[wid][pos] = x;
                                cand_i[wid][pos] = (int)c0 + e + j;
                            }
                        }
                    }
                }
            }
        } else {
            for (int e = lane; e < cn; e += kWarp) lm = fmaxf(lm, load_logit(rp + e));
            m = warp_max(lm);
            const float mc = __fmul_rn(m, c);
            if (m != -INFINITY)
                for (int e = lane; e < cn; e += kWarp) s += ex2(fmaf(load_logit(rp + e), c, -mc));
            const float theta = __shfl_sync(0xffffffffu, warp_sort_desc(lm, lane), k - 1);
            for (int e = lane; e < cn; e += kWarp) {
                const float x = load_logit(rp + e);
                if (x >= theta) {
                    const int pos = atomicAdd(&cand_n[wid], 1);
                    if (pos < kCandCap) {
                        cand_v[wid][pos] = x;
                        cand_i[wid][pos] = (int)c0 + e;
                    }
                }
            }
        }
        __syncwarp();
        const int nc = cand_n[wid];
        if (nc > kCandCap) {
            chunk_topk_fallback<T>(rp, cn, c0, k, lane, ev, ei);
        } else if (nc <= kWarp) {
            // the usual case: one warp sort of the candidates
            ev = lane < nc ? cand_v[wid][lane] : -INFINITY;
            ei = lane < nc ? cand_i[wid][lane] : INT_MAX;
            warp_sort_pairs(ev, ei, lane);
        } else {
            // k rounds of arg-max over the candidates; a taken one becomes
            // (-inf, INT_MAX), which every real token beats.
            for (int r = 0; r < k; ++r) {
                float bv = -INFINITY;
                int bi = INT_MAX, bp = -1;
                for (int q = lane; q < nc; q += kWarp)
                    if (better(cand_v[wid][q], cand_i[wid][q], bv, bi)) {
                        bv = cand_v[wid][q];
                        bi = cand_i[wid][q];
                        bp = q;
                    }
                float wv = bv;
                int wi = bi;
                warp_argmax(wv, wi);
                if (lane == r) {
                    ev = wv;
                    ei = wi;
                }
                if (wi != INT_MAX && bi == wi) {
                    cand_v[wid][bp] = -INFINITY;
                    cand_i[wid][bp] = INT_MAX;
                }
                __syncwarp();
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
        __syncwarp();
    }
}

constexpr int kRowStage = 1024;  // candidates staged in shared memory per warp

// One warp per row: the row's log-normaliser from its chunk sums (float64),
// and its top-k merged from the chunks' sorted lists.  The lists are first
// copied to shared memory in one coalesced pass (when they fit), then lane l
// walks the lists of chunks l, l+32, ...; k rounds of warp arg-max over the
// lanes' current heads.
__global__ void __launch_bounds__(kDThreads)
drafter_row_kernel(int64_t rows, int nch, int k, float c, double temp, BuildWs ws) {
    __shared__ float sv[kDThreads / kWarp][kRowStage];
    __shared__ int si[kDThreads / kWarp][kRowStage];
    const int lane = threadIdx.x & (kWarp - 1);
    const int wid = threadIdx.x / kWarp;
    const int wpb = blockDim.x / kWarp;
    for (int64_t row = (int64_t)blockIdx.x * wpb + wid; row < rows;
         row += (int64_t)gridDim.x * wpb) {
        const ChunkStat* cs = ws.chunk + row * nch;
        const int ncand = nch * k;
        const bool staged = ncand <= kRowStage;
        const float* gv = ws.cand_v + row * ncand;
        const int* gi = ws.cand_i + row * ncand;
        if (staged)
            for (int q = lane; q < ncand; q += kWarp) {
                sv[wid][q] = gv[q];
                si[wid][q] = gi[q];
            }
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
        __syncwarp();
        const float* cv = staged ? sv[wid] : gv;
        const int* ci = staged ? si[wid] : gi;
        int pos[kMaxListsPerLane];
        const int nj = (nch + kWarp - 1) / kWarp;
        for (int j = 0; j < nj; ++j) pos[j] = 0;
        float ev = -INFINITY;
        int ei = INT_MAX;
        for (int r = 0; r < k; ++r) {
            float hv = -INFINITY;
            int hi = INT_MAX, hj = -1;
            for (int j = 0; j < nj; ++j) {
                const int q = lane + kWarp * j;
                const int p = pos[j];
                if (q < nch && p < k) {
                    const float x = cv[q * k + p];
                    const int xi = ci[q * k + p];
                    if (xi != INT_MAX && better(x, xi, hv, hi)) {
                        hv = x;
                        hi = xi;
                        hj = j;
                    }
                }
            }
            float wv = hv;
            int wi = hi;
            warp_argmax(wv, wi);
            if (lane == r) {
                ev = wv;
                ei = wi;
            }
            if (wi != INT_MAX && hi == wi) ++pos[hj];
        }
        if (lane < k) {
            ws.top_id[row * k + lane] = ei;
            ws.top_zt[row * k + lane] = (double)ev / temp;
        }
        if (lane == 0) ws.lse[row] = lse;
        __syncwarp();
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
