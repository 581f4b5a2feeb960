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
// drafter_chunk_kernel  one warp per (row, 8 KB chunk), streaming: the chunk
//                       max, the sum of exp2(z*c - mc), and the maximum of
//                       each lane's slice of the chunk.
// drafter_row_kernel    one CTA per row: the LSE from the chunk sums; a
//                       bound theta <= the row's k-th largest logit (the k-th
//                       largest chunk maximum: k distinct chunks each hold a
//                       token at or above it); then only the lane slices
//                       whose maximum reaches theta are read again, and their
//                       tokens at or above theta give the exact top-k.
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

// Lane l's slice of a chunk: on the vectorised path the 16-byte vectors
// i*32 + l (i = 0..15); otherwise the tokens l, l+32, ....

// One warp per (row, 8 KB chunk), persistent over a grid stride.  Writes the
// chunk max and sum of exp2(z*c - mc) (ChunkStat) and the 32 lane-slice
// maxima.  On the vectorised path the next chunk's loads are issued as soon
// as the current chunk's per-lane work is done, so the warp sum and the
// stores overlap them; positions advance by carries.
template <typename T>
__global__ void __launch_bounds__(kDThreads)
drafter_chunk_kernel(const T* __restrict__ logits, int64_t rows, int64_t V, int nch, float c,
                     bool vec_ok, BuildWs ws) {
    pdl_entry();
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    constexpr int VEC = Lanes<T>::kVec;
    const int lane = threadIdx.x & (kWarp - 1);
    const int wpb = blockDim.x / kWarp;
    const int64_t total = rows * nch;
    const int64_t stride = (int64_t)gridDim.x * wpb;
    int64_t item = (int64_t)blockIdx.x * wpb + threadIdx.x / kWarp;
    if (item >= total) return;
    int64_t row = item / nch;
    int ch = (int)(item - row * nch);
    const int64_t drow = stride / nch;
    const int dch = (int)(stride - drow * nch);
    auto advance = [&]() {
        item += stride;
        ch += dch;
        const int carry = ch >= nch;
        ch -= carry ? nch : 0;
        row += drow + carry;
    };
    auto store = [&](int64_t it, float m, float s_lane, float lm) {
        const float s = warp_sum(s_lane);
        if (lane == 0) {
            ChunkStat st;
            st.m = m;
            st.s = s;
            st.r = 0.0f;
            st.amax = -1;
            ws.chunk[it] = st;
        }
        ws.lane_max[it * kWarp + lane] = lm;
    };

    if (!vec_ok) {  // unaligned rows or ragged V: element loads
        for (; item < total; advance()) {
            const int64_t c0 = (int64_t)ch * CE;
            const int cn = (int)min((int64_t)CE, V - c0);
            const T* rp = logits + row * V + c0;
            float lm = -INFINITY, s = 0.0f;
            for (int e = lane; e < cn; e += kWarp) lm = fmaxf(lm, load_logit(rp + e));
            const float m = warp_max(lm);
            const float mc = __fmul_rn(m, c);
            if (m != -INFINITY)
                for (int e = lane; e < cn; e += kWarp) s += ex2(fmaf(load_logit(rp + e), c, -mc));
            store(item, m, s, lm);
        }
        return;
    }

    uint4 buf[kVecPerLane];
    auto load = [&]() {
        const int64_t c0 = (int64_t)ch * CE;
        const bool in = TSD_IN(row, rows, kChkDrafter) && TSD_IN(ch, nch, kChkDrafter);
        const int cn = in ? (int)min((int64_t)CE, V - c0) : 0;
        const T* rp = logits + row * V + c0;
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) {
            const int e = (i * kWarp + lane) * VEC;
            buf[i] = (e < cn) ? ld_stream16(rp + e) : Lanes<T>::neg_inf();
        }
    };
    load();
    for (;;) {
        const float lm = Lanes<T>::block_max(buf);
        const float m = warp_max(lm);
        float s = 0.0f;
        if (m != -INFINITY) {
            const float mc = __fmul_rn(m, c);
            constexpr int NP = VEC / 2;
            const float2 cc = make_float2(c, c), nmc = make_float2(-mc, -mc);
            float2 acc[NP];
#pragma unroll
            for (int p = 0; p < NP; ++p) acc[p] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i)
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    const float2 y = __ffma2_rn(Lanes<T>::pair(buf[i], p), cc, nmc);
                    acc[p] = __fadd2_rn(acc[p], make_float2(ex2(y.x), ex2(y.y)));
                }
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                s += acc[p].x;
                s += acc[p].y;
            }
        }
        const int64_t cur = item;
        advance();
        if (item < total) load();
        store(cur, m, s, lm);
        if (item >= total) break;
    }
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

constexpr int kRThreads = 256;   // one CTA per drafter row
constexpr int kRTopThreads = kRThreads - kWarp;  // the warps that find the top-k (the last forms the LSE)
constexpr int kSliceCap = 2048;  // qualifying lane slices listed per row
constexpr int kRowCandCap = 1024;

// One CTA per row.  (1) The chunk statistics go to shared memory; theta =
// the k-th largest chunk maximum in (value desc, id asc) order, found by
// ranking every chunk maximum against the others (-inf when the row has fewer
// than k chunks).  (2) The slice maxima of every chunk whose maximum reaches
// theta are read at once; the slices reaching theta are listed.  (3) All
// 16-byte vectors (or tokens) of the listed slices are read at once, and the
// tokens at or above theta are listed.  Every token of the row's top-k is at
// or above theta, so (4) warp 0 selecting the top-k of that list by (logit
// desc, id asc) is exact.  A row whose lists overflow (many equal logits) is
// scanned token by token instead, still exactly.  The last warp leaves after
// (1) and forms the log-normaliser from the chunk sums in float64 (a chain of
// about 3k clocks on this GPU's narrow float64 pipe) while the others run
// (2)-(4) among themselves on a named barrier.
template <typename T>
__global__ void __launch_bounds__(kRThreads)
drafter_row_kernel(const T* __restrict__ logits, int64_t rows, int64_t V, int nch, int k, float c,
                   double temp, bool vec_ok, BuildWs ws) {
    pdl_entry();
    constexpr int CE = kChunkBytes / (int)sizeof(T);
    constexpr int VEC = Lanes<T>::kVec;
    __shared__ float cm[kMaxDrafterChunks];
    __shared__ int qlist[kMaxDrafterChunks];
    __shared__ int slist[kSliceCap];
    __shared__ float cand_v[kRowCandCap];
    __shared__ int cand_i[kRowCandCap];
    __shared__ float wmax[kRThreads / kWarp];
    __shared__ int wbad[kRThreads / kWarp];
    __shared__ int n_q, n_s, n_c;
    __shared__ float s_theta;
    const int tid = threadIdx.x, lane = tid & (kWarp - 1), wid = tid / kWarp;
    const int64_t row = blockIdx.x;
    const ChunkStat* cs = ws.chunk + row * nch;
    if (tid == 0) {
        n_q = 0;
        n_s = 0;
        n_c = 0;
        s_theta = -INFINITY;
    }
    // (1) chunk maxima, the row maximum, NaN sums
    float mloc = -INFINITY;
    bool bad = false;
    for (int q = tid; q < nch; q += kRThreads) {
        const ChunkStat st = cs[q];
        cm[q] = st.m;
        mloc = fmaxf(mloc, st.m);
        bad |= (st.s != st.s);
    }
    mloc = warp_max(mloc);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        wmax[wid] = mloc;
        wbad[wid] = bad;
    }
    __syncthreads();
    float m = -INFINITY;
    bad = false;
#pragma unroll
    for (int w = 0; w < kRThreads / kWarp; ++w) {
        m = fmaxf(m, wmax[w]);
        bad |= wbad[w] != 0;
    }
    if (wid == kRThreads / kWarp - 1) {  // the log-normaliser, beside (2)-(4)
        const float mc = __fmul_rn(m, c);
        double sum = 0.0;
        for (int q = lane; q < nch; q += kWarp)
            if (cm[q] != -INFINITY) sum += (double)cs[q].s * (double)ex2(__fmul_rn(cm[q], c) - mc);
        sum = warp_sum_d(sum);
        if (lane == 0) {
            const bool b = bad || m == -INFINITY || !(sum > 0.0);
            // LSE_j = ln 2 * (mc + log2 S), all relative to the same reference mc.
            // The exponents are float32, so the result can fall a few 1e-6
            // below the largest z / T_d, which the exact value never does: it
            // is raised to that floor (every kept token's log q is then <= 0).
            const double l = 0.6931471805599453 * ((double)mc + log2(sum));
            const double zmax = temp == 1.0 ? (double)m : (double)m / temp;
            ws.lse[row] = b ? __longlong_as_double(0x7ff8000000000000ll) : (l > zmax ? l : zmax);
        }
        return;
    }
    auto top_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kRTopThreads) : "memory"); };
    for (int q = tid; q < nch; q += kRTopThreads) {
        const float v = cm[q];
        if (v != v) continue;  // a NaN maximum ranks nowhere
        int rank = 0;
        for (int p = 0; p < nch; ++p) {
            const float w = cm[p];
            rank += (w > v) || (w == v && p < q);
        }
        if (rank == k - 1) s_theta = v;
    }
    top_sync();
    const float theta = s_theta;
    for (int q = tid; q < nch; q += kRTopThreads)
        if (cm[q] >= theta) {
            const int pos = atomicAdd(&n_q, 1);
            if (TSD_IN(pos, kMaxDrafterChunks, kChkDrafter)) qlist[pos] = q;
        }
    top_sync();
    // (2) qualifying slices
    const int nq = n_q;
    for (int t = tid; t < nq * kWarp; t += kRTopThreads) {
        const int q = qlist[t / kWarp], l = t & (kWarp - 1);
        if (ws.lane_max[(row * nch + q) * kWarp + l] >= theta) {
            const int pos = atomicAdd(&n_s, 1);
            if (pos < kSliceCap) slist[pos] = q * kWarp + l;
        }
    }
    top_sync();
    const int ns = n_s;
    bool overflow = ns > kSliceCap;
    // (3) candidate tokens
    if (!overflow) {
        const T* rrow = logits + row * V;
        auto offer = [&](float x, int id) {
            const int pos = atomicAdd(&n_c, 1);
            if (pos < kRowCandCap) {
                cand_v[pos] = x;
                cand_i[pos] = id;
            }
        };
        if (vec_ok) {
            for (int t = tid; t < ns * kVecPerLane; t += kRTopThreads) {
                const int sl = slist[t / kVecPerLane], i = t % kVecPerLane;
                const int q = sl / kWarp, l = sl & (kWarp - 1);
                const int64_t c0 = (int64_t)q * CE;
                const int e = (i * kWarp + l) * VEC;
                if (e < (int)min((int64_t)CE, V - c0)) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(rrow + c0 + e));
                    if (Lanes<T>::vmax(v) >= theta) {
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            const float x = Lanes<T>::get(v, j);
                            if (x >= theta) offer(x, (int)c0 + e + j);
                        }
                    }
                }
            }
        } else {
            constexpr int per = CE / kWarp;  // tokens of one slice: l, l+32, ...
            for (int t = tid; t < ns * per; t += kRTopThreads) {
                const int sl = slist[t / per], jj = t % per;
                const int q = sl / kWarp, l = sl & (kWarp - 1);
                const int64_t c0 = (int64_t)q * CE;
                const int e = l + kWarp * jj;
                if (e < (int)min((int64_t)CE, V - c0)) {
                    const float x = load_logit(rrow + c0 + e);
                    if (x >= theta) offer(x, (int)c0 + e);
                }
            }
        }
    }
    top_sync();
    const int nc = n_c;
    overflow |= nc > kRowCandCap;
    // (4) selection | log-normaliser
    if (wid == 0) {
        float ev = -INFINITY, tv = -INFINITY;
        int ei = INT_MAX, ti = INT_MAX;
        if (!overflow && nc <= kWarp) {
            ev = lane < nc ? cand_v[lane] : -INFINITY;
            ei = lane < nc ? cand_i[lane] : INT_MAX;
            warp_sort_pairs(ev, ei, lane);
        } else if (!overflow) {
            for (int b0 = 0; b0 < nc; b0 += kWarp) {
                const bool has = b0 + lane < nc;
                warp_list_offer(ev, ei, tv, ti, has, has ? cand_v[b0 + lane] : -INFINITY,
                                has ? cand_i[b0 + lane] : INT_MAX, k, lane);
            }
        } else {
            // every token of every chunk reaching theta, in order
            for (int q = 0; q < nch; ++q) {
                if (!(cm[q] >= theta)) continue;
                const int64_t c0 = (int64_t)q * CE;
                const int cn = (int)min((int64_t)CE, V - c0);
                const T* rp = logits + row * V + c0;
                for (int e0 = 0; e0 < cn; e0 += kWarp) {
                    const int e = e0 + lane;
                    const float x = e < cn ? load_logit(rp + e) : -INFINITY;
                    warp_list_offer(ev, ei, tv, ti, e < cn && x >= theta, x, (int)c0 + e, k, lane);
                }
            }
        }
        if (lane < k) {
            ws.top_id[row * k + lane] = ei;
            ws.top_zt[row * k + lane] = temp == 1.0 ? (double)ev : (double)ev / temp;  // z / T_d
        }
    }
}

cudaError_t launch_drafter_chunks(const void* logits, tsd_dtype dtype, int64_t rows, int64_t V,
                                  float c, const BuildWs& ws, cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    const bool vec_ok = ((uintptr_t)logits % 16 == 0) && ((V * es) % 16 == 0);
    const int wpb = kDThreads / kWarp;
    const int64_t want_chunks = (rows * nch + wpb - 1) / wpb;
    // persistent: one wave of resident CTAs, each warp streaming many chunks
    if (dtype == TSD_BF16) {
        auto kc = drafter_chunk_kernel<__nv_bfloat16>;
        return launch_pdl(kc, resident_grid((const void*)kc, kDThreads, 0, want_chunks), kDThreads,
                          0, stream, static_cast<const __nv_bfloat16*>(logits), rows, V, nch, c,
                          vec_ok, ws);
    }
    auto kc = drafter_chunk_kernel<float>;
    return launch_pdl(kc, resident_grid((const void*)kc, kDThreads, 0, want_chunks), kDThreads, 0,
                      stream, static_cast<const float*>(logits), rows, V, nch, c, vec_ok, ws);
}

cudaError_t launch_drafter_stats(const void* logits, tsd_dtype dtype, int64_t rows, int64_t V,
                                 int topk, float c, double temp, const BuildWs& ws,
                                 cudaStream_t stream) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    const int nch = (int)n_chunks(V, es);
    const bool vec_ok = ((uintptr_t)logits % 16 == 0) && ((V * es) % 16 == 0);
    if (cudaError_t e = launch_drafter_chunks(logits, dtype, rows, V, c, ws, stream); e != cudaSuccess)
        return e;
    if (dtype == TSD_BF16)
        return launch_pdl(drafter_row_kernel<__nv_bfloat16>, (unsigned)rows, kRThreads, 0, stream,
                          static_cast<const __nv_bfloat16*>(logits), rows, V, nch, topk, c, temp,
                          vec_ok, ws);
    return launch_pdl(drafter_row_kernel<float>, (unsigned)rows, kRThreads, 0, stream,
                      static_cast<const float*>(logits), rows, V, nch, topk, c, temp, vec_ok, ws);
}

TSD_CHECK_READER(checks_drafter)

}  // namespace tsd
