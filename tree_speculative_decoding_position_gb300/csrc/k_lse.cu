// k_lse.cu -- the mixture tree under the log-sum-exp score.
//
// "Multi-Future Drafting: Mixture Block Drafters for Tree-Verified
// Speculative Decoding", App. B "Max or log-sum-exp", Eq. 6: a prefix is
// scored by its mixture probability s_lse(v) = log sum_m pi_m Q_m(v).  That
// ranking is not a merge of per-mode searches, so the candidates are the
// distinct prefixes of the modes' per-depth lists, ranked by s_lse.
//
// A mode's depth-d list holds its B most probable length-d prefixes within
// the capped universe (the mode's k kept tokens per position).  Q_m
// factorises over positions, so the list is the best B children of the
// depth-(d-1) list, ordered by (path sum of z/T desc, parent's place asc,
// token rank asc).  Within one mode and depth every child carries the same
// summed log-normaliser, so path sums of z/T decide the order.
//
// lse_beam_kernel    one CTA per (mode, tree), depth by depth, in two warp
//                    groups.  Twelve warps rank: the children of the previous
//                    list form k runs, one per token rank, each already
//                    sorted; only children with (r+1)(i+1) <= B can be kept,
//                    and those runs are merged in log2(k) rounds of binary
//                    searches.  The first B are the new list, handed over
//                    (double-buffered, on named barriers) to four warps that
//                    score it while the next depth is ranked: each entry
//                    gathers its token's logit under every mode (full rows),
//                    extends the per-mode path sums, and takes s_lse = log
//                    sum_m exp(log pi_m + path sum - summed LSE), clamped to
//                    its parent's key; it also extends a hash of its token
//                    sequence.  Equal prefixes reached by several modes get
//                    bit-identical keys and hashes.
// lse_select_kernel  a cluster of two CTAs per tree, each taking half the
//                    depths.  Duplicates across modes are merged over groups
//                    of depths at once through a shared-memory hash on
//                    (depth, token-sequence hash), every merge then checked
//                    exactly (same depth, token and parent representative; by
//                    induction over depth that makes the classes exact); on a
//                    failed check rank 0 merges again depth by depth on
//                    (parent's representative, token).  The first appearance
//                    in (depth, mode, place) order represents a prefix.  Each
//                    CTA compacts its candidates; rank 0 appends rank 1's
//                    (distributed shared memory), a radix select on the 64-bit
//                    key image finds the B-th best, ties at it go by that
//                    order, and the kept entries ordered by counting give the
//                    node order (parents first).
#include <cooperative_groups.h>

#include "tsd_internal.cuh"

namespace tsd {

namespace cg = cooperative_groups;

constexpr int kSelThreads = 1024;
constexpr int kSelCluster = 2;  // CTAs per tree in the selection (a thread-block cluster)

__device__ __forceinline__ double load_logit(const void* logits, tsd_dtype dtype, int64_t off) {
    if (dtype == TSD_BF16)
        return (double)__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(logits)[off]);
    return (double)reinterpret_cast<const float*>(logits)[off];
}

// Named barriers of the list kernel (0 is __syncthreads): the ranking warps
// among themselves, and per list buffer "full" (a depth's list is ready for
// scoring) and "free" (its scoring has read it).
constexpr int kBeamThreads = 512;
constexpr int kScoreThreads = 128;                          // the last four warps
constexpr int kRankThreads = kBeamThreads - kScoreThreads;  // the first twelve
constexpr int kBarRank = 1, kBarScore = 2, kBarFull = 3, kBarFree = 5;
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Merge of kf sorted runs of (k0, k1) pairs, run r at [off[r], off[r+1]), in
// ceil(log2 kf) rounds, by the ranking threads: each round merges
// neighbouring groups of runs, and every element finds its place by one
// binary search in the other half of its group (keys are unique, so "less
// than" decides).  The second key is (i << 5) | r, so an element's run is its
// rank r (its low 5 bits).  Returns 1 when the result is in (d0, d1), 0 when
// in (k0, k1).
__device__ int merge_runs(unsigned long long* k0, unsigned* k1, unsigned long long* d0,
                          unsigned* d1, const int* off, int kf) {
    int flip = 0;
    for (int w = 1; w < kf; w <<= 1) {
        const unsigned long long* a0 = flip ? d0 : k0;
        const unsigned* a1 = flip ? d1 : k1;
        unsigned long long* b0 = flip ? k0 : d0;
        unsigned* b1 = flip ? k1 : d1;
        const int n = off[kf];
        for (int j = threadIdx.x; j < n; j += kRankThreads) {
            const unsigned long long x0 = a0[j];
            const unsigned x1 = a1[j];
            const int g = (int)(x1 & 31u) / (2 * w);  // the element's run is its rank
            const int lo = off[g * 2 * w], mid = off[min(g * 2 * w + w, kf)];
            const int hi = off[min(g * 2 * w + 2 * w, kf)];
            const bool left = j < mid;
            int blo = left ? mid : lo, bhi = left ? hi : mid;  // the other half
            while (blo < bhi) {
                const int m = (blo + bhi) >> 1;
                const bool less = a0[m] < x0 || (a0[m] == x0 && a1[m] < x1);
                if (less) blo = m + 1;
                else bhi = m;
            }
            const int pos = lo + (left ? j - lo : j - mid) + (blo - (left ? mid : lo));
            b0[pos] = x0;
            b1[pos] = x1;
        }
        named_sync(kBarRank, kRankThreads);
        flip ^= 1;
    }
    return flip;
}

// Image of -inf under order_key: the smallest image of a non-NaN double.
constexpr unsigned long long kNegInfImage = 0x000FFFFFFFFFFFFFull;

// Children that can be kept: at most sum over ranks r of B / (r+1) (rounded
// up to a power of two, at least 32).
static __host__ __device__ int lse_sort_cap(int B, int k) {
    int n = 0;
    for (int r = 0; r < k; ++r) n += B / (r + 1);
    return pow2_ceil(n < 32 ? 32 : n);
}

size_t lse_beam_smem(int K, int B, int k) {
    return sizeof(double) * (size_t)(2 * B * K + 4 * B + TSD_MAX_TOPK * (1 + TSD_MAX_MODES) + TSD_MAX_MODES) +
           sizeof(unsigned long long) * (size_t)(2 * B) +
           2 * (sizeof(unsigned long long) + sizeof(unsigned)) * (size_t)lse_sort_cap(B, k) +
           sizeof(int) * (size_t)(4 * B + TSD_MAX_TOPK);
}

// One CTA per (mode, tree).  The first twelve warps rank: depth by depth they
// build the mode's list (own-mode path sums only).  The last four score: a
// depth's list, once handed over, gets its path sums under every mode, its
// s_lse keys and its outputs, while the ranking warps already build the next
// depth's list.  The hand-over is double-buffered (parent places, ranks and
// the list size, by depth parity) on the "full" and "free" barriers.
__global__ void __launch_bounds__(kBeamThreads, 1)
lse_beam_kernel(const void* __restrict__ logits, tsd_dtype dtype, int K, int L, int64_t V, int k,
                int B, double temp, const float* __restrict__ log_prior, BuildWs bws, LseWs ws) {
    pdl_entry();
    extern __shared__ __align__(16) unsigned char sml[];
    const int m = blockIdx.x, t = blockIdx.y, tid = threadIdx.x;
    double* pm = reinterpret_cast<double*>(sml);  // [2][B][K] path sums under every mode (scoring)
    double* ps = pm + 2 * B * K;                  // [2][B] own-mode path sums (ranking)
    double* sk = ps + 2 * B;                      // [2][B] keys (scoring)
    double* zt = sk + 2 * B;                      // [k] this mode's kept z/T (ranking)
    double* zall = zt + TSD_MAX_TOPK;             // [k][K] those tokens' z/T under every mode (scoring)
    double* cst = zall + TSD_MAX_TOPK * TSD_MAX_MODES;  // [K] log prior - summed log-normalisers
    unsigned long long* ph = reinterpret_cast<unsigned long long*>(cst + TSD_MAX_MODES);  // [2][B] path hashes
    unsigned long long* ckey = ph + 2 * B;
    unsigned long long* ckey2 = ckey + lse_sort_cap(B, k);  // merge buffer
    unsigned* cidx = reinterpret_cast<unsigned*>(ckey2 + lse_sort_cap(B, k));
    unsigned* cidx2 = cidx + lse_sort_cap(B, k);
    int* par = reinterpret_cast<int*>(cidx2 + lse_sort_cap(B, k));  // [2][B] parent places (hand-over)
    int* rk = par + 2 * B;                                          // [2][B] token ranks (hand-over)
    int* tks = rk + 2 * B;                                          // [k] this mode's kept ids (scoring)
    __shared__ int s_bad, s_kf;
    __shared__ int s_nb[2];                  // list sizes (hand-over)
    __shared__ int s_off[TSD_MAX_TOPK + 1];  // offsets of the ranks' possible children
    const int64_t KB = (int64_t)K * B;
    const int64_t tree_rows = (int64_t)t * K * L;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    // a row without a finite log-normaliser poisons the tree: no lists at all
    for (int i = tid; i < K * L; i += blockDim.x)
        if (bws.lse[tree_rows + i] != bws.lse[tree_rows + i]) s_bad = 1;
    __syncthreads();
    if (s_bad) {
        for (int d = tid; d < L; d += blockDim.x) ws.nb[((int64_t)t * L + d) * K + m] = 0;
        return;
    }
    if (tid < kRankThreads) {
        // ranking: this mode's kept z/T one depth ahead
        double f_zt = 0.0;
        if (tid < k) f_zt = bws.top_zt[(tree_rows + (int64_t)m * L) * k + tid];
        int np = 1, cur = 0;
        for (int d = 0; d < L; ++d) {
            const int buf = d & 1;
            if (tid < k) zt[tid] = f_zt;
            if (tid < k && d + 1 < L) f_zt = bws.top_zt[(tree_rows + (int64_t)m * L + d + 1) * k + tid];
            const double* prev = ps + (cur ^ 1) * B;
            named_sync(kBarRank, kRankThreads);
            // Lists are sorted, and a lower rank has a larger z/T, so every
            // child (i', r2) with i' <= i and r2 < r precedes child (i, r): its
            // place is at least (r+1)(i+1) - 1, and only children with
            // (r+1)(i+1) <= B can be kept.  Those with mass are ordered by
            // (path sum desc, i asc, r asc) -- complemented order image, then
            // (i << 5) | r -- by merging the per-rank runs, and the first B
            // form the new list.
            if (tid < kWarp) {  // ranks with mass come first: kf of them
                const bool fin = tid < k && zt[tid] != -INFINITY;
                const int kf = __popc(__ballot_sync(0xffffffffu, fin));
                const int len = tid < kf ? min(np, B / (tid + 1)) : 0;
                int incl = len;
                for (int o = 1; o < kWarp; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += y;
                }
                if (tid < kf) s_off[tid] = incl - len;  // exclusive offsets
                if (tid == kWarp - 1) {                 // lane 31's inclusive sum is the total
                    s_off[kf] = incl;
                    s_kf = kf;
                }
            }
            named_sync(kBarRank, kRankThreads);
            const int kf = s_kf, nc = s_off[kf];
            // run r holds rank r's possible children in parent order: already
            // sorted by (complemented path-sum image, i k + r)
            for (int j = tid; j < nc; j += kRankThreads) {
                int r = 0;
                while (s_off[r + 1] <= j) ++r;
                const int i = j - s_off[r];
                ckey[j] = ~order_key((d == 0 ? 0.0 : prev[i]) + zt[r]);
                cidx[j] = ((unsigned)i << 5) | (unsigned)r;  // orders as (i, r); k <= 32
            }
            named_sync(kBarRank, kRankThreads);
            const bool in2 = merge_runs(ckey, cidx, ckey2, cidx2, s_off, kf) != 0;
            const unsigned long long* sk0 = in2 ? ckey2 : ckey;
            const unsigned* sk1 = in2 ? cidx2 : cidx;
            double* nps = ps + cur * B;
            const int nkeep = nc < B ? nc : B;
            if (d >= 2) named_sync(kBarFree + buf, kBeamThreads);  // depth d-2's list is scored
            int* bpar = par + buf * B;
            int* brk = rk + buf * B;
            for (int j = tid; j < nkeep; j += kRankThreads) {
                nps[j] = key_score(~sk0[j]);
                bpar[j] = (int)(sk1[j] >> 5);
                brk[j] = (int)(sk1[j] & 31u);
            }
            if (tid == 0) s_nb[buf] = nkeep;
            named_arrive(kBarFull + buf, kBeamThreads);
            np = nkeep;
            cur ^= 1;
        }
        return;
    }
    // scoring: every mode's log-normaliser and this mode's kept ids one depth
    // ahead, and the kept tokens' logits under every mode (gathered from the
    // full rows); the ids behind that gather two depths ahead
    const int st = tid - kRankThreads;
    double cum = 0.0, lpv = 0.0;
    if (st < K) lpv = log_prior ? (double)log_prior[(int64_t)t * K + st] : -log((double)K);
    double f_lse = 0.0, f_z = 0.0;
    int32_t f_tok = 0, f_id = 0;
    auto fetch_tok = [&](int d) {
        if (st < k * K) f_tok = bws.top_id[(tree_rows + (int64_t)m * L + d) * k + st / K];
    };
    auto fetch = [&](int d) {
        const int64_t row = tree_rows + (int64_t)m * L + d;
        if (st < k) f_id = bws.top_id[row * k + st];
        if (st < K) f_lse = bws.lse[tree_rows + (int64_t)st * L + d];
        if (st < k * K)
            f_z = load_logit(logits, dtype, (tree_rows + (int64_t)(st % K) * L + d) * V + f_tok);
    };
    fetch_tok(0);
    fetch(0);
    if (L > 1) fetch_tok(1);
    int cur = 0;
    for (int d = 0; d < L; ++d) {
        const int buf = d & 1;
        if (st < k) tks[st] = f_id;
        if (st < K) {
            cum += f_lse;
            cst[st] = lpv - cum;
        }
        if (st < k * K) zall[st] = temp == 1.0 ? f_z : f_z / temp;  // z / T_d
        if (d + 1 < L) fetch(d + 1);  // f_tok holds depth d+1's ids
        if (d + 2 < L) fetch_tok(d + 2);
        named_sync(kBarFull + buf, kBeamThreads);  // the list, and this group's inputs
        const int nb = s_nb[buf];
        const int* bpar = par + buf * B;
        const int* brk = rk + buf * B;
        const double* opm = pm + (cur ^ 1) * B * K;
        double* npm = pm + cur * B * K;
        const double* osk = sk + (cur ^ 1) * B;
        double* nsk = sk + cur * B;
        const unsigned long long* oph = ph + (cur ^ 1) * B;
        unsigned long long* nph = ph + cur * B;
        // s_lse of each entry: the terms log pi + log Q in float64 (path sum
        // plus the depth's constant log pi - summed LSE), the sum of
        // exp(term - largest) in fp32; one thread per entry, so that the
        // float64 instructions run on full warps
        for (int j = st; j < nb; j += kScoreThreads) {
            const int pj = bpar[j], rj = brk[j];
            if (!(TSD_IN(pj, B, kChkLse) && TSD_IN(rj, k, kChkLse))) continue;
            double a[TSD_MAX_MODES];
            double amax = -INFINITY;
#pragma unroll
            for (int m2 = 0; m2 < TSD_MAX_MODES; ++m2) {
                if (m2 >= K) break;
                const double P = (d == 0 ? 0.0 : opm[pj * K + m2]) + zall[rj * K + m2];
                npm[j * K + m2] = P;
                a[m2] = P + cst[m2];
                amax = fmax(amax, a[m2]);
            }
            double s = -INFINITY;
            if (amax > -INFINITY) {
                float acc = 0.0f;
#pragma unroll
                for (int m2 = 0; m2 < TSD_MAX_MODES; ++m2) {
                    if (m2 >= K) break;
                    acc += expf((float)(a[m2] - amax));
                }
                s = amax + (double)logf(acc);
            }
            const double up = d == 0 ? INFINITY : osk[pj];
            const double key = s < up ? s : up;
            nsk[j] = key;
            const int64_t f = (int64_t)t * L * KB + (int64_t)d * KB + (int64_t)m * B + j;
            const int32_t x = tks[rj];
            const unsigned long long hv = hash_step(d == 0 ? kRootHash : oph[pj], x);
            nph[j] = hv;
            ws.tok[f] = x;
            ws.par[f] = pj;
            ws.kimg[f] = ~order_key(key);
            ws.phash[f] = hv;
        }
        if (st == 0) ws.nb[((int64_t)t * L + d) * K + m] = nb;
        if (d + 2 < L) named_arrive(kBarFree + buf, kBeamThreads);
        named_sync(kBarScore, kScoreThreads);  // this depth's sums before the next depth's inputs
        cur ^= 1;
    }
}

// Exclusive block scan of one int per thread; *total gets the block sum.
__device__ int block_excl_scan_i(int x, int* red, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) red[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        const int y = lane < nw ? red[lane] : 0;
        int yi = y;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, yi, o);
            if (lane >= o) yi += z;
        }
        red[lane] = yi - y;
        if (lane == 31) red[32] = yi;
    }
    __syncthreads();
    const int r = red[wid] + inc - x;
    *total = red[32];
    __syncthreads();
    return r;
}

// Exclusive block scan of one 64-bit value per thread (two packed 32-bit
// counts add without carry as long as each stays below 2^32).
__device__ unsigned long long block_excl_scan_u64(unsigned long long x, unsigned long long* red,
                                                  unsigned long long* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    unsigned long long inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) red[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        const unsigned long long y = lane < nw ? red[lane] : 0ull;
        unsigned long long yi = y;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long z = __shfl_up_sync(0xffffffffu, yi, o);
            if (lane >= o) yi += z;
        }
        red[lane] = yi - y;
        if (lane == 31) red[32] = yi;
    }
    __syncthreads();
    const unsigned long long r = red[wid] + inc - x;
    *total = red[32];
    __syncthreads();
    return r;
}

// Block-wide AND and OR of one 64-bit value per thread, into *band / *bor.
__device__ void block_and_or(unsigned long long a, unsigned long long o, unsigned long long* red,
                             unsigned long long* band, unsigned long long* bor) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
        a &= __shfl_xor_sync(0xffffffffu, a, k);
        o |= __shfl_xor_sync(0xffffffffu, o, k);
    }
    if (lane == 0) {
        red[wid] = a;
        red[32 + wid] = o;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long A = ~0ull, O = 0ull;
        for (int w = 0; w < nw; ++w) {
            A &= red[w];
            O |= red[32 + w];
        }
        *band = A;
        *bor = O;
    }
    __syncthreads();
}

__device__ __forceinline__ bool pair_less(unsigned long long a0, unsigned long long a1,
                                          unsigned long long b0, unsigned long long b1) {
    return a0 < b0 || (a0 == b0 && a1 < b1);
}

constexpr unsigned long long kEmpty = ~0ull;
constexpr int kMaxSlotsPerThread = 4;  // n_modes * B <= 4096 over 1024 threads

// The merge over groups of depths: one table of kGroupSlots packed words
// (bits 19-63 a 45-bit hash of (depth, token sequence), bits 0-18 the flat
// index of the first appearance; equal prefixes agree above bit 18, so a
// 32-bit minimum of the low half keeps the first appearance), and each
// group entry's slot.  A group holds kGroupSlots / (2 K B) depths, so the
// table is at most half full.
constexpr int kGroupSlots = 16384;
constexpr int kFlatBits = 19;
constexpr unsigned long long kFlatMask = (1ull << kFlatBits) - 1;
static_assert((long long)TSD_MAX_L * kMaxLseModeBudget <= (long long)kFlatMask, "flat index in 19 bits");
static_assert(kGroupSlots >= 2 * kMaxLseModeBudget, "a group holds at least one depth");
constexpr int kGroupPer = kGroupSlots / 2 / kSelThreads;  // group entries a thread
#ifdef TSD_CHECKS
// The checked build keeps 6 bits of the group hash: matches then collide, the
// exact check fails and the depth-by-depth merge runs, and its test compares
// those outputs with the default build's.
constexpr unsigned long long kGroupKeyMask = 0x3Full;
#else
constexpr unsigned long long kGroupKeyMask = ~0ull >> kFlatBits;
#endif

// After the merge, the candidates (image, flat index) stay in shared memory,
// after the sort buffer, when every list entry fits there.
constexpr size_t kSelSmemCap = 220 * 1024;
constexpr int kSurvivors = 2048;  // the radix select's gathered bucket
// the kept entries twice (merged order, node order), then the gathered bucket
static __host__ __device__ size_t lse_sel_sort_bytes(int B) {
    return (size_t)4 * sizeof(unsigned long long) * pow2_ceil(B < 32 ? 32 : B) +
           sizeof(unsigned long long) * kSurvivors;
}
// Each CTA of a tree's pair compacts the candidates of its half of the
// depths there; rank 0 then appends rank 1's, so the buffer holds a tree's.
static __host__ __device__ bool lse_cands_in_smem(int K, int B, int L) {
    return lse_sel_sort_bytes(B) + (size_t)L * K * B * (sizeof(unsigned long long) + sizeof(int32_t)) <=
           kSelSmemCap;
}
size_t lse_select_smem(int K, int B, int L) {
    const size_t H = (size_t)pow2_ceil(2 * K * B);
    const size_t dedupe = H * (sizeof(unsigned long long) + sizeof(int)) + sizeof(int) * 2 * K * B;
    const size_t group = (size_t)kGroupSlots * sizeof(unsigned long long) + sizeof(int16_t) * (size_t)kGroupSlots / 2;
    size_t m = dedupe > group ? dedupe : group;
    const size_t sel = lse_sel_sort_bytes(B) +
                       (lse_cands_in_smem(K, B, L) ? (size_t)L * K * B * (sizeof(unsigned long long) + sizeof(int32_t)) : 0);
    return m > sel ? m : sel;
}

__global__ void __launch_bounds__(kSelThreads)
lse_select_kernel(int K, int L, int k, int B, BuildWs bws, LseWs ws, int32_t* __restrict__ parent,
                  int32_t* __restrict__ token, int32_t* __restrict__ depth,
                  float* __restrict__ score, int32_t* __restrict__ n_nodes,
                  int32_t* __restrict__ status, int32_t* __restrict__ n_cand) {
    pdl_entry();
    extern __shared__ __align__(16) unsigned char sms[];
    __shared__ int red[33];
    __shared__ unsigned hist[256];
    __shared__ int nbs[TSD_MAX_L * TSD_MAX_MODES];
    __shared__ int s_bad, s_bucket, s_need, s_count, s_ns;
    cg::cluster_group cl = cg::this_cluster();
    const int cr = (int)cl.block_rank();  // rank 0 merges the first half of the depths and finishes
    const int t = blockIdx.x / kSelCluster, tid = threadIdx.x;
    const int KB = K * B;
    const int64_t N = (int64_t)L * KB;
    const int64_t base = (int64_t)t * N;
    const int64_t out0 = (int64_t)t * (B + 1);
    const int H = pow2_ceil(2 * KB);
    unsigned long long* hkey = reinterpret_cast<unsigned long long*>(sms);
    int* hval = reinterpret_cast<int*>(hkey + H);
    int* rep_buf[2] = {hval + H, hval + H + KB};  // representatives of one depth, by (mode, place)
    if (tid == 0) s_bad = 0;
    for (int i = tid; i < L * K; i += blockDim.x) nbs[i] = ws.nb[(int64_t)t * L * K + i];
    __syncthreads();
    for (int i = tid; i < K * L * k; i += blockDim.x) {
        const double x = bws.top_zt[(int64_t)t * K * L * k + i];
        if (x != x) s_bad = 1;
    }
    for (int i = tid; i < K * L; i += blockDim.x) {
        const double x = bws.lse[(int64_t)t * K * L + i];
        if (x != x) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {  // both CTAs of the pair see it and leave
        if (cr != 0) return;
        for (int i = tid; i <= B; i += blockDim.x) {
            parent[out0 + i] = -1;
            token[out0 + i] = -1;
            depth[out0 + i] = -1;
            score[out0 + i] = -INFINITY;
        }
        if (tid == 0) {
            n_nodes[t] = 0;
            status[t] = kStatNonFinite;
            if (n_cand) n_cand[t] = 0;
        }
        return;
    }
    // 1. distinct prefixes: rep = flat index of the first appearance; every
    //    list entry is compacted, in flat order, into the candidate arrays
    //    when it is its own representative with mass.
    //    First, all depths of a group at once, keyed by each entry's hash of
    //    (depth, token sequence).  Every merge is then checked exactly: an
    //    entry and its representative have the same depth, the same token and
    //    parents with the same representative.  If all pass, a group's
    //    classes are exactly its distinct prefixes (by induction over depth).
    //    If one fails (a hash collision), the merge runs again depth by depth
    //    on (parent's representative, token), which needs no hash.
    __shared__ int s_fail, s_nf;
    __shared__ unsigned long long red64a[2 * 32], s_and, s_or;
    if (tid == 0) {
        s_and = 0ull;  // no common leading bits known (the depth-by-depth merge)
        s_or = ~0ull;
        s_nf = 0;
    }
    int n_f = 0;
    // The pair splits the depths: rank 0 the first Lh, rank 1 the rest.  Each
    // merges its depths in groups, the pair checks every merge, and each
    // compacts its own candidates, in shared memory after the sort buffer when
    // they fit (the grouped merge's table is dead by then), else in the
    // workspace at their flat places.
    const int Lh = (L + 1) / 2;
    const int dlo = cr == 0 ? 0 : Lh, dhi = cr == 0 ? Lh : L;
    const int64_t flo = (int64_t)dlo * KB, nloc = (int64_t)(dhi - dlo) * KB;
    const bool cand_smem = lse_cands_in_smem(K, B, L);
    unsigned long long* cimg_p = cand_smem ? reinterpret_cast<unsigned long long*>(sms + lse_sel_sort_bytes(B))
                                           : ws.cimg + base + flo;
    int32_t* cflat_p = cand_smem ? reinterpret_cast<int32_t*>(cimg_p + N) : ws.cflat + base + flo;
    if (tid == 0) s_fail = KB == 0;
    bool fail;
    {
        unsigned long long* gtab = reinterpret_cast<unsigned long long*>(sms);
        int16_t* gslot = reinterpret_cast<int16_t*>(gtab + kGroupSlots);
        const int G = KB > 0 ? kGroupSlots / (2 * KB) : 1;
        const FastDiv fKB((unsigned)(KB > 0 ? KB : 1)), fB((unsigned)(B > 0 ? B : 1));
        // an entry of depth d at e = mode * B + place: whether its place is
        // in the mode's list
        auto in_list = [&](int d, int e) {
            const int mm = (int)fB.div((unsigned)e);
            return e - mm * B < nbs[d * K + mm];
        };
        for (int h = tid; h < kGroupSlots; h += blockDim.x) gtab[h] = kEmpty;
        __syncthreads();
        for (int d0 = dlo; d0 < dhi && KB > 0; d0 += G) {
            const int nd = min(G, dhi - d0), ne = nd * KB;
            // the group's hashes first (at most kGroupPer a thread), then the inserts
            unsigned long long hv[kGroupPer];
            bool in[kGroupPer];
#pragma unroll
            for (int q = 0; q < kGroupPer; ++q) {
                const int i = tid + q * kSelThreads;
                const int qd = (int)fKB.div((unsigned)i);
                in[q] = i < ne && in_list(d0 + qd, i - qd * KB);
                hv[q] = in[q] ? ws.phash[base + (int64_t)d0 * KB + i] : 0ull;
            }
#pragma unroll
            for (int q = 0; q < kGroupPer; ++q) {
                const int i = tid + q * kSelThreads;
                if (i >= ne) continue;
                const int d = d0 + (int)fKB.div((unsigned)i);
                int slot = -1;
                if (in[q]) {
                    const int f = d0 * KB + i;
                    const unsigned long long key = (hash_step(hv[q], d) >> kFlatBits) & kGroupKeyMask;
                    const unsigned long long word = (key << kFlatBits) | (unsigned long long)f;
                    unsigned h = (unsigned)key & (unsigned)(kGroupSlots - 1);
                    for (int probe = 0; probe < kGroupSlots; ++probe) {
                        const unsigned long long old = atomicCAS(&gtab[h], kEmpty, word);
                        if (old == kEmpty) {
                            slot = (int)h;
                            break;
                        }
                        if ((old >> kFlatBits) == key) {
                            atomicMin(reinterpret_cast<unsigned*>(&gtab[h]), (unsigned)word);
                            slot = (int)h;
                            break;
                        }
                        h = (h + 1) & (unsigned)(kGroupSlots - 1);
                    }
                }
                gslot[i] = (int16_t)slot;
            }
            __syncthreads();
            for (int i = tid; i < ne; i += blockDim.x)
                if (gslot[i] >= 0) ws.rep[base + (int64_t)d0 * KB + i] = (int)(gtab[gslot[i]] & kFlatMask);
            __syncthreads();
            for (int h = tid; h < kGroupSlots; h += blockDim.x) gtab[h] = kEmpty;
            __syncthreads();
        }
        cl.sync();  // every representative of the tree is in the workspace
        // The exact check of every merge of this CTA's depths (a parent of
        // the first may be the other CTA's), with each entry's image and keep
        // mark staged at its place in this CTA's candidate buffer.
        bool bad_merge = false;
        unsigned long long and_img = ~0ull, or_img = 0ull;
        for (int64_t c0 = 0; c0 < nloc; c0 += 8 * blockDim.x) {
            int r[8];
            unsigned long long im[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int64_t i = c0 + q * blockDim.x + tid, c = flo + i;
                bool lv = false;
                if (i < nloc) {
                    const int d = (int)fKB.div((unsigned)c);
                    lv = in_list(d, (int)c - d * KB);
                }
                r[q] = lv ? ws.rep[base + c] : -1;
                im[q] = lv ? ws.kimg[base + c] : ~kNegInfImage;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int64_t i = c0 + q * blockDim.x + tid;
                if (i >= nloc) continue;
                const int f = (int)(flo + i);
                if (r[q] >= 0 && r[q] != f) {
                    const int rr = r[q], d = (int)fKB.div((unsigned)f), dr = (int)fKB.div((unsigned)rr);
                    bool same = dr == d && rr < f && ws.tok[base + rr] == ws.tok[base + f];
                    if (same && d > 0) {
                        const int pf = ws.par[base + f], pr = ws.par[base + rr];
                        const int mf = (int)fB.div((unsigned)(f - d * KB)), mr = (int)fB.div((unsigned)(rr - d * KB));
                        same = TSD_IN(pf, B, kChkLse) && TSD_IN(pr, B, kChkLse) &&
                               ws.rep[base + (int64_t)(d - 1) * KB + mf * B + pf] ==
                                   ws.rep[base + (int64_t)(d - 1) * KB + mr * B + pr];
                    }
                    bad_merge |= !same;
                }
                const bool kp = r[q] == f && im[q] != ~kNegInfImage;
                cimg_p[i] = im[q];
                cflat_p[i] = kp ? (int32_t)f : -1;
                if (kp) {
                    and_img &= im[q];
                    or_img |= im[q];
                }
            }
        }
        if (__syncthreads_or(bad_merge) && tid == 0) s_fail = 1;
        block_and_or(and_img, or_img, red64a, &s_and, &s_or);  // also orders the marks
        cl.sync();  // both CTAs' checks are in
        fail = s_fail != 0 || *cl.map_shared_rank(&s_fail, (unsigned)(cr ^ 1)) != 0;
        if (!fail) {
            // the kept ones moved forward chunk by chunk (a candidate's place
            // never exceeds its own, and a chunk is read before its scan's
            // barriers)
            for (int64_t c0 = 0; c0 < nloc; c0 += 4 * blockDim.x) {
                int32_t fl[4];
                unsigned long long im[4];
                int cnt = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t c = c0 + 4 * tid + q;
                    fl[q] = c < nloc ? cflat_p[c] : -1;
                    im[q] = c < nloc ? cimg_p[c] : 0ull;
                    cnt += fl[q] >= 0;
                }
                int tot;
                int pos = n_f + block_excl_scan_i(cnt, red, &tot);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (fl[q] < 0) continue;
                    cimg_p[pos] = im[q];
                    cflat_p[pos] = fl[q];
                    ++pos;
                }
                n_f += tot;
            }
            if (tid == 0) s_nf = n_f;
            __syncthreads();
        }
    }
    if (fail && KB > 0 && cr == 0) {
    // rank 0 alone, over every depth (the hash of this merge overlaps the
    // shared candidate buffer: its candidates go to the workspace)
    cimg_p = ws.cimg + base;
    cflat_p = ws.cflat + base;
    // thread tid holds entries e = S tid + q, q < S, of each depth (S = K B /
    // threads rounded up, at most 4); the next depth's tokens, parents and
    // images are loaded while this one hashes
    int32_t tk[kMaxSlotsPerThread], pp[kMaxSlotsPerThread];
    unsigned long long im[kMaxSlotsPerThread];
    bool lv[kMaxSlotsPerThread];
    const int S = (KB + blockDim.x - 1) / blockDim.x;
    auto load_depth = [&](int d, int32_t* tk_, int32_t* pp_, unsigned long long* im_, bool* lv_) {
#pragma unroll
        for (int q = 0; q < kMaxSlotsPerThread; ++q) {
            const int e = S * tid + q;
            lv_[q] = q < S && e < KB && (e % B) < nbs[d * K + e / B];
            const int64_t f = base + (int64_t)d * KB + e;
            tk_[q] = lv_[q] ? ws.tok[f] : 0;
            pp_[q] = lv_[q] && d > 0 ? ws.par[f] : -1;
            im_[q] = lv_[q] ? ws.kimg[f] : ~kNegInfImage;
        }
    };
    load_depth(0, tk, pp, im, lv);
    for (int d = 0; d < L; ++d) {
        int* rep_prev = rep_buf[(d & 1) ^ 1];
        int* rep_cur = rep_buf[d & 1];
        int32_t tk2[kMaxSlotsPerThread], pp2[kMaxSlotsPerThread];
        unsigned long long im2[kMaxSlotsPerThread];
        bool lv2[kMaxSlotsPerThread];
        if (d + 1 < L) load_depth(d + 1, tk2, pp2, im2, lv2);
        for (int h = tid; h < H; h += blockDim.x) {
            hkey[h] = kEmpty;
            hval[h] = INT_MAX;
        }
        __syncthreads();
        int slot[kMaxSlotsPerThread];
#pragma unroll
        for (int q = 0; q < kMaxSlotsPerThread; ++q) {
            slot[q] = -1;
            if (!lv[q]) continue;
            const int e = S * tid + q, m = e / B;
            const int f = d * KB + e;
            const int pr = d == 0 ? -1 : (TSD_IN(pp[q], B, kChkLse) ? rep_prev[m * B + pp[q]] : -1);
            const unsigned long long key =
                ((unsigned long long)(unsigned)(pr + 1) << 32) | (unsigned)tk[q];
            unsigned h = (unsigned)((key * 0x9E3779B97F4A7C15ull) >> 40) & (unsigned)(H - 1);
            for (int probe = 0; probe < H; ++probe) {
                const unsigned long long old = atomicCAS(&hkey[h], kEmpty, key);
                if (old == kEmpty || old == key) {
                    atomicMin(&hval[h], f);
                    slot[q] = (int)h;
                    break;
                }
                h = (h + 1) & (unsigned)(H - 1);
            }
        }
        __syncthreads();
        // representatives, and the compaction of those with mass in flat order
        int cnt = 0;
        bool keep[kMaxSlotsPerThread];
#pragma unroll
        for (int q = 0; q < kMaxSlotsPerThread; ++q) {
            const int e = S * tid + q;
            keep[q] = false;
            if (slot[q] < 0) continue;
            const int r = hval[slot[q]];
            rep_cur[e] = r;
            ws.rep[base + (int64_t)d * KB + e] = r;
            keep[q] = r == d * KB + e && im[q] != ~kNegInfImage;
            cnt += keep[q];
        }
        int tot;
        int pos = n_f + block_excl_scan_i(cnt, red, &tot);  // also orders rep_cur's writes
#pragma unroll
        for (int q = 0; q < kMaxSlotsPerThread; ++q) {
            if (!keep[q]) continue;
            ws.cimg[base + pos] = im[q];
            ws.cflat[base + pos] = d * KB + S * tid + q;
            ++pos;
        }
        n_f += tot;
#pragma unroll
        for (int q = 0; q < kMaxSlotsPerThread; ++q) {
            tk[q] = tk2[q];
            pp[q] = pp2[q];
            im[q] = im2[q];
            lv[q] = d + 1 < L && lv2[q];
        }
    }
    }  // the depth-by-depth merge
    cl.sync();  // each CTA's candidates are compacted (or rank 0 merged them all)
    if (cr != 0) {
        cl.sync();  // rank 0 has copied this CTA's candidates
        return;
    }
    // rank 0 appends rank 1's candidates to its own: the tree's, in flat
    // order (in the workspace the copy moves them down, chunk by chunk, each
    // read before it is written)
    if (!fail) {
        const int n1 = *cl.map_shared_rank(&s_nf, 1u);
        const unsigned long long* img1 = cand_smem ? cl.map_shared_rank(cimg_p, 1u) : ws.cimg + base + (int64_t)Lh * KB;
        const int32_t* fl1 = cand_smem ? cl.map_shared_rank(cflat_p, 1u) : ws.cflat + base + (int64_t)Lh * KB;
        for (int j0 = 0; j0 < n1; j0 += 4 * (int)blockDim.x) {
            unsigned long long im[4];
            int32_t fl[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = j0 + q * blockDim.x + tid;
                im[q] = j < n1 ? img1[j] : 0ull;
                fl[q] = j < n1 ? fl1[j] : -1;
            }
            __syncthreads();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = j0 + q * blockDim.x + tid;
                if (j < n1) {
                    cimg_p[n_f + j] = im[q];
                    cflat_p[n_f + j] = fl[q];
                }
            }
        }
        if (tid == 0) {
            s_and &= *cl.map_shared_rank(&s_and, 1u);
            s_or |= *cl.map_shared_rank(&s_or, 1u);
        }
        n_f += n1;
        __syncthreads();
    }
    cl.sync();  // rank 1's candidates are copied: it may leave
    const unsigned long long* cimg = cimg_p;
    const int32_t* cflat = cflat_p;
    // 2. radix select of the B-th best image among the candidates
    int take = n_f < B ? n_f : B;
    unsigned long long prefix = 0, mask = 0;
    int need = take;  // 1-based rank of the threshold among the remaining
    const bool cut = n_f > B;
    // the candidates' images agree above the highest bit where they differ:
    // the select starts at that bit's byte
    const unsigned long long diff = s_and ^ s_or;
    int shift0 = 56;
    if (take > 0 && cut) {
        if (diff == 0ull) {  // every candidate has the same image: it is the threshold
            shift0 = -8;
            mask = ~0ull;
            prefix = s_and;
        } else {
            shift0 = ((63 - __clzll((long long)diff)) / 8) * 8;
            if (shift0 < 56) {
                mask = ~((1ull << (shift0 + 8)) - 1);  // the bits above byte shift0
                prefix = s_and & mask;
            }
        }
    }
    if (take > 0 && cut) {
        // the passes read the candidates until the selected bucket holds at
        // most kSurvivors of them; those are then gathered (in any order: a
        // histogram needs none) and the later passes read only them
        unsigned long long* surv = reinterpret_cast<unsigned long long*>(sms) + 4 * pow2_ceil(B < 32 ? 32 : B);
        const unsigned long long* src = cimg;
        int nsrc = n_f;
        bool gathered = false;
        for (int shift = shift0; shift >= 0; shift -= 8) {
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            for (int c0 = 0; c0 < nsrc; c0 += 4 * blockDim.x) {
                unsigned long long v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = c0 + q * blockDim.x + tid;
                    v[q] = c < nsrc ? src[c] : ~0ull;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = c0 + q * blockDim.x + tid;
                    if (c < nsrc && (v[q] & mask) == prefix)
                        atomicAdd(&hist[(unsigned)(v[q] >> shift) & 255u], 1u);
                }
            }
            __syncthreads();
            if (tid < 32) {
                unsigned run = 0;
                unsigned v[8];
                for (int q = 0; q < 8; ++q) {
                    v[q] = hist[tid * 8 + q];
                    run += v[q];
                }
                unsigned incl = run;
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += y;
                }
                unsigned before = incl - run;
                // the lane whose range holds the need-th element
                if (before < (unsigned)need && (unsigned)need <= incl) {
                    for (int q = 0; q < 8; ++q) {
                        if ((unsigned)need <= before + v[q]) {
                            s_bucket = tid * 8 + q;
                            s_need = need - (int)before;
                            s_count = (int)v[q];
                            break;
                        }
                        before += v[q];
                    }
                }
            }
            if (tid == 0) s_ns = 0;
            __syncthreads();
            prefix |= (unsigned long long)s_bucket << shift;
            mask |= 255ull << shift;
            need = s_need;
            if (!gathered && shift > 0 && s_count <= kSurvivors) {
                for (int c = tid; c < nsrc; c += blockDim.x) {
                    const unsigned long long v = src[c];
                    if ((v & mask) == prefix) {
                        const int pos = atomicAdd(&s_ns, 1);
                        if (pos < kSurvivors) surv[pos] = v;
                    }
                }
                __syncthreads();
                src = surv;
                nsrc = min(s_ns, kSurvivors);
                gathered = true;
            }
            __syncthreads();
        }
    }
    const unsigned long long theta = prefix;
    // 3. compaction in flat order: every candidate below theta, and the first
    //    `need` equal to it
    unsigned long long* sk0 = reinterpret_cast<unsigned long long*>(sms);
    const int n2 = pow2_ceil(take < 32 ? 32 : take);
    unsigned long long* sk1 = sk0 + n2;
    __syncthreads();  // the hash table's space is reused
    {
        // position of a kept candidate = (candidates below theta before it) +
        // min(candidates equal to theta before it, need); one packed scan of
        // (below, equal) counts per four candidates a thread
        __shared__ unsigned long long red64[33];
        unsigned long long carry = 0;
        for (int c0 = 0; c0 < n_f; c0 += 4 * blockDim.x) {
            unsigned long long img[4];
            unsigned long long cnt = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c = c0 + 4 * tid + q;
                img[q] = c < n_f ? cimg[c] : ~0ull;
                if (c < n_f) cnt += (!cut || img[q] < theta) ? 1ull : (img[q] == theta ? 1ull << 32 : 0ull);
            }
            unsigned long long tot;
            unsigned long long run = carry + block_excl_scan_u64(cnt, red64, &tot);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c = c0 + 4 * tid + q;
                if (c >= n_f) continue;
                const int lt = (int)(run & 0xffffffffull), eq = (int)(run >> 32);
                const bool below = !cut || img[q] < theta;
                const bool equal = !below && img[q] == theta;
                if (below || (equal && eq < need)) {
                    const int pos = lt + min(eq, need);
                    if (pos < take) {
                        sk0[pos] = img[q];
                        sk1[pos] = (unsigned long long)cflat[c];
                    }
                }
                run += below ? 1ull : (equal ? 1ull << 32 : 0ull);
            }
            carry += tot;
        }
        const int kept = (int)(carry & 0xffffffffull) + min((int)(carry >> 32), cut ? need : 0);
        take = kept < take ? kept : take;  // equal unless the counts disagree
    }
    for (int i = take + tid; i < n2; i += blockDim.x) {
        sk0[i] = kEmpty;
        sk1[i] = kEmpty;
    }
    __syncthreads();
    // 4. order the kept entries by (image asc, flat index asc): an entry's
    //    place is the number of entries before it, counted by P threads
    unsigned long long* so0 = sk0 + 2 * pow2_ceil(B < 32 ? 32 : B);
    unsigned long long* so1 = so0 + pow2_ceil(B < 32 ? 32 : B);
    {
        int P = 1;
        while (P < 32 && take > 0 && 2 * P * take <= (int)blockDim.x) P <<= 1;
        for (int i0 = 0; i0 < take; i0 += blockDim.x / P) {  // block-uniform
            const int i = i0 + tid / P, sub = tid % P;
            int cnt = 0;
            unsigned long long a0 = 0ull, a1 = 0ull;
            if (i < take) {
                a0 = sk0[i];
                a1 = sk1[i];
                for (int j = sub; j < take; j += P) cnt += pair_less(sk0[j], sk1[j], a0, a1) ? 1 : 0;
            }
            for (int o = 1; o < P; o <<= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
            if (i < take && sub == 0 && cnt < take) {
                so0[cnt] = a0;
                so1[cnt] = a1;
            }
        }
    }
    __syncthreads();
    // 5. emit: node q+1 is the q-th kept entry; parents come first
    for (int q = tid; q < take; q += blockDim.x)
        if (so1[q] < (unsigned long long)N) ws.node_of[base + (int64_t)so1[q]] = q + 1;
    __syncthreads();
    for (int q = tid; q < B; q += blockDim.x) {
        const int64_t o = out0 + 1 + q;
        if (q < take && so1[q] < (unsigned long long)N) {
            const int64_t f = (int64_t)so1[q];
            const int d = (int)(f / KB), e = (int)(f - (int64_t)d * KB), m = e / B;
            int pn = 0;
            if (d > 0) {
                const int pp = ws.par[base + f];
                const int64_t r =
                    TSD_IN(pp, B, kChkLse) ? ws.rep[base + (int64_t)(d - 1) * KB + (int64_t)m * B + pp] : 0;
                pn = TSD_IN(r, N, kChkLse) ? ws.node_of[base + r] : 0;
            }
            if (!TSD_IN(pn, q + 1, kChkLse)) pn = 0;  // a parent precedes its child
            parent[o] = pn;
            token[o] = ws.tok[base + f];
            depth[o] = d + 1;
            const double key = key_score(~ws.kimg[base + f]);
            score[o] = (float)key;
            if (bws.score64) bws.score64[out0 + 1 + q] = key;
        } else {
            parent[o] = -1;
            token[o] = -1;
            depth[o] = -1;
            score[o] = -INFINITY;
        }
    }
    if (tid == 0) {
        parent[out0] = -1;
        token[out0] = -1;
        depth[out0] = 0;
        score[out0] = 0.0f;
        n_nodes[t] = take + 1;
        status[t] = kStatOk;
        if (n_cand) n_cand[t] = n_f;
    }
}

cudaError_t launch_lse_tree(const void* logits, tsd_dtype dtype, int n_trees, int K, int L,
                            int64_t V, int k, int B, double temp, const float* log_prior,
                            const BuildWs& bws, const LseWs& ws, int32_t* parent, int32_t* token,
                            int32_t* depth, float* score, int32_t* n_nodes, int32_t* status,
                            int32_t* n_cand, cudaStream_t stream) {
    const size_t sb = lse_beam_smem(K, B, k);
    cudaError_t e = cudaFuncSetAttribute(lse_beam_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sb);
    if (e != cudaSuccess) return e;
    e = launch_pdl(lse_beam_kernel, dim3((unsigned)K, (unsigned)n_trees), kBeamThreads, sb, stream,
                   logits, dtype, K, L, V, k, B, temp, log_prior, bws, ws);
    if (e != cudaSuccess) return e;
    const size_t ss = lse_select_smem(K, B, L);
    e = cudaFuncSetAttribute(lse_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss);
    if (e != cudaSuccess) return e;
    return launch_pdl_cluster(lse_select_kernel, (unsigned)(n_trees * kSelCluster), kSelCluster, kSelThreads,
                              ss, stream, K, L, k, B, bws, ws, parent, token, depth, score, n_nodes, status,
                              n_cand);
}

TSD_CHECK_READER(checks_lse)

}  // namespace tsd
