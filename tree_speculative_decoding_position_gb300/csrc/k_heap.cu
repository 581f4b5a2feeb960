// k_heap.cu -- best-first tree builder over the top-k universe, batched.
//
// "CAST: Cost-Aware Speculative Trees from One-Pass Block Drafters", Thm. 1
// and App. C "Candidate construction": the B prefixes with the largest
// plug-in score sum_j log q_j(y_j), expanded best-first; ties toward shorter
// prefixes, then lexicographic.
// "Multi-Future Drafting: Mixture Block Drafters for Tree-Verified
// Speculative Decoding", Sec. 3.4 Eq. 2, Sec. 4.3, App. B "Merged heap" and
// Prop. 6: entries (mode, prefix) keyed by that mode's score; taking an entry
// adds its next sibling (rank r+1) and its first child (rank 0 at the next
// position); a prefix taken again from another mode keeps its first node.
//
// The pages run this as a sequential heap on the host.  Here one CTA per tree
// builds it.  One mode takes the threshold expansion (below, thr_build): every
// prefix that can still reach the B best, depth by depth, under a rising bound.
// Several modes, and one mode when that declines, take rounds over a sorted
// frontier: each round takes the frontier's
// best M entries at once, merges them into the sorted list X of taken
// entries, and merges all k children of each (CAST App. C's push rule; the
// oracle's pins show it pops the same prefixes in the same order as the
// sibling + first-child rule) back into the frontier.  Because a prefix's
// children arrive one round after it, the number of rounds is about the depth
// of the tree.  Taking several entries per round may take some that a
// one-at-a-time heap would not reach, but never misses one: every entry not
// yet taken is worse than the frontier head, and the search stops only when
// the frontier holds nothing better than the B-th distinct prefix of X.  The
// frontier is pruned every round: until X holds B distinct prefixes, to
// entries no worse than the (K*B)-th entry of X and the frontier merged (at
// least B distinct prefixes are that good); after, to entries better than the
// B-th distinct prefix of X, and to at most its first K*B entries.
// The result is exactly the heap's: the B best distinct prefixes under the
// total order (score desc, depth asc, mode asc, rank sequence asc), listed in
// that order (= pop order).
//
// Scores: a prefix's sum of log q_j is evaluated as (the left-to-right sum of
// its tokens' z / T_d) - C_m(depth), with C_m(d) the sum of mode m's first d
// row log-normalisers.  Two prefixes of one depth and mode whose scaled logits
// sum to the same value therefore tie exactly (as they do in exact
// arithmetic), and the tie order decides them.  A child's key is at most its
// parent's: each log q is at most 0, and where the rounding of the two path
// sums would put a child above its parent, the child takes the parent's key,
// so that a parent always precedes its children.
//
// Entries are 32 bytes: a 64-bit order-preserving image of the float64 score,
// the 64-bit tie key depth << 59 | mode << 56 | rank digits (which also names
// the prefix within its mode), the prefix's z / T_d sum, and a 64-bit hash of
// the parent's token sequence (to tell equal prefixes of different modes
// apart; every hash match is confirmed by comparing the token sequences).
#include <float.h>

#include "tsd_internal.cuh"

namespace tsd {

constexpr int kBuildThreads = 512;
// successor slots per thread in child generation (the plan keeps M * k <= 512)
constexpr int kSlotsPerThread = (512 + kBuildThreads - 1) / kBuildThreads;

struct __align__(16) FEntry {
    unsigned long long key;   // order-preserving image of the score
    unsigned long long tb;    // depth << 59 | mode << 56 | rank digits
    double zsum;              // sum of z / T_d along the prefix (left to right)
    unsigned long long hpar;  // hash of the parent's token sequence
};
static_assert(sizeof(FEntry) == 32, "entry layout");

constexpr unsigned long long kSentinelKey = 0ull;  // below every real key
constexpr unsigned long long kRsMask = (1ull << 56) - 1;

__device__ __forceinline__ bool before(const FEntry& a, const FEntry& b) {
    return a.key > b.key || (a.key == b.key && a.tb < b.tb);
}
__device__ __forceinline__ int tb_depth(unsigned long long tb) { return (int)(tb >> 59); }
__device__ __forceinline__ int tb_mode(unsigned long long tb) { return (int)((tb >> 56) & 7); }

struct BuildPlan {
    int M;          // entries taken per round
    int fcap, xcap; // frontier / taken-list capacity
    int hcap;       // hash table size (power of two)
    size_t lists, fbytes, xbytes, sbytes, scode_bytes, hbytes, flag_bytes, smem_total;
    bool big_in_smem;
    size_t global_per_tree;
    // threshold expansion (one mode): candidate capacity (0 = rounds only),
    // depth of the fully enumerated levels and their prefix count
    int tcap, d0, n0;
    FastDiv kdiv;  // division by topk
};

// Threshold expansion: key bins of the selections, candidates kept at most,
// and the largest enumeration of the first levels.
constexpr int kThrBinBits = 11;
constexpr int kThrBins = 1 << kThrBinBits;
// bin counts in 32 rows of 64 plus one pad word: lane l of a warp owns row
// l, and a warp reading one word per lane across a row hits distinct banks
constexpr int kThrBinWords = kThrBins + kThrBins / 64;
constexpr int kThrCapMax = 3072;
constexpr int kThrSlots = 4096;  // (parent, rank) pairs evaluated per level
constexpr int kThrEnumMax = 1024;
// per candidate: key, tie key, z sum (8 B each); parent, node, bin-order
// slot, float z sum (4 B each)
constexpr size_t kThrBytesPer = 3 * sizeof(unsigned long long) + 4 * sizeof(int32_t);
// bin counts and bases, row sums, two pair lists; float lists, their
// magnitudes and the float log-normalisers
constexpr size_t kThrFixed = sizeof(int32_t) * (2 * kThrBinWords + 32 + 2 * kThrSlots) +
                             sizeof(float) * (TSD_MAX_L * TSD_MAX_TOPK + 2 * (TSD_MAX_L + 1));

__host__ __device__ inline int pow2_at_least(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

static BuildPlan build_plan(int n_modes, int L, int topk, int B) {
    BuildPlan p;
    // entries taken per round: their children (k each) fill the successor buffer
    p.M = (n_modes > 1 ? 256 : 512) / topk;
    if (p.M < 8) p.M = 8;
    if (p.M > 128) p.M = 128;
    // M * topk <= 512 (TSD_MAX_TOPK = 32): child generation gives each
    // thread at most kSlotsPerThread slots
    p.xcap = n_modes * (B + 1) + p.M;
    p.fcap = n_modes * (B + 1) + topk * p.M + n_modes * topk + 32;
    p.hcap = pow2_at_least(p.xcap + p.xcap / 2);  // load factor at most 2/3
    auto r16 = [](size_t b) { return (b + 15) & ~(size_t)15; };
    p.lists = r16((size_t)n_modes * L * topk * (sizeof(double) + sizeof(int32_t)) +
                  sizeof(double) * (size_t)n_modes * (L + 1));
    const size_t n2s = (size_t)pow2_at_least(topk * p.M < 32 ? 32 : topk * p.M);
    // successor order codes and the sort's second buffer
    p.scode_bytes = r16(2 * sizeof(unsigned long long) * n2s);
    p.sbytes = r16(sizeof(FEntry) * n2s) + p.scode_bytes;
    p.hbytes = r16((size_t)p.hcap * (sizeof(unsigned long long) + sizeof(int32_t)));
    p.flag_bytes = r16(sizeof(int32_t) * 2 * (size_t)p.xcap + 64);
    p.fbytes = r16(sizeof(FEntry) * 2 * (size_t)p.fcap);
    p.xbytes = r16(sizeof(FEntry) * 2 * (size_t)p.xcap);
    // frontier, taken list, hash table and marks go to global memory (one
    // region per tree) when shared memory cannot hold them
    const size_t big = p.fbytes + p.xbytes + p.hbytes + p.flag_bytes;
    p.big_in_smem = p.lists + p.sbytes + big <= 225 * 1024;  // of 227 KB per block
    p.smem_total = p.lists + p.sbytes + (p.big_in_smem ? big : 0);
    p.global_per_tree = p.big_in_smem ? 0 : big;
    // Threshold expansion for one mode: enumerate levels 1..d0 until they hold
    // B prefixes (one more while the enumeration stays within kThrEnumMax)
    p.tcap = p.d0 = p.n0 = 0;
    p.kdiv = FastDiv((unsigned)topk);
    if (n_modes == 1 && B > 0) {
        long long n = 0, lev = 1;
        int d = 0;
        while (d < L && n < B && n <= (1 << 22)) {
            ++d;
            lev *= topk;
            n += lev;
        }
        while (n >= B && d < L && n + lev * topk <= kThrEnumMax) {
            ++d;
            lev *= topk;
            n += lev;
        }
        const size_t fixed = r16(p.lists) + r16(kThrFixed);
        long long cap = fixed < 225 * 1024 ? (long long)((225 * 1024 - fixed) / kThrBytesPer) : 0;
        cap = (cap < kThrCapMax ? cap : kThrCapMax) & ~31LL;
        if (n >= B && 2 * n <= cap && 2LL * B <= cap) {
            p.tcap = (int)cap;
            p.d0 = d;
            p.n0 = (int)n;
            const size_t need = fixed + (size_t)cap * kThrBytesPer;
            if (need > p.smem_total) p.smem_total = need;
        }
    }
    return p;
}

size_t heap_spill_bytes(int n_modes, int L, int topk, int B) {
    return build_plan(n_modes, L, topk, B).global_per_tree;
}

// ---------------------------------------------------------------------------
// Block-wide helpers (all threads call them).
// ---------------------------------------------------------------------------
__device__ __forceinline__ FEntry shfl_xor_entry(const FEntry& x, int j) {
    FEntry y;
    y.key = __shfl_xor_sync(0xffffffffu, x.key, j);
    y.tb = __shfl_xor_sync(0xffffffffu, x.tb, j);
    y.zsum = __shfl_xor_sync(0xffffffffu, x.zsum, j);
    y.hpar = __shfl_xor_sync(0xffffffffu, x.hpar, j);
    return y;
}

// Bitonic steps (k, j) for j from jtop down to 1 on one 32-entry block held
// one entry per lane: partners differ in lane bits, so shuffles replace
// shared-memory exchanges and no block barrier is needed.
__device__ __forceinline__ FEntry bitonic_lane_steps(FEntry x, int e, int lane, int k, int jtop) {
    for (int j = jtop; j > 0; j >>= 1) {
        const FEntry y = shfl_xor_entry(x, j);
        const bool lower = (lane & j) == 0;
        const bool asc = (e & k) == 0;  // this k-block ends up in the total order
        const bool x_first = before(x, y);
        if ((lower == asc) != x_first) x = y;
    }
    return x;
}

// Bitonic sort of a[0, n2) (n2 a power of two, at least 32) into the total
// order.  Steps with partner distance below 32 run in registers per warp;
// only distances of 32 and more exchange through memory between barriers.
__device__ void sort_entries(FEntry* a, int n2) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nblk = n2 >> 5;
    for (int b = wid; b < nblk; b += nw) {  // k = 2 .. 32 inside each block
        const int e = (b << 5) + lane;
        FEntry x = a[e];
        for (int k = 2; k <= 32; k <<= 1) x = bitonic_lane_steps(x, e, lane, k, k >> 1);
        a[e] = x;
    }
    __syncthreads();
    for (int k = 64; k <= n2; k <<= 1) {
        for (int j = k >> 1; j >= 32; j >>= 1) {
            for (int i = threadIdx.x; i < n2; i += blockDim.x) {
                const int l = i ^ j;
                if (l > i) {
                    const FEntry x = a[i], y = a[l];
                    const bool up = (i & k) == 0;
                    if (up ? before(y, x) : before(x, y)) {
                        a[i] = y;
                        a[l] = x;
                    }
                }
            }
            __syncthreads();
        }
        for (int b = wid; b < nblk; b += nw) {
            const int e = (b << 5) + lane;
            a[e] = bitonic_lane_steps(a[e], e, lane, k, 16);
        }
        __syncthreads();
    }
}

// Part `part` of `nparts` of dst[0, na+nb) = merge of sorted a[0, na) and
// sorted b[0, nb) (merge path).  With `ord`, the j-th entry of b is
// b[ord[j] & 0xffff] (b itself unsorted).  No barrier.
__device__ void merge_part(FEntry* dst, const FEntry* a, int na, const FEntry* b, int nb,
                           const unsigned long long* ord, int part, int nparts) {
    auto bj = [&](int j) -> const FEntry& { return ord ? b[ord[j] & 0xffffull] : b[j]; };
    const int total = na + nb;
    const int per = (total + nparts - 1) / nparts;
    const int d0 = min(total, part * per), d1 = min(total, d0 + per);
    if (d0 < d1) {
        int lo = max(0, d0 - nb), hi = min(d0, na);
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (before(a[mid], bj(d0 - mid - 1))) lo = mid + 1;
            else hi = mid;
        }
        int ia = lo, ib = d0 - lo;
        for (int d = d0; d < d1; ++d) {
            if (ib >= nb || (ia < na && before(a[ia], bj(ib)))) dst[d] = a[ia++];
            else dst[d] = bj(ib++);
        }
    }
}

// Two independent merges in one phase, the block's threads split between
// them in proportion to their lengths; one barrier at the end.
__device__ void merge_two(FEntry* d1, const FEntry* a1, int na1, const FEntry* b1, int nb1,
                          FEntry* d2, const FEntry* a2, int na2, const FEntry* b2, int nb2,
                          const unsigned long long* ord2) {
    const int n1 = na1 + nb1, n2 = na2 + nb2, nt = blockDim.x;
    int t1 = n1 + n2 > 0 ? (int)(((long long)nt * n1 + (n1 + n2) / 2) / (n1 + n2)) : 0;
    if (n1 > 0 && t1 < 1) t1 = 1;
    if (n2 > 0 && t1 > nt - 1) t1 = nt - 1;
    if ((int)threadIdx.x < t1) merge_part(d1, a1, na1, b1, nb1, nullptr, threadIdx.x, t1);
    else merge_part(d2, a2, na2, b2, nb2, ord2, threadIdx.x - t1, nt - t1);
    __syncthreads();
}

// Smallest i in [lo, hi) with pred(i) false, for pred true then false over
// the range (hi if none): a 32-ary search by one warp (all lanes call it).
template <class P>
__device__ int warp_first_false(int lo, int hi, P pred) {
    const int lane = threadIdx.x & 31;
    while (hi - lo > 32) {
        const long long span = hi - lo;
        const bool tr = pred(lo + (int)(span * (lane + 1) / 33));
        const int c = __popc(__ballot_sync(0xffffffffu, tr));  // probes 0..c-1 hold
        const int nlo = c == 0 ? lo : lo + (int)(span * c / 33) + 1;
        const int nhi = c == 32 ? hi : lo + (int)(span * (c + 1) / 33);
        lo = nlo;
        hi = nhi;
    }
    const bool tr = lo + lane < hi && pred(lo + lane);
    return lo + __popc(__ballot_sync(0xffffffffu, tr));
}

// Sort of 64-bit codes c[0, n2) ascending (n2 a power of two, at least 32).
// Each 32-block is sorted in registers by one warp (bitonic, shuffles only);
// then sorted blocks of width w merge pairwise, w = 32, 64, ..., n2 / 2: an
// element's place in the merged block is its offset in its own block plus
// the number of partner-block elements before it (a binary search; left
// elements precede equal right ones, so equal codes keep distinct places).
// One barrier per doubling.  The blocks ping-pong between c and tmp; returns
// the buffer that holds the result.
__device__ unsigned long long* sort_codes(unsigned long long* c, unsigned long long* tmp, int n2) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int b = wid; b < (n2 >> 5); b += nw) {
        const int e = (b << 5) + lane;
        unsigned long long x = c[e];
        for (int k = 2; k <= 32; k <<= 1) {
            const bool asc = (lane & k) == 0;  // every 32-block ends ascending
            for (int j = k >> 1; j > 0; j >>= 1) {
                const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
                const bool lower = (lane & j) == 0;
                const unsigned long long lo = x < y ? x : y, hi = x < y ? y : x;
                x = (lower == asc) ? lo : hi;
            }
        }
        c[e] = x;
    }
    __syncthreads();
    unsigned long long *src = c, *dst = tmp;
    for (int w = 32; w < n2; w <<= 1) {
        for (int i = threadIdx.x; i < n2; i += blockDim.x) {
            const unsigned long long x = src[i];
            const int o = i & (w - 1), blk = i - o;
            const bool right = (blk & w) != 0;
            const unsigned long long* pb = src + (blk ^ w);
            int lo = 0, hi = w;
            while (lo < hi) {  // partner elements before x
                const int mid = (lo + hi) >> 1;
                if (right ? pb[mid] <= x : pb[mid] < x) lo = mid + 1;
                else hi = mid;
            }
            dst[(blk & ~w) + o + lo] = x;
        }
        __syncthreads();
        unsigned long long* t = src;
        src = dst;
        dst = t;
    }
    return src;
}

// The total order of a[0, n) (n <= 65536) as codes in *out[0, n): bits 63..16
// hold the complement of the top 48 bits of the score image (ascending code =
// descending score), bits 15..0 the entry's index.  Runs of equal 48-bit
// prefixes (scores within 2^-36 relative, exact ties among them) are then
// re-ordered by the full total order, one thread per run.  Returns false,
// leaving the codes unusable, when a run is longer than 32 (the caller then
// sorts the entries themselves).  buf holds 2 n2 codes, n2 = pow2 >= max(n, 32);
// *out points into it.
__device__ bool sort_order(const FEntry* a, int n, unsigned long long* buf, int n2, int* flag,
                           const unsigned long long** out) {
    for (int i = threadIdx.x; i < n2; i += blockDim.x)
        buf[i] = i < n ? ((~a[i].key & 0xffffffffffff0000ull) | (unsigned long long)i) : ~0ull;
    if (threadIdx.x == 0) *flag = 0;
    __syncthreads();
    unsigned long long* ord = sort_codes(buf, buf + n2, n2);
    for (int p = threadIdx.x; p < n; p += blockDim.x) {
        const unsigned long long hp = ord[p] >> 16;
        if ((p > 0 && (ord[p - 1] >> 16) == hp) || p + 1 >= n || (ord[p + 1] >> 16) != hp) continue;
        int q = p + 1;  // run [p, q) of equal prefixes, p its first element
        while (q < n && (ord[q] >> 16) == hp && q - p <= 32) ++q;
        if (q - p > 32) {
            *flag = 1;
            continue;
        }
        for (int u = p + 1; u < q; ++u) {  // insertion sort by the total order
            const unsigned long long cu = ord[u];
            int w = u - 1;
            while (w >= p && before(a[cu & 0xffffull], a[ord[w] & 0xffffull])) {
                ord[w + 1] = ord[w];
                --w;
            }
            ord[w + 1] = cu;
        }
    }
    __syncthreads();
    const bool ok = *flag == 0;
    __syncthreads();
    *out = ord;
    return ok;
}

// Inclusive block scan of one int per thread; *total = block sum.
__device__ int block_incl_scan_int(int x, int* red, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) red[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int y = lane < nw ? red[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        red[lane] = y;
    }
    __syncthreads();
    const int r = x + (wid > 0 ? red[wid - 1] : 0);
    *total = red[nw - 1];
    __syncthreads();
    return r;
}

struct Lists {
    const double* zt;   // [K][L][k] z / T_d of the kept tokens
    const double* cum;  // [K][L+1] cumulative row log-normalisers
    const int32_t* ids;
    int L, k, bits;
    __device__ int token(int m, int d, int r) const { return ids[(m * L + d - 1) * k + r]; }
    __device__ double zlog(int m, int d, int r) const { return zt[(m * L + d - 1) * k + r]; }
    __device__ double c(int m, int d) const { return cum[m * (L + 1) + d]; }
    // token at depth j+1 (j < d) of the prefix named by tie key tb
    __device__ int token_at(unsigned long long tb, int j) const {
        const int d = tb_depth(tb), m = tb_mode(tb);
        const int r = (int)(((tb & kRsMask) >> (bits * (d - 1 - j))) & ((1ull << bits) - 1));
        return token(m, j + 1, r);
    }
    __device__ int last_rank(unsigned long long tb) const {
        return (int)((tb & kRsMask) & ((1ull << bits) - 1));
    }
};

// Same token sequence for the first `len` positions of two prefixes.
__device__ bool same_tokens(const Lists& ls, unsigned long long ta, unsigned long long tbb, int len) {
    for (int j = 0; j < len; ++j)
        if (ls.token_at(ta, j) != ls.token_at(tbb, j)) return false;
    return true;
}

__device__ __forceinline__ unsigned long long entry_hash(const Lists& ls, const FEntry& e) {
    const int d = tb_depth(e.tb);
    return hash_step(e.hpar, ls.token(tb_mode(e.tb), d, ls.last_rank(e.tb)));
}

// Open addressing on the prefix hash: the bucket of entry i (claimed or found).
// Equal hashes of different prefixes are caught afterwards by comparing token
// sequences (a 2^-64 event per pair, reported as a failed tree, never merged).
__device__ int hash_bucket(unsigned long long h, unsigned long long* hkey, int hcap) {
    unsigned int b = (unsigned int)(h ^ (h >> 32)) & (hcap - 1);
    for (int probe = 0; probe < hcap; ++probe, b = (b + 1) & (hcap - 1)) {
        const unsigned long long old = atomicCAS(&hkey[b], 0ull, h);
        if (old == 0ull || old == h) return (int)b;
    }
    return -1;
}

// ---------------------------------------------------------------------------
// Threshold expansion (one mode).
//
// Scores never rise along a path (each log q is at most 0, and at equal score
// a parent's shorter tie key comes first), so for any lower bound theta of the
// B-th best key, the B best prefixes are the B best among the prefixes whose
// key is at least theta, and that set is closed under taking parents.  Every
// set of B prefixes gives such a bound: the key of its worst member.  The
// first d0 levels are enumerated in full and give the first bound; each
// further level keeps the children of the last level's kept prefixes whose
// key reaches the bound, and the bound then rises to the B-th best key of
// everything kept so far.  Keys are counted in bins of equal width below the
// best enumerated key; a bound is the lower edge of the bin that holds the
// B-th best key.  The B best kept prefixes under (key desc, tie key asc) are
// the tree, in that order: the same set and order as the rounds.
//
// A child's key is exact float64 (the rounds' arithmetic, clamped to its
// parent's key as there).  Float64 issues at
// one warp instruction per 64 clocks per SM quarter whatever the active lanes,
// so each level first bounds, in float32, how many of a parent's children can
// pass (they pass as a run from rank 0: its list is sorted), and evaluates
// only those (parent, rank) pairs, packed densely over the warps.
//
// Returns false when the candidates outgrow their arrays (or, which the
// clamped keys exclude, a child would precede its parent); the caller then
// runs the rounds, which rewrite every output.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int thr_pidx(int b) { return b + (b >> 6); }

__device__ __forceinline__ int warp_incl_scan(int x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// One warp: the bin that holds the B-th key (bin 0 holds the best keys), from
// the row sums and then the crossing row's bins; *upto = keys in bins up to
// it.  -1 when the counts read do not reach B.  Counts read while other warps
// add to them are at most the true counts of real candidates, so a bin found
// from them still has at least B real keys at or above it.
__device__ int thr_warp_bin(const int* hist, const int* rows, int B, int* upto) {
    const int lane = threadIdx.x & 31;
    const int rs = rows[lane];
    const int incl = warp_incl_scan(rs), excl = incl - rs;
    const unsigned int hit = __ballot_sync(0xffffffffu, excl < B && incl >= B);
    if (hit == 0u) return -1;
    const int c = __ffs(hit) - 1;
    const int cex = __shfl_sync(0xffffffffu, excl, c);
    const int h0 = hist[c * 65 + 2 * lane], h1 = hist[c * 65 + 2 * lane + 1];
    const int ex2 = cex + warp_incl_scan(h0 + h1) - h0 - h1;
    const int q = (ex2 < B && ex2 + h0 >= B) ? 0 : ((ex2 + h0 < B && ex2 + h0 + h1 >= B) ? 1 : -1);
    const unsigned int hit2 = __ballot_sync(0xffffffffu, q >= 0);
    if (hit2 == 0u) return -1;
    const int l2 = __ffs(hit2) - 1;
    const int q2 = __shfl_sync(0xffffffffu, q, l2);
    *upto = __shfl_sync(0xffffffffu, q == 0 ? ex2 + h0 : ex2 + h0 + h1, l2);
    return 64 * c + 2 * l2 + q2;
}

// float32 of a float64, rounded toward zero (integer operations only): within
// one float32 unit of the value, 0 below float32's normal range, infinite above it.
__device__ __forceinline__ float f32_trunc(double x) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(x);
    const unsigned int sign = (unsigned int)(u >> 32) & 0x80000000u;
    const int e = (int)((u >> 52) & 0x7FF);
    if (e == 0x7FF) return __uint_as_float(sign | 0x7F800000u | ((u << 12) != 0ull ? 0x400000u : 0u));
    const int E = e - 1023 + 127;
    if (E >= 255) return __uint_as_float(sign | 0x7F800000u);
    if (E <= 0) return __uint_as_float(sign);
    return __uint_as_float(sign | ((unsigned int)E << 23) | (unsigned int)((u >> 29) & 0x7FFFFFull));
}

// Shared scalars of the threshold expansion (set before the kernel's first barrier).
struct ThrState {
    unsigned long long whi[32], wlo[32];  // per warp: largest and least live key
    int wlive[32];                        // per warp: live keys
    int lev[3], slot[3];                  // per depth (mod 3): candidates, listed pairs
    int fail;
};
// The candidate arrays and tables, laid out after the lists in shared memory.
struct ThrMem {
    unsigned long long *key, *tb;
    double* zs;
    int *par, *node, *sidx;
    float* zf;  // z sums in float32
    int *hist, *hbase, *rows, *slots;
    float *ztf, *zmag, *cf;
};
__device__ __forceinline__ ThrMem thr_mem(uint8_t* base, int cap, int L, int k) {
    ThrMem m;
    m.key = reinterpret_cast<unsigned long long*>(base);
    m.tb = m.key + cap;
    m.zs = reinterpret_cast<double*>(m.tb + cap);
    m.par = reinterpret_cast<int*>(m.zs + cap);
    m.node = m.par + cap;  // node of a kept candidate, 0 otherwise
    m.sidx = m.node + cap;  // candidates in bin order
    m.zf = reinterpret_cast<float*>(m.sidx + cap);
    m.hist = reinterpret_cast<int*>(m.zf + cap);
    m.hbase = m.hist + kThrBinWords;
    m.rows = m.hbase + kThrBinWords;  // bins per row of 64
    m.slots = m.rows + 32;  // two lists of parent << 5 | rank, one per level parity
    m.ztf = reinterpret_cast<float*>(m.slots + 2 * kThrSlots);  // the lists' z / T_d in float32
    m.zmag = m.ztf + L * k;  // per depth: largest finite |ztf| (formed by integer maxima)
    m.cf = m.zmag + L;       // C(d) in float32, d = 0..L
    return m;
}

// The caller has zeroed the bin counts, row sums and magnitudes, set ztf and
// zmag from the lists and the state's counters to 0, behind one barrier.
__device__ bool thr_build(const Lists& ls, const ThrMem& tm, ThrState& ts, const BuildPlan& plan,
                          int L, int k, int B, int bits, int32_t* par, int32_t* tok,
                          int32_t* dep, float* sc, double* sc64, int32_t* rk, int32_t* md) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nthr = blockDim.x;
    const int nw = nthr >> 5;
    const int cap = plan.tcap, n0 = plan.n0, d0 = plan.d0;
    unsigned long long* ckey = tm.key;
    unsigned long long* ctb = tm.tb;
    double* czs = tm.zs;
    int* cpar = tm.par;
    int* cnode = tm.node;
    int* sidx = tm.sidx;
    float* czf = tm.zf;
    int* hist = tm.hist;
    int* hbase = tm.hbase;
    int* rows = tm.rows;
    int* slots = tm.slots;
    const float* ztf = tm.ztf;
    const float* zmag = tm.zmag;
    float* cf = tm.cf;
    int* s_lev = ts.lev;
    int* s_slot = ts.slot;
    int& s_fail = ts.fail;
    const unsigned long long live_min = order_key(-DBL_MAX);  // below: -inf
    if (tid <= L) cf[tid] = f32_trunc(ls.c(0, tid));

    // ---- levels 1..d0 in full, two levels a pass: level d from level d-1's
    // stored sums, level d+1 from them too (its parent's sum formed again,
    // by the same operations) ----
    unsigned long long hi = 0ull, lo = ~0ull;
    int live = 0;
    bool bad = false;
    if (tid < L) {
        const double c = ls.c(0, tid + 1);
        bad = !(c > -INFINITY && c < INFINITY);
    }
    {
        int off = 0, poff = 0, lev = k;  // level d starts at off, level d-1 at poff
        for (int d = 1; d <= d0; d += 2) {
            const bool two = d + 1 <= d0;
            const int n1 = lev, n2 = two ? lev * k : 0;
            const double c1 = ls.c(0, d), c2 = two ? ls.c(0, d + 1) : 0.0;
            for (int i = tid; i < n1 + n2; i += nthr) {
                int idx, pp;
                double z, cc;
                unsigned long long tb, kpar;  // kpar: the parent's key
                if (i < n1) {
                    const unsigned int q = plan.kdiv.div((unsigned int)i);
                    const int r = i - (int)q * k;
                    pp = d == 1 ? -1 : poff + (int)q;
                    z = (d == 1 ? 0.0 : czs[pp]) + ls.zlog(0, d, r);
                    kpar = d == 1 ? ~0ull : ckey[pp];
                    tb = ((unsigned long long)d << 59) |
                         (d == 1 ? 0ull : (((ctb[pp] & kRsMask) << bits) & kRsMask)) |
                         (unsigned long long)r;
                    idx = off + i;
                    cc = c1;
                } else {
                    const int j = i - n1;
                    const unsigned int q = plan.kdiv.div((unsigned int)j);  // parent in level d
                    const int r2 = j - (int)q * k;
                    const unsigned int q1 = plan.kdiv.div(q);  // grandparent in level d-1
                    const int r1 = (int)q - (int)q1 * k;
                    const int gp = d == 1 ? -1 : poff + (int)q1;
                    const double z1 = (d == 1 ? 0.0 : czs[gp]) + ls.zlog(0, d, r1);
                    z = z1 + ls.zlog(0, d + 1, r2);
                    const unsigned long long k1 = order_key(z1 - c1);  // the parent's key
                    kpar = d == 1 ? k1 : min(k1, ckey[gp]);
                    const unsigned long long t1 =
                        (d == 1 ? 0ull : (((ctb[gp] & kRsMask) << bits) & kRsMask)) |
                        (unsigned long long)r1;
                    tb = ((unsigned long long)(d + 1) << 59) | ((t1 << bits) & kRsMask) |
                         (unsigned long long)r2;
                    pp = off + (int)q;
                    idx = off + n1 + j;
                    cc = c2;
                }
                const double sv = z - cc;
                // a child's key is never above its parent's: where the rounding
                // of the two path sums would put it there, it takes the parent's
                const unsigned long long key = min(order_key(sv), kpar);
                if (sv != sv) bad = true;
                ckey[idx] = key;
                ctb[idx] = tb;
                czs[idx] = z;
                czf[idx] = f32_trunc(z);
                cpar[idx] = pp;
                cnode[idx] = 0;
                if (key >= live_min) {
                    hi = max(hi, key);
                    lo = min(lo, key);
                    ++live;
                }
            }
            poff = two ? off + n1 : off;  // the pass's last level
            off += n1 + n2;
            lev = two ? n2 * k : n1 * k;
            if (d + 2 <= d0) __syncthreads();  // the next pass reads these sums
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        live += __shfl_xor_sync(0xffffffffu, live, o);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) s_fail = 1;
    if (lane == 0) {
        ts.whi[wid] = hi;
        ts.wlo[wid] = lo;
        ts.wlive[wid] = live;
    }
    __syncthreads();
    if (s_fail != 0) return false;
    unsigned long long top = 0ull, bot = ~0ull;
    int nlive = 0;
    for (int w = 0; w < nw; ++w) {
        top = max(top, ts.whi[w]);
        bot = min(bot, ts.wlo[w]);
        nlive += ts.wlive[w];
    }
    if (nlive < B) return false;
    // bins of width 2^sh below the best key: bin(key) = (top - key) >> sh
    const unsigned long long span = top - bot;
    const int sh = span == 0ull ? 0 : max(0, 64 - __clzll((long long)span) - kThrBinBits);
    auto bin_of = [&](unsigned long long key) {
        const unsigned long long b = (top - key) >> sh;
        return (int)(b < (unsigned long long)kThrBins ? b : kThrBins - 1);
    };
    auto count_key = [&](unsigned long long key) {
        const int b = bin_of(key);
        atomicAdd(&hist[thr_pidx(b)], 1);
        atomicAdd(&rows[b >> 6], 1);
    };
    // the smallest key of bin b
    auto bin_floor = [&](int b) {
        if (b < 0) return live_min;
        const unsigned long long off = ((unsigned long long)b << sh) + ((1ull << sh) - 1ull);
        const unsigned long long f = top > off ? top - off : 0ull;
        return f > live_min ? f : live_min;
    };
    for (int i = tid; i < n0; i += nthr) {
        const unsigned long long key = ckey[i];
        if (key >= live_min) count_key(key);
    }
    __syncthreads();
    int upto = 0;
    unsigned long long theta = bin_floor(thr_warp_bin(hist, rows, B, &upto));

    // ---- levels d0+1, ...: kept children of the last level's kept prefixes ----
    // Per prefix, a float32 bound on its passing children: child r can pass
    // only if ztf[r] >= g.  The margin covers the error of every float32
    // operand and step (a few units of 2^-24 of the magnitudes involved,
    // against 2^-18 here; the absolute term covers values below float32's
    // normal range) and that of the float64 evaluation.  Where an operand does
    // not fit float32, g is not finite and every rank is evaluated.  A bound
    // formed with an earlier (lower) theta only lists more pairs: each pair's
    // exact key is tested against the current theta.
    auto bound = [&](float zsf, float thf, int dc) {  // dc: the children's depth
        const float cdf = cf[dc];
        const float m = 0x1p-18f * (fabsf(thf) + fabsf(cdf) + fabsf(zsf) + zmag[dc - 1]) + 1e-30f;
        const float g = ((thf - m) + cdf) - zsf;
        if (!(g > -INFINITY && g < INFINITY)) return k;
        const float* zr = ztf + (dc - 1) * k;
        int cb = 0;  // the list is sorted: the ranks that pass are a run from 0
        for (int r = 0; r < k; ++r) cb += zr[r] >= g ? 1 : 0;
        return cb;
    };
    // list the (prefix, rank) pairs of the lanes' prefixes for depth dc (all lanes call)
    auto list_pairs = [&](int p, int cb, int dc) {
        const int inc = warp_incl_scan(cb);
        int at = 0;
        if (lane == 31 && inc > 0) at = atomicAdd(&s_slot[dc % 3], inc);
        at = __shfl_sync(0xffffffffu, at, 31) + inc - cb;
        int* sl = slots + (dc & 1) * kThrSlots;
        for (int r = 0; r < cb; ++r) {
            if (at + r < kThrSlots) sl[at + r] = (p << 5) | r;
            else s_fail = 1;
        }
    };
    int pe = n0;
    if (d0 < L) {
        int lev = 1;
        for (int j = 0; j < d0; ++j) lev *= k;
        const float thf = f32_trunc(key_score(theta));
        for (int p0 = n0 - lev; p0 < n0; p0 += nthr) {  // level d0
            const int p = p0 + tid;
            const int cb = p < n0 && ckey[p] >= theta ? bound(czf[p], thf, d0 + 1) : 0;
            list_pairs(p, cb, d0 + 1);
        }
    }
    __syncthreads();
    if (s_fail != 0) return false;
    for (int d = d0 + 1; d <= L; ++d) {
        const int ns = s_slot[d % 3];
        if (ns == 0) break;
        const double cd = ls.c(0, d);
        int* cnt = &s_lev[d % 3];
        if (tid == 0) {  // last read before the previous barrier
            s_lev[(d + 1) % 3] = 0;
            s_slot[(d + 2) % 3] = 0;
        }
        // the exact keys of the listed pairs, packed over all threads; each
        // kept child lists its own pairs for the next depth (bounded with the
        // theta of this depth: later rises only drop more of them)
        const int* sl = slots + (d & 1) * kThrSlots;
        const float thf = f32_trunc(key_score(theta));
        for (int j0 = 0; j0 < ns; j0 += nthr) {
            const int j = j0 + tid;
            bool ok = false;
            int p = 0, r = 0;
            double z = 0.0;
            unsigned long long key = 0ull;
            if (j < ns) {
                p = sl[j] >> 5;
                r = sl[j] & 31;
                z = czs[p] + ls.zlog(0, d, r);
                key = min(order_key(z - cd), ckey[p]);  // never above the parent
                ok = key >= theta;
            }
            const unsigned int ball = __ballot_sync(0xffffffffu, ok);
            int at = 0;
            if (lane == 0 && ball != 0u) at = atomicAdd(cnt, __popc(ball));
            at = __shfl_sync(0xffffffffu, at, 0);
            int pos = -1, cb = 0;
            if (ok) {
                pos = pe + at + __popc(ball & ((1u << lane) - 1u));
                if (pos < cap) {
                    const float zf = f32_trunc(z);
                    ckey[pos] = key;
                    ctb[pos] = ((unsigned long long)d << 59) |
                               (((ctb[p] & kRsMask) << bits) & kRsMask) | (unsigned long long)r;
                    czs[pos] = z;
                    czf[pos] = zf;
                    cpar[pos] = p;
                    cnode[pos] = 0;
                    count_key(key);
                    if (d < L) cb = bound(zf, thf, d + 1);
                } else {
                    s_fail = 1;  // out of room
                }
            }
            list_pairs(pos, cb, d + 1);
        }
        {
            // the bound rises to the B-th best key kept so far, as each warp
            // sees the counts before the barrier (while others still add)
            const unsigned long long th = bin_floor(thr_warp_bin(hist, rows, B, &upto));
            theta = th > theta ? th : theta;
        }
        __syncthreads();
        if (s_fail != 0) return false;
        pe += *cnt;
    }
    const int N = pe;

    // ---- the B best: candidates of bins up to the B-th key's, ranked within bins ----
    // (no warp adds to the counts any more: every warp reads the same values)
    const int b1 = thr_warp_bin(hist, rows, B, &upto);
    const int M2 = upto;
    if (b1 < 0) return false;  // cannot happen: the counts hold at least B live keys
    for (int row = wid; row < 32; row += nw) {  // bases: keys in earlier bins
        const int rs = rows[lane];
        const int rbase = __shfl_sync(0xffffffffu, warp_incl_scan(rs) - rs, row);
        const int h0 = hist[row * 65 + 2 * lane], h1 = hist[row * 65 + 2 * lane + 1];
        const int ex2 = rbase + warp_incl_scan(h0 + h1) - h0 - h1;
        hbase[row * 65 + 2 * lane] = ex2;
        hbase[row * 65 + 2 * lane + 1] = ex2 + h0;
    }
    __syncthreads();
    for (int i = tid; i < N; i += nthr) {
        const unsigned long long key = ckey[i];
        if (key < live_min) continue;
        const int b = bin_of(key);
        if (b > b1) continue;
        const int sl = hbase[thr_pidx(b)] + atomicSub(&hist[thr_pidx(b)], 1) - 1;
        if (TSD_IN(sl, M2, kChkBuild)) sidx[sl] = i;
    }
    __syncthreads();
    int* ord = reinterpret_cast<int*>(czs);  // z sums are spent; 2 * cap >= B slots
    for (int sl = tid; sl < M2; sl += nthr) {
        const int c = sidx[sl];
        const unsigned long long key = ckey[c], tb = ctb[c];
        const int b = bin_of(key);
        const int lo = hbase[thr_pidx(b)], hi = b + 1 < kThrBins ? hbase[thr_pidx(b + 1)] : M2;
        int rank = lo;
        for (int j = lo; j < hi; ++j) {
            const int cj = sidx[j];
            const unsigned long long kj = ckey[cj];
            rank += (kj > key || (kj == key && ctb[cj] < tb)) ? 1 : 0;
        }
        if (rank < B) {
            ord[rank] = c;
            cnode[c] = rank + 1;
        }
    }
    __syncthreads();
    for (int pos = tid; pos < B; pos += nthr) {
        const int c = ord[pos], node = pos + 1;
        const unsigned long long tb = ctb[c];
        const int d = tb_depth(tb), r = ls.last_rank(tb);
        const double sv = key_score(ckey[c]);
        const int pp = cpar[c];
        const int pn = pp < 0 ? 0 : cnode[pp];
        if (pp >= 0 && (pn <= 0 || pn >= node)) s_fail = 1;  // a child before its parent
        par[node] = pn;
        tok[node] = ls.token(0, d, r);
        dep[node] = d;
        sc[node] = (float)sv;
        if (sc64) sc64[node] = sv;
        if (rk) rk[node] = r;
        if (md) md[node] = 0;
    }
    if (tid == 0) {
        par[0] = -1;
        tok[0] = -1;
        dep[0] = 0;
        sc[0] = 0.0f;
        if (sc64) sc64[0] = 0.0;
        if (rk) rk[0] = -1;
        if (md) md[0] = -1;
    }
    __syncthreads();
    return s_fail == 0;
}

__global__ void __launch_bounds__(kBuildThreads, 1)
build_tree_kernel(BuildWs ws, BuildPlan plan, int K, int L, int k, int B, int bits,
                  int32_t* __restrict__ parent, int32_t* __restrict__ token,
                  int32_t* __restrict__ depth, float* __restrict__ score,
                  int32_t* __restrict__ rank, int32_t* __restrict__ mode,
                  int32_t* __restrict__ n_nodes_out, int32_t* __restrict__ status) {
    pdl_entry();
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_bad, s_nF, s_nX, s_nS, s_D, s_posB, s_thr_on;
    __shared__ FEntry s_thr;  // pruning bound: entries not before it are dead
    __shared__ int red[32];
    const int t = blockIdx.x, tid = threadIdx.x;
    const int nl = K * L * k;
    uint8_t* p = smem;
    double* zt = reinterpret_cast<double*>(p);
    double* cum = zt + nl;
    int32_t* ids = reinterpret_cast<int32_t*>(cum + K * (L + 1));
    p += plan.lists;
    FEntry* S = reinterpret_cast<FEntry*>(p);
    unsigned long long* Scode = reinterpret_cast<unsigned long long*>(p + plan.sbytes - plan.scode_bytes);
    p += plan.sbytes;
    uint8_t* big = plan.big_in_smem ? p : ws.heap + (size_t)t * ws.heap_stride;
    FEntry* F[2] = {reinterpret_cast<FEntry*>(big), reinterpret_cast<FEntry*>(big) + plan.fcap};
    big += plan.fbytes;
    FEntry* X[2] = {reinterpret_cast<FEntry*>(big), reinterpret_cast<FEntry*>(big) + plan.xcap};
    big += plan.xbytes;
    unsigned long long* hkey = reinterpret_cast<unsigned long long*>(big);
    int* hval = reinterpret_cast<int*>(big + sizeof(unsigned long long) * plan.hcap);
    big += plan.hbytes;
    int* flag = reinterpret_cast<int*>(big);  // [xcap] first-occurrence marks, then ranks
    const Lists ls{zt, cum, ids, L, k, bits};
    const int stride = B + 1;
    // one mode: the threshold expansion's tables are set up beside the lists
    __shared__ ThrState s_ts;
    const bool thr_on = K == 1 && B > 0 && plan.tcap > 0;
    const ThrMem tm = thr_mem(smem + plan.lists, plan.tcap, L, k);

    if (tid == 0) {
        s_bad = 0;
        s_nF = 0;
        s_nX = 0;
        s_D = 0;
        for (int j = 0; j < 3; ++j) s_ts.lev[j] = s_ts.slot[j] = 0;
        s_ts.fail = 0;
    }
    if (thr_on) {
        for (int i = tid; i < kThrBinWords; i += blockDim.x) tm.hist[i] = 0;
        if (tid < 32) tm.rows[tid] = 0;
        if (tid < L) tm.zmag[tid] = 0.0f;
    }
    __syncthreads();
    for (int i = tid; i < nl; i += blockDim.x) {
        const double x = ws.top_zt[(int64_t)t * nl + i];
        zt[i] = x;
        ids[i] = ws.top_id[(int64_t)t * nl + i];
        if (x != x) s_bad = 1;
        if (thr_on) {
            // largest finite |z / T_d| per depth in float32; a finite value that
            // float32 cannot hold makes it infinite (the bound then lists every rank)
            const float xf = f32_trunc(x);
            tm.ztf[i] = xf;
            if (x > -INFINITY && x < INFINITY)
                atomicMax(reinterpret_cast<int*>(tm.zmag) + i / k, __float_as_int(fabsf(xf)));
        }
    }
    if (K == 1) {
        // C(d), summed left to right: warp 0 loads the L normalisers at once
        if (tid < 32) {
            const double l = tid < L ? ws.lse[(int64_t)t * L + tid] : 0.0;
            if (l != l) s_bad = 1;
            double c = 0.0;
            if (tid == 0) cum[0] = 0.0;
            for (int d = 0; d < L; ++d) {
                c = c + __shfl_sync(0xffffffffu, l, d);
                if (tid == d) cum[d + 1] = c;
            }
        }
    } else {
        for (int i = tid; i < K * L; i += blockDim.x) {  // the row log-normalisers, all at once
            const double l = ws.lse[(int64_t)t * K * L + i];
            if (l != l) s_bad = 1;
            cum[(i / L) * (L + 1) + i % L + 1] = l;
        }
        __syncthreads();
        for (int m = tid; m < K; m += blockDim.x) {  // C_m(d), summed left to right in place
            double c = 0.0;
            cum[m * (L + 1)] = 0.0;
            for (int d = 1; d <= L; ++d) {
                c = c + cum[m * (L + 1) + d];
                cum[m * (L + 1) + d] = c;
            }
        }
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    int fc = 0, xc = 0;  // current buffer indices
    int32_t* par = parent + (int64_t)t * stride;
    int32_t* tok = token + (int64_t)t * stride;
    int32_t* dep = depth + (int64_t)t * stride;
    float* sc = score + (int64_t)t * stride;
    int32_t* rk = rank ? rank + (int64_t)t * stride : nullptr;
    int32_t* md = mode ? mode + (int64_t)t * stride : nullptr;
    // one mode: threshold expansion first, the rounds when it declines
    bool done = false;
    if (!bad && thr_on)
        done = thr_build(ls, tm, s_ts, plan, L, k, B, bits, par, tok, dep, sc,
                         ws.score64 ? ws.score64 + (int64_t)t * stride : nullptr, rk, md);
    if (!bad && B > 0 && !done) {  // B = 0: the tree is the root alone
        // seeds: the root's children, all k first tokens of every mode
        const int n2 = pow2_at_least(K * k < 32 ? 32 : K * k);
        for (int i = tid; i < n2; i += blockDim.x) {
            FEntry e;
            e.key = kSentinelKey;
            e.tb = ~0ull;
            e.zsum = 0.0;
            e.hpar = kRootHash;
            if (i < K * k) {
                const int m = i / k, r = i % k;
                const double z = 0.0 + ls.zlog(m, 1, r);
                const double sv = z - ls.c(m, 1);
                if (sv != -INFINITY) {
                    e.key = order_key(sv);
                    e.tb = (1ull << 59) | ((unsigned long long)m << 56) | (unsigned long long)r;
                    e.zsum = z;
                }
            }
            F[0][i] = e;
        }
        __syncthreads();
        sort_entries(F[0], n2);
        if (tid == 0) {
            int nF = 0;
            while (nF < K * k && F[0][nF].key != kSentinelKey) ++nF;
            s_nF = nF;
            s_thr_on = 0;
        }
        __syncthreads();
        const int M = plan.M;
        for (int round = 0; round < (1 << 20); ++round) {
            const int nF = s_nF, nX = s_nX;
            if (nF == 0) break;
            const int bn = min(M, nF);
            // Children of the taken entries, one thread per (entry, rank) slot.
            // An entry's children are sorted by rank (its list is), and the
            // unusable ones (-inf, or not better than the pruning bound) form a
            // suffix; a block scan over the slots' flags packs the usable ones.
            const FEntry thr = s_thr;
            const bool thr_on = s_thr_on != 0;
            const int nslot = bn * k;
            // kSlotsPerThread slots per thread, kept in slot order: thread
            // tid owns slots kSlotsPerThread * tid + u
            FEntry ch[kSlotsPerThread];
            int okc[kSlotsPerThread];
            int nok = 0;
#pragma unroll
            for (int u = 0; u < kSlotsPerThread; ++u) {
                okc[u] = 0;
                const int c = kSlotsPerThread * tid + u;
                if (c < nslot) {
                    const int i = c / k, r = c - i * k;
                    const FEntry e = F[fc][i];
                    const int d = tb_depth(e.tb), m = tb_mode(e.tb);
                    if (d < L) {
                        const double z = e.zsum + ls.zlog(m, d + 1, r);
                        const double sv = z - ls.c(m, d + 1);
                        // never above the parent (rounding of the two path sums)
                        const unsigned long long kc = order_key(sv);
                        ch[u].key = kc < e.key ? kc : e.key;
                        ch[u].tb = ((unsigned long long)(d + 1) << 59) |
                                   ((unsigned long long)m << 56) |
                                   (((e.tb & kRsMask) << bits) & kRsMask) | (unsigned long long)r;
                        ch[u].zsum = z;
                        okc[u] = sv != -INFINITY && (!thr_on || before(ch[u], thr));
                        // one mode: a prefix is named by its tie key, no hash needed
                        ch[u].hpar = (okc[u] && K > 1) ? entry_hash(ls, e) : 0ull;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kSlotsPerThread; ++u) nok += okc[u];
            int written;
            int pos = block_incl_scan_int(nok, red, &written) - nok;
#pragma unroll
            for (int u = 0; u < kSlotsPerThread; ++u)
                if (okc[u] && TSD_IN(pos, M * k, kChkBuild)) S[pos++] = ch[u];
            if (tid == 0) s_nS = written;
            __syncthreads();
            const int nS = s_nS;
            // the successors' order: sorted 64-bit codes (S itself stays put),
            // or, after a long run of tied scores, S sorted in place
            const unsigned long long* Sord = nullptr;
            if (nS > 1) {
                const int n2S = pow2_at_least(nS < 32 ? 32 : nS);
                if (!sort_order(S, nS, Scode, n2S, &red[31], &Sord)) {
                    Sord = nullptr;
                    for (int i = nS + tid; i < n2S; i += blockDim.x) {
                        S[i].key = kSentinelKey;
                        S[i].tb = ~0ull;
                    }
                    __syncthreads();
                    sort_entries(S, n2S);
                }
            }
            if (nX + bn > plan.xcap || nF - bn + nS > plan.fcap) {  // cannot happen (see plan)
                if (tid == 0) s_bad = 3;
                __syncthreads();
                break;
            }
            // Taken entries join X (both sorted); the rest of the frontier
            // merges with the successors.
            merge_two(X[xc ^ 1], X[xc], nX, F[fc], bn, F[fc ^ 1], F[fc] + bn, nF - bn, S, nS, Sord);
            xc ^= 1;
            fc ^= 1;
            int nXn = nX + bn, nFn = nF - bn + nS;
            // Distinct prefixes in X: first occurrences in the sorted list.
            int D;
            if (K == 1) {
                D = nXn;
            } else {
                for (int i = tid; i < plan.hcap; i += blockDim.x) {
                    hkey[i] = 0ull;
                    hval[i] = INT_MAX;
                }
                __syncthreads();
                // first occurrence of each prefix = smallest X position in its bucket
                for (int i = tid; i < nXn; i += blockDim.x) {
                    const int b = hash_bucket(entry_hash(ls, X[xc][i]) | 1ull, hkey, plan.hcap);
                    flag[i] = b;
                    if (b < 0) s_bad = 2;
                    else atomicMin(&hval[b], i);
                }
                __syncthreads();
                for (int i = tid; i < nXn; i += blockDim.x) {
                    const int b = flag[i];
                    if (b < 0) continue;
                    const int j = hval[b];
                    if (j != i) {
                        const int d = tb_depth(X[xc][i].tb);
                        if (tb_depth(X[xc][j].tb) != d || !same_tokens(ls, X[xc][j].tb, X[xc][i].tb, d))
                            s_bad = 2;  // a hash collision: refuse rather than merge
                    }
                }
                __syncthreads();
                for (int i = tid; i < nXn; i += blockDim.x) flag[i] = (flag[i] >= 0 && hval[flag[i]] == i) ? 1 : 0;
                __syncthreads();
                // ranks of the first occurrences (block scan over chunks)
                int base = 0;
                for (int c0 = 0; c0 < nXn; c0 += blockDim.x) {
                    const int i = c0 + tid;
                    const int f = i < nXn ? flag[i] : 0;
                    int tot;
                    const int inc = block_incl_scan_int(f, red, &tot);
                    if (i < nXn) flag[plan.xcap + i] = f ? base + inc - 1 : -1;
                    base += tot;
                }
                D = base;
                __syncthreads();
            }
            if (D >= B) {
                // the B-th distinct prefix bounds everything worth keeping
                if (tid == 0) s_posB = (K == 1) ? B - 1 : -1;
                __syncthreads();
                if (K > 1)
                    for (int i = tid; i < nXn; i += blockDim.x)
                        if (flag[plan.xcap + i] == B - 1) s_posB = i;
                __syncthreads();
                const int posB = s_posB;
                const FEntry th = X[xc][posB];
                nXn = posB + 1;
                // frontier entries not before the bound can never be kept;
                // nor can entries past the frontier's first K*B: at most B of
                // its distinct prefixes can still be kept, and each prefix
                // appears at most K times (once per mode), so the best B are
                // among the first K*B.  (Without this cap the frontier can
                // outgrow its buffer when many candidates crowd the bound.)
                if (tid < 32) {
                    const FEntry* Fc = F[fc];
                    const int lo = warp_first_false(0, nFn, [&](int i) { return before(Fc[i], th); });
                    if (tid == 0) {
                        s_nF = min(lo, K * B);
                        s_thr = th;
                        s_thr_on = 1;
                    }
                }
            } else if (tid < 32) {
                // the (K*B)-th entry of X and the frontier merged: at least B
                // distinct prefixes are that good, so worse entries are dead
                const int want = K * B;
                int keepF = nFn;
                if (nXn + nFn >= want) {
                    // co-rank: ia entries of X and want - ia of F form the best `want`
                    const FEntry *Xc = X[xc], *Fc = F[fc];
                    const int ia = warp_first_false(max(0, want - nFn), min(want, nXn), [&](int mid) {
                        return before(Xc[mid], Fc[want - mid - 1]);
                    });
                    const int ib = want - ia;
                    // the want-th best is the worse of X[ia-1] and F[ib-1]
                    FEntry th;
                    if (ia == 0) th = F[fc][ib - 1];
                    else if (ib == 0) th = X[xc][ia - 1];
                    else th = before(X[xc][ia - 1], F[fc][ib - 1]) ? F[fc][ib - 1] : X[xc][ia - 1];
                    keepF = ib;  // F[ib..] are all after th
                    if (tid == 0) {
                        s_thr = th;
                        s_thr_on = 1;
                    }
                    // th itself may be kept (not "before" itself); keep F entries up to it
                }
                if (tid == 0) s_nF = keepF;
            }
            if (tid == 0) {
                s_nX = nXn;
                s_D = min(D, B);
            }
            __syncthreads();
        }
        __syncthreads();
    }
    // ---- output: nodes in X order (first occurrences), parents resolved ----
    const bool failed = bad || s_bad != 0;
    const int nX = failed ? 0 : s_nX;
    const int nn = failed ? 0 : (done ? B + 1 : s_D + 1);
    if (!failed && !done) {
        // node index of each kept entry: K == 1 -> position + 1; K > 1 ->
        // distinct rank + 1 for first occurrences
        // table: prefix -> node (keyed by the prefix hash, confirmed by tokens)
        for (int i = tid; i < plan.hcap; i += blockDim.x) {
            hkey[i] = 0ull;
            hval[i] = INT_MAX;
        }
        __syncthreads();
        // key of a node's prefix: its tie key for one mode (exact), else the
        // hash of its token sequence (matches confirmed by the tokens)
        auto node_key = [&](const FEntry& e) {
            return K == 1 ? e.tb : (entry_hash(ls, e) | 1ull);
        };
        auto first_bucket = [&](unsigned long long h) {
            const unsigned long long x = hash_step(h, 0);
            return (unsigned int)(x ^ (x >> 32)) & (plan.hcap - 1);
        };
        for (int i = tid; i < nX; i += blockDim.x) {
            const int node = (K == 1) ? i + 1 : flag[plan.xcap + i] + 1;
            if (node <= 0 || !TSD_IN(node, stride, kChkBuild)) continue;
            const FEntry e = X[xc][i];
            const unsigned long long h = node_key(e);
            unsigned int b = first_bucket(h);
            for (int probe = 0; probe < plan.hcap; ++probe, b = (b + 1) & (plan.hcap - 1)) {
                const unsigned long long old = atomicCAS(&hkey[b], 0ull, h);
                if (old == 0ull) {
                    hval[b] = i;  // X position of this node's entry
                    break;
                }
                if (old == h) {  // two distinct nodes with one hash
                    s_bad = 2;
                    break;
                }
            }
            const int d = tb_depth(e.tb), m = tb_mode(e.tb), r = ls.last_rank(e.tb);
            tok[node] = ls.token(m, d, r);
            dep[node] = d;
            sc[node] = (float)key_score(e.key);
            if (ws.score64) ws.score64[(int64_t)t * stride + node] = key_score(e.key);
            if (rk) rk[node] = r;
            if (md) md[node] = m;
        }
        __syncthreads();
        for (int i = tid; i < nX; i += blockDim.x) {
            const int node = (K == 1) ? i + 1 : flag[plan.xcap + i] + 1;
            if (node <= 0 || !TSD_IN(node, stride, kChkBuild)) continue;
            const FEntry e = X[xc][i];
            const int d = tb_depth(e.tb);
            int pn = 0;
            if (d > 1) {
                // the parent's key: its tie key (this one without its last rank
                // digit) for one mode, else the hash of its token sequence
                const unsigned long long h =
                    K == 1 ? (((unsigned long long)(d - 1) << 59) |
                              ((unsigned long long)tb_mode(e.tb) << 56) | ((e.tb & kRsMask) >> bits))
                           : (e.hpar | 1ull);
                unsigned int b = first_bucket(h);
                pn = -1;
                for (int probe = 0; probe < plan.hcap; ++probe, b = (b + 1) & (plan.hcap - 1)) {
                    const unsigned long long kk = hkey[b];
                    if (kk == 0ull) break;
                    if (kk == h) {
                        const int j = hval[b];
                        if (K == 1 || (tb_depth(X[xc][j].tb) == d - 1 &&
                                       same_tokens(ls, X[xc][j].tb, e.tb, d - 1))) {
                            pn = (K == 1) ? j + 1 : flag[plan.xcap + j] + 1;
                            break;
                        }
                    }
                }
            }
            par[node] = pn;
            if (pn < 0) s_bad = 2;
            else if (!TSD_IN(pn, node, kChkBuild)) s_bad = 2;  // a parent precedes its child
        }
        __syncthreads();
        if (tid == 0) {
            par[0] = -1;
            tok[0] = -1;
            dep[0] = 0;
            sc[0] = 0.0f;
            if (ws.score64) ws.score64[(int64_t)t * stride] = 0.0;
            if (rk) rk[0] = -1;
            if (md) md[0] = -1;
        }
    }
    for (int i = (failed ? 0 : nn) + tid; i <= B; i += blockDim.x) {
        par[i] = -1;
        tok[i] = -1;
        dep[i] = -1;
        sc[i] = -INFINITY;
        if (ws.score64) ws.score64[(int64_t)t * stride + i] = -INFINITY;
        if (rk) rk[i] = -1;
        if (md) md[i] = -1;
    }
    if (tid == 0) {
        n_nodes_out[t] = nn;
        status[t] = failed ? kStatNonFinite : kStatOk;
    }
}

cudaError_t launch_build_heap(const BuildWs& ws, int n_trees, int n_modes, int L, int topk, int B,
                              int32_t* parent, int32_t* token, int32_t* depth, float* score,
                              int32_t* rank, int32_t* mode, int32_t* n_nodes, int32_t* status,
                              cudaStream_t stream) {
    const BuildPlan p = build_plan(n_modes, L, topk, B);
    cudaError_t e = cudaFuncSetAttribute(build_tree_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)p.smem_total);
    if (e != cudaSuccess) return e;
    int bits = 0;
    while ((1 << bits) < topk) ++bits;
    if (cudaError_t e_ = launch_pdl(build_tree_kernel, n_trees, kBuildThreads, p.smem_total, stream, 
        ws, p, n_modes, L, topk, B, bits, parent, token, depth, score, rank, mode, n_nodes, status); e_ != cudaSuccess) return e_;
    return cudaGetLastError();
}

TSD_CHECK_READER(checks_heap)

}  // namespace tsd
