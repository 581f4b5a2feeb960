// tsd_internal.cuh -- device helpers and launch declarations shared by the
// kernels of the GB300 bounded-tree speculative decoding library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tsd.h"

namespace tsd {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// Bounds checks of a checked build (-DTSD_CHECKS).  Every index a kernel
// takes from memory (a parent, a child list offset, a token used as a
// column, a node id, a chunk or list position) passes TSD_IN(i, n, site)
// before its access: in a checked build a failing check sets bit `site` of
// this translation unit's check word and the access is skipped (no trap);
// in the default build the macro is the constant true and costs nothing.
// tsd_debug_check_failures() ORs and clears the words of every unit.
// ---------------------------------------------------------------------------
enum CheckSite : unsigned {
    kChkRowsItem = 0,   // rows_kernel: (tree, node, chunk) of a work item
    kChkChildList,      // a node's CSR child range and its child ids / tokens
    kChkPrep,           // verify_prep_kernel: sort keys, parents, node ids
    kChkAncestor,       // a parent read during an ancestor walk
    kChkExitNode,       // a drawn exit node, chunk or bonus token
    kChkWalk,           // the walk verifiers' staged tree, uniforms, children
    kChkPredraw,        // predraw-and-follow: draws and the followed child
    kChkBuild,          // the builder: list, frontier, successor, node positions
    kChkMask,           // tree_mask_kernel: ancestor bits
    kChkDrafter,        // drafter kernels: chunk, slice and candidate positions
    kChkLse,            // log-sum-exp lists and selection: places, reps, nodes
    kChkForest,         // shared-budget selection: ranks and kept nodes
    kChkExit,           // exit loss: rows and gathered tokens
};
#ifdef TSD_CHECKS
static __device__ unsigned int g_tsd_check_word;  // one per translation unit
__device__ __forceinline__ bool tsd_in_range(long long i, long long n, unsigned site) {
    if (i >= 0 && i < n) return true;
    atomicOr(&g_tsd_check_word, 1u << site);
    return false;
}
#define TSD_IN(i, n, site) ::tsd::tsd_in_range((long long)(i), (long long)(n), (site))
// The host reader of this unit's word: returns it and clears it.
#define TSD_CHECK_READER(name)                                                   \
    unsigned name() {                                                            \
        unsigned v = 0, z = 0;                                                   \
        cudaMemcpyFromSymbol(&v, g_tsd_check_word, sizeof(v));                   \
        cudaMemcpyToSymbol(g_tsd_check_word, &z, sizeof(z));                     \
        return v;                                                                \
    }
#else
#define TSD_IN(i, n, site) true
#define TSD_CHECK_READER(name) \
    unsigned name() { return 0u; }
#endif
unsigned checks_rows();
unsigned checks_tree();
unsigned checks_heap();
unsigned checks_mask();
unsigned checks_drafter();
unsigned checks_lse();
unsigned checks_forest();
unsigned checks_exit();
unsigned checks_fused();

// A logits row is processed in chunks of 8 KB (4096 bf16 or 2048 fp32
// tokens); one warp reduces one chunk with sixteen 16-byte loads per lane.
constexpr int kChunkBytes = 8192;
constexpr int kVecPerLane = kChunkBytes / (16 * kWarp);  // 16

__host__ __device__ constexpr int chunk_elems(int esize) { return kChunkBytes / esize; }
// The drafter's row kernel marks picked chunks in one 64-bit mask per lane, so
// a drafter row may span at most 2048 chunks (V <= 8388608 bf16 / 4194304 fp32).
constexpr int kMaxDrafterChunks = 2048;
__host__ __device__ inline int64_t n_chunks(int64_t V, int esize) {
    return (V + chunk_elems(esize) - 1) / chunk_elems(esize);
}

// Per-(row, chunk) reduction of a logits row.
//   m    the chunk's largest raw logit (-inf if every token is -inf)
//   s    sum over the chunk of exp2(z*c - mc), mc = fl(m*c), c = log2(e)/T
//   r    the same sum over tokens that are not drafted children of the row
//   amax lowest token id holding m (greedy); at T = 0, s is NaN when the
//        chunk holds a NaN or +inf logit and 0 otherwise.
struct ChunkStat {
    float m, s, r;
    int32_t amax;
};

// Per-node combination of its chunks (same reference mc for s and r).
struct NodeStat {
    float mc;      // fl(m*c) of the row maximum (greedy: the maximum itself)
    float s, r;    // row sums relative to mc
    int32_t amax;  // arg-max (lowest id) of the row
};

// ---------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 64x64 -> 128-bit multiplies with a Weyl key schedule.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t philox_x0(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3,
                                              uint64_t k0, uint64_t k1) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
        const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    return c0;
}

// The uniform on the 2^-24 grid for (seed; tree, node, stream).
__device__ __forceinline__ float uniform24(uint64_t seed, uint64_t tree, uint64_t node,
                                           uint64_t stream, uint64_t sub = 0) {
    const uint64_t x0 = philox_x0(tree, node, stream, sub, seed, 0);
    return (float)(x0 >> 40) * (1.0f / 16777216.0f);
}

// ---------------------------------------------------------------------------
// Element access.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float load_logit(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load_logit(const float* p) { return *p; }

// 16-byte streaming load (read once; do not keep in L1).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialization (launch_pdl below): it may be
// scheduled while the previous kernel in the stream is still finishing.  Its
// first statement is pdl_entry(), which waits until the previous kernel has
// completed and its memory is visible, and then lets the next kernel be
// scheduled.  No global memory is touched before that wait, so the stream's
// ordering is unchanged; only launch latency is hidden, one kernel ahead.
// (One exception, argued where it is: the exit loss's per-tree kernel reads
// its inputs before the wait, because its predecessor is always the chunk
// pass, which lets it be scheduled only after that pass's own wait.)
// (Letting the next kernel be scheduled before the wait instead hides a
// little more latency for a pair of kernels timed alone, but in a chain such
// as build, mask and verify, grids launched two or three kernels ahead sat on
// the SMs and slowed the whole step by about a tenth: measured 0.525 against
// 0.476 ms for the 32-tree B = 256 step.)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_entry() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The variant that lets the next kernel be scheduled first: for a kernel
// whose dependent is a handful of blocks that should already be resident
// when it completes (the per-tree finish of the small-launch verifier).
__device__ __forceinline__ void pdl_entry_early() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// MUFU base-2 exponential (ex2.approx.ftz: about 2 ulp).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Per-type access to one 16-byte vector of logits (8 bf16 or 4 fp32).
template <typename T>
struct Lanes;
template <>
struct Lanes<__nv_bfloat16> {
    static constexpr int kVec = 8;  // elements per 16-byte load
    static __device__ __forceinline__ float get(const uint4& q, int j) {
        const uint32_t w = (j >> 1) == 0 ? q.x : (j >> 1) == 1 ? q.y : (j >> 1) == 2 ? q.z : q.w;
        return (j & 1) ? bf16_hi(w) : bf16_lo(w);
    }
    static __device__ __forceinline__ uint4 neg_inf() {
        return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    }
    // Elements 2p and 2p+1 of a vector, widened to fp32.
    static __device__ __forceinline__ float2 pair(const uint4& q, int p) {
        const uint32_t w = p == 0 ? q.x : p == 1 ? q.y : p == 2 ? q.z : q.w;
        return make_float2(bf16_lo(w), bf16_hi(w));
    }
    static __device__ __forceinline__ float vmax(const uint4& q) {
        __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&q.x),
                                   *reinterpret_cast<const __nv_bfloat162*>(&q.y));
        a = __hmax2(a, __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&q.z),
                               *reinterpret_cast<const __nv_bfloat162*>(&q.w)));
        return fmaxf(__low2float(a), __high2float(a));
    }
    // Maximum over a lane's whole chunk slice: packed bf16 maxima in four
    // independent chains, widened once at the end.
    static __device__ __forceinline__ float block_max(const uint4 (&b)[kVecPerLane]) {
        __nv_bfloat162 a0 = *reinterpret_cast<const __nv_bfloat162*>(&b[0].x);
        __nv_bfloat162 a1 = *reinterpret_cast<const __nv_bfloat162*>(&b[0].y);
        __nv_bfloat162 a2 = *reinterpret_cast<const __nv_bfloat162*>(&b[0].z);
        __nv_bfloat162 a3 = *reinterpret_cast<const __nv_bfloat162*>(&b[0].w);
#pragma unroll
        for (int i = 1; i < kVecPerLane; ++i) {
            a0 = __hmax2(a0, *reinterpret_cast<const __nv_bfloat162*>(&b[i].x));
            a1 = __hmax2(a1, *reinterpret_cast<const __nv_bfloat162*>(&b[i].y));
            a2 = __hmax2(a2, *reinterpret_cast<const __nv_bfloat162*>(&b[i].z));
            a3 = __hmax2(a3, *reinterpret_cast<const __nv_bfloat162*>(&b[i].w));
        }
        a0 = __hmax2(__hmax2(a0, a1), __hmax2(a2, a3));
        return fmaxf(__low2float(a0), __high2float(a0));
    }
    // Maximum that is NaN when any element is NaN.
    static __device__ __forceinline__ float vmax_nan(const uint4& q) {
        __nv_bfloat162 a = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&q.x),
                                       *reinterpret_cast<const __nv_bfloat162*>(&q.y));
        a = __hmax2_nan(a, *reinterpret_cast<const __nv_bfloat162*>(&q.z));
        a = __hmax2_nan(a, *reinterpret_cast<const __nv_bfloat162*>(&q.w));
        return __bfloat162float(__hmax_nan(__low2bfloat16(a), __high2bfloat16(a)));
    }
};
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
template <>
struct Lanes<float> {
    static constexpr int kVec = 4;
    static __device__ __forceinline__ float get(const uint4& q, int j) {
        return __uint_as_float(j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w);
    }
    static __device__ __forceinline__ uint4 neg_inf() {
        return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
    }
    static __device__ __forceinline__ float2 pair(const uint4& q, int p) {
        return p == 0 ? make_float2(__uint_as_float(q.x), __uint_as_float(q.y))
                      : make_float2(__uint_as_float(q.z), __uint_as_float(q.w));
    }
    static __device__ __forceinline__ float vmax(const uint4& q) {
        return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                     fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
    }
    static __device__ __forceinline__ float block_max(const uint4 (&b)[kVecPerLane]) {
        float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) {
            a0 = fmaxf(a0, __uint_as_float(b[i].x));
            a1 = fmaxf(a1, __uint_as_float(b[i].y));
            a2 = fmaxf(a2, __uint_as_float(b[i].z));
            a3 = fmaxf(a3, __uint_as_float(b[i].w));
        }
        return fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
    }
    static __device__ __forceinline__ float vmax_nan(const uint4& q) {
        return fmax_nan(fmax_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                        fmax_nan(__uint_as_float(q.z), __uint_as_float(q.w)));
    }
};

// Order-preserving 64-bit image of a float64 score (larger score, larger
// key; -inf the smallest of the finite-or-infinite values), and its inverse.
// Division of 32-bit unsigned integers by a divisor fixed at run time, as a
// multiply-high and two shifts (Granlund and Montgomery, "Division by
// Invariant Integers using Multiplication", 1994, Sec. 4): with l = ceil(log2
// d) and m = floor(2^32 (2^l - d) / d) + 1, t = mulhi(m, x) gives
// x / d = (t + ((x - t) >> min(l, 1))) >> max(l - 1, 0) for every 32-bit x.
struct FastDiv {
    unsigned d = 1, m = 1, s1 = 0, s2 = 0;
    FastDiv() = default;
    __host__ __device__ explicit FastDiv(unsigned div) : d(div) {
        unsigned l = 0;
        while (l < 32 && (1ull << l) < div) ++l;
        m = (unsigned)(((((1ull << l) - div) << 32) / div) + 1);
        s1 = l < 1 ? l : 1;
        s2 = l > 1 ? l - 1 : 0;
    }
    __device__ __forceinline__ unsigned div(unsigned x) const {
        const unsigned t = __umulhi(m, x);
        return (t + ((x - t) >> s1)) >> s2;
    }
};

// Hash of a token sequence, one token at a time from the root's value: a
// strong 64-bit mix of (parent hash, token), a SplitMix64-style finaliser.
// Equal sequences get equal hashes; users confirm every match exactly.
constexpr unsigned long long kRootHash = 0x243F6A8885A308D3ull;
__device__ __forceinline__ unsigned long long hash_step(unsigned long long h, int tok) {
    unsigned long long x = h ^ ((unsigned long long)(uint32_t)tok * 0x9E3779B97F4A7C15ull);
    x ^= x >> 30;
    x *= 0xBF58476D1CE4E5B9ull;
    x ^= x >> 27;
    x *= 0x94D049BB133111EBull;
    x ^= x >> 31;
    return x;
}
__device__ __forceinline__ unsigned long long order_key(double s) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(s);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double key_score(unsigned long long k) {
    const unsigned long long u = (k >> 63) ? (k & 0x7fffffffffffffffull) : ~k;
    return __longlong_as_double((long long)u);
}

// (value desc, id asc) order on (logit, token) pairs.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
// Arg-max with ties to the lower id; every lane gets the result.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}
// Inclusive prefix sum across the warp.
__device__ __forceinline__ float warp_incl_scan(float x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

__device__ __forceinline__ bool is_bad_logit(float x) { return x != x || x == __int_as_float(0x7f800000); }

// ---------------------------------------------------------------------------
// Workspace layout of the verifiers (TEV and predraw), per call.
// ---------------------------------------------------------------------------
struct VerifyWs {
    int32_t* child_ptr;   // [n_trees][B+2] CSR offsets of each node's children
    int32_t* child_tok;   // [n_trees][B+1] children's tokens, sorted per node
    int32_t* child_node;  // [n_trees][B+1] the matching child node ids
    int32_t* depth;       // [n_trees][B+1]
    int32_t* tstat;       // [n_trees] internal per-tree status
    NodeStat* node;       // [n_trees][B+1]
    float* pedge;         // [n_trees][B+1] p_pa(u)(x_u)
    float* rho;           // [n_trees][B+1]
    int32_t* draws;       // [n_trees][B+1] predraw R_v
    ChunkStat* chunk;     // [n_trees][B+1][n_chunks]
};
size_t verify_ws_layout(int n_trees, int B, int64_t V, int esize, void* base, VerifyWs* out);

struct BuildWs {
    ChunkStat* chunk;    // [rows][n_chunks] (m, s)
    float* lane_max;     // [rows][n_chunks][32] maximum of each lane's slice of a chunk
    int32_t* top_id;     // [rows][topk]
    double* top_zt;      // [rows][topk] the kept tokens' z / T_d
    double* lse;         // [rows] log sum exp(z / T_d) over the row
    uint8_t* heap;       // [n_trees][heap bytes] spill space when shared memory is short
    size_t heap_stride;  // bytes per tree
    double* score64;     // nullable [n_trees][B+1]: each node's score in float64 (-inf past n_nodes)
};
size_t build_ws_layout(int n_trees, int n_modes, int L, int64_t V, int topk, int B, int esize,
                       void* base, BuildWs* out);

// ---------------------------------------------------------------------------
// Kernel launchers (one per .cu file).  All return cudaGetLastError().
// ---------------------------------------------------------------------------
cudaError_t launch_verify_prep(const int32_t* parent, const int32_t* token, const int32_t* n_nodes,
                               int n_trees, int B, int64_t V, const VerifyWs& ws,
                               cudaStream_t stream);
cudaError_t launch_rows(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                        float c, bool greedy, const int32_t* n_nodes, const VerifyWs& ws,
                        cudaStream_t stream);
cudaError_t launch_node_combine(const void* logits, tsd_dtype dtype, int n_trees, int B,
                                int64_t V, float c, bool greedy, const int32_t* n_nodes,
                                const VerifyWs& ws, cudaStream_t stream);
cudaError_t launch_tev_tree(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                            float c, bool greedy, uint64_t seed, const int32_t* parent,
                            const int32_t* n_nodes, const VerifyWs& ws, int32_t* exit_node,
                            int32_t* bonus, int32_t* accept_len, float* exit_mass,
                            float* prefix_prob, float* coverage, int32_t* status,
                            cudaStream_t stream);
// The two-kernel verifier of small launches (k_tev_fused.cu): a streaming
// row kernel that finds each row's children itself, then one block per tree.
// Usable when the logits rows are 16-byte aligned with V a multiple of the
// vector width, B <= kFusedMaxB (above it the batched chain is faster,
// measured) and a row has at most 128 chunks.  The event
// ev_between, if given, is recorded between its two kernels.
constexpr int kFusedMaxB = 128;
bool tev_fused_fits(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V);
cudaError_t launch_tev_fused(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                             float c, bool greedy, uint64_t seed, const int32_t* parent,
                             const int32_t* token, const int32_t* n_nodes, const VerifyWs& ws,
                             int32_t* exit_node, int32_t* bonus, int32_t* accept_len,
                             float* exit_mass, float* prefix_prob, float* coverage,
                             int32_t* status, cudaStream_t stream, cudaEvent_t ev_between);
cudaError_t launch_predraw_fused(const void* logits, tsd_dtype dtype, int n_trees, int B,
                                 int64_t V, float c, bool greedy, uint64_t seed,
                                 const int32_t* parent, const int32_t* token,
                                 const int32_t* n_nodes, const VerifyWs& ws, int32_t* exit_node,
                                 int32_t* bonus, int32_t* accept_len, int32_t* draws,
                                 int32_t* status, cudaStream_t stream);
cudaError_t launch_predraw(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                           float c, bool greedy, uint64_t seed, const int32_t* n_nodes,
                           const VerifyWs& ws, int32_t* exit_node, int32_t* bonus,
                           int32_t* accept_len, int32_t* draws, int32_t* status,
                           cudaStream_t stream);
cudaError_t launch_drafter_stats(const void* logits, tsd_dtype dtype, int64_t rows, int64_t V,
                                 int topk, float c, double temp, const BuildWs& ws,
                                 cudaStream_t stream);
cudaError_t launch_seqres_tree(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                               float c, bool greedy, uint64_t seed, const int32_t* n_nodes,
                               const VerifyWs& ws, int32_t* exit_node, int32_t* bonus,
                               int32_t* accept_len, int32_t* status, cudaStream_t stream);
cudaError_t launch_proposal_tree(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V,
                                 float c, bool greedy, uint64_t seed, const float* q_child,
                                 const int32_t* n_nodes, const VerifyWs& ws, int32_t* exit_node,
                                 int32_t* bonus, int32_t* accept_len, int32_t* status,
                                 cudaStream_t stream);
// Shared-budget selection over the trees of a launch (CAST App. B.4): each
// tree's candidates get their rank in the global merge and the batched
// stopping rule is tested there; every tree keeps its candidates ranked below
// the first failure (n_nodes = width + 1) and its slots past that are cleared.
constexpr int kMaxForestCandidates = 8192;
struct ForestWs {
    double* rho;    // [n_trees][B+1] candidate masses, candidate j at j
    double* pre;    // [n_trees][B+1] exclusive prefix sums of rho (entry cnt = total)
    int32_t* rank;  // [n_trees][B+1] place of candidate j in the global merge
    unsigned long long* img;  // [n_trees][B+1] order image of candidate j's score
    int32_t* cnt;   // [n_trees] candidates per tree (0 for a failed tree)
    int32_t* ctl;   // [2] first failing rank, candidate count
};
cudaError_t launch_forest_select(const double* score64, int32_t* depth, int n_trees, int B,
                                 int M_max, double l0, double c1, int32_t* n_nodes,
                                 const int32_t* status, int32_t* total, int32_t* parent,
                                 int32_t* token, float* score, const ForestWs& ws,
                                 cudaStream_t stream);
// Mixture tree under the log-sum-exp score (MFD App. B Eq. 6): per-mode
// per-depth lists, then distinct prefixes ranked by log sum_m pi_m Q_m(v).
// Entries are indexed flat by (depth, mode, place): f = (d K + m) B + i.
constexpr int kMaxLseModeBudget = 4096;  // n_modes * B: one depth's entries in the hash
constexpr int kMaxLseB = 2048;
struct LseWs {
    int32_t* tok;      // [n_trees][L*K*B] last token of each list entry
    int32_t* par;      // [n_trees][L*K*B] its parent's place one depth up (same mode)
    unsigned long long* kimg;  // [n_trees][L*K*B] ~order_key of the ranking key (s_lse clamped
                               // to the parent's key): ascending = better
    int32_t* rep;      // [n_trees][L*K*B] flat index of the first entry holding the same prefix
    int32_t* node_of;  // [n_trees][L*K*B] node index of a kept entry
    unsigned long long* cimg;  // [n_trees][L*K*B] candidates' images, compacted in flat order
    int32_t* cflat;            // [n_trees][L*K*B] their flat indices
    int32_t* nb;       // [n_trees][L][K] list sizes
    unsigned long long* phash;  // [n_trees][L*K*B] hash of each entry's token sequence
};
__host__ __device__ inline int pow2_ceil(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}
size_t lse_beam_smem(int K, int B, int k);
constexpr size_t kMaxLseSmem = 227 * 1024;
size_t lse_select_smem(int K, int B, int L);
cudaError_t launch_lse_tree(const void* logits, tsd_dtype dtype, int n_trees, int K, int L,
                            int64_t V, int k, int B, double temp, const float* log_prior,
                            const BuildWs& bws, const LseWs& ws, int32_t* parent, int32_t* token,
                            int32_t* depth, float* score, int32_t* n_nodes, int32_t* status,
                            int32_t* n_cand, cudaStream_t stream);
// The drafter's streaming pass alone (ws.chunk and ws.lane_max).
cudaError_t launch_drafter_chunks(const void* logits, tsd_dtype dtype, int64_t rows, int64_t V,
                                  float c, const BuildWs& ws, cudaStream_t stream);

// Workspace of the exit-guided loss, per call.
struct ExitWs {
    BuildWs rows;       // chunk statistics and lane maxima of the drafter rows
    double* lse;        // [n_trees][L] row log-normalisers of z / T_d
    double* wrow;       // [n_trees][L] summed weight of the nodes each row scores
    int32_t* tstat;     // [n_trees]
    double* norm;       // [2] N = sum over valid trees of (n_nodes - 1), then 1 / (T_d N) (0 if N = 0)
    unsigned* done;     // [1] completion counter of the per-tree kernel (zero between calls)
};
size_t exit_ws_layout(int n_trees, int L, int64_t V, int B, int esize, void* base, ExitWs* out);
cudaError_t launch_exit_loss(const void* logits, tsd_dtype dtype, int n_trees, int L, int64_t V,
                             float c, double temp, const int32_t* token, const int32_t* depth,
                             const int32_t* n_nodes, int B, const float* omega, double* loss_tree,
                             double* loss, float* grad, int32_t* status, const ExitWs& ws,
                             cudaStream_t stream);
cudaError_t launch_build_heap(const BuildWs& ws, int n_trees, int n_modes, int L, int topk, int B,
                              int32_t* parent, int32_t* token, int32_t* depth, float* score,
                              int32_t* rank, int32_t* mode, int32_t* n_nodes, int32_t* status,
                              cudaStream_t stream);
cudaError_t launch_tree_mask(const int32_t* parent, const int32_t* n_nodes, int n_trees, int B,
                             int prefix_len, uint32_t* anc_bits, int32_t* position_ids,
                             float* additive_mask, int64_t mask_ld, int32_t* status,
                             cudaStream_t stream);

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
// The same, with the grid's blocks in thread-block clusters of `cluster`
// along x (co-scheduled, with distributed shared memory and cluster barriers).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, unsigned cluster, unsigned block,
                               size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Grid for a persistent (grid-stride) kernel: min(want, SMs x the CTAs of
// `kernel` resident per SM at this block size and dynamic shared memory), at
// least 1.  Residency comes from the occupancy calculator, cached per device
// and kernel.
int resident_grid(const void* kernel, int threads, size_t smem, int64_t want);

// Internal per-tree status values (tstat) match tsd_status codes.
constexpr int32_t kStatOk = TSD_OK;
constexpr int32_t kStatBadTree = TSD_ERR_BAD_TREE;
constexpr int32_t kStatNonFinite = TSD_ERR_NONFINITE;

}  // namespace tsd
