// chunk_reduce.cuh -- per-chunk pieces of the node-row reduction of Tree
// Exit Verification ("Where Draft Trees Lose Target Mass: Exit-Guided
// Speculative Decoding", Sec. 3 Eq. 1, Sec. 3.1 Eq. 4, Eq. 7): one warp
// reduces one 8 KB chunk of a logits row held in registers (maximum, sums of
// exp2(z*c - mc) with and without the row's drafted children, or the arg-max
// at T = 0), and the walk of warp work items over (tree, node, chunk).
// Shared by the batched row kernel and the fused small-batch verifier.
#pragma once

#include "tsd_internal.cuh"

namespace tsd {

// First index in sorted a[lo, hi) with a[i] >= x.
__device__ __forceinline__ int lower_bound_i32(const int32_t* a, int lo, int hi, int64_t x) {
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)a[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// One lane's part of a chunk's statistics (see chunk_lane below).
struct LanePart {
    float m;   // chunk maximum (warp-reduced)
    float s;   // this lane's sum of exp2(z*c - mc)
    float r;   // the same without drafted children
    int amax;  // T = 0: this lane's first index holding m (INT_MAX: none)
    bool bad;  // T = 0: a NaN or +inf in this lane's slice
    bool kids; // T > 0: r differs from s (children fall in the chunk)
};

// Words of the per-lane child mask: one bit per element a lane holds in a
// chunk (kVecPerLane vectors of VEC elements).
template <typename T>
struct ExclMask {
    static constexpr int kWords = (kVecPerLane * Lanes<T>::kVec + 31) / 32;
    uint32_t w[kWords];
};

// Marks chunk offset o (0 <= o < the chunk's length) in the mask of the lane
// that holds it: vector o / VEC sits in lane (o / VEC) % 32 as that lane's
// vector (o / VEC) / 32.  Returns true if the bit was already set (the same
// token marked twice).
template <typename T>
__device__ __forceinline__ bool excl_mark(ExclMask<T>& m, int o, int lane) {
    constexpr int VEC = Lanes<T>::kVec;
    bool again = false;
    if (((o / VEC) & (kWarp - 1)) == lane) {
        const int bit = (o / (VEC * kWarp)) * VEC + (o % VEC);
        const uint32_t sel = 1u << (bit & 31);
#pragma unroll
        for (int w = 0; w < ExclMask<T>::kWords; ++w)
            if (w == (bit >> 5)) {
                again = (m.w[w] & sel) != 0;
                m.w[w] |= sel;
            }
    }
    return again;
}

// T = 0 part of a chunk: the warp-wide maximum and this lane's first index
// holding it.  Argmax with the smallest id among equal maxima: the maximum
// first (packed per-vector maxima), then the first element equal to it in
// index order.  Vector i*32 + lane sits in lane `lane`, so a lane's first hit
// is at its smallest i.  A NaN or +inf anywhere marks the chunk.
template <typename T>
__device__ __forceinline__ LanePart lane_argmax_part(const uint4 (&buf)[kVecPerLane], int cn,
                                                     int64_t c0, int lane) {
    constexpr int VEC = Lanes<T>::kVec;
    LanePart lp;
    lp.s = 0.0f;
    lp.r = 0.0f;
    lp.amax = INT_MAX;
    lp.bad = false;
    lp.kids = false;
    float vm[kVecPerLane];
    float lm = -INFINITY;
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
        vm[i] = Lanes<T>::vmax_nan(buf[i]);
        lp.bad |= is_bad_logit(vm[i]);
        lm = fmaxf(lm, vm[i]);
    }
    const float m = warp_max(lm);
    int hit = -1;
    uint4 hv = buf[0];
#pragma unroll
    for (int i = kVecPerLane - 1; i >= 0; --i)
        if (vm[i] == m && (i * kWarp + lane) * VEC < cn) {
            hit = i;
            hv = buf[i];
        }
    if (hit >= 0) {
        int j0 = VEC - 1;
#pragma unroll
        for (int j = VEC - 1; j >= 0; --j)
            if (Lanes<T>::get(hv, j) == m) j0 = j;
        lp.amax = (int)c0 + (hit * kWarp + lane) * VEC + j0;
    }
    lp.m = m;
    return lp;
}

// T > 0 sums of a chunk whose maximum m is finite and whose drafted
// children are marked in `excl`: this lane's sum of exp2(z*c - mc) and the
// same without the marked elements, mc = fl(m*c).  Packed fp32x2 fma/add
// (each lane rounds like fmaf / +); accumulator pair p holds element slots
// 2p and 2p+1 of every vector.
template <typename T>
__device__ __forceinline__ void lane_sums_excl(const uint4 (&buf)[kVecPerLane], float c, float mc,
                                               const ExclMask<T>& excl, LanePart& lp) {
    constexpr int VEC = Lanes<T>::kVec;
    constexpr int NP = VEC / 2;
    const float2 cc = make_float2(c, c), nmc = make_float2(-mc, -mc);
    float2 acc[NP], racc[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        acc[p] = make_float2(0.0f, 0.0f);
        racc[p] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i)
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const float2 y = __ffma2_rn(Lanes<T>::pair(buf[i], p), cc, nmc);
            const float2 e = make_float2(ex2(y.x), ex2(y.y));
            const int b0 = i * VEC + 2 * p, b1 = b0 + 1;
            acc[p] = __fadd2_rn(acc[p], e);
            racc[p] = __fadd2_rn(racc[p],
                                 make_float2(((excl.w[b0 >> 5] >> (b0 & 31)) & 1u) ? 0.0f : e.x,
                                             ((excl.w[b1 >> 5] >> (b1 & 31)) & 1u) ? 0.0f : e.y));
        }
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        lp.s += acc[p].x;
        lp.s += acc[p].y;
        lp.r += racc[p].x;
        lp.r += racc[p].y;
    }
}

// The same sums for a chunk without drafted children (the residual is the
// full sum).
template <typename T>
__device__ __forceinline__ void lane_sums_nokids(const uint4 (&buf)[kVecPerLane], float c,
                                                 float mc, LanePart& lp) {
    constexpr int VEC = Lanes<T>::kVec;
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
        lp.s += acc[p].x;
        lp.s += acc[p].y;
    }
    lp.r = lp.s;
}

// Statistics of one row chunk held in registers, in two parts so that a
// caller can start the next chunk's loads between them.  chunk_lane() uses
// the buffer: lane l holds vectors l, l+32, ... of the chunk (16 bytes each;
// vectors at or past cn elements hold -inf; cn is a multiple of the vector
// width).  It reduces the chunk maximum across the warp (the exponentials
// need it) but leaves the sums, or the arg-max candidates, per lane.  The
// drafted children of the row that fall in the chunk are ctok[clo, chi)
// (tokens).  chunk_finish() does the remaining warp reductions.
template <typename T, bool GREEDY>
__device__ __forceinline__ LanePart chunk_lane(const uint4 (&buf)[kVecPerLane], int cn, float c,
                                               const int32_t* __restrict__ ctok, int clo, int chi,
                                               int64_t c0, int lane) {
    if (GREEDY) return lane_argmax_part<T>(buf, cn, c0, lane);
    LanePart lp;
    lp.s = 0.0f;
    lp.r = 0.0f;
    lp.amax = INT_MAX;
    lp.bad = false;
    lp.kids = false;
    const float m = warp_max(Lanes<T>::block_max(buf));
    lp.m = m;
    if (m == -INFINITY) return lp;  // every token of the chunk is masked
    const float mc = __fmul_rn(m, c);
    if (chi == clo) {  // no drafted child in this chunk: the residual is the full sum
        lane_sums_nokids<T>(buf, c, mc, lp);
        return lp;
    }
    // Some children fall in this chunk: mark them in a per-lane bitmask over
    // the lane's kVecPerLane * VEC elements, then sum with and without them.
    lp.kids = true;
    ExclMask<T> excl;
#pragma unroll
    for (int w = 0; w < ExclMask<T>::kWords; ++w) excl.w[w] = 0u;
    for (int q = clo; q < chi; ++q) excl_mark<T>(excl, (int)((int64_t)ctok[q] - c0), lane);
    lane_sums_excl<T>(buf, c, mc, excl, lp);
    return lp;
}

// chunk_lane() for a caller that has already marked the children falling in
// the chunk (`kids` true if any lane marked one).
template <typename T, bool GREEDY>
__device__ __forceinline__ LanePart chunk_lane_marked(const uint4 (&buf)[kVecPerLane], int cn,
                                                      float c, const ExclMask<T>& excl, bool kids,
                                                      int64_t c0, int lane) {
    if (GREEDY) return lane_argmax_part<T>(buf, cn, c0, lane);
    LanePart lp;
    lp.s = 0.0f;
    lp.r = 0.0f;
    lp.amax = INT_MAX;
    lp.bad = false;
    lp.kids = false;
    const float m = warp_max(Lanes<T>::block_max(buf));
    lp.m = m;
    if (m == -INFINITY) return lp;
    const float mc = __fmul_rn(m, c);
    if (!kids) {
        lane_sums_nokids<T>(buf, c, mc, lp);
        return lp;
    }
    lp.kids = true;
    lane_sums_excl<T>(buf, c, mc, excl, lp);
    return lp;
}

template <bool GREEDY>
__device__ __forceinline__ ChunkStat chunk_finish(const LanePart& lp) {
    ChunkStat st;
    st.m = lp.m;
    if (GREEDY) {
        st.amax = __reduce_min_sync(0xffffffffu, lp.amax);
        st.s = __any_sync(0xffffffffu, lp.bad) ? __int_as_float(0x7fc00000) : 0.0f;
        st.r = 0.0f;
        return st;
    }
    st.amax = -1;
    st.s = warp_sum(lp.s);
    st.r = __any_sync(0xffffffffu, lp.kids) ? warp_sum(lp.r) : st.s;
    return st;
}

template <typename T>
__device__ __forceinline__ void load_chunk(uint4 (&buf)[kVecPerLane], const T* __restrict__ rp,
                                           int cn, int lane) {
    constexpr int VEC = Lanes<T>::kVec;
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
        const int e = (i * kWarp + lane) * VEC;
        buf[i] = (e < cn) ? ld_stream16(rp + e) : Lanes<T>::neg_inf();
    }
}

// Generic path for unaligned rows or ragged V: element loads, two passes.
template <typename T, bool GREEDY>
__device__ __noinline__ ChunkStat reduce_chunk_scalar(const T* __restrict__ rp, int cn, float c,
                                                      const int32_t* __restrict__ ctok, int clo,
                                                      int chi, int64_t c0, int lane) {
    ChunkStat st;
    float bm = -INFINITY;
    int bi = INT_MAX;
    bool bad = false;
    for (int e = lane; e < cn; e += kWarp) {
        const float x = load_logit(rp + e);
        bad |= is_bad_logit(x);
        if (better(x, (int)c0 + e, bm, bi)) {
            bm = x;
            bi = (int)c0 + e;
        }
    }
    warp_argmax(bm, bi);
    st.m = bm;
    if (GREEDY) {
        st.s = __any_sync(0xffffffffu, bad) ? __int_as_float(0x7fc00000) : 0.0f;
        st.r = 0.0f;
        st.amax = bi;
        return st;
    }
    st.amax = -1;
    if (bm == -INFINITY) {
        st.s = __any_sync(0xffffffffu, bad) ? __int_as_float(0x7fc00000) : 0.0f;
        st.r = 0.0f;
        return st;
    }
    const float mc = __fmul_rn(bm, c);
    float s = 0.0f, r = 0.0f;
    for (int e = lane; e < cn; e += kWarp) {
        const float x = load_logit(rp + e);
        const float v = ex2(fmaf(x, c, -mc));
        bool child = false;
        for (int q = clo; q < chi; ++q) child |= ((int64_t)ctok[q] == c0 + e);
        s += v;
        r += child ? 0.0f : v;
    }
    st.s = warp_sum(s);
    st.r = warp_sum(r);
    if (__any_sync(0xffffffffu, bad)) st.s = __int_as_float(0x7fc00000);
    return st;
}

// Position of a warp's work item, item = (t * (B+1) + v) * nch + ch, walked
// by a fixed stride with carries instead of divisions.
struct ItemPos {
    int64_t item;
    int t, v, ch;
};
struct ItemStep {
    int64_t stride;
    int dt, dv, dch;
};
__device__ __forceinline__ ItemPos item_pos(int64_t item, int R, int nch) {
    const int64_t row = item / nch;
    ItemPos p;
    p.item = item;
    p.ch = (int)(item - row * nch);
    p.t = (int)(row / R);
    p.v = (int)(row - (int64_t)p.t * R);
    return p;
}
__device__ __forceinline__ void item_advance(ItemPos& p, const ItemStep& s, int R, int nch) {
    p.item += s.stride;
    p.ch += s.dch;
    const int carry = p.ch >= nch;
    p.ch -= carry ? nch : 0;
    p.v += s.dv + carry;
    const int wrap = p.v >= R;
    p.v -= wrap ? R : 0;
    p.t += s.dt + wrap;
}

}  // namespace tsd
