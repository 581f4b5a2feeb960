// tsd_api.cu -- the C entry points declared in include/tsd.h: argument
// checks on the host, workspace layout, and the kernel launches.  Nothing here
// allocates or synchronises.
#include <math.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "tsd_internal.cuh"

namespace tsd {

int resident_grid(const void* kernel, int threads, size_t smem, int64_t want) {
    static std::mutex mu;
    // (device, kernel, block size, dynamic shared memory) -> (SMs, CTAs per SM)
    static std::map<std::tuple<int, const void*, int, size_t>, std::pair<int, int>> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::pair<int, int> r;
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto key = std::make_tuple(dev, kernel, threads, smem);
        auto it = cache.find(key);
        if (it == cache.end()) {
            int sms = 0, per = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                sms < 1)
                sms = 1;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, threads, smem) !=
                    cudaSuccess ||
                per < 1)
                per = 1;
            it = cache.emplace(key, std::make_pair(sms, per)).first;
        }
        r = it->second;
    }
    const int64_t cap = (int64_t)r.first * r.second;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

size_t heap_spill_bytes(int n_modes, int L, int topk, int B);  // k_heap.cu

// Which launches of Tree Exit Verification (and of predraw-and-follow) run the
// two-kernel path (k_tev_fused.cu), given its layout conditions (B <= 128 among them): every
// launch with B <= TSD_FUSED_ANY_SIZE_MAX_B (64), and launches of at most
// TSD_FUSED_MAX_ITEMS (node row, 8 KB chunk) items above that.  Measured on the V = 151936 grid: at B <= 64
// the two-kernel path was as fast or faster from 1 to 256 trees; at B = 128
// it was faster for one tree and 5-14% slower from 16 trees up (each tree's
// finish block then has more rows to combine than the batched combine
// kernel spreads over the GPU).  A build may set both bounds to compare paths.
#ifndef TSD_FUSED_MAX_ITEMS
#define TSD_FUSED_MAX_ITEMS 32768
#endif
#ifndef TSD_FUSED_ANY_SIZE_MAX_B
#define TSD_FUSED_ANY_SIZE_MAX_B 64
#endif
bool use_two_kernel_path(const void* logits, tsd_dtype dtype, int n_trees, int B, int64_t V) {
    const int es = dtype == TSD_BF16 ? 2 : 4;
    return tev_fused_fits(logits, dtype, n_trees, B, V) &&
           (B <= TSD_FUSED_ANY_SIZE_MAX_B ||
            (int64_t)n_trees * (B + 1) * n_chunks(V, es) <= TSD_FUSED_MAX_ITEMS);
}

namespace {

constexpr size_t kAlign = 256;

struct Carve {
    uint8_t* base;
    size_t off = 0;
    template <typename T>
    T* take(size_t count) {
        off = (off + kAlign - 1) & ~(kAlign - 1);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += sizeof(T) * count;
        return p;
    }
};

int dtype_size(tsd_dtype d) { return d == TSD_BF16 ? 2 : (d == TSD_F32 ? 4 : 0); }

bool temp_ok(float T) { return isfinite(T) && (T == 0.0f || T >= 1e-6f); }

// c = log2(e) / T rounded once to float; the kernels evaluate
// exp(z/T - m/T) as exp2(fma(z, c, -fl(m*c))).
float exp2_scale(double T) { return (float)(1.4426950408889634 / T); }

bool verify_args_ok(const void* logits, tsd_dtype dtype, const int32_t* parent,
                    const int32_t* token, const int32_t* n_nodes, int n_trees, int B, int64_t V,
                    float temperature, const int32_t* exit_node, const int32_t* bonus,
                    const int32_t* accept_len, const int32_t* status) {
    return logits && parent && token && n_nodes && exit_node && bonus && accept_len && status &&
           dtype_size(dtype) && n_trees >= 1 && B >= 0 && B <= TSD_MAX_B && V >= 1 &&
           V <= 0x7fffffff && temp_ok(temperature);
}

// The address through which the kernels read caller logits: device or
// managed memory as given; page-locked host memory through its mapped device
// address (the kernels then stream it over the host link).  Pageable host
// memory, or a pointer the runtime does not know, is refused.
bool logits_view(const void* p, const void** out) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of this query
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *out = p;
        return true;
    }
    if (a.type == cudaMemoryTypeHost && a.devicePointer) {
        *out = a.devicePointer;
        return true;
    }
    return false;
}

}  // namespace

size_t verify_ws_layout(int n_trees, int B, int64_t V, int esize, void* base, VerifyWs* out) {
    Carve cv{static_cast<uint8_t*>(base)};
    const size_t nt = (size_t)n_trees, nodes = nt * (size_t)(B + 1);
    VerifyWs ws;
    ws.child_ptr = cv.take<int32_t>(nt * (size_t)(B + 2));
    ws.child_tok = cv.take<int32_t>(nodes);
    ws.child_node = cv.take<int32_t>(nodes);
    ws.depth = cv.take<int32_t>(nodes);
    ws.tstat = cv.take<int32_t>(nt);
    ws.node = cv.take<NodeStat>(nodes);
    ws.pedge = cv.take<float>(nodes);
    ws.rho = cv.take<float>(nodes);
    ws.draws = cv.take<int32_t>(nodes);
    ws.chunk = cv.take<ChunkStat>(nodes * (size_t)n_chunks(V, esize));
    if (out) *out = ws;
    return (cv.off + kAlign - 1) & ~(kAlign - 1);
}

size_t exit_ws_layout(int n_trees, int L, int64_t V, int B, int esize, void* base, ExitWs* out) {
    (void)B;
    Carve cv{static_cast<uint8_t*>(base)};
    const size_t rows = (size_t)n_trees * L;
    const size_t nch = (size_t)n_chunks(V, esize);
    ExitWs ws = {};
    ws.rows.chunk = cv.take<ChunkStat>(rows * nch);
    ws.rows.lane_max = cv.take<float>(rows * nch * kWarp);
    ws.lse = cv.take<double>(rows);
    ws.wrow = cv.take<double>(rows);
    ws.tstat = cv.take<int32_t>((size_t)n_trees);
    ws.norm = cv.take<double>(2);
    ws.done = cv.take<unsigned>(1);
    if (out) *out = ws;
    return (cv.off + kAlign - 1) & ~(kAlign - 1);
}

size_t forest_ws_layout(int n_trees, int L, int64_t V, int topk, int B, int esize, void* base,
                        BuildWs* out, ForestWs* fout) {
    const size_t b = build_ws_layout(n_trees, 1, L, V, topk, B, esize, base, out);
    Carve cv{static_cast<uint8_t*>(base), b};
    const size_t slots = (size_t)n_trees * (size_t)(B + 1);
    double* s64 = cv.take<double>(slots);
    if (out) out->score64 = s64;
    ForestWs f;
    f.rho = cv.take<double>(slots);
    f.pre = cv.take<double>(slots);
    f.rank = cv.take<int32_t>(slots);
    f.img = cv.take<unsigned long long>(slots);
    f.cnt = cv.take<int32_t>((size_t)n_trees);
    f.ctl = cv.take<int32_t>(2);
    if (fout) *fout = f;
    return (cv.off + kAlign - 1) & ~(kAlign - 1);
}

size_t lse_ws_layout(int n_trees, int n_modes, int L, int64_t V, int topk, int B, int esize,
                     void* base, BuildWs* out, LseWs* lout) {
    Carve cv{static_cast<uint8_t*>(base)};
    const size_t rows = (size_t)n_trees * n_modes * L;
    const size_t nch = (size_t)n_chunks(V, esize);
    BuildWs ws;
    ws.chunk = cv.take<ChunkStat>(rows * nch);
    ws.lane_max = cv.take<float>(rows * nch * kWarp);
    ws.top_id = cv.take<int32_t>(rows * topk);
    ws.top_zt = cv.take<double>(rows * topk);
    ws.lse = cv.take<double>(rows);
    ws.heap = nullptr;
    ws.heap_stride = 0;
    ws.score64 = nullptr;
    const size_t ent = rows * (size_t)B;  // L * K * B entries per tree
    LseWs l;
    l.tok = cv.take<int32_t>(ent);
    l.par = cv.take<int32_t>(ent);
    l.kimg = cv.take<unsigned long long>(ent);
    l.rep = cv.take<int32_t>(ent);
    l.node_of = cv.take<int32_t>(ent);
    l.cimg = cv.take<unsigned long long>(ent);
    l.cflat = cv.take<int32_t>(ent);
    l.nb = cv.take<int32_t>(rows);
    l.phash = cv.take<unsigned long long>(ent);
    if (out) *out = ws;
    if (lout) *lout = l;
    return (cv.off + kAlign - 1) & ~(kAlign - 1);
}

size_t build_ws_layout(int n_trees, int n_modes, int L, int64_t V, int topk, int B, int esize,
                       void* base, BuildWs* out) {
    Carve cv{static_cast<uint8_t*>(base)};
    const size_t rows = (size_t)n_trees * n_modes * L;
    const size_t nch = (size_t)n_chunks(V, esize);
    BuildWs ws;
    ws.chunk = cv.take<ChunkStat>(rows * nch);
    ws.lane_max = cv.take<float>(rows * nch * kWarp);
    ws.top_id = cv.take<int32_t>(rows * topk);
    ws.top_zt = cv.take<double>(rows * topk);
    ws.lse = cv.take<double>(rows);
    ws.heap_stride = (heap_spill_bytes(n_modes, L, topk, B) + kAlign - 1) & ~(kAlign - 1);
    ws.heap = cv.take<uint8_t>((size_t)n_trees * ws.heap_stride);
    ws.score64 = nullptr;
    if (out) *out = ws;
    return (cv.off + kAlign - 1) & ~(kAlign - 1);
}

}  // namespace tsd

using namespace tsd;

extern "C" {

unsigned tsd_debug_check_failures(void) {
#ifdef TSD_CHECKS
    cudaDeviceSynchronize();
#endif
    return checks_rows() | checks_tree() | checks_heap() | checks_mask() | checks_drafter() |
           checks_lse() | checks_forest() | checks_exit() | checks_fused();
}

const char* tsd_status_string(tsd_status s) {
    switch (s) {
        case TSD_OK: return "ok";
        case TSD_ERR_INVALID_ARG: return "invalid argument";
        case TSD_ERR_CUDA: return "CUDA launch failed";
        case TSD_ERR_WORKSPACE: return "workspace too small or misaligned";
        case TSD_ERR_BAD_TREE: return "malformed tree";
        case TSD_ERR_NONFINITE: return "non-finite logits or a row without mass";
        case TSD_ERR_TIMEOUT: return "timed out";
    }
    return "unknown status";
}

static bool build_sizes_ok(int n_trees, int n_modes, int L, int64_t V, int topk, int B,
                           int esize) {
    if (n_chunks(V, esize) > kMaxDrafterChunks) return false;
    if (n_trees < 1 || n_modes < 1 || n_modes > TSD_MAX_MODES || L < 1 || L > TSD_MAX_L ||
        V < 1 || V > 0x7fffffff || topk < 1 || topk > TSD_MAX_TOPK || topk > V || B < 0 ||
        B > TSD_MAX_B)
        return false;
    int bits = 0;
    while ((1 << bits) < topk) ++bits;
    return (int64_t)L * bits <= 56;
}

static bool lse_sizes_ok(int n_trees, int n_modes, int L, int64_t V, int topk, int B, int esize) {
    return build_sizes_ok(n_trees, n_modes, L, V, topk, B, esize) && n_trees <= 65535 &&
           B <= kMaxLseB && n_modes * B <= kMaxLseModeBudget &&
           lse_beam_smem(n_modes, B, topk) <= kMaxLseSmem;
}

size_t tsd_workspace_size(tsd_op op, int n_trees, int n_modes, int L, int64_t V, int topk, int B,
                          tsd_dtype dtype) {
    const int es = dtype_size(dtype);
    if (!es) return 0;
    switch (op) {
        case TSD_OP_BUILD_TREE:
            if (!build_sizes_ok(n_trees, n_modes, L, V, topk, B, es)) return 0;
            return build_ws_layout(n_trees, n_modes, L, V, topk, B, es, nullptr, nullptr);
        case TSD_OP_VERIFY_TEV:
        case TSD_OP_VERIFY_DDTREE:
            if (n_trees < 1 || B < 0 || B > TSD_MAX_B || V < 1 || V > 0x7fffffff) return 0;
            return verify_ws_layout(n_trees, B, V, es, nullptr, nullptr);
        case TSD_OP_BUILD_FOREST:
            if (n_modes != 1 || !build_sizes_ok(n_trees, 1, L, V, topk, B, es) ||
                (int64_t)n_trees * B > kMaxForestCandidates)
                return 0;
            return forest_ws_layout(n_trees, L, V, topk, B, es, nullptr, nullptr, nullptr);
        case TSD_OP_BUILD_LSE:
            if (!lse_sizes_ok(n_trees, n_modes, L, V, topk, B, es)) return 0;
            return lse_ws_layout(n_trees, n_modes, L, V, topk, B, es, nullptr, nullptr, nullptr);
        case TSD_OP_EXIT_LOSS:
            if (n_trees < 1 || L < 1 || L > TSD_MAX_L || B < 0 || B > TSD_MAX_B || V < 1 ||
                V > 0x7fffffff || n_chunks(V, es) > kMaxDrafterChunks)
                return 0;
            return exit_ws_layout(n_trees, L, V, B, es, nullptr, nullptr);
    }
    return 0;
}

tsd_status tsd_build_tree(const void* drafter_logits, tsd_dtype dtype, int n_trees, int n_modes,
                          int L, int64_t V, int topk, int B, float drafter_temp,
                          int32_t* parent, int32_t* token, int32_t* depth, float* score,
                          int32_t* rank, int32_t* mode, int32_t* n_nodes, int32_t* status,
                          void* workspace, size_t ws_bytes, cudaStream_t stream) {
    if (!drafter_logits || !parent || !token || !depth || !score || !n_nodes || !status ||
        !dtype_size(dtype) || !build_sizes_ok(n_trees, n_modes, L, V, topk, B, dtype_size(dtype)) ||
        !(isfinite(drafter_temp) && drafter_temp >= 1e-6f))
        return TSD_ERR_INVALID_ARG;
    const int es = dtype_size(dtype);
    const size_t need = build_ws_layout(n_trees, n_modes, L, V, topk, B, es, nullptr, nullptr);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return TSD_ERR_WORKSPACE;
    if (!logits_view(drafter_logits, &drafter_logits)) return TSD_ERR_INVALID_ARG;
    BuildWs ws;
    build_ws_layout(n_trees, n_modes, L, V, topk, B, es, workspace, &ws);
    const int64_t rows = (int64_t)n_trees * n_modes * L;
    if (launch_drafter_stats(drafter_logits, dtype, rows, V, topk, exp2_scale(drafter_temp),
                             (double)drafter_temp, ws, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    if (launch_build_heap(ws, n_trees, n_modes, L, topk, B, parent, token, depth, score, rank,
                          mode, n_nodes, status, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

tsd_status tsd_build_lse_tree(const void* drafter_logits, tsd_dtype dtype, int n_trees,
                              int n_modes, int L, int64_t V, int topk, int B, float drafter_temp,
                              const float* log_prior, int32_t* parent, int32_t* token,
                              int32_t* depth, float* score, int32_t* n_nodes, int32_t* status,
                              int32_t* n_cand, void* workspace, size_t ws_bytes,
                              cudaStream_t stream) {
    if (!drafter_logits || !parent || !token || !depth || !score || !n_nodes || !status ||
        !dtype_size(dtype) || !lse_sizes_ok(n_trees, n_modes, L, V, topk, B, dtype_size(dtype)) ||
        !(isfinite(drafter_temp) && drafter_temp >= 1e-6f))
        return TSD_ERR_INVALID_ARG;
    const int es = dtype_size(dtype);
    const size_t need = lse_ws_layout(n_trees, n_modes, L, V, topk, B, es, nullptr, nullptr, nullptr);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return TSD_ERR_WORKSPACE;
    if (!logits_view(drafter_logits, &drafter_logits)) return TSD_ERR_INVALID_ARG;
    if (log_prior) {
        const void* lp = log_prior;
        if (!logits_view(lp, &lp)) return TSD_ERR_INVALID_ARG;
        log_prior = static_cast<const float*>(lp);
    }
    BuildWs ws;
    LseWs lws;
    lse_ws_layout(n_trees, n_modes, L, V, topk, B, es, workspace, &ws, &lws);
    const int64_t rows = (int64_t)n_trees * n_modes * L;
    if (launch_drafter_stats(drafter_logits, dtype, rows, V, topk, exp2_scale(drafter_temp),
                             (double)drafter_temp, ws, stream) != cudaSuccess ||
        launch_lse_tree(drafter_logits, dtype, n_trees, n_modes, L, V, topk, B,
                        (double)drafter_temp, log_prior, ws, lws, parent, token, depth, score,
                        n_nodes, status, n_cand, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

tsd_status tsd_tree_mask(const int32_t* parent, const int32_t* n_nodes, int n_trees, int B,
                         int prefix_len, uint32_t* anc_bits, int32_t* position_ids,
                         float* additive_mask, int64_t mask_ld, int32_t* status,
                         cudaStream_t stream) {
    if (!parent || !n_nodes || !anc_bits || !position_ids || !status || n_trees < 1 || B < 0 ||
        B > TSD_MAX_B || prefix_len < 0 ||
        (additive_mask && mask_ld < (int64_t)prefix_len + B + 1))
        return TSD_ERR_INVALID_ARG;
    if (launch_tree_mask(parent, n_nodes, n_trees, B, prefix_len, anc_bits, position_ids,
                         additive_mask, mask_ld, status, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

static tsd_status verify_tev_impl(const void* target_logits, tsd_dtype dtype,
                                  const int32_t* parent, const int32_t* token,
                                  const int32_t* n_nodes, int n_trees, int B, int64_t V,
                                  float temperature, uint64_t seed, int32_t* exit_node,
                                  int32_t* bonus_token, int32_t* accept_len, float* exit_mass,
                                  float* prefix_prob, float* coverage, int32_t* status,
                                  void* workspace, size_t ws_bytes, cudaStream_t stream,
                                  cudaEvent_t* ev) {
    if (!verify_args_ok(target_logits, dtype, parent, token, n_nodes, n_trees, B, V, temperature,
                        exit_node, bonus_token, accept_len, status))
        return TSD_ERR_INVALID_ARG;
    const int es = dtype_size(dtype);
    const size_t need = verify_ws_layout(n_trees, B, V, es, nullptr, nullptr);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return TSD_ERR_WORKSPACE;
    if (!logits_view(target_logits, &target_logits)) return TSD_ERR_INVALID_ARG;
    VerifyWs ws;
    verify_ws_layout(n_trees, B, V, es, workspace, &ws);
    const bool greedy = temperature == 0.0f;
    const float c = greedy ? 1.0f : exp2_scale(temperature);
    auto mark = [&](int i) { return ev ? cudaEventRecord(ev[i], stream) : cudaSuccess; };
    if (use_two_kernel_path(target_logits, dtype, n_trees, B, V)) {
        // a launch of a few waves of row chunks: the two-kernel path
        if (mark(0) != cudaSuccess || mark(1) != cudaSuccess ||
            launch_tev_fused(target_logits, dtype, n_trees, B, V, c, greedy, seed, parent, token,
                             n_nodes, ws, exit_node, bonus_token, accept_len, exit_mass,
                             prefix_prob, coverage, status, stream,
                             ev ? ev[2] : nullptr) != cudaSuccess ||
            mark(3) != cudaSuccess || mark(4) != cudaSuccess)
            return TSD_ERR_CUDA;
        return TSD_OK;
    }
    if (mark(0) != cudaSuccess ||
        launch_verify_prep(parent, token, n_nodes, n_trees, B, V, ws, stream) != cudaSuccess ||
        mark(1) != cudaSuccess ||
        launch_rows(target_logits, dtype, n_trees, B, V, c, greedy, n_nodes, ws, stream) != cudaSuccess ||
        mark(2) != cudaSuccess ||
        launch_node_combine(target_logits, dtype, n_trees, B, V, c, greedy, n_nodes, ws, stream) != cudaSuccess ||
        mark(3) != cudaSuccess ||
        launch_tev_tree(target_logits, dtype, n_trees, B, V, c, greedy, seed, parent, n_nodes, ws,
                        exit_node, bonus_token, accept_len, exit_mass, prefix_prob, coverage,
                        status, stream) != cudaSuccess ||
        mark(4) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

tsd_status tsd_verify_tev(const void* target_logits, tsd_dtype dtype, const int32_t* parent,
                          const int32_t* token, const int32_t* n_nodes, int n_trees, int B,
                          int64_t V, float temperature, uint64_t seed, int32_t* exit_node,
                          int32_t* bonus_token, int32_t* accept_len, float* exit_mass,
                          float* prefix_prob, float* coverage, int32_t* status, void* workspace,
                          size_t ws_bytes, cudaStream_t stream) {
    return verify_tev_impl(target_logits, dtype, parent, token, n_nodes, n_trees, B, V,
                           temperature, seed, exit_node, bonus_token, accept_len, exit_mass,
                           prefix_prob, coverage, status, workspace, ws_bytes, stream, nullptr);
}

tsd_status tsd_verify_tev_timed(const void* target_logits, tsd_dtype dtype, const int32_t* parent,
                                const int32_t* token, const int32_t* n_nodes, int n_trees, int B,
                                int64_t V, float temperature, uint64_t seed, int32_t* exit_node,
                                int32_t* bonus_token, int32_t* accept_len, float* exit_mass,
                                float* prefix_prob, float* coverage, int32_t* status,
                                void* workspace, size_t ws_bytes, cudaStream_t stream,
                                cudaEvent_t* stage_events) {
    if (!stage_events) return TSD_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i)
        if (!stage_events[i]) return TSD_ERR_INVALID_ARG;
    return verify_tev_impl(target_logits, dtype, parent, token, n_nodes, n_trees, B, V,
                           temperature, seed, exit_node, bonus_token, accept_len, exit_mass,
                           prefix_prob, coverage, status, workspace, ws_bytes, stream,
                           stage_events);
}

tsd_status tsd_verify_ddtree(const void* target_logits, tsd_dtype dtype, const int32_t* parent,
                             const int32_t* token, const int32_t* n_nodes, int n_trees, int B,
                             int64_t V, float temperature, uint64_t seed, int32_t* exit_node,
                             int32_t* bonus_token, int32_t* accept_len, int32_t* draws,
                             int32_t* status, void* workspace, size_t ws_bytes,
                             cudaStream_t stream) {
    if (!verify_args_ok(target_logits, dtype, parent, token, n_nodes, n_trees, B, V, temperature,
                        exit_node, bonus_token, accept_len, status))
        return TSD_ERR_INVALID_ARG;
    const int es = dtype_size(dtype);
    const size_t need = verify_ws_layout(n_trees, B, V, es, nullptr, nullptr);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return TSD_ERR_WORKSPACE;
    if (!logits_view(target_logits, &target_logits)) return TSD_ERR_INVALID_ARG;
    VerifyWs ws;
    verify_ws_layout(n_trees, B, V, es, workspace, &ws);
    const bool greedy = temperature == 0.0f;
    const float c = greedy ? 1.0f : exp2_scale(temperature);
    if (use_two_kernel_path(target_logits, dtype, n_trees, B, V)) {
        if (launch_predraw_fused(target_logits, dtype, n_trees, B, V, c, greedy, seed, parent, token,
                                 n_nodes, ws, exit_node, bonus_token, accept_len, draws, status,
                                 stream) != cudaSuccess)
            return TSD_ERR_CUDA;
        return TSD_OK;
    }
    if (launch_verify_prep(parent, token, n_nodes, n_trees, B, V, ws, stream) != cudaSuccess ||
        launch_rows(target_logits, dtype, n_trees, B, V, c, greedy, n_nodes, ws, stream) != cudaSuccess ||
        launch_node_combine(target_logits, dtype, n_trees, B, V, c, greedy, n_nodes, ws, stream) != cudaSuccess ||
        launch_predraw(target_logits, dtype, n_trees, B, V, c, greedy, seed, n_nodes, ws,
                       exit_node, bonus_token, accept_len, draws, status, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

tsd_status tsd_build_forest(const void* drafter_logits, tsd_dtype dtype, int n_trees, int L,
                            int64_t V, int topk, int B, float drafter_temp, int M_max, double l0,
                            double c1, int32_t* parent, int32_t* token, int32_t* depth,
                            float* score, int32_t* n_nodes, int32_t* status, int32_t* total,
                            void* workspace, size_t ws_bytes, cudaStream_t stream) {
    if (!drafter_logits || !parent || !token || !depth || !score || !n_nodes || !status || !total ||
        !dtype_size(dtype) || !build_sizes_ok(n_trees, 1, L, V, topk, B, dtype_size(dtype)) ||
        (int64_t)n_trees * B > kMaxForestCandidates || M_max < 0 || !(isfinite(l0) && l0 > 0.0) ||
        !(isfinite(c1) && c1 >= 0.0) || !(isfinite(drafter_temp) && drafter_temp >= 1e-6f))
        return TSD_ERR_INVALID_ARG;
    const int es = dtype_size(dtype);
    const size_t need = forest_ws_layout(n_trees, L, V, topk, B, es, nullptr, nullptr, nullptr);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return TSD_ERR_WORKSPACE;
    if (!logits_view(drafter_logits, &drafter_logits)) return TSD_ERR_INVALID_ARG;
    BuildWs ws;
    ForestWs fws;
    forest_ws_layout(n_trees, L, V, topk, B, es, workspace, &ws, &fws);
    const int64_t rows = (int64_t)n_trees * L;
    if (launch_drafter_stats(drafter_logits, dtype, rows, V, topk, exp2_scale(drafter_temp),
                             (double)drafter_temp, ws, stream) != cudaSuccess ||
        launch_build_heap(ws, n_trees, 1, L, topk, B, parent, token, depth, score, nullptr, nullptr,
                          n_nodes, status, stream) != cudaSuccess ||
        launch_forest_select(ws.score64, depth, n_trees, B, M_max, l0, c1, n_nodes, status, total,
                             parent, token, score, fws, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

// Argument checks, workspace and the three kernels every verifier shares
// (tree preparation, row reduction, per-node combination).
static tsd_status verify_front(const void** target_logits, tsd_dtype dtype, const int32_t* parent,
                               const int32_t* token, const int32_t* n_nodes, int n_trees, int B,
                               int64_t V, float temperature, const int32_t* exit_node,
                               const int32_t* bonus_token, const int32_t* accept_len,
                               const int32_t* status, void* workspace, size_t ws_bytes,
                               cudaStream_t stream, VerifyWs* ws, float* c, bool* greedy) {
    if (!verify_args_ok(*target_logits, dtype, parent, token, n_nodes, n_trees, B, V, temperature,
                        exit_node, bonus_token, accept_len, status))
        return TSD_ERR_INVALID_ARG;
    const int es = dtype_size(dtype);
    const size_t need = verify_ws_layout(n_trees, B, V, es, nullptr, nullptr);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return TSD_ERR_WORKSPACE;
    if (!logits_view(*target_logits, target_logits)) return TSD_ERR_INVALID_ARG;
    verify_ws_layout(n_trees, B, V, es, workspace, ws);
    *greedy = temperature == 0.0f;
    *c = *greedy ? 1.0f : exp2_scale(temperature);
    if (launch_verify_prep(parent, token, n_nodes, n_trees, B, V, *ws, stream) != cudaSuccess ||
        launch_rows(*target_logits, dtype, n_trees, B, V, *c, *greedy, n_nodes, *ws, stream) != cudaSuccess ||
        launch_node_combine(*target_logits, dtype, n_trees, B, V, *c, *greedy, n_nodes, *ws, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

tsd_status tsd_verify_seqres(const void* target_logits, tsd_dtype dtype, const int32_t* parent,
                             const int32_t* token, const int32_t* n_nodes, int n_trees, int B,
                             int64_t V, float temperature, uint64_t seed, int32_t* exit_node,
                             int32_t* bonus_token, int32_t* accept_len, int32_t* status,
                             void* workspace, size_t ws_bytes, cudaStream_t stream) {
    VerifyWs ws;
    float c;
    bool greedy;
    const tsd_status st = verify_front(&target_logits, dtype, parent, token, n_nodes, n_trees, B, V,
                                       temperature, exit_node, bonus_token, accept_len, status,
                                       workspace, ws_bytes, stream, &ws, &c, &greedy);
    if (st != TSD_OK) return st;
    if (launch_seqres_tree(target_logits, dtype, n_trees, B, V, c, greedy, seed, n_nodes, ws,
                           exit_node, bonus_token, accept_len, status, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

tsd_status tsd_verify_proposal(const void* target_logits, tsd_dtype dtype, const int32_t* parent,
                               const int32_t* token, const int32_t* n_nodes, const float* q_child,
                               int n_trees, int B, int64_t V, float temperature, uint64_t seed,
                               int32_t* exit_node, int32_t* bonus_token, int32_t* accept_len,
                               int32_t* status, void* workspace, size_t ws_bytes,
                               cudaStream_t stream) {
    if (!q_child) return TSD_ERR_INVALID_ARG;
    VerifyWs ws;
    float c;
    bool greedy;
    const tsd_status st = verify_front(&target_logits, dtype, parent, token, n_nodes, n_trees, B, V,
                                       temperature, exit_node, bonus_token, accept_len, status,
                                       workspace, ws_bytes, stream, &ws, &c, &greedy);
    if (st != TSD_OK) return st;
    if (launch_proposal_tree(target_logits, dtype, n_trees, B, V, c, greedy, seed, q_child,
                             n_nodes, ws, exit_node, bonus_token, accept_len, status,
                             stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

tsd_status tsd_exit_loss(const void* drafter_logits, tsd_dtype dtype, int n_trees, int L,
                         int64_t V, float drafter_temp, const int32_t* token, const int32_t* depth,
                         const int32_t* n_nodes, int B, const float* omega, double* loss_tree,
                         double* loss, float* grad, int32_t* status, void* workspace,
                         size_t ws_bytes, cudaStream_t stream) {
    const int es = dtype_size(dtype);
    if (!drafter_logits || !token || !depth || !n_nodes || !omega || !loss_tree || !loss ||
        !status || !es || n_trees < 1 || L < 1 || L > TSD_MAX_L || B < 0 || B > TSD_MAX_B ||
        V < 1 || V > 0x7fffffff || n_chunks(V, es) > kMaxDrafterChunks ||
        !(isfinite(drafter_temp) && drafter_temp >= 1e-6f))
        return TSD_ERR_INVALID_ARG;
    const size_t need = exit_ws_layout(n_trees, L, V, B, es, nullptr, nullptr);
    if (!workspace || ws_bytes < need || (uintptr_t)workspace % 16) return TSD_ERR_WORKSPACE;
    if (!logits_view(drafter_logits, &drafter_logits)) return TSD_ERR_INVALID_ARG;
    ExitWs ws;
    exit_ws_layout(n_trees, L, V, B, es, workspace, &ws);
    if (launch_exit_loss(drafter_logits, dtype, n_trees, L, V, exp2_scale(drafter_temp),
                         (double)drafter_temp, token, depth, n_nodes, B, omega, loss_tree, loss,
                         grad, status, ws, stream) != cudaSuccess)
        return TSD_ERR_CUDA;
    return TSD_OK;
}

}  // extern "C"
