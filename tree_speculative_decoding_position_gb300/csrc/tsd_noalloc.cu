// tsd_noalloc.cu -- tsd_verify_tev_noalloc: Tree Exit Verification for
// callers that cannot allocate device memory.
//
// Some callers own no device allocator: a plug-in that an inference engine
// hands only its input and output pointers, or a decode loop that must not
// call cudaMalloc because cudaMalloc can synchronise the device and stall
// work already queued.  This entry point takes the same inputs and outputs as
// tsd_verify_tev but no workspace: its scratch is the file-scope device array
// below, of TSD_NOALLOC_SCRATCH_BYTES, which every GPU that loads this library
// holds until the process exits.
//
// The host cannot pass the array's name to a kernel (in host code it is only
// a stand-in for the device symbol), so each call looks up the array's device
// address with cudaGetSymbolAddress, with the call's device current, and
// remembers it per device.  A call made while its stream is being captured
// into a CUDA graph does not look the address up (the runtime may refuse
// such queries during capture): it uses the address remembered by an earlier
// call on that device, and fails with TSD_ERR_CUDA if there was none.  So the
// first call on a device should come before any stream capture, and after a
// cudaDeviceReset the next call should again be made outside a capture (the
// reset reloads the module, and the remembered address is stale until a call
// outside capture looks it up again).
// Nothing here allocates, and no existing entry point changes.
#include <mutex>

#include "tsd_internal.cuh"

namespace {

static __device__ __align__(256) uint8_t g_tev_scratch[TSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_tev_scratch on the current device: looked up on every
// call outside stream capture, remembered for calls under capture.
cudaError_t scratch_address(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_tev_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    } else if (g_scratch_addr[dev] == nullptr) {
        return cudaErrorStreamCaptureUnsupported;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" tsd_status tsd_verify_tev_noalloc(const void* target_logits, tsd_dtype dtype,
                                             const int32_t* parent, const int32_t* token,
                                             const int32_t* n_nodes, int n_trees, int B,
                                             int64_t V, float temperature, uint64_t seed,
                                             int32_t* exit_node, int32_t* bonus_token,
                                             int32_t* accept_len, float* exit_mass,
                                             float* prefix_prob, float* coverage,
                                             int32_t* status, cudaStream_t stream) {
    if (!target_logits || !parent || !token || !n_nodes || !exit_node || !bonus_token ||
        !accept_len || !status)
        return TSD_ERR_INVALID_ARG;
    const size_t need = tsd_workspace_size(TSD_OP_VERIFY_TEV, n_trees, 1, 1, V, 1, B, dtype);
    if (need == 0) return TSD_ERR_INVALID_ARG;
    if (need > (size_t)TSD_NOALLOC_SCRATCH_BYTES) return TSD_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (scratch_address(stream, &scratch) != cudaSuccess) return TSD_ERR_CUDA;
    // Every scratch value the kernels read is first written by the same call,
    // so the previous call's contents need no clearing.
    return tsd_verify_tev(target_logits, dtype, parent, token, n_nodes, n_trees, B, V, temperature,
                          seed, exit_node, bonus_token, accept_len, exit_mass, prefix_prob,
                          coverage, status, scratch, (size_t)TSD_NOALLOC_SCRATCH_BYTES, stream);
}
