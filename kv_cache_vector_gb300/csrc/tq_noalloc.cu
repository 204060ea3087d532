// tq_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// Some callers of this library are not allowed to call cudaMalloc (or any
// allocator) while they run.  Examples: a plugin inside a host framework that
// owns every device allocation through its own memory planner; a serving
// loop whose device memory is fixed up front so that a step can never fail
// or stall on an allocation; code that must not take the allocator's global
// locks.  Such a caller cannot provide the split-K workspace that
// tq_attn_decode needs.  tq_attn_decode_noalloc runs the same kernels, but its
// scratch is a file-scope device array of fixed size, which the CUDA driver
// sets aside when the library's module is loaded on a GPU and keeps until the
// process exits.
#include <cmath>
#include <mutex>

#include "tq_internal.h"

namespace {

// Largest split-K workspace this entry point serves: 8 MiB.  Every GPU that
// loads the library holds this much device memory until exit.
constexpr size_t kScratchBytes = size_t(8) << 20;

__device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

// Host code cannot use g_attn_scratch as a device address (on the host the
// name is only a stand-in for the symbol).  The device address is looked up
// once per device, with that device current, and cached here.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" tq_status tq_attn_decode_noalloc(const tq_plan* plan, const void* q, int B, int Hq,
                                            int Hkv, tq_cache_view cache, int64_t ctx_len,
                                            int k_bits, int v_bits, float scale,
                                            float sparse_v_threshold, float* out,
                                            tq_stream_t stream) {
    // the same checks as tq_attn_decode, bar the caller's workspace
    bool nothing = false;
    tq_status st = tq::check_attn_decode_args(plan, q, B, Hq, Hkv, cache, ctx_len, k_bits, v_bits, scale,
                                              sparse_v_threshold, out, &nothing);
    if (st != TQ_OK || nothing) return st;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    const tq::AttnGeometry g = tq::attn_geometry(B, Hq, Hkv, ctx_len, tq::num_sms(), P->d, k_bits, v_bits,
                                                 sparse_v_threshold > 0.0f);
    if (tq::attn_workspace_bytes(B, Hq, P->d, g) > kScratchBytes) return TQ_ERR_WORKSPACE;
    void* ws = nullptr;
    cudaError_t e = scratch_for_current_device(&ws);
    if (e == cudaSuccess)
        e = tq::launch_attn_decode(*P, q, B, Hq, Hkv, cache, ctx_len, k_bits, v_bits, scale, sparse_v_threshold,
                                   out, nullptr, ws, g, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();  // leave no stale error for the caller's next launch check
        tq::set_last_cuda_error(e);
        return TQ_ERR_CUDA;
    }
    return TQ_OK;
}
