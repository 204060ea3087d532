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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

template <int D>
cudaError_t launch_d(int kb, int vb, const void* q, int B, int Hq, int Hkv, const tq_cache_view& c,
                     int64_t ctx, float* out, void* ws, const tq::AttnGeometry& g,
                     const tq::AttnParams& A, cudaStream_t st) {
    switch (kb) {
        case 2: return tq::launch_attn_dk<D, 2>(vb, q, B, Hq, Hkv, c, ctx, out, ws, g, A, st);
        case 3: return tq::launch_attn_dk<D, 3>(vb, q, B, Hq, Hkv, c, ctx, out, ws, g, A, st);
        default: return tq::launch_attn_dk<D, 4>(vb, q, B, Hq, Hkv, c, ctx, out, ws, g, A, st);
    }
}

}  // namespace

extern "C" tq_status tq_attn_decode_noalloc(const tq_plan* plan, const void* q, int B, int Hq,
                                            int Hkv, tq_cache_view cache, int64_t ctx_len,
                                            int k_bits, int v_bits, float scale,
                                            float sparse_v_threshold, float* out,
                                            tq_stream_t stream) {
    if (!plan || B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return TQ_ERR_INVALID_ARG;
    if (k_bits < 2 || k_bits > 4 || v_bits < 2 || v_bits > 4 || Hq / Hkv > 8)
        return TQ_ERR_UNSUPPORTED;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    if (P->d < 32) return TQ_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || !(sparse_v_threshold >= 0.0f) || !std::isfinite(sparse_v_threshold))
        return TQ_ERR_INVALID_ARG;
    if (ctx_len < 1 || ctx_len > cache.cap) return TQ_ERR_RANGE;
    if (B == 0) return TQ_OK;
    if (!q || !out || !cache.k_packed || !cache.k_norm || !cache.v_packed || !cache.v_norm)
        return TQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(cache.k_packed) ||
        !aligned16(cache.v_packed) || !aligned4(cache.k_norm) || !aligned4(cache.v_norm))
        return TQ_ERR_ALIGNMENT;
    const tq::AttnGeometry g = tq::attn_geometry(B, Hq, Hkv, ctx_len, tq::num_sms(), P->d, k_bits, v_bits);
    if (tq::attn_workspace_bytes(B, Hq, P->d, g) > kScratchBytes) return TQ_ERR_WORKSPACE;
    void* ws = nullptr;
    cudaError_t e = scratch_for_current_device(&ws);
    if (e != cudaSuccess) {
        tq::set_last_cuda_error(e);
        return TQ_ERR_CUDA;
    }
    tq::AttnParams A;
    tq::fill_attn_params(*P, k_bits, v_bits, scale, sparse_v_threshold, A);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (P->d) {
        case 32: e = launch_d<32>(k_bits, v_bits, q, B, Hq, Hkv, cache, ctx_len, out, ws, g, A, st); break;
        case 64: e = launch_d<64>(k_bits, v_bits, q, B, Hq, Hkv, cache, ctx_len, out, ws, g, A, st); break;
        case 128: e = launch_d<128>(k_bits, v_bits, q, B, Hq, Hkv, cache, ctx_len, out, ws, g, A, st); break;
        default: e = launch_d<256>(k_bits, v_bits, q, B, Hq, Hkv, cache, ctx_len, out, ws, g, A, st); break;
    }
    if (e != cudaSuccess) {
        tq::set_last_cuda_error(e);
        return TQ_ERR_CUDA;
    }
    return TQ_OK;
}
