// tq_launch.cu -- host helpers shared by the kernel files: SM count, resident
// blocks per SM, grid sizing, attention split geometry, and the device status
// word that kernels with bounded waits set when they give up.
#include <mutex>

#include "tq_internal.h"

namespace tq {

namespace dev {
__device__ int g_status = 0;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

// Resident blocks per SM of a kernel at a block size, asked once per kernel.
int blocks_per_sm(const void* fn, int block_threads, size_t dyn_smem) {
    static std::mutex mu;
    static const void* keys[512];
    static int vals[512];
    static int n = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (keys[i] == fn) return vals[i];
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, block_threads, dyn_smem) != cudaSuccess ||
        b < 1) {
        cudaGetLastError();
        b = 1;
    }
    if (n < 512) {
        keys[n] = fn;
        vals[n] = b;
        ++n;
    }
    return b;
}

// Grid-stride grids: one wave of resident blocks, or fewer if the work is small.
unsigned grid_for(const void* fn, int block_threads, int64_t items) {
    int64_t want = (items + block_threads - 1) / block_threads;
    const int64_t cap = (int64_t)num_sms() * blocks_per_sm(fn, block_threads, 0);
    if (want > cap) want = cap;
    return (unsigned)(want < 1 ? 1 : want);
}

// Split-K geometry of the decode attention: the longest split (<= 512
// positions) that still gives at least two CTAs per SM.
AttnGeometry attn_geometry(int B, int Hkv, int64_t ctx_len, int sms) {
    AttnGeometry g;
    int split = 512;
    const int64_t pairs = (int64_t)B * Hkv;
    const int64_t want = 2LL * (sms > 0 ? sms : 1);
    while (split > 64 && pairs * ((ctx_len + split - 1) / split) < want) split /= 2;
    g.split_len = split;
    g.n_splits = (int)((ctx_len + split - 1) / split);
    return g;
}

size_t attn_workspace_bytes(int B, int Hq, int d, const AttnGeometry& g) {
    return sizeof(float) * (size_t)B * Hq * g.n_splits * (d + 2);
}

cudaError_t read_device_status(int reset, int* out) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(out, dev::g_status, sizeof(int));
    if (e != cudaSuccess) return e;
    if (reset) {
        int zero = 0;
        e = cudaMemcpyToSymbol(dev::g_status, &zero, sizeof(int));
    }
    return e;
}

}  // namespace tq
