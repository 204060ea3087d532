// tq_launch.cu -- host helpers shared by the kernel files: SM count, resident
// blocks per SM, grid sizing, attention split geometry, and the device status
// word that kernels with bounded waits set when they give up.
#include <mutex>

#include <cudaTypedefs.h>

#include "tq_internal.h"

namespace tq {

namespace dev {
__device__ int g_status = 0;
}

int num_sms() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    if (n < 1) n = 1;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
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

namespace {
// Tuning parameter: the share of the last wave the d = 128 split geometry
// asks its work items to fill.
#ifndef TQ_ATTN3_FILL
#define TQ_ATTN3_FILL 0.97
#endif
// Tuning parameter: the shortest split of the CUDA-core decode attention.
#ifndef TQ_ATTN_MIN_SPLIT
#define TQ_ATTN_MIN_SPLIT 64
#endif
// d = 128: the longest per-warp range (256 down to 32 positions) whose work
// items fill the last wave of one-CTA-per-SM grids to at least TQ_ATTN3_FILL,
// else the one that fills it best; W warps per CTA.
AttnGeometry attn3_geometry(int64_t pairs, int64_t ctx_len, int sms, int W) {
    AttnGeometry g;
    const int64_t cap = sms > 0 ? sms : 1;
    int best = 256;
    double best_eff = -1.0;
    for (int wl = 256; wl >= 32; wl /= 2) {
        const int64_t seg = (int64_t)W * wl;
        const int64_t items = pairs * ((ctx_len + seg - 1) / seg);
        const int64_t grid = items < cap ? (items > 0 ? items : 1) : cap;
        const int64_t rounds = (items + grid - 1) / grid;
        const double eff = rounds > 0 ? (double)items / (double)(rounds * grid) : 1.0;
        if (eff >= TQ_ATTN3_FILL) {
            best = wl;
            break;
        }
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = wl;
        }
    }
    g.warp_len = best;
    g.split_len = W * best;
    g.n_splits = (int)((ctx_len + g.split_len - 1) / g.split_len);
    g.parts = 1;
    g.q16 = true;
    return g;
}
}  // namespace

AttnGeometry attn_qjl128_geometry(int B, int Hq, int Hkv, int64_t ctx_len, int sms, int kb, int vb) {
    return attn3_geometry((int64_t)B * Hkv, ctx_len, sms, attn3_warps(Hkv > 0 ? Hq / Hkv : 1, kb, vb, false, true));
}

size_t attn_qjl128_workspace_bytes(int B, int Hq, const AttnGeometry& g) {
    return 2 * attn3_prefix_bytes(B, Hq) + attn3_partial_bytes(B, Hq, g.n_splits) + attn3_meta_bytes(B, Hq, num_sms());
}

// Split-K geometry of the decode attention.  d = 128 (tensor-core kernel,
// one CTA of attn3_warps(G, kb, vb) warps per SM): attn3_geometry.  Otherwise
// the longest split (<= 512 positions) that still gives two CTAs per SM.
AttnGeometry attn_geometry(int B, int Hq, int Hkv, int64_t ctx_len, int sms, int d, int kb, int vb, bool sparse) {
    AttnGeometry g;
    const int64_t pairs = (int64_t)B * Hkv;
    if (d == 128) return attn3_geometry(pairs, ctx_len, sms, attn3_warps(Hkv > 0 ? Hq / Hkv : 1, kb, vb, sparse));
    // the generic kernel stages its whole range in shared memory: at most 512
    // positions (256 at d = 256) keep two CTAs per SM
    int split = d > 128 ? 256 : 512;
    const int64_t want = 2LL * (sms > 0 ? sms : 1);
    const int cap = split;
    while (split > TQ_ATTN_MIN_SPLIT && pairs * ((ctx_len + split - 1) / split) < want) split /= 2;
    g.split_len = split;
    g.n_splits = (int)((ctx_len + split - 1) / split);
    // At most 8 splits form one thread-block cluster and are merged inside it
    // (no combine launch).  Just past 8, take 8 splits of up to 5/4 the length.
    if (g.n_splits > 8) {
        const int64_t s8 = (ctx_len + 7) / 8;
        if (s8 <= cap && 4 * s8 <= 5 * (int64_t)split) {
            g.split_len = (int)s8;
            g.n_splits = (int)((ctx_len + s8 - 1) / s8);
        }
    }
    g.cluster = g.n_splits <= 8;
    g.parts = 1;
    g.warp_len = 0;
    g.q16 = false;
    return g;
}

AttnGeometry attn_qjl_geometry(int B, int Hq, int Hkv, int64_t ctx_len, int sms) {
    // the generic kernel's geometry (any d other than 128 takes that branch)
    return attn_geometry(B, Hq, Hkv, ctx_len, sms, 64, 2, 2, false);
}

size_t attn_qjl_workspace_bytes(int B, int Hq, int d, const AttnGeometry& g) {
    return sizeof(float) * (attn_qjl_prefix_floats(B, Hq, d) + (size_t)B * Hq * g.n_splits * g.parts * (d + 2));
}

AttnGeometry attn_geometry_paged(int B, int Hq, int Hkv, int64_t max_ctx, int sms, int kb, int vb) {
    // The CTAs' shares are balanced on the device from the actual lengths;
    // here only the slice length is chosen: the longest one that stays under
    // 1/8 of a warp's share if every sequence were max_ctx long.  Longer
    // slices measured faster with varied lengths (fewer items and pair
    // switches per CTA) although they balance more coarsely.
    AttnGeometry g;
    const int W = attn3_warps(Hkv > 0 ? Hq / Hkv : 1, kb, vb);
    const int64_t per_warp = (int64_t)B * Hkv * max_ctx / ((int64_t)W * (sms > 0 ? sms : 1));
    int wl = 256;
    while (wl > 32 && (int64_t)wl * 8 > per_warp) wl /= 2;
    g.warp_len = wl;
    g.split_len = W * wl;
    g.n_splits = (int)((max_ctx + g.split_len - 1) / g.split_len);
    g.parts = 1;
    g.q16 = true;
    return g;
}

size_t attn_paged_workspace_bound(int B, int Hq, int Hkv, int64_t max_ctx, int sms) {
    size_t most = 0;
    for (int kb = 2; kb <= 4; ++kb)
        for (int vb = 2; vb <= 4; ++vb) {
            const size_t w = attn_workspace_bytes(B, Hq, 128, attn_geometry_paged(B, Hq, Hkv, max_ctx, sms, kb, vb));
            if (w > most) most = w;
        }
    return most;
}

size_t attn_workspace_bound(int B, int Hq, int Hkv, int64_t ctx_len, int sms, int d) {
    size_t most = 0;
    for (int kb = 2; kb <= 4; ++kb)
        for (int vb = 2; vb <= 4; ++vb)
            for (int sp = 0; sp < 2; ++sp) {
                const size_t w =
                    attn_workspace_bytes(B, Hq, d, attn_geometry(B, Hq, Hkv, ctx_len, sms, d, kb, vb, sp != 0));
                if (w > most) most = w;
            }
    return most;
}

size_t attn_workspace_bytes(int B, int Hq, int d, const AttnGeometry& g) {
    if (g.q16)
        return attn3_prefix_bytes(B, Hq) + attn3_partial_bytes(B, Hq, g.n_splits) +
               attn3_meta_bytes(B, Hq, num_sms());
    return sizeof(float) * (size_t)B * Hq * g.n_splits * g.parts * (d + 2);
}

int* status_word() {
    static std::mutex mu;
    static int* ptr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, dev::g_status) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        ptr[dev] = static_cast<int*>(p);
    }
    return ptr[dev];
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}
}  // namespace

cudaError_t make_rows_map(CUtensorMap* map, const void* base, int esize, uint64_t d,
                          uint64_t n_rows, uint32_t box_rows) {
    auto fn = encode_tiled_fn();
    if (!fn) return cudaErrorNotSupported;
    const CUtensorMapDataType dt =
        esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t dims[2] = {d, n_rows};
    cuuint64_t strides[1] = {d * (uint64_t)esize};
    cuuint32_t box[2] = {(cuuint32_t)(128 / esize), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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
