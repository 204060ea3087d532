// tq_codec.cu -- sm_103a kernels of the row codec: encode, decode, append.
//
// Encode ("TurboQuant KV Cache Compression -- Spec", Steps 1-3 and As-Built
// Notes 1-2):  load row -> sign flip (xor of the fp32 sign bit) -> FWHT in
// registers -> norm -> bucket through an exact lookup table -> dense LSB-first
// pack -> store.  Decode reverses it: unpack -> centroid -> FWHT -> scale by
// norm / sqrt(d) -> sign -> store.  Rows are independent ("TurboQuantEngine --
// Specification", 7 Non-goals: each row encoded independently), so the grid
// simply strides over rows.
#include <cfloat>
#include <cuda_fp16.h>

#include "tq_async.cuh"
#include "tq_device.cuh"
#include "tq_umma.cuh"

namespace tq {
namespace dev {

constexpr int kBlock = 256;

// ------------------------------------------------------------------ encode

// Encode the thread's part of one row.  `valid` lanes store; the others only
// take part in the shuffle of the cross-thread stage.
template <int D, int BITS, typename T, bool LUT>
__device__ __forceinline__ void encode_part(const T* __restrict__ row, uint8_t* __restrict__ dst,
                                            float* __restrict__ dst_norm, int p, bool valid,
                                            const RowParams& P, const LutEntry* lut,
                                            const float* bnd_s) {
    constexpr int R = RowShape<D>::R, E = RowShape<D>::E;
    float v[E];
    load_signed<E>(row + p * E, v, P.sgn + p * E);
    // sum of squares of the row (signs do not matter), four partial sums
    float ss0 = 0.f, ss1 = 0.f, ss2 = 0.f, ss3 = 0.f;
#pragma unroll
    for (int i = 0; i < E; i += 4) {
        ss0 = fmaf(v[i], v[i], ss0);
        if (i + 1 < E) ss1 = fmaf(v[i + 1], v[i + 1], ss1);
        if (i + 2 < E) ss2 = fmaf(v[i + 2], v[i + 2], ss2);
        if (i + 3 < E) ss3 = fmaf(v[i + 3], v[i + 3], ss3);
    }
    float ss = (ss0 + ss1) + (ss2 + ss3);
    if constexpr (R == 2) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
    fwht_reg<E>(v);
    if constexpr (R == 2) fwht_cross<E>(v, p);
    if (P.two_sided) flip_rotated<D>(v, p, P.sgn2);
    float n = __fsqrt_rn(ss);
    // w = y * inv is the normalised coordinate u = (H s x / sqrt(d)) / n
    float inv = n > 0.f ? __fdiv_rn(P.inv_sqrt_d, n) : 0.f;
    if (!ss_in_range(ss)) {  // both threads of a row (R = 2) agree: ss is shared
        float m = 0.f;
        bool nf = false;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const float a = fabsf(v[i]);
            nf = nf || !(a <= FLT_MAX);
            m = fmaxf(m, a);
        }
        if constexpr (R == 2) {
            const unsigned am = __activemask();
            m = fmaxf(m, __shfl_xor_sync(am, m, 1));
            nf = __shfl_xor_sync(am, (int)nf, 1) != 0 || nf;
        }
        if (!nf && m > 0.f) {  // squares past fp32's range: the sums again on y S
            const float S = pow2_scale(m);
            float t = 0.f;
#pragma unroll
            for (int i = 0; i < E; ++i) t = fmaf(v[i] * S, v[i] * S, t);
            if constexpr (R == 2) t += __shfl_xor_sync(__activemask(), t, 1);
            scaled_norm<D>(t, S, n, inv);
        }
    }
    const float inv_s = inv * (float)kLutScale;

    constexpr int NW = (E * BITS + 31) / 32;
    uint32_t w[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        int id;
        if constexpr (LUT) id = bucket_lut(lut, v[i], inv, inv_s);
        else id = bucket_search<BITS>(bnd_s, v[i], inv);
        const int pos = i * BITS, wi = pos / 32, sh = pos % 32;
        w[wi] |= (uint32_t)id << sh;
        if (sh + BITS > 32) w[wi + 1] |= (uint32_t)id >> (32 - sh);
    }
    if (!valid) return;
    if constexpr (R == 1) {
        store_bytes<D * BITS / 8>(dst, w);
    } else {
        // split layout: two runs of E/2 indices
        constexpr int HB = E / 2 * BITS / 8;  // bytes per run
        store_bytes<HB>(dst + p * HB, w);
        store_bytes<HB>(dst + 2 * HB + p * HB, w + HB / 4);
    }
    if (p == 0) *dst_norm = n;
}

template <int D, int BITS, typename T>
__global__ void __launch_bounds__(kBlock) k_encode(const T* __restrict__ x, int64_t n_rows,
                                                   uint8_t* __restrict__ packed,
                                                   float* __restrict__ norms,
                                                   const __grid_constant__ RowParams P) {
    __shared__ LutEntry lut[kLutCells];
    build_lut(lut, P.bnd, (1 << BITS) - 1);
    __syncthreads();
    constexpr int R = RowShape<D>::R;
    constexpr int RB = D * BITS / 8;
    const int64_t n_items = n_rows * R;
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kBlock;
    for (int64_t base = (int64_t)blockIdx.x * kBlock + (threadIdx.x - lane); base < n_items;
         base += stride) {
        const int64_t item = base + lane;
        const bool valid = item < n_items;
        const int64_t row = valid ? item / R : n_rows - 1;
        const int p = (int)(item % R);
        encode_part<D, BITS, T, true>(x + row * D, packed + row * RB, norms + row, p, valid, P,
                                      lut, nullptr);
    }
}

// Append: blockIdx.y = 0 encodes the K rows, 1 the V rows.  Source row
// (b, h, i) of [B][Hkv][n_new][d] goes to cache row (b, h, pos + i) of
// [B][Hkv][cap].  Few rows per launch: binary-search bucketing, no table.
template <int D, int BITS, typename T>
__device__ __forceinline__ void append_rows(const T* __restrict__ src, uint8_t* __restrict__ pk,
                                            float* __restrict__ nrm, int64_t n_items,
                                            int64_t n_new, int64_t cap, int64_t pos,
                                            const RowParams& P, const float* bnd_s) {
    constexpr int R = RowShape<D>::R;
    constexpr int RB = D * BITS / 8;
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kBlock;
    for (int64_t base = (int64_t)blockIdx.x * kBlock + (threadIdx.x - lane); base < n_items;
         base += stride) {
        const int64_t item = base + lane;
        const bool valid = item < n_items;
        const int64_t srow = valid ? item / R : n_items / R - 1;
        const int p = (int)(item % R);
        const int64_t bh = srow / n_new, i = srow % n_new;
        const int64_t drow = bh * cap + pos + i;
        encode_part<D, BITS, T, false>(src + srow * D, pk + drow * RB, nrm + drow, p, valid, P,
                                       nullptr, bnd_s);
    }
}

template <int D, typename T>
__global__ void __launch_bounds__(kBlock) k_append(const T* __restrict__ k_new,
                                                   const T* __restrict__ v_new, int64_t n_rows,
                                                   int64_t n_new, tq_cache_view cache, int64_t pos,
                                                   int k_bits, int v_bits,
                                                   const __grid_constant__ RowParams PK,
                                                   const __grid_constant__ RowParams PV) {
    __shared__ float bnd_s[16];
    const bool is_v = blockIdx.y == 1;
    const RowParams& P = is_v ? PV : PK;
    if (threadIdx.x < 16) bnd_s[threadIdx.x] = P.bnd[threadIdx.x];
    __syncthreads();
    const int bits = is_v ? v_bits : k_bits;
    const T* src = is_v ? v_new : k_new;
    uint8_t* pk = is_v ? cache.v_packed : cache.k_packed;
    float* nrm = is_v ? cache.v_norm : cache.k_norm;
    const int64_t n_items = n_rows * RowShape<D>::R;
    switch (bits) {
        case 2: append_rows<D, 2, T>(src, pk, nrm, n_items, n_new, cache.cap, pos, P, bnd_s); break;
        case 3: append_rows<D, 3, T>(src, pk, nrm, n_items, n_new, cache.cap, pos, P, bnd_s); break;
        default: append_rows<D, 4, T>(src, pk, nrm, n_items, n_new, cache.cap, pos, P, bnd_s); break;
    }
}

// Append for d >= 32, built for latency (a decode step appends a few rows):
// one warp per row (warp_encode_indices, warp_pack_row), kAppWarps rows per
// block.  Launched with programmatic dependent launch: the sign tables are
// set up while the previous kernel of the stream finishes, and the rows and
// the cache are touched only after it has.
constexpr int kAppWarps = 4;

// PAGED: one new row per (sequence, KV head) (n_new = 1), written at position
// pa.lens[b] of a paged cache; a position or page id out of range writes
// nothing and sets the status word to kAppStatusRange.
constexpr int kAppStatusRange = 42;

template <int D, typename T, bool PAGED>
__global__ void __launch_bounds__(32 * kAppWarps) k_append_warp(const T* __restrict__ k_new,
                                                                const T* __restrict__ v_new, int64_t n_rows,
                                                                int64_t n_new, tq_cache_view cache,
                                                                int64_t pos, int k_bits, int v_bits,
                                                                const __grid_constant__ RowParams PK,
                                                                const __grid_constant__ RowParams PV,
                                                                const PagedArgs pa, int Hkv, int* status) {
    static_assert(D >= 32 && D <= kMaxD, "one warp per row");
    __shared__ uint32_t sg[D], sg2[D];
    __shared__ uint8_t idxbuf[kAppWarps][D];
    const bool is_v = blockIdx.y == 1;
    const RowParams& P = is_v ? PV : PK;
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
        sg[i] = sign_mask(P.sgnb, i);
        sg2[i] = sign_mask(P.sgn2b, i);
    }
    __syncthreads();
    griddep_wait();    // the new rows, and readers of the cache, of the previous kernel
    griddep_launch();  // the next kernel may set itself up; it waits for this grid
    const int bits = is_v ? v_bits : k_bits;
    const int nb = (1 << bits) - 1;
    const T* src = is_v ? v_new : k_new;
    uint8_t* pk = is_v ? cache.v_packed : cache.k_packed;
    float* nrm = is_v ? cache.v_norm : cache.k_norm;
    const int rb = D * bits / 8;  // bytes per packed row (a multiple of 4)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ib = idxbuf[warp];
    for (int64_t srow = (int64_t)blockIdx.x * kAppWarps + warp; srow < n_rows;
         srow += (int64_t)gridDim.x * kAppWarps) {
        const float n = warp_encode_indices<D, T>(src + srow * D, lane, sg, P.two_sided ? sg2 : nullptr, P, nb, ib);
        int64_t drow;
        if constexpr (PAGED) {
            const int64_t b = srow / Hkv;
            const int h = (int)(srow - b * Hkv);
            const int64_t p = __ldg(pa.lens + b);
            const int64_t cap = (int64_t)pa.max_pages << pa.page_shift;
            const int page = (p >= 0 && p < cap) ? __ldg(pa.bt + b * pa.max_pages + (p >> pa.page_shift)) : -1;
            if (page < 0 || page >= pa.n_pages) {  // warp-uniform: nothing is written for this row
                if (lane == 0 && status) atomicCAS(status, 0, kAppStatusRange);
                __syncwarp();
                continue;
            }
            drow = (((int64_t)page * Hkv + h) << pa.page_shift) + (p & ((int64_t(1) << pa.page_shift) - 1));
        } else {
            drow = (srow / n_new) * cache.cap + pos + srow % n_new;
        }
        warp_pack_row<D>(ib, lane, bits, pk + drow * rb);
        if (lane == 0) nrm[drow] = n;
        __syncwarp();
    }
}

// ------------------------------------------------------------------ decode

template <int D, int BITS, typename TO>
__device__ __forceinline__ void decode_part(const uint8_t* __restrict__ src, float norm,
                                            TO* __restrict__ dst, int p, bool valid,
                                            const RowParams& P, const float* cen_s) {
    constexpr int R = RowShape<D>::R, E = RowShape<D>::E;
    constexpr int NW = (E * BITS + 31) / 32;
    uint32_t w[NW];
    if constexpr (R == 1) {
        load_bytes<D * BITS / 8>(src, w);
    } else {
        constexpr int HB = E / 2 * BITS / 8;
        load_bytes<HB>(src + p * HB, w);
        load_bytes<HB>(src + 2 * HB + p * HB, w + HB / 4);
    }
    float v[E];
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = cen_s[unpack_one<BITS>(w, i)];
    if (P.two_sided) flip_rotated<D>(v, p, P.sgn2);
    fwht_reg<E>(v);
    if constexpr (R == 2) fwht_cross<E>(v, p);  // split -> contiguous
    const float sc = norm * P.inv_sqrt_d;
    const uint32_t* sg = P.sgn + p * E;
    if (!valid) return;
    TO* out = dst + p * E;
    if constexpr (sizeof(TO) == 4) {
#pragma unroll
        for (int k = 0; k < E; k += 4) {
            float4 o;
            o.x = __uint_as_float(__float_as_uint(v[k] * sc) ^ sg[k]);
            o.y = __uint_as_float(__float_as_uint(v[k + 1] * sc) ^ sg[k + 1]);
            o.z = __uint_as_float(__float_as_uint(v[k + 2] * sc) ^ sg[k + 2]);
            o.w = __uint_as_float(__float_as_uint(v[k + 3] * sc) ^ sg[k + 3]);
            reinterpret_cast<float4*>(out)[k / 4] = o;
        }
    } else {
        // bf16: round to nearest even; the sign flip commutes with rounding
#pragma unroll
        for (int k = 0; k < E; k += 8) {
            uint32_t q[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[k + 2 * m] * sc, v[k + 2 * m + 1] * sc);
                uint32_t bits = *reinterpret_cast<uint32_t*>(&h);
                bits ^= (sg[k + 2 * m] >> 16) | sg[k + 2 * m + 1];
                q[m] = bits;
            }
            reinterpret_cast<uint4*>(out)[k / 8] = make_uint4(q[0], q[1], q[2], q[3]);
        }
    }
}

template <int D, int BITS, typename TO>
__global__ void __launch_bounds__(kBlock) k_decode(const uint8_t* __restrict__ packed,
                                                   const float* __restrict__ norms,
                                                   int64_t n_rows, TO* __restrict__ y,
                                                   const __grid_constant__ RowParams P) {
    __shared__ float cen_s[16];
    if (threadIdx.x < 16) cen_s[threadIdx.x] = P.cen[threadIdx.x];
    __syncthreads();
    constexpr int R = RowShape<D>::R;
    constexpr int RB = D * BITS / 8;
    const int64_t n_items = n_rows * R;
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kBlock;
    for (int64_t base = (int64_t)blockIdx.x * kBlock + (threadIdx.x - lane); base < n_items;
         base += stride) {
        const int64_t item = base + lane;
        const bool valid = item < n_items;
        const int64_t row = valid ? item / R : n_rows - 1;
        const int p = (int)(item % R);
        decode_part<D, BITS, TO>(packed + row * RB, __ldg(norms + row), y + row * D, p, valid, P,
                                 cen_s);
    }
}

}  // namespace dev

namespace dev {

// ------------------------------------------------- encode, TMA-fed (v2)
//
// Persistent, warp-specialised: warp 4 issues 2-D TMA loads of 128-row tiles
// (128-byte boxes, 128-byte swizzle) into a ring of shared-memory stages;
// warps 0-3 take one row per thread, read it conflict-free from the swizzled
// stage, release the stage and encode the row in registers.  bf16 rows only.

constexpr int kTmaRows = 128;
constexpr int kTmaThreads = 160;

template <int D>
struct TmaEncodeShape {
    static constexpr int kBoxes = D * 2 / 128;                       // 128-byte boxes per row
    static constexpr int kStageBytes = kTmaRows * D * 2;
    static constexpr int kStages = kStageBytes <= 16384 ? 6 : 3;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kLutCells * 8 + 2 * kStages * 8;
};

template <int D, int BITS>
__global__ void __launch_bounds__(kTmaThreads, 2)
k_encode_tma(const __grid_constant__ CUtensorMap xmap, int64_t n_rows, uint8_t* __restrict__ packed,
             float* __restrict__ norms, int* status, const __grid_constant__ RowParams P) {
    using S = TmaEncodeShape<D>;
    constexpr int RB = D * BITS / 8;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle, by pointer arithmetic on
    // the shared array (keeps every access below a shared-memory access).
    unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char* stages = base;
    LutEntry* lut = reinterpret_cast<LutEntry*>(stages + S::kStages * S::kStageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(lut + kLutCells);
    uint64_t* empty = full + S::kStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 4);
        }
        mbar_fence_init();
    }
    build_lut(lut, P.bnd, (1 << BITS) - 1);
    __syncthreads();
    const int64_t n_tiles = (n_rows + kTmaRows - 1) / kTmaRows;

    if (warp == 4) {  // ---- producer
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            int it = 0;
            for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
                const int s = it % S::kStages;
                const uint32_t k = it / S::kStages;
                if (it >= S::kStages && !mbar_wait(&empty[s], (k - 1) & 1)) {
                    report_timeout(status, 1);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], S::kStageBytes);
#pragma unroll
                for (int b = 0; b < S::kBoxes; ++b)
                    tma_load_2d(stages + s * S::kStageBytes + b * kTmaRows * 128, &xmap, b * 64,
                                (int)(tile * kTmaRows), &full[s]);
            }
            // Loads still in flight must land before this CTA may exit.
            const int last = it;
            for (int j = (last > S::kStages ? last - S::kStages : 0); j < last; ++j) {
                if (!mbar_wait(&full[j % S::kStages], (j / S::kStages) & 1)) {
                    report_timeout(status, 2);
                    break;
                }
            }
        }
        return;
    }

    // ---- consumers: one row per thread
    const int r = threadIdx.x;  // 0..127
    int it = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
        const int s = it % S::kStages;
        if (!mbar_wait(&full[s], (it / S::kStages) & 1)) {
            report_timeout(status, 3);
            break;
        }
        float v[D];
        const unsigned char* st = stages + s * S::kStageBytes;
#pragma unroll
        for (int b = 0; b < S::kBoxes; ++b) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 q = *reinterpret_cast<const uint4*>(
                    st + b * kTmaRows * 128 + r * 128 + ((c ^ (r & 7)) << 4));
                const uint32_t* m = P.sgn + b * 64 + c * 8;
                float* o = v + b * 64 + c * 8;
                o[0] = bf16lo(q.x, m[0]);
                o[1] = bf16hi(q.x, m[1]);
                o[2] = bf16lo(q.y, m[2]);
                o[3] = bf16hi(q.y, m[3]);
                o[4] = bf16lo(q.z, m[4]);
                o[5] = bf16hi(q.z, m[5]);
                o[6] = bf16lo(q.w, m[6]);
                o[7] = bf16hi(q.w, m[7]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        F2 sa = f2(0.f, 0.f), sb = f2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < D; i += 4) {
            const F2 p0 = f2(v[i], v[i + 1]);
            const F2 p1 = f2(v[i + 2], v[i + 3]);
            sa = f2_fma(p0, p0, sa);
            sb = f2_fma(p1, p1, sb);
        }
        float s0, s1, s2, s3;
        f2_split(sa, s0, s1);
        f2_split(sb, s2, s3);
        const float ss = (s0 + s1) + (s2 + s3);
        fwht_reg2<D>(v);
        if (P.two_sided) flip_rotated<D>(v, 0, P.sgn2);
        float n = __fsqrt_rn(ss);
        float inv = n > 0.f ? __fdiv_rn(P.inv_sqrt_d, n) : 0.f;
        if (!ss_in_range(ss)) {
            float m = 0.f;
            bool nf = false;
#pragma unroll
            for (int i = 0; i < D; ++i) {
                const float a = fabsf(v[i]);
                nf = nf || !(a <= FLT_MAX);
                m = fmaxf(m, a);
            }
            if (!nf && m > 0.f) {  // squares past fp32's range: the sums again on y S
                const float S = pow2_scale(m);
                float t = 0.f;
#pragma unroll
                for (int i = 0; i < D; ++i) t = fmaf(v[i] * S, v[i] * S, t);
                scaled_norm<D>(t, S, n, inv);
            }
        }
        const float ks = inv * (float)kLutScale;
        const F2 K2 = f2(ks, ks);
        constexpr float kMagic = 12582912.0f + (float)kLutCenter;
        const F2 M2 = f2(kMagic, kMagic);
        constexpr int NW = D * BITS / 32;
        uint32_t w[NW];
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] = 0;
#pragma unroll
        for (int i = 0; i < D; i += 2) {
            float fx, fy;
            f2_split(f2_fma(f2(v[i], v[i + 1]), K2, M2), fx, fy);
            const LutEntry e0 = lut[__float_as_uint(fx) & (kLutCells - 1)];
            const LutEntry e1 = lut[__float_as_uint(fy) & (kLutCells - 1)];
            const int id0 = e0.lo + (fmaf(v[i], inv, -e0.thr) >= 0.0f ? 1 : 0);
            const int id1 = e1.lo + (fmaf(v[i + 1], inv, -e1.thr) >= 0.0f ? 1 : 0);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int id = h ? id1 : id0;
                const int pos = (i + h) * BITS, wi = pos / 32, sh = pos % 32;
                w[wi] += (uint32_t)id << sh;
                if (sh + BITS > 32) w[wi + 1] += (uint32_t)id >> (32 - sh);
            }
        }
        const int64_t row = tile * kTmaRows + r;
        if (row < n_rows) {
            store_bytes<RB>(packed + row * RB, w);
            norms[row] = n;
        }
    }
}

// ------------------------------------------- encode on tcgen05 (d = 128)
//
// y = H (s . x) for a tile of 128 rows is one GEMM, Y = X (D H): X (128 x 128
// bf16, TMA-loaded, K-major, 128-byte swizzle) times the constant +-1 matrix
// D H (bf16, built once per CTA in shared memory) on the tensor cores, fp32
// accumulation in tensor memory.  Warp roles: 0 = TMA producer, 1 = MMA
// issuer (and tensor-memory owner), 2-9 = two epilogue warpgroups taking
// alternate tiles; each epilogue thread reads its row from tensor memory
// (32x32b loads), forms the norm, buckets through the exact table and packs.

constexpr int kUmRows = 128;
constexpr int kUmStages = 3;
constexpr int kUmAcc = 4;             // tensor-memory accumulators of 128 columns
constexpr int kUmThreads = 10 * 32;
constexpr int kUmStageBytes = kUmRows * 128 * 2;
// Shared memory by absolute shared-window address.  The lane-replicated
// bucketing table sits at 64 KiB: entry (cell c, lane l) is at
// kUmRepAt + 256 c + 8 l, so its address is one byte permute of the cell's
// low byte.
constexpr uint32_t kUmHbAt = 2048;                              // D H (32 KB)
constexpr uint32_t kUmBarAt = kUmHbAt + 128 * 128 * 2;          // barriers, TMEM slot
constexpr uint32_t kUmRepAt = 65536;                            // replicated window (64 KB)
constexpr uint32_t kUmXsAt = 131072;                            // X stages
constexpr uint32_t kUmEnd = kUmXsAt + kUmStages * kUmStageBytes;
constexpr uint32_t kUmSgnAt = kUmBarAt + 256;  // s and s2 masks (1 KB), read when building D H
static_assert(kUmBarAt + (2 * kUmStages + 2 * kUmAcc) * 8 + 16 <= kUmSgnAt, "layout");
static_assert(kUmSgnAt + 1024 <= kUmRepAt, "layout");
static_assert(kUmEnd <= 232448, "shared memory");
// The tensor-core encoders' tables: cells k = rint(w * kUmLutScale) in
// [-64, 64], every finite row, indexed by one byte, k + 128.
constexpr int kRepCells = 256;

__device__ __forceinline__ LutEntry lds_entry(uint32_t addr) {
    LutEntry e;
    asm("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(e.lo), "=f"(e.thr) : "r"(addr));
    return e;
}

// Table entry of the cell k = rint(w * scale) (same rule as build_lut).
__device__ __forceinline__ LutEntry lut_cell(const float* bnd, int nb, int k, int scale) {
    const float lo = (float)(k - 0.5) / (float)scale;
    const float hi = (float)(k + 0.5) / (float)scale;
    LutEntry e;
    e.lo = 0;
    e.thr = __int_as_float(0x7F800000);
    for (int j = 0; j < nb; ++j) {
        const float b = bnd[j];
        if (b < lo) e.lo += 1;
        else if (b <= hi) e.thr = b;
    }
    return e;
}

template <int BITS>
__global__ void __launch_bounds__(kUmThreads, 1)
k_encode_umma(const __grid_constant__ CUtensorMap xmap, int64_t n_rows, uint8_t* __restrict__ packed,
              float* __restrict__ norms, int* status, const __grid_constant__ RowParams P) {
    constexpr int RB = 128 * BITS / 8;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t sbase = smem_addr(smem_raw);
    if (sbase > kUmHbAt) {  // the layout assumes dynamic memory starts lower
        if (threadIdx.x == 0) report_timeout(status, 17);
        return;
    }
    griddep_launch();
    auto at = [&](uint32_t a) { return smem_raw + (a - sbase); };
    unsigned char* xs = at(kUmXsAt);                            // stages of X
    unsigned char* hb = at(kUmHbAt);                            // D H, K-major
    uint64_t* full = reinterpret_cast<uint64_t*>(at(kUmBarAt));
    uint64_t* empty = full + kUmStages;
    uint64_t* accf = empty + kUmStages;
    uint64_t* acce = accf + kUmAcc;
    uint32_t* slot = reinterpret_cast<uint32_t*>(acce + kUmAcc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // B operand: element (n, k) = s2_n * (-1)^popcount(n & k) * s_k (s2 all
    // +1 unless the signs are two-sided), stored like a TMA 128-byte-swizzled
    // K-major tile (two 64-column halves of 16 KB).  The sign masks are staged
    // in shared memory first, from the bit words (a warp reads one word):
    // indexed reads of the parameter bank with a different index per lane
    // would be serialised.
    uint32_t* sg = reinterpret_cast<uint32_t*>(at(kUmSgnAt));
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
        sg[i] = sign_mask(P.sgnb, i);
        sg[128 + i] = sign_mask(P.sgn2b, i);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {
        const int n = i >> 7, k = i & 127;
        const bool neg = (((__popc(n & k) & 1) != 0) != (sg[k] != 0u)) != (sg[128 + n] != 0u);
        const int off = (k >> 6) * 16384 + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2;
        *reinterpret_cast<uint16_t*>(hb + off) = neg ? 0xBF80u : 0x3F80u;
    }
    for (int c = threadIdx.x; c < kRepCells; c += blockDim.x) {
        const LutEntry e = lut_cell(P.bnd, (1 << BITS) - 1, c - kRepCells / 2, kUmLutScale);
        LutEntry* row = reinterpret_cast<LutEntry*>(at(kUmRepAt + 256u * c));
#pragma unroll 4
        for (int l = 0; l < 32; ++l) row[l] = e;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kUmStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < kUmAcc; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], 4);
        }
        mbar_fence_init();
    }
    fence_proxy_async_smem();
    if (warp == 1) tmem_alloc<kUmAcc * 128>(slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    // the prologue above reads the parameters only; the rows and the outputs
    // may belong to the previous kernel in the stream
    griddep_wait();
    const int64_t n_tiles = (n_rows + kUmRows - 1) / kUmRows;

    if (warp == 0) {  // ---- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            int it = 0;
            for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
                const int s = it % kUmStages;
                if (it >= kUmStages && !mbar_wait(&empty[s], ((it / kUmStages) - 1) & 1)) {
                    report_timeout(status, 11);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], kUmStageBytes);
                tma_load_2d(xs + s * kUmStageBytes, &xmap, 0, (int)(tile * kUmRows), &full[s]);
                tma_load_2d(xs + s * kUmStageBytes + 16384, &xmap, 64, (int)(tile * kUmRows), &full[s]);
            }
            for (int j = (it > kUmStages ? it - kUmStages : 0); j < it; ++j)
                if (!mbar_wait(&full[j % kUmStages], (j / kUmStages) & 1)) {
                    report_timeout(status, 12);
                    break;
                }
        }
    } else if (warp == 1) {  // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16(128, 128, true);
            const uint32_t xs_a = smem_addr(xs), hb_a = smem_addr(hb);
            int it = 0;
            for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
                const int s = it % kUmStages, a = it % kUmAcc;
                if (!mbar_wait(&full[s], (it / kUmStages) & 1)) {
                    report_timeout(status, 13);
                    break;
                }
                if (it >= kUmAcc && !mbar_wait(&acce[a], ((it / kUmAcc) - 1) & 1)) {
                    report_timeout(status, 14);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    umma_f16(tmem + a * 128, umma_desc_sw128(xs_a + s * kUmStageBytes + off),
                             umma_desc_sw128(hb_a + off), idesc, kk > 0 ? 1u : 0u);
                }
                umma_commit(&empty[s]);
                umma_commit(&accf[a]);
            }
            // the last accumulators must be complete before tensor memory is freed
            for (int j = (it > kUmAcc ? it - kUmAcc : 0); j < it; ++j)
                if (!mbar_wait(&accf[j % kUmAcc], (j / kUmAcc) & 1)) {
                    report_timeout(status, 15);
                    break;
                }
        }
    } else {  // ---- epilogue: warps 2-5 take even tiles, 6-9 odd tiles
        const int wg = (warp - 2) >> 2, q = warp & 3;
        const int r = 32 * q + lane;
        constexpr int NW = 128 * BITS / 32;
        constexpr float kMagic = 12582912.0f + (float)(kRepCells / 2);
        const F2 M2 = f2(kMagic, kMagic);
        const uint32_t rep_slot = kUmRepAt + 8u * lane;
        int it = wg;
        for (int64_t tile = blockIdx.x + (int64_t)wg * gridDim.x; tile < n_tiles;
             tile += 2 * (int64_t)gridDim.x, it += 2) {
            const int a = it % kUmAcc;
            if (!mbar_wait(&accf[a], (it / kUmAcc) & 1)) {
                report_timeout(status, 16);
                break;
            }
            tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + a * 128;
            F2 sa = f2(0.f, 0.f), sb = f2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t y[32];
                tmem_ld32(ta + 32 * c, y);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const F2 p0 = f2(__uint_as_float(y[i]), __uint_as_float(y[i + 1]));
                    const F2 p1 = f2(__uint_as_float(y[i + 2]), __uint_as_float(y[i + 3]));
                    sa = f2_fma(p0, p0, sa);
                    sb = f2_fma(p1, p1, sb);
                }
            }
            float s0, s1, s2, s3;
            f2_split(sa, s0, s1);
            f2_split(sb, s2, s3);
            const float ss = (s0 + s1) + (s2 + s3);  // = d * ||x||^2
            float n = __fsqrt_rn(ss * (1.0f / 128.0f));
            float inv = ss > 0.f ? __frcp_rn(__fsqrt_rn(ss)) : 0.f;  // w = y / sqrt(ss) = u
            bool slow = false;  // a coordinate is not finite: binary search below
            const bool odd = !ss_in_range(ss);
            if (__any_sync(0xFFFFFFFFu, odd)) {
                // squares past fp32's range (or a zero or non-finite row): the
                // sums again on y S (rare; the tensor-memory loads are warp-wide)
                float m = 0.f;
                bool nf = false;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t y[32];
                    tmem_ld32(ta + 32 * c, y);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float a = fabsf(__uint_as_float(y[i]));
                        nf = nf || !(a <= FLT_MAX);
                        m = fmaxf(m, a);
                    }
                }
                const float S = (odd && !nf && m > 0.f) ? pow2_scale(m) : 1.f;
                float t = 0.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t y[32];
                    tmem_ld32(ta + 32 * c, y);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float a = __uint_as_float(y[i]) * S;
                        t = fmaf(a, a, t);
                    }
                }
                if (odd) {
                    if (nf) slow = true;
                    else if (m > 0.f) scaled_norm<128>(t, S, n, inv);
                }
            }
            const float ks = inv * (float)kUmLutScale;
            const F2 K2 = f2(ks, ks);
            uint32_t w[NW];
#pragma unroll
            for (int k = 0; k < NW; ++k) w[k] = 0;
            // Cells come from the replicated table (conflict-free: lane l
            // reads only its own column).  A finite row has |w| <= 1, so its
            // cells are 64 .. 192 and no coordinate needs a further check.
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t y[32];
                tmem_ld32(ta + 32 * c, y);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float y0 = __uint_as_float(y[i]), y1 = __uint_as_float(y[i + 1]);
                    float fx, fy;
                    f2_split(f2_fma(f2(y0, y1), K2, M2), fx, fy);
                    const uint32_t bx = __float_as_uint(fx), by = __float_as_uint(fy);
                    const LutEntry e0 = lds_entry(__byte_perm(bx, rep_slot, 0x7604));
                    const LutEntry e1 = lds_entry(__byte_perm(by, rep_slot, 0x7604));
                    const int id0 = e0.lo + (fmaf(y0, inv, -e0.thr) >= 0.0f ? 1 : 0);
                    const int id1 = e1.lo + (fmaf(y1, inv, -e1.thr) >= 0.0f ? 1 : 0);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int id = h ? id1 : id0;
                        const int pos = (32 * c + i + h) * BITS, wi = pos / 32, sh = pos % 32;
                        w[wi] += (uint32_t)id << sh;
                        if (sh + BITS > 32) w[wi + 1] += (uint32_t)id >> (32 - sh);
                    }
                }
            }
            // Rows with a NaN or infinite coordinate: exact binary search over
            // the boundaries, as the other encoders take it (the
            // tensor-memory loads are warp-wide).
            if (__any_sync(0xFFFFFFFFu, slow)) {
                if (slow) {
#pragma unroll
                    for (int k = 0; k < NW; ++k) w[k] = 0;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t y[32];
                    tmem_ld32(ta + 32 * c, y);
                    tmem_wait_ld();
                    if (slow) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int id = bucket_search<BITS>(P.bnd, __uint_as_float(y[i]), inv);
                            const int pos = (32 * c + i) * BITS, wi = pos / 32, sh = pos % 32;
                            w[wi] += (uint32_t)id << sh;
                            if (sh + BITS > 32) w[wi + 1] += (uint32_t)id >> (32 - sh);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[a]);
            const int64_t row = tile * kUmRows + r;
            if (row < n_rows) {
                store_bytes<RB>(packed + row * RB, w);
                norms[row] = n;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<kUmAcc * 128>(tmem);
    }
}

// ------------------------------------------- encode on tcgen05 (d = 256)
//
// H_256 = [[H, H], [H, -H]] (Sylvester order), so for a row x = [x0, x1] of
// 2 x 128 elements, y = H_256 (s . x) = [A0 + A1, A0 - A1] with
// A_p = H (s_p . x_p).  For a tile of 128 rows both A_p are tensor-core GEMMs
// against the constant +-1 matrices D_p H, as in the d = 128 encoder: X is
// TMA-loaded in 32 KB halves (columns 0..127, then 128..255) through three
// stages, and half p goes to accumulator columns 128 p of the tile's
// 256-column pair.  The epilogue forms A0 +- A1, the norm (||y||^2 =
// 2 (||A0||^2 + ||A1||^2) = d ||x||^2), the second signs when the plan has
// them (they differ between the two output halves, so they are not folded
// into D_p H), buckets and packs.  The bucketing table is the d = 128 one
// (count of boundaries below the cell, the boundary inside it), one column
// of 8 bytes per lane at cell stride 256 bytes from a 64 KiB base, so an
// entry's address is one byte permute; only the rows of finite rows' cells
// (64 .. 192) are stored, between the barriers and the X stages.

constexpr int kU2Rows = 128;
constexpr int kU2Stages = 3;               // X halves of 32 KB
constexpr int kU2Acc = 2;                  // accumulator pairs of 2 x 128 columns
constexpr int kU2Threads = 10 * 32;
constexpr int kU2HalfBytes = kU2Rows * 128 * 2;
constexpr uint32_t kU2HbAt = 2048;                                 // D0 H, D1 H (2 x 32 KB)
constexpr uint32_t kU2BarAt = kU2HbAt + 2 * 32768;                 // barriers, TMEM slot
constexpr uint32_t kU2SgnAt = kU2BarAt + 256;    // the sign masks s, then s2 (2 x 1 KB)
constexpr uint32_t kU2CellAt = kU2SgnAt + 2048;  // the table's cells, once each (2 KB)
constexpr uint32_t kU2RepAt = 65536;             // table row c at kU2RepAt + 256 c (rows 64 .. 192)
constexpr int kU2RowLo = 64, kU2RowHi = 192;
constexpr uint32_t kU2XsAt = 115712;             // X stages (1024-aligned), after the table's rows
constexpr uint32_t kU2End = kU2XsAt + kU2Stages * kU2HalfBytes;
static_assert(kU2XsAt % 1024 == 0, "swizzle atoms");
static_assert(kU2BarAt + (2 * kU2Stages + 2 * kU2Acc) * 8 + 16 <= kU2SgnAt, "layout");
static_assert(kU2CellAt + 8 * kRepCells <= kU2RepAt + 256u * kU2RowLo, "layout");
static_assert(kU2RepAt + 256u * (kU2RowHi + 1) <= kU2XsAt, "layout");
static_assert((kU2RepAt & 0xFF00u) == 0, "table base: cell byte free");
// a non-finite row's cell byte may name any row 0 .. 255: still inside the block's memory
static_assert(kU2RepAt >= kU2HbAt && kU2RepAt + 256u * 256u <= kU2End, "table rows in range");
static_assert(kU2End <= 232448, "shared memory");

// TS: the plan's second signs (two-sided), fixed per instantiation so that
// the per-element loop carries no test of it.
template <int BITS, bool TS>
__global__ void __launch_bounds__(kU2Threads, 1)
k_encode_umma256(const __grid_constant__ CUtensorMap xmap, int64_t n_rows, uint8_t* __restrict__ packed,
                 float* __restrict__ norms, int* status, const __grid_constant__ RowParams P) {
    constexpr int RB = 256 * BITS / 8, HB = RB / 2;  // bytes per row and per output half
    constexpr int NW = 128 * BITS / 32;              // packed words per output half
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t sbase = smem_addr(smem_raw);
    if (sbase > kU2HbAt) {  // the layout assumes dynamic memory starts lower
        if (threadIdx.x == 0) report_timeout(status, 67);
        return;
    }
    griddep_launch();
    auto at = [&](uint32_t a) { return smem_raw + (a - sbase); };
    unsigned char* xs = at(kU2XsAt);
    unsigned char* hb = at(kU2HbAt);
    uint64_t* full = reinterpret_cast<uint64_t*>(at(kU2BarAt));
    uint64_t* empty = full + kU2Stages;
    uint64_t* accf = empty + kU2Stages;
    uint64_t* acce = accf + kU2Acc;
    uint32_t* slot = reinterpret_cast<uint32_t*>(acce + kU2Acc);
    uint32_t* sg = reinterpret_cast<uint32_t*>(at(kU2SgnAt));
    const uint32_t* sg2 = sg + 256;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the sign masks, from the bit words of the parameter bank (indexed reads
    // of it with a different index per lane would be serialised)
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        sg[i] = sign_mask(P.sgnb, i);
        sg[256 + i] = sign_mask(P.sgn2b, i);
        reinterpret_cast<LutEntry*>(at(kU2CellAt))[i] = lut_cell(P.bnd, (1 << BITS) - 1, i - kRepCells / 2, kUmLutScale);
    }

    // Barriers first: the producer starts loading X while the other warps
    // build the operands and the table (a named barrier among warps 1-9).
    if (threadIdx.x == 0) {
        for (int i = 0; i < kU2Stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < kU2Acc; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], 4);
        }
        mbar_fence_init();
    }
    __syncthreads();
    uint32_t tmem = 0;
    if (warp > 0) {
        // B operands: D_p H, element (n, k) = (-1)^popcount(n & k) * s_{128 p + k},
        // each stored like a 128-byte-swizzled K-major tile of two 64-column
        // halves; 8 consecutive k per 16-byte store
        for (int i = threadIdx.x - 32; i < 2 * 128 * 16; i += blockDim.x - 32) {
            const int p = i >> 11, n = (i >> 4) & 127, k8 = i & 15;
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t h2 = 0;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 8 * k8 + 2 * j + e;
                    const bool neg = ((__popc(n & k) & 1) != 0) != (sg[128 * p + k] != 0u);
                    h2 |= (neg ? 0xBF80u : 0x3F80u) << (16 * e);
                }
                w[j] = h2;
            }
            const int off = p * 32768 + (k8 >> 3) * 16384 + n * 128 + (((k8 & 7) ^ (n & 7)) << 4);
            *reinterpret_cast<uint4*>(hb + off) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        // bucketing table: the cells of finite rows, replicated into 32
        // columns (consecutive threads write consecutive columns)
        const LutEntry* cells = reinterpret_cast<const LutEntry*>(at(kU2CellAt));
        for (int i = threadIdx.x - 32; i < (kU2RowHi - kU2RowLo + 1) * 32; i += blockDim.x - 32) {
            const int c = kU2RowLo + (i >> 5);
            *reinterpret_cast<LutEntry*>(at(kU2RepAt + 256u * c + 8u * (i & 31))) = cells[c];
        }
        fence_proxy_async_smem();  // the operands are read by the tensor cores
        if (warp == 1) tmem_alloc<kU2Acc * 256>(slot);
        tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"n"(kU2Threads - 32) : "memory");
        tc_fence_after();
        tmem = *slot;
    }
    // the prologue above reads the parameters only; the rows and the outputs
    // may belong to the previous kernel in the stream
    griddep_wait();
    const int64_t n_tiles = (n_rows + kU2Rows - 1) / kU2Rows;

    if (warp == 0) {  // ---- TMA producer: half h = 2 * (tile iteration) + p
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            int h = 0;
            for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
                for (int p = 0; p < 2; ++p, ++h) {
                    const int s = h % kU2Stages;
                    if (h >= kU2Stages && !mbar_wait(&empty[s], ((h / kU2Stages) - 1) & 1)) {
                        report_timeout(status, 61);
                        goto drain;
                    }
                    mbar_arrive_expect_tx(&full[s], kU2HalfBytes);
                    tma_load_2d(xs + s * kU2HalfBytes, &xmap, 128 * p, (int)(tile * kU2Rows), &full[s]);
                    tma_load_2d(xs + s * kU2HalfBytes + 16384, &xmap, 128 * p + 64, (int)(tile * kU2Rows), &full[s]);
                }
            }
        drain:
            for (int j = (h > kU2Stages ? h - kU2Stages : 0); j < h; ++j)
                if (!mbar_wait(&full[j % kU2Stages], (j / kU2Stages) & 1)) {
                    report_timeout(status, 62);
                    break;
                }
        }
    } else if (warp == 1) {  // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16(128, 128, true);
            const uint32_t xs_a = smem_addr(xs), hb_a = smem_addr(hb);
            int it = 0, h = 0;
            for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
                const int a = it % kU2Acc;
                if (it >= kU2Acc && !mbar_wait(&acce[a], ((it / kU2Acc) - 1) & 1)) {
                    report_timeout(status, 63);
                    break;
                }
                bool ok = true;
                for (int p = 0; p < 2; ++p, ++h) {
                    const int s = h % kU2Stages;
                    if (!mbar_wait(&full[s], (h / kU2Stages) & 1)) {
                        report_timeout(status, 64);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        umma_f16(tmem + a * 256 + p * 128, umma_desc_sw128(xs_a + s * kU2HalfBytes + off),
                                 umma_desc_sw128(hb_a + p * 32768 + off), idesc, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);
                }
                if (!ok) break;
                umma_commit(&accf[a]);
            }
            // the last accumulators must be complete before tensor memory is freed
            for (int j = (it > kU2Acc ? it - kU2Acc : 0); j < it; ++j)
                if (!mbar_wait(&accf[j % kU2Acc], (j / kU2Acc) & 1)) {
                    report_timeout(status, 65);
                    break;
                }
        }
    } else {  // ---- epilogue: warps 2-5 take even tiles, 6-9 odd tiles
        const int wg = (warp - 2) >> 2, q = warp & 3;
        const int r = 32 * q + lane;
        constexpr float kMagic = 12582912.0f + (float)(kRepCells / 2);
        const F2 M2 = f2(kMagic, kMagic);
        const uint32_t rep_slot = kU2RepAt + 8u * lane;
        int it = wg;
        for (int64_t tile = blockIdx.x + (int64_t)wg * gridDim.x; tile < n_tiles;
             tile += 2 * (int64_t)gridDim.x, it += 2) {
            const int a = it % kU2Acc;
            if (!mbar_wait(&accf[a], (it / kU2Acc) & 1)) {
                report_timeout(status, 66);
                break;
            }
            tc_fence_after();
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + a * 256;
            // The rare slow path below stays rolled over its chunks: with it
            // unrolled too, the code outgrows the instruction cache.
            F2 sa = f2(0.f, 0.f), sb = f2(0.f, 0.f);
            auto sumsq = [&](const uint32_t (&y)[32]) {
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const F2 p0 = f2(__uint_as_float(y[i]), __uint_as_float(y[i + 1]));
                    const F2 p1 = f2(__uint_as_float(y[i + 2]), __uint_as_float(y[i + 3]));
                    sa = f2_fma(p0, p0, sa);
                    sb = f2_fma(p1, p1, sb);
                }
            };
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // columns of A0 then A1
                uint32_t y[32];
                tmem_ld32(ta + 32 * c, y);
                tmem_wait_ld();
                sumsq(y);
            }
            float s0, s1, s2, s3;
            f2_split(sa, s0, s1);
            f2_split(sb, s2, s3);
            const float ss = 2.0f * ((s0 + s1) + (s2 + s3));  // = ||y||^2 = d ||x||^2
            float n = __fsqrt_rn(ss * (1.0f / 256.0f));
            float inv = ss > 0.f ? __frcp_rn(__fsqrt_rn(ss)) : 0.f;  // u = y * inv
            bool slow = false;  // a coordinate is not finite: binary search below
            const bool odd = !ss_in_range(ss);
            if (__any_sync(0xFFFFFFFFu, odd)) {
                // squares past fp32's range (or a zero or non-finite row): the
                // sums again on A S (rare; the tensor-memory loads are warp-wide)
                float m = 0.f;
                bool nf = false;
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t y[32];
                    tmem_ld32(ta + 32 * c, y);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float a = fabsf(__uint_as_float(y[i]));
                        nf = nf || !(a <= FLT_MAX);
                        m = fmaxf(m, a);
                    }
                }
                const float S = (odd && !nf && m > 0.f) ? pow2_scale(m) : 1.f;
                float t = 0.f;
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t y[32];
                    tmem_ld32(ta + 32 * c, y);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float a = __uint_as_float(y[i]) * S;
                        t = fmaf(a, a, t);
                    }
                }
                if (odd) {
                    if (nf) slow = true;
                    else if (m > 0.f) scaled_norm<256>(2.0f * t, S, n, inv);
                }
            }
            const float ks = inv * (float)kUmLutScale;
            const F2 K2 = f2(ks, ks);
            const int64_t row = tile * kU2Rows + r;
            const bool valid = row < n_rows;
            uint8_t* dst = packed + row * RB;
            // chunk c holds output dims 32c.. (low half) and 128 + 32c.. (high half):
            // 32 indices, CW words, per half
            constexpr int CW = BITS;
            auto put = [&](uint32_t (&w)[CW], int i, int id) {
                const int pos = i * BITS, wi = pos / 32, sh = pos % 32;
                w[wi] += (uint32_t)id << sh;
                if (sh + BITS > 32) w[wi + 1] += (uint32_t)id >> (32 - sh);
            };
            auto store = [&](int c, const uint32_t (&wl)[CW], const uint32_t (&wh)[CW]) {
                if (!valid) return;
                uint32_t* lo = reinterpret_cast<uint32_t*>(dst + 4 * BITS * c);
                uint32_t* hi = reinterpret_cast<uint32_t*>(dst + HB + 4 * BITS * c);
#pragma unroll
                for (int k = 0; k < CW; ++k) {
                    lo[k] = wl[k];
                    hi[k] = wh[k];
                }
            };
            auto halves = [&](const uint32_t (&a0)[32], const uint32_t (&a1)[32], int i, int c, float& ylo,
                              float& yhi) {
                ylo = __uint_as_float(a0[i]) + __uint_as_float(a1[i]);
                yhi = __uint_as_float(a0[i]) - __uint_as_float(a1[i]);
                if constexpr (TS) {
                    ylo = __uint_as_float(__float_as_uint(ylo) ^ sg2[32 * c + i]);
                    yhi = __uint_as_float(__float_as_uint(yhi) ^ sg2[128 + 32 * c + i]);
                }
            };
            // A chunk's packed words (CW per output half) leave as one vector
            // store per half where the width allows (16 bytes at 4 bits, 8 at 2):
            // 4-byte stores of 32 rows 128 bytes apart sent 8x the output
            // through the L1 write path.
            auto store_vec = [&](int c, const uint32_t (&wl)[CW], const uint32_t (&wh)[CW]) {
                if (!valid) return;
                uint8_t* lo = dst + 4 * BITS * c;
                uint8_t* hi = dst + HB + 4 * BITS * c;
                if constexpr (CW == 4) {
                    *reinterpret_cast<uint4*>(lo) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                    *reinterpret_cast<uint4*>(hi) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                } else if constexpr (CW == 2) {
                    *reinterpret_cast<uint2*>(lo) = make_uint2(wl[0], wl[1]);
                    *reinterpret_cast<uint2*>(hi) = make_uint2(wh[0], wh[1]);
                } else {
#pragma unroll
                    for (int k = 0; k < CW; ++k) {
                        reinterpret_cast<uint32_t*>(lo)[k] = wl[k];
                        reinterpret_cast<uint32_t*>(hi)[k] = wh[k];
                    }
                }
            };
            auto bucket_chunk = [&](const uint32_t (&a0)[32], const uint32_t (&a1)[32], int c) {
                uint32_t wl[CW], wh[CW];
#pragma unroll
                for (int k = 0; k < CW; ++k) wl[k] = wh[k] = 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float ylo, yhi;
                    halves(a0, a1, i, c, ylo, yhi);
                    float fx, fy;
                    f2_split(f2_fma(f2(ylo, yhi), K2, M2), fx, fy);
                    const uint32_t bx = __float_as_uint(fx), by = __float_as_uint(fy);
                    const LutEntry e0 = lds_entry(__byte_perm(bx, rep_slot, 0x7604));
                    const LutEntry e1 = lds_entry(__byte_perm(by, rep_slot, 0x7604));
                    put(wl, i, e0.lo + (fmaf(ylo, inv, -e0.thr) >= 0.0f ? 1 : 0));
                    put(wh, i, e1.lo + (fmaf(yhi, inv, -e1.thr) >= 0.0f ? 1 : 0));
                }
                store_vec(c, wl, wh);
            };
            // the common path rolled over the chunks (32 independent elements
            // each): unrolled, the code outgrew the instruction cache
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t a0[32], a1[32];
                tmem_ld32(ta + 32 * c, a0);
                tmem_ld32(ta + 128 + 32 * c, a1);
                tmem_wait_ld();
                bucket_chunk(a0, a1, c);
            }
            // rows with a NaN or infinite coordinate: exact binary search
            // over the boundaries, written over the fast path's bytes (the
            // tensor-memory loads are warp-wide); a finite row's cells are
            // 64 .. 192, all in the table
            if (__any_sync(0xFFFFFFFFu, slow)) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t a0[32], a1[32];
                    tmem_ld32(ta + 32 * c, a0);
                    tmem_ld32(ta + 128 + 32 * c, a1);
                    tmem_wait_ld();
                    if (slow) {
                        uint32_t wl[CW], wh[CW];
#pragma unroll
                        for (int k = 0; k < CW; ++k) wl[k] = wh[k] = 0;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float ylo, yhi;
                            halves(a0, a1, i, c, ylo, yhi);
                            put(wl, i, bucket_search<BITS>(P.bnd, ylo, inv));
                            put(wh, i, bucket_search<BITS>(P.bnd, yhi, inv));
                        }
                        store(c, wl, wh);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[a]);
            if (valid) norms[row] = n;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<kU2Acc * 256>(tmem);
    }
}

// ------------------------------------------------------- decode (v2)
//
// One row per thread, d <= 128: the next row's packed words and norm are
// loaded before the current row is transformed, so the load latency hides
// behind a row of arithmetic.  Centroids come from a 16-entry shared table
// (every entry in its own bank: conflict-free); field extraction produces the
// table's byte offsets directly.

template <int BITS, int D>
__device__ __forceinline__ void centroids_of(const uint32_t* w, const float (&cen)[16], float (&v)[D]) {
    const char* cb = reinterpret_cast<const char*>(cen);
    if constexpr (BITS == 4) {
#pragma unroll
        for (int k = 0; k < D / 8; ++k) {
            const uint32_t lo = (w[k] << 2) & 0x3C3C3C3Cu;  // fields 0,2,4,6 times 4
            const uint32_t hi = (w[k] >> 2) & 0x3C3C3C3Cu;  // fields 1,3,5,7 times 4
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * k + 2 * j] = *reinterpret_cast<const float*>(cb + __byte_perm(lo, 0, 0x4440 + j));
                v[8 * k + 2 * j + 1] = *reinterpret_cast<const float*>(cb + __byte_perm(hi, 0, 0x4440 + j));
            }
        }
    } else if constexpr (BITS == 2) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            const uint32_t m[4] = {(w[k] << 2) & 0x0C0C0C0Cu, w[k] & 0x0C0C0C0Cu,
                                   (w[k] >> 2) & 0x0C0C0C0Cu, (w[k] >> 4) & 0x0C0C0C0Cu};
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int f = 0; f < 4; ++f)
                    v[16 * k + 4 * j + f] = *reinterpret_cast<const float*>(cb + __byte_perm(m[f], 0, 0x4440 + j));
        }
    } else {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            const int pos = i * BITS, wi = pos / 32, sh = pos % 32;
            uint32_t x;
            if (sh + BITS <= 32) x = w[wi] >> sh;
            else x = __funnelshift_r(w[wi], w[wi + 1], sh);
            v[i] = *reinterpret_cast<const float*>(cb + ((x << 2) & 0x1Cu));
        }
    }
}

template <int D, int BITS, typename TO>
__global__ void __launch_bounds__(128, 3) k_decode2(const uint8_t* __restrict__ packed,
                                                 const float* __restrict__ norms, int64_t n_rows,
                                                 TO* __restrict__ y, const __grid_constant__ RowParams P) {
    __shared__ float cen_s[16];
    if (threadIdx.x < 16) cen_s[threadIdx.x] = P.cen[threadIdx.x];
    __syncthreads();
    constexpr int RB = D * BITS / 8, NW = RB / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // two rows in flight ahead of the one being transformed
    uint32_t wa[NW], wb[NW];
    float na = 0.f, nb = 0.f;
    if (row < n_rows) {
        load_bytes<RB>(packed + row * RB, wa);
        na = __ldg(norms + row);
    }
    if (row + stride < n_rows) {
        load_bytes<RB>(packed + (row + stride) * RB, wb);
        nb = __ldg(norms + row + stride);
    }
    for (; row < n_rows; row += stride) {
        uint32_t w[NW];
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            w[k] = wa[k];
            wa[k] = wb[k];
        }
        const float norm = na;
        na = nb;
        const int64_t nxt = row + 2 * stride;
        if (nxt < n_rows) {
            load_bytes<RB>(packed + nxt * RB, wb);
            nb = __ldg(norms + nxt);
        }
        float v[D];
        centroids_of<BITS, D>(w, cen_s, v);
        if (P.two_sided) flip_rotated<D>(v, 0, P.sgn2);
        fwht_reg2<D>(v);
        const float scs = norm * P.inv_sqrt_d;
        const F2 sc = f2(scs, scs);
        TO* out = y + row * D;
        if constexpr (sizeof(TO) == 4) {
#pragma unroll
            for (int k = 0; k < D; k += 4) {
                float ax, ay, bx, by;
                f2_split(f2_mul(f2(v[k], v[k + 1]), sc), ax, ay);
                f2_split(f2_mul(f2(v[k + 2], v[k + 3]), sc), bx, by);
                float4 o;
                o.x = __uint_as_float(__float_as_uint(ax) ^ P.sgn[k]);
                o.y = __uint_as_float(__float_as_uint(ay) ^ P.sgn[k + 1]);
                o.z = __uint_as_float(__float_as_uint(bx) ^ P.sgn[k + 2]);
                o.w = __uint_as_float(__float_as_uint(by) ^ P.sgn[k + 3]);
                reinterpret_cast<float4*>(out)[k / 4] = o;
            }
        } else {
#pragma unroll
            for (int k = 0; k < D; k += 8) {
                uint32_t q[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float ax, ay;
                    f2_split(f2_mul(f2(v[k + 2 * m], v[k + 2 * m + 1]), sc), ax, ay);
                    __nv_bfloat162 h = __floats2bfloat162_rn(ax, ay);
                    q[m] = *reinterpret_cast<uint32_t*>(&h) ^ ((P.sgn[k + 2 * m] >> 16) | P.sgn[k + 2 * m + 1]);
                }
                reinterpret_cast<uint4*>(out)[k / 8] = make_uint4(q[0], q[1], q[2], q[3]);
            }
        }
    }
}

// --------------------------------------------- decode to bf16, d = 128 (v3)
//
// As k_decode2, with the output staged per warp: 32 rows of bf16 (8 KB) are
// written thread-per-row into a 128-byte-swizzled shared buffer (conflict
// free) and leave as two 2-D TMA stores, so global writes are whole lines.
// Two buffers per warp; the packed rows of the next warp tile are loaded
// before the current one is transformed.

constexpr int kDec3Warps = 4;
constexpr int kDec3Smem = kDec3Warps * 2 * 8192 + 1024;

template <int BITS>
__global__ void __launch_bounds__(32 * kDec3Warps, 3)
k_decode3(const uint8_t* __restrict__ packed, const float* __restrict__ norms, int64_t n_rows,
          const __grid_constant__ CUtensorMap ymap, const __grid_constant__ RowParams P) {
    constexpr int D = 128, RB = D * BITS / 8, NW = RB / 4;
    __shared__ float cen_s[16];
    extern __shared__ __align__(1024) unsigned char dsm[];
    unsigned char* base = dsm + ((1024u - (smem_addr(dsm) & 1023u)) & 1023u);
    griddep_launch();
    if (threadIdx.x < 16) cen_s[threadIdx.x] = P.cen[threadIdx.x];
    __syncthreads();
    griddep_wait();  // the packed rows and the output may belong to the previous kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* buf = base + warp * 2 * 8192;
    const int64_t n_tiles = (n_rows + 31) / 32;
    const int64_t wstride = (int64_t)gridDim.x * kDec3Warps;
    int64_t tile = (int64_t)blockIdx.x * kDec3Warps + warp;
    uint32_t wn[NW];
    float nn = 0.f;
    auto fetch = [&](int64_t tl) {
        const int64_t row = tl * 32 + lane;
        if (tl < n_tiles && row < n_rows) {
            load_bytes<RB>(packed + row * RB, wn);
            nn = __ldg(norms + row);
        } else {
#pragma unroll
            for (int k = 0; k < NW; ++k) wn[k] = 0;
            nn = 0.f;
        }
    };
    fetch(tile);
    int it = 0;
    for (; tile < n_tiles; tile += wstride, ++it) {
        uint32_t w[NW];
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] = wn[k];
        const float norm = nn;
        fetch(tile + wstride);
        float v[D];
        centroids_of<BITS, D>(w, cen_s, v);
        if (P.two_sided) flip_rotated<D>(v, 0, P.sgn2);
        fwht_reg2<D>(v);
        const float scs = norm * P.inv_sqrt_d;
        const F2 sc = f2(scs, scs);
        unsigned char* b = buf + (it & 1) * 8192;
        // the store that last read this buffer (two tiles ago) must be done
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 16; ++c) {  // 16-byte chunk c = columns 8c .. 8c+7
            uint32_t q[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int k = 8 * c + 2 * m;
                float ax, ay;
                f2_split(f2_mul(f2(v[k], v[k + 1]), sc), ax, ay);
                __nv_bfloat162 h = __floats2bfloat162_rn(ax, ay);
                q[m] = *reinterpret_cast<uint32_t*>(&h) ^ ((P.sgn[k] >> 16) | P.sgn[k + 1]);
            }
            const int half = c >> 3, cc = c & 7;
            *reinterpret_cast<uint4*>(b + half * 4096 + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                make_uint4(q[0], q[1], q[2], q[3]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(&ymap, 0, (int)(tile * 32), b);
            tma_store_2d(&ymap, 64, (int)(tile * 32), b + 4096);
            bulk_commit();
        }
    }
    if (lane == 0) bulk_wait<0>();
}

// d = 256 with bf16 output: as k_decode3, two threads per row (lanes 2j and
// 2j + 1 hold the row's two "split" parts, see RowShape), so a warp tile is
// 16 rows; the transform ends with the cross-thread stage, leaving part p
// with output dims 128p .. 128p + 127.  The tile (16 rows of 512 B) is staged
// as four 128-byte-swizzled 64-column blocks and leaves as four 2-D TMA
// stores.
constexpr int kDec3bWarps = 4;
constexpr int kDec3bSmem = kDec3bWarps * 2 * 8192 + 1024;

template <int BITS>
__global__ void __launch_bounds__(32 * kDec3bWarps, 2)
k_decode3_256(const uint8_t* __restrict__ packed, const float* __restrict__ norms, int64_t n_rows,
              const __grid_constant__ CUtensorMap ymap, const __grid_constant__ RowParams P) {
    constexpr int D = 256, E = 128, RB = D * BITS / 8, HB = E / 2 * BITS / 8, NW = E * BITS / 32;
    __shared__ float cen_s[16];
    // the output pairs' sign masks of part p at sgh_s[65 p ..]: the lanes of
    // the two parts read different banks (a lane-varying index into the
    // parameter bank would be serialised)
    __shared__ uint32_t sgh_s[2 * 65];
    extern __shared__ __align__(1024) unsigned char dsm[];
    unsigned char* base = dsm + ((1024u - (smem_addr(dsm) & 1023u)) & 1023u);
    griddep_launch();
    if (threadIdx.x < 16) cen_s[threadIdx.x] = P.cen[threadIdx.x];
    if (threadIdx.x < 128) sgh_s[threadIdx.x + (threadIdx.x >> 6)] = P.sgnh[threadIdx.x];
    __syncthreads();
    griddep_wait();  // the packed rows and the output may belong to the previous kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rr = lane >> 1, p = lane & 1;  // row of the tile, part of the row
    unsigned char* buf = base + warp * 2 * 8192;
    const int64_t n_tiles = (n_rows + 15) / 16;
    const int64_t wstride = (int64_t)gridDim.x * kDec3bWarps;
    int64_t tile = (int64_t)blockIdx.x * kDec3bWarps + warp;
    uint32_t wn[NW];
    float nn = 0.f;
    auto fetch = [&](int64_t tl) {
        const int64_t row = tl * 16 + rr;
        if (tl < n_tiles && row < n_rows) {
            const uint8_t* src = packed + row * RB;
            load_bytes<HB>(src + p * HB, wn);
            load_bytes<HB>(src + 2 * HB + p * HB, wn + HB / 4);
            nn = __ldg(norms + row);
        } else {
#pragma unroll
            for (int k = 0; k < NW; ++k) wn[k] = 0;
            nn = 0.f;
        }
    };
    fetch(tile);
    int it = 0;
    for (; tile < n_tiles; tile += wstride, ++it) {
        uint32_t w[NW];
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] = wn[k];
        const float norm = nn;
        fetch(tile + wstride);
        float v[E];
        centroids_of<BITS, E>(w, cen_s, v);
        if (P.two_sided) flip_rotated<D>(v, p, P.sgn2);
        fwht_reg2<E>(v);
        fwht_cross<E>(v, p);  // split -> contiguous: dims 128p + j
        const float scs = norm * P.inv_sqrt_d;
        const F2 sc = f2(scs, scs);
        const uint32_t* sgh = sgh_s + 65 * p;
        unsigned char* b = buf + (it & 1) * 8192;
        // the stores that last read this buffer (two tiles ago) must be done
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 16; ++c) {  // 16-byte chunk c = dims 128p + 8c .. + 7
            uint32_t q[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int k = 8 * c + 2 * m;
                float ax, ay;
                f2_split(f2_mul(f2(v[k], v[k + 1]), sc), ax, ay);
                __nv_bfloat162 h = __floats2bfloat162_rn(ax, ay);
                q[m] = *reinterpret_cast<uint32_t*>(&h) ^ sgh[k >> 1];
            }
            const int blk = 2 * p + (c >> 3), cc = c & 7;
            *reinterpret_cast<uint4*>(b + blk * 2048 + rr * 128 + ((cc ^ (rr & 7)) << 4)) =
                make_uint4(q[0], q[1], q[2], q[3]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) tma_store_2d(&ymap, 64 * blk, (int)(tile * 16), b + blk * 2048);
            bulk_commit();
        }
    }
    if (lane == 0) bulk_wait<0>();
}

}  // namespace dev

// ---------------------------------------------------------------- launchers

namespace {

template <int D, int BITS>
cudaError_t enc_tma(const void* x, int64_t n, uint8_t* pk, float* nm, const RowParams& P, cudaStream_t s) {
    using Sh = dev::TmaEncodeShape<D>;
    CUtensorMap map;
    cudaError_t e = make_rows_map(&map, x, 2, D, (uint64_t)n, dev::kTmaRows);
    if (e != cudaSuccess) return e;
    auto fn = dev::k_encode_tma<D, BITS>;
    static int attr_dev_mask = 0;  // devices on which the smem opt-in was set
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 31 && !(attr_dev_mask & (1 << dev))) {
        e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_dev_mask |= 1 << dev;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void*)fn, dev::kTmaThreads, Sh::kSmemBytes) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int64_t tiles = (n + dev::kTmaRows - 1) / dev::kTmaRows;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > tiles) grid = tiles;
    fn<<<(unsigned)grid, dev::kTmaThreads, Sh::kSmemBytes, s>>>(map, n, pk, nm, status_word(), P);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t enc_umma(const void* x, int64_t n, uint8_t* pk, float* nm, const RowParams& P, cudaStream_t s) {
    CUtensorMap map;
    cudaError_t e = make_rows_map(&map, x, 2, 128, (uint64_t)n, dev::kUmRows);
    if (e != cudaSuccess) return e;
    auto fn = dev::k_encode_umma<BITS>;
    // absolute layout: ask for kUmEnd bytes (the dynamic block starts below kUmHbAt)
    e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev::kUmEnd);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (n + dev::kUmRows - 1) / dev::kUmRows;
    int64_t grid = num_sms();
    if (grid > tiles) grid = tiles;
    return dev::launch_pdl(fn, dim3((unsigned)grid), dim3(dev::kUmThreads), dev::kUmEnd, s, map, n, pk, nm,
                           status_word(), P);
}

template <int BITS>
cudaError_t enc_umma256(const void* x, int64_t n, uint8_t* pk, float* nm, const RowParams& P, cudaStream_t s) {
    CUtensorMap map;
    cudaError_t e = make_rows_map(&map, x, 2, 256, (uint64_t)n, dev::kU2Rows);
    if (e != cudaSuccess) return e;
    auto fn = P.two_sided ? dev::k_encode_umma256<BITS, true> : dev::k_encode_umma256<BITS, false>;
    // absolute layout: ask for kU2End bytes (the dynamic block starts below kU2HbAt)
    e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev::kU2End);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (n + dev::kU2Rows - 1) / dev::kU2Rows;
    int64_t grid = num_sms();
    if (grid > tiles) grid = tiles;
    return dev::launch_pdl(fn, dim3((unsigned)grid), dim3(dev::kU2Threads), dev::kU2End, s, map, n, pk, nm,
                           status_word(), P);
}

template <int D, int BITS, typename T>
cudaError_t enc(const void* x, int64_t n, uint8_t* pk, float* nm, const RowParams& P, cudaStream_t s) {
    // d = 128 and 256 bf16: the transform on the tensor cores; d = 64 bf16:
    // TMA-fed CUDA-core butterflies; other shapes: one thread per row (two at d = 256)
    if constexpr (D == 128 && sizeof(T) == 2) {
        return enc_umma<BITS>(x, n, pk, nm, P, s);
    } else if constexpr (D == 256 && sizeof(T) == 2) {
        return enc_umma256<BITS>(x, n, pk, nm, P, s);
    } else if constexpr (D == 64 && sizeof(T) == 2) {
        return enc_tma<D, BITS>(x, n, pk, nm, P, s);
    } else {
        auto fn = dev::k_encode<D, BITS, T>;
        unsigned g = grid_for((const void*)fn, dev::kBlock, n * dev::RowShape<D>::R);
        fn<<<g, dev::kBlock, 0, s>>>(static_cast<const T*>(x), n, pk, nm, P);
        return cudaGetLastError();
    }
}

template <int BITS>
cudaError_t dec3(const uint8_t* pk, const float* nm, int64_t n, void* y, const RowParams& P, cudaStream_t s) {
    CUtensorMap map;
    cudaError_t e = make_rows_map(&map, y, 2, 128, (uint64_t)n, 32);
    if (e != cudaSuccess) return e;
    auto fn = dev::k_decode3<BITS>;
    e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dev::kDec3Smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void*)fn, 32 * dev::kDec3Warps, dev::kDec3Smem) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int64_t warp_tiles = (n + 31) / 32;
    int64_t grid = (int64_t)num_sms() * per_sm;
    const int64_t need = (warp_tiles + dev::kDec3Warps - 1) / dev::kDec3Warps;
    if (grid > need) grid = need;
    return dev::launch_pdl(fn, dim3((unsigned)grid), dim3(32 * dev::kDec3Warps), dev::kDec3Smem, s, pk, nm, n, map,
                           P);
}

template <int BITS>
cudaError_t dec3_256(const uint8_t* pk, const float* nm, int64_t n, void* y, const RowParams& P, cudaStream_t s) {
    CUtensorMap map;
    cudaError_t e = make_rows_map(&map, y, 2, 256, (uint64_t)n, 16);
    if (e != cudaSuccess) return e;
    auto fn = dev::k_decode3_256<BITS>;
    e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dev::kDec3bSmem);
    if (e != cudaSuccess) return e;
    const int per_sm = blocks_per_sm((const void*)fn, 32 * dev::kDec3bWarps, dev::kDec3bSmem);
    const int64_t warp_tiles = (n + 15) / 16;
    int64_t grid = (int64_t)num_sms() * per_sm;
    const int64_t need = (warp_tiles + dev::kDec3bWarps - 1) / dev::kDec3bWarps;
    if (grid > need) grid = need;
    return dev::launch_pdl(fn, dim3((unsigned)grid), dim3(32 * dev::kDec3bWarps), dev::kDec3bSmem, s, pk, nm, n, map,
                           P);
}

template <int D, int BITS, typename TO>
cudaError_t dec(const uint8_t* pk, const float* nm, int64_t n, void* y, const RowParams& P, cudaStream_t s) {
    if constexpr (D == 128 && sizeof(TO) == 2) return dec3<BITS>(pk, nm, n, y, P, s);
    if constexpr (D == 256 && sizeof(TO) == 2) return dec3_256<BITS>(pk, nm, n, y, P, s);
    if constexpr (D == 64 || D == 128) {
        auto fn2 = dev::k_decode2<D, BITS, TO>;
        unsigned g = grid_for((const void*)fn2, 128, n);
        fn2<<<g, 128, 0, s>>>(pk, nm, n, static_cast<TO*>(y), P);
        return cudaGetLastError();
    }
    auto fn = dev::k_decode<D, BITS, TO>;
    unsigned g = grid_for((const void*)fn, dev::kBlock, n * dev::RowShape<D>::R);
    fn<<<g, dev::kBlock, 0, s>>>(pk, nm, n, static_cast<TO*>(y), P);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t app(const void* kn, const void* vn, int B, int Hkv, int64_t n_new, const tq_cache_view& c,
                int64_t pos, int kb, int vb, const RowParams& PK, const RowParams& PV, cudaStream_t s) {
    const int64_t rows = (int64_t)B * Hkv * n_new;
    if constexpr (D >= 32) {
        auto fn = dev::k_append_warp<D, T, false>;
        int64_t g = (rows + dev::kAppWarps - 1) / dev::kAppWarps;
        const int64_t cap = (int64_t)num_sms() * blocks_per_sm((const void*)fn, 32 * dev::kAppWarps, 0);
        if (g > cap) g = cap;
        return dev::launch_pdl(fn, dim3((unsigned)g, 2), dim3(32 * dev::kAppWarps), 0, s, static_cast<const T*>(kn),
                               static_cast<const T*>(vn), rows, n_new, c, pos, kb, vb, PK, PV, PagedArgs{}, Hkv,
                               (int*)nullptr);
    } else {
        auto fn = dev::k_append<D, T>;
        unsigned g = grid_for((const void*)fn, dev::kBlock, rows * dev::RowShape<D>::R);
        fn<<<dim3(g, 2), dev::kBlock, 0, s>>>(static_cast<const T*>(kn), static_cast<const T*>(vn), rows,
                                              n_new, c, pos, kb, vb, PK, PV);
    }
    return cudaGetLastError();
}

template <int D, int BITS>
cudaError_t enc_dt(tq_dtype dt, const void* x, int64_t n, uint8_t* pk, float* nm, const RowParams& P,
                   cudaStream_t s) {
    return dt == TQ_BF16 ? enc<D, BITS, __nv_bfloat16>(x, n, pk, nm, P, s)
                         : enc<D, BITS, float>(x, n, pk, nm, P, s);
}

template <int D, int BITS>
cudaError_t dec_dt(tq_dtype dt, const uint8_t* pk, const float* nm, int64_t n, void* y,
                   const RowParams& P, cudaStream_t s) {
    return dt == TQ_BF16 ? dec<D, BITS, __nv_bfloat16>(pk, nm, n, y, P, s)
                         : dec<D, BITS, float>(pk, nm, n, y, P, s);
}

}  // namespace

template <int D>
cudaError_t launch_encode_d(int bits, tq_dtype dt, const void* x, int64_t n_rows, uint8_t* packed,
                            float* norms, const RowParams& P, cudaStream_t s) {
    switch (bits) {
        case 2: return enc_dt<D, 2>(dt, x, n_rows, packed, norms, P, s);
        case 3: return enc_dt<D, 3>(dt, x, n_rows, packed, norms, P, s);
        default: return enc_dt<D, 4>(dt, x, n_rows, packed, norms, P, s);
    }
}

template <int D>
cudaError_t launch_decode_d(int bits, tq_dtype dt, const uint8_t* packed, const float* norms,
                            int64_t n_rows, void* y, const RowParams& P, cudaStream_t s) {
    switch (bits) {
        case 2: return dec_dt<D, 2>(dt, packed, norms, n_rows, y, P, s);
        case 3: return dec_dt<D, 3>(dt, packed, norms, n_rows, y, P, s);
        default: return dec_dt<D, 4>(dt, packed, norms, n_rows, y, P, s);
    }
}

template <int D>
cudaError_t launch_append_d(int k_bits, int v_bits, tq_dtype dt, const void* k_new,
                            const void* v_new, int B, int Hkv, int64_t n_new,
                            const tq_cache_view& cache, int64_t pos, const RowParams& PK,
                            const RowParams& PV, cudaStream_t s) {
    return dt == TQ_BF16
               ? app<D, __nv_bfloat16>(k_new, v_new, B, Hkv, n_new, cache, pos, k_bits, v_bits, PK, PV, s)
               : app<D, float>(k_new, v_new, B, Hkv, n_new, cache, pos, k_bits, v_bits, PK, PV, s);
}

template <int D>
cudaError_t launch_append_paged_d(int k_bits, int v_bits, tq_dtype dt, const void* k_new,
                                  const void* v_new, int B, int Hkv, const tq_cache_view& pages,
                                  const PagedArgs& pa, const RowParams& PK, const RowParams& PV,
                                  cudaStream_t s) {
    if constexpr (D >= 32) {
        const int64_t rows = (int64_t)B * Hkv;
        auto launch = [&](auto tag) {
            using T = decltype(tag);
            auto fn = dev::k_append_warp<D, T, true>;
            int64_t g = (rows + dev::kAppWarps - 1) / dev::kAppWarps;
            const int64_t cap = (int64_t)num_sms() * blocks_per_sm((const void*)fn, 32 * dev::kAppWarps, 0);
            if (g > cap) g = cap;
            return dev::launch_pdl(fn, dim3((unsigned)g, 2), dim3(32 * dev::kAppWarps), 0, s,
                                   static_cast<const T*>(k_new), static_cast<const T*>(v_new), rows, (int64_t)1,
                                   pages, (int64_t)0, k_bits, v_bits, PK, PV, pa, Hkv, status_word());
        };
        return dt == TQ_BF16 ? launch(__nv_bfloat16{}) : launch(float{});
    } else {
        return cudaErrorInvalidValue;
    }
}

#ifndef TQ_UNIT_D
#error "compile once per head dimension with -DTQ_UNIT_D=<d>"
#endif
template cudaError_t launch_encode_d<TQ_UNIT_D>(int, tq_dtype, const void*, int64_t, uint8_t*, float*,
                                                const RowParams&, cudaStream_t);
template cudaError_t launch_decode_d<TQ_UNIT_D>(int, tq_dtype, const uint8_t*, const float*, int64_t,
                                                void*, const RowParams&, cudaStream_t);
template cudaError_t launch_append_paged_d<TQ_UNIT_D>(int, int, tq_dtype, const void*, const void*, int, int,
                                                      const tq_cache_view&, const PagedArgs&,
                                                      const RowParams&, const RowParams&, cudaStream_t);
template cudaError_t launch_append_d<TQ_UNIT_D>(int, int, tq_dtype, const void*, const void*, int, int,
                                                int64_t, const tq_cache_view&, int64_t,
                                                const RowParams&, const RowParams&, cudaStream_t);

}  // namespace tq
