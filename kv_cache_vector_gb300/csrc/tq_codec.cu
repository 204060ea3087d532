// tq_codec.cu -- sm_103a kernels of the row codec: encode, decode, append.
//
// Encode ("TurboQuant KV Cache Compression -- Spec", Steps 1-3 and As-Built
// Notes 1-2):  load row -> sign flip (xor of the fp32 sign bit) -> FWHT in
// registers -> norm -> bucket through an exact lookup table -> dense LSB-first
// pack -> store.  Decode reverses it: unpack -> centroid -> FWHT -> scale by
// norm / sqrt(d) -> sign -> store.  Rows are independent ("TurboQuantEngine --
// Specification", 7 Non-goals: each row encoded independently), so the grid
// simply strides over rows.
#include "tq_device.cuh"

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
    const float n = __fsqrt_rn(ss);
    // w = y * inv is the normalised coordinate u = (H s x / sqrt(d)) / n
    const float inv = n > 0.f ? __fdiv_rn(P.inv_sqrt_d, n) : 0.f;
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

// ---------------------------------------------------------------- launchers

namespace {

template <int D, int BITS, typename T>
cudaError_t enc(const void* x, int64_t n, uint8_t* pk, float* nm, const RowParams& P, cudaStream_t s) {
    auto fn = dev::k_encode<D, BITS, T>;
    unsigned g = grid_for((const void*)fn, dev::kBlock, n * dev::RowShape<D>::R);
    fn<<<g, dev::kBlock, 0, s>>>(static_cast<const T*>(x), n, pk, nm, P);
    return cudaGetLastError();
}

template <int D, int BITS, typename TO>
cudaError_t dec(const uint8_t* pk, const float* nm, int64_t n, void* y, const RowParams& P, cudaStream_t s) {
    auto fn = dev::k_decode<D, BITS, TO>;
    unsigned g = grid_for((const void*)fn, dev::kBlock, n * dev::RowShape<D>::R);
    fn<<<g, dev::kBlock, 0, s>>>(pk, nm, n, static_cast<TO*>(y), P);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t app(const void* kn, const void* vn, int B, int Hkv, int64_t n_new, const tq_cache_view& c,
                int64_t pos, int kb, int vb, const RowParams& PK, const RowParams& PV, cudaStream_t s) {
    auto fn = dev::k_append<D, T>;
    const int64_t rows = (int64_t)B * Hkv * n_new;
    unsigned g = grid_for((const void*)fn, dev::kBlock, rows * dev::RowShape<D>::R);
    fn<<<dim3(g, 2), dev::kBlock, 0, s>>>(static_cast<const T*>(kn), static_cast<const T*>(vn), rows,
                                          n_new, c, pos, kb, vb, PK, PV);
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

#ifndef TQ_UNIT_D
#error "compile once per head dimension with -DTQ_UNIT_D=<d>"
#endif
template cudaError_t launch_encode_d<TQ_UNIT_D>(int, tq_dtype, const void*, int64_t, uint8_t*, float*,
                                                const RowParams&, cudaStream_t);
template cudaError_t launch_decode_d<TQ_UNIT_D>(int, tq_dtype, const uint8_t*, const float*, int64_t,
                                                void*, const RowParams&, cudaStream_t);
template cudaError_t launch_append_d<TQ_UNIT_D>(int, int, tq_dtype, const void*, const void*, int, int,
                                                int64_t, const tq_cache_view&, int64_t,
                                                const RowParams&, const RowParams&, cudaStream_t);

}  // namespace tq
