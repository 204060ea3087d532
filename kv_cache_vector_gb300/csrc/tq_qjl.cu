// tq_qjl.cu -- QJL residual keys: the Gaussian projection, encode and decode.
//
// "CITATIONS" (Atlas), Google TurboQuant entry: an MSE-optimal quantiser
// followed by a 1-bit quantised Johnson-Lindenstrauss transform of the
// residual makes inner products unbiased ("TurboQuant KV Cache Compression --
// Spec", Why not QJL?).  The pages give no formula; the format implemented
// here, for b bits per coordinate:
//   * the first b - 1 bits are the row codec's index on the (b - 1)-bit
//     codebook (the same rotation, norm and bucketing);
//   * r = u - c[idx] is the residual of the rotated normalised row u; its
//     projections p = S r by a d x d matrix S of i.i.d. N(0, 1) entries give
//     one sign bit each (bit k = 1 iff p_k >= 0), packed after the indices:
//     d * b / 8 bytes per row;
//   * gamma = n ||r|| (fp32) is stored beside the norm n;
//   * decode, in the rotated domain: n c[idx] + sqrt(pi/2)/d * gamma * S^T sgn
//     (sgn_k = +-1), then the inverse rotation.  E[sign(s.r) s] =
//     sqrt(2/pi) r / ||r|| for a standard Gaussian row s, so the correction
//     has expectation n r over S and <y, x_hat> is unbiased.
// S is drawn from the plan seed's splitmix64 stream (Vigna's published
// generator), after the 2d outputs of the sign vectors: entry k = i d + j is
// Box-Muller, sqrt(-2 ln(1 - U1)) cos(2 pi U2), on outputs 2d + 2k and
// 2d + 2k + 1, U = (out >> 11) / 2^53, computed in double and stored fp32.
//
// d = 128 runs the projections on the tensor cores (k_encode_qjl_tc,
// k_decode_qjl_tc, below).  CUDA-core work layout (d = 32, 64): a warp takes
// four rows at a time; lane l holds the E = d/32 coordinates l E .. l E + E -
// 1 through the transform and the projections k = l + 32 e, so that the sign
// bits of projection word e are one warp ballot.  The block keeps S in shared
// memory, row-major with a stride of d + 4 floats: lane reads of four
// consecutive floats of 32 different rows (encode) and of one row (decode)
// are both free of bank conflicts.  Each S load feeds the four rows of the
// warp.  Blocks of 12 warps.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_async.cuh"
#include "tq_device.cuh"

namespace tq {
namespace dev {

// Tuning parameters: warps per block, and rows per warp at a time (each S
// load feeds that many rows).
#ifndef TQ_QJL_WARPS
#define TQ_QJL_WARPS 12
#endif
constexpr int kQjlWarps = TQ_QJL_WARPS;
#ifndef TQ_QJL_ROWS
#define TQ_QJL_ROWS 4
#endif
constexpr int kQjlRows = TQ_QJL_ROWS;

template <int D>
struct QjlSmem {
    static constexpr int kStride = D + 4;                       // floats per row of S
    static constexpr int kS = D * kStride * 4;                  // bytes of S
    static constexpr int kR = kQjlWarps * kQjlRows * D * 4;     // residuals (encode) / rows (decode)
    static constexpr int kI = kQjlWarps * kQjlRows * D;         // index bytes (encode)
    static constexpr int kBytes = kS + kR + kI + 2 * D * 4;     // + sign masks
};

#if TQ_UNIT_D == 128  // the matrix kernel is built once
// Output i (0-based) of splitmix64 seeded with `seed`: the state after i + 1
// increments of the golden-ratio constant, through the published mix.
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void __launch_bounds__(256) k_qjl_matrix(uint64_t seed, int d, float* __restrict__ S) {
    const int64_t n = (int64_t)d * d;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t o = 2 * (uint64_t)d + 2 * (uint64_t)k;
        const double u1 = (double)(splitmix64_at(seed, o) >> 11) * 0x1p-53;
        const double u2 = (double)(splitmix64_at(seed, o + 1) >> 11) * 0x1p-53;
        S[k] = (float)(sqrt(-2.0 * log(1.0 - u1)) * cos(6.283185307179586 * u2));
    }
}
#endif

// Copy S [D][D] (global, row-major) into shared memory with row stride D + 4.
template <int D>
__device__ __forceinline__ void stage_matrix(const float* __restrict__ S, float* Ss) {
    constexpr int kStride = QjlSmem<D>::kStride;
    for (int i = threadIdx.x; i < D * D / 4; i += blockDim.x) {
        const int k = (4 * i) / D, j = (4 * i) % D;
        *reinterpret_cast<float4*>(Ss + k * kStride + j) = __ldg(reinterpret_cast<const float4*>(S) + i);
    }
}

// The in-warp transform: the E registers of each lane, then across lanes
// (element e of lane l is coordinate l E + e), unnormalised.
template <int E>
__device__ __forceinline__ void warp_fwht(float (&v)[E], int lane) {
    fwht_reg<E>(v);
#pragma unroll
    for (int b = 1; b < 32; b <<= 1) {
        const float sgn = (lane & b) ? -1.f : 1.f;  // (lo + hi, lo - hi) = o + (+-1) v, one rounding
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v[e], b);
            v[e] = fmaf(sgn, v[e], o);
        }
    }
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    return s;
}

// Encode: BITS total bits per coordinate (2..4), T the input type.  P holds
// the (BITS - 1)-bit codebook.
template <int D, int BITS, typename T>
__global__ void __launch_bounds__(32 * kQjlWarps) k_encode_qjl(const T* __restrict__ x, int64_t n_rows,
                                                               const float* __restrict__ S,
                                                               uint8_t* __restrict__ packed,
                                                               float* __restrict__ norms, float* __restrict__ rnorms,
                                                               const __grid_constant__ RowParams P) {
    constexpr int E = D / 32, MB = BITS - 1, NB = (1 << MB) - 1;
    constexpr int RB = D * BITS / 8, IB = D * MB / 8;
    constexpr int kStride = QjlSmem<D>::kStride;
    extern __shared__ __align__(16) unsigned char qjl_smem[];
    float* Ss = reinterpret_cast<float*>(qjl_smem);
    float* rbuf = reinterpret_cast<float*>(qjl_smem + QjlSmem<D>::kS);
    uint8_t* ibuf = qjl_smem + QjlSmem<D>::kS + QjlSmem<D>::kR;
    uint32_t* sg = reinterpret_cast<uint32_t*>(ibuf + QjlSmem<D>::kI);
    uint32_t* sg2 = sg + D;
    __shared__ float cen_s[16];  // centroids by lane-varying index: shared memory, not the parameter bank
    stage_matrix<D>(S, Ss);
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
        sg[i] = sign_mask(P.sgnb, i);
        sg2[i] = sign_mask(P.sgn2b, i);
    }
    if (threadIdx.x < 16) cen_s[threadIdx.x] = P.cen[threadIdx.x];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* rw = rbuf + warp * kQjlRows * D;
    uint8_t* iw = ibuf + warp * kQjlRows * D;
    for (int64_t r0 = ((int64_t)blockIdx.x * kQjlWarps + warp) * kQjlRows; r0 < n_rows;
         r0 += (int64_t)gridDim.x * kQjlWarps * kQjlRows) {
        float nrm[kQjlRows], gam[kQjlRows];
        // the rows' loads first, all in flight (rows past the end: zeros)
        float vq[kQjlRows][E];
#pragma unroll
        for (int q = 0; q < kQjlRows; ++q) {
            if (r0 + q < n_rows) {
                load_lane<E, T>(x + (r0 + q) * D, lane, sg, vq[q]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) vq[q][e] = 0.f;
            }
        }
        // ---- MSE stage and residual of each row
#pragma unroll
        for (int q = 0; q < kQjlRows; ++q) {
            float(&v)[E] = vq[q];
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
            ss = warp_sum(ss);
            warp_fwht<E>(v, lane);
            if (P.two_sided) {
#pragma unroll
                for (int e = 0; e < E; ++e) v[e] = __uint_as_float(__float_as_uint(v[e]) ^ sg2[lane * E + e]);
            }
            float n = __fsqrt_rn(ss);
            float inv = n > 0.f ? __fdiv_rn(P.inv_sqrt_d, n) : 0.f;
            if (!ss_in_range(ss)) warp_rescaled_norm<D, E>(v, n, inv);  // squares past fp32's range
            float rr = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                int id = 0;
#pragma unroll
                for (int j = 0; j < NB; ++j) id += fmaf(v[e], inv, -P.bnd[j]) >= 0.0f ? 1 : 0;
                const float r = fmaf(v[e], inv, -cen_s[id]);
                rr = fmaf(r, r, rr);
                iw[q * D + lane * E + e] = (uint8_t)id;
                rw[q * D + lane * E + e] = r;
            }
            rr = warp_sum(rr);
            nrm[q] = n;
            gam[q] = n * __fsqrt_rn(rr);
        }
        __syncwarp();
        // ---- projections p_k = sum_j S[k][j] r_j, k = lane + 32 e
        float acc[kQjlRows][E];
#pragma unroll
        for (int q = 0; q < kQjlRows; ++q)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[q][e] = 0.f;
#pragma unroll 4
        for (int j = 0; j < D; j += 4) {
            float4 rv[kQjlRows];
#pragma unroll
            for (int q = 0; q < kQjlRows; ++q) rv[q] = *reinterpret_cast<const float4*>(rw + q * D + j);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float4 s = *reinterpret_cast<const float4*>(Ss + (lane + 32 * e) * kStride + j);
#pragma unroll
                for (int q = 0; q < kQjlRows; ++q) {
                    acc[q][e] = fmaf(s.x, rv[q].x, acc[q][e]);
                    acc[q][e] = fmaf(s.y, rv[q].y, acc[q][e]);
                    acc[q][e] = fmaf(s.z, rv[q].z, acc[q][e]);
                    acc[q][e] = fmaf(s.w, rv[q].w, acc[q][e]);
                }
            }
        }
        // ---- store: indices, sign words, norm and gamma
#pragma unroll
        for (int q = 0; q < kQjlRows; ++q) {
            uint32_t mine = 0u;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const uint32_t w = __ballot_sync(0xFFFFFFFFu, acc[q][e] >= 0.f);
                if (lane == e) mine = w;
            }
            if (r0 + q < n_rows) {  // warp-uniform
                uint8_t* dst = packed + (r0 + q) * RB;
                warp_pack_row<D>(iw + q * D, lane, MB, dst);
                if (lane < E) reinterpret_cast<uint32_t*>(dst + IB)[lane] = mine;
                if (lane == 0) {
                    norms[r0 + q] = nrm[q];
                    rnorms[r0 + q] = gam[q];
                }
            }
        }
        __syncwarp();
    }
}

// Decode: y = s1 . H (s2 . (n c[idx] + kappa gamma S^T sgn)) / sqrt(d), kappa =
// sqrt(pi/2)/d; lane l computes coordinates l E .. l E + E - 1.  S^T sgn is
// taken as 2 t - c, t the sum of the rows of S whose sign bit is set (one
// predicated add per element) and c the column sums of S.
template <int D, int BITS, typename TO>
__global__ void __launch_bounds__(32 * kQjlWarps) k_decode_qjl(const uint8_t* __restrict__ packed,
                                                               const float* __restrict__ norms,
                                                               const float* __restrict__ rnorms, int64_t n_rows,
                                                               const float* __restrict__ S, TO* __restrict__ y,
                                                               const __grid_constant__ RowParams P, float kappa) {
    constexpr int E = D / 32, MB = BITS - 1;
    constexpr int RB = D * BITS / 8, IB = D * MB / 8;
    constexpr int kStride = QjlSmem<D>::kStride;
    extern __shared__ __align__(16) unsigned char qjl_smem[];
    float* Ss = reinterpret_cast<float*>(qjl_smem);
    __shared__ float csum[D];    // column sums of S
    __shared__ float cen_s[16];  // centroids by lane-varying index: shared memory, not the parameter bank
    stage_matrix<D>(S, Ss);
    if (threadIdx.x < 16) cen_s[threadIdx.x] = P.cen[threadIdx.x];
    __syncthreads();
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
        float c = 0.f;
        for (int k = 0; k < D; ++k) c += Ss[k * kStride + i];
        csum[i] = c;
    }
    __syncthreads();
    float cs[E];
    uint32_t sgl[E], sg2l[E];  // the lane's sign masks, read once (lane-varying parameter reads serialise)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        cs[e] = csum[lane * E + e];
        sgl[e] = sign_mask(P.sgnb, lane * E + e);
        sg2l[e] = P.two_sided ? sign_mask(P.sgn2b, lane * E + e) : 0u;
    }
    for (int64_t r0 = ((int64_t)blockIdx.x * kQjlWarps + warp) * kQjlRows; r0 < n_rows;
         r0 += (int64_t)gridDim.x * kQjlWarps * kQjlRows) {
        uint32_t sw[kQjlRows][E];  // sign words of each row (every lane holds all)
        uint32_t ib[kQjlRows];     // the lane's E indices
        float nrm[kQjlRows], gk[kQjlRows];
#pragma unroll
        for (int q = 0; q < kQjlRows; ++q) {
            const bool ok = r0 + q < n_rows;
            const uint8_t* row = packed + (ok ? r0 + q : 0) * RB;
            const uint32_t* w = reinterpret_cast<const uint32_t*>(row + IB);
#pragma unroll
            for (int e = 0; e < E; ++e) sw[q][e] = ok ? __ldg(w + e) : 0u;
            // bits [lane E MB, (lane + 1) E MB) of the index stream
            const int bit0 = lane * E * MB, wi = bit0 / 32, sh = bit0 % 32;
            const uint32_t* iwp = reinterpret_cast<const uint32_t*>(row);
            uint32_t v = ok ? __ldg(iwp + wi) >> sh : 0u;
            if (ok && sh + E * MB > 32) v |= __ldg(iwp + wi + 1) << (32 - sh);
            ib[q] = v;
            nrm[q] = ok ? __ldg(norms + r0 + q) : 0.f;
            gk[q] = ok ? __ldg(rnorms + r0 + q) * kappa : 0.f;
        }
        // t_i = sum of S[k][i] over the projections k with sgn_k = +1
        float t[kQjlRows][E];
#pragma unroll
        for (int q = 0; q < kQjlRows; ++q)
#pragma unroll
            for (int e = 0; e < E; ++e) t[q][e] = 0.f;
#pragma unroll
        for (int kw = 0; kw < E; ++kw) {
#pragma unroll
            for (int b = 0; b < 32; ++b) {
                const int k = 32 * kw + b;
                float s[E];
                if constexpr (E == 4) {
                    const float4 f = *reinterpret_cast<const float4*>(Ss + k * kStride + lane * 4);
                    s[0] = f.x; s[1] = f.y; s[2] = f.z; s[3] = f.w;
                } else if constexpr (E == 2) {
                    const float2 f = *reinterpret_cast<const float2*>(Ss + k * kStride + lane * 2);
                    s[0] = f.x; s[1] = f.y;
                } else {
                    s[0] = Ss[k * kStride + lane];
                }
#pragma unroll
                for (int q = 0; q < kQjlRows; ++q)
                    if (sw[q][kw] & (1u << b)) {
#pragma unroll
                        for (int e = 0; e < E; ++e) t[q][e] += s[e];
                    }
            }
        }
#pragma unroll
        for (int q = 0; q < kQjlRows; ++q) {
            if (r0 + q >= n_rows) break;  // warp-uniform
            float v[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float c = cen_s[(ib[q] >> (e * MB)) & ((1u << MB) - 1)];
                v[e] = fmaf(gk[q], fmaf(2.f, t[q][e], -cs[e]), nrm[q] * c);
                v[e] = __uint_as_float(__float_as_uint(v[e]) ^ sg2l[e]);
            }
            warp_fwht<E>(v, lane);
            TO* dst = y + (r0 + q) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float o = __uint_as_float(__float_as_uint(v[e] * P.inv_sqrt_d) ^ sgl[e]);
                if constexpr (sizeof(TO) == 2) dst[e] = __float2bfloat16_rn(o);
                else dst[e] = o;
            }
        }
    }
}

#if TQ_UNIT_D == 128
// ---- d = 128: the projections on the tensor cores (mma.sync m16n8k16, fp16
// operands, fp32 accumulation), a warp taking 16 rows at a time.
//
// Encode: the MSE stage computes what the CUDA-core kernel does, so indices,
// norms and gammas are the same; the indices are packed by shuffles and
// stored as soon as a row's are known.  The residuals, times 2^10, go to shared
// memory as fp16 high and low parts, and P = R S^T is taken as R_hi S_hi +
// R_lo S_hi + R_hi S_lo: each operand carried to about 22 bits, so a sign can
// differ from an exact projection's only within about 1e-6 ||r|| of zero.  The
// sign bits come from four ballots per tile of 8 projections.
// Decode: S^T sgn = SGN S with A = the signs as fp16 +-1 (exact), B = S as
// fp16 high and low parts, then the CUDA-core kernel's epilogue per row.
// S sits in shared memory as fp16 high and low parts in rows of 136 halves:
// [projection][dim] for the encode, [dim][projection] for the decode, so that
// each operand's ldmatrix reads 8 rows of 16 bytes from distinct banks.
// Row data reaches a warp through its own staging buffer in shared memory,
// filled by cp.async one tile ahead: the encoder's next 16 bf16 rows (4 KB,
// issued once the current rows have been read, so the copy runs under the
// projections), the decoder's next 16 packed rows with their norms and gammas
// (two buffers, since a tile's rows are read until its end).  Bytes past the
// last row are zero-filled.
#ifndef TQ_QJL_TC_WARPS
#define TQ_QJL_TC_WARPS 12
#endif
constexpr int kQtcWarps = TQ_QJL_TC_WARPS;
// rows the encoder's MSE stage takes side by side
#ifndef TQ_QJL_TC_SIDE
#define TQ_QJL_TC_SIDE 4
#endif
constexpr int kQtcSide = TQ_QJL_TC_SIDE;
constexpr int kQtcRow = 136;                                     // halves per row of an fp16 tile
constexpr int kQtcS = 2 * 128 * kQtcRow * 2;                     // S high and low parts
constexpr int kQtcEncWarp = 2 * 16 * kQtcRow * 2;                // residual parts
constexpr int kQtcEncXb = 16 * 128 * 2;                          // staged bf16 rows of a tile
constexpr int kQtcEncXbAt = kQtcS + kQtcWarps * kQtcEncWarp + 2 * 128 * 4;  // after the sign masks
constexpr int kQtcEncSmem = kQtcEncXbAt + kQtcWarps * kQtcEncXb;
constexpr int kQtcDecWarp = 16 * kQtcRow * 4;                    // S^T sgn of 16 rows, fp32
constexpr int kQtcDecXb = 16 * 64 + 2 * 16 * 4;                  // packed rows (at most 64 B), norms, gammas
constexpr int kQtcDecXbAt = kQtcS + kQtcWarps * kQtcDecWarp;
constexpr int kQtcDecSmem = kQtcDecXbAt + kQtcWarps * 2 * kQtcDecXb;
static_assert(kQtcEncXbAt % 16 == 0 && kQtcDecXbAt % 16 == 0 && kQtcDecXb % 16 == 0, "16-byte copies");
static_assert(kQtcEncSmem + 256 <= 232448 && kQtcDecSmem + 256 <= 232448, "shared memory per block");

// All of this thread's cp.async groups but the last one committed have landed.
__device__ __forceinline__ void qtc_cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void qtc_mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void qtc_ldsm4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// x as fp16 high and low parts (x = hi + lo to about 22 bits), packed pairwise.
__device__ __forceinline__ void qtc_split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
    const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
    hi = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
    lo = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
}
// S (fp32 [projection][dim]) as fp16 high and low parts in rows of kQtcRow
// halves, [projection][dim] or, TRANS, [dim][projection].
template <bool TRANS>
__device__ __forceinline__ void qtc_stage_s(const float* __restrict__ S, __half* sh, __half* sl) {
    for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {
        const int k = i >> 7, j = i & 127;
        const float v = __ldg(S + i);
        const __half h = __float2half_rn(v);
        const int at = TRANS ? j * kQtcRow + k : k * kQtcRow + j;
        sh[at] = h;
        sl[at] = __float2half_rn(v - __half2float(h));
    }
}
// bits 0..3 of e to bits 0, 2, 4, 6
__device__ __forceinline__ uint32_t qtc_spread4(uint32_t e) {
    return (e & 1u) | ((e & 2u) << 1) | ((e & 4u) << 2) | ((e & 8u) << 3);
}
// The MB-bit indices of dims 4l .. 4l + 3, bytes of lane l's ids, into the
// row's dense LSB-first stream at dst (16 MB bytes, 4-byte aligned): each
// lane's 4 MB-bit field, concatenated with its neighbours' by shuffles.
template <int MB>
__device__ __forceinline__ void qtc_pack_indices(uint32_t ids, int lane, uint8_t* dst) {
    const uint32_t f = (ids & 0xFFu) | (((ids >> 8) & 0xFFu) << MB) | (((ids >> 16) & 0xFFu) << (2 * MB)) |
                       ((ids >> 24) << (3 * MB));
    uint32_t* o = reinterpret_cast<uint32_t*>(dst);
    if constexpr (MB == 1) {  // 4-bit fields: 8 lanes per word
        uint32_t x = f;
        x |= __shfl_down_sync(0xFFFFFFFFu, x, 1) << 4;
        x |= __shfl_down_sync(0xFFFFFFFFu, x, 2) << 8;
        x |= __shfl_down_sync(0xFFFFFFFFu, x, 4) << 16;
        if ((lane & 7) == 0) o[lane >> 3] = x;
    } else if constexpr (MB == 2) {  // 8-bit fields: 4 lanes per word
        uint32_t x = f;
        x |= __shfl_down_sync(0xFFFFFFFFu, x, 1) << 8;
        x |= __shfl_down_sync(0xFFFFFFFFu, x, 2) << 16;
        if ((lane & 3) == 0) o[lane >> 2] = x;
    } else {  // 12-bit fields: 8 lanes per 3 words
        const uint32_t p = f | (__shfl_down_sync(0xFFFFFFFFu, f, 1) << 12);  // 24 bits (even lanes)
        const uint64_t q = (uint64_t)p | ((uint64_t)__shfl_down_sync(0xFFFFFFFFu, p, 2) << 24);  // 48 bits (lanes 4k)
        const uint32_t plo = __shfl_down_sync(0xFFFFFFFFu, (uint32_t)q, 4);
        const uint32_t phi = __shfl_down_sync(0xFFFFFFFFu, (uint32_t)(q >> 32), 4);
        const uint64_t partner = ((uint64_t)phi << 32) | plo;  // lanes 4k + 4 .. 4k + 7
        const uint64_t lo = q | (partner << 48);
        if ((lane & 7) == 0) {
            o[3 * (lane >> 3)] = (uint32_t)lo;
            o[3 * (lane >> 3) + 1] = (uint32_t)(lo >> 32);
            o[3 * (lane >> 3) + 2] = (uint32_t)(partner >> 16);
        }
    }
}
// warp_fwht and warp_sum on R rows side by side: each row's operations are
// those of the one-row versions, and the rows' shuffles overlap.
template <int R, int E>
__device__ __forceinline__ void warp_fwht_rows(float (&v)[R][E], int lane) {
#pragma unroll
    for (int q = 0; q < R; ++q) fwht_reg<E>(v[q]);
#pragma unroll
    for (int b = 1; b < 32; b <<= 1) {
        // (lo + hi, lo - hi) as one fused multiply-add, o + (+-1) v: the
        // product is exact, so the one rounding is that of the add
        const float sgn = (lane & b) ? -1.f : 1.f;
#pragma unroll
        for (int q = 0; q < R; ++q)
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float o = __shfl_xor_sync(0xFFFFFFFFu, v[q][e], b);
                v[q][e] = fmaf(sgn, v[q][e], o);
            }
    }
}
template <int R>
__device__ __forceinline__ void warp_sum_rows(float (&s)[R]) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int q = 0; q < R; ++q) s[q] += __shfl_xor_sync(0xFFFFFFFFu, s[q], o);
}

template <int BITS, typename T>
__global__ void __launch_bounds__(32 * kQtcWarps, 1) k_encode_qjl_tc(const T* __restrict__ x, int64_t n_rows,
                                                                  const float* __restrict__ S,
                                                                  uint8_t* __restrict__ packed,
                                                                  float* __restrict__ norms,
                                                                  float* __restrict__ rnorms,
                                                                  const __grid_constant__ RowParams P) {
    constexpr int D = 128, E = 4, MB = BITS - 1, NB = (1 << MB) - 1;
    constexpr int RB = D * BITS / 8, IB = D * MB / 8;
    extern __shared__ __align__(16) unsigned char qtc_smem[];
    __half* Sh = reinterpret_cast<__half*>(qtc_smem);
    __half* Sl = Sh + 128 * kQtcRow;
    uint32_t* sg = reinterpret_cast<uint32_t*>(qtc_smem + kQtcS + kQtcWarps * kQtcEncWarp);
    uint32_t* sg2 = sg + D;
    // centroids and boundaries by lane-varying index: shared memory, not the parameter bank
    __shared__ float cen_s[16], bnd_s[16];
    qtc_stage_s<false>(S, Sh, Sl);
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
        sg[i] = sign_mask(P.sgnb, i);
        sg2[i] = sign_mask(P.sgn2b, i);
    }
    if (threadIdx.x < 16) {
        cen_s[threadIdx.x] = P.cen[threadIdx.x];
        bnd_s[threadIdx.x] = threadIdx.x < NB ? P.bnd[threadIdx.x] : 0.f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* wb = qtc_smem + kQtcS + warp * kQtcEncWarp;
    uint32_t* Rh = reinterpret_cast<uint32_t*>(wb);                       // [16][kQtcRow / 2] half pairs
    uint32_t* Rl = Rh + 16 * kQtcRow / 2;
    const uint32_t sRh = smem_addr(Rh), sSh = smem_addr(Sh), sSl = smem_addr(Sl);
    const uint32_t sRl = smem_addr(Rl);
    // bf16 rows come through the warp's staging buffer (fp32 rows, twice the
    // bytes, are loaded directly)
    constexpr bool kStaged = sizeof(T) == 2;
    const unsigned char* xb = qtc_smem + kQtcEncXbAt + warp * kQtcEncXb;
    const uint32_t sXb = smem_addr(xb);
    auto stage = [&](int64_t t0) {  // tile t0 .. t0 + 15: 256 pieces of 16 bytes, 8 per lane
        const unsigned char* src = reinterpret_cast<const unsigned char*>(x + t0 * D);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int p = lane + 32 * k;  // row p / 16
            const bool in = t0 + (p >> 4) < n_rows;
            cp_async16(sXb + 16u * p, in ? src + 16 * p : src, in ? 16u : 0u);
        }
        cp_async_commit();
    };
    const int64_t r_step = (int64_t)gridDim.x * kQtcWarps * 16;
    int64_t r0 = ((int64_t)blockIdx.x * kQtcWarps + warp) * 16;
    if constexpr (kStaged) {
        if (r0 < n_rows) stage(r0);
    }
    for (; r0 < n_rows; r0 += r_step) {
        if constexpr (kStaged) {
            cp_async_wait_all();
            __syncwarp();
        }
        // ---- MSE stage and residual of each row, kQtcSide rows side by side
        // (their loads first; rows past the end: zeros)
#pragma unroll 1
        for (int q0 = 0; q0 < 16; q0 += kQtcSide) {
            float vq[kQtcSide][E];
#pragma unroll
            for (int q = 0; q < kQtcSide; ++q) {
                if (r0 + q0 + q < n_rows) {
                    if constexpr (kStaged) {
                        const uint2 u = *reinterpret_cast<const uint2*>(xb + (q0 + q) * 256 + 8 * lane);
                        const uint32_t h[E] = {u.x << 16, u.x & 0xFFFF0000u, u.y << 16, u.y & 0xFFFF0000u};
#pragma unroll
                        for (int e = 0; e < E; ++e) vq[q][e] = __uint_as_float(h[e] ^ sg[lane * E + e]);
                    } else {
                        load_lane<E, T>(x + (r0 + q0 + q) * D, lane, sg, vq[q]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) vq[q][e] = 0.f;
                }
            }
            float ss[kQtcSide];
#pragma unroll
            for (int q = 0; q < kQtcSide; ++q) {
                ss[q] = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) ss[q] = fmaf(vq[q][e], vq[q][e], ss[q]);
            }
            warp_sum_rows<kQtcSide>(ss);
            warp_fwht_rows<kQtcSide, E>(vq, lane);
            float rr[kQtcSide];
#pragma unroll
            for (int q = 0; q < kQtcSide; ++q) {
                const int row = q0 + q;
                float(&v)[E] = vq[q];
                if (P.two_sided) {
#pragma unroll
                    for (int e = 0; e < E; ++e) v[e] = __uint_as_float(__float_as_uint(v[e]) ^ sg2[lane * E + e]);
                }
                float n = __fsqrt_rn(ss[q]);
                float inv = n > 0.f ? __fdiv_rn(P.inv_sqrt_d, n) : 0.f;
                if (!ss_in_range(ss[q])) warp_rescaled_norm<D, E>(v, n, inv);  // squares past fp32's range
                ss[q] = n;
                float rs[E];
                uint32_t ids = 0u;
                rr[q] = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    // the number of boundaries at or below the coordinate; the
                    // test is monotone in the boundary, so a binary search
                    // finds the count
                    int id = 0;
#pragma unroll
                    for (int step = (NB + 1) / 2; step >= 1; step >>= 1)
                        if (fmaf(v[e], inv, -bnd_s[id + step - 1]) >= 0.0f) id += step;
                    const float r = fmaf(v[e], inv, -cen_s[id]);
                    rr[q] = fmaf(r, r, rr[q]);
                    ids |= (uint32_t)id << (8 * e);
                    rs[e] = r * 1024.f;  // exact; keeps the low parts out of the fp16 subnormals
                }
                if (r0 + row < n_rows) qtc_pack_indices<MB>(ids, lane, packed + (r0 + row) * RB);  // warp-uniform
                uint32_t h0, l0, h1, l1;
                qtc_split2(rs[0], rs[1], h0, l0);
                qtc_split2(rs[2], rs[3], h1, l1);
                *reinterpret_cast<uint2*>(Rh + row * (kQtcRow / 2) + 2 * lane) = make_uint2(h0, h1);
                *reinterpret_cast<uint2*>(Rl + row * (kQtcRow / 2) + 2 * lane) = make_uint2(l0, l1);
            }
            warp_sum_rows<kQtcSide>(rr);
            if (lane == 0) {
#pragma unroll
                for (int q = 0; q < kQtcSide; ++q)
                    if (r0 + q0 + q < n_rows) {
                        norms[r0 + q0 + q] = ss[q];
                        rnorms[r0 + q0 + q] = ss[q] * __fsqrt_rn(rr[q]);
                    }
            }
        }
        __syncwarp();
        // every lane has read the staged rows: the next tile's copy runs
        // under this tile's projections
        if constexpr (kStaged) {
            if (r0 + r_step < n_rows) stage(r0 + r_step);
        }
        // ---- P = R S^T: A fragments of the 8 k-steps (16 dims each), then
        // tiles of 8 projections
        uint32_t ah[8][4], al[8][4];
        {
            const uint32_t off = (uint32_t)(((lane & 15) * kQtcRow + (lane >> 4) * 8) * 2);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                qtc_ldsm4(sRh + off + 32u * kk, ah[kk]);
                qtc_ldsm4(sRl + off + 32u * kk, al[kk]);
            }
        }
        const uint32_t boff = (uint32_t)(((lane & 7) * kQtcRow + (lane >> 3) * 8) * 2);
        // sign word w of each row: projections 32 w .. 32 w + 31, four tiles
#pragma unroll 1
        for (int w = 0; w < 4; ++w) {
            uint32_t word = 0u;  // lane r < 16: row r's
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nt = 4 * w + j;
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < 8; kk += 2) {
                    uint32_t bh[4], bl[4];
                    const uint32_t off = boff + (uint32_t)((8 * nt * kQtcRow + 16 * kk) * 2);
                    qtc_ldsm4(sSh + off, bh);  // k-steps kk (regs 0, 1) and kk + 1 (regs 2, 3)
                    qtc_ldsm4(sSl + off, bl);
                    qtc_mma(c, ah[kk], bh[0], bh[1]);
                    qtc_mma(c, al[kk], bh[0], bh[1]);
                    qtc_mma(c, ah[kk], bl[0], bl[1]);
                    qtc_mma(c, ah[kk + 1], bh[2], bh[3]);
                    qtc_mma(c, al[kk + 1], bh[2], bh[3]);
                    qtc_mma(c, ah[kk + 1], bl[2], bl[3]);
                }
                // c: rows g, g + 8, projections 8 nt + 2t, 8 nt + 2t + 1 (lane 4g + t)
                const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, c[0] >= 0.f);
                const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, c[1] >= 0.f);
                const uint32_t b2 = __ballot_sync(0xFFFFFFFFu, c[2] >= 0.f);
                const uint32_t b3 = __ballot_sync(0xFFFFFFFFu, c[3] >= 0.f);
                const uint32_t sh = 4u * (uint32_t)(lane & 7);
                const uint32_t e0 = ((lane < 8 ? b0 : b2) >> sh) & 0xFu, e1 = ((lane < 8 ? b1 : b3) >> sh) & 0xFu;
                word |= (qtc_spread4(e0) | (qtc_spread4(e1) << 1)) << (8 * j);
            }
            if (lane < 16 && r0 + lane < n_rows) reinterpret_cast<uint32_t*>(packed + (r0 + lane) * RB + IB)[w] = word;
        }
        __syncwarp();
    }
}

template <int BITS, typename TO>
__global__ void __launch_bounds__(32 * kQtcWarps, 1) k_decode_qjl_tc(const uint8_t* __restrict__ packed,
                                                                  const float* __restrict__ norms,
                                                                  const float* __restrict__ rnorms,
                                                                  int64_t n_rows, const float* __restrict__ S,
                                                                  TO* __restrict__ y,
                                                                  const __grid_constant__ RowParams P, float kappa) {
    constexpr int D = 128, E = 4, MB = BITS - 1;
    constexpr int RB = D * BITS / 8, IB = D * MB / 8;
    extern __shared__ __align__(16) unsigned char qtc_smem[];
    __half* Sh = reinterpret_cast<__half*>(qtc_smem);  // [dim][projection]
    __half* Sl = Sh + 128 * kQtcRow;
    __shared__ float cen_s[16];  // centroids by lane-varying index: shared memory, not the parameter bank
    qtc_stage_s<true>(S, Sh, Sl);
    if (threadIdx.x < 16) cen_s[threadIdx.x] = P.cen[threadIdx.x];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    float* Tb = reinterpret_cast<float*>(qtc_smem + kQtcS + warp * kQtcDecWarp);  // [16][kQtcRow]
    uint32_t sgl[E], sg2l[E];  // the lane's sign masks, read once (lane-varying parameter reads serialise)
#pragma unroll
    for (int e = 0; e < E; ++e) {
        sgl[e] = sign_mask(P.sgnb, lane * E + e);
        sg2l[e] = P.two_sided ? sign_mask(P.sgn2b, lane * E + e) : 0u;
    }
    const uint32_t sSh = smem_addr(Sh), sSl = smem_addr(Sl);
    const uint32_t boff = (uint32_t)(((lane & 7) * kQtcRow + (lane >> 3) * 8) * 2);
    // staging buffer b of the warp: the tile's packed rows (16 RB bytes), then
    // its 16 norms and 16 gammas
    const unsigned char* xb0 = qtc_smem + kQtcDecXbAt + warp * 2 * kQtcDecXb;
    const uint32_t sXb0 = smem_addr(xb0);
    auto stage = [&](int64_t t0, int b) {  // always commits a group, empty past the end
        if (t0 < n_rows) {
            const uint32_t dst = sXb0 + (uint32_t)(b * kQtcDecXb);
            const uint8_t* src = packed + t0 * RB;
            const int64_t have = n_rows - t0;  // rows of the tile that exist (may exceed 16)
            for (int p = lane; p < RB; p += 32) {  // RB pieces of 16 bytes, RB / 16 per row
                const bool in = p / (RB / 16) < have;
                cp_async16(dst + 16u * p, in ? src + 16 * p : src, in ? 16u : 0u);
            }
            const int r = lane & 15;
            const bool in = r < have;
            cp_async4(dst + 16u * RB + 4u * lane, (lane < 16 ? norms : rnorms) + t0 + (in ? r : 0), in ? 4u : 0u);
        }
        cp_async_commit();
    };
    const int64_t r_step = (int64_t)gridDim.x * kQtcWarps * 16;
    int64_t r0 = ((int64_t)blockIdx.x * kQtcWarps + warp) * 16;
    stage(r0, 0);
    for (int it = 0; r0 < n_rows; r0 += r_step, ++it) {
        stage(r0 + r_step, (it + 1) & 1);
        qtc_cp_async_wait_prev();  // this tile's group
        __syncwarp();
        const unsigned char* xb = xb0 + (it & 1) * kQtcDecXb;
        const float* xn = reinterpret_cast<const float*>(xb + 16 * RB);  // norms, then gammas
        // sign words: lane r < 16 reads row r's, then each lane takes rows g and g + 8
        uint4 wv = make_uint4(0u, 0u, 0u, 0u);
        if (lane < 16) wv = *reinterpret_cast<const uint4*>(xb + lane * RB + IB);
        const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t wg[4], wg8[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            wg[i] = __shfl_sync(0xFFFFFFFFu, w4[i], g);
            wg8[i] = __shfl_sync(0xFFFFFFFFu, w4[i], g + 8);
        }
        // A: sgn_k as fp16 +1 (bit set) or -1; k-step kk is projections
        // 16 kk .. 16 kk + 15, bits 16 (kk & 1) + .. of word kk / 2
        auto pm = [](uint32_t z) { return 0x3C003C00u | ((~z & 1u) << 15) | ((~z & 2u) << 30); };
        uint32_t a[8][4];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int b = 16 * (kk & 1) + 2 * t;
            a[kk][0] = pm(wg[kk >> 1] >> b);
            a[kk][1] = pm(wg8[kk >> 1] >> b);
            a[kk][2] = pm(wg[kk >> 1] >> (b + 8));
            a[kk][3] = pm(wg8[kk >> 1] >> (b + 8));
        }
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
                uint32_t bh[4], bl[4];
                const uint32_t off = boff + (uint32_t)((8 * nt * kQtcRow + 16 * kk) * 2);
                qtc_ldsm4(sSh + off, bh);
                qtc_ldsm4(sSl + off, bl);
                qtc_mma(c, a[kk], bh[0], bh[1]);
                qtc_mma(c, a[kk], bl[0], bl[1]);
                qtc_mma(c, a[kk + 1], bh[2], bh[3]);
                qtc_mma(c, a[kk + 1], bl[2], bl[3]);
            }
            // rows g, g + 8, dims 8 nt + 2t, + 1
            *reinterpret_cast<float2*>(Tb + g * kQtcRow + 8 * nt + 2 * t) = make_float2(c[0], c[1]);
            *reinterpret_cast<float2*>(Tb + (g + 8) * kQtcRow + 8 * nt + 2 * t) = make_float2(c[2], c[3]);
        }
        __syncwarp();
        // ---- per row: n c[idx] + kappa gamma S^T sgn, then the inverse transform
#pragma unroll 1
        for (int q0 = 0; q0 < 16; q0 += 4) {
            uint32_t ib[4];
            float nrm[4], gk[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // rows past the end read the zero fill
                const int bit0 = lane * E * MB, wi = bit0 / 32, sh = bit0 % 32;
                const uint32_t* iwp = reinterpret_cast<const uint32_t*>(xb + (q0 + q) * RB);
                uint32_t v = iwp[wi] >> sh;
                if (sh + E * MB > 32) v |= iwp[wi + 1] << (32 - sh);
                ib[q] = v;
                nrm[q] = xn[q0 + q];
                gk[q] = xn[16 + q0 + q] * kappa;
            }
            float v[4][E];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 tv = *reinterpret_cast<const float4*>(Tb + (q0 + q) * kQtcRow + 4 * lane);
                const float tt[E] = {tv.x, tv.y, tv.z, tv.w};
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float c = cen_s[(ib[q] >> (e * MB)) & ((1u << MB) - 1)];
                    v[q][e] = fmaf(gk[q], tt[e], nrm[q] * c);
                    v[q][e] = __uint_as_float(__float_as_uint(v[q][e]) ^ sg2l[e]);
                }
            }
            warp_fwht_rows<4, E>(v, lane);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (r0 + q0 + q >= n_rows) continue;  // warp-uniform
                float o[E];
#pragma unroll
                for (int e = 0; e < E; ++e)
                    o[e] = __uint_as_float(__float_as_uint(v[q][e] * P.inv_sqrt_d) ^ sgl[e]);
                TO* dst = y + (r0 + q0 + q) * D + lane * E;  // 16-byte aligned rows
                if constexpr (sizeof(TO) == 2) {
                    const __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]), b = __floats2bfloat162_rn(o[2], o[3]);
                    *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<const uint32_t*>(&a),
                                                                *reinterpret_cast<const uint32_t*>(&b));
                } else {
                    *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
                }
            }
        }
        __syncwarp();
    }
}
#endif

}  // namespace dev

namespace {

template <typename K>
unsigned qjl_grid(K fn, int64_t n_rows, int smem) {
    const int64_t per_block = (int64_t)dev::kQjlWarps * dev::kQjlRows;
    int64_t g = (n_rows + per_block - 1) / per_block;
    const int64_t cap = (int64_t)num_sms() * blocks_per_sm((const void*)fn, 32 * dev::kQjlWarps, smem);
    if (g > cap) g = cap;
    return (unsigned)(g < 1 ? 1 : g);
}

template <int D, int BITS, typename T>
cudaError_t enc_qjl(const void* x, int64_t n, const float* S, uint8_t* pk, float* nm, float* rn,
                    const RowParams& P, cudaStream_t s) {
    auto fn = dev::k_encode_qjl<D, BITS, T>;
    constexpr int smem = dev::QjlSmem<D>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fn<<<qjl_grid(fn, n, smem), 32 * dev::kQjlWarps, smem, s>>>(static_cast<const T*>(x), n, S, pk, nm, rn, P);
    return cudaGetLastError();
}

template <int D, int BITS, typename TO>
cudaError_t dec_qjl(const uint8_t* pk, const float* nm, const float* rn, int64_t n, const float* S, void* y,
                    const RowParams& P, cudaStream_t s) {
    auto fn = dev::k_decode_qjl<D, BITS, TO>;
    constexpr int smem = dev::QjlSmem<D>::kS;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const float kappa = (float)(1.2533141373155003 / D);  // sqrt(pi / 2) / d
    fn<<<qjl_grid(fn, n, smem), 32 * dev::kQjlWarps, smem, s>>>(pk, nm, rn, n, S, static_cast<TO*>(y), P, kappa);
    return cudaGetLastError();
}

#if TQ_UNIT_D == 128
template <int BITS, typename T>
cudaError_t enc_qjl_tc(const void* x, int64_t n, const float* S, uint8_t* pk, float* nm, float* rn,
                       const RowParams& P, cudaStream_t s) {
    auto fn = dev::k_encode_qjl_tc<BITS, T>;
    constexpr int smem = dev::kQtcEncSmem;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t per_block = (int64_t)dev::kQtcWarps * 16;
    int64_t g = (n + per_block - 1) / per_block;
    const int64_t cap = (int64_t)num_sms() * blocks_per_sm((const void*)fn, 32 * dev::kQtcWarps, smem);
    if (g > cap) g = cap;
    fn<<<(unsigned)(g < 1 ? 1 : g), 32 * dev::kQtcWarps, smem, s>>>(static_cast<const T*>(x), n, S, pk, nm, rn, P);
    return cudaGetLastError();
}

template <int BITS, typename TO>
cudaError_t dec_qjl_tc(const uint8_t* pk, const float* nm, const float* rn, int64_t n, const float* S, void* y,
                       const RowParams& P, cudaStream_t s) {
    auto fn = dev::k_decode_qjl_tc<BITS, TO>;
    constexpr int smem = dev::kQtcDecSmem;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t per_block = (int64_t)dev::kQtcWarps * 16;
    int64_t g = (n + per_block - 1) / per_block;
    const int64_t cap = (int64_t)num_sms() * blocks_per_sm((const void*)fn, 32 * dev::kQtcWarps, smem);
    if (g > cap) g = cap;
    const float kappa = (float)(1.2533141373155003 / 128);  // sqrt(pi / 2) / d
    fn<<<(unsigned)(g < 1 ? 1 : g), 32 * dev::kQtcWarps, smem, s>>>(pk, nm, rn, n, S, static_cast<TO*>(y), P,
                                                                    kappa);
    return cudaGetLastError();
}
#endif

}  // namespace

template <int D>
cudaError_t launch_encode_qjl_d(int bits, tq_dtype dt, const void* x, int64_t n_rows, const float* S,
                                uint8_t* packed, float* norms, float* rnorms, const RowParams& P,
                                cudaStream_t s) {
    auto go = [&](auto tag) {
        using T = decltype(tag);
#if TQ_UNIT_D == 128
        if constexpr (D == 128) {  // the projections on the tensor cores
            switch (bits) {
                case 2: return enc_qjl_tc<2, T>(x, n_rows, S, packed, norms, rnorms, P, s);
                case 3: return enc_qjl_tc<3, T>(x, n_rows, S, packed, norms, rnorms, P, s);
                default: return enc_qjl_tc<4, T>(x, n_rows, S, packed, norms, rnorms, P, s);
            }
        } else
#endif
        {
            switch (bits) {
                case 2: return enc_qjl<D, 2, T>(x, n_rows, S, packed, norms, rnorms, P, s);
                case 3: return enc_qjl<D, 3, T>(x, n_rows, S, packed, norms, rnorms, P, s);
                default: return enc_qjl<D, 4, T>(x, n_rows, S, packed, norms, rnorms, P, s);
            }
        }
    };
    return dt == TQ_BF16 ? go(__nv_bfloat16{}) : go(float{});
}

template <int D>
cudaError_t launch_decode_qjl_d(int bits, tq_dtype dt, const uint8_t* packed, const float* norms,
                                const float* rnorms, int64_t n_rows, const float* S, void* y, const RowParams& P,
                                cudaStream_t s) {
    auto go = [&](auto tag) {
        using TO = decltype(tag);
#if TQ_UNIT_D == 128
        if constexpr (D == 128) {  // the projections on the tensor cores
            switch (bits) {
                case 2: return dec_qjl_tc<2, TO>(packed, norms, rnorms, n_rows, S, y, P, s);
                case 3: return dec_qjl_tc<3, TO>(packed, norms, rnorms, n_rows, S, y, P, s);
                default: return dec_qjl_tc<4, TO>(packed, norms, rnorms, n_rows, S, y, P, s);
            }
        } else
#endif
        {
            switch (bits) {
                case 2: return dec_qjl<D, 2, TO>(packed, norms, rnorms, n_rows, S, y, P, s);
                case 3: return dec_qjl<D, 3, TO>(packed, norms, rnorms, n_rows, S, y, P, s);
                default: return dec_qjl<D, 4, TO>(packed, norms, rnorms, n_rows, S, y, P, s);
            }
        }
    };
    return dt == TQ_BF16 ? go(__nv_bfloat16{}) : go(float{});
}

#if TQ_UNIT_D == 128
cudaError_t launch_qjl_matrix(uint64_t seed, int d, float* S, cudaStream_t s) {
    const int64_t n = (int64_t)d * d;
    dev::k_qjl_matrix<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(seed, d, S);
    return cudaGetLastError();
}
#endif

#if !defined(TQ_UNIT_D)
#error "compile once per head dimension with -DTQ_UNIT_D=<d>"
#endif
template cudaError_t launch_encode_qjl_d<TQ_UNIT_D>(int, tq_dtype, const void*, int64_t, const float*, uint8_t*,
                                                    float*, float*, const RowParams&, cudaStream_t);
template cudaError_t launch_decode_qjl_d<TQ_UNIT_D>(int, tq_dtype, const uint8_t*, const float*, const float*,
                                                    int64_t, const float*, void*, const RowParams&, cudaStream_t);

}  // namespace tq
