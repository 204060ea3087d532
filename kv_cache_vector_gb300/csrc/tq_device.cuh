// tq_device.cuh -- device building blocks of the sm_103a row codec.
//
// A row of d elements is held by R = d/E threads (E <= 128 elements in
// registers each; R = 2 only for d = 256).  The Walsh-Hadamard transform runs
// as log2(E) register-only butterfly stages plus, for R = 2, one stage that
// pairs the two threads through a shuffle ("TurboQuant KV Cache Compression
// -- Spec", Hadamard Transform Detail: stages commute, so the cross-thread
// stage can come last on encode and last on decode).
//
// Element layouts for R = 2 (E = 128, d = 256), thread part p in {0, 1}:
//   "contiguous":  slot s <-> element p*E + s
//   "split":       slot s <  E/2 <-> element p*E/2 + s
//                  slot s >= E/2 <-> element E + p*E/2 + (s - E/2)
// Encode loads contiguous and leaves split after the cross stage; decode
// loads split and leaves contiguous.  The packed bit stream of a split part
// is two contiguous runs of E/2 indices, so both sides stay vectorised.
#pragma once

#include <cstdint>

#include <cfloat>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tq {
namespace dev {

template <int D>
struct RowShape {
    static constexpr int R = (D > 128) ? 2 : 1;  // threads per row
    static constexpr int E = D / R;              // elements per thread
};

// Coordinate of element i of part p in the rotated domain.  With two threads
// per row the rotated coordinates are split: part p holds [p E/2, (p+1) E/2)
// and [E + p E/2, E + (p+1) E/2), the order of the packed row.
template <int D>
__device__ __forceinline__ int rotated_coord(int p, int i) {
    constexpr int R = RowShape<D>::R, E = RowShape<D>::E;
    if constexpr (R == 1) return i;
    else return i < E / 2 ? p * (E / 2) + i : E + p * (E / 2) + (i - E / 2);
}

// Two-sided signs: flip the rotated-domain values of part p by s2.
template <int D, int E>
__device__ __forceinline__ void flip_rotated(float (&v)[E], int p, const uint32_t* sgn2) {
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = __uint_as_float(__float_as_uint(v[i]) ^ sgn2[rotated_coord<D>(p, i)]);
}

// ------------------------------------------------------------- load + sign

// v[s] = s_i * x_i for the thread's E elements starting at element `first`
// (contiguous layout).  The sign is an xor of the fp32 sign bit with the
// per-element mask from the parameter bank.
template <int E>
__device__ __forceinline__ void load_signed(const float* __restrict__ src, float (&v)[E],
                                            const uint32_t* sgn) {
    static_assert(E % 4 == 0 || E < 4, "vector width");
    if constexpr (E >= 4) {
        const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
        for (int k = 0; k < E / 4; ++k) {
            uint4 w = __ldg(p + k);
            v[4 * k + 0] = __uint_as_float(w.x ^ sgn[4 * k + 0]);
            v[4 * k + 1] = __uint_as_float(w.y ^ sgn[4 * k + 1]);
            v[4 * k + 2] = __uint_as_float(w.z ^ sgn[4 * k + 2]);
            v[4 * k + 3] = __uint_as_float(w.w ^ sgn[4 * k + 3]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < E; ++k) v[k] = __uint_as_float(__float_as_uint(src[k]) ^ sgn[k]);
    }
}

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ float bf16lo(uint32_t w, uint32_t m) {
    return __uint_as_float((w << 16) ^ m);
}
__device__ __forceinline__ float bf16hi(uint32_t w, uint32_t m) {
    return __uint_as_float((w & 0xFFFF0000u) ^ m);
}

template <int E>
__device__ __forceinline__ void load_signed(const __nv_bfloat16* __restrict__ src, float (&v)[E],
                                            const uint32_t* sgn) {
    static_assert(E % 8 == 0, "bf16 rows are loaded 16 bytes at a time");
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int k = 0; k < E / 8; ++k) {
        uint4 w = __ldg(p + k);
        const uint32_t* m = sgn + 8 * k;
        v[8 * k + 0] = bf16lo(w.x, m[0]);
        v[8 * k + 1] = bf16hi(w.x, m[1]);
        v[8 * k + 2] = bf16lo(w.y, m[2]);
        v[8 * k + 3] = bf16hi(w.y, m[3]);
        v[8 * k + 4] = bf16lo(w.z, m[4]);
        v[8 * k + 5] = bf16hi(w.z, m[5]);
        v[8 * k + 6] = bf16lo(w.w, m[6]);
        v[8 * k + 7] = bf16hi(w.w, m[7]);
    }
}

// ------------------------------------------------------------------ FWHT

// The xor mask of sign j (0x80000000 for a negative sign) from its bit in
// 32-bit words (AttnParams::sgnb / sgn2b).
__device__ __forceinline__ uint32_t sign_mask(const uint32_t* bits, int j) {
    return ((bits[j >> 5] >> (j & 31)) & 1u) << 31;
}

// Unnormalised butterfly over the E registers: stages len = 1 .. E/2,
// (a, b) -> (a + b, a - b).  Every loop has a constant trip count (stage st,
// butterfly q; the pair is (i, i + 2^st) with i = q with a zero bit inserted
// at position st), so full unrolling turns every index into a constant and
// the row stays in registers.
template <int E>
__device__ __forceinline__ void fwht_reg(float (&v)[E]) {
#pragma unroll
    for (int st = 0; (1 << st) < E; ++st) {
#pragma unroll
        for (int q = 0; q < E / 2; ++q) {
            const int len = 1 << st;
            const int i = ((q >> st) << (st + 1)) | (q & (len - 1));
            const float a = v[i], b = v[i + len];
            v[i] = a + b;
            v[i + len] = a - b;
        }
    }
}

// Packed fp32x2 arithmetic on a register pair (inline PTX on .b64 operands;
// the pair is packed and unpacked with mov, which register allocation folds).
struct F2 {
    unsigned long long r;
};
__device__ __forceinline__ F2 f2(float lo, float hi) {
    F2 o;
    asm("mov.b64 %0, {%1, %2};" : "=l"(o.r) : "f"(lo), "f"(hi));
    return o;
}
__device__ __forceinline__ void f2_split(F2 a, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.r));
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    F2 o;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(o.r) : "l"(a.r), "l"(b.r));
    return o;
}
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
    F2 o;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(o.r) : "l"(a.r), "l"(b.r));
    return o;
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
    F2 o;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(o.r) : "l"(a.r), "l"(b.r));
    return o;
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
    F2 o;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(o.r) : "l"(a.r), "l"(b.r), "l"(c.r));
    return o;
}

// The same transform with packed fp32x2 arithmetic: stage len = 1 is scalar,
// every later stage pairs registers (i, i+1) with (i+len, i+len+1), so one
// instruction does two butterflies.  Same lane-op count, half the issue slots.
template <int E>
__device__ __forceinline__ void fwht_reg2(float (&v)[E]) {
#pragma unroll
    for (int j = 0; j < E; j += 2) {
        const float a = v[j], b = v[j + 1];
        v[j] = a + b;
        v[j + 1] = a - b;
    }
#pragma unroll
    for (int st = 1; (1 << st) < E; ++st) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {  // q-th pair of butterflies of this stage
            const int len = 1 << st;
            const int i = (((2 * q) >> st) << (st + 1)) | ((2 * q) & (len - 1));
            const F2 a = f2(v[i], v[i + 1]);
            const F2 b = f2(v[i + len], v[i + len + 1]);
            f2_split(f2_add(a, b), v[i], v[i + 1]);
            f2_split(f2_sub(a, b), v[i + len], v[i + len + 1]);
        }
    }
}

// The butterfly stage that pairs slot s of part 0 with slot s of part 1
// (lanes l and l^1).  Part 0 computes both outputs of slots [0, E/2), part 1
// those of slots [E/2, E); afterwards slot j (j < E/2) holds the part-0
// output and slot E/2 + j the part-1 output of the slot it computed.
template <int E>
__device__ __forceinline__ void fwht_cross(float (&v)[E], int p) {
    constexpr int H = E / 2;
#pragma unroll
    for (int j = 0; j < H; ++j) {
        float send = p ? v[j] : v[H + j];
        float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 1);
        float a = p ? recv : v[j];
        float b = p ? v[H + j] : recv;
        v[j] = a + b;
        v[H + j] = a - b;
    }
}

// ------------------------------------------------------------- bucketing

struct LutEntry {
    int lo;     // #{ j : beta_j < cell_lo }
    float thr;  // the one boundary inside the closed cell, or +inf
};

// Fill the bucketing table from the fp32 boundaries (every thread of the
// block takes part; the caller synchronises).  Exact by construction: every
// closed cell holds at most one boundary (checked on the host when the plan
// is built), so for any w in cell g,
//   #{ j : w >= beta_j } = lo_g + [w >= thr_g].
__device__ __forceinline__ void build_lut(LutEntry* lut, const float* bnd, int nb) {
    for (int g = threadIdx.x; g < kLutCells; g += blockDim.x) {
        float lo = (float)(g - kLutCenter - 0.5) / (float)kLutScale;
        float hi = (float)(g - kLutCenter + 0.5) / (float)kLutScale;
        int cnt = 0;
        float thr = __int_as_float(0x7F800000);
        for (int j = 0; j < nb; ++j) {
            float b = bnd[j];
            if (b < lo) cnt += 1;
            else if (b <= hi) thr = b;
        }
        lut[g].lo = cnt;
        lut[g].thr = thr;
    }
}

// Rows whose sum of squares leaves fp32's range.  The encoders take a row's
// norm from its sum of squares; for a row of finite norm that sum can still
// overflow (norms above about 1.8e19) or underflow (below about 1e-19), and
// the norm and every index would come out wrong.  Such a row -- and a zero or
// non-finite one, which share the test -- is measured again on y S, S the
// power of two that brings the row's largest |y| to [1, 4): an exact
// scaling, so the normalised coordinates and the stored norm are the ones
// the unscaled arithmetic would give had it the range.
__device__ __forceinline__ bool ss_in_range(float ss) { return ss >= 0x1p-120f && ss <= 0x1p+120f; }
// S = 2^(127 - e) for the biased exponent e of m (m > 0 finite; S <= 2^127).
__device__ __forceinline__ float pow2_scale(float m) {
    const uint32_t e = min((__float_as_uint(m) >> 23) & 0xFFu, 253u);
    return __uint_as_float((254u - e) << 23);
}
// Norm and normaliser of a row from ss2 = sum of (y S)^2 over its D
// coordinates (y = H s x, unnormalised): n = ||x|| = sqrt(ss2 / D) / S and
// inv = 1 / (sqrt(D) n) = S / sqrt(ss2), so that y * inv = u.
template <int D>
__device__ __forceinline__ void scaled_norm(float ss2, float S, float& n, float& inv) {
    n = __fdiv_rn(__fsqrt_rn(ss2 * (1.0f / (float)D)), S);
    inv = __frcp_rn(__fsqrt_rn(ss2)) * S;
}
// The same for a row spread over a warp, E transformed coordinates per lane
// (call warp-uniformly).  A zero row or one with a non-finite coordinate keeps
// n and inv.
template <int D, int E>
__device__ __forceinline__ void warp_rescaled_norm(const float (&v)[E], float& n, float& inv) {
    float m = 0.f;
    bool nf = false;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float a = fabsf(v[e]);
        nf = nf || !(a <= FLT_MAX);
        m = fmaxf(m, a);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    nf = __any_sync(0xFFFFFFFFu, nf);
    if (!nf && m > 0.f) {
        const float S = pow2_scale(m);
        float t = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) t = fmaf(v[e] * S, v[e] * S, t);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
        scaled_norm<D>(t, S, n, inv);
    }
}

// Level index of w = y * inv (exact product), via the table.  The cell is
// rint(w * kLutScale) + kLutCenter, read off the mantissa of a single FMA
// with 1.5 * 2^23 (its unit in the last place is 1, so the FMA rounds the
// exact product to the nearest integer); the compare is one FMA whose sign is
// exact.  y * inv_s (inv_s = inv * kLutScale) equals w * kLutScale exactly.
__device__ __forceinline__ int bucket_lut(const LutEntry* lut, float y, float inv, float inv_s) {
    constexpr float kMagic = 12582912.0f + (float)kLutCenter;
    float f = fmaf(y, inv_s, kMagic);
    uint32_t g = __float_as_uint(f) & (uint32_t)(kLutCells - 1);
    LutEntry e = lut[g];
    float r = fmaf(y, inv, -e.thr);
    return e.lo + (r >= 0.0f ? 1 : 0);
}

// Reference bucketing by binary search over the fp32 boundaries (used where
// building the table would cost more than it saves: a few rows per launch).
template <int BITS>
__device__ __forceinline__ int bucket_search(const float* bnd, float y, float inv) {
    int idx = 0;
#pragma unroll
    for (int step = (1 << BITS) / 2; step >= 1; step >>= 1) {
        float r = fmaf(y, inv, -bnd[idx + step - 1]);
        if (r >= 0.0f) idx += step;
    }
    return idx;
}

// --------------------------------------------------------------- packing

// Pack N indices (N * BITS a multiple of 32) into N*BITS/32 words, dense
// LSB-first.
template <int N, int BITS>
__device__ __forceinline__ void pack_words(const int* idx, uint32_t* w) {
    constexpr int NW = N * BITS / 32;
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const int pos = i * BITS;
        const int wi = pos / 32, sh = pos % 32;
        w[wi] |= (uint32_t)idx[i] << sh;
        if (sh + BITS > 32) w[wi + 1] |= (uint32_t)idx[i] >> (32 - sh);
    }
}

// Extract index i (compile-time) from a word array.
template <int BITS>
__device__ __forceinline__ int unpack_one(const uint32_t* w, int i) {
    const int pos = i * BITS;
    const int wi = pos / 32, sh = pos % 32;
    uint32_t v = w[wi] >> sh;
    if (sh + BITS > 32) v |= w[wi + 1] << (32 - sh);
    return (int)(v & ((1u << BITS) - 1));
}

// Store / load `bytes` bytes (compile-time) at a pointer aligned to the
// largest power of two dividing `bytes` (at most 16).
template <int BYTES>
__device__ __forceinline__ void store_bytes(uint8_t* dst, const uint32_t* w) {
    if constexpr (BYTES % 16 == 0) {
#pragma unroll
        for (int k = 0; k < BYTES / 16; ++k)
            reinterpret_cast<uint4*>(dst)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    } else if constexpr (BYTES % 8 == 0) {
#pragma unroll
        for (int k = 0; k < BYTES / 8; ++k)
            reinterpret_cast<uint2*>(dst)[k] = make_uint2(w[2 * k], w[2 * k + 1]);
    } else if constexpr (BYTES % 4 == 0) {
#pragma unroll
        for (int k = 0; k < BYTES / 4; ++k) reinterpret_cast<uint32_t*>(dst)[k] = w[k];
    } else {
#pragma unroll
        for (int k = 0; k < BYTES; ++k) dst[k] = (uint8_t)(w[k / 4] >> (8 * (k % 4)));
    }
}

template <int BYTES>
__device__ __forceinline__ void load_bytes(const uint8_t* src, uint32_t* w) {
    if constexpr (BYTES % 16 == 0) {
#pragma unroll
        for (int k = 0; k < BYTES / 16; ++k) {
            uint4 q = __ldg(reinterpret_cast<const uint4*>(src) + k);
            w[4 * k] = q.x; w[4 * k + 1] = q.y; w[4 * k + 2] = q.z; w[4 * k + 3] = q.w;
        }
    } else if constexpr (BYTES % 8 == 0) {
#pragma unroll
        for (int k = 0; k < BYTES / 8; ++k) {
            uint2 q = __ldg(reinterpret_cast<const uint2*>(src) + k);
            w[2 * k] = q.x; w[2 * k + 1] = q.y;
        }
    } else if constexpr (BYTES % 4 == 0) {
#pragma unroll
        for (int k = 0; k < BYTES / 4; ++k) w[k] = __ldg(reinterpret_cast<const uint32_t*>(src) + k);
    } else {
#pragma unroll
        for (int k = 0; k < (BYTES + 3) / 4; ++k) w[k] = 0;
#pragma unroll
        for (int k = 0; k < BYTES; ++k) w[k / 4] |= (uint32_t)__ldg(src + k) << (8 * (k % 4));
    }
}

// ---------------------------------------------------------- one row per warp
// The row codec with one warp per row, E = d / 32 consecutive elements per
// lane, for the decode-time append of a few rows.  The transform runs over
// the element bits in registers and over the lane bits with shuffles, in the
// same bit order and with the same adds as the in-register transform; each
// index is the count of boundaries below the coordinate (the same comparison
// as the other encoders).

template <int E, typename T>
__device__ __forceinline__ void load_lane(const T* __restrict__ row, int lane, const uint32_t* sg,
                                          float (&v)[E]) {
    if constexpr (sizeof(T) == 2) {
        const uint16_t* p = reinterpret_cast<const uint16_t*>(row) + lane * E;
        uint32_t h[E];
        if constexpr (E == 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(p);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                h[2 * k] = w[k] & 0xFFFFu;
                h[2 * k + 1] = w[k] >> 16;
            }
        } else if constexpr (E == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            h[0] = u.x & 0xFFFFu;
            h[1] = u.x >> 16;
            h[2] = u.y & 0xFFFFu;
            h[3] = u.y >> 16;
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) h[e] = p[e];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = __uint_as_float((h[e] << 16) ^ sg[lane * E + e]);
    } else {
        const float* p = reinterpret_cast<const float*>(row) + lane * E;
        if constexpr (E % 4 == 0) {
#pragma unroll
            for (int k = 0; k < E / 4; ++k) {
                const float4 u = reinterpret_cast<const float4*>(p)[k];
                v[4 * k] = u.x;
                v[4 * k + 1] = u.y;
                v[4 * k + 2] = u.z;
                v[4 * k + 3] = u.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = p[e];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = __uint_as_float(__float_as_uint(v[e]) ^ sg[lane * E + e]);
    }
}

// Sign-flip, transform and bucket one row; the indices go to ib[0, D) (a
// per-warp byte buffer) and the row's L2 norm is returned.  sg: the sign masks
// in shared memory; sg2: the second sign masks in shared memory (two-sided
// signs) or null; nb = 2^bits - 1 boundaries of P are used.
template <int D, typename T>
__device__ __forceinline__ float warp_encode_indices(const T* __restrict__ row, int lane, const uint32_t* sg,
                                                     const uint32_t* sg2, const RowParams& P, int nb,
                                                     uint8_t* ib) {
    constexpr int E = D / 32;
    float v[E];
    load_lane<E, T>(row, lane, sg, v);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    fwht_reg<E>(v);
#pragma unroll
    for (int b = 1; b < 32; b <<= 1) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v[e], b);
            v[e] = (lane & b) ? o - v[e] : v[e] + o;  // (lo + hi, lo - hi)
        }
    }
    if (sg2) {  // element e of lane l is rotated coordinate l E + e
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = __uint_as_float(__float_as_uint(v[e]) ^ sg2[lane * E + e]);
    }
    float n = __fsqrt_rn(ss);
    float inv = n > 0.f ? __fdiv_rn(P.inv_sqrt_d, n) : 0.f;
    if (!ss_in_range(ss)) warp_rescaled_norm<D, E>(v, n, inv);  // warp-uniform: ss is the warp's sum
#pragma unroll
    for (int e = 0; e < E; ++e) {
        int id = 0;
        for (int j = 0; j < nb; ++j) id += fmaf(v[e], inv, -P.bnd[j]) >= 0.0f ? 1 : 0;
        ib[lane * E + e] = (uint8_t)id;
    }
    __syncwarp();
    return n;
}

// Pack the D indices of ib into the dense LSB-first stream at dst (d * bits / 8
// bytes, 4-byte aligned): lane l writes word l, stream bits [32 l, 32 l + 32).
template <int D>
__device__ __forceinline__ void warp_pack_row(const uint8_t* ib, int lane, int bits, uint8_t* dst) {
    const int rb = D * bits / 8;
    if (4 * lane < rb) {
        const int b0 = 32 * lane;
        const int i0 = b0 / bits, i1 = min(D - 1, (b0 + 31) / bits);
        uint32_t word = 0u;
        for (int i = i0; i <= i1; ++i) {
            const int sh = i * bits - b0;
            const uint32_t x = ib[i];
            word |= sh >= 0 ? x << sh : x >> -sh;
        }
        reinterpret_cast<uint32_t*>(dst)[lane] = word;
    }
}

// Unnormalised Walsh-Hadamard transform of `nvec` vectors of length D held in
// shared memory (every thread of the block takes part).
template <int D>
__device__ void fwht_smem(float* v, int nvec) {
    for (int len = 1; len < D; len <<= 1) {
        __syncthreads();
        for (int t = threadIdx.x; t < nvec * D / 2; t += blockDim.x) {
            const int vec = t / (D / 2), k = t % (D / 2);
            const int i = (k / len) * 2 * len + (k % len);
            float* x = v + vec * D;
            const float a = x[i], b = x[i + len];
            x[i] = a + b;
            x[i + len] = a - b;
        }
    }
    __syncthreads();
}

// The same transform with a warp per row: lane l holds elements l E .. l E +
// E - 1 (E = D / 32); the stages over the element bits run in registers and
// those over the lane bits by shuffles, in the order len = 1, 2, .., D/2 and
// with the same adds as fwht_smem, so the result is the same; two CTA
// barriers instead of log2(D) + 1.  Rows r, r + warps, .. go to warp r.
template <int D>
__device__ void fwht_rows_warp(float* v, int nvec) {
    constexpr int E = D / 32;
    __syncthreads();  // the rows were written by other threads
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int r = warp; r < nvec; r += nw) {  // warp-uniform
        float* x = v + r * D + lane * E;
        float e[E];
#pragma unroll
        for (int k = 0; k < E; ++k) e[k] = x[k];
        fwht_reg<E>(e);
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int k = 0; k < E; ++k) {
                const float o = __shfl_xor_sync(0xFFFFFFFFu, e[k], m);
                e[k] = upper ? o - e[k] : e[k] + o;  // (lo + hi, lo - hi)
            }
        }
#pragma unroll
        for (int k = 0; k < E; ++k) x[k] = e[k];
    }
    __syncthreads();
}

// ------------------------------------------------- query rotation (d = 128)
// One block of 128 threads rotates one query row for the tensor-core
// attention: q~ = s2 . H (s . q) / sqrt(d) (s2 only with two-sided signs),
// times the plan's query multiplier scale * log2(e) / (sqrt(d) * s_k),
// written as fp16 high and low parts (q16_row[0, 128) and [128, 256)) of the
// row divided by a power of two (*qexp_out) that keeps them below 2^14.
__device__ __forceinline__ void rotate_q_row(const __nv_bfloat16* __restrict__ q_row, __half* __restrict__ q16_row,
                                             float* __restrict__ qexp_out, const AttnParams& P) {
    __shared__ float v[128];
    __shared__ float wmax[4];
    const int j = threadIdx.x;
    const float x = __bfloat162float(q_row[j]);
    v[j] = __uint_as_float(__float_as_uint(x) ^ sign_mask(P.sgnb, j));
    fwht_smem<128>(v, 1);
    const float y = __uint_as_float(__float_as_uint(v[j]) ^ (P.two_sided ? sign_mask(P.sgn2b, j) : 0u)) * P.q_mul;
    float a = fabsf(y);
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    if ((j & 31) == 0) wmax[j >> 5] = a;
    __syncthreads();
    const float M = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    int e = 0;
    if (M > 0.f && M <= FLT_MAX) {
        int ex = 0;
        frexpf(M, &ex);  // M in [2^(ex-1), 2^ex)
        e = min(100, max(-100, ex - 14));
    }
    const float ys = ldexpf(y, -e);
    const __half hi = __float2half_rn(ys);
    const __half lo = __float2half_rn(ys - __half2float(hi));
    q16_row[j] = hi;
    q16_row[128 + j] = lo;
    if (j == 0) *qexp_out = ldexpf(1.f, e);
}

}  // namespace dev
}  // namespace tq
