// tq_attn.cu -- decode attention over the packed cache, in the rotated domain.
//
// "TurboQuant KV Cache Compression -- Spec", Optimization: Fused dequant-dot:
// rotate q once, score each cached position against its centroids
// ((Rq).(Rk) = q.k), accumulate V in the rotated domain, rotate the output
// back once.  Split-K flash-decode: CTA (split, kv head, batch) handles a
// contiguous range of positions for all Hq/Hkv query heads of the GQA group
// and writes fp32 partials (running max m, denominator l, accumulator acc[d]);
// a second kernel merges the splits by log-sum-exp, normalises and
// un-rotates.  "CITATIONS", Sparse V dequant: a V row is skipped when every
// head's exp(sigma - m) is below the threshold; it still counts in l.
#include <cfloat>

#include <cuda_fp16.h>

#include "tq_device.cuh"

namespace tq {
namespace dev {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kMaxGroup = 8;

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

template <int BITS, int D>
__device__ __forceinline__ void load_packed_row(const uint8_t* p, uint32_t (&w)[(D * BITS + 31) / 32]) {
    load_bytes<D * BITS / 8>(p, w);
}

template <int D, int KB, int VB>
__global__ void __launch_bounds__(kAttnThreads)
k_attn_split(const __nv_bfloat16* __restrict__ q, int Hq, int Hkv, tq_cache_view cache,
             int64_t ctx_len, int split_len, int n_splits, float* __restrict__ ws,
             const __grid_constant__ AttnParams P) {
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = Hq / Hkv;
    const int64_t t0 = (int64_t)split * split_len;
    const int len = (int)min((int64_t)split_len, ctx_len - t0);

    extern __shared__ float smem[];
    float* qrot = smem;                          // [G][D]
    float* sc = qrot + kMaxGroup * D;            // [G][split_len]: scores, then exp
    float* accs = sc + kMaxGroup * split_len;    // [G][D] cross-warp sum
    float* red = accs + kMaxGroup * D;           // [kAttnWarps][kMaxGroup]
    float* mh = red + kAttnWarps * kMaxGroup;    // [kMaxGroup] max per head
    float* lh = mh + kMaxGroup;                  // [kMaxGroup] denominators
    float* kcen = lh + kMaxGroup;                // [16]
    float* vcen = kcen + 16;                     // [16]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 16) {
        kcen[tid] = P.kcen[tid];
        vcen[tid] = P.vcen[tid];
    }
    // ---- rotate the group's queries: qrot = H (s . q) / sqrt(d), times scale
    for (int i = tid; i < G * D; i += blockDim.x) {
        const int h = i / D, j = i % D;
        const float x = __bfloat162float(q[((int64_t)b * Hq + g * G + h) * D + j]);
        qrot[i] = __uint_as_float(__float_as_uint(x) ^ P.sgn[j]);
    }
    fwht_smem<D>(qrot, G);
    for (int i = tid; i < G * D; i += blockDim.x) qrot[i] *= P.inv_sqrt_d * P.scale;
    __syncthreads();

    const int64_t row0 = ((int64_t)b * Hkv + g) * cache.cap + t0;
    constexpr int KRB = D * KB / 8, VRB = D * VB / 8;

    // ---- pass 1: scores sigma = n_k * (qrot . c_k) for every position
    float mloc[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) mloc[h] = -FLT_MAX;
    for (int t = tid; t < len; t += blockDim.x) {
        uint32_t w[(D * KB + 31) / 32];
        load_packed_row<KB, D>(cache.k_packed + (row0 + t) * KRB, w);
        const float nk = __ldg(cache.k_norm + row0 + t);
        float acc[kMaxGroup];
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) acc[h] = 0.f;
#pragma unroll
        for (int j = 0; j < D; ++j) {
            const float c = kcen[unpack_one<KB>(w, j)];
#pragma unroll
            for (int h = 0; h < kMaxGroup; ++h)
                if (h < G) acc[h] = fmaf(qrot[h * D + j], c, acc[h]);
        }
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h)
            if (h < G) {
                const float s = acc[h] * nk;
                sc[h * split_len + t] = s;
                mloc[h] = fmaxf(mloc[h], s);
            }
    }
    // block max per head
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
        float m = mloc[h];
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) red[warp * kMaxGroup + h] = m;
    }
    __syncthreads();
    if (tid < kMaxGroup) {
        float m = -FLT_MAX;
        for (int w = 0; w < kAttnWarps; ++w) m = fmaxf(m, red[w * kMaxGroup + tid]);
        mh[tid] = m;
    }
    __syncthreads();
    // ---- exp and denominators
    float lloc[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) lloc[h] = 0.f;
    for (int t = tid; t < len; t += blockDim.x) {
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h)
            if (h < G) {
                const float e = __expf(sc[h * split_len + t] - mh[h]);
                sc[h * split_len + t] = e;
                lloc[h] += e;
            }
    }
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
        float l = lloc[h];
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
        if (lane == 0) red[warp * kMaxGroup + h] = l;
    }
    __syncthreads();
    if (tid < kMaxGroup) {
        float l = 0.f;
        for (int w = 0; w < kAttnWarps; ++w) l += red[w * kMaxGroup + tid];
        lh[tid] = l;
    }
    for (int i = tid; i < G * D; i += blockDim.x) accs[i] = 0.f;
    __syncthreads();

    // ---- pass 2: acc += p_t * n_v * c_v in the rotated domain.  A warp takes
    // one position at a time; lane l owns elements [l*EPL, (l+1)*EPL).
    constexpr int EPL = D / 32;
    constexpr int LBITS = EPL * VB;  // bits per lane per row (<= 32)
    float acc[kMaxGroup][EPL];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
    const float thr = P.sparse_thr;
    for (int t = warp; t < len; t += kAttnWarps) {
        float pm = 0.f;
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h)
            if (h < G) pm = fmaxf(pm, sc[h * split_len + t]);
        if (pm < thr) continue;  // warp-uniform
        const uint8_t* vr = cache.v_packed + (row0 + t) * VRB;
        const int bit0 = lane * LBITS;
        const uint32_t* vw = reinterpret_cast<const uint32_t*>(vr);
        const int wi = bit0 / 32, sh = bit0 % 32;
        uint32_t bitsv = __ldg(vw + wi) >> sh;
        if (sh + LBITS > 32) bitsv |= __ldg(vw + wi + 1) << (32 - sh);
        const float nv = __ldg(cache.v_norm + row0 + t);
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float c = vcen[(bitsv >> (e * VB)) & ((1u << VB) - 1)] * nv;
#pragma unroll
            for (int h = 0; h < kMaxGroup; ++h)
                if (h < G) acc[h][e] = fmaf(sc[h * split_len + t], c, acc[h][e]);
        }
    }
    // fixed-order cross-warp reduction
    for (int w = 0; w < kAttnWarps; ++w) {
        if (warp == w) {
#pragma unroll
            for (int h = 0; h < kMaxGroup; ++h)
                if (h < G)
#pragma unroll
                    for (int e = 0; e < EPL; ++e) accs[h * D + lane * EPL + e] += acc[h][e];
        }
        __syncthreads();
    }
    // ---- partials: ws[b][h][split][D + 2] = acc..., m, l
    for (int i = tid; i < G * (D + 2); i += blockDim.x) {
        const int h = i / (D + 2), j = i % (D + 2);
        const float v = j < D ? accs[h * D + j] : (j == D ? mh[h] : lh[h]);
        ws[(((int64_t)b * Hq + g * G + h) * n_splits + split) * (D + 2) + j] = v;
    }
}

// Merge the splits of one (batch, query head) by log-sum-exp, normalise and
// rotate back: out = s . (H o_rot) / sqrt(d).
template <int D>
__global__ void __launch_bounds__(D) k_attn_combine(const float* __restrict__ ws, int n_splits,
                                                    float* __restrict__ out,
                                                    const __grid_constant__ AttnParams P) {
    __shared__ float o[D];
    const int bh = blockIdx.x, j = threadIdx.x;
    const float* base = ws + (int64_t)bh * n_splits * (D + 2);
    float M = -FLT_MAX;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, base[s * (D + 2) + D]);
    float L = 0.f, a = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const float f = __expf(base[s * (D + 2) + D] - M);
        L = fmaf(f, base[s * (D + 2) + D + 1], L);
        a = fmaf(f, base[s * (D + 2) + j], a);
    }
    o[j] = a / L;
    fwht_smem<D>(o, 1);
    out[(int64_t)bh * D + j] = __uint_as_float(__float_as_uint(o[j] * P.inv_sqrt_d) ^ P.sgn[j]);
}

// ============================================================ v2, d = 128
//
// Tensor-core flash-decode (mma.sync m16n8k16, fp16 operands, fp32
// accumulation).  Per warp and 16-position tile:
//   S = Q K^T   rows = the G query heads of the group (padded to 16), columns =
//               8 positions per MMA; A = q (rotated once, scaled by
//               scale*log2(e), fp16, in registers), B = K centroids straight
//               from a lane-replicated shared table.  The 128 contraction dims
//               are permuted so that lane t reads one contiguous chunk (dims
//               32t..32t+31) of each K row; q is loaded with the same
//               permutation, and a dot product does not depend on the order.
//   softmax     exp2 with a lazily updated running max (rescale only when the
//               tile max exceeds it by more than kLazy, or at once when norms
//               are large), fp32 denominators.
//   O += P V    the S accumulators are exactly the A fragments of P (heads x
//               positions); V rows are dequantised by the warp into a
//               swizzled shared tile (16 x 128 fp16) and read with
//               ldmatrix.trans; the V norm is folded into P.
// Work items (batch, KV head, 512-position split) are spread over persistent
// CTAs of 4 warps; each warp owns 128 positions and writes its own partial
// (acc[128], m, l) with m in log2 units; a combine kernel merges them.

constexpr int kA2Warps = 4;
constexpr int kA2Threads = 32 * kA2Warps;
constexpr int kA2WarpPos = 128;
constexpr int kA2Split = kA2Warps * kA2WarpPos;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;  // log2 units: p <= 256 before a forced rescale

template <int BITS>
struct PairTable {  // (2*BITS)-bit index -> two fp16 centroids of consecutive dims
    static constexpr int kEntries = 1 << (2 * BITS);
};

__device__ __forceinline__ uint32_t h2u(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// table[e * 32 + lane] = (c[e & m], c[e >> BITS]): one copy per lane, so a
// warp's lookups never collide in a bank.
template <int BITS>
__device__ void fill_pair_table(uint32_t* t, const float* cen) {
    constexpr int N = PairTable<BITS>::kEntries, M = (1 << BITS) - 1;
    for (int i = threadIdx.x; i < N * 32; i += blockDim.x) {
        const int e = i >> 5;
        t[i] = h2u(cen[e & M], cen[(e >> BITS) & M]);
    }
}

// Pair p of a bit stream held in words w: bits [p*2*BITS, p*2*BITS + 2*BITS).
template <int BITS>
__device__ __forceinline__ uint32_t pair_at(const uint32_t* w, int p) {
    constexpr int PB = 2 * BITS;
    const int pos = p * PB, wi = pos / 32, sh = pos % 32;
    uint32_t x;
    if (sh + PB <= 32) x = w[wi] >> sh;
    else x = __funnelshift_r(w[wi], w[wi + 1], sh);
    return x & ((1u << PB) - 1);
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <int BYTES>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t* w) {
    load_bytes<BYTES>(p, w);
}

// q rotation: q16[b][h][j] = fp16( (H (s . q) / sqrt(d))_j * scale * log2(e) )
static __global__ void __launch_bounds__(128) k_attn_qrot(const __nv_bfloat16* __restrict__ q,
                                                   __half* __restrict__ q16,
                                                   const __grid_constant__ AttnParams P) {
    __shared__ float v[128];
    const int bh = blockIdx.x, j = threadIdx.x;
    const float x = __bfloat162float(q[(int64_t)bh * 128 + j]);
    v[j] = __uint_as_float(__float_as_uint(x) ^ P.sgn[j]);
    fwht_smem<128>(v, 1);
    q16[(int64_t)bh * 128 + j] = __float2half_rn(v[j] * (P.inv_sqrt_d * P.scale * kLog2e));
}

template <int KB, int VB>
struct A2Smem {
    static constexpr int kKTable = PairTable<KB>::kEntries * 32 * 4;
    static constexpr int kVTable = PairTable<VB>::kEntries * 32 * 4;
    static constexpr int kVTile = 16 * 128 * 2;  // per warp
    static constexpr int kBytes = kKTable + kVTable + kA2Warps * kVTile;
};

template <int KB, int VB>
__global__ void __launch_bounds__(kA2Threads)
k_attn2_split(const __half* __restrict__ q16, int Hq, int Hkv, tq_cache_view cache,
              int64_t ctx_len, int n_splits, int64_t n_items, float* __restrict__ part,
              const __grid_constant__ AttnParams P) {
    constexpr int D = 128;
    constexpr int KRB = D * KB / 8, VRB = D * VB / 8;
    constexpr int KCH = 4 * KB;  // bytes of a K row per lane (32 dims)
    constexpr int VCH = 8 * VB;  // bytes of a V row per lane (64 dims)
    extern __shared__ __align__(128) unsigned char a2_smem[];
    uint32_t* ktab = reinterpret_cast<uint32_t*>(a2_smem);
    uint32_t* vtab = reinterpret_cast<uint32_t*>(a2_smem + A2Smem<KB, VB>::kKTable);
    unsigned char* vtiles = a2_smem + A2Smem<KB, VB>::kKTable + A2Smem<KB, VB>::kVTable;
    fill_pair_table<KB>(ktab, P.kcen);
    fill_pair_table<VB>(vtab, P.vcen);
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int G = Hq / Hkv;
    const int n_parts = n_splits * kA2Warps;
    const uint32_t* kt = ktab + lane;
    const uint32_t* vt = vtab + lane;
    unsigned char* vtile = vtiles + warp * A2Smem<KB, VB>::kVTile;
    const uint32_t vtile_s = static_cast<uint32_t>(__cvta_generic_to_shared(vtile));
    const float thr = P.sparse_thr;
    const bool head_ok = g < G;

    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int split = (int)(item % n_splits);
        const int64_t bh = item / n_splits;
        const int gh = (int)(bh % Hkv);
        const int64_t b = bh / Hkv;
        const int64_t start = (int64_t)split * kA2Split + warp * kA2WarpPos;
        const int64_t end = min(start + kA2WarpPos, ctx_len);
        const int head = gh * G + g;  // query head of this lane's row (if g < G)
        float* out = part + (((b * Hq + head) * n_parts) + (int64_t)split * kA2Warps + warp) * (D + 2);

        float O[16][4];
#pragma unroll
        for (int j = 0; j < 16; ++j) O[j][0] = O[j][1] = O[j][2] = O[j][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;

        if (start < end) {
            // q fragments (permuted dims): qa[kk] = q[32t+4kk .. +1], qb[kk] = q[32t+4kk+2 .. +3]
            uint32_t qa[8], qb[8];
            if (head_ok) {
                const uint2* qp = reinterpret_cast<const uint2*>(q16 + (b * Hq + head) * D + 32 * t);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint2 u = __ldg(qp + kk);
                    qa[kk] = u.x;
                    qb[kk] = u.y;
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) qa[kk] = qb[kk] = 0u;
            }
            const int64_t row0 = (b * Hkv + gh) * cache.cap;
            const uint8_t* kbase = cache.k_packed + row0 * KRB + KCH * t;
            const float* knorm = cache.k_norm + row0;
            const float* vnorm = cache.v_norm + row0;

            for (int64_t t0 = start; t0 < end; t0 += 16) {
                // ---- scores for 16 positions (two n-tiles of 8)
                float sc[2][2];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int64_t pk = min(t0 + 8 * nt + g, end - 1);
                    uint32_t kw[KB];
                    load_words<KCH>(kbase + pk * KRB, kw);
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t b0 = kt[pair_at<KB>(kw, 2 * kk) * 32];
                        const uint32_t b1 = kt[pair_at<KB>(kw, 2 * kk + 1) * 32];
                        mma16816(acc, qa[kk], 0u, qb[kk], 0u, b0, b1);
                    }
                    sc[nt][0] = acc[0];
                    sc[nt][1] = acc[1];
                }
                // positions of this lane's scores: t0 + 8nt + 2t + e
                float nk[2][2], nv[2][2];
                bool ok[2][2];
                float tmax = -INFINITY, nvmax = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int64_t ps = t0 + 8 * nt + 2 * t + e;
                        ok[nt][e] = ps < end;
                        const int64_t pc = ok[nt][e] ? ps : end - 1;
                        nk[nt][e] = __ldg(knorm + pc);
                        nv[nt][e] = __ldg(vnorm + pc);
                        sc[nt][e] = ok[nt][e] ? sc[nt][e] * nk[nt][e] : -INFINITY;
                        tmax = fmaxf(tmax, sc[nt][e]);
                        nvmax = fmaxf(nvmax, nv[nt][e]);
                    }
                tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 1));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, 2));
                // Rescale when this tile's max runs ahead of the running max by
                // more than kLazy, or at all when large V norms could push
                // p * n_v past the fp16 range.
                const float lazy = nvmax > 200.f ? 0.f : kLazy;
                const bool need = head_ok && tmax > m_run + lazy;
                if (__any_sync(0xFFFFFFFFu, need)) {
                    const float m_new = fmaxf(m_run, tmax);
                    const float alpha = fast_exp2(m_run - m_new);  // m_run = -inf -> 0
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        O[j][0] *= alpha;
                        O[j][1] *= alpha;
                    }
                    l_run *= alpha;
                    m_run = m_new;
                }
                float p[2][2];
                float pmax = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        p[nt][e] = (head_ok && ok[nt][e]) ? fast_exp2(sc[nt][e] - m_run) : 0.f;
                        l_run += p[nt][e];
                        pmax = fmaxf(pmax, p[nt][e]);
                    }
                // sparse-V: skip the tile's V rows when no head of the group
                // reaches the threshold anywhere in the tile
                if (!__any_sync(0xFFFFFFFFu, pmax >= thr)) continue;
                const uint32_t pa0 = h2u(p[0][0] * nv[0][0], p[0][1] * nv[0][1]);
                const uint32_t pa2 = h2u(p[1][0] * nv[1][0], p[1][1] * nv[1][1]);

                // ---- V tile: lane -> position (lane & 15), dims 64*(lane >> 4) .. +63
                {
                    const int vp = lane & 15, hh = lane >> 4;
                    const int64_t pv = min(t0 + vp, end - 1);
                    uint32_t vw[VCH / 4 + 1];
                    load_words<VCH>(cache.v_packed + (row0 + pv) * VRB + VCH * hh, vw);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {  // 8 chunks of 8 dims
                        uint4 q4;
                        q4.x = vt[pair_at<VB>(vw, 4 * c + 0) * 32];
                        q4.y = vt[pair_at<VB>(vw, 4 * c + 1) * 32];
                        q4.z = vt[pair_at<VB>(vw, 4 * c + 2) * 32];
                        q4.w = vt[pair_at<VB>(vw, 4 * c + 3) * 32];
                        const int chunk = 8 * hh + c;
                        *reinterpret_cast<uint4*>(vtile + vp * 256 + ((chunk ^ (vp & 7)) << 4)) = q4;
                    }
                }
                __syncwarp();
                // ---- O += P V over 16 n-tiles of 8 dims
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = lane;
                    const int pos = ((i >> 3) & 1) * 8 + (i & 7);
                    const int chunk = 2 * j + (i >> 4);
                    uint32_t r[4];
                    ldsm_x4_trans(r, vtile_s + pos * 256 + ((chunk ^ (pos & 7)) << 4));
                    mma16816(O[2 * j], pa0, 0u, pa2, 0u, r[0], r[1]);
                    mma16816(O[2 * j + 1], pa0, 0u, pa2, 0u, r[2], r[3]);
                }
                __syncwarp();
            }
        }
        l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 1);
        l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 2);
        if (head_ok) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                *reinterpret_cast<float2*>(out + 8 * j + 2 * t) = make_float2(O[j][0], O[j][1]);
            if (t == 0) {
                out[D] = m_run;
                out[D + 1] = l_run;
            }
        }
    }
}

// Merge the partials of one (batch, query head) (m in log2 units), normalise
// and rotate back.
static __global__ void __launch_bounds__(128) k_attn2_combine(const float* __restrict__ part, int n_parts,
                                                       float* __restrict__ out,
                                                       const __grid_constant__ AttnParams P) {
    __shared__ float o[128];
    const int bh = blockIdx.x, j = threadIdx.x;
    const float* base = part + (int64_t)bh * n_parts * 130;
    float M = -INFINITY;
    for (int s = 0; s < n_parts; ++s) M = fmaxf(M, base[s * 130 + 128]);
    float L = 0.f, a = 0.f;
    for (int s = 0; s < n_parts; ++s) {
        const float ms = base[s * 130 + 128];
        const float f = ms == -INFINITY ? 0.f : fast_exp2(ms - M);
        L = fmaf(f, base[s * 130 + 129], L);
        a = fmaf(f, base[s * 130 + j], a);
    }
    o[j] = a / L;
    fwht_smem<128>(o, 1);
    out[(int64_t)bh * 128 + j] = __uint_as_float(__float_as_uint(o[j] * P.inv_sqrt_d) ^ P.sgn[j]);
}

template <int KB, int VB>
cudaError_t attn2_launch(const void* q, int B, int Hq, int Hkv, const tq_cache_view& cache,
                         int64_t ctx_len, float* out, void* ws, const AttnGeometry& geo,
                         const AttnParams& P, cudaStream_t s) {
    __half* q16 = static_cast<__half*>(ws);
    float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + attn2_q16_bytes(B, Hq));
    k_attn_qrot<<<B * Hq, 128, 0, s>>>(static_cast<const __nv_bfloat16*>(q), q16, P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto fn = k_attn2_split<KB, VB>;
    constexpr int smem = A2Smem<KB, VB>::kBytes;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void*)fn, kA2Threads, smem) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int64_t items = (int64_t)B * Hkv * geo.n_splits;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > items) grid = items;
    fn<<<(unsigned)grid, kA2Threads, smem, s>>>(q16, Hq, Hkv, cache, ctx_len, geo.n_splits, items, part, P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_attn2_combine<<<B * Hq, 128, 0, s>>>(part, geo.n_splits * kA2Warps, out, P);
    return cudaGetLastError();
}

template <int D, int KB, int VB>
cudaError_t attn_launch(const void* q, int B, int Hq, int Hkv, const tq_cache_view& cache,
                        int64_t ctx_len, float* out, void* ws, const AttnGeometry& geo,
                        const AttnParams& P, cudaStream_t s) {
    auto fn = k_attn_split<D, KB, VB>;
    const size_t smem = sizeof(float) * (kMaxGroup * D * 2 + (size_t)kMaxGroup * geo.split_len +
                                         kAttnWarps * kMaxGroup + 2 * kMaxGroup + 32);
    dim3 grid(geo.n_splits, Hkv, B);
    fn<<<grid, kAttnThreads, smem, s>>>(static_cast<const __nv_bfloat16*>(q), Hq, Hkv, cache, ctx_len,
                                       geo.split_len, geo.n_splits, static_cast<float*>(ws), P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_attn_combine<D><<<B * Hq, D, 0, s>>>(static_cast<const float*>(ws), geo.n_splits, out, P);
    return cudaGetLastError();
}

template <int D, int KB>
cudaError_t attn_vb(int vb, const void* q, int B, int Hq, int Hkv, const tq_cache_view& c,
                    int64_t ctx, float* out, void* ws, const AttnGeometry& geo, const AttnParams& P,
                    cudaStream_t s) {
    if constexpr (D == 128) {
        switch (vb) {
            case 2: return attn2_launch<KB, 2>(q, B, Hq, Hkv, c, ctx, out, ws, geo, P, s);
            case 3: return attn2_launch<KB, 3>(q, B, Hq, Hkv, c, ctx, out, ws, geo, P, s);
            default: return attn2_launch<KB, 4>(q, B, Hq, Hkv, c, ctx, out, ws, geo, P, s);
        }
    }
    switch (vb) {
        case 2: return attn_launch<D, KB, 2>(q, B, Hq, Hkv, c, ctx, out, ws, geo, P, s);
        case 3: return attn_launch<D, KB, 3>(q, B, Hq, Hkv, c, ctx, out, ws, geo, P, s);
        default: return attn_launch<D, KB, 4>(q, B, Hq, Hkv, c, ctx, out, ws, geo, P, s);
    }
}

}  // namespace dev

template <int D, int KB>
cudaError_t launch_attn_dk(int v_bits, const void* q, int B, int Hq, int Hkv,
                           const tq_cache_view& cache, int64_t ctx_len, float* out, void* workspace,
                           const AttnGeometry& g, const AttnParams& P, cudaStream_t s) {
    return dev::attn_vb<D, KB>(v_bits, q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, P, s);
}

#if !defined(TQ_UNIT_D) || !defined(TQ_UNIT_KB)
#error "compile once per head dimension and K width with -DTQ_UNIT_D=<d> -DTQ_UNIT_KB=<bits>"
#endif
template cudaError_t launch_attn_dk<TQ_UNIT_D, TQ_UNIT_KB>(int, const void*, int, int, int,
                                                           const tq_cache_view&, int64_t, float*,
                                                           void*, const AttnGeometry&,
                                                           const AttnParams&, cudaStream_t);

}  // namespace tq
