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
