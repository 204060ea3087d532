// tq_attn_generic.cu -- decode attention on the CUDA cores: head dimensions
// other than 128, and keys in the QJL residual format.
//
// "TurboQuant KV Cache Compression -- Spec", Optimization: Fused dequant-dot:
// rotate q once, score each cached position against its centroids
// ((Rq).(Rk) = q.k), accumulate V in the rotated domain, rotate the output
// back once.  Split-K flash-decode: CTA (split, KV head, sequence) handles a
// range of positions for all G = Hq/Hkv query heads of the group and writes
// fp32 partials (max m, denominator l, accumulator acc[d]); k_attn_combine
// merges the splits by log-sum-exp, normalises and un-rotates.  "CITATIONS",
// Sparse V dequant: a V row is skipped when every head's exp(sigma - m) is
// below the threshold; it still counts in l.
//
// Memory: the CTA first issues asynchronous copies of its whole range (K rows
// and norms, and, for a dense call, V rows and norms) into shared memory, so
// that every load of the range is in flight at once; the query rotation runs
// meanwhile.  With a sparse-V threshold the V rows are copied after the
// scores, and only those some head keeps.  A range holds at most 512
// positions (256 at d = 256), which keeps two CTAs resident per SM.
//
// Scores: a warp per position, lane l holding dims [l E, (l + 1) E) (E =
// d/32).  The GP partial dot products of a lane (GP = G rounded up to 2, 4 or
// 8) are summed across the warp by a reduce-scatter: each of the first
// log2(GP) shuffle steps halves the set of heads a lane carries, so the GP
// sums cost GP - 1 + 5 - log2(GP) shuffles (6 for GP = 4) instead of 5 GP.
#include <cfloat>
#include <type_traits>

#include <cuda_fp16.h>

#include "tq_async.cuh"
#include "tq_device.cuh"

namespace tq {
namespace dev {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kMaxGroup = 8;

// Cache row of position p of (sequence b, KV head g): contiguous, or through
// the block table (-1 for a page id out of range, which is not read).
template <bool PAGED>
__device__ __forceinline__ int64_t attn_row(const tq_cache_view& cache, const PagedArgs& pa, int Hkv, int b, int g,
                                            int64_t p) {
    if constexpr (PAGED) {
        const int page = __ldg(pa.bt + (int64_t)b * pa.max_pages + (p >> pa.page_shift));
        if (page < 0 || page >= pa.n_pages) return -1;
        return (((int64_t)page * Hkv + g) << pa.page_shift) + (p & ((int64_t(1) << pa.page_shift) - 1));
    } else {
        return ((int64_t)b * Hkv + g) * cache.cap + p;
    }
}

// The lane's LB <= 32 bits of a packed row in shared memory, starting at bit
// LB * lane.
template <int LB>
__device__ __forceinline__ uint32_t lane_bits_s(const uint8_t* row, int lane) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(row);
    const int bit0 = lane * LB, wi = bit0 / 32, sh = bit0 % 32;
    uint32_t x = w[wi] >> sh;
    if (sh + LB > 32) x |= w[wi + 1] << (32 - sh);
    return x;
}

// Copy granularity of a row of RB bytes: the largest of 16, 8, 4 dividing it.
__host__ __device__ constexpr int copy_unit(int rb) { return rb % 16 == 0 ? 16 : (rb % 8 == 0 ? 8 : 4); }

template <int N>
__device__ __forceinline__ void cp_async_n(uint32_t dst, const void* src) {
    if constexpr (N == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(N) : "memory");
}

// Issue the copies of positions t0 .. t0 + n - 1 of a per-position array of
// RB-byte rows (packed rows, or 4-byte norms) into dst (row t at t RB), by
// the whole block.  Rows whose page is out of range, and, with `keep`, rows
// whose flag is 0, are not copied.
template <int RB, bool PAGED>
__device__ __forceinline__ void stage_rows(uint8_t* dst, const void* src, const tq_cache_view& cache,
                                           const PagedArgs& pa, int Hkv, int b, int g, int64_t t0, int n,
                                           const uint8_t* keep) {
    constexpr int U = copy_unit(RB), PER = RB / U;
    const uint32_t base = smem_addr(dst);
    const uint8_t* s = static_cast<const uint8_t*>(src);
    for (int c = threadIdx.x; c < n * PER; c += blockDim.x) {
        const int t = c / PER, piece = c - t * PER;
        if (keep && !keep[t]) continue;
        const int64_t row = attn_row<PAGED>(cache, pa, Hkv, b, g, t0 + t);
        if (row < 0) continue;
        cp_async_n<U>(base + t * RB + piece * U, s + row * RB + piece * U);
    }
}

// Sum v[0, GP) over the warp, scattered: afterwards lane l holds the full sum
// of head head_of<GP>(l) in v[0].
template <int GP>
__device__ __forceinline__ void reduce_scatter(float (&v)[GP], int lane) {
    int c = GP;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        if (c > 1) {
            const int half = c / 2;
            const bool up = (lane & m) != 0;
#pragma unroll
            for (int j = 0; j < GP / 2; ++j) {
                if (j < half) {
                    const float send = up ? v[j] : v[j + half];
                    const float keep = up ? v[j + half] : v[j];
                    v[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
                }
            }
            c = half;
        } else {
            v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], m);
        }
    }
}

// Head whose sum lane l holds after reduce_scatter<GP>: the upper-half choices
// made at masks 16, 8, 4 (as many as log2(GP)), high bit first.
template <int GP>
__device__ __forceinline__ int head_of(int lane) {
    if constexpr (GP == 1) return 0;
    else if constexpr (GP == 2) return (lane >> 4) & 1;
    else if constexpr (GP == 4) return ((lane >> 3) & 2) | ((lane >> 3) & 1);
    else return ((lane >> 2) & 4) | ((lane >> 2) & 2) | ((lane >> 2) & 1);
}

// Thread-block clusters: the CTA's rank in its cluster, a shared-memory
// address of another CTA of the cluster, a load from it, and a barrier of
// every thread of the cluster (release / acquire).
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    // volatile: kept after the cluster barrier (also volatile); no memory
    // clobber, so the loads of several ranks are issued back to back
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The generic split kernel.  D: head dimension; KB, VB: K and V widths (for
// QJL keys KB is the total width: a (KB - 1)-bit index per coordinate, then
// d sign bits of the projected residual, with k_rnorm holding gamma; the score
// is n <q~, c[idx]> + gamma <q', sgn>, q~ the rotated scaled query and q' =
// sqrt(pi/2)/d S q~, both read from qpre, written by k_qjl_query).  PAGED:
// positions through the block table; the sequence's length is lens[b] +
// len_plus clamped to [0, ctx_len] (len_plus = 1 when lens holds the
// positions just appended).  GP: the group size rounded up (2, 4 or 8).
// CL: the splits of one (batch, KV head) form a thread-block cluster (at most
// 8); after its partial each CTA waits at a cluster barrier, and the CTA of
// rank 0 merges the partials straight from its peers' shared memory into
// out, as k_attn_combine would from the workspace; a second barrier keeps
// the peers' memory until it has.
template <int D, int KB, int VB, bool PAGED, bool QJL, int GP, bool CL = false>
__global__ void __launch_bounds__(kAttnThreads, 2)
k_attn_split(const __nv_bfloat16* __restrict__ q, int Hq, int Hkv, tq_cache_view cache, int64_t ctx_len,
             int split_len, int n_splits, float* __restrict__ ws, const __grid_constant__ AttnParams P,
             const PagedArgs pa, int len_plus, int* status, const float* __restrict__ qpre,
             const float* __restrict__ k_rnorm, float* __restrict__ out) {
    // the previous kernel in the stream may have written the cache or the
    // queries: wait for it, then let the combine be scheduled
    griddep_wait();
    griddep_launch();
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int G = Hq / Hkv;
    int64_t Ls = ctx_len;
    if constexpr (PAGED) {
        const int64_t l = (int64_t)__ldg(pa.lens + b) + len_plus;
        Ls = l < 0 ? 0 : (l < ctx_len ? l : ctx_len);
    }
    const int64_t t0 = (int64_t)split * split_len;
    const int len = (int)(Ls - t0 < 0 ? 0 : (Ls - t0 < split_len ? Ls - t0 : split_len));
    constexpr int EPL = D / 32;  // dims per lane
    constexpr int KRB = D * KB / 8, VRB = D * VB / 8;
    constexpr int MB = QJL ? KB - 1 : KB;  // index bits per key coordinate
    constexpr int KIB = D * MB / 8;        // index bytes of a key row

    extern __shared__ __align__(16) float smem[];
    float* qrot = smem;                          // [G][D]
    float* qT = qrot + kMaxGroup * D;            // [G * EPL][32]: dim l EPL + e of head h at (h EPL + e) 32 + l
    float* sc = qT + kMaxGroup * D;              // [G][split_len]: scores, then exp
    float* accs = sc + kMaxGroup * split_len;    // [G][D] cross-warp sum (QJL: the projections first)
    float* red = accs + kMaxGroup * D;           // [kAttnWarps][kMaxGroup]
    float* mh = red + kAttnWarps * kMaxGroup;    // [kMaxGroup] max per head
    float* lh = mh + kMaxGroup;                  // [kMaxGroup] denominators
    float* kcen = lh + kMaxGroup;                // [16]
    float* vcen = kcen + 16;                     // [16]
    uint8_t* ks = reinterpret_cast<uint8_t*>(vcen + 16);   // [split_len][KRB]
    uint8_t* vs = ks + split_len * KRB;                    // [split_len][VRB]
    float* kn = reinterpret_cast<float*>(vs + split_len * VRB);  // [split_len]
    float* vn = kn + split_len;                            // [split_len]
    float* kg = vn + split_len;                            // [split_len] (QJL)
    uint8_t* keep = reinterpret_cast<uint8_t*>(kg + split_len);  // [split_len] (sparse V)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!CL && len == 0) {  // block-uniform: an empty partial (in a cluster the body below gives it)
        for (int i = tid; i < G * (D + 2); i += blockDim.x) {
            const int h = i / (D + 2), j = i % (D + 2);
            ws[(((int64_t)b * Hq + g * G + h) * n_splits + split) * (D + 2) + j] = j == D ? -FLT_MAX : 0.f;
        }
        return;
    }
    const float thr = P.sparse_thr;
    const bool sparse = thr > 0.f;
    // ---- the range's copies, all in flight at once
    stage_rows<KRB, PAGED>(ks, cache.k_packed, cache, pa, Hkv, b, g, t0, len, nullptr);
    stage_rows<4, PAGED>(reinterpret_cast<uint8_t*>(kn), cache.k_norm, cache, pa, Hkv, b, g, t0, len, nullptr);
    if constexpr (QJL)
        stage_rows<4, PAGED>(reinterpret_cast<uint8_t*>(kg), k_rnorm, cache, pa, Hkv, b, g, t0, len, nullptr);
    if (!sparse) {
        stage_rows<VRB, PAGED>(vs, cache.v_packed, cache, pa, Hkv, b, g, t0, len, nullptr);
        stage_rows<4, PAGED>(reinterpret_cast<uint8_t*>(vn), cache.v_norm, cache, pa, Hkv, b, g, t0, len, nullptr);
    }
    cp_async_commit();

    if (tid < 16) {
        kcen[tid] = P.kcen[tid];
        vcen[tid] = P.vcen[tid];
    }
    if constexpr (QJL) {
        // rotated queries and their projections; the projections wait in the
        // cross-warp sum buffer, which is cleared only after pass 1
        for (int i = tid; i < G * D; i += blockDim.x) {
            const int h = i / D, j = i % D;
            const float* src = qpre + ((int64_t)b * Hq + g * G + h) * 2 * D;
            qrot[i] = src[j];
            accs[i] = src[D + j];
        }
    } else {
        // ---- rotate the group's queries: qrot = H (s . q) / sqrt(d), times scale
        for (int i = tid; i < G * D; i += blockDim.x) {
            const int h = i / D, j = i % D;
            const float x = __bfloat162float(q[((int64_t)b * Hq + g * G + h) * D + j]);
            qrot[i] = __uint_as_float(__float_as_uint(x) ^ sign_mask(P.sgnb, j));
        }
        fwht_rows_warp<D>(qrot, G);
        for (int i = tid; i < G * D; i += blockDim.x) {
            const uint32_t m = P.two_sided ? sign_mask(P.sgn2b, i % D) : 0u;
            qrot[i] = __uint_as_float(__float_as_uint(qrot[i]) ^ m) * (P.inv_sqrt_d * P.scale);
        }
    }
    __syncthreads();
    // heads past G read zeros
    for (int i = tid; i < GP * D; i += blockDim.x) {
        const int h = i / D, j = i % D;
        qT[(h * EPL + j % EPL) * 32 + j / EPL] = h < G ? qrot[i] : 0.f;
        if constexpr (QJL)
            if (h >= G) accs[i] = 0.f;
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- pass 1: sigma = n_k (q~ . c_k) (+ gamma q' . sgn), a warp per position.
    // The lane's query values (and projections) are the same for every
    // position: held in registers where they fit (the score stores into the
    // same shared array would otherwise force a reload per position).
    constexpr bool HOIST = (QJL ? 2 : 1) * GP * EPL <= 48;
    float qreg[HOIST ? GP : 1][HOIST ? EPL : 1];
    float preg[HOIST && QJL ? GP : 1][HOIST && QJL ? EPL : 1];
    if constexpr (HOIST) {
#pragma unroll
        for (int h = 0; h < GP; ++h)
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                qreg[h][e] = qT[(h * EPL + e) * 32 + lane];
                if constexpr (QJL) preg[h][e] = accs[h * D + 32 * e + lane];
            }
    }
    auto qv = [&](int h, int e) { if constexpr (HOIST) return qreg[h][e]; else return qT[(h * EPL + e) * 32 + lane]; };
    auto pv = [&](int h, int e) {
        if constexpr (HOIST && QJL) return preg[h][e]; else return accs[h * D + 32 * e + lane];
    };
    const int myh = head_of<GP>(lane);
    const bool writer = (lane & (32 / GP - 1)) == 0;
    float mloc = -FLT_MAX;
    for (int t = warp; t < len; t += kAttnWarps) {
        if constexpr (PAGED) {
            if (attn_row<PAGED>(cache, pa, Hkv, b, g, t0 + t) < 0) {  // warp-uniform: not read
                if (lane == 0) {
                    report_timeout(status, 33);
                    for (int h = 0; h < G; ++h) sc[h * split_len + t] = -FLT_MAX;
                }
                continue;
            }
        }
        const uint8_t* krow = ks + t * KRB;
        const uint32_t bits = lane_bits_s<EPL * MB>(krow, lane);
        float part[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) part[h] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float c = kcen[(bits >> (e * MB)) & ((1u << MB) - 1)];
#pragma unroll
            for (int h = 0; h < GP; ++h) part[h] = fmaf(qv(h, e), c, part[h]);
        }
        if constexpr (QJL) {
            uint32_t sw[EPL];
            if constexpr (EPL == 4 && KIB % 16 == 0) {
                const uint4 w = *reinterpret_cast<const uint4*>(krow + KIB);
                sw[0] = w.x; sw[1] = w.y; sw[2] = w.z; sw[3] = w.w;
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) sw[e] = reinterpret_cast<const uint32_t*>(krow + KIB)[e];
            }
            float sp[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) sp[h] = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                // projection k = 32 e + lane: its sign is bit `lane` of word e
                const uint32_t neg = (~sw[e] >> lane) << 31;
#pragma unroll
                for (int h = 0; h < GP; ++h) sp[h] += __uint_as_float(__float_as_uint(pv(h, e)) ^ neg);
            }
            const float nk = kn[t], gk = kg[t];
#pragma unroll
            for (int h = 0; h < GP; ++h) part[h] = fmaf(nk, part[h], gk * sp[h]);
        } else {
            const float nk = kn[t];
#pragma unroll
            for (int h = 0; h < GP; ++h) part[h] *= nk;
        }
        reduce_scatter<GP>(part, lane);
        if (writer && myh < G) {
            sc[myh * split_len + t] = part[0];
            mloc = fmaxf(mloc, part[0]);
        }
    }
    // block max per head: the writer lanes of each warp hold their head's
    if (writer && myh < G) red[warp * kMaxGroup + myh] = mloc;
    __syncthreads();
    if (tid < G) {
        float m = -FLT_MAX;
        for (int w = 0; w < kAttnWarps; ++w) m = fmaxf(m, red[w * kMaxGroup + tid]);
        mh[tid] = m;
    }
    __syncthreads();
    // ---- exp, denominators, and (sparse V) the rows some head keeps
    float lloc[kMaxGroup];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) lloc[h] = 0.f;
    for (int t = tid; t < len; t += blockDim.x) {
        float pm = 0.f;
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h)
            if (h < G) {
                const float e = __expf(sc[h * split_len + t] - mh[h]);
                sc[h * split_len + t] = e;
                lloc[h] += e;
                pm = fmaxf(pm, e);
            }
        if (sparse) keep[t] = pm >= thr ? 1 : 0;
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
    if (sparse) {  // block-uniform: copy the kept rows' V now
        stage_rows<VRB, PAGED>(vs, cache.v_packed, cache, pa, Hkv, b, g, t0, len, keep);
        stage_rows<4, PAGED>(reinterpret_cast<uint8_t*>(vn), cache.v_norm, cache, pa, Hkv, b, g, t0, len, keep);
        cp_async_commit();
        cp_async_wait_all();
    }
    __syncthreads();

    // ---- pass 2: acc += p_t * n_v * c_v in the rotated domain.  A warp takes
    // one position at a time; lane l owns elements [l*EPL, (l+1)*EPL).
    float acc[GP][EPL];
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
    int nread = 0;  // rows whose V this warp reads
    for (int t = warp; t < len; t += kAttnWarps) {
        if (sparse && !keep[t]) continue;  // warp-uniform
        if constexpr (PAGED) {
            if (attn_row<PAGED>(cache, pa, Hkv, b, g, t0 + t) < 0) continue;  // warp-uniform
        }
        ++nread;
        float p[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) p[h] = h < G ? sc[h * split_len + t] : 0.f;
        const uint32_t bitsv = lane_bits_s<EPL * VB>(vs + t * VRB, lane);
        const float nv = vn[t];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float c = vcen[(bitsv >> (e * VB)) & ((1u << VB) - 1)] * nv;
#pragma unroll
            for (int h = 0; h < GP; ++h) acc[h][e] = fmaf(p[h], c, acc[h][e]);
        }
    }
    if (P.v_rows && lane == 0 && nread > 0) atomicAdd(P.v_rows + (int64_t)b * Hkv + g, nread);
    // fixed-order cross-warp reduction: accs = ((0 + acc_0) + acc_1) + ...
    if (kAttnWarps * G <= 2 * kMaxGroup) {  // block-uniform: the warps' partials fit in qrot and qT
        // (both free since pass 1): written side by side, then summed in warp
        // order by every thread for its elements; two barriers instead of one per warp
        float* part = qrot;  // [kAttnWarps][G][D]
#pragma unroll
        for (int h = 0; h < GP; ++h)
            if (h < G)
#pragma unroll
                for (int e = 0; e < EPL; ++e) part[(warp * G + h) * D + lane * EPL + e] = acc[h][e];
        __syncthreads();
        for (int i = tid; i < G * D; i += blockDim.x) {
            float a = accs[i];
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) a += part[w * G * D + i];
            accs[i] = a;
        }
        __syncthreads();
    } else {
        for (int w = 0; w < kAttnWarps; ++w) {
            if (warp == w) {
#pragma unroll
                for (int h = 0; h < GP; ++h)
                    if (h < G)
#pragma unroll
                        for (int e = 0; e < EPL; ++e) accs[h * D + lane * EPL + e] += acc[h][e];
            }
            __syncthreads();
        }
    }
    if constexpr (!CL) {
        // ---- partials: ws[b][h][split][D + 2] = acc..., m, l
        for (int i = tid; i < G * (D + 2); i += blockDim.x) {
            const int h = i / (D + 2), j = i % (D + 2);
            const float v = j < D ? accs[h * D + j] : (j == D ? mh[h] : lh[h]);
            ws[(((int64_t)b * Hq + g * G + h) * n_splits + split) * (D + 2) + j] = v;
        }
    } else {
        // ---- merge: the same arithmetic as k_attn_combine, the splits in
        // rank order (rank = split).  Every rank merges the elements i with
        // i mod n_splits = its rank, reading the splits' accumulators from
        // their shared memory, and stores the merged values into rank 0's
        // buffer; rank 0 then rotates back and writes the output.
        __shared__ float cml[2][8][kMaxGroup];  // every split's m and l, in every rank
        if (tid < G) {  // handed to every rank before the barrier (remote stores)
            for (int r = 0; r < n_splits; ++r) {
                st_cluster_f32(cluster_map(smem_addr(&cml[0][split][tid]), (uint32_t)r), mh[tid]);
                st_cluster_f32(cluster_map(smem_addr(&cml[1][split][tid]), (uint32_t)r), lh[tid]);
            }
        }
        cluster_sync_all();  // every partial is in its CTA's shared memory, m and l in every rank's
        const int rank = (int)cluster_rank();
        float* o = qrot;  // [G][D], free since the cross-warp sum
        const uint32_t a_accs = smem_addr(accs), o0 = cluster_map(smem_addr(o), 0);
        for (int i = rank + tid * n_splits; i < G * D; i += blockDim.x * n_splits) {
            const int h = i / D, j = i % D;
            float x[8];  // the splits' accumulators, loads all in flight (ranks past the last: the last)
#pragma unroll
            for (int r = 0; r < 8; ++r)
                x[r] = ld_cluster_f32(cluster_map(a_accs + 4u * i, (uint32_t)(r < n_splits ? r : n_splits - 1)));
            float M = -FLT_MAX;
            for (int r = 0; r < n_splits; ++r) M = fmaxf(M, cml[0][r][h]);
            float L = 0.f, a = 0.f;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if (r < n_splits) {
                    const float f = __expf(cml[0][r][h] - M);
                    L = fmaf(f, cml[1][r][h], L);
                    a = fmaf(f, x[r], a);
                }
            }
            const float v = L > 0.f ? a / L : 0.f;  // a sequence with no positions gives zeros
            st_cluster_f32(o0 + 4u * i, __uint_as_float(__float_as_uint(v) ^ (P.two_sided ? sign_mask(P.sgn2b, j) : 0u)));
        }
        cluster_sync_all();  // rank 0's buffer is complete; no rank reads another's memory after this
        if (rank == 0) {
            fwht_rows_warp<D>(o, G);  // synchronises the CTA first
            for (int i = tid; i < G * D; i += blockDim.x) {
                const int h = i / D, j = i % D;
                out[((int64_t)b * Hq + g * G + h) * D + j] = __uint_as_float(__float_as_uint(o[i] * P.inv_sqrt_d) ^ sign_mask(P.sgnb, j));
            }
        }
    }
}

// Merge the splits of one (batch, query head) by log-sum-exp, normalise and
// rotate back: out = s . (H o_rot) / sqrt(d).
template <int D>
__global__ void __launch_bounds__(D) k_attn_combine(const float* __restrict__ ws, int n_splits,
                                                    float* __restrict__ out,
                                                    const __grid_constant__ AttnParams P) {
    __shared__ float o[D];
    griddep_wait();  // the split kernel's partials
    griddep_launch();
    const int bh = blockIdx.x, j = threadIdx.x;
    const float* base = ws + (int64_t)bh * n_splits * (D + 2);
    float M = -FLT_MAX;
#pragma unroll 4
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, base[s * (D + 2) + D]);
    float L = 0.f, a = 0.f;
#pragma unroll 4  // several partials' loads in flight
    for (int s = 0; s < n_splits; ++s) {
        const float f = __expf(base[s * (D + 2) + D] - M);
        L = fmaf(f, base[s * (D + 2) + D + 1], L);
        a = fmaf(f, base[s * (D + 2) + j], a);
    }
    const float v = L > 0.f ? a / L : 0.f;  // a sequence with no positions gives zeros
    o[j] = __uint_as_float(__float_as_uint(v) ^ (P.two_sided ? sign_mask(P.sgn2b, j) : 0u));
    fwht_rows_warp<D>(o, 1);
    out[(int64_t)bh * D + j] = __uint_as_float(__float_as_uint(o[j] * P.inv_sqrt_d) ^ sign_mask(P.sgnb, j));
}

// QJL keys: the rotated query of one (batch, query head), times the softmax
// scale, and its projection by the QJL matrix times sqrt(pi/2)/d, written to
// qpre[bh][0, D) and [D, 2D).  One block of D threads per head; thread k
// forms projection k from row k of S, which passes through shared memory 32
// columns at a time (read coalesced, row stride 33 floats, so that the lanes
// reading one column of 32 rows hit distinct banks).
template <int D>
__global__ void __launch_bounds__(D) k_qjl_query(const __nv_bfloat16* __restrict__ q,
                                                 const float* __restrict__ S, float* __restrict__ qpre,
                                                 const __grid_constant__ AttnParams P, float kappa) {
    __shared__ float v[D];
    __shared__ float ss[D * 33];
    griddep_wait();
    griddep_launch();
    const int bh = blockIdx.x, j = threadIdx.x;
    const float x = __bfloat162float(q[(int64_t)bh * D + j]);
    v[j] = __uint_as_float(__float_as_uint(x) ^ sign_mask(P.sgnb, j));
    fwht_rows_warp<D>(v, 1);
    const uint32_t m = P.two_sided ? sign_mask(P.sgn2b, j) : 0u;
    const float r = __uint_as_float(__float_as_uint(v[j]) ^ m) * (P.inv_sqrt_d * P.scale);
    __syncthreads();
    v[j] = r;
    __syncthreads();
    float p = 0.f;
    for (int c = 0; c < D; c += 32) {
        if (c > 0) __syncthreads();  // the previous columns' reads done
#pragma unroll 8
        for (int f = j; f < D * 32; f += D) ss[(f >> 5) * 33 + (f & 31)] = __ldg(S + (f >> 5) * D + c + (f & 31));
        __syncthreads();
#pragma unroll 8
        for (int i = 0; i < 32; ++i) p = fmaf(ss[j * 33 + i], v[c + i], p);
    }
    qpre[(int64_t)bh * 2 * D + j] = r;
    qpre[(int64_t)bh * 2 * D + D + j] = p * kappa;
}

// Dynamic shared memory of k_attn_split for a range of `split_len` positions.
template <int D, int KB, int VB>
constexpr size_t split_smem(int split_len) {
    return sizeof(float) * (kMaxGroup * D * 3 + (size_t)kMaxGroup * split_len + kAttnWarps * kMaxGroup +
                            2 * kMaxGroup + 32) +
           (size_t)split_len * (D * KB / 8 + D * VB / 8 + 3 * sizeof(float) + 1);
}

// A launch with programmatic stream serialization and, cx > 0, clusters of
// cx CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*fn)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               unsigned cx, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cx;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cx > 0 ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, static_cast<KArgs>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The split kernel, then, unless its splits merge inside their cluster, the
// combine.  A cluster launch that the device refuses (a cluster it cannot
// place) is retried without clusters.
template <int D, int KB, int VB, bool PAGED, bool QJL>
cudaError_t split_launch(const void* q, int B, int Hq, int Hkv, const tq_cache_view& cache, int64_t ctx_len,
                         float* part, float* out, const AttnGeometry& geo, const AttnParams& P, cudaStream_t s,
                         const PagedArgs& pa, int len_plus, const float* qpre, const float* k_rnorm) {
    const int G = Hq / Hkv;
    const size_t smem = split_smem<D, KB, VB>(geo.split_len);
    dim3 grid(geo.n_splits, Hkv, B);
    auto go = [&](auto fn, unsigned cx) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_pdl_cluster(fn, grid, dim3(kAttnThreads), smem, s, cx, static_cast<const __nv_bfloat16*>(q),
                                  Hq, Hkv, cache, ctx_len, geo.split_len, geo.n_splits, part, P, pa, len_plus,
                                  status_word(), qpre, k_rnorm, out);
    };
    auto pick = [&](auto cl) {
        constexpr bool C = decltype(cl)::value;
        const unsigned cx = C ? (unsigned)geo.n_splits : 0u;
        if (G <= 2) return go(k_attn_split<D, KB, VB, PAGED, QJL, 2, C>, cx);
        if (G <= 4) return go(k_attn_split<D, KB, VB, PAGED, QJL, 4, C>, cx);
        return go(k_attn_split<D, KB, VB, PAGED, QJL, 8, C>, cx);
    };
    if (geo.cluster) {
        const cudaError_t e = pick(std::true_type{});
        if (e != cudaErrorInvalidClusterSize && e != cudaErrorLaunchOutOfResources) return e;
        cudaGetLastError();  // not a sticky error: take the two-launch path
    }
    cudaError_t e = pick(std::false_type{});
    if (e != cudaSuccess) return e;
    return launch_pdl(k_attn_combine<D>, dim3(B * Hq), dim3(D), 0, s, (const float*)part, geo.n_splits, out, P);
}

template <int D, int KB, int VB, bool PAGED = false>
cudaError_t attn_launch(const void* q, int B, int Hq, int Hkv, const tq_cache_view& cache,
                        int64_t ctx_len, float* out, void* ws, const AttnGeometry& geo,
                        const AttnParams& P, cudaStream_t s, const PagedArgs& pa = PagedArgs{},
                        int len_plus = 0) {
    float* part = static_cast<float*>(ws);
    return split_launch<D, KB, VB, PAGED, false>(q, B, Hq, Hkv, cache, ctx_len, part, out, geo, P, s, pa, len_plus,
                                                 nullptr, nullptr);
}

// QJL keys (contiguous cache): the query prologue, the split kernel with QJL
// scoring over the workspace after the prologue's qpre, and (without
// clusters) the combine.
template <int D, int KB, int VB>
cudaError_t attn_qjl_launch(const void* q, const float* S, int B, int Hq, int Hkv, const tq_cache_view& cache,
                            const float* k_rnorm, int64_t ctx_len, float* out, void* ws, const AttnGeometry& geo,
                            const AttnParams& P, cudaStream_t s) {
    float* qpre = static_cast<float*>(ws);
    float* part = qpre + attn_qjl_prefix_floats(B, Hq, D);
    cudaError_t e = launch_pdl(k_qjl_query<D>, dim3(B * Hq), dim3(D), 0, s, static_cast<const __nv_bfloat16*>(q), S,
                               qpre, P, (float)(1.2533141373155003 / D));
    if (e != cudaSuccess) return e;
    return split_launch<D, KB, VB, false, true>(q, B, Hq, Hkv, cache, ctx_len, part, out, geo, P, s, PagedArgs{}, 0,
                                                qpre, k_rnorm);
}

}  // namespace dev

#if !defined(TQ_UNIT_D) || !defined(TQ_UNIT_KB)
#error "compile once per head dimension and K width with -DTQ_UNIT_D=<d> -DTQ_UNIT_KB=<bits>"
#endif

#if TQ_UNIT_D != 128
// Head dimensions other than 128: contiguous and paged caches.
template <int D, int KB>
cudaError_t launch_attn_dk(int v_bits, const void* q, int B, int Hq, int Hkv, const tq_cache_view& cache,
                           int64_t ctx_len, float* out, void* workspace, const AttnGeometry& g, const AttnParams& P,
                           cudaStream_t s) {
    switch (v_bits) {
        case 2: return dev::attn_launch<D, KB, 2>(q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, P, s);
        case 3: return dev::attn_launch<D, KB, 3>(q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, P, s);
        default: return dev::attn_launch<D, KB, 4>(q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, P, s);
    }
}
template cudaError_t launch_attn_dk<TQ_UNIT_D, TQ_UNIT_KB>(int, const void*, int, int, int, const tq_cache_view&,
                                                           int64_t, float*, void*, const AttnGeometry&,
                                                           const AttnParams&, cudaStream_t);

// len_plus = 1 when pa.lens holds the positions just appended.
template <int D, int KB>
cudaError_t launch_attn_generic_paged(int v_bits, const void* q, int B, int Hq, int Hkv,
                                      const tq_cache_view& pages, int64_t max_ctx, float* out, void* workspace,
                                      const AttnGeometry& g, const AttnParams& P, const PagedArgs& pa,
                                      int len_plus, cudaStream_t s) {
    switch (v_bits) {
        case 2: return dev::attn_launch<D, KB, 2, true>(q, B, Hq, Hkv, pages, max_ctx, out, workspace, g, P, s, pa, len_plus);
        case 3: return dev::attn_launch<D, KB, 3, true>(q, B, Hq, Hkv, pages, max_ctx, out, workspace, g, P, s, pa, len_plus);
        default: return dev::attn_launch<D, KB, 4, true>(q, B, Hq, Hkv, pages, max_ctx, out, workspace, g, P, s, pa, len_plus);
    }
}
template cudaError_t launch_attn_generic_paged<TQ_UNIT_D, TQ_UNIT_KB>(int, const void*, int, int, int,
                                                                       const tq_cache_view&, int64_t, float*, void*,
                                                                       const AttnGeometry&, const AttnParams&,
                                                                       const PagedArgs&, int, cudaStream_t);
#endif

#if TQ_UNIT_D <= 128
template <int D, int KB>
cudaError_t launch_attn_qjl(int v_bits, const void* q, const float* S, int B, int Hq, int Hkv,
                            const tq_cache_view& cache, const float* k_rnorm, int64_t ctx_len, float* out,
                            void* workspace, const AttnGeometry& g, const AttnParams& P, cudaStream_t s) {
    switch (v_bits) {
        case 2: return dev::attn_qjl_launch<D, KB, 2>(q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, P, s);
        case 3: return dev::attn_qjl_launch<D, KB, 3>(q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, P, s);
        default: return dev::attn_qjl_launch<D, KB, 4>(q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, P, s);
    }
}
template cudaError_t launch_attn_qjl<TQ_UNIT_D, TQ_UNIT_KB>(int, const void*, const float*, int, int, int,
                                                            const tq_cache_view&, const float*, int64_t, float*,
                                                            void*, const AttnGeometry&, const AttnParams&,
                                                            cudaStream_t);
#endif

}  // namespace tq
