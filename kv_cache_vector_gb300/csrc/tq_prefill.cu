// tq_prefill.cu -- prefill (multi-query, causal) attention over the packed
// cache, d = 128, on the 5th-generation tensor cores.
//
// A chunk of T query tokens per sequence, token t at absolute position
// q_start[b] + t, each attending over positions [0, q_start[b] + t] of its
// KV head: the decode attention of "TurboQuant KV Cache Compression --
// Spec" (Optimization: Fused dequant-dot -- scores against the centroids in
// the rotated domain, V accumulated rotated, one inverse rotation of the
// output) with many queries per KV head, which turns both contractions into
// dense matrix products.
//
// One CTA of four warps takes 128 query rows of one (sequence, KV head):
// 128 / G consecutive tokens times the G query heads of the group (row r =
// token (r / G), head (r % G)).  Per block of 128 KV positions:
//   1. the packed K and V rows and their norms are staged in shared memory;
//   2. the threads turn K into fp16 centroids c * s_k (a 128 x 128 tile in
//      the 128-byte-swizzled K-major layout; lookups in a table of centroid
//      pairs of two consecutive dims);
//   3. one thread issues S = Q_hi K^T + Q_lo K^T (tcgen05.mma kind::f16, fp32
//      accumulator in tensor memory): the rotated query is split into fp16
//      high and low parts, so it keeps about 22 significant bits;
//   4. meanwhile the threads turn V into fp16 centroids c * s_v, transposed
//      (positions contiguous per dim; lookups in a table of centroid pairs of
//      two consecutive positions);
//   5. each thread reads its row of S from tensor memory, applies the query's
//      power-of-two scale, the K norms and the causal mask, and updates its
//      running max and denominator (log2 units); P = exp2(s - m) times the V
//      norm over 2^E (E fixed per CTA from the largest V norm it reads, so P
//      <= 1) goes to shared memory as fp16 high and low parts;
//   6. one thread issues O_blk = P_hi V + P_lo V into tensor memory; each
//      thread folds its row into the running output held in registers,
//      O = O * exp2(m_old - m_new) + O_blk.
// At the end the row is divided by the denominator, scaled by 2^E / s_v and
// rotated back (s . H (s2 . o) / sqrt(d)) in registers.
//
// Every wait on an mbarrier is bounded (2 s); a wait that gives up sets the
// device status word, the CTA stops, waits (bounded) for its MMAs in flight,
// frees its tensor memory and returns.
#include <cfloat>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_async.cuh"
#include "tq_device.cuh"
#include "tq_umma.cuh"

namespace tq {
namespace dev {

constexpr int kPfRows = 128;   // query rows per CTA
constexpr int kPfBlock = 128;  // KV positions per block
// shared memory, offsets from a 1024-aligned base
constexpr uint32_t kPfQH = 0;          // Q high parts, 128 x 128 fp16
constexpr uint32_t kPfQL = 32768;      // Q low parts
constexpr uint32_t kPfKT = 65536;      // K centroids of the block, [position][dim]
constexpr uint32_t kPfVT = 98304;      // V centroids of the block, [dim][position]
constexpr uint32_t kPfPH = 131072;     // P high parts, [row][position]
constexpr uint32_t kPfPL = 163840;     // P low parts
constexpr uint32_t kPfKS = 196608;     // packed K rows of the block, 64-byte stride
constexpr uint32_t kPfVS = 204800;     // packed V rows
constexpr uint32_t kPfKN = 212992;     // K norms of the block (128 floats)
constexpr uint32_t kPfVN = 213504;     // V norms
constexpr uint32_t kPfTK = 214016;     // K pair table (up to 256 words)
constexpr uint32_t kPfTV = 215040;     // V pair table
constexpr uint32_t kPfBar = 216064;    // two mbarriers
constexpr uint32_t kPfMisc = 216080;   // tensor-memory base, reduction scratch
constexpr uint32_t kPfEnd = 216128;
constexpr uint32_t kPfSmem = kPfEnd + 1024;  // plus alignment slack
constexpr int kPfStatusWait = 51;      // an MMA completion wait gave up
constexpr int kPfStatusRange = 52;     // q_start[b] + T exceeds the cache capacity, or q_start < 0

// Offset of the 16-byte chunk holding elements [8 k8, 8 k8 + 8) of `row` in a
// 128 x 128 fp16 K-major tile with the 128-byte swizzle (two 64-column
// halves of 16 KB, rows of 128 bytes, chunk index xor row % 8).
__device__ __forceinline__ uint32_t pf_chunk(int row, int k8) {
    return (uint32_t)((k8 >> 3) * 16384 + row * 128 + (((k8 & 7) ^ (row & 7)) << 4));
}

// The 32 bits of a packed row from bit `pos` on (the row is read as 32-bit
// words; when `pos` is not word aligned the next word is read too, which for
// the last fields of a row lies in the row's 64-byte staging slot and only
// feeds bits above the ones used).
__device__ __forceinline__ uint32_t pf_bits(const uint32_t* w, int pos) {
    const int i = pos >> 5, sh = pos & 31;
    return sh == 0 ? w[i] : __funnelshift_r(w[i], w[i + 1], sh);
}

__device__ __forceinline__ uint32_t pf_pack_half2(float a, float b) {
    return (uint32_t)__half_as_ushort(__float2half_rn(a)) | ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
}

__device__ __forceinline__ float pf_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A row of the prefill output attends over [0, pos]; rows past the chunk
// (the last tile of a (sequence, KV head)) attend nowhere and write nothing.
template <int KB, int VB>
__global__ void __launch_bounds__(128, 1)
k_attn_prefill(const __half* __restrict__ q16, const float* __restrict__ qexp, int Hq, int Hkv, int T,
               const int32_t* __restrict__ q_start, tq_cache_view cache, float* __restrict__ out,
               int* status, const __grid_constant__ AttnParams P) {
    extern __shared__ __align__(1024) unsigned char pf_raw[];
    unsigned char* sm = pf_raw + ((1024u - (smem_addr(pf_raw) & 1023u)) & 1023u);
    const uint32_t sa = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hq / Hkv, tpr = kPfRows / G;
    const int bg = blockIdx.y, b = bg / Hkv, g = bg - b * Hkv;
    const int rows_total = T * G;
    const int grow = blockIdx.x * kPfRows + tid;  // this thread's row within (b, g)
    const bool rvalid = grow < rows_total;
    const int tok = rvalid ? grow / G : 0, hh = grow - (grow / G) * G;
    int64_t qs = __ldg(q_start + b);
    const int last_tok = min(T, (int)(blockIdx.x + 1) * tpr) - 1;
    if (qs < 0 || qs + T > cache.cap) {  // nothing sensible to read: report and write zeros
        if (tid == 0) report_timeout(status, kPfStatusRange);
        qs = -1;
    }
    const int64_t pos = qs + tok;                            // this row attends [0, pos]
    const int64_t kv_end = qs < 0 ? 0 : qs + last_tok + 1;   // rows this CTA reads
    uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + kPfBar);
    uint64_t* bar_pv = bar_s + 1;
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kPfMisc);
    float* red = reinterpret_cast<float*>(sm + kPfMisc + 16);
    uint32_t* tk = reinterpret_cast<uint32_t*>(sm + kPfTK);
    uint32_t* tv = reinterpret_cast<uint32_t*>(sm + kPfTV);
    float* kn_s = reinterpret_cast<float*>(sm + kPfKN);
    float* vn_s = reinterpret_cast<float*>(sm + kPfVN);

    // pair tables: entry e = (c[e % 2^b], c[e / 2^b]) as two fp16 halves
    for (int e = tid; e < (1 << (2 * KB)); e += 128)
        tk[e] = pf_pack_half2(P.kcen_h[e & ((1 << KB) - 1)], P.kcen_h[e >> KB]);
    for (int e = tid; e < (1 << (2 * VB)); e += 128)
        tv[e] = pf_pack_half2(P.vcen_h[e & ((1 << VB) - 1)], P.vcen_h[e >> VB]);
    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_pv, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc<256>(slot);

    // E: the largest V norm this CTA reads is below 2^E
    const int64_t crow0 = (int64_t)bg * cache.cap;  // cache row of position 0
    float vmax = 0.f;
    for (int64_t t = tid; t < kv_end; t += 128) vmax = fmaxf(vmax, fabsf(__ldg(cache.v_norm + crow0 + t)));
    for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, o));
    if (lane == 0) red[warp] = vmax;

    // Q tile: row tid, high and low parts
    {
        const uint4* src = reinterpret_cast<const uint4*>(q16 + ((int64_t)bg * rows_total + grow) * 256);
#pragma unroll 4
        for (int k8 = 0; k8 < 16; ++k8) {
            const uint4 h = rvalid ? __ldg(src + k8) : make_uint4(0, 0, 0, 0);
            const uint4 l = rvalid ? __ldg(src + 16 + k8) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sm + kPfQH + pf_chunk(tid, k8)) = h;
            *reinterpret_cast<uint4*>(sm + kPfQL + pf_chunk(tid, k8)) = l;
        }
    }
    const float qx = rvalid ? __ldg(qexp + (int64_t)bg * rows_total + grow) : 0.f;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    int E = 0;
    {
        const float vm = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        if (vm > 0.f && vm <= FLT_MAX) frexpf(vm, &E);  // vm < 2^E
    }
    const float inv2E = ldexpf(1.f, -E);
    const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16);  // this warp's lanes
    constexpr uint32_t idesc = umma_idesc_f16(128, 128, false);

    float O[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) O[j] = 0.f;
    float m = -INFINITY, l = 0.f;
    bool bad = false;
    int pend = 0;  // 1: the S MMAs of block `blk` may be in flight; 2: the PV MMAs
    int pend_par = 0;
    const int nblk = (int)((kv_end + kPfBlock - 1) / kPfBlock);
    constexpr int RBK = 16 * KB, RBV = 16 * VB;  // packed bytes per row

    for (int blk = 0; blk < nblk; ++blk) {
        const int64_t t0 = (int64_t)blk * kPfBlock;
        const int nv = kv_end - t0 < kPfBlock ? (int)(kv_end - t0) : kPfBlock;
        // 1. stage the packed rows and norms of positions t0 .. t0 + 127 (zeros past kv_end)
        {
            const int64_t crow = crow0 + t0 + tid;
            uint4* ks = reinterpret_cast<uint4*>(sm + kPfKS + tid * 64);
            uint4* vs = reinterpret_cast<uint4*>(sm + kPfVS + tid * 64);
            const bool in = tid < nv;
#pragma unroll
            for (int i = 0; i < RBK / 16; ++i)
                ks[i] = in ? __ldg(reinterpret_cast<const uint4*>(cache.k_packed + crow * RBK) + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < RBV / 16; ++i)
                vs[i] = in ? __ldg(reinterpret_cast<const uint4*>(cache.v_packed + crow * RBV) + i) : make_uint4(0, 0, 0, 0);
            kn_s[tid] = in ? __ldg(cache.k_norm + crow) : 0.f;
            vn_s[tid] = in ? __ldg(cache.v_norm + crow) : 0.f;
        }
        __syncthreads();
        // 2. K tile: thread tid = position tid, 16 chunks of 8 dims (4 pair lookups each)
        {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(sm + kPfKS + tid * 64);
#pragma unroll 4
            for (int k8 = 0; k8 < 16; ++k8) {
                const uint32_t f = pf_bits(w, k8 * 8 * KB);
                uint4 c;
                c.x = tk[f & ((1u << (2 * KB)) - 1)];
                c.y = tk[(f >> (2 * KB)) & ((1u << (2 * KB)) - 1)];
                c.z = tk[(f >> (4 * KB)) & ((1u << (2 * KB)) - 1)];
                c.w = tk[(f >> (6 * KB)) & ((1u << (2 * KB)) - 1)];
                *reinterpret_cast<uint4*>(sm + kPfKT + pf_chunk(tid, k8)) = c;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // 3. S = Q K^T (high and low parts of Q)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_f16(tmem, umma_desc_sw128(sa + kPfQH + off), umma_desc_sw128(sa + kPfKT + off), idesc,
                         kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_f16(tmem, umma_desc_sw128(sa + kPfQL + off), umma_desc_sw128(sa + kPfKT + off), idesc, 1u);
            }
            umma_commit(bar_s);
        }
        pend = 1;
        pend_par = blk & 1;
        // 4. V tile: thread = (8 positions, 16 dims); entry (c[idx(t, j)], c[idx(t + 1, j)])
        {
            const int t8 = tid & 15, dg = tid >> 4;
            uint64_t f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t* w = reinterpret_cast<const uint32_t*>(sm + kPfVS + (8 * t8 + i) * 64);
                const int bp = dg * 16 * VB;  // bit offset of dim 16 dg
                const int wi = bp >> 5, sh = bp & 31;
                const uint64_t x = (uint64_t)w[wi] | ((uint64_t)w[wi + 1] << 32);
                f[i] = x >> sh;  // 16 fields of VB bits in the low 16 VB bits
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                uint32_t c[4];
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    const uint32_t a = (uint32_t)(f[2 * pp] >> (jj * VB)) & ((1u << VB) - 1);
                    const uint32_t bb = (uint32_t)(f[2 * pp + 1] >> (jj * VB)) & ((1u << VB) - 1);
                    c[pp] = tv[a | (bb << VB)];
                }
                *reinterpret_cast<uint4*>(sm + kPfVT + pf_chunk(16 * dg + jj, t8)) = make_uint4(c[0], c[1], c[2], c[3]);
            }
        }
        fence_proxy_async_smem();
        // 5. softmax of this thread's row
        const bool ok_s = mbar_wait(bar_s, blk & 1);
        if (__syncthreads_or(!ok_s)) {
            if (tid == 0) report_timeout(status, kPfStatusWait);
            bad = true;
            break;
        }
        pend = 0;
        tc_fence_after();
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t s[32];
            tmem_ld32(t_row + 32 * c, s);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int k = 32 * c + i;
                const bool valid = rvalid && k < nv && t0 + k <= pos;
                const float v = __uint_as_float(s[i]) * qx * kn_s[k];
                mx = valid ? fmaxf(mx, v) : mx;
            }
        }
        const float m_new = fmaxf(m, mx);
        const float alpha = (m_new == -INFINITY || m == -INFINITY) ? 0.f : pf_exp2(m - m_new);
        float lb = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t s[32];
            tmem_ld32(t_row + 32 * c, s);
            tmem_wait_ld();
#pragma unroll
            for (int k8 = 0; k8 < 4; ++k8) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {
                    float w2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int i = 8 * k8 + 2 * pr + u, k = 32 * c + i;
                        const bool valid = rvalid && k < nv && t0 + k <= pos;
                        const float p = valid ? pf_exp2(__uint_as_float(s[i]) * qx * kn_s[k] - m_new) : 0.f;
                        lb += p;
                        w2[u] = p * vn_s[k] * inv2E;
                    }
                    const __half h0 = __float2half_rn(w2[0]), h1 = __float2half_rn(w2[1]);
                    hi[pr] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                    lo[pr] = pf_pack_half2(w2[0] - __half2float(h0), w2[1] - __half2float(h1));
                }
                const int kc = 4 * c + k8;  // chunk of 8 positions
                *reinterpret_cast<uint4*>(sm + kPfPH + pf_chunk(tid, kc)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(sm + kPfPL + pf_chunk(tid, kc)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        l = l * alpha + lb;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // 6. O_blk = P V (high and low parts of P), folded into the running output
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_f16(tmem + 128, umma_desc_sw128(sa + kPfPH + off), umma_desc_sw128(sa + kPfVT + off), idesc,
                         kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_f16(tmem + 128, umma_desc_sw128(sa + kPfPL + off), umma_desc_sw128(sa + kPfVT + off), idesc,
                         1u);
            }
            umma_commit(bar_pv);
        }
        pend = 2;
        pend_par = blk & 1;
        const bool ok_pv = mbar_wait(bar_pv, blk & 1);
        if (__syncthreads_or(!ok_pv)) {
            if (tid == 0) report_timeout(status, kPfStatusWait);
            bad = true;
            break;
        }
        pend = 0;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(t_row + 128 + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) O[32 * c + i] = fmaf(O[32 * c + i], alpha, __uint_as_float(o[i]));
        }
        m = m_new;
        tc_fence_before();
        __syncthreads();  // S, O_blk and the staging buffers are free for the next block
    }

    if (bad && pend) mbar_wait(pend == 1 ? bar_s : bar_pv, pend_par);  // bounded: let MMAs in flight finish
    // normalise, rotate back (s . H (s2 . o) / sqrt(d)) and store the row
    if (rvalid && !bad) {
        const float sc = l > 0.f ? ldexpf(P.out_mul, E) / l : 0.f;
        if (P.two_sided) {
#pragma unroll
            for (int j = 0; j < 128; ++j) O[j] = __uint_as_float(__float_as_uint(O[j]) ^ P.sgn2[j]);
        }
        fwht_reg<128>(O);
        float* dst = out + (((int64_t)b * T + tok) * Hq + g * G + hh) * 128;
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
            float4 v;
            v.x = __uint_as_float(__float_as_uint(O[j] * sc * P.inv_sqrt_d) ^ P.sgn[j]);
            v.y = __uint_as_float(__float_as_uint(O[j + 1] * sc * P.inv_sqrt_d) ^ P.sgn[j + 1]);
            v.z = __uint_as_float(__float_as_uint(O[j + 2] * sc * P.inv_sqrt_d) ^ P.sgn[j + 2]);
            v.w = __uint_as_float(__float_as_uint(O[j + 3] * sc * P.inv_sqrt_d) ^ P.sgn[j + 3]);
            reinterpret_cast<float4*>(dst)[j / 4] = v;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<256>(tmem);
    }
}

// Query rotation for the prefill: block (b, t, h) rotates q[b][t][h] into
// row (t G + h % G) of (b, h / G) in the layout the prefill kernel reads.
static __global__ void __launch_bounds__(128) k_prefill_q(const __nv_bfloat16* __restrict__ q,
                                                          __half* __restrict__ q16, float* __restrict__ qexp,
                                                          int T, int Hq, int Hkv,
                                                          const __grid_constant__ AttnParams P) {
    const int64_t i = blockIdx.x;  // (b T + t) Hq + h
    const int h = (int)(i % Hq);
    const int64_t bt = i / Hq;
    const int t = (int)(bt % T);
    const int64_t b = bt / T;
    const int G = Hq / Hkv;
    const int64_t row = (b * Hkv + h / G) * ((int64_t)T * G) + (int64_t)t * G + h % G;
    rotate_q_row(q + i * 128, q16 + row * 256, qexp + row, P);
}

template <int KB, int VB>
cudaError_t prefill_launch(const void* q, int B, int T, int Hq, int Hkv, const int32_t* q_start,
                           const tq_cache_view& cache, float* out, void* ws, const AttnParams& P, cudaStream_t s) {
    __half* q16 = static_cast<__half*>(ws);
    float* qexp = reinterpret_cast<float*>(static_cast<char*>(ws) + (size_t)B * T * Hq * 512);
    k_prefill_q<<<(unsigned)((int64_t)B * T * Hq), 128, 0, s>>>(static_cast<const __nv_bfloat16*>(q), q16, qexp, T,
                                                               Hq, Hkv, P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto fn = k_attn_prefill<KB, VB>;
    static int attr_done[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPfSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = 1;
    }
    const int G = Hq / Hkv;
    const dim3 grid((unsigned)(((int64_t)T * G + kPfRows - 1) / kPfRows), (unsigned)(B * Hkv));
    fn<<<grid, 128, kPfSmem, s>>>(q16, qexp, Hq, Hkv, T, q_start, cache, out, status_word(), P);
    return cudaGetLastError();
}

}  // namespace dev

template <int KB>
cudaError_t launch_attn_prefill(int v_bits, const void* q, int B, int T, int Hq, int Hkv, const int32_t* q_start,
                                const tq_cache_view& cache, float* out, void* workspace, const AttnParams& P,
                                cudaStream_t s) {
    switch (v_bits) {
        case 2: return dev::prefill_launch<KB, 2>(q, B, T, Hq, Hkv, q_start, cache, out, workspace, P, s);
        case 3: return dev::prefill_launch<KB, 3>(q, B, T, Hq, Hkv, q_start, cache, out, workspace, P, s);
        default: return dev::prefill_launch<KB, 4>(q, B, T, Hq, Hkv, q_start, cache, out, workspace, P, s);
    }
}

#if !defined(TQ_UNIT_KB)
#error "compile once per K width with -DTQ_UNIT_KB=<bits>"
#endif
template cudaError_t launch_attn_prefill<TQ_UNIT_KB>(int, const void*, int, int, int, int, const int32_t*,
                                                     const tq_cache_view&, float*, void*, const AttnParams&,
                                                     cudaStream_t);

}  // namespace tq
