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
// One CTA of sixteen warps takes 128 query rows of one (sequence, KV head):
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
//   5. four threads share a row of S (a quarter of the columns each): they
//      read it from tensor memory, apply the query's power-of-two scale, the
//      K norms and the causal mask, merge their maxima through shared memory
//      and update the running max and denominator (log2 units); P = exp2(s -
//      m) times the V norm over 2^E (E fixed per CTA from the largest V norm
//      it reads, so P <= 1) goes to shared memory as fp16 high and low parts;
//   6. one thread issues O_blk = P_hi V + P_lo V into tensor memory; each
//      thread folds its quarter of the row into the running output held in
//      registers, O = O * exp2(m_old - m_new) + O_blk.
// At the end the rows are divided by the denominator, scaled by 2^E / s_v
// and rotated back (s . H (s2 . o) / sqrt(d)): butterflies over a thread's
// quarter in registers, the two across quarters through shared memory.
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

constexpr int kPfRows = 128;     // query rows per CTA
constexpr int kPfBlock = 128;    // KV positions per block
constexpr int kPfThreads = 512;  // 16 warps; warp w reads tensor-memory lanes 32 (w % 4) .. + 31,
                                 // columns 32 (w / 4) .. + 31 of its rows
// shared memory, offsets from a 1024-aligned base
constexpr uint32_t kPfQH = 0;          // Q high parts, 128 x 128 fp16 (the output rows at the end)
constexpr uint32_t kPfQL = 32768;      // Q low parts
constexpr uint32_t kPfKT = 65536;      // K centroids of the block, [position][dim]
constexpr uint32_t kPfVT = 98304;      // V centroids of the block, [dim][position]
constexpr uint32_t kPfPH = 131072;     // P high parts, [row][position]
constexpr uint32_t kPfPL = 163840;     // P low parts
constexpr uint32_t kPfTK = 196608;     // K pair table, 4 copies (up to 256 x 4 words)
constexpr uint32_t kPfTV = 200704;     // V pair table, 4 copies
constexpr uint32_t kPfSK = 204800;     // staged packed K rows of the next block, 64-byte stride
constexpr uint32_t kPfSV = 212992;     // staged packed V rows
constexpr uint32_t kPfSKN = 221184;    // staged K norms (128 floats)
constexpr uint32_t kPfSVN = 221696;    // staged V norms
constexpr uint32_t kPfKN = 222208;     // K norms of the block (128 floats)
constexpr uint32_t kPfVN = 222720;     // V norms of the block over 2^E
constexpr uint32_t kPfRed = 223232;    // [4][128] floats: per-quarter row maxima / sums
constexpr uint32_t kPfBar = 225280;    // two mbarriers
constexpr uint32_t kPfMisc = 225296;   // tensor-memory base, reduction scratch (16 floats)
constexpr uint32_t kPfEnd = 225424;
constexpr int kPfCopies = 4;           // table copies: lane l reads copy l % 4 (fewer bank conflicts)
constexpr uint32_t kPfSmem = kPfEnd + 1024;  // plus alignment slack
constexpr int kPfStatusWait = 51;      // an MMA completion wait gave up
constexpr int kPfStatusRange = 52;     // q_start[b] + T exceeds the cache capacity, or q_start < 0

// Offset of the 16-byte chunk holding elements [8 k8, 8 k8 + 8) of `row` in a
// 128 x 128 fp16 K-major tile with the 128-byte swizzle (two 64-column
// halves of 16 KB, rows of 128 bytes, chunk index xor row % 8).
__device__ __forceinline__ uint32_t pf_chunk(int row, int k8) {
    return (uint32_t)((k8 >> 3) * 16384 + row * 128 + (((k8 & 7) ^ (row & 7)) << 4));
}

// N bits (N <= 32) of a staged packed row from bit `pos` on, in the low
// bits; the row is read as 32-bit words, the next word only when the field
// crosses into it.
template <int N>
__device__ __forceinline__ uint32_t pf_bits(const uint32_t* w, int pos) {
    const int i = pos >> 5, sh = pos & 31;
    const uint32_t lo = w[i];
    if (sh == 0) return lo;
    return sh + N > 32 ? __funnelshift_r(lo, w[i + 1], sh) : lo >> sh;
}

// Stage the packed K and V rows and the norms of positions t0 .. t0 + 127 of
// cache rows crow0 + .. with cp.async (zero fill past n valid rows; the
// source of a zero-filled copy is row crow0, which exists).
template <int KB, int VB>
__device__ __forceinline__ void pf_stage(uint32_t sa, const tq_cache_view& cache, int64_t crow0, int64_t t0,
                                         int n, int tid) {
    constexpr int KP = KB, VP = VB;  // 16-byte parts per packed row (16 * bits bytes)
    if (tid < 128 * KP) {
        const int row = tid / KP, part = tid - row * KP;
        const bool in = row < n;
        const uint8_t* src = cache.k_packed + (crow0 + (in ? t0 + row : 0)) * (16 * KB) + part * 16;
        cp_async16(sa + kPfSK + row * 64 + part * 16, src, in ? 16u : 0u);
    }
    if (tid < 128 * VP) {
        const int row = tid / VP, part = tid - row * VP;
        const bool in = row < n;
        const uint8_t* src = cache.v_packed + (crow0 + (in ? t0 + row : 0)) * (16 * VB) + part * 16;
        cp_async16(sa + kPfSV + row * 64 + part * 16, src, in ? 16u : 0u);
    }
    if (tid < 256) {  // norms, one per copy (a norm row is only 4-byte aligned); zeros past n
        const int k = tid & 127, side = tid >> 7;
        const float* nrm = side ? cache.v_norm : cache.k_norm;
        cp_async4(sa + (side ? kPfSVN : kPfSKN) + 4 * k, nrm + crow0 + (k < n ? t0 + k : 0), k < n ? 4u : 0u);
    }
    cp_async_commit();
}

__device__ __forceinline__ uint32_t pf_pack_half2(float a, float b) {
    return (uint32_t)__half_as_ushort(__float2half_rn(a)) | ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
}

__device__ __forceinline__ float pf_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Tiles of a (sequence, KV head) are taken last first: with a causal mask the
// last tiles read the most KV blocks, so the longest CTAs start first.
template <int KB, int VB>
__global__ void __launch_bounds__(kPfThreads, 1)
k_attn_prefill(const __half* __restrict__ q16, const float* __restrict__ qexp, int Hq, int Hkv, int T,
               const int32_t* __restrict__ q_start, tq_cache_view cache, float* __restrict__ out,
               int* status, const __grid_constant__ AttnParams P) {
    extern __shared__ __align__(1024) unsigned char pf_raw[];
    unsigned char* sm = pf_raw + ((1024u - (smem_addr(pf_raw) & 1023u)) & 1023u);
    const uint32_t sa = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = 32 * (warp & 3) + lane;  // this thread's query row in the tile
    const int cq = warp >> 2;              // and its quarter of the columns
    const int G = Hq / Hkv, tpr = kPfRows / G;
    const int bg = blockIdx.y, b = bg / Hkv, g = bg - b * Hkv;
    const int mt = (int)(gridDim.x - 1 - blockIdx.x);
    const int rows_total = T * G;
    const int grow = mt * kPfRows + r;  // this thread's row within (b, g)
    const bool rvalid = grow < rows_total;
    const int tok = rvalid ? grow / G : 0, hh = grow - (grow / G) * G;
    int64_t qs = __ldg(q_start + b);
    const int last_tok = min(T, (mt + 1) * tpr) - 1;
    if (qs < 0 || qs + T > cache.cap) {  // nothing sensible to read: report and write zeros
        if (tid == 0) report_timeout(status, kPfStatusRange);
        qs = -1;
    }
    const int64_t pos = qs + tok;                            // this row attends [0, pos]
    const int64_t kv_end = qs < 0 ? 0 : qs + last_tok + 1;   // rows this CTA reads
    uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + kPfBar);
    uint64_t* bar_pv = bar_s + 1;
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kPfMisc);
    volatile int* wflag = reinterpret_cast<volatile int*>(sm + kPfMisc + 8);
    // One thread waits (bounded) for an MMA to complete and the block's
    // barrier releases the others: no warp spins on the mbarrier while others
    // still have work.  Returns false for every thread if the wait gave up.
    auto block_wait = [&](uint64_t* bar, int parity) {
        if (tid == 0) *wflag = mbar_wait(bar, parity) ? 1 : 0;
        __syncthreads();
        return *wflag != 0;
    };
    float* wred = reinterpret_cast<float*>(sm + kPfMisc + 16);
    uint32_t* tk = reinterpret_cast<uint32_t*>(sm + kPfTK);
    uint32_t* tv = reinterpret_cast<uint32_t*>(sm + kPfTV);
    float* kn_s = reinterpret_cast<float*>(sm + kPfKN);
    float* vn_s = reinterpret_cast<float*>(sm + kPfVN);
    float* red = reinterpret_cast<float*>(sm + kPfRed);

    // pair tables: entry e = (c[e % 2^b], c[e / 2^b]) as two fp16 halves, copy
    // c of entry e at word 8 e + c
    for (int i = tid; i < (kPfCopies << (2 * KB)); i += kPfThreads) {
        const int e = i / kPfCopies;
        tk[i] = pf_pack_half2(P.kcen_h[e & ((1 << KB) - 1)], P.kcen_h[e >> KB]);
    }
    for (int i = tid; i < (kPfCopies << (2 * VB)); i += kPfThreads) {
        const int e = i / kPfCopies;
        tv[i] = pf_pack_half2(P.vcen_h[e & ((1 << VB) - 1)], P.vcen_h[e >> VB]);
    }
    const uint32_t* tkl = tk + (lane & (kPfCopies - 1));  // this lane's copy
    const uint32_t* tvl = tv + (lane & (kPfCopies - 1));
    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_pv, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc<512>(slot);  // S 0-127, O_blk 128-255, P high 256-319, P low 320-383

    // E: the largest V norm this CTA reads is below 2^E
    const int64_t crow0 = (int64_t)bg * cache.cap;  // cache row of position 0
    float vmax = 0.f;
    for (int64_t t = tid; t < kv_end; t += kPfThreads) vmax = fmaxf(vmax, fabsf(__ldg(cache.v_norm + crow0 + t)));
    for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, o));
    if (lane == 0) wred[warp] = vmax;

    // Q tile: row r, chunks 4 cq .. 4 cq + 3 of the high and low parts
    {
        const uint4* src = reinterpret_cast<const uint4*>(q16 + ((int64_t)bg * rows_total + grow) * 256);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k8 = 4 * cq + i;
            const uint4 h = rvalid ? __ldg(src + k8) : make_uint4(0, 0, 0, 0);
            const uint4 l = rvalid ? __ldg(src + 16 + k8) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sm + kPfQH + pf_chunk(r, k8)) = h;
            *reinterpret_cast<uint4*>(sm + kPfQL + pf_chunk(r, k8)) = l;
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
        float vm = 0.f;
#pragma unroll
        for (int w = 0; w < kPfThreads / 32; ++w) vm = fmaxf(vm, wred[w]);
        if (vm > 0.f && vm <= FLT_MAX) frexpf(vm, &E);  // vm < 2^E
    }
    const float inv2E = ldexpf(1.f, -E);
    const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * cq;  // this thread's S columns
    constexpr uint32_t idesc = umma_idesc_f16(128, 128, false);

    float O[32];  // columns 32 cq .. 32 cq + 31 of the output row (rotated, units of 2^E s_v)
#pragma unroll
    for (int j = 0; j < 32; ++j) O[j] = 0.f;
    float m = -INFINITY, lp = 0.f;  // running max of the row (s' units) and this quarter's sum
    bool bad = false;
    int pend = 0;  // 1: the S MMAs of the current block may be in flight; 2: the PV MMAs
    int pend_par = 0;
    const int nblk = (int)((kv_end + kPfBlock - 1) / kPfBlock);
    if (nblk > 0) pf_stage<KB, VB>(sa, cache, crow0, 0, kv_end < kPfBlock ? (int)kv_end : kPfBlock, tid);
    // The K tile of block j + 1 is built while the PV product of block j runs
    // (the K tile is free once S_j is done), and S_{j+1} is issued before the
    // V tile of block j + 1 is built.
    auto stage_k = [&]() {
        // the staged rows of the block have landed; the norms move to their own
        // arrays (the staging area takes the next block during this one)
        cp_async_wait_all();
        __syncthreads();
        if (tid < 128) kn_s[tid] = reinterpret_cast<const float*>(sm + kPfSKN)[tid];
        else if (tid < 256) vn_s[tid - 128] = reinterpret_cast<const float*>(sm + kPfSVN)[tid - 128] * inv2E;
        // K tile: lanes take the 16 chunks of 8 dims of a row (consecutive words
        // of the staged row, conflict-free tile stores); row (tid / 16) + 32 i;
        // 4 pair lookups per chunk
        {
            const int k8 = tid & 15;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = (tid >> 4) + 32 * i;
                const uint32_t f =
                    pf_bits<8 * KB>(reinterpret_cast<const uint32_t*>(sm + kPfSK + t * 64), k8 * 8 * KB);
                constexpr uint32_t M = (1u << (2 * KB)) - 1;
                uint4 c;
                c.x = tkl[kPfCopies * (f & M)];
                c.y = tkl[kPfCopies * ((f >> (2 * KB)) & M)];
                c.z = tkl[kPfCopies * ((f >> (4 * KB)) & M)];
                c.w = tkl[kPfCopies * ((f >> (6 * KB)) & M)];
                *reinterpret_cast<uint4*>(sm + kPfKT + pf_chunk(t, k8)) = c;
            }
        }
    };
    auto issue_s = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // S = Q K^T (high and low parts of Q)
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
    };
    if (nblk > 0) {
        stage_k();
        issue_s();
        pend = 1;
        pend_par = 0;
    }

    for (int blk = 0; blk < nblk; ++blk) {
        const int64_t t0 = (int64_t)blk * kPfBlock;
        const int nv = kv_end - t0 < kPfBlock ? (int)(kv_end - t0) : kPfBlock;
        // V tile: lanes take consecutive dim pairs (2 jp, 2 jp + 1) of the same
        // rows; thread = (dim pair tid % 64, position groups (tid / 64) + 8 i of
        // 8 positions); entry (c[idx(t, j)], c[idx(t + 1, j)])
        {
            const int jp = tid & 63;
            constexpr uint32_t M = (1u << VB) - 1;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int t8 = (tid >> 6) + 8 * i;
                uint32_t f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    f[u] = pf_bits<2 * VB>(reinterpret_cast<const uint32_t*>(sm + kPfSV + (8 * t8 + u) * 64),
                                           2 * jp * VB);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    uint32_t c[4];
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        const uint32_t a = (f[2 * pp] >> (jj * VB)) & M;
                        const uint32_t bb = (f[2 * pp + 1] >> (jj * VB)) & M;
                        c[pp] = tvl[kPfCopies * (a | (bb << VB))];
                    }
                    *reinterpret_cast<uint4*>(sm + kPfVT + pf_chunk(2 * jp + jj, t8)) =
                        make_uint4(c[0], c[1], c[2], c[3]);
                }
            }
        }
        fence_proxy_async_smem();
        // softmax: this thread's 32 columns of its row
        if (!block_wait(bar_s, blk & 1)) {
            if (tid == 0) report_timeout(status, kPfStatusWait);
            bad = true;
            break;
        }
        pend = 0;
        if (blk + 1 < nblk) {  // the staging area is free: fetch the next block during this one
            const int64_t t1 = t0 + kPfBlock;
            pf_stage<KB, VB>(sa, cache, crow0, t1, kv_end - t1 < kPfBlock ? (int)(kv_end - t1) : kPfBlock, tid);
        }
        tc_fence_after();
        // s' = S * |k| per column; the row's scores in log2 units are s' * qx
        // (qx > 0), so the running max is kept in s' units and
        // p = exp2(s' qx - m qx).  Columns inside the row's range for the whole
        // quarter skip the per-column mask.
        float sv[32];
        {
            uint32_t sr[32];
            tmem_ld32(t_row, sr);
            tmem_wait_ld();
            const float4* kn4 = reinterpret_cast<const float4*>(kn_s + 32 * cq);
            const bool full = rvalid && 32 * cq + 31 < nv && t0 + 32 * cq + 31 <= pos;
            float mx = -INFINITY;
            if (full) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 kk = kn4[j];
                    f2_split(f2_mul(f2(__uint_as_float(sr[4 * j]), __uint_as_float(sr[4 * j + 1])), f2(kk.x, kk.y)),
                             sv[4 * j], sv[4 * j + 1]);
                    f2_split(f2_mul(f2(__uint_as_float(sr[4 * j + 2]), __uint_as_float(sr[4 * j + 3])), f2(kk.z, kk.w)),
                             sv[4 * j + 2], sv[4 * j + 3]);
                    mx = fmaxf(mx, fmaxf(fmaxf(sv[4 * j], sv[4 * j + 1]), fmaxf(sv[4 * j + 2], sv[4 * j + 3])));
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int k = 32 * cq + i;
                    const bool valid = rvalid && k < nv && t0 + k <= pos;
                    sv[i] = valid ? __uint_as_float(sr[i]) * kn_s[k] : -INFINITY;
                    mx = fmaxf(mx, sv[i]);
                }
            }
            red[cq * 128 + r] = mx;
        }
        __syncthreads();
        const float m_new = fmaxf(m, fmaxf(fmaxf(red[r], red[128 + r]), fmaxf(red[256 + r], red[384 + r])));
        const float qxs = rvalid ? qx : 1.f;
        const float alpha = (m_new == -INFINITY || m == -INFINITY) ? 0.f : pf_exp2((m - m_new) * qxs);
        const float nmq = m_new == -INFINITY ? 0.f : -m_new * qxs;  // masked columns: exp2(-inf) = 0
        const F2 QX = f2(qxs, qxs), NMQ = f2(nmq, nmq);
        F2 LB = f2(0.f, 0.f);
        const float4* vn4 = reinterpret_cast<const float4*>(vn_s + 32 * cq);  // |v| / 2^E
        uint32_t hi16[16], lo16[16];  // this quarter's 32 positions of P as fp16 pairs
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {
            uint32_t* hi = hi16 + 4 * k8;
            uint32_t* lo = lo16 + 4 * k8;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const float4 vv = vn4[2 * k8 + h2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int i = 8 * k8 + 4 * h2 + 2 * u;
                    float a0, a1;
                    f2_split(f2_fma(f2(sv[i], sv[i + 1]), QX, NMQ), a0, a1);
                    const F2 pp = f2(pf_exp2(a0), pf_exp2(a1));
                    LB = f2_add(LB, pp);
                    float w0, w1;
                    f2_split(f2_mul(pp, u == 0 ? f2(vv.x, vv.y) : f2(vv.z, vv.w)), w0, w1);
                    const __half2 hh2 = __floats2half2_rn(w0, w1);
                    const float2 hf = __half22float2(hh2);
                    const __half2 ll2 = __floats2half2_rn(w0 - hf.x, w1 - hf.y);
                    hi[2 * h2 + u] = *reinterpret_cast<const uint32_t*>(&hh2);
                    lo[2 * h2 + u] = *reinterpret_cast<const uint32_t*>(&ll2);
                }
            }
        }
        // P to tensor memory, row r, columns 16 cq .. 16 cq + 15 of each part
        {
            const uint32_t t_p = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256 + 16 * cq;
            tmem_st16(t_p, hi16);
            tmem_st16(t_p + 64, lo16);
            tmem_wait_st();
        }
        float lb0, lb1;
        f2_split(LB, lb0, lb1);
        const float lb = lb0 + lb1;
        lp = lp * alpha + lb;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // O_blk = P V (high and low parts of P), folded into the running output
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_f16_ts(tmem + 128, tmem + 256 + 8 * kk, umma_desc_sw128(sa + kPfVT + off), idesc,
                            kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                umma_f16_ts(tmem + 128, tmem + 320 + 8 * kk, umma_desc_sw128(sa + kPfVT + off), idesc, 1u);
            }
            umma_commit(bar_pv);
        }
        pend = 2;
        pend_par = blk & 1;
        if (blk + 1 < nblk) stage_k();  // K tile of the next block while PV runs
        if (!block_wait(bar_pv, blk & 1)) {
            if (tid == 0) report_timeout(status, kPfStatusWait);
            bad = true;
            break;
        }
        pend = 0;
        tc_fence_after();
        {
            uint32_t o[32];
            tmem_ld32(t_row + 128, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) O[i] = fmaf(O[i], alpha, __uint_as_float(o[i]));
        }
        m = m_new;
        if (blk + 1 < nblk) {  // its barrier also ends this block: S, O_blk and red are free
            issue_s();
            pend = 1;
            pend_par = (blk + 1) & 1;
        } else {
            tc_fence_before();
            __syncthreads();
        }
    }

    cp_async_wait_all();  // no copy of this thread is left in flight
    if (bad && pend) mbar_wait(pend == 1 ? bar_s : bar_pv, pend_par);  // bounded: let MMAs in flight finish
    // normalise (the row's sum over its four quarters) and rotate back,
    // s . H (s2 . o) / sqrt(d): H over the 7 index bits of a row is the
    // butterflies over bits 0-4 (a thread's quarter, in registers) and over
    // bits 5 and 6 (between the four threads of the row, through shared
    // memory laid out [quarter][element][row] so that a warp's accesses hit
    // 32 banks).  The Q region holds the exchange buffer (64 KB).
    red[cq * 128 + r] = lp;
    __syncthreads();
    {
        const float l = red[r] + red[128 + r] + red[256 + r] + red[384 + r];
        const float sc = l > 0.f ? ldexpf(P.out_mul, E) / l : 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float v = O[i] * sc;
            O[i] = P.two_sided ? __uint_as_float(__float_as_uint(v) ^ P.sgn2[32 * cq + i]) : v;
        }
    }
    fwht_reg<32>(O);
    float* xs = reinterpret_cast<float*>(sm + kPfQH);
#pragma unroll
    for (int bit = 1; bit <= 2; bit <<= 1) {  // quarter index bits: index bits 5 and 6
#pragma unroll
        for (int i = 0; i < 32; ++i) xs[(cq * 32 + i) * 128 + r] = O[i];
        __syncthreads();
        const int pq = cq ^ bit;
        const bool upper = (cq & bit) != 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float o = xs[(pq * 32 + i) * 128 + r];
            O[i] = upper ? o - O[i] : O[i] + o;  // (lo + hi, lo - hi)
        }
        __syncthreads();
    }
    if (rvalid && !bad) {
        float4* dst = reinterpret_cast<float4*>(out + (((int64_t)b * T + tok) * Hq + g * G + hh) * 128 + 32 * cq);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            const int j = 32 * cq + i;
            float4 v;
            v.x = __uint_as_float(__float_as_uint(O[i] * P.inv_sqrt_d) ^ P.sgn[j]);
            v.y = __uint_as_float(__float_as_uint(O[i + 1] * P.inv_sqrt_d) ^ P.sgn[j + 1]);
            v.z = __uint_as_float(__float_as_uint(O[i + 2] * P.inv_sqrt_d) ^ P.sgn[j + 2]);
            v.w = __uint_as_float(__float_as_uint(O[i + 3] * P.inv_sqrt_d) ^ P.sgn[j + 3]);
            dst[i / 4] = v;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<512>(tmem);
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
    fn<<<grid, kPfThreads, kPfSmem, s>>>(q16, qexp, Hq, Hkv, T, q_start, cache, out, status_word(), P);
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
