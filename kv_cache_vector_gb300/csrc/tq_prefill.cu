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
// Precision.  The products run on fp16 operands with fp32 accumulation, and
// every operand whose rounding the output can see is carried in two fp16
// parts: the rotated query (high and low), the key centroids (the fp16
// value nearest c * s_k and the fp16 rest c * s_k - that), and P (high and
// low), so S = Q_hi K^T + Q_lo K^T + Q_hi Dk^T and O = P_hi V + P_lo V.  Only
// the V centroids stay single (fp16 nearest c * s_v, within 2.2e-5 relative
// at 3 bits): early causal tokens average few rows, so their outputs are
// nearly raw V values, and the 2e-3 absolute bound has to hold on them.
//
// Two kernels.  Every (sequence, KV head) has many query tiles, and each of
// them reads the whole prefix, so the packed rows are expanded once, not once
// per tile:
//   k_prefill_expand  turns each block of 128 cached positions into a tile
//     image in the workspace: the K centroid high and low parts
//     [position][dim] and the V centroids [dim][position] as fp16, all in the
//     128-byte-swizzled K-major layout the tensor cores read, then the 128 K
//     norms and the 128 V norms (97 KB; norms past the sequence's last
//     position are zero, centroids there c[0]), and the block's largest V
//     norm.  One extra block writes the query rotation s2 . H . s as a bf16
//     matrix of +-1.
//   k_attn_prefill  takes 128 query rows of one (sequence, KV head): 128 / G
//     consecutive tokens times the G query heads of the group (row r = token
//     r / G, head r % G), with warp roles:
//       warp 0    streams the K tiles (high and low) of block j into K stage
//                 j % 2 once S of block j - 2 is done (bulk copies);
//       warp 10   streams the V tile and norms into V stage j % 2 once the PV
//                 product of block j - 2 is done;
//       warp 1    issues the query rotation (bf16 rows times the +-1 matrix,
//                 exact products, fp32 sums), then per block S into
//                 tensor-memory buffer j % 2 (24 MMAs, the query read from
//                 tensor memory) and the PV product of block j - 1 (16 MMAs,
//                 P read from tensor memory);
//       warps 2-9 two threads per query row, 64 columns each: the query's
//                 high and low parts (under a power-of-two scale per row)
//                 into tensor memory from the rotated rows, then per block
//                 the scores times the K norms and the query's scale, the
//                 causal mask, the row max merged through shared memory, and
//                 P = exp2(s - m) times the V norm over 2^E (E fixed per CTA
//                 from the largest V norm it reads) as fp16 high and low
//                 parts over the thread's own S columns.
//     Tensor memory: S/P buffers at columns 0 and 128, the output at 256, the
//     query's high parts at 384 and low parts at 448.  The output
//     accumulates in tensor memory.  The reference max m of a row moves only
//     when a block raises the row max by more than 8 (log2 units), so P
//     stays below 2^8; when it moves, the softmax threads rescale their
//     output columns in tensor memory after the previous PV product is done.
//     At the end the rows are divided by the denominator, scaled by 2^E / s_v
//     and rotated back (s . H (s2 . o) / sqrt(d)): butterflies over a
//     thread's 64 columns in registers, the last one through shared memory,
//     and the rows leave through bulk stores.
//
// Every wait on an mbarrier is bounded (2 s); a wait that gives up sets the
// device status word and a flag that ends every other wait of the CTA, the
// MMA thread waits (bounded) for its products in flight, the copy threads for
// their copies, and the CTA frees its tensor memory and returns.
#include <cfloat>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_async.cuh"
#include "tq_device.cuh"
#include "tq_umma.cuh"
#include "tq_tmem.cuh"

#if !defined(TQ_UNIT_KB)
#error "compile once per K width with -DTQ_UNIT_KB=<bits>"
#endif

namespace tq {
namespace dev {

constexpr int kPfBlock = 128;    // KV positions per block
// tile image of one block, offsets within it
constexpr uint32_t kPfImgK = 0;        // K centroid high parts, 128 x 128 fp16, [position][dim]
constexpr uint32_t kPfImgD = 32768;    // K centroid low parts, the same layout
constexpr uint32_t kPfImgV = 65536;    // V centroids, [dim][position]
constexpr uint32_t kPfImgKN = 98304;   // K norms (128 floats)
constexpr uint32_t kPfImgVN = 98816;   // V norms
static_assert(kPfImgVN + 512 == kPfImgBytes, "tile image layout");

// ---- expansion kernel: the image is built in two halves in one 64 KB buffer
// (the K tiles, then the V tile and norms)
constexpr int kPxThreads = 256;
constexpr uint32_t kPxBuf = 0;
constexpr uint32_t kPxStage = 65536;         // two stages of packed rows: K (8 KB) then V (8 KB)
constexpr uint32_t kPxStageBytes = 16384;
constexpr uint32_t kPxTK = kPxStage + 2 * kPxStageBytes;  // K high-part pair table, 4 copies (256 x 4 words)
constexpr uint32_t kPxTD = kPxTK + 4096;     // K low-part pair table
constexpr uint32_t kPxTV = kPxTD + 4096;     // V pair table
constexpr uint32_t kPxBar = kPxTV + 4096;    // two mbarriers, a flag
constexpr uint32_t kPxSmem = kPxBar + 32;
constexpr int kPxStatusWait = 53;            // a staging wait of the expansion gave up
constexpr int kPfCopies = 4;                 // table copies: lane l reads copy l % 4 (fewer bank conflicts)

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

__device__ __forceinline__ uint32_t pf_pack_half2(float a, float b) {
    return (uint32_t)__half_as_ushort(__float2half_rn(a)) | ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
}

// 1-D bulk copy of `bytes` bytes from shared address `src` to global memory
// (both 16-byte aligned, bytes % 16 == 0), in this thread's bulk group.
__device__ __forceinline__ void pf_bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

// ------------------------------------------------------------------ expansion

// Block (x, bg), x < gridDim.x - 1, expands blocks x, x + gridDim.x - 1, ..
// of (sequence, KV head) bg into img + (bg nbmax + j) kPfImgBytes, and the
// block's largest |V norm| into bmax[bg nbmax + j]; block (gridDim.x - 1, 0)
// writes the query rotation matrix.  Blocks at or past the sequence's last
// position q_start[b] + T are not read; a sequence whose range is invalid is
// skipped (the attention kernel reports it).  Thread 0 fetches the packed
// rows of the next block (one bulk copy per side, rows below the capacity
// only) while the block builds the current image, and sends each half of the
// image out with one bulk store.
template <int KB, int VB>
__global__ void __launch_bounds__(kPxThreads, 2)
k_prefill_expand(const int32_t* __restrict__ q_start, int T, int Hkv, tq_cache_view cache, int nbmax,
                 unsigned char* __restrict__ img, float* __restrict__ bmax, uint4* __restrict__ rot,
                 int* status, const __grid_constant__ AttnParams P) {
    extern __shared__ __align__(16) unsigned char px_raw[];
    unsigned char* sm = px_raw;
    const uint32_t sa = smem_addr(sm);
    const int tid = threadIdx.x, lane = tid & 31;
    const int bg = blockIdx.y, b = bg / Hkv;
    const int nx = gridDim.x - 1;  // blocks per (sequence, KV head); the last column has one job
    if ((int)blockIdx.x == nx) {
        if (blockIdx.y != 0) return;
        // the query rotation as a bf16 matrix R[j][i] = s2_j H_ji s_i (entries
        // +-1, H_ji = (-1)^popcount(i & j)), rows j in the 128-byte-swizzled
        // K-major layout: 16-byte chunk c holds row j = (c / 8) % 128, elements
        // 64 (c / 1024) + 8 ((c % 8) ^ (j % 8)) + 0 .. 7
        for (int c = tid; c < 2048; c += kPxThreads) {
            const int j = (c >> 3) & 127;
            const int i0 = 64 * (c >> 10) + 8 * ((c & 7) ^ (j & 7));
            const uint32_t s2 = P.two_sided ? P.sgn2[j] : 0u;
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t h2 = 0;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int i = i0 + 2 * k + u;
                    const uint32_t sg = ((P.sgn[i] ^ s2) >> 16) ^ ((__popc(i & j) & 1) ? 0x8000u : 0u);
                    h2 |= (0x3F80u | (sg & 0x8000u)) << (16 * u);
                }
                w[k] = h2;
            }
            rot[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        return;
    }
    const int64_t qs = __ldg(q_start + b);
    if (qs < 0 || qs + T > cache.cap) return;
    const int64_t kv_end = qs + T;
    const int nb = (int)((kv_end + kPfBlock - 1) / kPfBlock);
    if ((int)blockIdx.x >= nb) return;
    const int64_t crow0 = (int64_t)bg * cache.cap;  // cache row of position 0
    uint32_t* tk = reinterpret_cast<uint32_t*>(sm + kPxTK);
    uint32_t* td = reinterpret_cast<uint32_t*>(sm + kPxTD);
    uint32_t* tv = reinterpret_cast<uint32_t*>(sm + kPxTV);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kPxBar);  // [2] the stage's rows have landed
    volatile int* okf = reinterpret_cast<volatile int*>(sm + kPxBar + 16);
    // pair tables: entry e = (c[e % 2^b], c[e / 2^b]) as two fp16 halves, copy
    // c of entry e at word 4 e + c
    for (int i = tid; i < (kPfCopies << (2 * KB)); i += kPxThreads) {
        const int e = i / kPfCopies;
        tk[i] = pf_pack_half2(P.kcen_h[e & ((1 << KB) - 1)], P.kcen_h[e >> KB]);
        td[i] = pf_pack_half2(P.kcen_l[e & ((1 << KB) - 1)], P.kcen_l[e >> KB]);
    }
    for (int i = tid; i < (kPfCopies << (2 * VB)); i += kPxThreads) {
        const int e = i / kPfCopies;
        tv[i] = pf_pack_half2(P.vcen_h[e & ((1 << VB) - 1)], P.vcen_h[e >> VB]);
    }
    const uint32_t* tkl = tk + (lane & (kPfCopies - 1));  // this lane's copy
    const uint32_t* tdl = td + (lane & (kPfCopies - 1));
    const uint32_t* tvl = tv + (lane & (kPfCopies - 1));
    // rows of block j that exist in the cache (at least the n of the sequence)
    auto rows_of = [&](int j) {
        const int64_t t0 = (int64_t)j * kPfBlock;
        return cache.cap - t0 < kPfBlock ? (int)(cache.cap - t0) : kPfBlock;
    };
    auto stage = [&](int j, int s) {  // thread 0: the packed rows of block j into stage s
        const int64_t t0 = (int64_t)j * kPfBlock;
        const uint32_t nr = (uint32_t)rows_of(j);
        const uint32_t dst = sa + kPxStage + s * kPxStageBytes;
        mbar_arrive_expect_tx(&bars[s], nr * 16 * (KB + VB));
        bulk_load(dst, cache.k_packed + (crow0 + t0) * (16 * KB), nr * 16 * KB, &bars[s]);
        bulk_load(dst + 8192, cache.v_packed + (crow0 + t0) * (16 * VB), nr * 16 * VB, &bars[s]);
    };
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_fence_init();
        *okf = 1;
        stage(blockIdx.x, 0);
    }
    __syncthreads();

    int k = 0, pre = 0;  // items started, and whether the next one's rows were requested
    for (int j = blockIdx.x; j < nb; j += nx, ++k) {
        const int s = k & 1;
        const int64_t t0 = (int64_t)j * kPfBlock;
        const int n = kv_end - t0 < kPfBlock ? (int)(kv_end - t0) : kPfBlock;
        const int nr = rows_of(j);
        unsigned char* dsti = img + ((int64_t)bg * nbmax + j) * kPfImgBytes;
        if (tid == 0) {
            // the next block's rows into the other stage (free: the block that
            // used it was built before the last barrier), then wait for this
            // block's rows (bounded) and for the last image store to have read
            // shared memory
            pre = j + nx < nb;
            if (pre) stage(j + nx, s ^ 1);
            const bool ok = mbar_wait(&bars[s], (k >> 1) & 1);
            if (!ok) report_timeout(status, kPxStatusWait);
            bulk_wait_read<0>();
            *okf = ok ? 1 : 0;
        }
        __syncthreads();
        if (!*okf) break;
        const unsigned char* sk = sm + kPxStage + s * kPxStageBytes;
        const unsigned char* sv = sk + 8192;
        // K tiles, high and low parts: lanes take the 16 chunks of 8 dims of a
        // row (consecutive words of the staged row, conflict-free tile stores);
        // rows (tid / 16) + 16 i; 4 pair lookups per chunk and part; rows past
        // the capacity read index 0
        {
            const int k8 = tid & 15;
            constexpr uint32_t M = (1u << (2 * KB)) - 1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = (tid >> 4) + 16 * i;
                const uint32_t f = t < nr ? pf_bits<8 * KB>(reinterpret_cast<const uint32_t*>(sk + t * (16 * KB)),
                                                            k8 * 8 * KB)
                                          : 0u;
                const uint32_t e0 = f & M, e1 = (f >> (2 * KB)) & M, e2 = (f >> (4 * KB)) & M, e3 = (f >> (6 * KB)) & M;
                const uint32_t off = pf_chunk(t, k8);
                *reinterpret_cast<uint4*>(sm + kPxBuf + off) =
                    make_uint4(tkl[kPfCopies * e0], tkl[kPfCopies * e1], tkl[kPfCopies * e2], tkl[kPfCopies * e3]);
                *reinterpret_cast<uint4*>(sm + kPxBuf + kPfImgD + off) =
                    make_uint4(tdl[kPfCopies * e0], tdl[kPfCopies * e1], tdl[kPfCopies * e2], tdl[kPfCopies * e3]);
            }
        }
        fence_proxy_async_smem();  // the image goes out through the async proxy
        __syncthreads();
        if (tid == 0) {
            pf_bulk_store(dsti + kPfImgK, sa + kPxBuf, 65536);
            bulk_commit();
            bulk_wait_read<0>();  // the buffer takes the second half
        }
        __syncthreads();
        {  // norms (after the V tile in the buffer); zeros past n
            const int kk = tid & 127;
            const float* nrm = tid < 128 ? cache.k_norm : cache.v_norm;
            reinterpret_cast<float*>(sm + kPxBuf + (tid < 128 ? kPfImgKN : kPfImgVN) - kPfImgV)[kk] =
                kk < n ? __ldg(nrm + crow0 + t0 + kk) : 0.f;
        }
        // V tile: lanes take consecutive dim pairs (2 jp, 2 jp + 1) of the same
        // rows; thread = (dim pair tid % 64, groups (tid / 64) + 4 i of 8
        // positions); entry (c[idx(t, j)], c[idx(t + 1, j)])
        {
            const int jp = tid & 63;
            constexpr uint32_t M = (1u << VB) - 1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t8 = (tid >> 6) + 4 * i;
                uint32_t f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    f[u] = 8 * t8 + u < nr ? pf_bits<2 * VB>(reinterpret_cast<const uint32_t*>(sv + (8 * t8 + u) * (16 * VB)),
                                                             2 * jp * VB)
                                           : 0u;
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    uint32_t c[4];
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        const uint32_t a = (f[2 * pp] >> (jj * VB)) & M;
                        const uint32_t bb = (f[2 * pp + 1] >> (jj * VB)) & M;
                        c[pp] = tvl[kPfCopies * (a | (bb << VB))];
                    }
                    *reinterpret_cast<uint4*>(sm + kPxBuf + pf_chunk(2 * jp + jj, t8)) =
                        make_uint4(c[0], c[1], c[2], c[3]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid >= 128 && tid < 160) {  // the block's largest |V norm|
            const float* vn = reinterpret_cast<const float*>(sm + kPxBuf + kPfImgVN - kPfImgV);
            float v = fmaxf(fmaxf(fabsf(vn[lane]), fabsf(vn[lane + 32])), fmaxf(fabsf(vn[lane + 64]), fabsf(vn[lane + 96])));
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
            if (lane == 0) bmax[(int64_t)bg * nbmax + j] = v;
        }
        if (tid == 0) {
            pf_bulk_store(dsti + kPfImgV, sa + kPxBuf, kPfImgBytes - kPfImgV);
            bulk_commit();
        }
    }
    if (tid == 0) {
        bulk_wait<0>();  // the image stores are complete before the block leaves
        if (!*okf) {  // after a wait that gave up: the staging copies in flight land first (bounded)
            mbar_wait(&bars[k & 1], (k >> 1) & 1);
            if (pre) mbar_wait(&bars[(k + 1) & 1], ((k + 1) >> 1) & 1);
        }
    }
}

// ------------------------------------------------------------------ attention
// The attention kernel does not depend on the bit widths: one copy, in the
// unit of K width 4.
#if TQ_UNIT_KB == 4

// ---- attention kernel
constexpr int kPfRows = 128;           // query rows per CTA
constexpr int kPfThreads = 352;        // warp 0 K copies, warp 1 MMAs, warps 2-9 softmax, warp 10 V copies
constexpr int kPfSoftmax = 256;
constexpr uint32_t kPfKStage = 65536;  // a K stage: the high and low K tiles of a block
constexpr uint32_t kPfKS = 0;          // two K stages (1024-aligned); the exchange and output tiles at the end
constexpr uint32_t kPfQB = kPfKS + kPfKStage;         // prologue, in K stage 1: the bf16 query rows
constexpr uint32_t kPfRot = kPfQB + 32768;            // and the rotation matrix
constexpr uint32_t kPfVS = kPfKS + 2 * kPfKStage;     // two V stages: V tile, K norms, V norms of a block
constexpr uint32_t kPfVStage = kPfImgBytes - kPfImgV;  // 33792 bytes (1024-aligned)
constexpr uint32_t kPfRed = kPfVS + 2 * kPfVStage;     // [2][2][128] floats: per-half row maxima
constexpr uint32_t kPfBar = kPfRed + 2048;             // 15 mbarriers
constexpr uint32_t kPfMisc = kPfBar + 128;             // tensor-memory base, abort flag
constexpr uint32_t kPfQX = kPfMisc + 16;               // the rows' power-of-two query scales (128 floats)
constexpr uint32_t kPfEnd = kPfQX + 512;
constexpr uint32_t kPfSmem = kPfEnd + 1024;            // plus alignment slack
static_assert(kPfSmem <= 232448, "shared memory per CTA");
constexpr uint32_t kPfTO = 256;        // tensor-memory column of the output (and of the rotated rows first)
constexpr uint32_t kPfTQ = 384;        // of the query's high parts; the low parts 64 further
constexpr int kPfStatusWait = 51;      // an MMA, copy or softmax wait gave up
constexpr int kPfStatusRange = 52;     // q_start[b] + T exceeds the cache capacity, or q_start < 0
constexpr float kPfRescale = 8.f;      // move the reference max when the row max grows by more (log2)
constexpr uint32_t kPfOutStride = 528;  // output tile row stride in shared memory at the end
static_assert(128 * kPfOutStride <= 2 * kPfKStage, "the output tile fits the K stages");

// 2^e for -126 <= e <= 127, from the exponent field.
__device__ __forceinline__ float pf_pow2(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

__device__ __forceinline__ float pf_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Barrier among the softmax warps (named barrier 1).
__device__ __forceinline__ void pf_softmax_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kPfSoftmax) : "memory");
}

// Bounded wait for the phase of `bar` with parity `parity`.  Gives up at once
// if the CTA's abort flag is set; a wait that runs out of time sets it and
// the status word.  Returns false if it gave up.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, int parity, volatile int* abort_f, int* status) {
    if (mbar_try_wait(bar, (uint32_t)parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, (uint32_t)parity)) {
        if (*abort_f) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_f = 1;
            report_timeout(status, kPfStatusWait);
            return false;
        }
    }
    return true;
}

// Block (bg, y) takes query tile gridDim.y - 1 - y of (sequence, KV head) bg:
// blocks start in x-fastest order, so the last tiles of every head, which
// read the most KV blocks under the causal mask, start first.
__global__ void __launch_bounds__(kPfThreads, 1)
k_attn_prefill(const __nv_bfloat16* __restrict__ q, const unsigned char* __restrict__ rot,
               const unsigned char* __restrict__ img, int nbmax, int Hq, int Hkv, int T,
               const int32_t* __restrict__ q_start, const float* __restrict__ bmax, int64_t cap,
               float* __restrict__ out, int* status, const __grid_constant__ AttnParams P) {
    extern __shared__ __align__(1024) unsigned char pf_raw[];
    unsigned char* sm = pf_raw + ((1024u - (smem_addr(pf_raw) & 1023u)) & 1023u);
    const uint32_t sa = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hq / Hkv, tpr = kPfRows / G;
    const int bg = blockIdx.x, b = bg / Hkv, g = bg - b * Hkv;
    const int mt = (int)(gridDim.y - 1 - blockIdx.y);
    const int rows_total = T * G;
    int64_t qs = __ldg(q_start + b);
    const int last_tok = min(T, (mt + 1) * tpr) - 1;
    if (qs < 0 || qs + T > cap) {  // nothing sensible to read: report and write zeros
        if (tid == 0) report_timeout(status, kPfStatusRange);
        qs = -1;
    }
    const int64_t kv_end = qs < 0 ? 0 : qs + last_tok + 1;  // positions this CTA reads
    const int nblk = (int)((kv_end + kPfBlock - 1) / kPfBlock);
    // Block j: K stage, V stage and tensor-memory S/P buffer j % 2.
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kPfBar);
    uint64_t* kfull = bars;         // [2] the K tiles of the stage's block have landed
    uint64_t* vfull = bars + 2;     // [2] its V tile and norms have landed
    uint64_t* s_full = bars + 4;    // [2] S of the block is done (its K stage is free)
    uint64_t* p_full = bars + 6;    // [2] the eight softmax warps wrote P over it
    uint64_t* pv_done = bars + 8;   // [2] its PV product completed: V stage and buffer free, O current
    uint64_t* q_in = bars + 10;     // the bf16 query rows and the rotation matrix are in shared memory
    uint64_t* rot_done = bars + 11; // the rotated rows are in tensor memory (the output columns)
    uint64_t* q_full = bars + 12;   // the softmax warps wrote the query's parts to tensor memory
    uint64_t* drain = bars + 13;    // the MMA thread's products in flight, on the abort path
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + kPfMisc);
    volatile int* abort_f = reinterpret_cast<volatile int*>(sm + kPfMisc + 4);
    float* red = reinterpret_cast<float*>(sm + kPfRed);
    float* qx_s = reinterpret_cast<float*>(sm + kPfQX);

    if (tid == 0) {
        for (int i = 0; i < 14; ++i) mbar_init(&bars[i], (i == 6 || i == 7 || i == 12) ? 8u : (i == 10 ? 9u : 1u));
        *abort_f = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc<512>(slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    constexpr uint32_t idesc = umma_idesc_f16(128, 128, false);

    if (warp == 0 || warp == 10) {
        // ---- copies: warp 0 the K tiles of block j into K stage j % 2 once S
        // of block j - 2 is done (block 1 once the rotation has read the
        // prologue's operands there), warp 10 the V tile and norms into V stage
        // j % 2 once the PV product of block j - 2 is
        if (lane == 0) {
            const bool kside = warp == 0;
            uint64_t* fb = kside ? kfull : vfull;
            if (kside) {  // the rotation matrix, B operand of the query rotation
                mbar_arrive_expect_tx(q_in, 32768);
                bulk_load(sa + kPfRot, rot, 32768, q_in);
            }
            int issued = 0;
            for (int j = 0; j < nblk; ++j) {
                const int s = j & 1;
                bool ok = true;
                if (kside && j == 1) ok = pf_wait(rot_done, 0, abort_f, status);
                if (ok && j >= 2) ok = pf_wait(kside ? &s_full[s] : &pv_done[s], ((j - 2) >> 1) & 1, abort_f, status);
                if (!ok) break;
                const unsigned char* src = img + ((int64_t)bg * nbmax + j) * kPfImgBytes;
                if (kside) {
                    mbar_arrive_expect_tx(&kfull[s], kPfKStage);
                    bulk_load(sa + kPfKS + s * kPfKStage, src + kPfImgK, kPfKStage, &kfull[s]);
                } else {
                    mbar_arrive_expect_tx(&vfull[s], kPfVStage);
                    bulk_load(sa + kPfVS + s * kPfVStage, src + kPfImgV, kPfVStage, &vfull[s]);
                }
                issued = j + 1;
            }
            // the copies issued have landed before the CTA leaves (bounded;
            // regardless of the abort flag)
            for (int j = issued >= 2 ? issued - 2 : 0; j < issued; ++j) mbar_wait(&fb[j & 1], (j >> 1) & 1);
            if (kside) mbar_wait(q_in, 0);
        }
    } else if (warp == 1) {
        // ---- MMAs: the query rotation, then S of block j and the PV product
        // of block j - 1
        if (lane == 0) {
            // the query rotation: rows (bf16, A) times the rotation matrix (B)
            bool ok = pf_wait(q_in, 0, abort_f, status);
            if (ok) {
                tc_fence_after();
                constexpr uint32_t idesc_bf = umma_idesc_f16(128, 128, true);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    umma_f16(tmem + kPfTO, umma_desc_sw128(sa + kPfQB + off), umma_desc_sw128(sa + kPfRot + off),
                             idesc_bf, kk > 0 ? 1u : 0u);
                }
                umma_commit(rot_done);
                ok = pf_wait(q_full, 0, abort_f, status);
            }
            for (int j = 0; ok && j <= nblk; ++j) {
                if (j < nblk) {
                    const int s = j & 1;
                    // the buffer last held P of block j - 2
                    ok = pf_wait(&kfull[s], (j >> 1) & 1, abort_f, status) &&
                         (j < 2 || pf_wait(&pv_done[s], ((j - 2) >> 1) & 1, abort_f, status));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kt = sa + kPfKS + s * kPfKStage;
                    const uint32_t d = tmem + 128 * s;
                    // S = Q_hi K_hi^T + Q_lo K_hi^T + Q_hi K_lo^T; dims 16 kk ..
                    // 16 kk + 15 of the query at column 8 kk of its part
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        umma_f16_ts(d, tmem + kPfTQ + 8 * kk, umma_desc_sw128(kt + off), idesc, kk > 0 ? 1u : 0u);
                    }
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        umma_f16_ts(d, tmem + kPfTQ + 64 + 8 * kk, umma_desc_sw128(kt + off), idesc, 1u);
                    }
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        umma_f16_ts(d, tmem + kPfTQ + 8 * kk, umma_desc_sw128(kt + kPfImgD + off), idesc, 1u);
                    }
                    umma_commit(&s_full[s]);
                }
                if (j >= 1) {
                    const int jj = j - 1, s = jj & 1;
                    ok = pf_wait(&vfull[s], (jj >> 1) & 1, abort_f, status) &&
                         pf_wait(&p_full[s], (jj >> 1) & 1, abort_f, status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t vt = sa + kPfVS + s * kPfVStage;
                    // P of positions 16 kk .. 16 kk + 15: high parts at column
                    // 64 (kk / 4) + 8 (kk % 4) of the buffer, low parts 32 further
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint32_t a = tmem + 128 * s + 64 * (kk >> 2) + 8 * (kk & 3);
                        umma_f16_ts(tmem + kPfTO, a, umma_desc_sw128(vt + off), idesc, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint32_t a = tmem + 128 * s + 64 * (kk >> 2) + 8 * (kk & 3) + 32;
                        umma_f16_ts(tmem + kPfTO, a, umma_desc_sw128(vt + off), idesc, 1u);
                    }
                    umma_commit(&pv_done[s]);
                }
            }
            if (!ok) {  // the products in flight finish before the tensor memory is freed (bounded)
                umma_commit(drain);
                mbar_wait(drain, 0);
            }
        }
    } else {
        // ---- softmax (warps 2-9): row r of the tile, columns 64 hf .. 64 hf + 63
        const int qd = warp & 3, hf = (warp - 2) >> 2;
        const int r = 32 * qd + lane;
        const int grow = mt * kPfRows + r;  // the row within (b, g)
        const bool rvalid = grow < rows_total;
        const int tok = rvalid ? grow / G : 0;
        const uint32_t t_lane = tmem + ((uint32_t)(32 * qd) << 16);
        // Query: warp w stages rows 16 (w - 2) .. + 15 as bf16 (zero rows past
        // the chunk's last token) for the rotation product; from the rotated
        // rows each thread then writes its 64 columns as fp16 high and low parts
        // over a power of two 2^e per row that keeps them below 2^14, into the
        // query's tensor-memory columns, and the MMA thread takes them through
        // q_full
        {
            uint2 raw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int gr = mt * kPfRows + 16 * (warp - 2) + i;
                raw[i] = make_uint2(0u, 0u);
                if (gr < rows_total) {
                    const int tk = gr / G, hd = gr - tk * G;
                    raw[i] = __ldg(reinterpret_cast<const uint2*>(q + (((int64_t)b * T + tk) * Hq + g * G + hd) * 128) +
                                   lane);
                }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
                *reinterpret_cast<uint2*>(sm + kPfQB + pf_chunk(16 * (warp - 2) + i, lane >> 1) + (lane & 1) * 8) =
                    raw[i];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_in);
        // E: the largest V norm this CTA reads is below 2^E (from the blocks' maxima)
        int E = 0;
        {
            float vm = 0.f;
            for (int t = lane; t < nblk; t += 32) vm = fmaxf(vm, __ldg(bmax + (int64_t)bg * nbmax + t));
            for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, o));
            if (vm > 0.f && vm <= FLT_MAX) frexpf(vm, &E);  // vm < 2^E
        }
        {
            pf_wait(rot_done, 0, abort_f, status);
            __syncwarp();
            tc_fence_after();
            uint32_t y0[32], y1[32];
            tmem_ld32(t_lane + kPfTO + 64 * hf, y0);
            tmem_ld32(t_lane + kPfTO + 64 * hf + 32, y1);
            tmem_wait_ld();
            float y[64];
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                y[i] = __uint_as_float(y0[i]) * P.q_mul;
                y[32 + i] = __uint_as_float(y1[i]) * P.q_mul;
                a = fmaxf(a, fmaxf(fabsf(y[i]), fabsf(y[32 + i])));
            }
            red[hf * 128 + r] = a;
            pf_softmax_sync();
            a = fmaxf(red[r], red[128 + r]);
            int e = 0;
            if (a > 0.f && a <= FLT_MAX) {
                const int ex = (int)((__float_as_uint(a) >> 23) & 0xFFu) - 126;  // a in [2^(ex-1), 2^ex)
                e = min(100, max(-100, ex - 14));
            }
            const float inv = pf_pow2(-e);  // exact scaling by a power of two
            uint32_t qh[32], ql[32];  // dims 64 hf + 2 u, + 1 as fp16 pairs
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const float v0 = y[2 * u] * inv, v1 = y[2 * u + 1] * inv;
                const __half2 hh2 = __floats2half2_rn(v0, v1);
                const float2 hf2 = __half22float2(hh2);
                const __half2 ll2 = __floats2half2_rn(v0 - hf2.x, v1 - hf2.y);
                qh[u] = *reinterpret_cast<const uint32_t*>(&hh2);
                ql[u] = *reinterpret_cast<const uint32_t*>(&ll2);
            }
            tmem_st32(t_lane + kPfTQ + 32 * hf, qh);
            tmem_st32(t_lane + kPfTQ + 64 + 32 * hf, ql);
            tmem_wait_st();
            if (hf == 0) qx_s[r] = rvalid ? pf_pow2(e) : 0.f;
        }
        tc_fence_before();
        pf_softmax_sync();
        if (lane == 0) mbar_arrive(q_full);
        const float qx = qx_s[r];

        const int64_t pos = qs + tok;  // this row attends [0, pos]
        const float qxs = rvalid ? qx : 1.f;
        const float inv2E = ldexpf(1.f, -E);
        const F2 QX = f2(qxs, qxs), IE = f2(inv2E, inv2E);
        float m = -INFINITY, l = 0.f;  // reference max (s' units) and this half's sum
        for (int j = 0; j < nblk; ++j) {
            const int s = j & 1, ph = (j >> 1) & 1;
            const int64_t t0 = (int64_t)j * kPfBlock;
            const int nv = kv_end - t0 < kPfBlock ? (int)(kv_end - t0) : kPfBlock;
            pf_wait(&vfull[s], ph, abort_f, status);  // the norms of the block
            pf_wait(&s_full[s], ph, abort_f, status);
            __syncwarp();
            tc_fence_after();
            const unsigned char* stg = sm + kPfVS + s * kPfVStage - kPfImgV;  // image offsets
            const float* kn = reinterpret_cast<const float*>(stg + kPfImgKN) + 64 * hf;
            const float2* vn2 = reinterpret_cast<const float2*>(stg + kPfImgVN) + 32 * hf;
            const uint32_t t_buf = t_lane + 128 * s + 64 * hf;
            // s' = S |k| per column; the row's scores in log2 units are s' qx
            // (qx > 0), so the max is kept in s' units and p = exp2(s' qx - m qx).
            // Columns inside the row's range for the whole half skip the mask.
            float sv[64];
            float mx = -INFINITY;
            {
                uint32_t sr0[32], sr1[32];
                tmem_ld32(t_buf, sr0);
                tmem_ld32(t_buf + 32, sr1);
                tmem_wait_ld();
                const bool whole = rvalid && 64 * hf + 63 < nv && t0 + 64 * hf + 63 <= pos;
                if (whole) {
                    const float4* kn4 = reinterpret_cast<const float4*>(kn);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float4 kk = kn4[i];
                        const uint32_t* sr = i < 8 ? sr0 + 4 * i : sr1 + 4 * (i - 8);
                        f2_split(f2_mul(f2(__uint_as_float(sr[0]), __uint_as_float(sr[1])), f2(kk.x, kk.y)),
                                 sv[4 * i], sv[4 * i + 1]);
                        f2_split(f2_mul(f2(__uint_as_float(sr[2]), __uint_as_float(sr[3])), f2(kk.z, kk.w)),
                                 sv[4 * i + 2], sv[4 * i + 3]);
                        mx = fmaxf(mx, fmaxf(fmaxf(sv[4 * i], sv[4 * i + 1]), fmaxf(sv[4 * i + 2], sv[4 * i + 3])));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int k = 64 * hf + i;
                        const bool valid = rvalid && k < nv && t0 + k <= pos;
                        const uint32_t raw = i < 32 ? sr0[i] : sr1[i - 32];
                        sv[i] = valid ? __uint_as_float(raw) * kn[i] : -INFINITY;
                        mx = fmaxf(mx, sv[i]);
                    }
                }
            }
            red[(s * 2 + hf) * 128 + r] = mx;
            pf_softmax_sync();
            const float m_new = fmaxf(m, fmaxf(red[(s * 2) * 128 + r], red[(s * 2 + 1) * 128 + r]));
            // both threads of a row take the same decisions (same inputs)
            const bool move = m == -INFINITY || (m_new - m) * qxs > kPfRescale;
            const bool rescale = move && m != -INFINITY;  // O holds earlier blocks: scale it
            if (__any_sync(0xFFFFFFFFu, rescale)) {
                // the PV product of block j - 1 is the last one that wrote O
                pf_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_f, status);
                __syncwarp();
                tc_fence_after();
                const float alpha = rescale ? pf_exp2((m - m_new) * qxs) : 1.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_lane + kPfTO + 64 * hf + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(t_lane + kPfTO + 64 * hf + 32 * c, o);
                }
                if (rescale) l *= alpha;
            }
            if (move) m = m_new;
            const float nmq = m == -INFINITY ? 0.f : -m * qxs;  // masked columns: exp2(-inf) = 0
            const F2 NMQ = f2(nmq, nmq);
            F2 LB = f2(0.f, 0.f);
            uint32_t ph2[32], pl2[32];  // P of positions 64 hf + 2 u, + 1 as fp16 pairs
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                float a0, a1;
                f2_split(f2_fma(f2(sv[2 * u], sv[2 * u + 1]), QX, NMQ), a0, a1);
                const F2 pp = f2(pf_exp2(a0), pf_exp2(a1));
                LB = f2_add(LB, pp);
                const float2 vv = vn2[u];
                float w0, w1;
                f2_split(f2_mul(pp, f2_mul(f2(vv.x, vv.y), IE)), w0, w1);
                const __half2 hh2 = __floats2half2_rn(w0, w1);
                const float2 hf2 = __half22float2(hh2);
                const __half2 ll2 = __floats2half2_rn(w0 - hf2.x, w1 - hf2.y);
                ph2[u] = *reinterpret_cast<const uint32_t*>(&hh2);
                pl2[u] = *reinterpret_cast<const uint32_t*>(&ll2);
            }
            tmem_st32(t_buf, ph2);
            tmem_st32(t_buf + 32, pl2);
            tmem_wait_st();
            {
                float lb0, lb1;
                f2_split(LB, lb0, lb1);
                l += lb0 + lb1;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[s]);
        }

        // ---- epilogue: normalise (the row's sum over its two halves) and
        // rotate back, s . H (s2 . o) / sqrt(d): H over the 7 index bits of a
        // row is the butterflies over bits 0-5 (a thread's half, in
        // registers) and over bit 6 (between the two threads of the row,
        // through shared memory laid out [half][element / 4][row] in float4;
        // the K stages, free once the last product is done).
        float O[64];
        if (nblk > 0) {
            const int jl = nblk - 1;
            pf_wait(&pv_done[jl & 1], (jl >> 1) & 1, abort_f, status);
            __syncwarp();
            tc_fence_after();
            uint32_t o0[32], o1[32];
            tmem_ld32(t_lane + kPfTO + 64 * hf, o0);
            tmem_ld32(t_lane + kPfTO + 64 * hf + 32, o1);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                O[i] = __uint_as_float(o0[i]);
                O[32 + i] = __uint_as_float(o1[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) O[i] = 0.f;
        }
        float* lsum = red + ((nblk & 1) * 2) * 128;  // the buffer block nblk - 1 did not use
        lsum[hf * 128 + r] = l;
        pf_softmax_sync();
        const float lt = lsum[r] + lsum[128 + r];
        const float sc = lt > 0.f ? ldexpf(P.out_mul, E) / lt * P.inv_sqrt_d : 0.f;
        if (P.two_sided) {
#pragma unroll
            for (int i = 0; i < 64; ++i) O[i] = __uint_as_float(__float_as_uint(O[i]) ^ P.sgn2[64 * hf + i]);
        }
        fwht_reg2<64>(O);
        float4* xs = reinterpret_cast<float4*>(sm + kPfKS);
#pragma unroll
        for (int i = 0; i < 16; ++i) xs[(hf * 16 + i) * 128 + r] = make_float4(O[4 * i], O[4 * i + 1], O[4 * i + 2], O[4 * i + 3]);
        pf_softmax_sync();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 o = xs[((hf ^ 1) * 16 + i) * 128 + r];
            const float oo[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) O[4 * i + k] = hf ? oo[k] - O[4 * i + k] : O[4 * i + k] + oo[k];  // (lo + hi, lo - hi)
        }
        pf_softmax_sync();  // the exchange is read: the K stages take the output tile
        // The output tile, row-major with rows kPfOutStride bytes apart (512
        // bytes of data and 16 of padding, so the per-row writes hit distinct
        // banks).  Lanes 0-15 of each softmax warp then send 16 rows with one
        // bulk store each, and wait only until shared memory has been read.
        unsigned char* ot = sm + kPfKS;
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
            const int jd = 64 * hf + i;
            float4 v;
            v.x = __uint_as_float(__float_as_uint(O[i] * sc) ^ P.sgn[jd]);
            v.y = __uint_as_float(__float_as_uint(O[i + 1] * sc) ^ P.sgn[jd + 1]);
            v.z = __uint_as_float(__float_as_uint(O[i + 2] * sc) ^ P.sgn[jd + 2]);
            v.w = __uint_as_float(__float_as_uint(O[i + 3] * sc) ^ P.sgn[jd + 3]);
            *reinterpret_cast<float4*>(ot + r * kPfOutStride + jd * 4) = v;
        }
        fence_proxy_async_smem();
        pf_softmax_sync();
        if (lane < 16 && *abort_f == 0) {
            const int rr = 16 * (warp - 2) + lane;
            const int gr = mt * kPfRows + rr;
            if (gr < rows_total) {
                const int tk = gr / G, hd = gr - tk * G;
                pf_bulk_store(out + (((int64_t)b * T + tk) * Hq + g * G + hd) * 128, sa + kPfKS + rr * kPfOutStride,
                              512);
                bulk_commit();
                bulk_wait_read<0>();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<512>(tmem);
    }
}

#endif  // TQ_UNIT_KB == 4

static cudaError_t set_smem_once(const void* fn, int bytes, int* done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
    return e;
}

template <int KB, int VB>
cudaError_t prefill_expand(int B, int T, int Hkv, const int32_t* q_start, const tq_cache_view& cache,
                           unsigned char* ws, const AttnParams& P, cudaStream_t s) {
    unsigned char* img = ws + kPfRotBytes;
    float* bmax = reinterpret_cast<float*>(img + attn_prefill_img_bytes(B, Hkv, cache.cap));
    auto fn = k_prefill_expand<KB, VB>;
    static int attr_done[64] = {};
    cudaError_t e = set_smem_once((const void*)fn, (int)kPxSmem, attr_done);
    if (e != cudaSuccess) return e;
    const int nbmax = (int)((cache.cap + kPfBlock - 1) / kPfBlock);
    const int groups = B * Hkv;
    int x = 608 / groups;  // about four CTAs per SM in all
    x = x < 1 ? 1 : (x > nbmax ? nbmax : x);
    fn<<<dim3((unsigned)x + 1, (unsigned)groups), kPxThreads, kPxSmem, s>>>(q_start, T, Hkv, cache, nbmax, img, bmax,
                                                                          reinterpret_cast<uint4*>(ws), status_word(), P);
    return cudaGetLastError();
}

}  // namespace dev

#if TQ_UNIT_KB == 4
cudaError_t launch_prefill_attention(const void* q, int B, int T, int Hq, int Hkv, const int32_t* q_start,
                                     const tq_cache_view& cache, float* out, void* workspace,
                                     const AttnParams& P, cudaStream_t s) {
    using namespace dev;
    const unsigned char* rot = static_cast<const unsigned char*>(workspace);
    const unsigned char* img = rot + kPfRotBytes;
    static int attr_done[64] = {};
    cudaError_t e = set_smem_once((const void*)k_attn_prefill, (int)kPfSmem, attr_done);
    if (e != cudaSuccess) return e;
    const int G = Hq / Hkv;
    const int nbmax = (int)((cache.cap + kPfBlock - 1) / kPfBlock);
    const dim3 grid((unsigned)(B * Hkv), (unsigned)(((int64_t)T * G + kPfRows - 1) / kPfRows));
    const float* bmax = reinterpret_cast<const float*>(img + attn_prefill_img_bytes(B, Hkv, cache.cap));
    k_attn_prefill<<<grid, kPfThreads, kPfSmem, s>>>(static_cast<const __nv_bfloat16*>(q), rot, img, nbmax, Hq, Hkv,
                                                     T, q_start, bmax, cache.cap, out, status_word(), P);
    return cudaGetLastError();
}
#endif

template <int KB>
cudaError_t launch_attn_prefill(int v_bits, const void* q, int B, int T, int Hq, int Hkv, const int32_t* q_start,
                                const tq_cache_view& cache, float* out, void* workspace, const AttnParams& P,
                                cudaStream_t s) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    cudaError_t e;
    switch (v_bits) {
        case 2: e = dev::prefill_expand<KB, 2>(B, T, Hkv, q_start, cache, ws, P, s); break;
        case 3: e = dev::prefill_expand<KB, 3>(B, T, Hkv, q_start, cache, ws, P, s); break;
        default: e = dev::prefill_expand<KB, 4>(B, T, Hkv, q_start, cache, ws, P, s); break;
    }
    if (e != cudaSuccess) return e;
    return launch_prefill_attention(q, B, T, Hq, Hkv, q_start, cache, out, workspace, P, s);
}

template cudaError_t launch_attn_prefill<TQ_UNIT_KB>(int, const void*, int, int, int, int, const int32_t*,
                                                     const tq_cache_view&, float*, void*, const AttnParams&,
                                                     cudaStream_t);

}  // namespace tq
