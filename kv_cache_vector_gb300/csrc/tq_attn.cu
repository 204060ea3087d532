// tq_attn.cu -- decode attention over the packed cache at d = 128, on the
// tensor cores (the other head dimensions and QJL keys: tq_attn_generic.cu).
//
// "TurboQuant KV Cache Compression -- Spec", Optimization: Fused dequant-dot:
// rotate q once, score each cached position against its centroids
// ((Rq).(Rk) = q.k), accumulate V in the rotated domain, rotate the output
// back once.  Split-K flash-decode with fp32 partials merged by log-sum-exp.
// "CITATIONS", Sparse V dequant: a V row is skipped when every head's
// exp(sigma - m) is below the threshold; it still counts in l.
#include <cfloat>
#include <type_traits>

#include <cuda_fp16.h>

#include "tq_async.cuh"
#include "tq_device.cuh"

namespace tq {
namespace dev {

// ============================================================ d = 128
//
// Tensor-core flash-decode (mma.sync m16n8k16: fp16 operands, fp32
// accumulation) over chunks of 32 positions, processed as two sub-tiles of
// 16 positions.
//
//   S^T = K Q~    A = K centroids of 16 positions (rows) x 16 dims, looked
//                 up as pairs (two consecutive dims, fp16 x 2) in a lane-
//                 replicated table; B = the rotated query, 8 columns = 4
//                 query heads x (fp16 high part, fp16 low part).  The score
//                 of a head is the sum of its two columns, so the query keeps
//                 about 22 significant bits.  The 128 contraction dims are
//                 permuted so that lane t reads dims 32t..32t+31 of a K row;
//                 a dot product does not depend on the order.
//   softmax       exp2 with a lazily updated running maximum (updated only
//                 when a chunk's maximum exceeds it by more than kLazy, so
//                 p <= 2^kLazy), fp32 denominators.
//   O^T += V^T P  A = V centroids, 16 dims (rows) x 16 positions, from pair
//                 lookups of four positions and byte permutes; B = p times the
//                 V norm, 8 columns = 4 heads x (high, low part).  Row g of
//                 m-tile mt is dim 16g + 2mt, row g + 8 is dim 16g + 2mt + 1,
//                 so lane row g ends up holding dims 16g..16g+15.
// The tables hold fp16 values of c * s, with the scale s chosen on the host
// so that every centroid of the width is close to its fp16 value (worst
// relative error about 1e-4 at 4 bits, 3e-5 at 3 bits); 1/s_k is folded into
// the query and 1/s_v into the output.  Query heads go in groups of four:
// NG = 1 for G <= 4, NG = 2 for G <= 8.
//
// Data movement: CTAs of W warps take contiguous ranges of work items
// (batch, KV head, segment of W * warp_len positions); the segment is cut
// into chunks of 32 positions and warp w takes chunks w, w + W, w + 2W, ...,
// so the rows of a segment that a sequence fills spread evenly over the
// warps.  A warp streams its own chunks through a ring of 2 or 3 stages in
// shared memory: one lane issues 1-D bulk copies (cp.async.bulk) of the
// chunk's packed K and V rows, each lane copies the two norms of one
// position (cp.async, 4 bytes), and one mbarrier per stage completes when
// all of it has landed.  When the (batch, KV head) of the items changes and
// at the end of the range, the warps merge their partials through shared
// memory and write one partial (acc[128], m, l) per query head;
// k_attn3_combine merges a (batch, head)'s partials.

constexpr int kA3Chunk = 32;
constexpr int kA3MergeStride = kAttn3MergeRow / 4;  // floats per (warp, head) row of the merge buffer
constexpr float kLazy = 8.0f;        // log2 units
// Shared memory is addressed by absolute shared-window address.  The pair
// table starts at 128 KiB: entry e of lane l's column is at
// kA3TableAt + e * 256 + 4 * l (K) or + 128 + 4 * l (V), so a lookup address
// is (e << 8) | slot, one byte permute for a 4-bit pair.
constexpr uint32_t kA3RingAt = kAttn3RingAt;
constexpr uint32_t kA3TableAt = kAttn3TableAt;
// Device status codes.
constexpr int kA3StatusWait = 31;    // a ring stage did not complete within the bound
constexpr int kA3StatusLayout = 32;  // dynamic shared memory starts above kA3RingAt
constexpr int kA3StatusPage = 33;    // a paged cache's block table names a page out of range
constexpr int kA3StatusAppend = 42;  // an appended row's position or page is out of range (as the append)

// Warps, ring stages and the shared-memory plan per CTA (attn3_plan): up to
// 16 warps x 2 stages for up to four query heads per KV head, 8 x 3 for up to
// eight.
// QJL: keys in the QJL residual format, KB bits in total (a KB - 1 bit index
// per coordinate, then the 128 sign bits of the projected residual).
template <int KB, int VB, int NG, bool SP = false, bool QJL = false>
struct A3Shape {
    static constexpr Attn3Plan kPlan = attn3_plan(4 * NG, KB, VB, SP, QJL);
    static constexpr int kWarps = kPlan.warps;
    static constexpr int kStages = kPlan.stages;
    static constexpr int kThreads = 32 * kWarps;
    static_assert(kWarps > 0, "no shared-memory plan");
};

template <int KB, int VB, int NG, bool SP = false, bool QJL = false>
struct A3Layout {
    static_assert(!(SP && QJL), "QJL keys run dense");
    static constexpr Attn3Plan kPlan = A3Shape<KB, VB, NG, SP, QJL>::kPlan;
    static constexpr int kWarps = kPlan.warps, kStages = kPlan.stages;
    static constexpr int kMB = QJL ? KB - 1 : KB;            // index bits per key coordinate
    static constexpr int kSignOff = 16 * kMB;                 // QJL: the sign words of a key row
    static constexpr int kKRow = 16 * KB, kVRow = 16 * VB;  // bytes of a d = 128 row
    static constexpr int kVOff = kA3Chunk * kKRow;  // V rows in the stage (not SP)
    static constexpr int kKnOff = kA3Chunk * (kKRow + (SP ? 0 : kVRow));
    static constexpr int kVnOff = kKnOff + 4 * kA3Chunk;
    static constexpr int kGnOff = kVnOff + 4 * kA3Chunk;      // QJL: the keys' gammas
    static constexpr int kStage = (QJL ? kGnOff : kVnOff) + 4 * kA3Chunk;
    static constexpr int kVBuf = kA3Chunk * kVRow;  // SP: one chunk's V rows; two per warp after its stages
    static constexpr int kWarpRing = kPlan.stages * kStage + (SP ? 2 * kVBuf : 0);
    static_assert(kWarpRing == attn3_warp_ring_bytes(KB, VB, kPlan.stages, SP, QJL), "ring size");
    static constexpr int kEntries = 256;  // rows of the pair table (one byte of index)
    static constexpr int kHeads = 4 * NG;
    // keys that carry their rest: 8-byte key entries (high and low fp16
    // pairs), 16 columns shared by lanes l and l + 16
    static constexpr bool kRest = attn3_key_rest(kMB);
    static constexpr int kMergeHeads = kPlan.merge_heads;
    static constexpr uint32_t kMergeAt = (uint32_t)kPlan.merge;
    static constexpr uint32_t kBarAt = (uint32_t)kPlan.bars;
    static constexpr uint32_t kEnd = (uint32_t)kPlan.end;
    static_assert(kStage % 16 == 0, "stage alignment");
    static_assert(kA3RingAt + kWarps * kWarpRing <= kA3TableAt, "ring overlaps the table");
    static_assert(kBarAt % 8 == 0 && kMergeAt % 16 == 0, "alignment");
    static_assert(kEnd <= (uint32_t)kAttn3SmemTop, "more than 227 KiB of shared memory");
};

__device__ __forceinline__ uint32_t h2u(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Unsigned keys that order as the floats do (for an integer atomic maximum).
__device__ __forceinline__ uint32_t f2ord(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Work items are split over the CTAs of the grid as contiguous ranges:
// CTA c takes items [n_items c / grid, n_items (c + 1) / grid).  The CTA that
// takes item i:
__host__ __device__ __forceinline__ int attn3_cta_of(int64_t i, int grid, int64_t n_items) {
    return (int)(((i + 1) * grid - 1) / n_items);
}

// Table lookup (the table is written once, before the first barrier).
__device__ __forceinline__ uint32_t lds_tab(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
// Both fp16 parts of a key pair (x: the values nearest c * s_k, y: their rests).
__device__ __forceinline__ uint2 lds_tab2(uint32_t addr) {
    uint2 v;
    asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
// Loads of ring data: volatile, so that they stay after the stage's wait.
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) { return __uint_as_float(lds_u32(addr)); }
__device__ __forceinline__ uint2 lds_v2(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Lookup address of pair q (stream order) of a packed field held in the NW
// words w: the byte holding the pair's first bit -- of w itself, or of w
// shifted right by the pair's bit offset within a byte -- lands in bits
// 8..15 of `slot` (table base + column) by one byte permute.  The table has
// 256 rows and row e holds the pair e mod 2^(2 BITS), so the bits of the next
// pair that share the byte do not matter.  Shifted words with the same
// (offset, word) are common subexpressions across q.
template <int BITS, int NW>
__device__ __forceinline__ uint32_t pair_addr(const uint32_t (&w)[NW], int q, uint32_t slot) {
    const int o = q * 2 * BITS, sh = o & 7, byte = o >> 3, wi = byte >> 2, bi = byte & 3;
    uint32_t x;
    if (sh == 0) x = w[wi];
    else if (wi + 1 < NW) x = __funnelshift_r(w[wi], w[wi + 1], sh);
    else x = w[wi] >> sh;
    return __byte_perm(x, slot, 0x7604u | ((uint32_t)bi << 4));
}

// The 32 dims 32t..32t+31 of a K row (KB words).
template <int KB>
__device__ __forceinline__ void load_kfield(uint32_t addr, uint32_t (&w)[KB]) {
    if constexpr (KB == 4) {
        const uint4 u = lds_v4(addr);
        w[0] = u.x;
        w[1] = u.y;
        w[2] = u.z;
        w[3] = u.w;
    } else if constexpr (KB == 3) {
        w[0] = lds_u32(addr);
        w[1] = lds_u32(addr + 4);
        w[2] = lds_u32(addr + 8);
    } else {
        const uint2 u = lds_v2(addr);
        w[0] = u.x;
        w[1] = u.y;
    }
}

// The 16 dims 16g..16g+15 of a V row starting at `row`, as bits 0.. of f.
template <int VB>
__device__ __forceinline__ void load_vfield(uint32_t row, int g, uint32_t (&f)[2]) {
    if constexpr (VB == 4) {
        const uint2 u = lds_v2(row + 8 * g);
        f[0] = u.x;
        f[1] = u.y;
    } else if constexpr (VB == 3) {
        // 6 bytes at byte 6g: read the aligned 8 bytes holding them
        const uint32_t a = row + ((6u * g) & ~3u);
        const uint32_t w0 = lds_u32(a), w1 = lds_u32(a + 4);
        const uint32_t sh = (g & 1) << 4;
        f[0] = __funnelshift_r(w0, w1, sh);
        f[1] = w1 >> sh;
    } else {
        f[0] = lds_u32(row + 4 * g);
        f[1] = 0u;
    }
}

// Rotated queries: y = H (s . q) * q_mul (q_mul = scale * log2(e) /
// (sqrt(d) * s_k)), stored per (batch, head) as qexp = 2^e and fp16 high and
// low parts of y / 2^e, with e chosen so that max |y| / 2^e is in
// [2^13, 2^14).  q16 layout: [B * Hq][2 (high, low)][128].
__device__ __forceinline__ void attn3_rotate_q(const __nv_bfloat16* __restrict__ q, __half* __restrict__ q16,
                                               float* __restrict__ qexp, const AttnParams& P) {
    const int64_t bh = blockIdx.x;
    rotate_q_row(q + bh * 128, q16 + bh * 256, qexp + bh, P);
}

// The same rotation with one warp per (batch, head), eight per block: lane l
// holds elements 4 l .. 4 l + 3, the butterflies over index bits 0 and 1 are
// in registers and those over bits 2-6 between lanes, in the order len = 1,
// 2, .., 64, and the scale and the fp16 parts are those of rotate_q_row.
// y_out (or nullptr): the lane's four elements of s2 . H (s . q) before the
// scale, for the QJL projection.
__device__ __forceinline__ void attn3_q_warp(const __nv_bfloat16* __restrict__ q, __half* __restrict__ q16,
                                             float* __restrict__ qexp, const AttnParams& P, int64_t bh, int lane,
                                             float* y_out) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(q + bh * 128) + lane);
    float x[4];
    {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        x[0] = a.x;
        x[1] = a.y;
        x[2] = c.x;
        x[3] = c.y;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = __uint_as_float(__float_as_uint(x[k]) ^ sign_mask(P.sgnb, 4 * lane + k));
    {
        const float a0 = x[0] + x[1], a1 = x[0] - x[1], a2 = x[2] + x[3], a3 = x[2] - x[3];
        x[0] = a0 + a2;
        x[1] = a1 + a3;
        x[2] = a0 - a2;
        x[3] = a1 - a3;
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, x[k], m);
            x[k] = upper ? o - x[k] : x[k] + o;  // (lo + hi, lo - hi)
        }
    }
    float M = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x[k] = __uint_as_float(__float_as_uint(x[k]) ^ (P.two_sided ? sign_mask(P.sgn2b, 4 * lane + k) : 0u));
        if (y_out) y_out[k] = x[k];
        x[k] *= P.q_mul;
        M = fmaxf(M, fabsf(x[k]));
    }
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    int e = 0;
    if (M > 0.f && M <= FLT_MAX) {
        int ex = 0;
        frexpf(M, &ex);  // M in [2^(ex-1), 2^ex)
        e = min(100, max(-100, ex - 14));
    }
    __half hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float ys = ldexpf(x[k], -e);
        hi[k] = __float2half_rn(ys);
        lo[k] = __float2half_rn(ys - __half2float(hi[k]));
    }
    __half* row = q16 + bh * 256;
    *reinterpret_cast<uint2*>(row + 4 * lane) =
        make_uint2((uint32_t)__half_as_ushort(hi[0]) | ((uint32_t)__half_as_ushort(hi[1]) << 16),
                   (uint32_t)__half_as_ushort(hi[2]) | ((uint32_t)__half_as_ushort(hi[3]) << 16));
    *reinterpret_cast<uint2*>(row + 128 + 4 * lane) =
        make_uint2((uint32_t)__half_as_ushort(lo[0]) | ((uint32_t)__half_as_ushort(lo[1]) << 16),
                   (uint32_t)__half_as_ushort(lo[2]) | ((uint32_t)__half_as_ushort(lo[3]) << 16));
    if (lane == 0) qexp[bh] = ldexpf(1.f, e);
}

// gmax (sparse V, or nullptr): the split kernel's running maxima, cleared here.
static __global__ void __launch_bounds__(256) k_attn3_q(const __nv_bfloat16* __restrict__ q,
                                                        __half* __restrict__ q16,
                                                        float* __restrict__ qexp,
                                                        const __grid_constant__ AttnParams P, int64_t n_rows,
                                                        uint32_t* __restrict__ gmax) {
    griddep_wait();    // the queries, and readers of this call's workspace, of the previous kernel
    griddep_launch();  // the split kernel may start its table build now
    const int lane = threadIdx.x & 31;
    const int64_t bh = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (bh >= n_rows) return;  // the whole warp
    if (gmax && lane == 0) gmax[bh] = 0u;  // below every score's key
    attn3_q_warp(q, q16, qexp, P, bh, lane, nullptr);
}

// The query rotation of the paged attention with the decode step's append
// folded in ("TurboQuant KV Cache Compression -- Spec", fa_tq_attention_cached:
// quantise the new K and V into the cache, then attend).  Block (b, h) rotates
// query head h of sequence b as k_attn3_q does.  The first block of each KV
// head's query group also encodes that head's new K row (warp 0) and V row
// (warp 1) with the row codec of the append and writes them at position
// pa.lens[b]; a position or page id out of range writes nothing and sets the
// status word to 42.  Block (b, 0) writes the attended length pa.lens[b] + 1
// to len1[b] for the planning and split kernels, which run after this launch.
template <typename T>
static __global__ void __launch_bounds__(128) k_attn3_q_append(const __nv_bfloat16* __restrict__ q,
                                                               __half* __restrict__ q16, float* __restrict__ qexp,
                                                               const __grid_constant__ AttnParams P, int Hq, int Hkv,
                                                               const T* __restrict__ k_new, const T* __restrict__ v_new,
                                                               tq_cache_view cache, const PagedArgs pa,
                                                               const __grid_constant__ RowParams PK,
                                                               const __grid_constant__ RowParams PV, int k_bits,
                                                               int v_bits, int32_t* __restrict__ len1, int* status) {
    __shared__ uint32_t sg[128], sg2[128];
    __shared__ uint8_t ib[2][128];
    const int j = threadIdx.x;
    sg[j] = sign_mask(P.sgnb, j);
    sg2[j] = sign_mask(P.sgn2b, j);
    griddep_wait();  // the queries, new rows and cache, and readers of the workspace, of the previous kernel
    griddep_launch();
    const int b = blockIdx.x / Hq, h = blockIdx.x - b * Hq, G = Hq / Hkv;
    const int64_t p = __ldg(pa.lens + b);
    if (h == 0 && j == 0) len1[b] = p < 0 ? 0 : (p >= INT32_MAX ? INT32_MAX : (int32_t)(p + 1));
    attn3_rotate_q(q, q16, qexp, P);  // synchronises the block, so sg is complete
    if (h % G != 0 || j >= 64) return;
    const int warp = j >> 5, lane = j & 31, kvh = h / G;
    const bool is_v = warp == 1;
    const RowParams& R = is_v ? PV : PK;
    const int bits = is_v ? v_bits : k_bits;
    const int64_t cap = (int64_t)pa.max_pages << pa.page_shift;
    const int page = (p >= 0 && p < cap) ? __ldg(pa.bt + (int64_t)b * pa.max_pages + (p >> pa.page_shift)) : -1;
    if (page < 0 || page >= pa.n_pages) {  // warp-uniform: nothing is written for this row
        if (lane == 0) atomicCAS(status, 0, kA3StatusAppend);
        return;
    }
    const int64_t drow = (((int64_t)page * Hkv + kvh) << pa.page_shift) + (p & ((int64_t(1) << pa.page_shift) - 1));
    const T* src = (is_v ? v_new : k_new) + ((int64_t)b * Hkv + kvh) * 128;
    const float n = warp_encode_indices<128, T>(src, lane, sg, P.two_sided ? sg2 : nullptr, R, (1 << bits) - 1,
                                                ib[warp]);
    warp_pack_row<128>(ib[warp], lane, bits, (is_v ? cache.v_packed : cache.k_packed) + drow * (16 * bits));
    if (lane == 0) (is_v ? cache.v_norm : cache.k_norm)[drow] = n;
}

// Work partition of the paged kernel (written by k_attn3_plan): CTA c takes
// items [cta_begin[c], cta_begin[c + 1]); slot_base[c] counts the CTAs before
// c that take any item; c0 / clast hold the first and last CTA taking items
// of each (batch, KV head).
struct A3Meta {
    int32_t* cta_begin;
    int32_t* slot_base;
    int32_t* c0;
    int32_t* clast;
    uint32_t* gmax;  // sparse V: largest score per (batch, query head) so far, zeroed by the query rotation
    // QJL keys: the projected queries (fp16 high and low parts, [B Hq][2][128])
    // and their powers of two, and the keys' gammas [B][Hkv][cap]
    const __half* qp16;
    const float* qpexp;
    const float* k_rnorm;
};
// Weights of the work partition, in rows of the busiest warp: an item that
// holds rows costs its busiest warp's rows plus kA3ItemCost, an empty item
// kA3EmptyCost (the consumer steps over it), and the first item of a
// (batch, KV head) also kA3RunCost (merging the warps' partials and loading
// the query).
constexpr int kA3ItemCost = 4;
constexpr int kA3EmptyCost = 1;
constexpr int kA3RunCost = 128;
constexpr int kA3PlanSmemPairs = 8192;  // pair prefixes kept in shared memory up to this count

// Block-wide inclusive scan over 1024 threads; `total` gets the sum.
__device__ __forceinline__ int64_t block1024_scan(int64_t v, int64_t* wsum, int64_t& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) wsum[wid] = v;
    __syncthreads();
    if (wid == 0) {
        int64_t x = wsum[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t t = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += t;
        }
        wsum[lane] = x;
    }
    __syncthreads();
    const int64_t r = v + (wid > 0 ? wsum[wid - 1] : 0);
    total = wsum[31];
    __syncthreads();
    return r;
}

// The items of one (batch, KV head) with L rows, in split order: nf full
// segments, then a partial one of r rows if r > 0, then empty ones.
struct A3PairCost {
    int64_t nf, wf, wp;
    int has_p;
    __device__ A3PairCost(int64_t L, int64_t seg, int W, int nC) {
        nf = L / seg;
        const int64_t r = L - nf * seg;
        has_p = r > 0;
        wf = (int64_t)nC * kA3Chunk + kA3ItemCost;
        const int64_t f = (r + kA3Chunk - 1) / kA3Chunk;
        wp = (f + W - 1) / W * kA3Chunk + kA3ItemCost;
    }
    // weight of items [0, j)
    __device__ int64_t before(int64_t j) const {
        if (j <= 0) return 0;
        int64_t e = kA3RunCost + (j < nf ? j : nf) * wf;
        if (j > nf && has_p) e += wp;
        const int64_t ne = j - nf - has_p;
        if (ne > 0) e += ne * kA3EmptyCost;
        return e;
    }
};

// One block of 1024 threads.  The W warps of a CTA share each item's chunks
// round robin, so the warp with the most chunks (warp 0) sets the CTA's time
// and the items are weighed in its rows (A3PairCost).  Items are cut into
// `grid` contiguous ranges of about equal weight: item i goes to CTA
// floor(P_i grid / total), P_i the weight of the items before it, so CTA c
// starts at the first item with P_i >= ceil(c total / grid), found by a
// binary search over the pairs' prefix weights and one within the pair.  A
// CTA's range thus runs through consecutive splits of one (batch, KV head)
// at a time.  The kernel runs beside the query rotation launched before it
// (programmatic dependent launch) and waits for it at the end, so that the
// split kernel, which waits for this one, sees the rotated queries too;
// lens_from_prev: lens is written by that launch, so wait for it first.
static __global__ void __launch_bounds__(1024) k_attn3_plan(const int32_t* __restrict__ lens, int Hkv,
                                                            int n_splits, int64_t seg, int warp_len,
                                                            int64_t max_ctx, int n_pairs, int grid, A3Meta m,
                                                            bool lens_from_prev) {
    extern __shared__ __align__(16) unsigned char plan_smem[];
    __shared__ int64_t wsum[32];
    __shared__ int32_t cb[1025];
    if (lens_from_prev) griddep_wait();
    griddep_launch();
    const int tid = threadIdx.x;
    const int W = (int)(seg / warp_len), nC = warp_len / kA3Chunk;
    // exclusive prefix weight of each pair: shared memory, or the c0/clast
    // area of the workspace (8 bytes per pair fit in its 8 bytes per query head)
    int64_t* pre = n_pairs <= kA3PlanSmemPairs ? reinterpret_cast<int64_t*>(plan_smem)
                                               : reinterpret_cast<int64_t*>(m.c0);
    auto pair_len = [&](int bh) {
        int64_t L = __ldg(lens + bh / Hkv);
        return L < 0 ? 0 : (L > max_ctx ? max_ctx : L);
    };
    int64_t carry = 0;
    for (int base = 0; base < n_pairs; base += 1024) {
        const int bh = base + tid;
        const int64_t w = bh < n_pairs ? A3PairCost(pair_len(bh), seg, W, nC).before(n_splits) : 0;
        int64_t chunk_total;
        const int64_t incl = block1024_scan(w, wsum, chunk_total);
        if (bh < n_pairs) pre[bh] = carry + incl - w;
        carry += chunk_total;
    }
    const int64_t total = carry;
    __syncthreads();
    // CTA c's first item
    const int64_t n_items = (int64_t)n_pairs * n_splits;
    if (tid <= grid) {
        int64_t first;
        if (tid == 0) {
            first = 0;
        } else if (tid == grid) {
            first = n_items;
        } else {
            const int64_t t = ((int64_t)tid * total + grid - 1) / grid;  // ceil(c total / grid) > 0
            // the last pair whose prefix is below t (pair 0's is 0 < t)
            int lo = 0, hi = n_pairs;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (pre[mid] < t) lo = mid;
                else hi = mid;
            }
            const A3PairCost pc(pair_len(lo), seg, W, nC);
            const int64_t need = t - pre[lo];
            // the first split j in [1, n_splits] with before(j) >= need; n_splits: the next pair's item 0
            int64_t jl = 0, jh = n_splits;  // before(jl) < need <= before(jh) or jh = n_splits
            while (jh - jl > 1) {
                const int64_t mid = (jl + jh) >> 1;
                if (pc.before(mid) < need) jl = mid;
                else jh = mid;
            }
            first = (int64_t)lo * n_splits + jh;
        }
        cb[tid] = (int32_t)first;
        m.cta_begin[tid] = (int32_t)first;
    }
    __syncthreads();
    // slot bases: a dense numbering of the CTAs that take items
    {
        const int64_t ne = tid < grid ? (cb[tid + 1] > cb[tid] ? 1 : 0) : 0;
        int64_t tot;
        const int64_t incl = block1024_scan(ne, wsum, tot);
        if (tid <= grid) m.slot_base[tid] = (int32_t)(incl - ne);
    }
    // first and last CTA of each pair: the last CTA whose range starts at or before the item
    auto cta_of = [&](int64_t item) {
        int lo = 0, hi = grid;  // cb[lo] <= item < cb[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cb[mid] <= item) lo = mid;
            else hi = mid;
        }
        return lo;
    };
    for (int bh = tid; bh < n_pairs; bh += 1024) {
        const int a = cta_of((int64_t)bh * n_splits), z = cta_of((int64_t)bh * n_splits + n_splits - 1);
        m.c0[bh] = a;
        m.clast[bh] = z;
    }
    griddep_wait();  // the query rotation has completed
}

// PAGED: the cache is paged (PagedArgs), each sequence attends over its own
// length (at most ctx_len) and CTA ranges come from k_attn3_plan; otherwise
// rows are [B][Hkv][cap], every sequence attends over ctx_len and CTA c takes
// items [n_items c / grid, n_items (c + 1) / grid).
// SP (contiguous cache, sparse-V threshold > 0): the producer copies a
// chunk's K rows and norms; the V rows are copied only after the chunk's
// scores, when some query head keeps one of its rows ("CITATIONS", Sparse V
// dequant), and their product is taken one chunk later, with the chunk's
// weights rescaled if the running maximum moves in between.
template <int KB, int VB, int NG, bool PAGED, bool SP, bool QJL = false>
__global__ void __launch_bounds__(A3Shape<KB, VB, NG, SP, QJL>::kThreads, 1)
k_attn3_split(const __half* __restrict__ q16, const float* __restrict__ qexp, int Hq, int Hkv,
              tq_cache_view cache, int64_t ctx_len, int warp_len, int n_splits, int64_t n_items,
              float* __restrict__ part, int* status, const __grid_constant__ AttnParams P,
              const PagedArgs pa, const A3Meta meta) {
    static_assert(!(SP && PAGED), "sparse-V copies are for the contiguous cache");
    static_assert(!(QJL && PAGED), "QJL keys: contiguous cache");
    using L = A3Layout<KB, VB, NG, SP, QJL>;
    constexpr int W = L::kWarps, S = L::kStages, T = A3Shape<KB, VB, NG, SP, QJL>::kThreads;
    constexpr int MB = L::kMB;  // index bits of a key coordinate
    constexpr uint32_t kAll = 0xFFFFFFFFu;
    extern __shared__ __align__(16) unsigned char a3_smem[];
    griddep_launch();  // the combine may be scheduled; it waits for this grid
    const uint32_t base = smem_addr(a3_smem);
    if (base > kA3RingAt) {  // the layout below assumes dynamic memory starts lower
        if (threadIdx.x == 0) report_timeout(status, kA3StatusLayout);
        return;
    }
    auto gptr = [&](uint32_t abs) { return a3_smem + (abs - base); };

    // ---- pair tables and the per-warp barriers
    {
        constexpr int MK = (1 << MB) - 1, MV = (1 << VB) - 1;
        for (int i = threadIdx.x; i < L::kEntries * 64; i += T) {
            const int e = i >> 6, s = i & 63;  // row e holds the pair e mod 2^(2 bits)
            uint32_t v;
            if (s >= 32)
                v = h2u(P.vcen_h[e & MV], P.vcen_h[(e >> VB) & MV]);
            else if (L::kRest && (s & 1))  // words 2c, 2c + 1 of column c: high and low key parts
                v = h2u(P.kcen_l[e & MK], P.kcen_l[(e >> MB) & MK]);
            else
                v = h2u(P.kcen_h[e & MK], P.kcen_h[(e >> MB) & MK]);
            *reinterpret_cast<uint32_t*>(gptr(kA3TableAt + 256u * e + 4u * s)) = v;
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(gptr(L::kBarAt)) + warp * S;
    uint64_t* vbars = reinterpret_cast<uint64_t*>(gptr(L::kBarAt)) + W * S + warp * 2;  // SP: the V buffers
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bars + s, 32);
        if constexpr (SP) {
            mbar_init(vbars, 1);
            mbar_init(vbars + 1, 1);
        }
        mbar_fence_init();
    }
    __syncthreads();
    // everything above depends on the parameters only; from here on the
    // rotated queries (and, paged, the work partition and appended rows) of
    // the previous kernels are read
    griddep_wait();

    const int g = lane >> 2, t = lane & 3;
    const int G = Hq / Hkv;
    const uint32_t kslot = kA3TableAt + (L::kRest ? 8u * (lane & 15) : 4u * lane);
    const uint32_t vslot = kA3TableAt + 128u + 4u * lane;
    const uint32_t ring = kA3RingAt + (uint32_t)(warp * L::kWarpRing);
    const uint32_t vbuf = ring + (uint32_t)(S * L::kStage);  // SP: V buffers 0 and 1
    float* merge = reinterpret_cast<float*>(gptr(L::kMergeAt));
    // Work items, (batch, KV head) pairs and positions fit in 32 bits (the
    // host checks it); only cache row indices take 64.
    const int i_begin = PAGED ? meta.cta_begin[blockIdx.x] : (int)(n_items * blockIdx.x / gridDim.x);
    const int i_end = PAGED ? meta.cta_begin[blockIdx.x + 1] : (int)(n_items * (blockIdx.x + 1) / gridDim.x);
    const int nC = warp_len / kA3Chunk;
    const int seg = W * warp_len;
    const int wofs = warp * kA3Chunk;  // first chunk of the warp in a segment
    const int ctx32 = (int)ctx_len;
    constexpr int kStride = W * kA3Chunk;             // from one of its chunks to the next
    bool bad = false;  // warp-uniform: a wait gave up; compute is skipped from then on
    int inflight = 0;  // stages issued and not yet waited for

    // Producer cursor: the next chunk slot to look at.  Only slots that hold
    // rows of the sequence go through the ring: the consumer computes the
    // same row counts, so both sides skip the empty slots and take stages and
    // phases in the same order, and the producer stays S non-empty slots
    // ahead.  Position and cache row advance by additions.
    int p_item = i_begin, p_bh = i_begin / n_splits;
    int p_c = 0, p_split = i_begin % n_splits, p_st = 0;
    int p_pos = p_split * seg + wofs;
    // paged: the sequence, head and context length of p_bh, cached per pair
    int p_ctx = ctx32, p_cbh = -1, p_b = 0;
    int p_h = 0;
    auto next_item = [&]() {
        p_c = 0;
        ++p_item;
        if (++p_split == n_splits) {
            p_split = 0;
            ++p_bh;
        }
        p_pos = p_split * seg + wofs;
    };
    // seek() moves the cursor to the next slot that holds rows (or to the end
    // of the range), finds its row count and, paged, loads its page id.  It
    // runs before the consumer works on its current chunk and the page id is
    // first used in issue(), after that work, so the load's latency is hidden.
    int q_n = 0;  // rows of the slot found
    int q_page = 0;
    auto seek = [&]() {
        q_n = 0;
        while (p_item < i_end && !bad) {
            if constexpr (PAGED) {
                if (p_bh != p_cbh) {
                    p_cbh = p_bh;
                    p_b = p_bh / Hkv;
                    p_h = p_bh - p_b * Hkv;
                    const int len = __ldg(pa.lens + p_b);
                    p_ctx = len < 0 ? 0 : (len < ctx32 ? len : ctx32);
                }
            }
            const int rem = p_ctx - p_pos;
            if (rem <= 0) {  // the item's later slots of this warp lie further out
                next_item();
                continue;
            }
            q_n = rem >= kA3Chunk ? kA3Chunk : rem;
            if constexpr (PAGED) q_page = __ldg(pa.bt + (int64_t)p_b * pa.max_pages + (p_pos >> pa.page_shift));
            return;
        }
    };
    auto issue = [&]() {
        if (q_n == 0 || bad) return;
        const int n = q_n;
        int64_t row = (int64_t)p_bh * cache.cap + p_pos;
        bool ok = true;
        if constexpr (PAGED) {
            if (q_page < 0 || q_page >= pa.n_pages) {
                if (lane == 0) report_timeout(status, kA3StatusPage);
                ok = false;
            } else {
                row = (((int64_t)q_page * Hkv + p_h) << pa.page_shift) + (p_pos & ((1 << pa.page_shift) - 1));
            }
        }
        uint64_t* bar = bars + p_st;
        const uint32_t sb = ring + (uint32_t)(p_st * L::kStage);
        if (ok) {
            if (lane == 0) {
                fence_async_smem();  // earlier generic reads of this stage come first
                mbar_expect_tx(bar, (uint32_t)(n * (L::kKRow + (SP ? 0 : L::kVRow))));
                bulk_load(sb, cache.k_packed + row * L::kKRow, (uint32_t)(n * L::kKRow), bar);
                if constexpr (!SP)
                    bulk_load(sb + L::kVOff, cache.v_packed + row * L::kVRow, (uint32_t)(n * L::kVRow), bar);
            }
            // lanes past the end copy nothing (source size 0) from a valid row;
            // position l's norms go to slot 4 (l % 8) + l / 8, so that lane
            // (g, t) finds positions g, g + 8, g + 16, g + 24 in one 16-byte load
            const int64_t r = row + (lane < n ? lane : n - 1);
            const uint32_t sz = lane < n ? 4u : 0u;
            const uint32_t slot = 4u * (4u * (lane & 7) + (lane >> 3));
            cp_async4(sb + L::kKnOff + slot, cache.k_norm + r, sz);
            cp_async4(sb + L::kVnOff + slot, cache.v_norm + r, sz);
            if constexpr (QJL) cp_async4(sb + L::kGnOff + slot, meta.k_rnorm + r, sz);
            cp_async_arrive(bar);
        } else {
            mbar_arrive(bar);  // a bad page: nothing is copied, the chunk's result is undefined
        }
        if (++p_c == nC) {
            next_item();
        } else {
            p_pos += kStride;
        }
        if (++p_st == S) p_st = 0;
        ++inflight;
        q_n = 0;
    };
    for (int i = 0; i < S; ++i) {
        seek();
        issue();
    }

    float O[NG][8][4];
    float m_run[NG], l_run[NG], qx[NG];
    uint32_t qb[NG][8][2];
    // QJL: the projected query's B fragments and powers of two
    uint32_t qpb[QJL ? NG : 1][QJL ? 8 : 1][2];
    float qpx[QJL ? NG : 1];
    bool hok[NG];
    int vexp = 0;  // the V accumulators are in units of 2^vexp
    float vlim = 128.f, vsc = 1.f;
    int cur_bh = -1;
    int ctx_run = ctx32;  // context length of the current (batch, KV head) run
    const float thr = P.sparse_thr;
    const bool sparse = thr > 0.f;
    const int srcA = 8 * t + (g >> 1), srcB = srcA + 4;
    const bool odd = (g & 1) != 0;

    // SP: the kept chunk whose V product is still to come (its V buffer,
    // weights, V norms and valid rows); V buffers with a copy in flight; V
    // barrier phases
    bool pend = false;
    int pvi = 0;
    float pp[NG][2][2], pvn[2][2];
    bool pok[2][2];
    uint32_t pkeep = 0u;  // SP: sub-tiles of the pending chunk that some head keeps (bits u)
    // SP: the largest score of the lane's head seen anywhere in the grid so far
    // (log2 units; meta.gmax, one order-preserving key per (batch, query head)),
    // as this warp last read or raised it, and that head's slot
    float m_ref[NG];
    uint32_t* gslot[NG];
    const float lthr = SP ? __log2f(thr) : 0.f;
    uint32_t vfl = 0u, vph = 0u;
    int vcount = 0;  // rows whose V this warp read in the current (batch, KV head) run

    // Scores of one chunk of 32 positions at shared address sb (FULL: all 32
    // valid): the weights p relative to the running maximum, the V norms and
    // the valid rows; updates the running maximum and denominators.
    auto scores = [&](uint32_t sb, int n, auto full_tag, float (&p)[NG][2][2], float (&vn)[2][2],
                      bool (&ok)[2][2], uint32_t& ukeep) {
        constexpr bool FULL = decltype(full_tag)::value;
        const uint32_t sK = sb;
        uint32_t gseen[NG];  // SP: the grid's maximum, loaded now and used after the MMAs
        if constexpr (SP) {
#pragma unroll
            for (int hg = 0; hg < NG; ++hg) gseen[hg] = *reinterpret_cast<volatile uint32_t*>(gslot[hg]);
        }
        // ---- scores, one 16-position sub-tile at a time (fewer live registers)
        float sacc[2][NG][4];
        float ssg[QJL ? 2 : 1][QJL ? NG : 1][4];  // QJL: the sign part, its own accumulators
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            uint32_t kw[2][MB];
#pragma unroll
            for (int hg = 0; hg < NG; ++hg) sacc[u][hg][0] = sacc[u][hg][1] = sacc[u][hg][2] = sacc[u][hg][3] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                load_kfield<MB>(sK + (uint32_t)((16 * u + 8 * h + g) * L::kKRow + 4 * MB * t), kw[h]);
            if constexpr (L::kRest) {
                // S = (K_hi + K_lo) (Q_hi + Q_lo) with the keys' fp16 rests:
                // one MMA per 8 positions, whose A rows g and g + 8 are the
                // high parts and the rests of the same position, so that one
                // 8-byte table entry (high pair, rest pair) is two consecutive
                // A registers; the two row halves are summed afterwards
                float ra[2][NG][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int hg = 0; hg < NG; ++hg) ra[h][hg][0] = ra[h][hg][1] = ra[h][hg][2] = ra[h][hg][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint2 e0 = lds_tab2(pair_addr<MB>(kw[h], 2 * kk, kslot));
                        const uint2 e1 = lds_tab2(pair_addr<MB>(kw[h], 2 * kk + 1, kslot));
#pragma unroll
                        for (int hg = 0; hg < NG; ++hg)
                            mma16816(ra[h][hg], e0.x, e0.y, e1.x, e1.y, qb[hg][kk][0], qb[hg][kk][1]);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int hg = 0; hg < NG; ++hg) {
                        sacc[u][hg][2 * h] = ra[h][hg][0] + ra[h][hg][2];
                        sacc[u][hg][2 * h + 1] = ra[h][hg][1] + ra[h][hg][3];
                    }
            } else {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t a0 = lds_tab(pair_addr<MB>(kw[0], 2 * kk, kslot));
                    const uint32_t a2 = lds_tab(pair_addr<MB>(kw[0], 2 * kk + 1, kslot));
                    const uint32_t a1 = lds_tab(pair_addr<MB>(kw[1], 2 * kk, kslot));
                    const uint32_t a3 = lds_tab(pair_addr<MB>(kw[1], 2 * kk + 1, kslot));
#pragma unroll
                    for (int hg = 0; hg < NG; ++hg)
                        mma16816(sacc[u][hg], a0, a1, a2, a3, qb[hg][kk][0], qb[hg][kk][1]);
                }
            }
            if constexpr (QJL) {
                // <q', sgn>: A = +-1 from the sign bits (bit set: +1).  Lane t
                // reads sign word t of its rows (projections 32t .. 32t + 31).
                // For MMA kk its fp16 pairs are bits (kk, kk + 16) (a0, a1) and
                // (kk + 8, kk + 24) (a2, a3): one constant shift puts both bits
                // of a pair on the fp16 sign positions (bits 15 and 31).  The
                // projected query is stored in the same order (k_attn3_qjl_q).
                uint32_t sw[2];
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    sw[h] = lds_u32(sK + (uint32_t)((16 * u + 8 * h + g) * L::kKRow + L::kSignOff + 4 * t));
#pragma unroll
                for (int hg = 0; hg < NG; ++hg) ssg[u][hg][0] = ssg[u][hg][1] = ssg[u][hg][2] = ssg[u][hg][3] = 0.f;
                auto pm1 = [](uint32_t z) { return (z & 0x80008000u) ^ 0xBC00BC00u; };
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t a0 = pm1(sw[0] << (15 - kk)), a2 = pm1(sw[0] << (7 - kk));
                    const uint32_t a1 = pm1(sw[1] << (15 - kk)), a3 = pm1(sw[1] << (7 - kk));
#pragma unroll
                    for (int hg = 0; hg < NG; ++hg)
                        mma16816(ssg[u][hg], a0, a1, a2, a3, qpb[hg][kk][0], qpb[hg][kk][1]);
                }
            }
        }
        // lane (g, t): positions 16u + 8h + g of head 4hg + t; their norms are
        // the 4 consecutive slots 4g + 2u + h
        float sc[NG][2][2];
        float nvl = 0.f;
        const uint4 kn4 = lds_v4(sb + L::kKnOff + 16u * g), vn4 = lds_v4(sb + L::kVnOff + 16u * g);
        const uint32_t knw[4] = {kn4.x, kn4.y, kn4.z, kn4.w}, vnw[4] = {vn4.x, vn4.y, vn4.z, vn4.w};
        uint32_t gnw[4] = {0u, 0u, 0u, 0u};  // QJL: the keys' gammas, the same slots
        if constexpr (QJL) {
            const uint4 gn4 = lds_v4(sb + L::kGnOff + 16u * g);
            gnw[0] = gn4.x;
            gnw[1] = gn4.y;
            gnw[2] = gn4.z;
            gnw[3] = gn4.w;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = 16 * u + 8 * h + g;
                ok[u][h] = FULL || r < n;
                const float kn = __uint_as_float(knw[2 * u + h]);
                vn[u][h] = __uint_as_float(vnw[2 * u + h]);
                if (FULL) nvl = fmaxf(nvl, vn[u][h]);
                else if (ok[u][h]) nvl = fmaxf(nvl, vn[u][h]);
#pragma unroll
                for (int hg = 0; hg < NG; ++hg) {
                    float v = (sacc[u][hg][2 * h] + sacc[u][hg][2 * h + 1]) * (kn * qx[hg]);
                    if constexpr (QJL)
                        v = fmaf(ssg[u][hg][2 * h] + ssg[u][hg][2 * h + 1],
                                 __uint_as_float(gnw[2 * u + h]) * qpx[hg], v);
                    sc[hg][u][h] = ok[u][h] ? v : -INFINITY;
                }
            }
        bool need = false;
        float tmax[NG];
#pragma unroll
        for (int hg = 0; hg < NG; ++hg) {
            float mx = fmaxf(fmaxf(sc[hg][0][0], sc[hg][0][1]), fmaxf(sc[hg][1][0], sc[hg][1][1]));
            mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 16));
            tmax[hg] = mx;
            need = need || mx > m_run[hg] + kLazy;
        }
        if constexpr (SP) {
            // Gate against the largest score of the head seen anywhere in the
            // grid so far (at most the global maximum, so every row the
            // method keeps is kept): a sub-tile's V is needed when some valid
            // row of some head has sigma - m >= log2(threshold).  The warp
            // raises the grid's value only when it holds a new maximum.
            ukeep = 0u;
#pragma unroll
            for (int hg = 0; hg < NG; ++hg) {
                if (hok[hg]) {
                    m_ref[hg] = fmaxf(m_ref[hg], ord2f(gseen[hg]));
                    if (tmax[hg] > m_ref[hg]) {
                        m_ref[hg] = tmax[hg];
                        if (g == 0) atomicMax(gslot[hg], f2ord(tmax[hg]));
                    }
                    const float gate = m_ref[hg] + lthr;
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        if ((ok[u][0] && sc[hg][u][0] >= gate) || (ok[u][1] && sc[hg][u][1] >= gate)) ukeep |= 1u << u;
                }
            }
            ukeep = __reduce_or_sync(kAll, ukeep);
        }
        // rare: the running maximum moves, or a V norm would take p * n_v
        // (p <= 2^kLazy) past the fp16 range in units of 2^vexp
        if (__any_sync(kAll, need || nvl > vlim)) {
#pragma unroll
            for (int hg = 0; hg < NG; ++hg) {
                const float mn = fmaxf(m_run[hg], tmax[hg]);
                const float al = mn == -INFINITY ? 1.f : fast_exp2(m_run[hg] - mn);
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    O[hg][mt][0] *= al;
                    O[hg][mt][1] *= al;
                    O[hg][mt][2] *= al;
                    O[hg][mt][3] *= al;
                }
                l_run[hg] *= al;
                m_run[hg] = mn;
                if constexpr (SP) {  // the pending chunk's weights follow the new maximum
                    if (pend) {
                        pp[hg][0][0] *= al;
                        pp[hg][0][1] *= al;
                        pp[hg][1][0] *= al;
                        pp[hg][1][1] *= al;
                    }
                }
            }
            float w = nvl;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w = fmaxf(w, __shfl_xor_sync(kAll, w, o));
            if (w > vlim) {
                const int e2 = (int)((__float_as_uint(w) >> 23) & 0xFFu) - 126;  // w < 2^e2
                const int en = max(vexp, e2 - 7);
                const float f = ldexpf(1.f, vexp - en);
#pragma unroll
                for (int hg = 0; hg < NG; ++hg)
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        O[hg][mt][0] *= f;
                        O[hg][mt][1] *= f;
                        O[hg][mt][2] *= f;
                        O[hg][mt][3] *= f;
                    }
                vexp = en;
                vlim = ldexpf(1.f, en + 7);
                vsc = ldexpf(1.f, -en);
            }
        }
#pragma unroll
        for (int hg = 0; hg < NG; ++hg)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    p[hg][u][h] = fast_exp2(sc[hg][u][h] - m_run[hg]);
                    l_run[hg] += p[hg][u][h];
                }
    };

    // O^T += V^T P over the chunk whose V rows are at shared address sV, per sub-tile.
    auto pv = [&](uint32_t sV, const float (&p)[NG][2][2], const float (&vn)[2][2], const bool (&ok)[2][2],
                  uint32_t ukeep) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if constexpr (SP) {
                if (!(ukeep & (1u << u))) continue;
            } else if (sparse) {  // skip when every head is below the threshold
                bool keep = false;
#pragma unroll
                for (int hg = 0; hg < NG; ++hg)
                    keep = keep || (hok[hg] && fmaxf(p[hg][u][0], p[hg][u][1]) >= thr);
                if (!__any_sync(kAll, keep)) continue;
            }
            uint32_t pb0[NG], pb1[NG];
#pragma unroll
            for (int hg = 0; hg < NG; ++hg) {
                const float x0 = p[hg][u][0] * (vn[u][0] * vsc);
                const float x1 = p[hg][u][1] * (vn[u][1] * vsc);
                const float y0 = ok[u][0] ? x0 : 0.f, y1 = ok[u][1] ? x1 : 0.f;
                const __half2 hh = __floats2half2_rn(y0, y1);
                const float2 hf = __half22float2(hh);
                const __half2 hl = __floats2half2_rn(y0 - hf.x, y1 - hf.y);
                const uint32_t uH = *reinterpret_cast<const uint32_t*>(&hh);
                const uint32_t uL = *reinterpret_cast<const uint32_t*>(&hl);
                const uint32_t hA = __shfl_sync(kAll, uH, srcA);
                const uint32_t hB = __shfl_sync(kAll, uH, srcB);
                const uint32_t lA = __shfl_sync(kAll, uL, srcA);
                const uint32_t lB = __shfl_sync(kAll, uL, srcB);
                const uint32_t sA = odd ? lA : hA, sB = odd ? lB : hB;
                pb0[hg] = __byte_perm(sA, sB, 0x5410);  // positions 2t, 2t + 1
                pb1[hg] = __byte_perm(sA, sB, 0x7632);  // positions 2t + 8, 2t + 9
            }
            uint32_t fA[2], fB[2], fC[2], fD[2];
            const uint32_t r0 = sV + (uint32_t)((16 * u + 2 * t) * L::kVRow);
            load_vfield<VB>(r0, g, fA);
            load_vfield<VB>(r0 + L::kVRow, g, fB);
            load_vfield<VB>(r0 + 8 * L::kVRow, g, fC);
            load_vfield<VB>(r0 + 9 * L::kVRow, g, fD);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const uint32_t uA = lds_tab(pair_addr<VB>(fA, mt, vslot));
                const uint32_t uB = lds_tab(pair_addr<VB>(fB, mt, vslot));
                const uint32_t uC = lds_tab(pair_addr<VB>(fC, mt, vslot));
                const uint32_t uD = lds_tab(pair_addr<VB>(fD, mt, vslot));
                const uint32_t a0 = __byte_perm(uA, uB, 0x5410), a1 = __byte_perm(uA, uB, 0x7632);
                const uint32_t a2 = __byte_perm(uC, uD, 0x5410), a3 = __byte_perm(uC, uD, 0x7632);
#pragma unroll
                for (int hg = 0; hg < NG; ++hg) mma16816(O[hg][mt], a0, a1, a2, a3, pb0[hg], pb1[hg]);
            }
        }
    };

    // SP: take the pending chunk's V product once its V rows have landed in
    // its buffer.
    auto flush = [&]() {
        if constexpr (SP) {
            if (!pend) return;
            pend = false;
            if (!bad) {
                const bool okw = mbar_wait(vbars + pvi, (vph >> pvi) & 1u);
                if (!__all_sync(kAll, okw)) {
                    if (lane == 0) report_timeout(status, kA3StatusWait);
                    bad = true;  // the copy stays in vfl: waited for again before exit
                } else {
                    vph ^= 1u << pvi;
                    vfl &= ~(1u << pvi);
                    pv(vbuf + (uint32_t)(pvi * L::kVBuf), pp, pvn, pok, pkeep);
                }
            }
        }
    };

    // Merge the warps' running partials of the (batch, KV head) run_bh into
    // one partial per query head; its slot is this CTA's offset from the
    // first CTA whose items reach run_bh.
    auto publish = [&](int64_t run_bh) {
        if (P.v_rows && lane == 0 && vcount > 0) atomicAdd(P.v_rows + run_bh, vcount);
        vcount = 0;
        const float mul = ldexpf(P.out_mul, vexp);
        float lsum[NG];
#pragma unroll
        for (int hg = 0; hg < NG; ++hg) {
            float l = l_run[hg];
            l += __shfl_xor_sync(kAll, l, 4);
            l += __shfl_xor_sync(kAll, l, 8);
            l += __shfl_xor_sync(kAll, l, 16);
            lsum[hg] = l;
        }
        const int64_t b = run_bh / Hkv;
        const int gh = (int)(run_bh % Hkv);
        const int slot = PAGED ? meta.slot_base[blockIdx.x] - meta.slot_base[meta.c0[run_bh]]
                               : (int)blockIdx.x - attn3_cta_of(run_bh * n_splits, gridDim.x, n_items);
        // the merge buffer holds MH heads of every warp: heads h0 .. h0 + MH - 1 per pass
        constexpr int MH = L::kMergeHeads;
        for (int h0 = 0; h0 < G; h0 += MH) {
#pragma unroll
            for (int hg = 0; hg < NG; ++hg) {
                const int hh = 4 * hg + t;
                if (hok[hg] && hh >= h0 && hh < h0 + MH) {
                    float* row = merge + (warp * MH + (hh - h0)) * kA3MergeStride;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float4 v;
                        v.x = (O[hg][2 * i][0] + O[hg][2 * i][1]) * mul;
                        v.y = (O[hg][2 * i][2] + O[hg][2 * i][3]) * mul;
                        v.z = (O[hg][2 * i + 1][0] + O[hg][2 * i + 1][1]) * mul;
                        v.w = (O[hg][2 * i + 1][2] + O[hg][2 * i + 1][3]) * mul;
                        *reinterpret_cast<float4*>(row + 16 * g + 4 * i) = v;
                    }
                    if (g == 0) {
                        row[128] = m_run[hg];
                        row[129] = lsum[hg];
                    }
                }
            }
            __syncthreads();
            const int nh = G - h0 < MH ? G - h0 : MH;
            for (int i = threadIdx.x; i < nh * 128; i += T) {
                const int h = i >> 7, dim = i & 127;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < W; ++w) M = fmaxf(M, merge[(w * MH + h) * kA3MergeStride + 128]);
                float Ls = 0.f, A = 0.f;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float* row = merge + (w * MH + h) * kA3MergeStride;
                    const float f = row[128] == -INFINITY ? 0.f : fast_exp2(row[128] - M);
                    Ls = fmaf(f, row[129], Ls);
                    A = fmaf(f, row[dim], A);
                }
                float* o = part + ((b * Hq + gh * G + h0 + h) * n_splits + slot) * 130;
                o[dim] = A;
                if (dim == 0) {
                    o[128] = M;
                    o[129] = Ls;
                }
            }
            __syncthreads();
        }
    };

    // Items of one (batch, KV head) are consecutive: the warps accumulate
    // across them and publish when the pair changes and at the end.
    int split = i_begin % n_splits, cst = 0;
    uint32_t cph = 0;
    int bh = i_begin / n_splits;
    for (int item = i_begin; item <= i_end; ++item) {
        if (item == i_end || bh != cur_bh) {
            flush();
            if (cur_bh >= 0) publish(cur_bh);
            if (item == i_end) break;
            cur_bh = bh;
#pragma unroll
            for (int hg = 0; hg < NG; ++hg) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) O[hg][mt][0] = O[hg][mt][1] = O[hg][mt][2] = O[hg][mt][3] = 0.f;
                m_run[hg] = -INFINITY;
                l_run[hg] = 0.f;
            }
            vexp = 0;
            vlim = 128.f;
            vsc = 1.f;
            const int64_t b = bh / Hkv;
            const int gh = (int)(bh % Hkv);
            if constexpr (PAGED) {
                const int len = __ldg(pa.lens + b);
                ctx_run = len < 0 ? 0 : (len < ctx32 ? len : ctx32);
            }
#pragma unroll
            for (int hg = 0; hg < NG; ++hg) {
                const int hc = 4 * hg + (g >> 1);  // head of this lane's B column
                if (hc < G) {
                    const uint4* qp = reinterpret_cast<const uint4*>(
                        q16 + ((b * Hq + gh * G + hc) * 2 + (g & 1)) * 128 + 32 * t);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 u = __ldg(qp + i);
                        qb[hg][2 * i][0] = u.x;
                        qb[hg][2 * i][1] = u.y;
                        qb[hg][2 * i + 1][0] = u.z;
                        qb[hg][2 * i + 1][1] = u.w;
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) qb[hg][kk][0] = qb[hg][kk][1] = 0u;
                }
                if constexpr (QJL) {  // the same fragment layout over the projections
                    if (hc < G) {
                        const uint4* qpp = reinterpret_cast<const uint4*>(
                            meta.qp16 + ((b * Hq + gh * G + hc) * 2 + (g & 1)) * 128 + 32 * t);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4 u = __ldg(qpp + i);
                            qpb[hg][2 * i][0] = u.x;
                            qpb[hg][2 * i][1] = u.y;
                            qpb[hg][2 * i + 1][0] = u.z;
                            qpb[hg][2 * i + 1][1] = u.w;
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) qpb[hg][kk][0] = qpb[hg][kk][1] = 0u;
                    }
                }
                hok[hg] = 4 * hg + t < G;
                qx[hg] = hok[hg] ? __ldg(qexp + b * Hq + gh * G + 4 * hg + t) : 0.f;
                if constexpr (QJL) qpx[hg] = hok[hg] ? __ldg(meta.qpexp + b * Hq + gh * G + 4 * hg + t) : 0.f;
                if constexpr (SP) {
                    m_ref[hg] = -INFINITY;
                    gslot[hg] = meta.gmax + (b * Hq + gh * G + (hok[hg] ? 4 * hg + t : 0));
                }
            }
        }

        int pos = split * seg + wofs;
        for (int c = 0; c < nC; ++c, pos += kStride) {
            const int rem = ctx_run - pos;
            if (rem <= 0) break;  // this slot and the item's later ones hold no rows
            const int n = rem >= kA3Chunk ? kA3Chunk : rem;
            if constexpr (!SP) seek();  // paged: the page id loads while this chunk computes
            if (!bad) {
                const bool ok = mbar_wait(bars + cst, cph);
                if (!__all_sync(kAll, ok)) {
                    if (lane == 0) report_timeout(status, kA3StatusWait);
                    bad = true;  // cst and cph stay at the stage that gave up
                } else {
                    --inflight;
                }
            }
            bool release = true;  // SP refills the K stage itself, right after the scores
            if (!bad) {
                const uint32_t sb = ring + (uint32_t)(cst * L::kStage);
                float p[NG][2][2], vn[2][2];
                bool ok[2][2];
                uint32_t ukeep = 3u;
                if (n == kA3Chunk) scores(sb, n, std::true_type{}, p, vn, ok, ukeep);
                else scores(sb, n, std::false_type{}, p, vn, ok, ukeep);
                if constexpr (SP) {
                    const bool keep = ukeep != 0u;  // warp-uniform
                    const int vi = pend ? (pvi ^ 1) : 0;  // the buffer the pending chunk does not hold
                    if (keep && lane == 0) {
                        uint64_t* vb = vbars + vi;
                        fence_async_smem();  // earlier generic reads of the buffer come first
                        mbar_arrive_expect_tx(vb, (uint32_t)(n * L::kVRow));
                        bulk_load(vbuf + (uint32_t)(vi * L::kVBuf),
                                  cache.v_packed + ((int64_t)cur_bh * cache.cap + pos) * L::kVRow,
                                  (uint32_t)(n * L::kVRow), vb);
                    }
                    if (keep) vfl |= 1u << vi;
                    // the K stage is done with: the producer refills it now
                    __syncwarp();
                    seek();
                    issue();
                    release = false;
                    flush();  // the previous kept chunk's V product, while this chunk's V loads
                    if (keep) {
                        pend = true;
                        pvi = vi;
#pragma unroll
                        for (int hg = 0; hg < NG; ++hg)
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                pp[hg][u][0] = p[hg][u][0];
                                pp[hg][u][1] = p[hg][u][1];
                            }
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            pvn[u][0] = vn[u][0];
                            pvn[u][1] = vn[u][1];
                            pok[u][0] = ok[u][0];
                            pok[u][1] = ok[u][1];
                        }
                        pkeep = ukeep;
                        vcount += n;
                    }
                } else {
                    pv(sb + L::kVOff, p, vn, ok, 3u);
                    vcount += n;
                }
            }
            if (release) {
                __syncwarp();
                if constexpr (SP) seek();
                issue();
            }
            if (!bad && ++cst == S) {
                cst = 0;
                cph ^= 1u;
            }
        }
        if (++split == n_splits) {
            split = 0;
            ++bh;
        }
    }
    // A wait gave up: wait, again for a bounded time each, for the copies
    // this warp still has in flight before its shared memory is released.
    if (bad) {
        for (int k = 0; k < inflight; ++k) {
            mbar_wait(bars + cst, cph);
            if (++cst == S) {
                cst = 0;
                cph ^= 1u;
            }
        }
        if constexpr (SP) {
            for (int s = 0; s < 2; ++s)
                if (vfl & (1u << s)) mbar_wait(vbars + s, (vph >> s) & 1u);
        }
    }
}

// Merge the partials of one (batch, query head) (m in log2 units), normalise
// and rotate back: out = s . H (s2 . o) / sqrt(d).  One warp per (batch,
// query head), eight per block; lane l owns dims 2l, 2l + 1, 64 + 2l and
// 65 + 2l (8-byte loads: a partial row is 130 floats).  The butterflies
// over index bits 0 and 6 are in registers, those over bits 1-5 between
// lanes, in the order len = 1, 2, .., 64.
static __global__ void __launch_bounds__(128) k_attn3_combine(const float* __restrict__ part, int n_splits,
                                                              int grid, int64_t n_items, int Hq, int Hkv,
                                                              int64_t n_bh, float* __restrict__ out,
                                                              const __grid_constant__ AttnParams P,
                                                              bool paged, const A3Meta meta) {
    griddep_wait();    // the partials of the split kernel
    griddep_launch();  // a later kernel of the stream may set itself up; it waits for this grid
    __shared__ float red[3][132];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t bh = blockIdx.x;
    // partials of this (batch, query head): one per CTA whose items reach its KV head
    const int64_t bhk = (bh / Hq) * Hkv + (bh % Hq) / (Hq / Hkv);
    const int n_parts = paged ? meta.slot_base[meta.clast[bhk]] - meta.slot_base[meta.c0[bhk]] + 1
                              : attn3_cta_of((bhk + 1) * n_splits - 1, grid, n_items) -
                                    attn3_cta_of(bhk * n_splits, grid, n_items) + 1;
    const float* base = part + bh * n_splits * 130;
    float M = -INFINITY;
    for (int s = lane; s < n_parts; s += 32) M = fmaxf(M, __ldcg(base + s * 130 + 128));
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    // the four warps take every fourth partial
    float L = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 4
    for (int s = w; s < n_parts; s += 4) {  // unrolled: the loads of several partials in flight
        const float* row = base + s * 130;
        const float ms = __ldcg(row + 128);
        const float wt = ms == -INFINITY ? 0.f : fast_exp2(ms - M);
        L = fmaf(wt, __ldcg(row + 129), L);
        const float2 x = __ldcg(reinterpret_cast<const float2*>(row) + lane);
        const float2 y = __ldcg(reinterpret_cast<const float2*>(row + 64) + lane);
        a0 = fmaf(wt, x.x, a0);
        a1 = fmaf(wt, x.y, a1);
        a2 = fmaf(wt, y.x, a2);
        a3 = fmaf(wt, y.y, a3);
    }
    if (w > 0) {
        *reinterpret_cast<float4*>(&red[w - 1][4 * lane]) = make_float4(a0, a1, a2, a3);
        if (lane == 0) red[w - 1][128] = L;
    }
    __syncthreads();
    if (w > 0) return;
#pragma unroll
    for (int k = 0; k < 3; ++k) {  // fixed order
        const float4 r = *reinterpret_cast<const float4*>(&red[k][4 * lane]);
        a0 += r.x;
        a1 += r.y;
        a2 += r.z;
        a3 += r.w;
        L += red[k][128];
    }
    // an empty context (paged, length 0) gives zeros
    float v[4] = {L > 0.f ? a0 / L : 0.f, L > 0.f ? a1 / L : 0.f, L > 0.f ? a2 / L : 0.f, L > 0.f ? a3 / L : 0.f};
    const int dim[4] = {2 * lane, 2 * lane + 1, 64 + 2 * lane, 65 + 2 * lane};
    if (P.two_sided) {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __uint_as_float(__float_as_uint(v[k]) ^ sign_mask(P.sgn2b, dim[k]));
    }
    {  // index bit 0
        const float p0 = v[0] + v[1], p1 = v[0] - v[1], p2 = v[2] + v[3], p3 = v[2] - v[3];
        v[0] = p0;
        v[1] = p1;
        v[2] = p2;
        v[3] = p3;
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {  // index bits 1-5: lane bits 0-4
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v[k], m);
            v[k] = upper ? o - v[k] : v[k] + o;  // (lo + hi, lo - hi)
        }
    }
    {  // index bit 6
        const float p0 = v[0] + v[2], p2 = v[0] - v[2], p1 = v[1] + v[3], p3 = v[1] - v[3];
        v[0] = p0;
        v[1] = p1;
        v[2] = p2;
        v[3] = p3;
    }
    float* o = out + bh * 128;
    float2 r0, r1;
    r0.x = __uint_as_float(__float_as_uint(v[0] * P.inv_sqrt_d) ^ sign_mask(P.sgnb, dim[0]));
    r0.y = __uint_as_float(__float_as_uint(v[1] * P.inv_sqrt_d) ^ sign_mask(P.sgnb, dim[1]));
    r1.x = __uint_as_float(__float_as_uint(v[2] * P.inv_sqrt_d) ^ sign_mask(P.sgnb, dim[2]));
    r1.y = __uint_as_float(__float_as_uint(v[3] * P.inv_sqrt_d) ^ sign_mask(P.sgnb, dim[3]));
    reinterpret_cast<float2*>(o)[lane] = r0;
    reinterpret_cast<float2*>(o + 64)[lane] = r1;
}

template <int KB, int VB, int NG, bool PAGED, bool SP, bool QJL = false>
cudaError_t attn3_split_launch(const __half* q16, const float* qexp, int Hq, int Hkv,
                               const tq_cache_view& cache, int64_t ctx_len, const AttnGeometry& geo,
                               int64_t items, int grid, float* part, const AttnParams& P,
                               const PagedArgs& pa, const A3Meta& meta, cudaStream_t s) {
    using L = A3Layout<KB, VB, NG, SP, QJL>;
    auto fn = k_attn3_split<KB, VB, NG, PAGED, SP, QJL>;
    // The kernel addresses shared memory from window address 0, so it asks
    // for kEnd bytes (the dynamic block starts at or below kA3RingAt).
    static int attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kEnd);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = 1;
    }
    return launch_pdl(fn, dim3((unsigned)grid), dim3(A3Shape<KB, VB, NG, SP, QJL>::kThreads), L::kEnd, s, q16, qexp, Hq,
                      Hkv, cache, ctx_len, geo.warp_len, geo.n_splits, items, part, status_word(), P, pa, meta);
}

template <int KB, int VB, bool PAGED = false>
cudaError_t attn3_launch(const void* q, int B, int Hq, int Hkv, const tq_cache_view& cache,
                         int64_t ctx_len, float* out, void* ws, const AttnGeometry& geo,
                         const AttnParams& P, cudaStream_t s, const PagedArgs& pa_in = PagedArgs{},
                         const AttnAppend* app = nullptr) {
    __half* q16 = static_cast<__half*>(ws);
    float* qexp = reinterpret_cast<float*>(static_cast<char*>(ws) + (size_t)B * Hq * 512);
    float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + attn3_prefix_bytes(B, Hq));
    const int sms = num_sms();
    A3Meta meta{};
    meta.cta_begin = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(part) + attn3_partial_bytes(B, Hq, geo.n_splits));
    meta.slot_base = meta.cta_begin + (sms + 1);
    meta.c0 = meta.slot_base + (sms + 1);
    meta.clast = meta.c0 + (size_t)B * Hq;
    meta.gmax = reinterpret_cast<uint32_t*>(meta.clast + (size_t)B * Hq + B);
    PagedArgs pa = pa_in;
    cudaError_t e;
    if (PAGED && app) {
        int32_t* len1 = meta.clast + (size_t)B * Hq;  // attended lengths, written by the append launch
        auto qb = static_cast<const __nv_bfloat16*>(q);
        if (app->bf16)
            e = launch_pdl(k_attn3_q_append<__nv_bfloat16>, dim3(B * Hq), dim3(128), 0, s, qb, q16, qexp, P, Hq, Hkv,
                           static_cast<const __nv_bfloat16*>(app->k_new),
                           static_cast<const __nv_bfloat16*>(app->v_new), cache, pa, *app->PK, *app->PV, KB, VB,
                           len1, status_word());
        else
            e = launch_pdl(k_attn3_q_append<float>, dim3(B * Hq), dim3(128), 0, s, qb, q16, qexp, P, Hq, Hkv,
                           static_cast<const float*>(app->k_new), static_cast<const float*>(app->v_new), cache, pa,
                           *app->PK, *app->PV, KB, VB, len1, status_word());
        pa.lens = len1;
    } else {
        e = launch_pdl(k_attn3_q, dim3((unsigned)(((int64_t)B * Hq + 7) / 8)), dim3(256), 0, s,
                       static_cast<const __nv_bfloat16*>(q), q16, qexp, P, (int64_t)B * Hq,
                       (!PAGED && P.sparse_thr > 0.f) ? meta.gmax : (uint32_t*)nullptr);
    }
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)B * Hkv * geo.n_splits;
    int grid = (int)(items < sms ? items : sms);  // one CTA per SM
    if (PAGED) {
        if (grid > 1024) grid = 1024;  // the planning block gives one thread to each CTA
        const int n_pairs = B * Hkv;
        const size_t plan_smem = n_pairs <= kA3PlanSmemPairs ? sizeof(int64_t) * (size_t)n_pairs : 0;
        static int plan_attr[64] = {};
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || !plan_attr[dev]) {
            e = cudaFuncSetAttribute((const void*)k_attn3_plan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(sizeof(int64_t) * kA3PlanSmemPairs));
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) plan_attr[dev] = 1;
        }
        e = launch_pdl(k_attn3_plan, dim3(1), dim3(1024), plan_smem, s, (const int32_t*)pa.lens, Hkv, geo.n_splits,
                       (int64_t)geo.split_len, geo.warp_len, ctx_len, n_pairs, grid, meta, app != nullptr);
        if (e != cudaSuccess) return e;
    }
    // contiguous cache with a sparse-V threshold: the variant that copies V
    // only for the chunks some head keeps
    const bool sp = !PAGED && P.sparse_thr > 0.f;
    if (Hq / Hkv <= 4)
        e = sp ? attn3_split_launch<KB, VB, 1, false, true>(q16, qexp, Hq, Hkv, cache, ctx_len, geo, items, grid,
                                                            part, P, pa, meta, s)
               : attn3_split_launch<KB, VB, 1, PAGED, false>(q16, qexp, Hq, Hkv, cache, ctx_len, geo, items,
                                                             grid, part, P, pa, meta, s);
    else
        e = sp ? attn3_split_launch<KB, VB, 2, false, true>(q16, qexp, Hq, Hkv, cache, ctx_len, geo, items, grid,
                                                            part, P, pa, meta, s)
               : attn3_split_launch<KB, VB, 2, PAGED, false>(q16, qexp, Hq, Hkv, cache, ctx_len, geo, items,
                                                             grid, part, P, pa, meta, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_attn3_combine, dim3((unsigned)(B * Hq)), dim3(128), 0, s, (const float*)part, geo.n_splits,
                      grid, items, Hq, Hkv, (int64_t)B * Hq, out, P, PAGED, meta);
}

// QJL keys: the rotated and the projected queries of eight (batch, query
// head) rows per block of 256 threads.  Warp w rotates row 8 blockIdx.x + w
// as k_attn3_q does (q16, qexp) and keeps y = s2 . H (s . q) (unnormalised)
// in shared memory.  The projection is q' = proj_mul * S y with proj_mul =
// scale * log2(e) * sqrt(pi/2) / (d sqrt(d)), so that gamma <q', sgn> is the
// sign part of the score in log2 units.  S (row k = projection k) passes
// through shared memory in two halves of 64 columns with a row stride of 65
// floats, so that the 32 lanes reading one column of 32 rows hit distinct
// banks; thread (h4, k) forms projection k of rows 4 h4 .. 4 h4 + 3.  Each
// row is stored as fp16 high and low parts of q' / 2^e (|q' / 2^e| < 2^14) at
// qp16[bh][2][128] and 2^e at qpexp[bh].  Projection 32t + j sits at 32t +
// 4 (j mod 8) + m, m = 0, 2, 1, 3 for j in [0, 8), [8, 16), [16, 24), [24,
// 32): the order in which the split kernel's sign fragments pair the bits.
static __global__ void __launch_bounds__(256) k_attn3_qjl_q(const __nv_bfloat16* __restrict__ q,
                                                            const float* __restrict__ S, __half* __restrict__ q16,
                                                            float* __restrict__ qexp, __half* __restrict__ qp16,
                                                            float* __restrict__ qpexp,
                                                            const __grid_constant__ AttnParams P, float proj_mul,
                                                            int64_t n_rows) {
    __shared__ __align__(16) float ys[8][128];
    __shared__ float ss[128 * 65];
    __shared__ float wmax[8][4];
    griddep_wait();  // the queries and S, and readers of the workspace, of the previous kernel
    griddep_launch();
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int64_t row0 = (int64_t)blockIdx.x * 8;
    {
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        if (row0 + w < n_rows) attn3_q_warp(q, q16, qexp, P, row0 + w, lane, y);
        *reinterpret_cast<float4*>(&ys[w][4 * lane]) = make_float4(y[0], y[1], y[2], y[3]);
    }
    const int k = tid & 127, h4 = tid >> 7;
    float p[4] = {0.f, 0.f, 0.f, 0.f};
    for (int half = 0; half < 2; ++half) {
        __syncthreads();  // ys written; the previous half's reads of ss done
#pragma unroll
        for (int r = 0; r < 8; ++r) {  // 128 rows x 16 float4 of this half
            const int f = tid + 256 * r, sr = f >> 4, c4 = f & 15;
            const float4 v = __ldg(reinterpret_cast<const float4*>(S + sr * 128 + 64 * half) + c4);
            float* d = ss + sr * 65 + 4 * c4;
            d[0] = v.x;
            d[1] = v.y;
            d[2] = v.z;
            d[3] = v.w;
        }
        __syncthreads();
        const float* srow = ss + k * 65;
#pragma unroll 4
        for (int i = 0; i < 64; i += 4) {
            const float s0 = srow[i], s1 = srow[i + 1], s2 = srow[i + 2], s3 = srow[i + 3];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float4 y = *reinterpret_cast<const float4*>(&ys[4 * h4 + h][64 * half + i]);
                p[h] = fmaf(s0, y.x, p[h]);
                p[h] = fmaf(s1, y.y, p[h]);
                p[h] = fmaf(s2, y.z, p[h]);
                p[h] = fmaf(s3, y.w, p[h]);
            }
        }
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        p[h] *= proj_mul;
        float M = fabsf(p[h]);
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        if (lane == 0) wmax[w][h] = M;
    }
    __syncthreads();
    const int r = k & 31, slot = (int)((0x3120u >> (4 * (r >> 3))) & 0xFu);  // 0, 2, 1, 3
    const int at = (k & ~31) + 4 * (r & 7) + slot;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int64_t bh = row0 + 4 * h4 + h;
        if (bh >= n_rows) break;
        const float M = fmaxf(fmaxf(wmax[4 * h4][h], wmax[4 * h4 + 1][h]), fmaxf(wmax[4 * h4 + 2][h], wmax[4 * h4 + 3][h]));
        int e = 0;
        if (M > 0.f && M <= FLT_MAX) {
            int ex = 0;
            frexpf(M, &ex);  // M in [2^(ex-1), 2^ex)
            e = min(100, max(-100, ex - 14));
        }
        const float ps = ldexpf(p[h], -e);
        const __half hi = __float2half_rn(ps);
        const __half lo = __float2half_rn(ps - __half2float(hi));
        qp16[bh * 256 + at] = hi;
        qp16[bh * 256 + 128 + at] = lo;
        if (k == 0) qpexp[bh] = ldexpf(1.f, e);
    }
}

// QJL keys (KB bits in total, contiguous cache): the rotated and projected
// queries, the split kernel with the QJL scores, the combine.  The
// workspace is the d = 128 layout with the projected queries' prefix after
// the rotated queries'.
template <int KB, int VB>
cudaError_t attn3_qjl_launch(const void* q, const float* S, int B, int Hq, int Hkv, const tq_cache_view& cache,
                             const float* k_rnorm, int64_t ctx_len, float* out, void* ws, const AttnGeometry& geo,
                             const AttnParams& P, float proj_mul, cudaStream_t s) {
    __half* q16 = static_cast<__half*>(ws);
    float* qexp = reinterpret_cast<float*>(static_cast<char*>(ws) + (size_t)B * Hq * 512);
    char* pre2 = static_cast<char*>(ws) + attn3_prefix_bytes(B, Hq);
    __half* qp16 = reinterpret_cast<__half*>(pre2);
    float* qpexp = reinterpret_cast<float*>(pre2 + (size_t)B * Hq * 512);
    float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * attn3_prefix_bytes(B, Hq));
    const int sms = num_sms();
    A3Meta meta{};
    meta.cta_begin = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(part) + attn3_partial_bytes(B, Hq, geo.n_splits));
    meta.slot_base = meta.cta_begin + (sms + 1);
    meta.c0 = meta.slot_base + (sms + 1);
    meta.clast = meta.c0 + (size_t)B * Hq;
    meta.gmax = nullptr;
    meta.qp16 = qp16;
    meta.qpexp = qpexp;
    meta.k_rnorm = k_rnorm;
    const auto qb = static_cast<const __nv_bfloat16*>(q);
    cudaError_t e = launch_pdl(k_attn3_qjl_q, dim3((unsigned)(((int64_t)B * Hq + 7) / 8)), dim3(256), 0, s, qb, S, q16,
                               qexp, qp16, qpexp, P, proj_mul, (int64_t)B * Hq);
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)B * Hkv * geo.n_splits;
    const int grid = (int)(items < sms ? items : sms);  // one CTA per SM
    if (Hq / Hkv <= 4)
        e = attn3_split_launch<KB, VB, 1, false, false, true>(q16, qexp, Hq, Hkv, cache, ctx_len, geo, items, grid,
                                                              part, P, PagedArgs{}, meta, s);
    else
        e = attn3_split_launch<KB, VB, 2, false, false, true>(q16, qexp, Hq, Hkv, cache, ctx_len, geo, items, grid,
                                                              part, P, PagedArgs{}, meta, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_attn3_combine, dim3((unsigned)(B * Hq)), dim3(128), 0, s, (const float*)part, geo.n_splits,
                      grid, items, Hq, Hkv, (int64_t)B * Hq, out, P, false, meta);
}

}  // namespace dev

#if !defined(TQ_UNIT_D) || !defined(TQ_UNIT_KB) || TQ_UNIT_D != 128
#error "compile for d = 128, once per K width, with -DTQ_UNIT_D=128 -DTQ_UNIT_KB=<bits>"
#endif

template <int D, int KB>
cudaError_t launch_attn_dk(int v_bits, const void* q, int B, int Hq, int Hkv, const tq_cache_view& cache,
                           int64_t ctx_len, float* out, void* workspace, const AttnGeometry& g, const AttnParams& P,
                           cudaStream_t s) {
    static_assert(D == 128, "the tensor-core kernel is d = 128 only");
    switch (v_bits) {
        case 2: return dev::attn3_launch<KB, 2>(q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, P, s);
        case 3: return dev::attn3_launch<KB, 3>(q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, P, s);
        default: return dev::attn3_launch<KB, 4>(q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, P, s);
    }
}
template cudaError_t launch_attn_dk<128, TQ_UNIT_KB>(int, const void*, int, int, int, const tq_cache_view&, int64_t,
                                                     float*, void*, const AttnGeometry&, const AttnParams&,
                                                     cudaStream_t);

template <int KB>
cudaError_t launch_attn128_paged(int v_bits, const void* q, int B, int Hq, int Hkv,
                                 const tq_cache_view& pages, int64_t max_ctx, float* out,
                                 void* workspace, const AttnGeometry& g, const AttnParams& P,
                                 const PagedArgs& pa, cudaStream_t s, const AttnAppend* app) {
    switch (v_bits) {
        case 2: return dev::attn3_launch<KB, 2, true>(q, B, Hq, Hkv, pages, max_ctx, out, workspace, g, P, s, pa, app);
        case 3: return dev::attn3_launch<KB, 3, true>(q, B, Hq, Hkv, pages, max_ctx, out, workspace, g, P, s, pa, app);
        default: return dev::attn3_launch<KB, 4, true>(q, B, Hq, Hkv, pages, max_ctx, out, workspace, g, P, s, pa, app);
    }
}
#if TQ_UNIT_KB >= 3
// QJL keys of TQ_UNIT_KB bits in total (a TQ_UNIT_KB - 1 bit index).
template <int KB>
cudaError_t launch_attn3_qjl(int v_bits, const void* q, const float* S, int B, int Hq, int Hkv,
                             const tq_cache_view& cache, const float* k_rnorm, int64_t ctx_len, float* out,
                             void* workspace, const AttnGeometry& g, const AttnParams& P, float proj_mul,
                             cudaStream_t s) {
    switch (v_bits) {
        case 2: return dev::attn3_qjl_launch<KB, 2>(q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, P, proj_mul, s);
        case 3: return dev::attn3_qjl_launch<KB, 3>(q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, P, proj_mul, s);
        default: return dev::attn3_qjl_launch<KB, 4>(q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, P, proj_mul, s);
    }
}
template cudaError_t launch_attn3_qjl<TQ_UNIT_KB>(int, const void*, const float*, int, int, int, const tq_cache_view&,
                                                  const float*, int64_t, float*, void*, const AttnGeometry&,
                                                  const AttnParams&, float, cudaStream_t);
#endif
template cudaError_t launch_attn128_paged<TQ_UNIT_KB>(int, const void*, int, int, int, const tq_cache_view&,
                                                      int64_t, float*, void*, const AttnGeometry&,
                                                      const AttnParams&, const PagedArgs&, cudaStream_t,
                                                      const AttnAppend*);

}  // namespace tq
