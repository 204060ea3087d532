// tq_internal.h -- declarations shared by the host entry points (tq_api.cpp)
// and the kernel files.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/tq.h"

namespace tq {

constexpr int kMaxD = 256;

// Per-launch constants of the row codec, passed by value (they live in the
// kernel-parameter constant bank, so uniform reads cost no instruction).
struct RowParams {
    uint32_t sgn[kMaxD];  // 0x80000000 where s_i = -1, else 0 (xor mask on fp32 bits)
    float cen[16];        // fp32 centroids, ascending (2^bits used)
    float bnd[16];        // fp32 boundaries, ascending (2^bits - 1 used), rest +inf
    float inv_sqrt_d;
    // Two-sided signs (R = S2 H S1 / sqrt(d)): masks of the second diagonal,
    // applied after the forward transform and before the inverse one.
    int two_sided;
    uint32_t sgn2[kMaxD];
    uint32_t sgnb[kMaxD / 32];   // the signs one bit each (as AttnParams::sgnb)
    uint32_t sgn2b[kMaxD / 32];
    // the signs of elements 2j and 2j + 1 on the sign bits of a bf16 pair
    // (bits 15 and 31): one xor flips a packed output pair
    uint32_t sgnh[kMaxD / 2];
};

// Constants of the attention kernels.
struct AttnParams {
    uint32_t sgn[kMaxD];
    float kcen[16];
    float vcen[16];
    float inv_sqrt_d;
    float scale;       // softmax scale applied to q . k
    float sparse_thr;  // 0 = dense
    // d = 128 tensor-core kernels: the fp16 values nearest c * s_k and c * s_v
    // (s per width makes every one of them close: within 8.3e-5 relative at 4
    // bits, 2.2e-5 at 3), the query multiplier scale * log2(e) / (sqrt(d) *
    // s_k) and the output multiplier 1 / s_v; kcen_l is the rest of c * s_k,
    // c * s_k - kcen_h (fp16 holds it to 2^-11 of itself), for the prefill's
    // key low part.
    float kcen_h[16];
    float vcen_h[16];
    float kcen_l[16];
    float q_mul;
    float out_mul;
    int two_sided;  // as RowParams
    uint32_t sgn2[kMaxD];
    // The same signs one bit each (bit j of word j / 32 set: element j
    // negative).  A warp whose lanes take consecutive elements reads one or a
    // few words, where a per-element array read would take one parameter-bank
    // access per distinct lane address.
    uint32_t sgnb[kMaxD / 32];
    uint32_t sgn2b[kMaxD / 32];
    // [B][Hkv] rows whose V bytes the call read (zeroed before the launch),
    // or nullptr
    int32_t* v_rows;
};

// Host plan (the public tq_plan).
struct Plan {
    int d;
    uint64_t seed;
    uint32_t flags;  // TQ_PLAN_* of tq_plan_create_ex
    int8_t signs[kMaxD];
    int8_t signs2[kMaxD];  // all +1 unless TQ_PLAN_TWO_SIDED_SIGNS
    double c64[5][16], b64[5][16];  // index by bits (1..4)
    float c32[5][16], b32[5][16];
    // Per width: a scale s in [1, 2) that puts every c32 * s close to an fp16
    // value, and those fp16 values (the fp16 tensor-core attention).
    float hscale[5];
    float hcen[5][16];
};

void fill_attn_params(const Plan& P, int k_bits, int v_bits, float scale, float sparse_thr,
                      AttnParams& A);

// Argument checks of the contiguous decode attention, shared by
// tq_attn_decode and tq_attn_decode_noalloc: everything but the workspace,
// including that every buffer is one the device can dereference.  TQ_OK with
// *nothing = true when B == 0 (nothing to launch).
tq_status check_attn_decode_args(const tq_plan* plan, const void* q, int B, int Hq, int Hkv,
                                 const tq_cache_view& cache, int64_t ctx_len, int k_bits, int v_bits,
                                 float scale, float sparse_v_threshold, const float* out, bool* nothing);
// Launch of the contiguous decode attention on checked arguments, with the
// workspace `workspace` (geometry g) and the head-dimension dispatch of
// tq_attn_decode.
struct AttnGeometry;
// v_rows: the [B][Hkv] row counts of tq_attn_decode_ex, or nullptr.
cudaError_t launch_attn_decode(const Plan& P, const void* q, int B, int Hq, int Hkv, const tq_cache_view& cache,
                               int64_t ctx_len, int k_bits, int v_bits, float scale, float sparse_v_threshold,
                               float* out, int32_t* v_rows, void* workspace, const AttnGeometry& g,
                               cudaStream_t st);

// Bucketing lookup table geometry (encode): cell g covers the normalised
// coordinate w with rint(w * kLutScale) = g - kLutCenter, i.e. the closed
// interval [(g - kLutCenter - 0.5) / kLutScale, (g - kLutCenter + 0.5) / kLutScale].
constexpr int kLutScale = 256;
constexpr int kLutCenter = 512;
constexpr int kLutCells = 1024;  // covers w in [-2, 2); |w| <= 1 for finite rows
// The tensor-core encoders' tables (d = 128 and 256): cells of width 1/64 (a
// power of two, so y * inv * 64 is the exact product), k = rint(w * 64) in
// [-64, 64] for every finite row, indexed by one byte (k + 128).  Exact when
// no closed cell holds two boundaries: the codebooks' boundaries are at least
// 1.45 (d = 128) and 1.03 (d = 256) cells apart; plan creation checks it.
constexpr int kUmLutScale = 64;

// Launchers, one explicit instantiation per head dimension D (each kernel
// file is compiled once per D, in parallel).  They validate nothing: the
// caller (tq_api.cpp) has checked every argument.
template <int D>
cudaError_t launch_encode_d(int bits, tq_dtype dt, const void* x, int64_t n_rows, uint8_t* packed,
                            float* norms, const RowParams& P, cudaStream_t s);
template <int D>
cudaError_t launch_decode_d(int bits, tq_dtype dt, const uint8_t* packed, const float* norms,
                            int64_t n_rows, void* y, const RowParams& P, cudaStream_t s);
template <int D>
cudaError_t launch_append_d(int k_bits, int v_bits, tq_dtype dt, const void* k_new,
                            const void* v_new, int B, int Hkv, int64_t n_new,
                            const tq_cache_view& cache, int64_t pos, const RowParams& PK,
                            const RowParams& PV, cudaStream_t s);

// QJL residual keys (d = 32, 64, 128): the seeded Gaussian matrix S [d][d]
// (fp32, row-major), encode and decode with P the (bits - 1)-bit row
// parameters, and the decode attention over a contiguous cache whose keys are
// in that format (P from fill_attn_params with k_bits - 1).  The attention
// workspace is the prefix of rotated and projected queries (2 d floats per
// query head, rounded up to 64 floats) followed by the split partials of the
// generic geometry (attn_qjl_geometry).
cudaError_t launch_qjl_matrix(uint64_t seed, int d, float* S, cudaStream_t s);
template <int D>
cudaError_t launch_encode_qjl_d(int bits, tq_dtype dt, const void* x, int64_t n_rows, const float* S,
                                uint8_t* packed, float* norms, float* rnorms, const RowParams& P,
                                cudaStream_t s);
template <int D>
cudaError_t launch_decode_qjl_d(int bits, tq_dtype dt, const uint8_t* packed, const float* norms,
                                const float* rnorms, int64_t n_rows, const float* S, void* y, const RowParams& P,
                                cudaStream_t s);
struct AttnGeometry;
template <int KB>
cudaError_t launch_attn3_qjl(int v_bits, const void* q, const float* S, int B, int Hq, int Hkv,
                             const tq_cache_view& cache, const float* k_rnorm, int64_t ctx_len, float* out,
                             void* workspace, const AttnGeometry& g, const AttnParams& P, float proj_mul,
                             cudaStream_t s);
template <int D, int KB>
cudaError_t launch_attn_qjl(int v_bits, const void* q, const float* S, int B, int Hq, int Hkv,
                            const tq_cache_view& cache, const float* k_rnorm, int64_t ctx_len, float* out,
                            void* workspace, const AttnGeometry& g, const AttnParams& P, cudaStream_t s);
inline size_t attn_qjl_prefix_floats(int B, int Hq, int d) {
    return ((size_t)B * Hq * 2 * d + 63) / 64 * 64;
}

// Shared-memory plan of the d = 128 attention kernel, in absolute
// shared-window addresses (the dynamic block starts at or below
// kAttn3RingAt).  Each warp streams 32-position chunks (packed K and V rows
// plus two fp32 norms each) through its own ring of `stages` stages starting
// at kAttn3RingAt.  The centroid-pair table sits at kAttn3TableAt, 64 KiB
// aligned, so that a lookup address is one byte permute: row e (256 bytes)
// holds the pair of levels e, keys in bytes 0..127 and values in 128..255.
// A value entry is one fp16 pair per lane (32 columns of 4 bytes).  A key
// entry is one fp16 pair per lane, or, for widths that carry the rest of
// each centroid (attn3_key_rest), the pair of values nearest c * s_k and the
// pair of their rests, 8 bytes read by one 64-bit load: such a load is served
// a half-warp at a time, so lanes l and l + 16 share a column without a bank
// conflict (16 columns of 8 bytes).  The merge buffer holds `merge_heads`
// query heads of every warp at a time (merge passes = heads / merge_heads).
// Up to four query heads per KV head: 2 stages and as many warps (at most
// TQ_ATTN3_WARP_CAP) as fit; up to eight: 3 stages and at most 8 warps.
// The sparse-V variant (contiguous cache) copies a chunk's V rows only after
// its scores and takes their product one chunk later: its stages hold K rows
// and norms only, and each warp has two V buffers of one chunk after its
// stages, each with its own barrier.
constexpr int kAttn3RingAt = 2048;
constexpr int kAttn3TableAt = 131072;
constexpr int kAttn3SmemTop = 232448;    // 227 KiB, the most a block may use
constexpr int kAttn3MergeRow = 132 * 4;  // bytes per (warp, head) row of the merge buffer
// Tuning parameters: the most warps per CTA for up to four query heads per
// KV head, and the smallest key width whose centroids carry their fp16 rest.
#ifndef TQ_ATTN3_WARP_CAP
#define TQ_ATTN3_WARP_CAP 16
#endif
#ifndef TQ_ATTN3_REST_MIN_BITS
#define TQ_ATTN3_REST_MIN_BITS 3
#endif
// QJL keys (qjl): kb is the row's total width and a stage also holds each
// position's gamma (4 more bytes per position).
constexpr int attn3_stage_bytes(int kb, int vb, bool qjl = false) { return 32 * (16 * kb + 16 * vb + (qjl ? 12 : 8)); }
// Ring bytes of one warp: its stages, and with sparse V its two V buffers.
constexpr int attn3_warp_ring_bytes(int kb, int vb, int stages, bool sparse, bool qjl = false) {
    return sparse ? stages * 32 * (16 * kb + 8) + 2 * 32 * 16 * vb : stages * attn3_stage_bytes(kb, vb, qjl);
}
constexpr bool attn3_key_rest(int kb) { return kb >= TQ_ATTN3_REST_MIN_BITS; }

struct Attn3Plan {
    int warps, stages, merge_heads;
    int merge;  // merge buffer
    int bars;   // 8-byte mbarriers: one per (warp, stage), then two per warp for sparse V
    int end;    // bytes of dynamic shared memory to ask for
};

// The QJL-key kernel carries the projected query and a second set of score
// accumulators: at most 12 warps (170 registers per thread).
constexpr int kAttn3QjlWarpCap = 12;

constexpr Attn3Plan attn3_plan(int G, int kb, int vb, bool sparse = false, bool qjl = false) {
    const int heads = G <= 4 ? 4 : 8;
    const int stages = G <= 4 ? 2 : 3;
    const int high = kAttn3TableAt + 65536;  // first byte above the table
    for (int w = (G <= 4 ? (qjl ? kAttn3QjlWarpCap : TQ_ATTN3_WARP_CAP) : 8); w >= 1; --w) {
        const int ring_end = kAttn3RingAt + w * attn3_warp_ring_bytes(kb, vb, stages, sparse, qjl);
        if (ring_end > kAttn3TableAt) continue;
        const int bars_bytes = 8 * w * (stages + (sparse ? 2 : 0));
        for (int mh = heads; mh >= 1; mh /= 2) {
            const int mb = w * mh * kAttn3MergeRow;
            // merge and barriers above the table, else in the gap below it
            if (high + mb + bars_bytes <= kAttn3SmemTop) return Attn3Plan{w, stages, mh, high, high + mb, high + mb + bars_bytes};
            if (ring_end + mb + bars_bytes <= kAttn3TableAt) return Attn3Plan{w, stages, mh, ring_end, ring_end + mb, high};
        }
    }
    return Attn3Plan{0, 0, 0, 0, 0, 0};
}
constexpr int attn3_warps(int G, int kb, int vb, bool sparse = false, bool qjl = false) {
    return attn3_plan(G, kb, vb, sparse, qjl).warps;
}

struct AttnGeometry {
    int n_splits;
    int split_len;         // positions per split
    int parts;             // partials written per split
    int warp_len;          // d = 128: positions per warp and split
    bool q16;              // the workspace starts with the rotated fp16 queries
    bool cluster = false;  // other d: the splits of a (batch, KV head) form one cluster (<= 8)
};
// `sparse`: the call has a sparse-V threshold (the d = 128 kernel then runs
// its sparse variant, with its own warp count).
AttnGeometry attn_geometry(int B, int Hq, int Hkv, int64_t ctx_len, int num_sms, int d, int kb,
                           int vb, bool sparse = false);
// d = 128, paged cache with a length per sequence: shorter warp slices, so a
// sequence's last, partly filled split wastes little of a CTA's time.
AttnGeometry attn_geometry_paged(int B, int Hq, int Hkv, int64_t max_ctx, int num_sms, int kb, int vb);
size_t attn_paged_workspace_bound(int B, int Hq, int Hkv, int64_t max_ctx, int num_sms);
// Workspace that covers every K/V width pair and both the dense and the
// sparse-V kernel (the public size query takes neither).
size_t attn_workspace_bound(int B, int Hq, int Hkv, int64_t ctx_len, int num_sms, int d);
size_t attn_workspace_bytes(int B, int Hq, int d, const AttnGeometry& g);
// QJL keys: the generic (CUDA-core) split geometry at any d, and the bytes of
// its workspace (query prefix and partials).
AttnGeometry attn_qjl_geometry(int B, int Hq, int Hkv, int64_t ctx_len, int num_sms);
size_t attn_qjl_workspace_bytes(int B, int Hq, int d, const AttnGeometry& g);
// QJL keys of 3 and 4 bits at d = 128: the tensor-core kernel.  Its workspace
// is the d = 128 layout with a second query prefix (the projected query,
// fp16 high and low parts, and its powers of two) after the first.
AttnGeometry attn_qjl128_geometry(int B, int Hq, int Hkv, int64_t ctx_len, int num_sms, int kb, int vb);
size_t attn_qjl128_workspace_bytes(int B, int Hq, const AttnGeometry& g);
// d = 128: rotated queries (fp16 high and low parts, 512 bytes per head) and
// their power-of-two scales (4 bytes per head), rounded up to 256 bytes.
// d = 128, paged attention: the work partition written by the planning
// kernel after the partials: int32 CTA range starts [sms + 1], slot bases
// [sms + 1], first and last CTA per (batch, KV head) [B * Hq] each (Hq bounds
// Hkv), the attended lengths of the fused append [B]; then, for the sparse-V
// kernel, the largest score seen so far per (batch, query head) [B * Hq] as
// order-preserving uint32 keys; rounded up to 256 bytes.
inline size_t attn3_meta_bytes(int B, int Hq, int sms) {
    return ((size_t)4 * (2 * ((size_t)sms + 1) + 3 * (size_t)B * Hq + (size_t)B) + 255) / 256 * 256;
}
inline size_t attn3_partial_bytes(int B, int Hq, int n_splits) {
    return ((size_t)4 * B * Hq * n_splits * 130 + 255) / 256 * 256;
}
inline size_t attn3_prefix_bytes(int B, int Hq) {
    return ((size_t)B * Hq * (512 + 4) + 255) / 256 * 256;
}
template <int D, int KB>
cudaError_t launch_attn_dk(int v_bits, const void* q, int B, int Hq, int Hkv,
                           const tq_cache_view& cache, int64_t ctx_len, float* out, void* workspace,
                           const AttnGeometry& g, const AttnParams& P, cudaStream_t s);

// Paged-cache addressing: sequence b keeps position p at offset
// p & (2^page_shift - 1) of page bt[b * max_pages + (p >> page_shift)]; a page
// holds every KV head, [page][Hkv][page_size] rows.  `lens` holds the context
// length (attention) or the position written (append) of each sequence.
struct PagedArgs {
    const int32_t* bt;
    const int32_t* lens;
    int64_t n_pages;
    int max_pages;
    int page_shift;
};
// The decode step's append folded into the paged attention: one new K and V
// row per (sequence, KV head), [B][Hkv][128] fp32 or bf16, written at the
// position pa.lens[b] before the attention reads lengths pa.lens[b] + 1.
struct AttnAppend {
    const void* k_new;
    const void* v_new;
    bool bf16;
    const RowParams* PK;
    const RowParams* PV;
};
// d = 128 paged attention (tq_attn.cu, compiled in the d = 128 units); the
// tq_cache_view carries the page arrays (its cap is unused).  With `app`, the
// rows of app are appended first (same launches, the append rides on the
// query rotation).
template <int KB>
cudaError_t launch_attn128_paged(int v_bits, const void* q, int B, int Hq, int Hkv,
                                 const tq_cache_view& pages, int64_t max_ctx, float* out,
                                 void* workspace, const AttnGeometry& g, const AttnParams& P,
                                 const PagedArgs& pa, cudaStream_t s, const AttnAppend* app = nullptr);
// Paged attention for head dimensions other than 128 (tq_attn.cu, compiled
// in the d units other than 128): the generic kernel over the block table,
// lengths pa.lens[b] + len_plus.
template <int D, int KB>
cudaError_t launch_attn_generic_paged(int v_bits, const void* q, int B, int Hq, int Hkv,
                                      const tq_cache_view& pages, int64_t max_ctx, float* out, void* workspace,
                                      const AttnGeometry& g, const AttnParams& P, const PagedArgs& pa,
                                      int len_plus, cudaStream_t s);
// Prefill (multi-query, causal) attention, d = 128 (tq_prefill.cu, one unit
// per K width).  workspace: the query rotation as a 128 x 128 bf16 matrix
// (kPfRotBytes), one expanded tile image of kPfImgBytes per block of 128
// cache positions per (sequence, KV head), then each block's largest V norm
// (a float).
constexpr size_t kPfImgBytes = 99328;
constexpr size_t kPfRotBytes = 32768;
inline size_t attn_prefill_img_bytes(int B, int Hkv, int64_t cap) {
    return (size_t)B * Hkv * (size_t)((cap + 127) / 128) * kPfImgBytes;
}
inline size_t attn_prefill_ws_bytes(int B, int Hkv, int64_t cap) {
    return kPfRotBytes + attn_prefill_img_bytes(B, Hkv, cap) +
           ((size_t)B * Hkv * (size_t)((cap + 127) / 128) * 4 + 15) / 16 * 16;
}
template <int KB>
cudaError_t launch_attn_prefill(int v_bits, const void* q, int B, int T, int Hq, int Hkv, const int32_t* q_start,
                                const tq_cache_view& cache, float* out, void* workspace, const AttnParams& P,
                                cudaStream_t s);
// The attention kernel of the prefill (after the tile images are written).
cudaError_t launch_prefill_attention(const void* q, int B, int T, int Hq, int Hkv, const int32_t* q_start,
                                     const tq_cache_view& cache, float* out, void* workspace,
                                     const AttnParams& P, cudaStream_t s);
// Paged append of one token per sequence, d >= 32 (tq_codec.cu).
template <int D>
cudaError_t launch_append_paged_d(int k_bits, int v_bits, tq_dtype dt, const void* k_new,
                                  const void* v_new, int B, int Hkv, const tq_cache_view& pages,
                                  const PagedArgs& pa, const RowParams& PK, const RowParams& PV,
                                  cudaStream_t s);

// Shared launch helpers (tq_launch.cpp).
int num_sms();
int blocks_per_sm(const void* kernel, int block_threads, size_t dyn_smem);
unsigned grid_for(const void* kernel, int block_threads, int64_t items);

// Device address of the status word on the current device (kernels with
// bounded waits write it when they give up); nullptr if unavailable.
int* status_word();

// 2-D TMA descriptor over rows: n_rows x d elements of `esize` bytes, boxes of
// 128 bytes (inner) x box_rows rows, 128-byte swizzle, zero fill past the end.
cudaError_t make_rows_map(CUtensorMap* map, const void* base, int esize, uint64_t d,
                          uint64_t n_rows, uint32_t box_rows);

// Records the cudaError_t that tq_last_cuda_error reports for this thread.
void set_last_cuda_error(cudaError_t e);

// Device status word (bounded waits that gave up).
cudaError_t read_device_status(int reset, int* out);

}  // namespace tq
