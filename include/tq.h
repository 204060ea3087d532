/*
 * tq.h -- C ABI of the GB300 (sm_103a) TurboQuant KV-cache codec and the
 * decode attention that reads its packed output.
 *
 * The method (page titles and sections it follows):
 *  "TurboQuant KV Cache Compression -- Spec" (Foundry attention/spec.md):
 *     Step 1 Random Orthogonal Rotation, As-Built Notes 1-2 (signs before the
 *     Hadamard transform; L2-norm normalisation), Step 2 Lloyd-Max Scalar
 *     Quantization, Step 3 Packing, Codebook Generation, Hadamard Transform
 *     Detail, API (fa_tq_init / fa_tq_quantize / fa_tq_dequantize /
 *     fa_tq_attention_cached), Optimization: Fused dequant-dot.
 *  "TurboQuantEngine -- Specification" (larql): 2.2 Memory contract (fp32
 *     norm + ceil(head_dim*bits/8) bytes per head and row), 6 P1 follow-ups
 *     (incremental encode of the new row only).
 *  "CITATIONS" (Atlas): Sparse V dequant; Asymmetric K/V dtype.
 *
 * Row codec.  For a row x of length d (a power of two, 8 <= d <= 256):
 *   n = ||x||_2 (stored as fp32);  y = H (s . x) / sqrt(d)  with s the seeded
 *   +-1 diagonal and H the Sylvester Hadamard matrix;  u = y / n (u = 0 when
 *   n = 0);  idx_i = #{ j : u_i >= beta_j } over the 2^bits - 1 fp32
 *   boundaries of the Lloyd-Max codebook of one coordinate of a uniform unit
 *   vector in R^d;  the indices are packed as a dense LSB-first bit stream
 *   (index i in stream bits [i*bits, i*bits+bits); stream bit k is bit k%8 of
 *   byte k/8), d*bits/8 bytes per row.  Decode: x_hat = n * s . (H c_idx) /
 *   sqrt(d).  The sign diagonal: s_i = -1 iff the top bit of the i-th output
 *   of splitmix64 seeded with `seed` is set.
 *
 * Conventions for every call below:
 *  - Device buffers are owned by the caller.  The library allocates only host
 *    memory, and only in tq_plan_create.  No call allocates device memory.
 *  - Hot calls (tq_encode, tq_decode, tq_append, tq_attn_decode) validate
 *    their arguments on the host, return an error before launching anything
 *    if they are wrong, and otherwise enqueue their kernels on `stream`
 *    (asynchronous; a NULL stream is the legacy default stream).  A launch
 *    failure is reported as TQ_ERR_CUDA (see tq_last_cuda_error); faults
 *    during execution surface at the caller's next synchronisation.
 *  - Pointers to device memory must be 16-byte aligned (TQ_ERR_ALIGNMENT).
 *  - Kernels never trap; a kernel that gives up a bounded wait records it in
 *    a device status word read by tq_device_status.
 *  - Calls are thread-safe as long as plans are not destroyed while in use.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, without the CUDA headers. */
typedef struct CUstream_st *tq_stream_t;

typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, Hq % Hkv != 0 ... */
    TQ_ERR_UNSUPPORTED = 2, /* d or bits or dtype outside the supported set   */
    TQ_ERR_ALIGNMENT = 3,   /* a device pointer is not 16-byte aligned        */
    TQ_ERR_RANGE = 4,       /* pos / ctx_len outside the cache capacity       */
    TQ_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required     */
    TQ_ERR_CUDA = 6,        /* a CUDA runtime call failed                      */
    TQ_ERR_NOMEM = 7        /* host allocation failed                          */
} tq_status;

typedef enum { TQ_F32 = 0, TQ_BF16 = 1 } tq_dtype;

/* Opaque plan: d, seed, sign diagonal and the fp32 codebooks for bits 2..4
 * (the pages' fa_tq_state).  Host memory only. */
typedef struct tq_plan tq_plan;

/* One layer of a packed KV cache, caller-owned device memory:
 *   k_packed [B][Hkv][cap][d*k_bits/8]   k_norm [B][Hkv][cap]  (fp32)
 *   v_packed [B][Hkv][cap][d*v_bits/8]   v_norm [B][Hkv][cap]  (fp32)
 * (the pages' per-token compressed entry: packed indices per head plus the
 * stored norm, laid out per head and position as in their per-head
 * [n_kv_head, max_seq, head_dim] cache). */
typedef struct {
    uint8_t *k_packed;
    float *k_norm;
    uint8_t *v_packed;
    float *v_norm;
    int64_t cap;
} tq_cache_view;

/* Lloyd-Max codebook for one coordinate of a uniform unit vector in R^d
 * (density proportional to (1-x^2)^((d-3)/2) on [-1,1]), 2^bits levels:
 * "TurboQuant KV Cache Compression -- Spec", Step 2 and Codebook Generation
 * (Lloyd iteration -- centroids are conditional means of their cells,
 * boundaries are midpoints -- run to convergence).  Pure host function,
 * deterministic.  d >= 3, 1 <= bits <= 4.
 *   centroids:  2^bits doubles, ascending (caller-owned host memory)
 *   boundaries: 2^bits - 1 doubles, ascending, middle one exactly 0
 * Errors: TQ_ERR_INVALID_ARG (null), TQ_ERR_UNSUPPORTED (d or bits). */
tq_status tq_codebook_init(int d, int bits, double *centroids, double *boundaries);

/* The Lloyd-Max codebook of N(0, 1/d) (TQ_PLAN_GAUSSIAN_CODEBOOK), same
 * layout; d >= 1. */
tq_status tq_codebook_init_gaussian(int d, int bits, double *centroids, double *boundaries);

/* Build a plan for head dimension d (power of two, 8..256) and sign seed
 * (the pages' fa_tq_init(head_dim, config, seed)).  Computes the codebooks
 * for bits 2, 3, 4 and the sign diagonal.  *out receives a host object that
 * the caller releases with tq_plan_destroy.
 * Errors: TQ_ERR_INVALID_ARG (null out), TQ_ERR_UNSUPPORTED (d, or a codebook
 * with two boundaries closer than the encoders' bucketing cells: 1/256, and
 * 1/64 at d = 128 and 256 -- no codebook the library builds is), TQ_ERR_NOMEM. */
tq_status tq_plan_create(int d, uint64_t seed, tq_plan **out);

/* Format variants of the plan, for interoperability with caches written by
 * the turbo3/turbo4-style kernels ("CITATIONS", N(0, 1/d) codebook
 * replacement; Two-sided Rademacher signs in WHT):
 *   TQ_PLAN_GAUSSIAN_CODEBOOK: the Lloyd-Max codebook of N(0, 1/d), the
 *     large-d limit of the coordinate density, instead of the exact one.
 *   TQ_PLAN_TWO_SIDED_SIGNS: the rotation is S2 H S1 / sqrt(d), with s1 the
 *     first d outputs of the seed's sign stream and s2 the next d; decode and
 *     the attention's output rotation use S1 H S2 / sqrt(d).  Dot products are
 *     preserved, so attention over such a cache is unchanged in form.
 * tq_plan_create(d, seed, out) is tq_plan_create_ex(d, seed, 0, out).
 * Errors: TQ_ERR_UNSUPPORTED for unknown flag bits, as tq_plan_create else. */
enum { TQ_PLAN_GAUSSIAN_CODEBOOK = 1, TQ_PLAN_TWO_SIDED_SIGNS = 2 };
tq_status tq_plan_create_ex(int d, uint64_t seed, uint32_t flags, tq_plan **out);

/* The second sign vector s2 (d entries of -1/+1; all +1 without
 * TQ_PLAN_TWO_SIDED_SIGNS). */
tq_status tq_plan_signs2(const tq_plan *plan, int8_t *signs);
tq_status tq_plan_destroy(tq_plan *plan);

/* Inspection helpers (host memory): the d signs (+1/-1) of the plan, and the
 * fp32 codebook the kernels use for `bits` (2^bits centroids, 2^bits - 1
 * boundaries). */
tq_status tq_plan_signs(const tq_plan *plan, int8_t *signs);
tq_status tq_plan_codebook(const tq_plan *plan, int bits, float *centroids, float *boundaries);

/* Encode n_rows rows ("fa_tq_quantize" on a batch of rows).
 *   x:      [n_rows][d] fp32 or bf16 (x_dtype), device, 16-byte aligned
 *   packed: [n_rows][d*bits/8] bytes, device, 16-byte aligned
 *   norms:  [n_rows] fp32, device
 * bits in {2,3,4}.  n_rows = 0 is a no-op. */
tq_status tq_encode(const tq_plan *plan, int bits, const void *x, tq_dtype x_dtype,
                    int64_t n_rows, uint8_t *packed, float *norms, tq_stream_t stream);

/* Decode n_rows rows ("fa_tq_dequantize"): y = n * s . (H c_idx) / sqrt(d).
 *   packed: [n_rows][d*bits/8], norms: [n_rows] fp32 (device)
 *   y:      [n_rows][d] fp32 or bf16 (y_dtype, round to nearest even), device */
tq_status tq_decode(const tq_plan *plan, int bits, const uint8_t *packed, const float *norms,
                    int64_t n_rows, void *y, tq_dtype y_dtype, tq_stream_t stream);

/* Append n_new tokens of K and V into one layer of the cache at positions
 * [pos, pos + n_new): the incremental encode of only the new rows
 * ("TurboQuantEngine -- Specification", 6 P1 follow-ups, W3).  One launch
 * encodes the K rows with k_bits and the V rows with v_bits.
 *   k_new, v_new: [B][Hkv][n_new][d] fp32 or bf16 (dtype), device
 * Errors: TQ_ERR_RANGE if pos < 0 or pos + n_new > cache.cap. */
tq_status tq_append(const tq_plan *plan, int k_bits, int v_bits, const void *k_new,
                    const void *v_new, tq_dtype dtype, int B, int Hkv, int64_t n_new,
                    tq_cache_view cache, int64_t pos, tq_stream_t stream);

/* Workspace bytes tq_attn_decode needs for these sizes on the current device
 * (split-K partials).  0 for invalid sizes. */
size_t tq_attn_workspace_bytes(int B, int Hq, int Hkv, int d, int64_t ctx_len);

/* Workspace bytes tq_attn_decode_paged needs for these sizes on the current
 * device (split-K partials, and for d = 128 the work partition).  0 for
 * invalid sizes or d not in {32, 64, 128, 256}. */
size_t tq_attn_paged_workspace_bytes(int B, int Hq, int Hkv, int d, int64_t max_ctx);

/* Decode attention over the packed cache, one query token per sequence
 * ("TurboQuant KV Cache Compression -- Spec", fa_tq_attention_cached and
 * Optimization: Fused dequant-dot; "CITATIONS", Sparse V dequant and
 * Asymmetric K/V dtype).  For batch b and query head h (KV head
 * g = h / (Hq/Hkv)), over positions t in [0, ctx_len):
 *   sigma_t = scale * q . k_hat_t,  p = softmax(sigma),
 *   out = sum_t p_t v_hat_t
 * computed in the rotated domain: q is rotated once, scores are taken against
 * the centroids, V is accumulated rotated and the output is rotated back
 * once.  fp32 accumulation and softmax.
 *   q:   [B][Hq][d] bf16, device
 *   out: [B][Hq][d] fp32, device
 *   sparse_v_threshold: 0 = dense.  Otherwise a V row is skipped (treated as
 *     zero, still counted in the softmax denominator) when, for every head of
 *     the GQA group, exp(sigma_t - m) < threshold, with m the running maximum
 *     of that head at the time (m <= the global maximum, so the rows kept
 *     include every row with exp(sigma_t - max) >= threshold).
 *   workspace: device scratch of at least tq_attn_workspace_bytes(...) bytes;
 *     no initial contents needed.
 * Errors: TQ_ERR_RANGE if ctx_len < 1 or ctx_len > cache.cap;
 *   TQ_ERR_INVALID_ARG if Hq % Hkv != 0; TQ_ERR_WORKSPACE. */
tq_status tq_attn_decode(const tq_plan *plan, const void *q, int B, int Hq, int Hkv,
                         tq_cache_view cache, int64_t ctx_len, int k_bits, int v_bits,
                         float scale, float sparse_v_threshold, float *out, void *workspace,
                         size_t workspace_bytes, tq_stream_t stream);

/* tq_attn_decode, also reporting how many cached rows' V bytes each (batch,
 * KV head) read ("CITATIONS", Sparse V dequant: the gate saves the V loads
 * and the dequantisation of rows no query head needs).
 *   v_rows_read: [B][Hkv] int32, device, 4-byte aligned, or NULL; the call
 *     writes it (no initial contents needed).  A dense call reads every row,
 *     ctx_len per entry.  With sparse_v_threshold > 0 and d = 128 the kernel
 *     copies the V rows of a 32-position chunk only when, for some query head
 *     of the group, some row of the chunk has exp(sigma_t - m) >= threshold
 *     (m that head's running maximum at the time, so no row the method keeps
 *     is skipped); ctx_len - v_rows_read[b][g] rows of V were skipped.  Other
 *     head dimensions gate row by row.
 * tq_attn_decode is this call with v_rows_read = NULL; arguments, workspace
 * and errors are otherwise the same (TQ_ERR_ALIGNMENT for a misaligned
 * v_rows_read). */
tq_status tq_attn_decode_ex(const tq_plan *plan, const void *q, int B, int Hq, int Hkv,
                            tq_cache_view cache, int64_t ctx_len, int k_bits, int v_bits,
                            float scale, float sparse_v_threshold, float *out, int32_t *v_rows_read,
                            void *workspace, size_t workspace_bytes, tq_stream_t stream);

/* Decode attention that allocates nothing, for callers that are not allowed
 * to allocate device memory while they run -- a plugin inside a framework
 * that owns every device allocation through its own memory planner, or a
 * serving loop whose device memory is fixed up front so that no step can fail
 * or stall on an allocation.  Such callers cannot hand tq_attn_decode a
 * workspace.  This call computes exactly what tq_attn_decode computes, with
 * the same kernels and arguments minus the workspace.  The pages have no
 * counterpart of it.
 *   Scratch: a fixed device array of 8 MiB inside the library (every GPU
 *   that loads the library holds it until the process exits).  If the split-K
 *   partials for these sizes and bit widths need more than that, the call
 *   returns TQ_ERR_WORKSPACE and launches nothing.  tq_attn_workspace_bytes
 *   is an upper bound over all bit widths: a result <= 8388608 guarantees
 *   the sizes fit; a larger one may still fit for the widths of the call.
 *   No part of the scratch needs to start at zero: each call writes every
 *   partial before it reads it.
 *   Set-up: the first call on a device looks up the array's device address
 *   (with that device current) and caches it for the life of the process;
 *   make that first call before any stream capture on that device.  A
 *   cudaDeviceReset reloads the library's device code and leaves that cached
 *   address (and the one of the tq_device_status word) stale: make no call
 *   of this library on a device after resetting it.
 *   All calls on a device share the one array: calls whose kernels overlap on
 *   the GPU (different streams, or concurrent host threads) race and produce
 *   wrong results.  Serialise them, e.g. on one stream.
 *   Calls no cudaMalloc, cudaFree or other allocating routine.
 * Errors: as tq_attn_decode, with TQ_ERR_WORKSPACE meaning "needs more than
 * the 8 MiB array". */
tq_status tq_attn_decode_noalloc(const tq_plan *plan, const void *q, int B, int Hq, int Hkv,
                                 tq_cache_view cache, int64_t ctx_len, int k_bits, int v_bits,
                                 float scale, float sparse_v_threshold, float *out,
                                 tq_stream_t stream);

/* One layer of a paged KV cache ("CITATIONS" (Atlas), N(0, 1/d) codebook
 * replacement and Sparse V dequant: the paged write path and the
 * paged_decode_attn kernels; "TurboQuant KV Cache Compression -- Spec", API:
 * fa_tq_attention_cached).  Fixed-size pages of page_size positions, each page
 * holding every KV head, caller-owned device memory:
 *   k_packed [n_pages][Hkv][page_size][d*k_bits/8]   k_norm [n_pages][Hkv][page_size]
 *   v_packed [n_pages][Hkv][page_size][d*v_bits/8]   v_norm [n_pages][Hkv][page_size]
 * Sequence b keeps position p at offset p % page_size of page
 * block_table[b * max_pages + p / page_size] (int32 on the device).  page_size
 * is a power of two, at least 32. */
typedef struct {
    uint8_t *k_packed;
    float *k_norm;
    uint8_t *v_packed;
    float *v_norm;
    int64_t n_pages;
    int32_t page_size;
} tq_paged_cache;

/* Append one new token per sequence to a paged cache: the pages' write path
 * (quantize into the cache) with the row codec of tq_encode.
 *   k_new, v_new: [B][Hkv][d] (dtype), device
 *   block_table:  [B][max_pages] int32 page ids, device
 *   positions:    [B] int32, device: the position written for sequence b
 * The rows land at positions[b] of every KV head of sequence b.  Positions and
 * page ids are read on the device: a position outside [0, max_pages *
 * page_size) or a page id outside [0, n_pages) writes nothing for that
 * sequence and sets the device status word (tq_device_status) to 42.
 * d >= 32.  Errors: TQ_ERR_UNSUPPORTED (d < 32, page_size not a power of two
 * >= 32, bits, dtype), TQ_ERR_INVALID_ARG, TQ_ERR_ALIGNMENT. */
tq_status tq_append_paged(const tq_plan *plan, int k_bits, int v_bits, const void *k_new,
                          const void *v_new, tq_dtype dtype, int B, int Hkv, tq_paged_cache cache,
                          const int32_t *block_table, int max_pages, const int32_t *positions,
                          tq_stream_t stream);

/* Decode attention over a paged cache with a context length per sequence:
 * for sequence b and query head h, the tq_attn_decode result over positions
 * [0, min(ctx_lens[b], max_ctx)) of sequence b (an empty context gives a zero
 * output row).  d in {32, 64, 128, 256}: the tensor-core kernel at d = 128,
 * the CUDA-core one otherwise.
 *   q:   [B][Hq][d] bf16, device;  out: [B][Hq][d] fp32, device
 *   block_table: [B][max_pages] int32, device;  ctx_lens: [B] int32, device
 *   max_ctx: an upper bound of the lengths, <= max_pages * page_size; it sizes
 *     the split-K geometry: the workspace is
 *     tq_attn_paged_workspace_bytes(B, Hq, Hkv, 128, max_ctx) bytes.
 * A page id outside [0, n_pages) is not read; the device status word is set
 * to 33 and that chunk's result is undefined.
 * Errors: as tq_attn_decode; TQ_ERR_UNSUPPORTED also for d not in {32, 64,
 * 128, 256}, B > 65535, max_ctx > 2^30 or a page_size that is not a power of
 * two >= 32; TQ_ERR_RANGE if max_ctx < 1 or max_ctx > max_pages * page_size. */
tq_status tq_attn_decode_paged(const tq_plan *plan, const void *q, int B, int Hq, int Hkv,
                               tq_paged_cache cache, const int32_t *block_table, int max_pages,
                               const int32_t *ctx_lens, int64_t max_ctx, int k_bits, int v_bits,
                               float scale, float sparse_v_threshold, float *out, void *workspace,
                               size_t workspace_bytes, tq_stream_t stream);

/* One decode step on a paged cache: append each sequence's new token, then
 * attend over the sequence including it ("TurboQuant KV Cache Compression --
 * Spec", fa_tq_attention_cached: the new K and V are quantised into the cache
 * and the cached K and V are read for attention).  For sequence b the new
 * rows are written at position positions[b], exactly as tq_append_paged
 * writes them, and the output is the tq_attn_decode_paged result over
 * positions [0, min(positions[b] + 1, max_ctx)).  At d = 128 the append rides
 * on the attention's first launch (no launch is added); at d in {32, 64, 256}
 * the append is its own launch before the attention.
 *   q:      [B][Hq][d] bf16, device;  out: [B][Hq][d] fp32, device
 *   k_new, v_new: [B][Hkv][d] (kv_dtype), device
 *   block_table: [B][max_pages] int32, device;  positions: [B] int32, device
 *   max_ctx: an upper bound of positions[b] + 1, <= max_pages * page_size; the
 *     workspace is tq_attn_paged_workspace_bytes(B, Hq, Hkv, 128, max_ctx).
 * A position outside [0, max_pages * page_size) or a page id outside
 * [0, n_pages) writes nothing for that sequence and sets the device status
 * word to 42; its attention still runs over min(positions[b] + 1, max_ctx)
 * positions (none if positions[b] < 0).
 * Errors: as tq_attn_decode_paged; TQ_ERR_UNSUPPORTED also for kv_dtype. */
tq_status tq_attn_decode_append_paged(const tq_plan *plan, const void *q, const void *k_new,
                                      const void *v_new, tq_dtype kv_dtype, int B, int Hq, int Hkv,
                                      tq_paged_cache cache, const int32_t *block_table, int max_pages,
                                      const int32_t *positions, int64_t max_ctx, int k_bits, int v_bits,
                                      float scale, float sparse_v_threshold, float *out, void *workspace,
                                      size_t workspace_bytes, tq_stream_t stream);

/* Workspace bytes tq_attn_prefill needs for a cache of capacity `cap`: 32 KB
 * for the query rotation matrix, then the expanded K/V tiles, 99332 bytes per
 * 128 cache positions per sequence and KV head (about 6.5 times the packed
 * K4/V3 cache they expand); 0 for
 * invalid sizes, cap < T or d != 128.  B, T, Hq are checked only. */
size_t tq_attn_prefill_workspace_bytes(int B, int T, int Hq, int Hkv, int64_t cap, int d);

/* Prefill (chunked, multi-query) attention over the packed cache: a chunk of
 * T query tokens per sequence, token t of sequence b at absolute position
 * q_start[b] + t, attending causally over positions [0, q_start[b] + t] of
 * the contiguous cache (the chunk's own K/V rows already appended).  This is
 * the decode attention ("TurboQuant KV Cache Compression -- Spec",
 * fa_tq_attention_cached; Optimization: Fused dequant-dot -- scores against
 * the centroids in the rotated domain, V accumulated rotated, one inverse
 * rotation per output) with one query per token; both contractions run on
 * the tensor cores.  d = 128, Hq / Hkv in {1, 2, 4, 8}; dense (no sparse-V).
 *   q:   [B][T][Hq][d] bf16, device;  out: [B][T][Hq][d] fp32, device
 *   q_start: [B] int32, device; every q_start[b] + T must be <= cache.cap
 *     (checked on the device: a sequence that breaks it gets zero rows and
 *     the device status word 52).
 *   workspace: tq_attn_prefill_workspace_bytes(B, T, Hq, Hkv, cache.cap, 128)
 *     bytes; the prefix of every sequence is expanded there once into fp16
 *     centroid tiles, then read by every query tile of its KV head.
 * Errors: TQ_ERR_UNSUPPORTED (d, group size, bits; B * Hkv > 65535 or
 * T * Hq / Hkv > 65535 * 128), TQ_ERR_RANGE (cap < T),
 * TQ_ERR_INVALID_ARG, TQ_ERR_ALIGNMENT, TQ_ERR_WORKSPACE. */
tq_status tq_attn_prefill(const tq_plan *plan, const void *q, int B, int T, int Hq, int Hkv,
                          tq_cache_view cache, const int32_t *q_start, int k_bits, int v_bits,
                          float scale, float *out, void *workspace, size_t workspace_bytes,
                          tq_stream_t stream);

/* Text for a status code (static storage). */
/* ------------------------------------------------------ QJL residual keys
 * "CITATIONS" (Atlas), Google TurboQuant entry: an MSE-optimal quantiser
 * followed by a 1-bit quantised Johnson-Lindenstrauss transform of the
 * residual gives unbiased inner products ("TurboQuant KV Cache Compression --
 * Spec", Why not QJL?, which keeps MSE-only for softmax attention).  The
 * pages print no formula; the format here, for d in {32, 64, 128} and
 * b = bits in {2, 3, 4}:
 *   row bytes d*b/8: the d indices of the (b-1)-bit codec (same rotation,
 *   norm and bucketing, (b-1)-bit codebook of the plan), packed as tq_encode
 *   packs them, then d sign bits (stream bit k = 1 iff (S r)_k >= 0) where
 *   r = u - c[idx] is the residual of the rotated normalised row u;
 *   norms[i] = n = ||x_i||, rnorms[i] = gamma = n * ||r|| (fp32);
 *   decode: x_hat = s1 . H (s2 . (n c[idx] + sqrt(pi/2)/d * gamma * S^T sgn))
 *   / sqrt(d), sgn_k = +-1.  Over Gaussian S, E[<y, x_hat>] = <y, x>.
 * S is [d][d] fp32, row-major, caller-owned device memory (16-byte aligned),
 * filled by tq_qjl_matrix: S_ij = sqrt(-2 ln(1 - U1)) cos(2 pi U2) with
 * U = (out >> 11) / 2^53 on outputs 2d + 2k and 2d + 2k + 1 (k = i d + j) of
 * the plan seed's splitmix64 stream, in double, rounded to fp32.
 * Errors: TQ_ERR_UNSUPPORTED for other d, bits or dtypes; otherwise as
 * tq_encode / tq_decode / tq_attn_decode. */
tq_status tq_qjl_matrix(const tq_plan *plan, float *S, tq_stream_t stream);
/* x [n_rows][d] fp32 or bf16 -> packed [n_rows][d*bits/8], norms, rnorms [n_rows]. */
tq_status tq_encode_qjl(const tq_plan *plan, int bits, const float *S, const void *x, tq_dtype x_dtype,
                        int64_t n_rows, uint8_t *packed, float *norms, float *rnorms, tq_stream_t stream);
/* packed, norms, rnorms as tq_encode_qjl writes them -> y [n_rows][d]. */
tq_status tq_decode_qjl(const tq_plan *plan, int bits, const float *S, const uint8_t *packed,
                        const float *norms, const float *rnorms, int64_t n_rows, void *y, tq_dtype y_dtype,
                        tq_stream_t stream);
/* Decode attention (dense) over a contiguous cache whose K rows are in the
 * QJL format of k_bits (cache.k_packed [B][Hkv][cap][d*k_bits/8], cache.k_norm
 * the norms, k_rnorm [B][Hkv][cap] the gammas) and whose V rows are plain
 * tq_encode rows of v_bits: out = softmax(scale * q . K_hat) V_hat per query
 * head, with q [B][Hq][d] bf16 and out [B][Hq][d] fp32.  The scores are
 * n <R q, c[idx]> + sqrt(pi/2)/d * gamma <S R q, sgn>: S meets only the query.
 * workspace: at least tq_attn_qjl_workspace_bytes(B, Hq, Hkv, d, ctx_len). */
size_t tq_attn_qjl_workspace_bytes(int B, int Hq, int Hkv, int d, int64_t ctx_len);
tq_status tq_attn_decode_qjl(const tq_plan *plan, const float *S, const void *q, int B, int Hq, int Hkv,
                             tq_cache_view cache, const float *k_rnorm, int64_t ctx_len, int k_bits,
                             int v_bits, float scale, float *out, void *workspace, size_t workspace_bytes,
                             tq_stream_t stream);

const char *tq_status_string(tq_status status);

/* The cudaError_t value behind the most recent TQ_ERR_CUDA of this thread. */
int tq_last_cuda_error(void);

/* Device status word of the current device: 0 if no kernel of this library
 * has given up a bounded wait since the last reset (reset = 1 clears it).
 * Synchronises the device. */
tq_status tq_device_status(int reset, int *status_out);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
