/*
 * tq_oracle.h -- plain, slow, double-precision CPU oracle for the TurboQuant
 * KV-cache codec and the decode attention that reads its packed output.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library (kv_cache_vector_gb300/)
 * includes, links or calls this code; only tests/, the smoke check and the
 * CPU-baseline leg of bench.py do.  It shares no header, helper, table or
 * constant generator with the CUDA path.
 *
 * Sources (page title, section):
 *  [FS]  "TurboQuant KV Cache Compression -- Spec" (Foundry attention/spec.md):
 *        As-Built Notes 1-2; Step 1 Random Orthogonal Rotation; Step 2
 *        Lloyd-Max Scalar Quantization; Step 3 Packing; Codebook Generation;
 *        Hadamard Transform Detail; Optimization: Fused dequant-dot.
 *  [LS]  "TurboQuantEngine -- Specification" (larql turbo-quant-engine.md):
 *        2.1 Accuracy contract; 2.2 Memory contract (4-byte norm per row).
 *  [AC]  "CITATIONS" (Atlas feature/tq-plus-integration): N(0,1/d) codebook
 *        note; Sparse V dequant.
 *  [KS]  "Implementation specification: TurboAngle and TurboQuant-style KV
 *        compression" (kvcompress): Core implementation contract; Required
 *        invariants.
 *
 * Readings where the pages are silent or disagree (each is listed in the
 * design notes of the repository):
 *  - sign diagonal: s_i = -1 iff the top bit of the i-th splitmix64 output
 *    (seeded with `seed`) is set; the pages say "random +-1 signs from a seed"
 *    and name no generator.
 *  - D is applied before H ([FS] As-Built Note 1), y = H (s . x) / sqrt(d).
 *  - density of one rotated coordinate: (1-x^2)^((d-3)/2) on [-1,1], the exact
 *    marginal of a uniform unit vector (the pages' "Beta(d/2,d/2) on [0,1]" is
 *    this family after an affine change of variable, with a different shape
 *    parameter; the exact marginal is taken).
 *  - Lloyd iteration is run to convergence, not a fixed ~20 iterations.
 *  - codebook values are stored as fp32 ([FS] Step 2 struct: float arrays),
 *    and the bucket decision compares the fp32 coordinate with the fp32
 *    boundaries: idx = #{ j : u >= beta_j } (what a binary search into
 *    boundaries[] returns, ties going to the higher level).
 *  - a zero row has u = 0, norm 0, and decodes to exact zeros.
 *  - packing is a dense LSB-first bit stream, d*b/8 bytes per row
 *    ([LS] 2.2 ceil(head_dim*bits/8); [FS] memory table K3 = 48 B per head).
 *  - sparse-V: row t is dropped for head h iff exp(sigma_t - max_t sigma) <
 *    threshold; dropped rows still count in the softmax denominator and
 *    contribute a zero V row ([AC] Sparse V dequant).
 */
#ifndef TQ_ORACLE_H
#define TQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* splitmix64 (Vigna): advance *state and return the next output. */
uint64_t orc_splitmix64_next(uint64_t *state);

/* s[i] in {-1,+1} for i < d, from the splitmix64 stream seeded with seed. */
void orc_signs(uint64_t seed, int d, int8_t *s);

/* In-place unnormalised Walsh-Hadamard butterfly (Sylvester order), d = 2^k.
 * [FS] Hadamard Transform Detail. */
void orc_fwht(double *v, int d);

/* y = H (s . x) / sqrt(d)   ([FS] As-Built Note 1, Hadamard Transform Detail);
 * with s2 (not NULL) y = s2 . H (s . x) / sqrt(d) ([AC] Two-sided Rademacher
 * signs in WHT: signs1 before, signs2 after the butterfly). */
void orc_rotate(const int8_t *s, const int8_t *s2, int d, const double *x, double *y);
/* x = s . (H y) / sqrt(d)   (the inverse: H/sqrt(d) and D are self-inverse);
 * with s2: x = s . H (s2 . y) / sqrt(d). */
void orc_unrotate(const int8_t *s, const int8_t *s2, int d, const double *y, double *x);

/* Lloyd-Max codebook of N(0, 1/d) ([AC] N(0,1/d) codebook replacement): same
 * layout as orc_codebook; returns the iteration count, or -1. */
int orc_codebook_gauss(int d, int bits, double *centroids, double *boundaries);
/* E[(X - Q(X))^2] of a codebook for X ~ N(0, 1/d). */
double orc_codebook_gauss_mse(int d, int bits, const double *centroids, const double *boundaries);

/* Lloyd-Max codebook for one coordinate of a uniform unit vector in R^d,
 * 2^bits levels, bits in [1, 8], d >= 3.  Writes 2^bits centroids and
 * 2^bits - 1 boundaries, ascending, in double.  Returns the number of Lloyd
 * iterations, or -1 on bad arguments / no convergence.  [FS] Step 2,
 * Codebook Generation. */
int orc_codebook(int d, int bits, double *centroids, double *boundaries);

/* Per-coordinate mean squared error E[(X - Q(X))^2] of a codebook under the
 * coordinate density for dimension d (all cells, normalised density). */
double orc_codebook_mse(int d, int bits, const double *centroids,
                        const double *boundaries);

/* Probability mass of the coordinate density on [a, b] (-1 <= a <= b <= 1). */
double orc_density_mass(int d, double a, double b);

/* Level index of the fp32 coordinate u: #{ j : u >= boundaries[j] }. */
int orc_bucket(float u, int bits, const float *boundaries);

/* Dense LSB-first bit packing of d indices of `bits` bits: d*bits/8 bytes. */
void orc_pack(const uint8_t *idx, int d, int bits, uint8_t *out);
void orc_unpack(const uint8_t *in, int d, int bits, uint8_t *idx);

/* Encode n_rows rows of x (double; the caller converts fp32/bf16 exactly).
 *  packed: [n_rows][d*bits/8], norms: [n_rows] fp32 (round to nearest of the
 *  exact-in-double L2 norm).  u_out (optional, may be NULL): [n_rows][d], the
 *  normalised rotated coordinate in double before the fp32 decision. */
void orc_encode(const int8_t *s, const int8_t *s2, int d, int bits, const float *boundaries,
                const double *x, int64_t n_rows, uint8_t *packed, float *norms,
                double *u_out);

/* Decode: x_hat = norm * s . (H c_idx) / sqrt(d), in double (with s2:
 * norm * s . H (s2 . c_idx) / sqrt(d)).  s2 may be NULL in every call. */
void orc_decode(const int8_t *s, const int8_t *s2, int d, int bits, const float *centroids,
                const uint8_t *packed, const float *norms, int64_t n_rows,
                double *out);

/* Decode attention in the unrotated domain (plain definition).
 *  q:    [B][Hq][d] double
 *  k_packed [B][Hkv][cap][d*kb/8], k_norm [B][Hkv][cap]; same for v.
 *  Query head h reads KV head h / (Hq/Hkv).  Attends positions [0, ctx_len).
 *  sigma_t = scale * q . k_hat_t;  p = exp(sigma - max) / sum exp(sigma - max)
 *  o = sum_t p_t v_hat_t, where rows with exp(sigma_t - max) < sparse_thr
 *  contribute zero (sparse_thr = 0: dense).
 *  out: [B][Hq][d] double; kept (optional): [B][Hq] number of V rows used. */
void orc_attention(const int8_t *s, const int8_t *s2, int d, int B, int Hq, int Hkv, int64_t cap,
                   int64_t ctx_len, int k_bits, const float *k_centroids,
                   const uint8_t *k_packed, const float *k_norm, int v_bits,
                   const float *v_centroids, const uint8_t *v_packed,
                   const float *v_norm, const double *q, double scale,
                   double sparse_thr, double *out, int64_t *kept);

/* Prefill (multi-query) attention: token t of sequence b attends over
 * positions [0, q_start[b] + t] (causal), otherwise as orc_attention.
 *  q: [B][T][Hq][d] double; out: [B][T][Hq][d] double; the cache must hold
 *  q_start[b] + T rows of every sequence. */
void orc_attention_prefill(const int8_t *s, const int8_t *s2, int d, int B, int T, int Hq, int Hkv,
                           int64_t cap, const int32_t *q_start, int k_bits,
                           const float *k_centroids, const uint8_t *k_packed, const float *k_norm,
                           int v_bits, const float *v_centroids, const uint8_t *v_packed,
                           const float *v_norm, const double *q, double scale, double *out);

/* ------------------------------------------------------ QJL residual keys
 * "CITATIONS" (Atlas), Google TurboQuant entry: for inner products, an
 * MSE-optimal quantiser followed by a 1-bit quantised Johnson-Lindenstrauss
 * transform of the residual removes the bias ("TurboQuant KV Cache
 * Compression -- Spec", Why not QJL?; "Implementation specification ...",
 * TurboQuant path: residual / QJL-style correction).  The pages print no
 * formula; the reading taken here:
 *  - b bits per coordinate: the first b - 1 are the MSE codec's index, on the
 *    (b - 1)-bit codebook; then one sign bit per projection, d projections.
 *    Row layout: the d indices of b - 1 bits (dense LSB-first), then the d
 *    signs (bit k = 1 iff projection k >= 0), d*b/8 bytes.
 *  - the residual of the rotated normalised row, r = u - c[idx] (u as the
 *    encoder computes it, c the fp32 centroids), is projected by S (d x d,
 *    i.i.d. N(0,1)); gamma = n * ||r|| is stored beside the norm n.
 *  - decode (rotated domain): n c[idx] + sqrt(pi/2)/d * gamma * S^T sgn,
 *    sgn_k = +-1; E over S of the second term is n r (E[sign(s.r) s] =
 *    sqrt(2/pi) r/||r|| for a standard Gaussian s), so inner products with
 *    the decoded row are unbiased.
 *  - S_ij: Box-Muller, sqrt(-2 ln(1 - U1)) cos(2 pi U2), on the outputs
 *    o = 2d + 2k and 2d + 2k + 1 (k = i d + j) of the splitmix64 stream of
 *    `seed` (the stream whose first 2d outputs give s1 and s2), U = (out >>
 *    11) / 2^53. */
void orc_qjl_matrix(uint64_t seed, int d, double *S);

/* packed: [n_rows][d*bits/8] as above; norms, rnorms: [n_rows] fp32 (n and
 * gamma).  c_mse / b_mse: the (bits-1)-bit codebook (fp32).  proj_out
 * (optional): [n_rows][d] the projections S r in double. */
void orc_encode_qjl(const int8_t *s, const int8_t *s2, int d, int bits, const float *c_mse,
                    const float *b_mse, const double *S, const double *x, int64_t n_rows,
                    uint8_t *packed, float *norms, float *rnorms, double *proj_out);
/* x_hat = unrotate(n c[idx] + sqrt(pi/2)/d * gamma * S^T sgn), in double. */
void orc_decode_qjl(const int8_t *s, const int8_t *s2, int d, int bits, const float *c_mse,
                    const double *S, const uint8_t *packed, const float *norms, const float *rnorms,
                    int64_t n_rows, double *out);
/* orc_attention with keys in the QJL format (k_rnorm [B][Hkv][cap] holds
 * gamma) and values in the plain format; dense. */
void orc_attention_qjl(const int8_t *s, const int8_t *s2, int d, int B, int Hq, int Hkv, int64_t cap,
                       int64_t ctx_len, int k_bits, const float *k_c_mse, const double *S,
                       const uint8_t *k_packed, const float *k_norm, const float *k_rnorm, int v_bits,
                       const float *v_centroids, const uint8_t *v_packed, const float *v_norm,
                       const double *q, double scale, double *out);

#ifdef __cplusplus
}
#endif

#endif /* TQ_ORACLE_H */
