/*
 * tq_oracle.c -- plain, slow, double-precision CPU oracle.  TEST
 * INFRASTRUCTURE ONLY: see tq_oracle.h for the sources it follows, the
 * readings it takes where the pages are silent, and who may call it.
 *
 * Everything here is the definition written out: explicit loops, no blocking,
 * no fusion, no reordering beyond what the definitions state.
 */
#include "tq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

/* ------------------------------------------------------------------ signs */

/* splitmix64, as published by S. Vigna (public-domain reference generator):
 * add the golden-ratio increment, then two xor-shift-multiply mixing rounds
 * and a final xor-shift. */
uint64_t orc_splitmix64_next(uint64_t *state) {
    *state += 0x9E3779B97F4A7C15ULL;
    uint64_t z = *state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Seeded Rademacher diagonal D ([FS] Step 1: "a diagonal of random +1/-1
 * signs (one d-element array, generated from seed)"). */
void orc_signs(uint64_t seed, int d, int8_t *s) {
    uint64_t state = seed;
    for (int i = 0; i < d; ++i) {
        uint64_t r = orc_splitmix64_next(&state);
        s[i] = (r >> 63) ? (int8_t)-1 : (int8_t)1;
    }
}

/* ------------------------------------------------------------- rotation */

/* [FS] Hadamard Transform Detail: butterfly with len = 1, 2, 4, ..., d/2;
 * (u, v) -> (u + v, u - v).  Unnormalised. */
void orc_fwht(double *v, int d) {
    for (int len = 1; len < d; len *= 2) {
        for (int i = 0; i < d; i += 2 * len) {
            for (int j = i; j < i + len; ++j) {
                double a = v[j];
                double b = v[j + len];
                v[j] = a + b;
                v[j + len] = a - b;
            }
        }
    }
}

/* [FS] As-Built Note 1: the sign diagonal is applied before the FWHT,
 * rotate(x) = H (D x) / sqrt(d). */
void orc_rotate(const int8_t *s, const int8_t *s2, int d, const double *x, double *y) {
    for (int i = 0; i < d; ++i) y[i] = (double)s[i] * x[i];
    orc_fwht(y, d);
    double inv = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i) y[i] *= inv;
    /* "CITATIONS", Two-sided Rademacher signs in WHT: signs2 after the butterfly */
    if (s2)
        for (int i = 0; i < d; ++i) y[i] *= (double)s2[i];
}

/* [FS] Hadamard Transform Detail: "Inverse: same operation (FWHT is its own
 * inverse up to scaling, and D is its own inverse)", applied in reverse
 * order: x = D H y / sqrt(d). */
void orc_unrotate(const int8_t *s, const int8_t *s2, int d, const double *y, double *x) {
    for (int i = 0; i < d; ++i) x[i] = s2 ? (double)s2[i] * y[i] : y[i];
    orc_fwht(x, d);
    double inv = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i) x[i] = (double)s[i] * x[i] * inv;
}

/* ------------------------------------------------------------- codebook */

/* Gauss-Legendre nodes and weights on [-1, 1]: roots of P_n by Newton's
 * method on the three-term recurrence (n P_n = (2n-1) x P_{n-1} - (n-1)
 * P_{n-2}), weights 2 / ((1 - x^2) P_n'(x)^2). */
#define GL_N 20
static double gl_x[GL_N], gl_w[GL_N];
static int gl_ready = 0;

static void gl_init(void) {
    if (gl_ready) return;
    for (int i = 0; i < GL_N; ++i) {
        double x = cos(M_PI * (i + 0.75) / (GL_N + 0.5));
        double dp = 1.0;
        for (int it = 0; it < 100; ++it) {
            double p0 = 1.0, p1 = x;
            for (int k = 2; k <= GL_N; ++k) {
                double p2 = ((2.0 * k - 1.0) * x * p1 - (k - 1.0) * p0) / k;
                p0 = p1;
                p1 = p2;
            }
            dp = GL_N * (x * p1 - p0) / (x * x - 1.0);
            double dx = p1 / dp;
            x -= dx;
            if (fabs(dx) < 1e-16) break;
        }
        gl_x[i] = x;
        gl_w[i] = 2.0 / ((1.0 - x * x) * dp * dp);
    }
    gl_ready = 1;
}

/* Under x = sin(theta), the unnormalised density (1 - x^2)^((d-3)/2) dx
 * becomes cos(theta)^(d-2) dtheta, which is smooth on [-pi/2, pi/2] for every
 * d >= 3.  Integrate cos^(d-2) * sin^m over [ta, tb] (0 <= ta <= tb <= pi/2)
 * by composite Gauss-Legendre with panels no wider than 1/(4 sqrt(d)) rad. */
static double theta_moment(int d, int m, double ta, double tb) {
    if (tb <= ta) return 0.0;
    /* Beyond this angle cos^(d-2) is below 1e-40 of its peak: the tail adds
     * nothing visible in double precision. */
    double tcut = (d > 3) ? acos(exp(log(1e-40) / (double)(d - 2))) : M_PI / 2;
    if (ta >= tcut) return 0.0;
    if (tb > tcut) tb = tcut;
    double pw = 0.25 / sqrt((double)d);
    int np = (int)ceil((tb - ta) / pw);
    if (np < 1) np = 1;
    double h = (tb - ta) / np, sum = 0.0;
    for (int p = 0; p < np; ++p) {
        double a = ta + p * h, mid = a + 0.5 * h;
        for (int i = 0; i < GL_N; ++i) {
            double t = mid + 0.5 * h * gl_x[i];
            double f = pow(cos(t), (double)(d - 2));
            if (m == 1) f *= sin(t);
            if (m == 2) f *= sin(t) * sin(t);
            sum += 0.5 * h * gl_w[i] * f;
        }
    }
    return sum;
}

/* Mass of the unnormalised density on [xa, xb], 0 <= xa <= xb <= 1. */
static double half_mass(int d, double xa, double xb) {
    return theta_moment(d, 0, asin(xa), asin(xb));
}

/* First moment on [xa, xb] in closed form: the antiderivative of
 * x (1-x^2)^((d-3)/2) is -(1-x^2)^((d-1)/2) / (d-1). */
static double half_first_moment(int d, double xa, double xb) {
    double A = 0.5 * (double)(d - 1);
    return (pow(1.0 - xa * xa, A) - pow(1.0 - xb * xb, A)) / (double)(d - 1);
}

double orc_density_mass(int d, double a, double b) {
    gl_init();
    if (d < 3 || a > b) return 0.0;
    double z = 2.0 * half_mass(d, 0.0, 1.0);
    /* split at zero and fold the negative part by symmetry */
    double m = 0.0;
    if (a < 0.0) {
        double lo = -a, hi = (b < 0.0) ? -b : 0.0;
        m += half_mass(d, hi, lo);
    }
    if (b > 0.0) {
        double lo = (a > 0.0) ? a : 0.0;
        m += half_mass(d, lo, b);
    }
    return m / z;
}

/* [FS] Codebook Generation: Lloyd iteration -- centroids are conditional
 * expectations over the current cells, boundaries are midpoints of adjacent
 * centroids -- for the coordinate density (1-x^2)^((d-3)/2).  The density is
 * symmetric, so the positive half is iterated with a fixed boundary at 0 and
 * mirrored.  Run until the centroids stop moving (the density is log-concave
 * for d >= 3, so the fixed point is unique). */
int orc_codebook(int d, int bits, double *centroids, double *boundaries) {
    gl_init();
    if (d < 3 || bits < 1 || bits > 8 || !centroids || !boundaries) return -1;
    int L = 1 << bits, H = L / 2;
    double *beta = (double *)malloc(sizeof(double) * (H + 1));
    double *c = (double *)malloc(sizeof(double) * H);
    if (!beta || !c) { free(beta); free(c); return -1; }
    /* Start: uniform cells on [0, w] with w = min(1, 3/sqrt(d)), the last
     * cell reaching to 1 (uniform boundaries as in the pages' step 1, over
     * the range where the coordinate actually lives). */
    double w = 3.0 / sqrt((double)d);
    if (w > 1.0) w = 1.0;
    beta[0] = 0.0;
    for (int k = 1; k < H; ++k) beta[k] = w * k / H;
    beta[H] = 1.0;
    /* Stop when the largest centroid move is at machine level, or when it
     * has stopped shrinking (a rounding-level limit cycle) below 1e-12. */
    int it, converged = 0, since_best = 0;
    double best = INFINITY;
    for (it = 1; it <= 200000; ++it) {
        double delta = 0.0, cmax = 0.0;
        for (int k = 0; k < H; ++k) {
            double m0 = half_mass(d, beta[k], beta[k + 1]);
            double m1 = half_first_moment(d, beta[k], beta[k + 1]);
            double ck = m1 / m0;
            if (it > 1 && fabs(ck - c[k]) > delta) delta = fabs(ck - c[k]);
            c[k] = ck;
            if (fabs(ck) > cmax) cmax = fabs(ck);
        }
        for (int k = 1; k < H; ++k) beta[k] = 0.5 * (c[k - 1] + c[k]);
        if (it == 1) continue;
        if (delta <= 4e-15 * cmax) { converged = 1; break; }
        if (delta < 0.5 * best) { best = delta; since_best = 0; }
        else if (++since_best > 500 && best <= 1e-12 * cmax) { converged = 1; break; }
    }
    if (converged) {
        for (int k = 0; k < H; ++k) {
            centroids[H + k] = c[k];
            centroids[H - 1 - k] = -c[k];
        }
        boundaries[H - 1] = 0.0;
        for (int k = 1; k < H; ++k) {
            boundaries[H - 1 + k] = beta[k];
            boundaries[H - 1 - k] = -beta[k];
        }
    }
    free(beta);
    free(c);
    return converged ? it : -1;
}

/* ---------------------------------------------- Gaussian codebook
 * "CITATIONS", N(0, 1/d) codebook replacement: the Lloyd-Max codebook of a
 * Gaussian with variance 1/d (the per-coordinate variance after the
 * transform).  For X ~ N(0, sigma^2) and a cell (a, b) (a = -inf or b = +inf
 * allowed): P = (erfc(a/(sigma sqrt 2)) - erfc(b/(sigma sqrt 2))) / 2 and
 * E[X 1{a<X<b}] = sigma^2 (phi(a) - phi(b)), phi the N(0, sigma^2) density.
 * All 2^b cells are iterated (no use of symmetry), from levels evenly spread
 * over [-3 sigma, 3 sigma].  The iteration converges linearly and slowly, so
 * it runs until the step reaches rounding level: no centroid moves by more
 * than 1e-15 sigma, or the step has stayed below 1e-13 sigma without a new
 * minimum for 2000 iterations (the floor set by the libm's erfc and exp). */
static double gauss_pdf(double x, double sigma) {
    if (isinf(x)) return 0.0;
    double z = x / sigma;
    return exp(-0.5 * z * z) / (sigma * sqrt(2.0 * M_PI));
}
static double gauss_mass(double a, double b, double sigma) {
    double k = 1.0 / (sigma * sqrt(2.0));
    return 0.5 * (erfc(a * k) - erfc(b * k));
}

int orc_codebook_gauss(int d, int bits, double *centroids, double *boundaries) {
    int L = 1 << bits;
    double sigma = 1.0 / sqrt((double)d);
    double c[16];
    for (int i = 0; i < L; ++i) c[i] = sigma * (-3.0 + 6.0 * (i + 0.5) / L);
    double best = INFINITY;
    int stall = 0;
    for (int it = 1; it <= 2000000; ++it) {
        double moved = 0.0;
        double edge[17];
        edge[0] = -INFINITY;
        edge[L] = INFINITY;
        for (int i = 1; i < L; ++i) edge[i] = 0.5 * (c[i - 1] + c[i]);
        for (int i = 0; i < L; ++i) {
            double p = gauss_mass(edge[i], edge[i + 1], sigma);
            double m1 = sigma * sigma * (gauss_pdf(edge[i], sigma) - gauss_pdf(edge[i + 1], sigma));
            double ci = m1 / p;
            if (!isfinite(ci)) return -1;
            if (fabs(ci - c[i]) > moved) moved = fabs(ci - c[i]);
            c[i] = ci;
        }
        if (moved < best) {
            best = moved;
            stall = 0;
        } else {
            ++stall;
        }
        if (moved < 1e-15 * sigma || (best < 1e-13 * sigma && stall > 2000)) {
            /* The density is symmetric, so the exact quantiser is: remove the
             * rounding-level asymmetry, which puts the middle boundary at 0. */
            for (int i = 0; i < L / 2; ++i) {
                double a = 0.5 * (c[L - 1 - i] - c[i]);
                c[i] = -a;
                c[L - 1 - i] = a;
            }
            for (int i = 0; i < L; ++i) centroids[i] = c[i];
            for (int i = 1; i < L; ++i) boundaries[i - 1] = 0.5 * (c[i - 1] + c[i]);
            return it;
        }
    }
    return -1;
}

/* E[(X - Q(X))^2] for X ~ N(0, 1/d): per cell, the second moment about the
 * centroid, sigma^2 P + sigma^2 (a phi(a) - b phi(b)) - 2 c sigma^2 (phi(a) -
 * phi(b)) + c^2 P, with x phi(x) = 0 at infinity. */
double orc_codebook_gauss_mse(int d, int bits, const double *centroids, const double *boundaries) {
    int L = 1 << bits;
    double sigma = 1.0 / sqrt((double)d), s2 = sigma * sigma, mse = 0.0;
    for (int i = 0; i < L; ++i) {
        double a = (i == 0) ? -INFINITY : boundaries[i - 1];
        double b = (i == L - 1) ? INFINITY : boundaries[i];
        double p = gauss_mass(a, b, sigma);
        double pa = gauss_pdf(a, sigma), pb = gauss_pdf(b, sigma);
        double apa = isinf(a) ? 0.0 : a * pa, bpb = isinf(b) ? 0.0 : b * pb;
        double m1 = s2 * (pa - pb), m2 = s2 * p + s2 * (apa - bpb);
        mse += m2 - 2.0 * centroids[i] * m1 + centroids[i] * centroids[i] * p;
    }
    return mse;
}

double orc_codebook_mse(int d, int bits, const double *centroids,
                        const double *boundaries) {
    gl_init();
    int L = 1 << bits, H = L / 2;
    double z = half_mass(d, 0.0, 1.0);
    double mse = 0.0;
    /* positive half: cells [b_{H-1+k}, b_{H+k}] with centroid c_{H+k};
     * the negative half contributes the same by symmetry. */
    for (int k = 0; k < H; ++k) {
        double xa = boundaries[H - 1 + k];
        double xb = (k == H - 1) ? 1.0 : boundaries[H + k];
        double ck = centroids[H + k];
        double ta = asin(xa), tb = asin(xb);
        double m0 = theta_moment(d, 0, ta, tb);
        double m1 = theta_moment(d, 1, ta, tb);
        double m2 = theta_moment(d, 2, ta, tb);
        mse += m2 - 2.0 * ck * m1 + ck * ck * m0;
    }
    return mse / z;
}

/* ---------------------------------------------------------- quantiser */

/* [FS] Step 2: "binary search into boundaries[] to get the level index":
 * the index is the number of boundaries at or below u. */
int orc_bucket(float u, int bits, const float *boundaries) {
    int L = 1 << bits, idx = 0;
    for (int j = 0; j < L - 1; ++j)
        if (u >= boundaries[j]) idx += 1;
    return idx;
}

/* Stream bit k is bit (k mod 8) of byte k/8; index i occupies stream bits
 * [i*bits, i*bits + bits), least significant bit first. */
void orc_pack(const uint8_t *idx, int d, int bits, uint8_t *out) {
    int nbytes = d * bits / 8;
    memset(out, 0, (size_t)nbytes);
    for (int i = 0; i < d; ++i) {
        for (int k = 0; k < bits; ++k) {
            int bit = (idx[i] >> k) & 1;
            int pos = i * bits + k;
            out[pos / 8] |= (uint8_t)(bit << (pos % 8));
        }
    }
}

void orc_unpack(const uint8_t *in, int d, int bits, uint8_t *idx) {
    for (int i = 0; i < d; ++i) {
        int v = 0;
        for (int k = 0; k < bits; ++k) {
            int pos = i * bits + k;
            v |= ((in[pos / 8] >> (pos % 8)) & 1) << k;
        }
        idx[i] = (uint8_t)v;
    }
}

/* --------------------------------------------------------- encode/decode */

void orc_encode(const int8_t *s, const int8_t *s2, int d, int bits, const float *boundaries,
                const double *x, int64_t n_rows, uint8_t *packed, float *norms,
                double *u_out) {
    int rb = d * bits / 8;
    double *y = (double *)malloc(sizeof(double) * d);
    uint8_t *idx = (uint8_t *)malloc((size_t)d);
    for (int64_t r = 0; r < n_rows; ++r) {
        const double *xr = x + r * d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += xr[i] * xr[i];
        double n = sqrt(ss);                     /* [FS] As-Built Note 2 */
        orc_rotate(s, s2, d, xr, y);
        norms[r] = (float)n;                     /* stored fp32 ([LS] 2.2) */
        for (int i = 0; i < d; ++i) {
            double u = (n > 0.0) ? y[i] / n : 0.0;
            if (u_out) u_out[r * d + i] = u;
            idx[i] = (uint8_t)orc_bucket((float)u, bits, boundaries);
        }
        orc_pack(idx, d, bits, packed + r * rb);
    }
    free(y);
    free(idx);
}

void orc_decode(const int8_t *s, const int8_t *s2, int d, int bits, const float *centroids,
                const uint8_t *packed, const float *norms, int64_t n_rows,
                double *out) {
    int rb = d * bits / 8;
    double *c = (double *)malloc(sizeof(double) * d);
    uint8_t *idx = (uint8_t *)malloc((size_t)d);
    for (int64_t r = 0; r < n_rows; ++r) {
        orc_unpack(packed + r * rb, d, bits, idx);
        for (int i = 0; i < d; ++i) c[i] = (double)centroids[idx[i]];
        double *o = out + r * d;
        orc_unrotate(s, s2, d, c, o);
        for (int i = 0; i < d; ++i) o[i] *= (double)norms[r];
    }
    free(c);
    free(idx);
}

/* ------------------------------------------------------------ attention */

void orc_attention(const int8_t *s, const int8_t *s2, int d, int B, int Hq, int Hkv, int64_t cap,
                   int64_t ctx_len, int k_bits, const float *k_centroids,
                   const uint8_t *k_packed, const float *k_norm, int v_bits,
                   const float *v_centroids, const uint8_t *v_packed,
                   const float *v_norm, const double *q, double scale,
                   double sparse_thr, double *out, int64_t *kept) {
    int G = Hq / Hkv;
    int rbk = d * k_bits / 8, rbv = d * v_bits / 8;
    double *kh = (double *)malloc(sizeof(double) * (size_t)(ctx_len * d + 1));
    double *vh = (double *)malloc(sizeof(double) * (size_t)(ctx_len * d + 1));
    double *sig = (double *)malloc(sizeof(double) * (size_t)(ctx_len + 1));
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < Hkv; ++g) {
            int64_t row0 = ((int64_t)b * Hkv + g) * cap;
            orc_decode(s, s2, d, k_bits, k_centroids, k_packed + row0 * rbk,
                       k_norm + row0, ctx_len, kh);
            orc_decode(s, s2, d, v_bits, v_centroids, v_packed + row0 * rbv,
                       v_norm + row0, ctx_len, vh);
            for (int hh = 0; hh < G; ++hh) {
                int h = g * G + hh;
                const double *qh = q + ((int64_t)b * Hq + h) * d;
                double *o = out + ((int64_t)b * Hq + h) * d;
                double m = -INFINITY;
                for (int64_t t = 0; t < ctx_len; ++t) {
                    double dot = 0.0;
                    for (int j = 0; j < d; ++j) dot += qh[j] * kh[t * d + j];
                    sig[t] = scale * dot;
                    if (sig[t] > m) m = sig[t];
                }
                double l = 0.0;
                for (int64_t t = 0; t < ctx_len; ++t) l += exp(sig[t] - m);
                for (int j = 0; j < d; ++j) o[j] = 0.0;
                int64_t used = 0;
                for (int64_t t = 0; t < ctx_len; ++t) {
                    double e = exp(sig[t] - m);
                    if (e < sparse_thr) continue;   /* [AC] Sparse V dequant */
                    used += 1;
                    for (int j = 0; j < d; ++j) o[j] += (e / l) * vh[t * d + j];
                }
                if (kept) kept[(int64_t)b * Hq + h] = used;
            }
        }
    }
    free(kh);
    free(vh);
    free(sig);
}

/* Prefill (multi-query) attention over the packed cache, plain definition:
 * token t of sequence b (absolute position q_start[b] + t) attends, for query
 * head h, over positions [0, q_start[b] + t] of KV head h / (Hq/Hkv) -- the
 * decode attention above with one query per token and a causal length.
 *  q:   [B][T][Hq][d] double;  out: [B][T][Hq][d] double. */
void orc_attention_prefill(const int8_t *s, const int8_t *s2, int d, int B, int T, int Hq, int Hkv,
                           int64_t cap, const int32_t *q_start, int k_bits,
                           const float *k_centroids, const uint8_t *k_packed, const float *k_norm,
                           int v_bits, const float *v_centroids, const uint8_t *v_packed,
                           const float *v_norm, const double *q, double scale, double *out) {
    int G = Hq / Hkv;
    int rbk = d * k_bits / 8, rbv = d * v_bits / 8;
    for (int b = 0; b < B; ++b) {
        int64_t n = (int64_t)q_start[b] + T; /* rows the chunk can reach */
        double *kh = (double *)malloc(sizeof(double) * (size_t)(n * d + 1));
        double *vh = (double *)malloc(sizeof(double) * (size_t)(n * d + 1));
        double *sig = (double *)malloc(sizeof(double) * (size_t)(n + 1));
        for (int g = 0; g < Hkv; ++g) {
            int64_t row0 = ((int64_t)b * Hkv + g) * cap;
            orc_decode(s, s2, d, k_bits, k_centroids, k_packed + row0 * rbk, k_norm + row0, n, kh);
            orc_decode(s, s2, d, v_bits, v_centroids, v_packed + row0 * rbv, v_norm + row0, n, vh);
            for (int t = 0; t < T; ++t) {
                int64_t ctx = (int64_t)q_start[b] + t + 1;
                for (int hh = 0; hh < G; ++hh) {
                    int h = g * G + hh;
                    const double *qh = q + (((int64_t)b * T + t) * Hq + h) * d;
                    double *o = out + (((int64_t)b * T + t) * Hq + h) * d;
                    double m = -INFINITY, l = 0.0;
                    for (int64_t u = 0; u < ctx; ++u) {
                        double dot = 0.0;
                        for (int j = 0; j < d; ++j) dot += qh[j] * kh[u * d + j];
                        sig[u] = scale * dot;
                        if (sig[u] > m) m = sig[u];
                    }
                    for (int64_t u = 0; u < ctx; ++u) l += exp(sig[u] - m);
                    for (int j = 0; j < d; ++j) o[j] = 0.0;
                    for (int64_t u = 0; u < ctx; ++u) {
                        double p = exp(sig[u] - m) / l;
                        for (int j = 0; j < d; ++j) o[j] += p * vh[u * d + j];
                    }
                }
            }
        }
        free(kh);
        free(vh);
        free(sig);
    }
}

/* ------------------------------------------------------ QJL residual keys */

/* The Gaussian projection of the QJL stage (reading in tq_oracle.h). */
void orc_qjl_matrix(uint64_t seed, int d, double *S) {
    uint64_t state = seed;
    for (int i = 0; i < 2 * d; ++i) orc_splitmix64_next(&state); /* s1, s2 */
    const double two53 = 9007199254740992.0;
    for (int64_t k = 0; k < (int64_t)d * d; ++k) {
        double u1 = (double)(orc_splitmix64_next(&state) >> 11) / two53;
        double u2 = (double)(orc_splitmix64_next(&state) >> 11) / two53;
        S[k] = sqrt(-2.0 * log(1.0 - u1)) * cos(2.0 * M_PI * u2);
    }
}

void orc_encode_qjl(const int8_t *s, const int8_t *s2, int d, int bits, const float *c_mse,
                    const float *b_mse, const double *S, const double *x, int64_t n_rows,
                    uint8_t *packed, float *norms, float *rnorms, double *proj_out) {
    int rb = d * bits / 8, ib = d * (bits - 1) / 8;
    double *y = (double *)malloc(sizeof(double) * d);
    double *r = (double *)malloc(sizeof(double) * d);
    uint8_t *idx = (uint8_t *)malloc((size_t)d);
    uint8_t *sg = (uint8_t *)malloc((size_t)d);
    for (int64_t row = 0; row < n_rows; ++row) {
        const double *xr = x + row * d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += xr[i] * xr[i];
        double n = sqrt(ss);
        orc_rotate(s, s2, d, xr, y);
        norms[row] = (float)n;
        /* MSE stage on b - 1 bits, then the residual of the normalised row */
        double rr = 0.0;
        for (int i = 0; i < d; ++i) {
            double u = (n > 0.0) ? y[i] / n : 0.0;
            idx[i] = (uint8_t)orc_bucket((float)u, bits - 1, b_mse);
            r[i] = u - (double)c_mse[idx[i]];
            rr += r[i] * r[i];
        }
        rnorms[row] = (float)(n * sqrt(rr));
        /* QJL stage: the signs of S r */
        for (int k = 0; k < d; ++k) {
            double p = 0.0;
            for (int j = 0; j < d; ++j) p += S[(int64_t)k * d + j] * r[j];
            if (proj_out) proj_out[row * d + k] = p;
            sg[k] = p >= 0.0 ? 1 : 0;
        }
        orc_pack(idx, d, bits - 1, packed + row * rb);
        orc_pack(sg, d, 1, packed + row * rb + ib);
    }
    free(y);
    free(r);
    free(idx);
    free(sg);
}

void orc_decode_qjl(const int8_t *s, const int8_t *s2, int d, int bits, const float *c_mse,
                    const double *S, const uint8_t *packed, const float *norms, const float *rnorms,
                    int64_t n_rows, double *out) {
    int rb = d * bits / 8, ib = d * (bits - 1) / 8;
    double *yr = (double *)malloc(sizeof(double) * d);
    uint8_t *idx = (uint8_t *)malloc((size_t)d);
    uint8_t *sg = (uint8_t *)malloc((size_t)d);
    const double kappa = sqrt(M_PI / 2.0) / (double)d;
    for (int64_t row = 0; row < n_rows; ++row) {
        orc_unpack(packed + row * rb, d, bits - 1, idx);
        orc_unpack(packed + row * rb + ib, d, 1, sg);
        double n = (double)norms[row], g = (double)rnorms[row];
        for (int i = 0; i < d; ++i) {
            double t = 0.0;
            for (int k = 0; k < d; ++k) t += S[(int64_t)k * d + i] * (sg[k] ? 1.0 : -1.0);
            yr[i] = n * (double)c_mse[idx[i]] + kappa * g * t;
        }
        orc_unrotate(s, s2, d, yr, out + row * d);
    }
    free(yr);
    free(idx);
    free(sg);
}

void orc_attention_qjl(const int8_t *s, const int8_t *s2, int d, int B, int Hq, int Hkv, int64_t cap,
                       int64_t ctx_len, int k_bits, const float *k_c_mse, const double *S,
                       const uint8_t *k_packed, const float *k_norm, const float *k_rnorm, int v_bits,
                       const float *v_centroids, const uint8_t *v_packed, const float *v_norm,
                       const double *q, double scale, double *out) {
    int G = Hq / Hkv;
    int rbk = d * k_bits / 8, rbv = d * v_bits / 8;
    double *kh = (double *)malloc(sizeof(double) * (size_t)(ctx_len * d + 1));
    double *vh = (double *)malloc(sizeof(double) * (size_t)(ctx_len * d + 1));
    double *sig = (double *)malloc(sizeof(double) * (size_t)(ctx_len + 1));
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < Hkv; ++g) {
            int64_t row0 = ((int64_t)b * Hkv + g) * cap;
            orc_decode_qjl(s, s2, d, k_bits, k_c_mse, S, k_packed + row0 * rbk, k_norm + row0,
                           k_rnorm + row0, ctx_len, kh);
            orc_decode(s, s2, d, v_bits, v_centroids, v_packed + row0 * rbv, v_norm + row0, ctx_len, vh);
            for (int hh = 0; hh < G; ++hh) {
                int h = g * G + hh;
                const double *qh = q + ((int64_t)b * Hq + h) * d;
                double *o = out + ((int64_t)b * Hq + h) * d;
                double m = -INFINITY;
                for (int64_t t = 0; t < ctx_len; ++t) {
                    double dot = 0.0;
                    for (int j = 0; j < d; ++j) dot += qh[j] * kh[t * d + j];
                    sig[t] = scale * dot;
                    if (sig[t] > m) m = sig[t];
                }
                double l = 0.0;
                for (int64_t t = 0; t < ctx_len; ++t) l += exp(sig[t] - m);
                for (int j = 0; j < d; ++j) o[j] = 0.0;
                for (int64_t t = 0; t < ctx_len; ++t) {
                    double p = exp(sig[t] - m) / l;
                    for (int j = 0; j < d; ++j) o[j] += p * vh[t * d + j];
                }
            }
        }
    }
    free(kh);
    free(vh);
    free(sig);
}
