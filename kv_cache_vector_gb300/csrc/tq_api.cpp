// tq_api.cpp -- the C ABI: plan construction (codebooks, signs), argument
// validation, and dispatch to the sm_103a kernels.  See include/tq.h.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <new>
#include <type_traits>

#include "tq_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

tq_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return TQ_ERR_CUDA;
}

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// A pointer the GPU cannot dereference (pageable host memory on a system
// without pageable-memory access) is turned into an error instead of a fault.
// Unknown answers are let through.  Where the device reads pageable memory
// every pointer qualifies, so no per-pointer query is made (the answer is
// cached per device).
bool pageable_access() {
    static int cached[64] = {};  // 0 unknown, 1 no, 2 yes
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev] == 2;
    int pageable = 0;
    if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (dev >= 0 && dev < 64) cached[dev] = pageable ? 2 : 1;
    return pageable != 0;
}

bool device_accessible(const void* p) {
    if (pageable_access()) return true;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return a.type != cudaMemoryTypeUnregistered;
}

// ------------------------------------------------------------ signs

// splitmix64 (S. Vigna): the state advances by the 64-bit golden-ratio
// constant and each output is that state passed through two
// xor-shift/multiply rounds and a final xor-shift.
uint64_t splitmix64(uint64_t& st) {
    st += 0x9E3779B97F4A7C15ULL;
    uint64_t z = st;
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

// ---------------------------------------------------------- codebook
//
// One coordinate X of a uniform unit vector in R^d has density proportional
// to (1 - x^2)^((d-3)/2) on [-1, 1].  With x = sin(t) the mass of [0, x] is
// W_{d-2}(asin x), where W_n(T) = int_0^T cos^n is given in closed form by
// the reduction W_n = cos^{n-1}(T) sin(T) / n + (n-1)/n W_{n-2}, W_0 = T,
// W_1 = sin T; the first moment of [a, b] is
// ((1-a^2)^{(d-1)/2} - (1-b^2)^{(d-1)/2}) / (d-1).

double cos_power_integral(int n, double T) {
    const double s = std::sin(T), c = std::cos(T);
    double w = (n % 2 == 0) ? T : s;
    double cpow = (n % 2 == 0) ? c : c * c;  // cos^{k-1} for the first k below
    for (int k = (n % 2 == 0) ? 2 : 3; k <= n; k += 2) {
        w = cpow * s / k + (double)(k - 1) / k * w;
        cpow *= c * c;
    }
    return w;
}

struct SphereHalf {
    int d;
    double mass(double a, double b) const {  // 0 <= a <= b <= 1
        return cos_power_integral(d - 2, std::asin(b)) - cos_power_integral(d - 2, std::asin(a));
    }
    double moment(double a, double b) const {
        const double e = 0.5 * (d - 1);
        return (std::pow(1.0 - a * a, e) - std::pow(1.0 - b * b, e)) / (double)(d - 1);
    }
};

// N(0, 1/d), the large-d limit of the coordinate density ("CITATIONS", N(0,
// 1/d) codebook replacement: after the transform the per-coordinate variance
// is 1/d).  With sigma = 1/sqrt(d), the mass of [a, b] is
// (erfc(a / (sigma sqrt 2)) - erfc(b / (sigma sqrt 2))) / 2 and the first
// moment sigma^2 (phi(a) - phi(b)), phi the N(0, sigma^2) density; b may be
// +infinity.
struct GaussHalf {
    double sigma;
    double mass(double a, double b) const {
        const double k = 1.0 / (sigma * std::sqrt(2.0));
        return 0.5 * (std::erfc(a * k) - std::erfc(b * k));
    }
    double moment(double a, double b) const {
        auto g = [&](double x) { return std::isinf(x) ? 0.0 : std::exp(-0.5 * (x / sigma) * (x / sigma)); };
        return sigma / std::sqrt(2.0 * 3.14159265358979323846) * (g(a) - g(b));
    }
};

// Lloyd iteration on the positive half-line (both densities are symmetric
// and log-concave, so the optimum is symmetric and unique): centroids are
// conditional means of their cells, interior boundaries midpoints of
// neighbouring centroids.  Starts from cells evenly spread over
// [0, 2.5/sqrt(d)] and runs until the centroids settle at rounding level.
// `top` is the end of the support (1 for the sphere, +infinity for N(0, 1/d)).
template <class Density>
bool lloyd_half(const Density& f, int d, double top, int bits, double* c, double* beta) {
    const int H = (1 << bits) / 2;
    double w = 2.5 / std::sqrt((double)d);
    if (w > 1.0) w = 1.0;
    beta[0] = 0.0;
    beta[H] = top;
    for (int k = 1; k < H; ++k) beta[k] = w * k / H;
    double best = std::numeric_limits<double>::infinity();
    int stall = 0;
    for (int it = 0; it < 400000; ++it) {
        double moved = 0.0, big = 0.0;
        for (int k = 0; k < H; ++k) {
            double ck = f.moment(beta[k], beta[k + 1]) / f.mass(beta[k], beta[k + 1]);
            if (!std::isfinite(ck)) return false;
            if (it > 0) moved = std::fmax(moved, std::fabs(ck - c[k]));
            c[k] = ck;
            big = std::fmax(big, std::fabs(ck));
        }
        for (int k = 1; k < H; ++k) beta[k] = 0.5 * (c[k - 1] + c[k]);
        if (it == 0) continue;
        if (moved <= 4e-15 * big) return true;
        if (moved < 0.5 * best) {
            best = moved;
            stall = 0;
        } else if (++stall > 500 && best <= 1e-12 * big) {
            return true;
        }
    }
    return false;
}

bool codebook(int d, int bits, double* cen, double* bnd, bool gaussian = false) {
    const int L = 1 << bits, H = L / 2;
    double c[8], beta[9];
    const bool ok = gaussian ? lloyd_half(GaussHalf{1.0 / std::sqrt((double)d)}, d,
                                          std::numeric_limits<double>::infinity(), bits, c, beta)
                             : lloyd_half(SphereHalf{d}, d, 1.0, bits, c, beta);
    if (!ok) return false;
    for (int k = 0; k < H; ++k) {
        cen[H + k] = c[k];
        cen[H - 1 - k] = -c[k];
    }
    bnd[H - 1] = 0.0;
    for (int k = 1; k < H; ++k) {
        bnd[H - 1 + k] = beta[k];
        bnd[H - 1 - k] = -beta[k];
    }
    return true;
}

// The encode kernels bucket through a table of cells of width 1/scale; it
// is exact when no closed cell holds two boundaries.
bool lut_exact(const float* b32, int nb, int scale) {
    for (int j = 0; j + 1 < nb; ++j) {
        double gap = (double)b32[j + 1] - (double)b32[j];
        if (gap <= 1.0 / scale + 1e-12) return false;
    }
    return true;
}

void fill_row_params(const tq::Plan& P, int bits, tq::RowParams& R) {
    for (int w = 0; w < tq::kMaxD / 32; ++w) R.sgnb[w] = R.sgn2b[w] = 0u;
    for (int i = 0; i < tq::kMaxD; ++i) {
        R.sgn[i] = (i < P.d && P.signs[i] < 0) ? 0x80000000u : 0u;
        R.sgn2[i] = (i < P.d && P.signs2[i] < 0) ? 0x80000000u : 0u;
        if (R.sgn[i]) R.sgnb[i >> 5] |= 1u << (i & 31);
        if (R.sgn2[i]) R.sgn2b[i >> 5] |= 1u << (i & 31);
    }
    for (int j = 0; j < tq::kMaxD / 2; ++j) R.sgnh[j] = (R.sgn[2 * j] >> 16) | R.sgn[2 * j + 1];
    R.two_sided = (P.flags & TQ_PLAN_TWO_SIDED_SIGNS) ? 1 : 0;
    for (int i = 0; i < 16; ++i) {
        R.cen[i] = P.c32[bits][i];
        R.bnd[i] = P.b32[bits][i];
    }
    R.inv_sqrt_d = (float)(1.0 / std::sqrt((double)P.d));
}

// Nearest fp16 value of x (ties to even), for x inside the normal fp16 range:
// 11 significant bits.
double round_to_half(double x) {
    int e = 0;
    const double m = std::frexp(x, &e);  // x = m * 2^e, 0.5 <= |m| < 1
    return std::ldexp(std::nearbyint(std::ldexp(m, 11)), e - 11);
}

// The d = 128 attention multiplies fp16 centroids on the tensor cores.  A
// common scale s leaves the attention unchanged once 1/s is applied to the
// result, and a good s brings every centroid of the width close to an fp16
// value: s is the best of 2^14 evenly spaced candidates in [1, 2) for the
// worst relative rounding error (centroids are symmetric, so the positive
// half decides).
void half_scale(const float* c, int L, float* s_out, float* h_out) {
    double best = std::numeric_limits<double>::infinity(), best_s = 1.0;
    for (int i = 0; i < (1 << 14); ++i) {
        const double s = 1.0 + i / 16384.0;
        double worst = 0.0;
        for (int k = L / 2; k < L && worst < best; ++k) {
            const double v = (double)c[k] * s;
            worst = std::fmax(worst, std::fabs(round_to_half(v) - v) / std::fabs(v));
        }
        if (worst < best) {
            best = worst;
            best_s = s;
        }
    }
    *s_out = (float)best_s;  // 15 significant bits: exact
    for (int k = 0; k < 16; ++k) h_out[k] = k < L ? (float)round_to_half((double)c[k] * best_s) : 0.0f;
}

template <int V>
using IntC = std::integral_constant<int, V>;

// Call f(IntC<d>) for the supported head dimensions.
template <typename F>
cudaError_t dispatch_d(int d, F&& f) {
    switch (d) {
        case 8: return f(IntC<8>{});
        case 16: return f(IntC<16>{});
        case 32: return f(IntC<32>{});
        case 64: return f(IntC<64>{});
        case 128: return f(IntC<128>{});
        case 256: return f(IntC<256>{});
    }
    return cudaErrorInvalidValue;
}

template <typename F>
cudaError_t dispatch_attn_d(int d, F&& f) {
    switch (d) {
        case 32: return f(IntC<32>{});
        case 64: return f(IntC<64>{});
        case 128: return f(IntC<128>{});
        case 256: return f(IntC<256>{});
    }
    return cudaErrorInvalidValue;
}

// QJL residual keys: head dimensions whose matrix fits in shared memory.
bool qjl_d(int d) { return d == 32 || d == 64 || d == 128; }

template <typename F>
cudaError_t dispatch_qjl_d(int d, F&& f) {
    switch (d) {
        case 32: return f(IntC<32>{});
        case 64: return f(IntC<64>{});
        case 128: return f(IntC<128>{});
    }
    return cudaErrorInvalidValue;
}

bool valid_bits(int b) { return b >= 2 && b <= 4; }
bool valid_dtype(tq_dtype t) { return t == TQ_F32 || t == TQ_BF16; }

}  // namespace

void tq::set_last_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

void tq::fill_attn_params(const Plan& P, int k_bits, int v_bits, float scale, float sparse_thr,
                          AttnParams& A) {
    for (int w = 0; w < kMaxD / 32; ++w) A.sgnb[w] = A.sgn2b[w] = 0u;
    for (int i = 0; i < kMaxD; ++i) {
        A.sgn[i] = (i < P.d && P.signs[i] < 0) ? 0x80000000u : 0u;
        A.sgn2[i] = (i < P.d && P.signs2[i] < 0) ? 0x80000000u : 0u;
        if (A.sgn[i]) A.sgnb[i >> 5] |= 1u << (i & 31);
        if (A.sgn2[i]) A.sgn2b[i >> 5] |= 1u << (i & 31);
    }
    A.two_sided = (P.flags & TQ_PLAN_TWO_SIDED_SIGNS) ? 1 : 0;
    for (int i = 0; i < 16; ++i) {
        A.kcen[i] = P.c32[k_bits][i];
        A.vcen[i] = P.c32[v_bits][i];
        A.kcen_h[i] = P.hcen[k_bits][i];
        A.vcen_h[i] = P.hcen[v_bits][i];
    }
    const double sd = std::sqrt((double)P.d);
    A.inv_sqrt_d = (float)(1.0 / sd);
    A.scale = scale;
    A.sparse_thr = sparse_thr;
    const double ks = P.hscale[k_bits] > 0.0f ? P.hscale[k_bits] : 1.0;
    const double vs = P.hscale[v_bits] > 0.0f ? P.hscale[v_bits] : 1.0;
    for (int i = 0; i < 16; ++i) A.kcen_l[i] = (float)((double)P.c32[k_bits][i] * ks - (double)P.hcen[k_bits][i]);
    A.q_mul = (float)((double)scale * 1.4426950408889634 / (sd * ks));
    A.out_mul = (float)(1.0 / vs);
    A.v_rows = nullptr;
}

tq_status tq::check_attn_decode_args(const tq_plan* plan, const void* q, int B, int Hq, int Hkv,
                                     const tq_cache_view& cache, int64_t ctx_len, int k_bits, int v_bits,
                                     float scale, float sparse_v_threshold, const float* out, bool* nothing) {
    *nothing = false;
    if (!plan || B < 0 || Hq <= 0 || Hkv <= 0) return TQ_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return TQ_ERR_INVALID_ARG;
    if (!valid_bits(k_bits) || !valid_bits(v_bits)) return TQ_ERR_UNSUPPORTED;
    if (Hq / Hkv > 8) return TQ_ERR_UNSUPPORTED;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    if (P->d < 32) return TQ_ERR_UNSUPPORTED;
    if (!(std::isfinite(scale)) || !(sparse_v_threshold >= 0.0f) || !std::isfinite(sparse_v_threshold))
        return TQ_ERR_INVALID_ARG;
    if (ctx_len < 1 || ctx_len > cache.cap) return TQ_ERR_RANGE;
    // the d = 128 kernel counts work items and positions in 32 bits
    if (ctx_len > (int64_t(1) << 30) || (int64_t)B * Hkv * ((ctx_len + 31) / 32) > INT32_MAX)
        return TQ_ERR_UNSUPPORTED;
    if (B == 0) {
        *nothing = true;
        return TQ_OK;
    }
    if (!q || !out || !cache.k_packed || !cache.k_norm || !cache.v_packed || !cache.v_norm)
        return TQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(cache.k_packed) ||
        !aligned16(cache.v_packed) || !aligned4(cache.k_norm) || !aligned4(cache.v_norm))
        return TQ_ERR_ALIGNMENT;
    if (!device_accessible(q) || !device_accessible(out) || !device_accessible(cache.k_packed) ||
        !device_accessible(cache.v_packed) || !device_accessible(cache.k_norm) ||
        !device_accessible(cache.v_norm))
        return TQ_ERR_INVALID_ARG;
    return TQ_OK;
}

cudaError_t tq::launch_attn_decode(const Plan& P, const void* q, int B, int Hq, int Hkv,
                                   const tq_cache_view& cache, int64_t ctx_len, int k_bits, int v_bits,
                                   float scale, float sparse_v_threshold, float* out, int32_t* v_rows,
                                   void* workspace, const AttnGeometry& g, cudaStream_t st) {
    tq::AttnParams A;
    tq::fill_attn_params(P, k_bits, v_bits, scale, sparse_v_threshold, A);
    if (v_rows) {  // counted by the split kernels, one add per warp and (batch, KV head) run
        const cudaError_t e = cudaMemsetAsync(v_rows, 0, sizeof(int32_t) * (size_t)B * Hkv, st);
        if (e != cudaSuccess) return e;
        A.v_rows = v_rows;
    }
    return dispatch_attn_d(P.d, [&](auto D) {
        constexpr int d = decltype(D)::value;
        switch (k_bits) {
            case 2: return tq::launch_attn_dk<d, 2>(v_bits, q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, A, st);
            case 3: return tq::launch_attn_dk<d, 3>(v_bits, q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, A, st);
            default: return tq::launch_attn_dk<d, 4>(v_bits, q, B, Hq, Hkv, cache, ctx_len, out, workspace, g, A, st);
        }
    });
}

extern "C" {

tq_status tq_codebook_init(int d, int bits, double* centroids, double* boundaries) {
    if (!centroids || !boundaries) return TQ_ERR_INVALID_ARG;
    if (d < 3 || d > 65536 || bits < 1 || bits > 4) return TQ_ERR_UNSUPPORTED;
    return codebook(d, bits, centroids, boundaries) ? TQ_OK : TQ_ERR_UNSUPPORTED;
}

tq_status tq_codebook_init_gaussian(int d, int bits, double* centroids, double* boundaries) {
    if (!centroids || !boundaries) return TQ_ERR_INVALID_ARG;
    if (d < 1 || d > 65536 || bits < 1 || bits > 4) return TQ_ERR_UNSUPPORTED;
    return codebook(d, bits, centroids, boundaries, true) ? TQ_OK : TQ_ERR_UNSUPPORTED;
}

tq_status tq_plan_create(int d, uint64_t seed, tq_plan** out) { return tq_plan_create_ex(d, seed, 0u, out); }

tq_status tq_plan_create_ex(int d, uint64_t seed, uint32_t flags, tq_plan** out) {
    if (!out) return TQ_ERR_INVALID_ARG;
    *out = nullptr;
    if (flags & ~(uint32_t)(TQ_PLAN_GAUSSIAN_CODEBOOK | TQ_PLAN_TWO_SIDED_SIGNS)) return TQ_ERR_UNSUPPORTED;
    if (!is_pow2(d) || d < 8 || d > tq::kMaxD) return TQ_ERR_UNSUPPORTED;
    tq::Plan* P = new (std::nothrow) tq::Plan;
    if (!P) return TQ_ERR_NOMEM;
    std::memset(P, 0, sizeof(*P));
    P->d = d;
    P->seed = seed;
    P->flags = flags;
    // s1 = the stream's first d outputs; two-sided: s2 = the next d
    uint64_t st = seed;
    for (int i = 0; i < d; ++i) P->signs[i] = (splitmix64(st) >> 63) ? -1 : 1;
    for (int i = 0; i < d; ++i)
        P->signs2[i] = (flags & TQ_PLAN_TWO_SIDED_SIGNS) ? ((splitmix64(st) >> 63) ? -1 : 1) : 1;
    const bool gauss = (flags & TQ_PLAN_GAUSSIAN_CODEBOOK) != 0;
    for (int bits = 1; bits <= 4; ++bits) {
        const int L = 1 << bits;
        if (!codebook(d, bits, P->c64[bits], P->b64[bits], gauss)) {
            delete P;
            return TQ_ERR_UNSUPPORTED;
        }
        for (int i = 0; i < 16; ++i) {
            P->c32[bits][i] = i < L ? (float)P->c64[bits][i] : 0.0f;
            P->b32[bits][i] = i < L - 1 ? (float)P->b64[bits][i]
                                        : std::numeric_limits<float>::infinity();
        }
        if (bits >= 2 && (!lut_exact(P->b32[bits], L - 1, tq::kLutScale) ||
                          ((d == 128 || d == 256) && !lut_exact(P->b32[bits], L - 1, tq::kUmLutScale)))) {
            delete P;
            return TQ_ERR_UNSUPPORTED;
        }
        if (bits >= 2 && d == 128) half_scale(P->c32[bits], L, &P->hscale[bits], P->hcen[bits]);
    }
    *out = reinterpret_cast<tq_plan*>(P);
    return TQ_OK;
}

tq_status tq_plan_destroy(tq_plan* plan) {
    delete reinterpret_cast<tq::Plan*>(plan);
    return TQ_OK;
}

tq_status tq_plan_signs(const tq_plan* plan, int8_t* signs) {
    if (!plan || !signs) return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    std::memcpy(signs, P->signs, (size_t)P->d);
    return TQ_OK;
}

tq_status tq_plan_signs2(const tq_plan* plan, int8_t* signs) {
    if (!plan || !signs) return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    std::memcpy(signs, P->signs2, (size_t)P->d);
    return TQ_OK;
}

tq_status tq_plan_codebook(const tq_plan* plan, int bits, float* centroids, float* boundaries) {
    if (!plan || !centroids || !boundaries) return TQ_ERR_INVALID_ARG;
    if (bits < 1 || bits > 4) return TQ_ERR_UNSUPPORTED;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    const int L = 1 << bits;
    std::memcpy(centroids, P->c32[bits], sizeof(float) * L);
    std::memcpy(boundaries, P->b32[bits], sizeof(float) * (L - 1));
    return TQ_OK;
}

tq_status tq_encode(const tq_plan* plan, int bits, const void* x, tq_dtype x_dtype,
                    int64_t n_rows, uint8_t* packed, float* norms, tq_stream_t stream) {
    if (!plan || n_rows < 0) return TQ_ERR_INVALID_ARG;
    if (!valid_bits(bits) || !valid_dtype(x_dtype)) return TQ_ERR_UNSUPPORTED;
    if (n_rows == 0) return TQ_OK;
    if (!x || !packed || !norms) return TQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(packed) || !aligned4(norms)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(x) || !device_accessible(packed) || !device_accessible(norms))
        return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    tq::RowParams R;
    fill_row_params(*P, bits, R);
    cudaError_t e = dispatch_d(P->d, [&](auto D) {
        return tq::launch_encode_d<decltype(D)::value>(bits, x_dtype, x, n_rows, packed, norms, R,
                                                       reinterpret_cast<cudaStream_t>(stream));
    });
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_decode(const tq_plan* plan, int bits, const uint8_t* packed, const float* norms,
                    int64_t n_rows, void* y, tq_dtype y_dtype, tq_stream_t stream) {
    if (!plan || n_rows < 0) return TQ_ERR_INVALID_ARG;
    if (!valid_bits(bits) || !valid_dtype(y_dtype)) return TQ_ERR_UNSUPPORTED;
    if (n_rows == 0) return TQ_OK;
    if (!y || !packed || !norms) return TQ_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(packed) || !aligned4(norms)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(y) || !device_accessible(packed) || !device_accessible(norms))
        return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    tq::RowParams R;
    fill_row_params(*P, bits, R);
    cudaError_t e = dispatch_d(P->d, [&](auto D) {
        return tq::launch_decode_d<decltype(D)::value>(bits, y_dtype, packed, norms, n_rows, y, R,
                                                       reinterpret_cast<cudaStream_t>(stream));
    });
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_append(const tq_plan* plan, int k_bits, int v_bits, const void* k_new,
                    const void* v_new, tq_dtype dtype, int B, int Hkv, int64_t n_new,
                    tq_cache_view cache, int64_t pos, tq_stream_t stream) {
    if (!plan || B < 0 || Hkv < 0 || n_new < 0) return TQ_ERR_INVALID_ARG;
    if (!valid_bits(k_bits) || !valid_bits(v_bits) || !valid_dtype(dtype))
        return TQ_ERR_UNSUPPORTED;
    if (pos < 0 || cache.cap < 0 || pos + n_new > cache.cap) return TQ_ERR_RANGE;
    if ((int64_t)B * Hkv * n_new == 0) return TQ_OK;
    if (!k_new || !v_new || !cache.k_packed || !cache.k_norm || !cache.v_packed || !cache.v_norm)
        return TQ_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(cache.k_packed) ||
        !aligned16(cache.v_packed) || !aligned4(cache.k_norm) || !aligned4(cache.v_norm))
        return TQ_ERR_ALIGNMENT;
    if (!device_accessible(k_new) || !device_accessible(v_new) ||
        !device_accessible(cache.k_packed) || !device_accessible(cache.v_packed) ||
        !device_accessible(cache.k_norm) || !device_accessible(cache.v_norm))
        return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    tq::RowParams PK, PV;
    fill_row_params(*P, k_bits, PK);
    fill_row_params(*P, v_bits, PV);
    cudaError_t e = dispatch_d(P->d, [&](auto D) {
        return tq::launch_append_d<decltype(D)::value>(k_bits, v_bits, dtype, k_new, v_new, B, Hkv,
                                                       n_new, cache, pos, PK, PV,
                                                       reinterpret_cast<cudaStream_t>(stream));
    });
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

size_t tq_attn_workspace_bytes(int B, int Hq, int Hkv, int d, int64_t ctx_len) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || ctx_len < 1 || !is_pow2(d) ||
        d > tq::kMaxD)
        return 0;
    return tq::attn_workspace_bound(B, Hq, Hkv, ctx_len, tq::num_sms(), d);
}

size_t tq_attn_paged_workspace_bytes(int B, int Hq, int Hkv, int d, int64_t max_ctx) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_ctx < 1) return 0;
    if (d == 128) return tq::attn_paged_workspace_bound(B, Hq, Hkv, max_ctx, tq::num_sms());
    if (d != 32 && d != 64 && d != 256) return 0;
    return tq::attn_workspace_bound(B, Hq, Hkv, max_ctx, tq::num_sms(), d);
}

tq_status tq_attn_decode_ex(const tq_plan* plan, const void* q, int B, int Hq, int Hkv,
                            tq_cache_view cache, int64_t ctx_len, int k_bits, int v_bits,
                            float scale, float sparse_v_threshold, float* out, int32_t* v_rows_read,
                            void* workspace, size_t workspace_bytes, tq_stream_t stream) {
    bool nothing = false;
    tq_status st = tq::check_attn_decode_args(plan, q, B, Hq, Hkv, cache, ctx_len, k_bits, v_bits, scale,
                                              sparse_v_threshold, out, &nothing);
    if (st != TQ_OK || nothing) return st;
    if (v_rows_read && (!aligned4(v_rows_read))) return TQ_ERR_ALIGNMENT;
    if (v_rows_read && !device_accessible(v_rows_read)) return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    const tq::AttnGeometry g = tq::attn_geometry(B, Hq, Hkv, ctx_len, tq::num_sms(), P->d, k_bits, v_bits,
                                                 sparse_v_threshold > 0.0f);
    if (!workspace || workspace_bytes < tq::attn_workspace_bytes(B, Hq, P->d, g)) return TQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(workspace)) return TQ_ERR_INVALID_ARG;
    const cudaError_t e = tq::launch_attn_decode(*P, q, B, Hq, Hkv, cache, ctx_len, k_bits, v_bits, scale,
                                                 sparse_v_threshold, out, v_rows_read, workspace, g,
                                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_attn_decode(const tq_plan* plan, const void* q, int B, int Hq, int Hkv,
                         tq_cache_view cache, int64_t ctx_len, int k_bits, int v_bits,
                         float scale, float sparse_v_threshold, float* out, void* workspace,
                         size_t workspace_bytes, tq_stream_t stream) {
    return tq_attn_decode_ex(plan, q, B, Hq, Hkv, cache, ctx_len, k_bits, v_bits, scale, sparse_v_threshold,
                             out, nullptr, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------ QJL residual keys

tq_status tq_qjl_matrix(const tq_plan* plan, float* S, tq_stream_t stream) {
    if (!plan || !S) return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    if (!qjl_d(P->d)) return TQ_ERR_UNSUPPORTED;
    if (!aligned16(S)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(S)) return TQ_ERR_INVALID_ARG;
    const cudaError_t e = tq::launch_qjl_matrix(P->seed, P->d, S, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_encode_qjl(const tq_plan* plan, int bits, const float* S, const void* x, tq_dtype x_dtype,
                        int64_t n_rows, uint8_t* packed, float* norms, float* rnorms, tq_stream_t stream) {
    if (!plan || n_rows < 0) return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    if (!valid_bits(bits) || !valid_dtype(x_dtype) || !qjl_d(P->d)) return TQ_ERR_UNSUPPORTED;
    if (n_rows == 0) return TQ_OK;
    if (!S || !x || !packed || !norms || !rnorms) return TQ_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(x) || !aligned16(packed) || !aligned4(norms) || !aligned4(rnorms))
        return TQ_ERR_ALIGNMENT;
    if (!device_accessible(S) || !device_accessible(x) || !device_accessible(packed) ||
        !device_accessible(norms) || !device_accessible(rnorms))
        return TQ_ERR_INVALID_ARG;
    tq::RowParams R;
    fill_row_params(*P, bits - 1, R);
    cudaError_t e = dispatch_qjl_d(P->d, [&](auto D) {
        return tq::launch_encode_qjl_d<decltype(D)::value>(bits, x_dtype, x, n_rows, S, packed, norms, rnorms, R,
                                                           reinterpret_cast<cudaStream_t>(stream));
    });
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_decode_qjl(const tq_plan* plan, int bits, const float* S, const uint8_t* packed, const float* norms,
                        const float* rnorms, int64_t n_rows, void* y, tq_dtype y_dtype, tq_stream_t stream) {
    if (!plan || n_rows < 0) return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    if (!valid_bits(bits) || !valid_dtype(y_dtype) || !qjl_d(P->d)) return TQ_ERR_UNSUPPORTED;
    if (n_rows == 0) return TQ_OK;
    if (!S || !y || !packed || !norms || !rnorms) return TQ_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(y) || !aligned16(packed) || !aligned4(norms) || !aligned4(rnorms))
        return TQ_ERR_ALIGNMENT;
    if (!device_accessible(S) || !device_accessible(y) || !device_accessible(packed) ||
        !device_accessible(norms) || !device_accessible(rnorms))
        return TQ_ERR_INVALID_ARG;
    tq::RowParams R;
    fill_row_params(*P, bits - 1, R);
    cudaError_t e = dispatch_qjl_d(P->d, [&](auto D) {
        return tq::launch_decode_qjl_d<decltype(D)::value>(bits, y_dtype, packed, norms, rnorms, n_rows, S, y, R,
                                                           reinterpret_cast<cudaStream_t>(stream));
    });
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

size_t tq_attn_qjl_workspace_bytes(int B, int Hq, int Hkv, int d, int64_t ctx_len) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || ctx_len < 1 || !qjl_d(d)) return 0;
    size_t most = tq::attn_qjl_workspace_bytes(B, Hq, d, tq::attn_qjl_geometry(B, Hq, Hkv, ctx_len, tq::num_sms()));
    if (d == 128 && Hq / Hkv <= 8) {  // 3- and 4-bit keys: the tensor-core kernel
        for (int kb = 3; kb <= 4; ++kb)
            for (int vb = 2; vb <= 4; ++vb) {
                const size_t w = tq::attn_qjl128_workspace_bytes(
                    B, Hq, tq::attn_qjl128_geometry(B, Hq, Hkv, ctx_len, tq::num_sms(), kb, vb));
                if (w > most) most = w;
            }
    }
    return most;
}

tq_status tq_attn_decode_qjl(const tq_plan* plan, const float* S, const void* q, int B, int Hq, int Hkv,
                             tq_cache_view cache, const float* k_rnorm, int64_t ctx_len, int k_bits, int v_bits,
                             float scale, float* out, void* workspace, size_t workspace_bytes,
                             tq_stream_t stream) {
    if (!plan) return TQ_ERR_INVALID_ARG;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    if (!qjl_d(P->d)) return TQ_ERR_UNSUPPORTED;
    bool nothing = false;
    tq_status st = tq::check_attn_decode_args(plan, q, B, Hq, Hkv, cache, ctx_len, k_bits, v_bits, scale, 0.0f,
                                              out, &nothing);
    if (st != TQ_OK || nothing) return st;
    if (!S || !k_rnorm) return TQ_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned4(k_rnorm)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(S) || !device_accessible(k_rnorm)) return TQ_ERR_INVALID_ARG;
    // 3- and 4-bit keys at d = 128 run on the tensor cores, the rest on the CUDA cores
    const bool tc = P->d == 128 && k_bits >= 3;
    const tq::AttnGeometry g = tc ? tq::attn_qjl128_geometry(B, Hq, Hkv, ctx_len, tq::num_sms(), k_bits, v_bits)
                                  : tq::attn_qjl_geometry(B, Hq, Hkv, ctx_len, tq::num_sms());
    const size_t need = tc ? tq::attn_qjl128_workspace_bytes(B, Hq, g) : tq::attn_qjl_workspace_bytes(B, Hq, P->d, g);
    if (!workspace || workspace_bytes < need) return TQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(workspace)) return TQ_ERR_INVALID_ARG;
    tq::AttnParams A;
    tq::fill_attn_params(*P, k_bits - 1, v_bits, scale, 0.0f, A);
    if (tc) {
        // q' = scale log2(e) sqrt(pi/2) / (d sqrt(d)) S y, y the unnormalised rotated query
        const float proj_mul = (float)((double)scale * 1.4426950408889634 * 1.2533141373155003 / (128.0 * std::sqrt(128.0)));
        const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        const cudaError_t e3 =
            k_bits == 3 ? tq::launch_attn3_qjl<3>(v_bits, q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, A,
                                                  proj_mul, s)
                        : tq::launch_attn3_qjl<4>(v_bits, q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, A,
                                                  proj_mul, s);
        return e3 == cudaSuccess ? TQ_OK : cuda_fail(e3);
    }
    cudaError_t e = dispatch_qjl_d(P->d, [&](auto D) {
        constexpr int d = decltype(D)::value;
        const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
        switch (k_bits) {
            case 2: return tq::launch_attn_qjl<d, 2>(v_bits, q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, A, s);
            case 3: return tq::launch_attn_qjl<d, 3>(v_bits, q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, A, s);
            default: return tq::launch_attn_qjl<d, 4>(v_bits, q, S, B, Hq, Hkv, cache, k_rnorm, ctx_len, out, workspace, g, A, s);
        }
    });
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

// ------------------------------------------------------------ paged cache

namespace {
// page_size a power of two >= 32: its log2, else -1.
int page_shift_of(int32_t page_size) {
    if (page_size < 32 || (page_size & (page_size - 1)) != 0) return -1;
    int sh = 0;
    while ((1 << sh) < page_size) ++sh;
    return sh;
}
bool paged_pointers_ok(const tq_paged_cache& c) {
    return c.k_packed && c.k_norm && c.v_packed && c.v_norm;
}
bool paged_aligned(const tq_paged_cache& c) {
    return aligned16(c.k_packed) && aligned16(c.v_packed) && aligned4(c.k_norm) && aligned4(c.v_norm);
}
bool paged_accessible(const tq_paged_cache& c) {
    return device_accessible(c.k_packed) && device_accessible(c.v_packed) &&
           device_accessible(c.k_norm) && device_accessible(c.v_norm);
}
tq_cache_view paged_as_view(const tq_paged_cache& c) {
    tq_cache_view v;
    v.k_packed = c.k_packed;
    v.k_norm = c.k_norm;
    v.v_packed = c.v_packed;
    v.v_norm = c.v_norm;
    v.cap = 0;  // unused on the paged paths
    return v;
}

// Paged attention for d != 128 (the generic kernel), after the common checks:
// sequence b attends over lens[b] + len_plus positions, clamped to max_ctx.
tq_status generic_paged(const tq::Plan& P, const void* q, int B, int Hq, int Hkv, const tq_paged_cache& cache,
                        const int32_t* block_table, int max_pages, const int32_t* lens, int len_plus,
                        int64_t max_ctx, int shift, int k_bits, int v_bits, float scale, float sparse_v_threshold,
                        float* out, void* workspace, size_t workspace_bytes, tq_stream_t stream) {
    const tq::AttnGeometry g = tq::attn_geometry(B, Hq, Hkv, max_ctx, tq::num_sms(), P.d, k_bits, v_bits);
    if (!workspace || workspace_bytes < tq::attn_workspace_bytes(B, Hq, P.d, g)) return TQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(q) || !device_accessible(out) || !device_accessible(workspace) ||
        !device_accessible(block_table) || !device_accessible(lens) || !paged_accessible(cache))
        return TQ_ERR_INVALID_ARG;
    tq::AttnParams A;
    tq::fill_attn_params(P, k_bits, v_bits, scale, sparse_v_threshold, A);
    const tq::PagedArgs pa{block_table, lens, cache.n_pages, max_pages, shift};
    const tq_cache_view view = paged_as_view(cache);
    auto st = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = dispatch_attn_d(P.d, [&](auto D) -> cudaError_t {
        constexpr int d = decltype(D)::value;
        if constexpr (d == 128) {
            return cudaErrorInvalidValue;  // the d = 128 kernel has its own paged path
        } else {
            switch (k_bits) {
                case 2: return tq::launch_attn_generic_paged<d, 2>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, len_plus, st);
                case 3: return tq::launch_attn_generic_paged<d, 3>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, len_plus, st);
                default: return tq::launch_attn_generic_paged<d, 4>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, len_plus, st);
            }
        }
    });
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}
}  // namespace

tq_status tq_append_paged(const tq_plan* plan, int k_bits, int v_bits, const void* k_new,
                          const void* v_new, tq_dtype dtype, int B, int Hkv, tq_paged_cache cache,
                          const int32_t* block_table, int max_pages, const int32_t* positions,
                          tq_stream_t stream) {
    if (!plan || B < 0 || Hkv <= 0 || max_pages < 1 || cache.n_pages < 1) return TQ_ERR_INVALID_ARG;
    if (!valid_bits(k_bits) || !valid_bits(v_bits) || !valid_dtype(dtype)) return TQ_ERR_UNSUPPORTED;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    const int shift = page_shift_of(cache.page_size);
    if (P->d < 32 || shift < 0) return TQ_ERR_UNSUPPORTED;
    if (B == 0) return TQ_OK;
    if (!k_new || !v_new || !block_table || !positions || !paged_pointers_ok(cache)) return TQ_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned4(block_table) || !aligned4(positions) ||
        !paged_aligned(cache))
        return TQ_ERR_ALIGNMENT;
    if (!device_accessible(k_new) || !device_accessible(v_new) || !device_accessible(block_table) ||
        !device_accessible(positions) || !paged_accessible(cache))
        return TQ_ERR_INVALID_ARG;
    tq::RowParams PK, PV;
    fill_row_params(*P, k_bits, PK);
    fill_row_params(*P, v_bits, PV);
    const tq::PagedArgs pa{block_table, positions, cache.n_pages, max_pages, shift};
    const tq_cache_view view = paged_as_view(cache);
    cudaError_t e = dispatch_d(P->d, [&](auto D) {
        return tq::launch_append_paged_d<decltype(D)::value>(k_bits, v_bits, dtype, k_new, v_new, B, Hkv,
                                                             view, pa, PK, PV,
                                                             reinterpret_cast<cudaStream_t>(stream));
    });
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_attn_decode_paged(const tq_plan* plan, const void* q, int B, int Hq, int Hkv,
                               tq_paged_cache cache, const int32_t* block_table, int max_pages,
                               const int32_t* ctx_lens, int64_t max_ctx, int k_bits, int v_bits,
                               float scale, float sparse_v_threshold, float* out, void* workspace,
                               size_t workspace_bytes, tq_stream_t stream) {
    if (!plan || B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_pages < 1 || cache.n_pages < 1)
        return TQ_ERR_INVALID_ARG;
    if (!valid_bits(k_bits) || !valid_bits(v_bits) || Hq / Hkv > 8) return TQ_ERR_UNSUPPORTED;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    const int shift = page_shift_of(cache.page_size);
    if ((P->d != 128 && P->d != 32 && P->d != 64 && P->d != 256) || shift < 0) return TQ_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || !(sparse_v_threshold >= 0.0f) || !std::isfinite(sparse_v_threshold))
        return TQ_ERR_INVALID_ARG;
    if (max_ctx < 1 || max_ctx > ((int64_t)max_pages << shift)) return TQ_ERR_RANGE;
    if (max_ctx > (int64_t(1) << 30) || B > 65535) return TQ_ERR_UNSUPPORTED;  // 32-bit positions; grid
    if (B == 0) return TQ_OK;
    if (!q || !out || !block_table || !ctx_lens || !paged_pointers_ok(cache)) return TQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned4(block_table) || !aligned4(ctx_lens) ||
        !paged_aligned(cache))
        return TQ_ERR_ALIGNMENT;
    if (P->d != 128)
        return generic_paged(*P, q, B, Hq, Hkv, cache, block_table, max_pages, ctx_lens, 0, max_ctx, shift, k_bits,
                             v_bits, scale, sparse_v_threshold, out, workspace, workspace_bytes, stream);
    tq::AttnGeometry g = tq::attn_geometry_paged(B, Hq, Hkv, max_ctx, tq::num_sms(), k_bits, v_bits);
    if ((int64_t)B * Hkv * g.n_splits > INT32_MAX) return TQ_ERR_UNSUPPORTED;  // work items are int32
    if (!workspace || workspace_bytes < tq::attn_workspace_bytes(B, Hq, P->d, g)) return TQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(q) || !device_accessible(out) || !device_accessible(workspace) ||
        !device_accessible(block_table) || !device_accessible(ctx_lens) || !paged_accessible(cache))
        return TQ_ERR_INVALID_ARG;
    tq::AttnParams A;
    tq::fill_attn_params(*P, k_bits, v_bits, scale, sparse_v_threshold, A);
    const tq::PagedArgs pa{block_table, ctx_lens, cache.n_pages, max_pages, shift};
    const tq_cache_view view = paged_as_view(cache);
    auto st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (k_bits) {
        case 2: e = tq::launch_attn128_paged<2>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, st); break;
        case 3: e = tq::launch_attn128_paged<3>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, st); break;
        default: e = tq::launch_attn128_paged<4>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, st); break;
    }
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_attn_decode_append_paged(const tq_plan* plan, const void* q, const void* k_new,
                                      const void* v_new, tq_dtype kv_dtype, int B, int Hq, int Hkv,
                                      tq_paged_cache cache, const int32_t* block_table, int max_pages,
                                      const int32_t* positions, int64_t max_ctx, int k_bits, int v_bits,
                                      float scale, float sparse_v_threshold, float* out, void* workspace,
                                      size_t workspace_bytes, tq_stream_t stream) {
    if (!plan || B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_pages < 1 || cache.n_pages < 1)
        return TQ_ERR_INVALID_ARG;
    if (!valid_bits(k_bits) || !valid_bits(v_bits) || Hq / Hkv > 8 || !valid_dtype(kv_dtype))
        return TQ_ERR_UNSUPPORTED;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    const int shift = page_shift_of(cache.page_size);
    if ((P->d != 128 && P->d != 32 && P->d != 64 && P->d != 256) || shift < 0) return TQ_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || !(sparse_v_threshold >= 0.0f) || !std::isfinite(sparse_v_threshold))
        return TQ_ERR_INVALID_ARG;
    if (max_ctx < 1 || max_ctx > ((int64_t)max_pages << shift)) return TQ_ERR_RANGE;
    if (max_ctx > (int64_t(1) << 30) || B > 65535) return TQ_ERR_UNSUPPORTED;  // 32-bit positions; grid
    if (B == 0) return TQ_OK;
    if (!q || !k_new || !v_new || !out || !block_table || !positions || !paged_pointers_ok(cache))
        return TQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out) || !aligned4(block_table) ||
        !aligned4(positions) || !paged_aligned(cache))
        return TQ_ERR_ALIGNMENT;
    if (P->d != 128) {
        // the append, then the attention over positions[b] + 1 rows: two launches
        if (!device_accessible(k_new) || !device_accessible(v_new)) return TQ_ERR_INVALID_ARG;
        tq::RowParams PK, PV;
        fill_row_params(*P, k_bits, PK);
        fill_row_params(*P, v_bits, PV);
        const tq::PagedArgs pa{block_table, positions, cache.n_pages, max_pages, shift};
        const tq_cache_view view = paged_as_view(cache);
        const cudaError_t e = dispatch_d(P->d, [&](auto D) {
            return tq::launch_append_paged_d<decltype(D)::value>(k_bits, v_bits, kv_dtype, k_new, v_new, B, Hkv,
                                                                 view, pa, PK, PV,
                                                                 reinterpret_cast<cudaStream_t>(stream));
        });
        if (e != cudaSuccess) return cuda_fail(e);
        return generic_paged(*P, q, B, Hq, Hkv, cache, block_table, max_pages, positions, 1, max_ctx, shift, k_bits,
                             v_bits, scale, sparse_v_threshold, out, workspace, workspace_bytes, stream);
    }
    tq::AttnGeometry g = tq::attn_geometry_paged(B, Hq, Hkv, max_ctx, tq::num_sms(), k_bits, v_bits);
    if ((int64_t)B * Hkv * g.n_splits > INT32_MAX) return TQ_ERR_UNSUPPORTED;  // work items are int32
    if (!workspace || workspace_bytes < tq::attn_workspace_bytes(B, Hq, P->d, g)) return TQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(q) || !device_accessible(k_new) || !device_accessible(v_new) ||
        !device_accessible(out) || !device_accessible(workspace) || !device_accessible(block_table) ||
        !device_accessible(positions) || !paged_accessible(cache))
        return TQ_ERR_INVALID_ARG;
    tq::AttnParams A;
    tq::fill_attn_params(*P, k_bits, v_bits, scale, sparse_v_threshold, A);
    tq::RowParams PK, PV;
    fill_row_params(*P, k_bits, PK);
    fill_row_params(*P, v_bits, PV);
    const tq::AttnAppend app{k_new, v_new, kv_dtype == TQ_BF16, &PK, &PV};
    const tq::PagedArgs pa{block_table, positions, cache.n_pages, max_pages, shift};
    const tq_cache_view view = paged_as_view(cache);
    auto st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (k_bits) {
        case 2: e = tq::launch_attn128_paged<2>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, st, &app); break;
        case 3: e = tq::launch_attn128_paged<3>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, st, &app); break;
        default: e = tq::launch_attn128_paged<4>(v_bits, q, B, Hq, Hkv, view, max_ctx, out, workspace, g, A, pa, st, &app); break;
    }
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

size_t tq_attn_prefill_workspace_bytes(int B, int T, int Hq, int Hkv, int64_t cap, int d) {
    if (B < 0 || T < 1 || Hq <= 0 || Hkv <= 0 || cap < T || d != 128) return 0;
    return tq::attn_prefill_ws_bytes(B, Hkv, cap);
}

tq_status tq_attn_prefill(const tq_plan* plan, const void* q, int B, int T, int Hq, int Hkv, tq_cache_view cache,
                          const int32_t* q_start, int k_bits, int v_bits, float scale, float* out,
                          void* workspace, size_t workspace_bytes, tq_stream_t stream) {
    if (!plan || B < 0 || T < 1 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return TQ_ERR_INVALID_ARG;
    if (!valid_bits(k_bits) || !valid_bits(v_bits)) return TQ_ERR_UNSUPPORTED;
    const tq::Plan* P = reinterpret_cast<const tq::Plan*>(plan);
    const int G = Hq / Hkv;
    if (P->d != 128 || (G != 1 && G != 2 && G != 4 && G != 8)) return TQ_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return TQ_ERR_INVALID_ARG;
    if (cache.cap < T) return TQ_ERR_RANGE;
    if (B == 0) return TQ_OK;
    // grid limits: (sequence, KV head) pairs and 128-row query tiles per pair
    if ((int64_t)B * Hkv > 65535 || (int64_t)B * T * Hq > INT32_MAX || (int64_t)T * G > 65535LL * 128)
        return TQ_ERR_UNSUPPORTED;
    if (!q || !out || !q_start || !cache.k_packed || !cache.k_norm || !cache.v_packed || !cache.v_norm)
        return TQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned4(q_start) || !aligned16(cache.k_packed) ||
        !aligned16(cache.v_packed) || !aligned4(cache.k_norm) || !aligned4(cache.v_norm))
        return TQ_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < tq::attn_prefill_ws_bytes(B, Hkv, cache.cap)) return TQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TQ_ERR_ALIGNMENT;
    if (!device_accessible(q) || !device_accessible(out) || !device_accessible(q_start) ||
        !device_accessible(workspace) || !device_accessible(cache.k_packed) || !device_accessible(cache.v_packed) ||
        !device_accessible(cache.k_norm) || !device_accessible(cache.v_norm))
        return TQ_ERR_INVALID_ARG;
    tq::AttnParams A;
    tq::fill_attn_params(*P, k_bits, v_bits, scale, 0.0f, A);
    auto st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (k_bits) {
        case 2: e = tq::launch_attn_prefill<2>(v_bits, q, B, T, Hq, Hkv, q_start, cache, out, workspace, A, st); break;
        case 3: e = tq::launch_attn_prefill<3>(v_bits, q, B, T, Hq, Hkv, q_start, cache, out, workspace, A, st); break;
        default: e = tq::launch_attn_prefill<4>(v_bits, q, B, T, Hq, Hkv, q_start, cache, out, workspace, A, st); break;
    }
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID_ARG: return "invalid argument";
        case TQ_ERR_UNSUPPORTED: return "unsupported head dimension, bit width or dtype";
        case TQ_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
        case TQ_ERR_RANGE: return "position or context length outside the cache";
        case TQ_ERR_WORKSPACE: return "workspace missing or too small";
        case TQ_ERR_CUDA: return "CUDA runtime error";
        case TQ_ERR_NOMEM: return "host allocation failed";
    }
    return "unknown status";
}

int tq_last_cuda_error(void) { return g_last_cuda_error; }

tq_status tq_device_status(int reset, int* status_out) {
    if (!status_out) return TQ_ERR_INVALID_ARG;
    cudaError_t e = tq::read_device_status(reset, status_out);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // extern "C"
