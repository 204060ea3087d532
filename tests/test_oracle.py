"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: a
library routine for a special case (scipy's Sylvester Hadamard matrix, numpy's
bit packing and binary search, mpmath quadrature), a closed form, a textbook
table, a published generator output, an invariant, or a figure the pages print.
CPU only.
"""
import math

import mpmath
import numpy as np
import pytest
import scipy.linalg
import scipy.special

from conftest import read_golden
from kv_cache_vector_gb300 import synth
from oracle import oracle as O

# --------------------------------------------------------------- generator


def test_splitmix64_reference_vector():
    """Published splitmix64 outputs for state 0 (fixture cites the source)."""
    want = [int(r[0], 16) for r in read_golden("splitmix64_seed0.txt")]
    got = [int(v) for v in O.splitmix64_stream(0, len(want))]
    assert got == want


@pytest.mark.parametrize("seed", [0, 42, 12345])
def test_signs_follow_generator_definition(seed):
    """s_i = -1 iff the top bit of the i-th output is set; checked against an
    independent (numpy, counter-based) implementation of the same generator."""
    d = 256
    s = O.signs(seed, d)
    r = synth.splitmix64_at(seed, np.arange(d))
    want = np.where((r >> np.uint64(63)) == 1, -1, 1).astype(np.int8)
    assert np.array_equal(s, want)
    assert set(np.unique(s)) <= {-1, 1}
    # the first 128 signs of d = 256 are the signs of d = 128
    assert np.array_equal(O.signs(seed, 128), s[:128])


def test_signs_balanced():
    s = np.concatenate([O.signs(seed, 256) for seed in range(64)]).astype(np.float64)
    assert abs(s.mean()) < 4.0 / math.sqrt(s.size)   # 4 sigma of a fair coin


# ---------------------------------------------------------------- rotation


@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128, 256])
def test_fwht_is_sylvester_hadamard(d):
    """Butterfly == scipy.linalg.hadamard (Sylvester construction) matmul."""
    rng = np.random.default_rng(d)
    v = rng.standard_normal((5, d))
    H = scipy.linalg.hadamard(d).astype(np.float64)
    assert np.allclose(O.fwht(v), v @ H.T, rtol=0, atol=1e-12 * d)


@pytest.mark.parametrize("d", [8, 64, 128, 256])
def test_rotation_matches_matrix_and_is_orthonormal(d):
    s = O.signs(42, d)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    R = H @ np.diag(s.astype(np.float64)) / math.sqrt(d)      # y = H D x / sqrt(d)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((9, d))
    y = O.rotate(s, x)
    assert np.allclose(y, x @ R.T, atol=1e-12)
    # R R^T = I  (Foundry spec, Testing Strategy 2)
    Rb = O.rotate(s, np.eye(d))          # rows: R e_j = column j of R
    assert np.allclose(Rb @ Rb.T, np.eye(d), atol=1e-12)
    # norm preserved (kvcompress, Required invariants)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    # inverse: D H y / sqrt(d) returns x (Foundry spec, Hadamard Transform Detail)
    assert np.allclose(O.unrotate(s, y), x, atol=1e-12)
    # dot products preserved: (Rq).(Rk) = q.k (Foundry spec, fused dequant-dot)
    assert np.allclose((y[:4] * y[4:8]).sum(1), (x[:4] * x[4:8]).sum(1), atol=1e-11)
    # a basis vector spreads evenly: every |y_i| = 1/sqrt(d)
    assert np.allclose(np.abs(Rb), 1.0 / math.sqrt(d), atol=1e-14)


def test_rotation_applies_signs_before_hadamard():
    """D first (Foundry spec As-Built Note 1): a constant vector maps to the
    Hadamard transform of the sign vector, not to a single spike."""
    d = 64
    s = O.signs(42, d)
    y = O.rotate(s, np.ones((1, d)))[0]
    H = scipy.linalg.hadamard(d)
    assert np.allclose(y, H @ s.astype(np.float64) / math.sqrt(d), atol=1e-12)


# ---------------------------------------------------------------- codebook


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_d3_is_uniform_quantiser(bits):
    """d = 3: the coordinate density (1-x^2)^0 is uniform on [-1, 1], whose
    Lloyd-Max quantiser is the uniform one (closed form)."""
    L = 1 << bits
    c, b, _ = O.codebook(3, bits)
    assert np.allclose(c, -1 + (2 * np.arange(L) + 1) / L, atol=1e-13)
    assert np.allclose(b, -1 + 2 * np.arange(1, L) / L, atol=1e-13)
    mse = O.codebook_mse(3, bits, c, b)
    assert mse == pytest.approx(1.0 / (3 * L * L), rel=1e-10)


@pytest.mark.parametrize("d", [3, 4, 8, 64, 128, 256, 1000])
def test_codebook_one_bit_closed_form(d):
    """One bit: the centroid is E[X | X > 0] = Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2))
    for one coordinate of a uniform unit vector in R^d."""
    c, b, _ = O.codebook(d, 1)
    want = math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
    assert c[1] == pytest.approx(want, rel=1e-12)
    assert c[0] == -c[1] and b[0] == 0.0


def _mp_cell_centroid(d, a, b):
    a_ = (d - 3) / mpmath.mpf(2)
    f = lambda x: (1 - x * x) ** a_
    num = mpmath.quad(lambda x: x * f(x), [a, b])
    den = mpmath.quad(f, [a, b])
    return num / den


@pytest.mark.parametrize("d,bits", [(5, 4), (16, 3), (128, 2), (128, 3), (128, 4), (256, 4)])
def test_codebook_fixed_point_conditions(d, bits):
    """Lloyd-Max conditions, checked with 30-digit mpmath quadrature:
    every centroid is the conditional mean of its cell, every boundary the
    midpoint of its neighbours; codebook symmetric and ascending."""
    mpmath.mp.dps = 30
    c, b, _ = O.codebook(d, bits)
    L = 1 << bits
    assert np.all(np.diff(c) > 0) and np.all(np.diff(b) > 0)
    assert np.array_equal(c, -c[::-1]) and np.array_equal(b, -b[::-1])
    assert np.allclose(b, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    edges = [-1.0] + list(b) + [1.0]
    scale = 1.0 / math.sqrt(d)
    for k in range(L // 2, L):          # positive half (symmetry checked above)
        want = float(_mp_cell_centroid(d, mpmath.mpf(edges[k]), mpmath.mpf(edges[k + 1])))
        assert abs(c[k] - want) < 1e-12 * scale, (k, c[k], want)


def test_codebook_gaussian_limit(golden):
    """sqrt(d) * codebook -> Gaussian Lloyd-Max quantiser (Max 1960) as d grows."""
    d = 65536
    for row in golden("gaussian_lloyd_max.txt"):
        L = int(row[0])
        bits = L.bit_length() - 1
        levels = [float(v) for v in row[1].split()]
        thr = [] if row[2] == "-" else [float(v) for v in row[2].split()]
        c, b, _ = O.codebook(d, bits)
        got_c = c[L // 2:] * math.sqrt(d)
        got_b = b[L // 2:] * math.sqrt(d)
        assert np.allclose(got_c, levels, atol=1.5e-3), (L, got_c, levels)
        assert np.allclose(got_b, thr, atol=1.5e-3), (L, got_b, thr)
        mse = O.codebook_mse(d, bits, c, b) * d
        assert mse == pytest.approx(float(row[3]), rel=2e-3)


def test_density_mass_closed_forms():
    # d = 3 uniform; d = 5: density (3/4)(1 - x^2), CDF (3/4)(x - x^3/3) + 1/2
    assert O.density_mass(3, -0.3, 0.5) == pytest.approx(0.4, abs=1e-14)
    F = lambda x: 0.75 * (x - x ** 3 / 3) + 0.5
    assert O.density_mass(5, -0.2, 0.7) == pytest.approx(F(0.7) - F(-0.2), abs=1e-14)
    for d in (8, 128, 256):
        assert O.density_mass(d, -1.0, 1.0) == pytest.approx(1.0, abs=1e-13)
        assert O.density_mass(d, -1.0, 0.0) == pytest.approx(0.5, abs=1e-13)
    # d = 128 against scipy's regularised incomplete beta: X^2 ~ Beta(1/2, (d-1)/2)
    d, t = 128, 0.05
    want = scipy.special.betainc(0.5, (d - 1) / 2, t * t)
    assert O.density_mass(128, -t, t) == pytest.approx(want, abs=1e-13)


@pytest.mark.parametrize("d", [8, 64, 128, 256])
def test_codebook_mse_strictly_decreasing(d):
    """Error falls as resolution grows (kvcompress, Required invariants)."""
    mses = [O.codebook_mse(d, b, *O.codebook(d, b)[:2]) for b in (1, 2, 3, 4)]
    assert all(m1 > m2 for m1, m2 in zip(mses, mses[1:]))


# -------------------------------------------------------------- quantiser


@pytest.mark.parametrize("d,bits", [(128, 2), (128, 3), (128, 4), (256, 4), (16, 3)])
def test_bucket_is_binary_search_and_nearest_level(d, bits):
    """idx(u) == numpy binary search (side='right') over the fp32 boundaries,
    and == the nearest fp32 centroid away from the boundaries."""
    cf, bf = O.codebook_f32(d, bits)
    rng = np.random.default_rng(bits)
    u = np.concatenate([rng.uniform(-1, 1, 2000), rng.normal(0, 1 / math.sqrt(d), 4000),
                        bf, np.nextafter(bf, np.float32(-2)), [0.0, -0.0, 1.0, -1.0]]).astype(np.float32)
    got = np.array([O.bucket(float(v), bits, bf) for v in u])
    assert np.array_equal(got, np.searchsorted(bf, u, side="right"))
    away = np.min(np.abs(u[:, None].astype(np.float64) - bf[None, :].astype(np.float64)), axis=1) > 1e-6
    nearest = np.argmin(np.abs(u[:, None].astype(np.float64) - cf[None, :].astype(np.float64)), axis=1)
    assert np.array_equal(got[away], nearest[away])


def test_bucket_ties_go_up():
    cf, bf = O.codebook_f32(128, 4)
    for j, bj in enumerate(bf):
        assert O.bucket(float(bj), 4, bf) == j + 1
    assert O.bucket(0.0, 4, bf) == 8 and O.bucket(-0.0, 4, bf) == 8


# ---------------------------------------------------------------- packing


def test_pack_worked_examples(golden):
    for row in golden("pack_examples.txt"):
        bits = int(row[0])
        idx = np.array([int(v) for v in row[1].split()], np.uint8)
        want = bytes.fromhex(row[2].replace(" ", ""))
        assert O.pack(idx, bits).tobytes() == want
        assert np.array_equal(O.unpack(np.frombuffer(want, np.uint8), len(idx), bits), idx)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("d", [8, 16, 64, 128, 256])
def test_pack_matches_numpy_packbits_and_roundtrips(bits, d):
    """Round trip over every level value (Foundry spec, Testing Strategy 8) and
    agreement with numpy.packbits(bitorder='little')."""
    L = 1 << bits
    rng = np.random.default_rng(d * bits)
    idx = np.stack([np.arange(d) % L, rng.integers(0, L, d), np.full(d, L - 1)]).astype(np.uint8)
    p = O.pack(idx, bits)
    assert p.shape == (3, d * bits // 8)
    bitsarr = ((idx[..., None] >> np.arange(bits)) & 1).astype(np.uint8).reshape(3, -1)
    assert np.array_equal(p, np.packbits(bitsarr, axis=1, bitorder="little"))
    assert np.array_equal(O.unpack(p, d, bits), idx)


# ---------------------------------------------------------- encode/decode


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_zero_row(bits):
    d = 128
    s = O.signs(42, d)
    packed, norms = O.encode(s, bits, np.zeros((2, d)))
    assert np.all(norms == 0)
    assert np.all(O.unpack(packed, d, bits) == (1 << (bits - 1)))
    assert np.all(O.decode(s, bits, packed, norms) == 0.0)


def test_encode_power_of_two_scaling():
    """x and 2^k x give identical indices, and norms exactly 2^k apart."""
    d, bits = 128, 4
    s = O.signs(42, d)
    x = synth.normal_rows(3, 64, d).double().numpy()
    p0, n0 = O.encode(s, bits, x)
    for k in (-8, 5):
        p1, n1 = O.encode(s, bits, x * 2.0 ** k)
        assert np.array_equal(p0, p1)
        assert np.array_equal(n1, n0 * np.float32(2.0 ** k))


def test_encode_deterministic_and_seed_dependent():
    """Same seed -> identical bytes (Foundry Testing Strategy 5; kvcompress
    Required invariants); another seed -> other bytes."""
    d, bits = 128, 4
    x = synth.normal_rows(5, 32, d).double().numpy()
    a = O.encode(O.signs(42, d), bits, x)[0]
    b = O.encode(O.signs(42, d), bits, x)[0]
    c = O.encode(O.signs(43, d), bits, x)[0]
    assert np.array_equal(a, b) and not np.array_equal(a, c)


@pytest.mark.parametrize("bits", [2, 4])
def test_encode_u_and_decode_match_explicit_matrices(bits):
    d = 64
    s = O.signs(9, d)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    x = synth.normal_rows(11, 16, d).double().numpy()
    packed, norms, u = O.encode(s, bits, x, want_u=True)
    n = np.linalg.norm(x, axis=1, keepdims=True)
    assert np.allclose(u, (x * s) @ H.T / math.sqrt(d) / n, atol=1e-13)
    assert np.allclose(norms, n[:, 0].astype(np.float32), rtol=0, atol=0)
    cf, bf = O.codebook_f32(d, bits)
    idx = np.searchsorted(bf, u.astype(np.float32), side="right")
    assert np.array_equal(O.unpack(packed, d, bits), idx)
    xhat = O.decode(s, bits, packed, norms)
    want = (cf[idx].astype(np.float64) @ H.T) * s / math.sqrt(d) * norms[:, None].astype(np.float64)
    assert np.allclose(xhat, want, atol=1e-12)


@pytest.mark.parametrize("d", [128, 256])
def test_roundtrip_cosine_contract(d, golden):
    """Random-direction unit rows: per-row cosine >= 0.88 (4-bit) and >= 0.85
    (3-bit) (TurboQuantEngine spec 2.1); the mean matches sqrt(1 - d*MSE) of the
    codebook (the centroid condition makes x.x_hat = |x_hat|^2); error falls
    strictly with the bit width."""
    gate = {k: float(v) for k, v in golden("quality_contract.txt")}
    s = O.signs(42, d)
    x = synth.unit_rows(21, 512, d).double().numpy()
    mean_err = []
    for bits in (1, 2, 3, 4):
        p, nrm = O.encode(s, bits, x)
        xh = O.decode(s, bits, p, nrm)
        cos = (x * xh).sum(1) / np.linalg.norm(x, axis=1) / np.linalg.norm(xh, axis=1)
        if bits == 4:
            assert cos.min() >= gate["roundtrip_cos_min_4bit"]
        if bits == 3:
            assert cos.min() >= gate["roundtrip_cos_min_3bit"]
        mse = O.codebook_mse(d, bits, *O.codebook(d, bits)[:2]) * d
        assert cos.mean() == pytest.approx(math.sqrt(1 - mse), abs=3e-3)
        mean_err.append(((x - xh) ** 2).sum(1).mean())
    assert all(a > b for a, b in zip(mean_err, mean_err[1:]))


# ---------------------------------------------------------------- attention


def _cache(seed, B, Hkv, cap, d, kb, vb, s, kgen=None):
    nrows = B * Hkv * cap
    k = synth.normal_rows(seed, nrows, d, stream=1).double().numpy() if kgen is None else kgen
    v = synth.normal_rows(seed, nrows, d, stream=2).double().numpy()
    kp, kn = O.encode(s, kb, k)
    vp, vn = O.encode(s, vb, v)
    return (kp.reshape(B, Hkv, cap, -1), kn.reshape(B, Hkv, cap),
            vp.reshape(B, Hkv, cap, -1), vn.reshape(B, Hkv, cap))


def test_attention_brute_force_tiny():
    """Against scipy softmax + numpy matmuls over the oracle's decoded rows."""
    B, Hq, Hkv, d, cap, ctx, kb, vb = 2, 4, 2, 16, 7, 5, 4, 3
    s = O.signs(1, d)
    kp, kn, vp, vn = _cache(1, B, Hkv, cap, d, kb, vb, s)
    q = synth.normal_rows(2, B * Hq, d).double().numpy().reshape(B, Hq, d)
    out = O.attention(s, q, kp, kn, vp, vn, kb, vb, ctx, 0.25)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            K = O.decode(s, kb, kp[b, g, :ctx], kn[b, g, :ctx])
            V = O.decode(s, vb, vp[b, g, :ctx], vn[b, g, :ctx])
            p = scipy.special.softmax(0.25 * K @ q[b, h])
            assert np.allclose(out[b, h], p @ V, atol=1e-13)


def test_attention_special_cases():
    B, Hq, Hkv, d, cap, kb, vb = 1, 4, 2, 32, 9, 4, 2
    s = O.signs(3, d)
    kp, kn, vp, vn = _cache(4, B, Hkv, cap, d, kb, vb, s)
    q = synth.normal_rows(5, B * Hq, d).double().numpy().reshape(B, Hq, d)
    V = [O.decode(s, vb, vp[0, g], vn[0, g]) for g in range(Hkv)]
    # one position: the output is that V row exactly
    o1 = O.attention(s, q, kp, kn, vp, vn, kb, vb, 1, 0.3)
    for h in range(Hq):
        assert np.allclose(o1[0, h], V[h // 2][0], atol=1e-14)
    # q = 0 or scale = 0: uniform weights -> mean of the kv head's V rows (GQA:
    # heads 0,1 read kv head 0 and heads 2,3 read kv head 1)
    for qq, sc in ((np.zeros_like(q), 0.3), (q, 0.0)):
        o = O.attention(s, qq, kp, kn, vp, vn, kb, vb, 6, sc)
        for h in range(Hq):
            assert np.allclose(o[0, h], V[h // 2][:6].mean(0), atol=1e-13)
        assert not np.allclose(o[0, 0], o[0, 2])
    # identical keys -> uniform weights -> mean
    kp2 = np.broadcast_to(kp[:, :, :1], kp.shape).copy()
    kn2 = np.broadcast_to(kn[:, :, :1], kn.shape).copy()
    o = O.attention(s, q, kp2, kn2, vp, vn, kb, vb, 9, 0.3)
    for h in range(Hq):
        assert np.allclose(o[0, h], V[h // 2].mean(0), atol=1e-13)


def test_attention_rotated_domain_identity():
    """(Rq).(Rk) = q.k: scores and values taken in the rotated domain straight
    from the centroids, then one inverse rotation of the output, agree with the
    plain (unrotated) oracle (Foundry spec, Optimization: Fused dequant-dot)."""
    B, Hq, Hkv, d, cap, ctx, kb, vb = 1, 8, 2, 128, 40, 37, 4, 3
    s = O.signs(42, d)
    kp, kn, vp, vn = _cache(6, B, Hkv, cap, d, kb, vb, s)
    q = synth.normal_rows(7, B * Hq, d).double().numpy().reshape(B, Hq, d)
    out = O.attention(s, q, kp, kn, vp, vn, kb, vb, ctx, 1 / math.sqrt(d))
    kc, _ = O.codebook_f32(d, kb)
    vc, _ = O.codebook_f32(d, vb)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        qt = O.rotate(s, q[0, h][None])[0]
        Kc = kc[O.unpack(kp[0, g, :ctx], d, kb)].astype(np.float64) * kn[0, g, :ctx, None]
        Vc = vc[O.unpack(vp[0, g, :ctx], d, vb)].astype(np.float64) * vn[0, g, :ctx, None]
        p = scipy.special.softmax(Kc @ qt / math.sqrt(d))
        o = O.unrotate(s, (p @ Vc)[None])[0]
        assert np.allclose(out[0, h], o, atol=1e-12)


def test_attention_sparse_v_limits():
    """threshold 0 == dense; threshold 1 keeps only the maximising row, whose
    weight is exp(0)/l (rows below the threshold stay in the denominator)."""
    B, Hq, Hkv, d, cap, ctx, kb, vb = 1, 2, 1, 16, 20, 20, 3, 2
    s = O.signs(8, d)
    kp, kn, vp, vn = _cache(9, B, Hkv, cap, d, kb, vb, s)
    q = 3 * synth.normal_rows(10, B * Hq, d).double().numpy().reshape(B, Hq, d)
    dense = O.attention(s, q, kp, kn, vp, vn, kb, vb, ctx, 0.5)
    zero, kept0 = O.attention(s, q, kp, kn, vp, vn, kb, vb, ctx, 0.5, 0.0, want_kept=True)
    assert np.array_equal(dense, zero) and np.all(kept0 == ctx)
    one, kept1 = O.attention(s, q, kp, kn, vp, vn, kb, vb, ctx, 0.5, 1.0, want_kept=True)
    K = O.decode(s, kb, kp[0, 0, :ctx], kn[0, 0, :ctx])
    V = O.decode(s, vb, vp[0, 0, :ctx], vn[0, 0, :ctx])
    for h in range(Hq):
        sig = 0.5 * K @ q[0, h]
        t = int(np.argmax(sig))
        l = np.exp(sig - sig.max()).sum()
        assert kept1[0, h] == 1
        assert np.allclose(one[0, h], V[t] / l, atol=1e-13)


@pytest.mark.parametrize("kb,vb,key", [(4, 2, "attn_cos_k4v2_gaussian"),
                                       (4, 3, "attn_cos_k4v3_gaussian"),
                                       (4, 4, "attn_cos_k4v4_gaussian")])
def test_attention_quality_matches_pages(kb, vb, key, golden):
    """Attention-output cosine, FP vs compressed, on Gaussian data: the pages'
    measured figures (~0.94 K4/V2, ~0.98 K4/V3, ~0.99 K4/V4), loosely."""
    want = {k: float(v) for k, v in golden("quality_contract.txt")}[key]
    B, Hq, Hkv, d, ctx = 1, 8, 2, 128, 256
    s = O.signs(42, d)
    k = synth.normal_rows(31, B * Hkv * ctx, d, stream=1).double().numpy()
    v = synth.normal_rows(31, B * Hkv * ctx, d, stream=2).double().numpy()
    kp, kn, vp, vn = _cache(31, B, Hkv, ctx, d, kb, vb, s, kgen=k)
    q = synth.normal_rows(32, B * Hq, d).double().numpy().reshape(B, Hq, d)
    out = O.attention(s, q, kp, kn, vp, vn, kb, vb, ctx, 1 / math.sqrt(d))
    K = k.reshape(Hkv, ctx, d)
    V = v.reshape(Hkv, ctx, d)
    cos = []
    for h in range(Hq):
        p = scipy.special.softmax(K[h // 4] @ q[0, h] / math.sqrt(d))
        ref = p @ V[h // 4]
        cos.append(ref @ out[0, h] / np.linalg.norm(ref) / np.linalg.norm(out[0, h]))
    assert np.mean(cos) == pytest.approx(want, abs=0.03)
