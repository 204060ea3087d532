"""Pins of the oracle's format variants ("CITATIONS", Two-sided Rademacher
signs in WHT; N(0, 1/d) codebook replacement) against things other than the
oracle: scipy's Sylvester Hadamard matrix, the published splitmix64 generator
(an independent counter-based implementation), Max's 1960 table of the
Gaussian Lloyd-Max quantiser, closed forms, and scipy quadrature of the
Gaussian density.  CPU only.
"""
import math

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import scipy.stats

from conftest import read_golden
from kv_cache_vector_gb300 import synth
from oracle import oracle as O

# ------------------------------------------------------- two-sided signs


@pytest.mark.parametrize("seed", [0, 42, 7])
def test_signs2_are_the_next_d_outputs(seed):
    """s2 is the top bit of outputs d .. 2d-1 of the seed's splitmix64 stream,
    checked against an independent counter-based implementation."""
    for d in (64, 128, 256):
        r = synth.splitmix64_at(seed, np.arange(d, 2 * d))
        want = np.where((r >> np.uint64(63)) == 1, -1, 1).astype(np.int8)
        assert np.array_equal(O.signs2(seed, d), want)


def _explicit(s1, s2, d):
    H = scipy.linalg.hadamard(d).astype(np.float64)
    return np.diag(s2.astype(np.float64)) @ H @ np.diag(s1.astype(np.float64)) / math.sqrt(d)


@pytest.mark.parametrize("d", [8, 64, 128, 256])
def test_two_sided_rotation_is_s2_h_s1(d):
    """rotate(s1, x, s2) = S2 H S1 x / sqrt(d) and unrotate is its transpose,
    against scipy's Hadamard matrix; orthonormal, preserves dot products."""
    rng = np.random.default_rng(d)
    s1, s2 = O.signs(3, d), O.signs2(3, d)
    R = _explicit(s1, s2, d)
    x = rng.standard_normal((6, d))
    y = O.rotate(s1, x, s2)
    assert np.allclose(y, x @ R.T, atol=1e-13)
    assert np.allclose(O.unrotate(s1, y, s2), x, atol=1e-13)
    assert np.allclose(O.unrotate(s1, y, s2), y @ R, atol=1e-13)
    assert np.allclose(R @ R.T, np.eye(d), atol=1e-13)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    assert np.dot(O.rotate(s1, q, s2), O.rotate(s1, k, s2)) == pytest.approx(np.dot(q, k), abs=1e-12)


def test_two_sided_with_all_plus_s2_is_one_sided():
    d = 128
    rng = np.random.default_rng(1)
    s1 = O.signs(42, d)
    x = rng.standard_normal((4, d))
    ones = np.ones(d, np.int8)
    assert np.array_equal(O.rotate(s1, x, ones), O.rotate(s1, x))
    assert np.array_equal(O.unrotate(s1, x, ones), O.unrotate(s1, x))


@pytest.mark.parametrize("kind", ["sphere", "gauss"])
def test_two_sided_encode_decode_follow_the_explicit_matrix(kind):
    """Encode buckets u = (S2 H S1 x / sqrt d) / ||x|| and decode returns
    n S1 H S2 c / sqrt(d), with the rotation taken as an explicit matrix."""
    d, bits = 128, 3
    s1, s2 = O.signs(9, d), O.signs2(9, d)
    R = _explicit(s1, s2, d)
    x = synth.normal_rows(4, 20, d).double().numpy()
    packed, norms = O.encode(s1, bits, x, s2=s2, kind=kind)
    cen, bnd = O.codebook_f32(d, bits, kind)
    u = (x @ R.T) / np.linalg.norm(x, axis=1, keepdims=True)
    idx = np.searchsorted(bnd, u.astype(np.float32), side="right")
    assert np.array_equal(O.unpack(packed, d, bits), idx.astype(np.uint8))
    xh = O.decode(s1, bits, packed, norms, s2=s2, kind=kind)
    want = norms.astype(np.float64)[:, None] * (cen[idx].astype(np.float64) @ R)
    assert np.allclose(xh, want, atol=1e-12)


# ------------------------------------------------------ Gaussian codebook


def _ulp_of_printed(v: str) -> float:
    """One unit in the last digit of a printed table value."""
    return 10.0 ** -(len(v.split(".")[1]) if "." in v else 0)


def test_gauss_codebook_matches_max_table():
    """sqrt(d) times the N(0, 1/d) codebook is Max's unit-variance quantiser
    (the golden fixture cites the table), for d = 1 and d = 128, to one unit
    in the last printed digit (the table has four significant figures)."""
    for d in (1, 128):
        for row in read_golden("gaussian_lloyd_max.txt"):
            L = int(row[0])
            bits = L.bit_length() - 1
            levels = row[1].split()
            thr = [] if row[2] == "-" else row[2].split()
            c, b, _ = O.codebook(d, bits, "gauss")
            for k, v in enumerate(levels):
                assert abs(c[L // 2 + k] * math.sqrt(d) - float(v)) <= _ulp_of_printed(v), (d, L, k)
                assert abs(-c[L // 2 - 1 - k] * math.sqrt(d) - float(v)) <= _ulp_of_printed(v), (d, L, k)
            for k, v in enumerate(thr):
                assert abs(b[L // 2 + k] * math.sqrt(d) - float(v)) <= _ulp_of_printed(v), (d, L, k)
            mse = O.codebook_mse(d, bits, c, b, "gauss") * d
            assert mse == pytest.approx(float(row[3]), rel=1e-3)


def test_gauss_codebook_one_bit_closed_form():
    """One bit: levels +-sigma sqrt(2/pi), threshold 0, MSE sigma^2 (1 - 2/pi)."""
    for d in (1, 64, 128):
        sg = 1 / math.sqrt(d)
        c, b, _ = O.codebook(d, 1, "gauss")
        assert c[1] == pytest.approx(sg * math.sqrt(2 / math.pi), rel=1e-12)
        assert c[0] == pytest.approx(-sg * math.sqrt(2 / math.pi), rel=1e-12)
        assert b[0] == pytest.approx(0.0, abs=1e-15)
        assert O.codebook_mse(d, 1, c, b, "gauss") == pytest.approx(sg * sg * (1 - 2 / math.pi), rel=1e-12)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_gauss_codebook_is_a_lloyd_fixed_point(bits):
    """Each centroid is the conditional mean of its cell and each boundary the
    midpoint of its neighbours, with the means taken by scipy quadrature of
    the N(0, 1/d) density; the codebook scales as 1/sqrt(d)."""
    d = 128
    sg = 1 / math.sqrt(d)
    c, b, _ = O.codebook(d, bits, "gauss")
    assert np.allclose(b, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    edges = np.concatenate([[-np.inf], b, [np.inf]])
    pdf = scipy.stats.norm(0, sg).pdf
    for i in range(len(c)):
        lo, hi = edges[i], edges[i + 1]
        m0 = scipy.integrate.quad(pdf, lo, hi, epsabs=1e-15, epsrel=1e-13)[0]
        m1 = scipy.integrate.quad(lambda x: x * pdf(x), lo, hi, epsabs=1e-15, epsrel=1e-13)[0]
        assert c[i] == pytest.approx(m1 / m0, rel=1e-9, abs=1e-12)
    c1, _, _ = O.codebook(1, bits, "gauss")
    assert np.allclose(c * math.sqrt(d), c1, rtol=1e-11, atol=1e-13)


def test_gauss_mse_matches_quadrature():
    d, bits = 128, 3
    sg = 1 / math.sqrt(d)
    c, b, _ = O.codebook(d, bits, "gauss")
    edges = np.concatenate([[-np.inf], b, [np.inf]])
    pdf = scipy.stats.norm(0, sg).pdf
    want = sum(scipy.integrate.quad(lambda x, ci=ci: (x - ci) ** 2 * pdf(x), edges[i], edges[i + 1],
                                    epsabs=1e-16, epsrel=1e-12)[0] for i, ci in enumerate(c))
    assert O.codebook_mse(d, bits, c, b, "gauss") == pytest.approx(want, rel=1e-9)


def test_gauss_and_sphere_codebooks_differ_at_head_dims():
    """The two codebooks are distinct formats at d = 128 (the Gaussian one is
    the sphere's large-d limit): their fp32 boundaries differ."""
    for bits in (2, 3, 4):
        _, bs = O.codebook_f32(128, bits, "sphere")
        _, bg = O.codebook_f32(128, bits, "gauss")
        assert not np.array_equal(bs, bg)
        assert np.allclose(bs, bg, rtol=0.05)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_gauss_codebook_is_exactly_symmetric(bits):
    """The N(0, 1/d) density is symmetric, so the quantiser is: c[L-1-i] =
    -c[i] and the middle boundary is exactly 0 (a zero row buckets there)."""
    c, b, _ = O.codebook(128, bits, "gauss")
    L = 1 << bits
    assert np.array_equal(c[::-1], -c)
    assert b[L // 2 - 1] == 0.0
    assert np.array_equal(b[::-1], -b)
