"""Pins of the oracle's QJL residual keys ("CITATIONS", Google TurboQuant
entry: an MSE-optimal quantiser followed by a 1-bit quantised JL transform of
the residual; "TurboQuant KV Cache Compression -- Spec", Why not QJL?).

The reading: b bits per coordinate are a (b - 1)-bit MSE index plus one sign of
the Gaussian projection S r of the rotated normalised residual r; gamma =
n ||r|| is stored beside the norm; decode adds sqrt(pi/2)/d * gamma * S^T sgn
to the MSE reconstruction in the rotated domain.  Pinned here against the
published splitmix64 generator (an independent counter-based implementation),
scipy's normal distribution, scipy's Sylvester Hadamard matrix, the already
pinned (b - 1)-bit codec, unbiasedness of the inner-product estimator in
expectation over seeds (the property the second stage exists for), and a scipy
softmax over decoded rows.  CPU only.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.special
import scipy.stats

from kv_cache_vector_gb300 import synth
from oracle import oracle as O

# ------------------------------------------------------------ the projection


@pytest.mark.parametrize("seed", [42, 7])
def test_matrix_is_standard_gaussian(seed):
    """The 128 x 128 entries pass a Kolmogorov-Smirnov test against N(0, 1),
    with mean, variance and lag-1 correlation inside four standard errors."""
    S = O.qjl_matrix(seed, 128)
    v = S.ravel()
    n = v.size
    assert scipy.stats.kstest(v, "norm").pvalue > 1e-3
    assert abs(v.mean()) < 4 / math.sqrt(n)
    assert abs(v.var() - 1.0) < 4 * math.sqrt(2.0 / n)
    assert abs(np.corrcoef(v[:-1], v[1:])[0, 1]) < 4 / math.sqrt(n)
    # rows are near orthogonal at rate 1/sqrt(d)
    G = S @ S.T / 128
    assert np.abs(np.diag(G) - 1).max() < 0.5
    assert np.abs(G - np.diag(np.diag(G))).max() < 6 / math.sqrt(128)


@pytest.mark.parametrize("d", [8, 128])
def test_matrix_uses_outputs_after_the_signs(d):
    """S_ij is Box-Muller on outputs 2d + 2k and 2d + 2k + 1 (k = i d + j) of
    the seed's splitmix64 stream, taken from an independent counter-based
    implementation of the published generator."""
    k = np.arange(d * d, dtype=np.int64)
    o1 = synth.splitmix64_at(42, 2 * d + 2 * k)
    o2 = synth.splitmix64_at(42, 2 * d + 2 * k + 1)
    u1 = (o1 >> np.uint64(11)).astype(np.float64) / 2.0 ** 53
    u2 = (o2 >> np.uint64(11)).astype(np.float64) / 2.0 ** 53
    want = (np.sqrt(-2 * np.log1p(-u1)) * np.cos(2 * np.pi * u2)).reshape(d, d)
    np.testing.assert_allclose(O.qjl_matrix(42, d), want, rtol=1e-13, atol=1e-13)
    assert not np.array_equal(O.qjl_matrix(42, d), O.qjl_matrix(43, d))


# ------------------------------------------------------------ the encoder


def _rows(n, d, seed):
    return np.random.default_rng(seed).standard_normal((n, d)) * np.random.default_rng(seed + 1).uniform(
        0.1, 20, (n, 1))


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_mse_stage_is_the_b_minus_1_bit_codec(bits):
    """The leading d(b-1)/8 bytes and the norm are the pinned (b - 1)-bit
    codec's encoding of the same rows."""
    d = 128
    s = O.signs(42, d)
    x = _rows(64, d, bits)
    S = O.qjl_matrix(42, d)
    p, n, g = O.encode_qjl(s, bits, x, S)
    pm, nm = O.encode(s, bits - 1, x)
    assert p.shape == (64, d * bits // 8)
    assert np.array_equal(p[:, :d * (bits - 1) // 8], pm)
    assert np.array_equal(n, nm)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_gamma_is_the_residual_norm(bits):
    """gamma = ||x - x_mse|| with x_mse the (b - 1)-bit codec's decode, taken
    in the original domain (the rotation is orthogonal)."""
    d = 128
    s = O.signs(42, d)
    x = _rows(64, d, 10 + bits)
    S = O.qjl_matrix(42, d)
    p, n, g = O.encode_qjl(s, bits, x, S)
    pm, nm = O.encode(s, bits - 1, x)
    xm = O.decode(s, bits - 1, pm, nm)
    np.testing.assert_allclose(g, np.linalg.norm(x - xm, axis=1), rtol=2e-6)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_signs_are_the_projection_signs(bits):
    """Sign bit k is set iff (S r)_k >= 0, with r = rotate(x)/n - c[idx]
    rebuilt in numpy from the explicit Hadamard matrix and the fp32 codebook."""
    d = 128
    s = O.signs(42, d)
    x = _rows(48, d, 20 + bits)
    S = O.qjl_matrix(42, d)
    p, n, g, proj = O.encode_qjl(s, bits, x, S, want_proj=True)
    ib = d * (bits - 1) // 8
    idx = O.unpack(p[:, :ib], d, bits - 1)
    sg = O.unpack(p[:, ib:], d, 1)
    R = scipy.linalg.hadamard(d) * s[None, :].astype(np.float64) / math.sqrt(d)
    u = (x @ R.T) / np.linalg.norm(x, axis=1, keepdims=True)
    cen, _ = O.codebook_f32(d, bits - 1)
    r = u - cen.astype(np.float64)[idx]
    want = r @ S.T
    np.testing.assert_allclose(proj, want, atol=1e-12)
    clear = np.abs(want) > 1e-9
    assert clear.mean() > 0.999
    assert np.array_equal(sg[clear], (want[clear] >= 0).astype(np.uint8))


def test_scaling_and_zero_rows():
    """x -> 2x leaves the bytes alone and doubles n and gamma exactly; a zero
    row has n = gamma = 0 and decodes to exact zeros."""
    d = 128
    s = O.signs(42, d)
    S = O.qjl_matrix(42, d)
    x = _rows(16, d, 31)
    p1, n1, g1 = O.encode_qjl(s, 3, x, S)
    p2, n2, g2 = O.encode_qjl(s, 3, 2 * x, S)
    assert np.array_equal(p1, p2) and np.array_equal(2 * n1, n2) and np.array_equal(2 * g1, g2)
    z = np.zeros((2, d))
    pz, nz, gz = O.encode_qjl(s, 3, z, S)
    assert np.all(nz == 0) and np.all(gz == 0)
    assert np.all(O.decode_qjl(s, 3, pz, nz, gz, S) == 0)


# ------------------------------------------------------------ the decoder


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("two_sided", [False, True])
def test_decode_against_explicit_matrices(bits, two_sided):
    """decode = R^T (n c[idx] + sqrt(pi/2)/d gamma S^T (2 sgn - 1)) with R the
    explicit rotation matrix, on d = 16."""
    d = 16
    s = O.signs(5, d)
    s2 = O.signs2(5, d) if two_sided else None
    S = O.qjl_matrix(5, d)
    x = _rows(40, d, 40 + bits)
    p, n, g = O.encode_qjl(s, bits, x, S, s2=s2)
    ib = d * (bits - 1) // 8
    idx = O.unpack(p[:, :ib], d, bits - 1)
    sg = O.unpack(p[:, ib:], d, 1).astype(np.float64) * 2 - 1
    cen, _ = O.codebook_f32(d, bits - 1)
    R = scipy.linalg.hadamard(d) * s[None, :].astype(np.float64) / math.sqrt(d)
    if two_sided:
        R = s2.astype(np.float64)[:, None] * R
    yr = n.astype(np.float64)[:, None] * cen.astype(np.float64)[idx] + \
        math.sqrt(math.pi / 2) / d * g.astype(np.float64)[:, None] * (sg @ S)
    np.testing.assert_allclose(O.decode_qjl(s, bits, p, n, g, S, s2=s2), yr @ R, atol=1e-12)


@pytest.mark.parametrize("bits", [2, 3])
def test_inner_products_are_unbiased_over_seeds(bits):
    """Averaged over 400 seeds (each a fresh rotation and projection), the QJL
    estimate of <y, x> has no bias beyond four standard errors, while the
    (b - 1)-bit MSE-only estimate shows its known shrinkage by many standard
    errors (the reason the pages give for the second stage)."""
    d = 128
    rng = np.random.default_rng(99)
    x = rng.standard_normal((4, d))
    y = x + 0.5 * rng.standard_normal((4, d))
    truth = np.sum(x * y, axis=1)
    est_q, est_m = [], []
    for seed in range(1000, 1400):
        s = O.signs(seed, d)
        S = O.qjl_matrix(seed, d)
        p, n, g = O.encode_qjl(s, bits, x, S)
        est_q.append(np.sum(O.decode_qjl(s, bits, p, n, g, S) * y, axis=1))
        pm, nm = O.encode(s, bits - 1, x)
        est_m.append(np.sum(O.decode(s, bits - 1, pm, nm) * y, axis=1))
    for est, unbiased in ((np.array(est_q), True), (np.array(est_m), False)):
        bias = est.mean(axis=0) - truth
        se = est.std(axis=0, ddof=1) / math.sqrt(est.shape[0])
        if unbiased:
            assert np.all(np.abs(bias) < 4 * se), (bias, se)
        else:
            assert np.all(np.abs(bias) > 10 * se), (bias, se)


def test_sign_projection_expectation():
    """The identity the estimator rests on: E[sign(s.r) s] = sqrt(2/pi) r/||r||
    for a standard Gaussian s; the 128 rows of 60 matrices give 7680 draws."""
    d = 128
    r = np.random.default_rng(3).standard_normal(d)
    acc = np.zeros(d)
    m = 0
    for seed in range(60):
        S = O.qjl_matrix(seed, d)
        acc += (np.sign(S @ r)[:, None] * S).sum(axis=0)
        m += d
    est = acc / m
    want = math.sqrt(2 / math.pi) * r / np.linalg.norm(r)
    # each coordinate's draw has variance at most 1
    assert np.abs(est - want).max() < 4.5 / math.sqrt(m)


# ------------------------------------------------------------ attention


def test_attention_with_qjl_keys():
    """Softmax attention over the QJL-decoded keys and the plain-decoded
    values, restated with scipy's softmax, with GQA (4 query heads per KV head)
    and a partly filled cache."""
    d, B, Hq, Hkv, cap, L, kb, vb = 16, 2, 8, 2, 24, 19, 3, 2
    rng = np.random.default_rng(5)
    s = O.signs(42, d)
    S = O.qjl_matrix(42, d)
    k = rng.standard_normal((B, Hkv, cap, d))
    v = rng.standard_normal((B, Hkv, cap, d))
    kp, kn, kg = O.encode_qjl(s, kb, k.reshape(-1, d), S)
    vp, vn = O.encode(s, vb, v.reshape(-1, d))
    q = rng.standard_normal((B, Hq, d))
    scale = 1 / math.sqrt(d)
    got = O.attention_qjl(s, q, kp.reshape(B, Hkv, cap, -1), kn.reshape(B, Hkv, cap), kg.reshape(B, Hkv, cap),
                          S, vp.reshape(B, Hkv, cap, -1), vn.reshape(B, Hkv, cap), kb, vb, L, scale)
    kh = O.decode_qjl(s, kb, kp, kn, kg, S).reshape(B, Hkv, cap, d)
    vh = O.decode(s, vb, vp, vn).reshape(B, Hkv, cap, d)
    for b in range(B):
        for h in range(Hq):
            gkv = h // (Hq // Hkv)
            p = scipy.special.softmax(scale * kh[b, gkv, :L] @ q[b, h])
            np.testing.assert_allclose(got[b, h], p @ vh[b, gkv, :L], atol=1e-12)
