"""GPU parity of the QJL residual keys ("CITATIONS", Google TurboQuant entry;
"TurboQuant KV Cache Compression -- Spec", Why not QJL?) against the oracle.

The projection S is an input of the method.  The library's generator is
checked against the oracle's; every other test hands both sides the oracle's
matrix rounded to fp32 (the oracle computing with those values in double), so
that the two differ only by the library's fp32 arithmetic.

Bars:
* the (b - 1)-bit indices: bit-exact except within 1e-6 of a boundary (the
  codec's own rule), norms to 1e-5 relative;
* sign bits: a flip only where the oracle's projection |(S r)_k| is within
  2e-4 ||r|| of zero (an fp32 chain of d products of a row of S, about
  sqrt(d) in norm, with r: below 1e-4 ||r|| even in the worst case), at most
  1e-3 of the signs; gamma to 1e-5 relative;
* decode within 1e-5 ||y|| / sqrt(d) per element (plus one bf16 unit);
* attention within 2e-3 absolute.
"""
import math

import numpy as np
import pytest
import torch

from kv_cache_vector_gb300 import abi, synth
from oracle import oracle as O
from parity import ATTN_ATOL, DECODE_REL, bf16_ulp, compare_encode

pytestmark = pytest.mark.gpu

SIGN_TOL = 2e-4
MAX_FLIP_FRACTION = 1e-3
GAMMA_RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kv_cache_vector_gb300 import build
    build.build()
    abi.lib()
    abi.tq_device_status(reset=True)


def _s32(seed, d):
    return np.ascontiguousarray(O.qjl_matrix(seed, d).astype(np.float32))


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("seed", [42, 7])
def test_matrix_matches_oracle(d, seed):
    """The device generator (splitmix64 + Box-Muller in double, rounded to
    fp32) against the oracle's double matrix: within one fp32 unit, nearly all
    identical after rounding."""
    got = abi.tq_qjl_matrix(abi.Plan(d, seed)).cpu().numpy().astype(np.float64)
    want = O.qjl_matrix(seed, d)
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - want) <= ulp)
    assert np.mean(got == want.astype(np.float32)) > 0.999


def _check_qjl_encode(s, bits, x64, S32, pk, nm, rn, s2=None, kind="sphere"):
    """Returns the flip fraction; asserts every bar above."""
    n, d = x64.shape
    ib = d * (bits - 1) // 8
    opk, onm, org, proj = O.encode_qjl(s, bits, x64, S32.astype(np.float64), s2=s2, kind=kind, want_proj=True)
    compare_encode(s, bits - 1, x64, np.ascontiguousarray(pk[:, :ib]), nm, s2=s2, kind=kind)
    same = np.all(pk[:, :ib] == opk[:, :ib], axis=1)
    gs = O.unpack(np.ascontiguousarray(pk[same, ib:]), d, 1)
    os_ = O.unpack(np.ascontiguousarray(opk[same, ib:]), d, 1)
    flips = gs != os_
    rnorm = np.where(onm[same] > 0, org[same].astype(np.float64) / np.maximum(onm[same], 1e-30), 0.0)
    if flips.any():
        margin = np.abs(proj[same]) / np.maximum(rnorm[:, None], 1e-30)
        assert margin[flips].max() <= SIGN_TOL, f"a sign flipped {margin[flips].max():.3g} ||r|| from zero"
    frac = float(flips.mean()) if flips.size else 0.0
    assert frac <= MAX_FLIP_FRACTION, f"{flips.sum()} sign flips"
    np.testing.assert_allclose(rn[same], org[same], rtol=GAMMA_RTOL, atol=0)
    return frac


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_encode_parity_ragged(d, bits, dtype):
    n = 333  # not a multiple of the 32 rows a block takes
    plan = abi.Plan(d, 42)
    S32 = _s32(42, d)
    x = synth.normal_rows(700 + d + bits, n, d, dtype)
    pk, nm, rn = abi.tq_encode_qjl(plan, bits, torch.from_numpy(S32).cuda(), x.cuda())
    torch.cuda.synchronize()
    _check_qjl_encode(O.signs(42, d), bits, x.double().numpy(), S32, pk.cpu().numpy(), nm.cpu().numpy(),
                      rn.cpu().numpy())


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_encode_rows_beyond_fp32_squares(d, dtype):
    """Rows of finite norm whose sum of squares leaves fp32's range (2^+-100
    scalings) beside unscaled ones: indices, signs, norms and gammas as the
    oracle's."""
    bits = 4
    plan = abi.Plan(d, 42)
    S32 = _s32(42, d)
    base = synth.normal_rows(4100 + d, 12, d).double()
    scale = torch.tensor([2.0 ** 100, 2.0 ** -100, 1.0] * 4, dtype=torch.float64)[:, None]
    x = (base * scale).to(dtype)
    pk, nm, rn = abi.tq_encode_qjl(plan, bits, torch.from_numpy(S32).cuda(), x.cuda())
    torch.cuda.synchronize()
    _check_qjl_encode(O.signs(42, d), bits, x.double().numpy(), S32, pk.cpu().numpy(), nm.cpu().numpy(),
                      rn.cpu().numpy())


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codec_parity_several_grid_passes(bits):
    """d = 128, 40,001 bf16 low-rank rows with outlier channels: more rows
    than one pass of the persistent grid takes (152 blocks of 12 warps x 16
    rows), with a ragged last group.  Encode against the oracle as above;
    decode of the library's own encoding against the oracle's decode of the
    same bytes."""
    d, n = 128, 40001
    plan = abi.Plan(d, 42)
    S32 = _s32(42, d)
    Sd = torch.from_numpy(S32).cuda()
    x = synth.lowrank_rows(1500 + bits, n, d)
    pk, nm, rn = abi.tq_encode_qjl(plan, bits, Sd, x.cuda())
    torch.cuda.synchronize()
    pk, nm, rn = pk.cpu().numpy(), nm.cpu().numpy(), rn.cpu().numpy()
    s = O.signs(42, d)
    _check_qjl_encode(s, bits, x.double().numpy(), S32, pk, nm, rn)
    y = abi.tq_decode_qjl(plan, bits, Sd, torch.from_numpy(pk).cuda(), torch.from_numpy(nm).cuda(),
                          torch.from_numpy(rn).cuda(), torch.float32)
    torch.cuda.synchronize()
    want = O.decode_qjl(s, bits, pk, nm, rn, S32.astype(np.float64))
    tol = DECODE_REL * np.linalg.norm(want, axis=1, keepdims=True) / math.sqrt(d)
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - want) <= tol)


@pytest.mark.parametrize("flags", [abi.PLAN_TWO_SIDED_SIGNS, abi.PLAN_GAUSSIAN_CODEBOOK | abi.PLAN_TWO_SIDED_SIGNS])
def test_encode_parity_format_variants(flags):
    d, bits = 128, 3
    plan = abi.Plan(d, 42, flags)
    S32 = _s32(42, d)
    x = synth.normal_rows(71, 200, d, torch.bfloat16)
    pk, nm, rn = abi.tq_encode_qjl(plan, bits, torch.from_numpy(S32).cuda(), x.cuda())
    torch.cuda.synchronize()
    kind = "gauss" if flags & abi.PLAN_GAUSSIAN_CODEBOOK else "sphere"
    _check_qjl_encode(O.signs(42, d), bits, x.double().numpy(), S32, pk.cpu().numpy(), nm.cpu().numpy(),
                      rn.cpu().numpy(), s2=O.signs2(42, d), kind=kind)


def test_encode_edge_rows_and_sizes():
    """Zero rows (n = gamma = 0), one-hot and constant rows, 2^k scalings; a
    single row; no rows."""
    d, bits = 128, 4
    plan = abi.Plan(d, 42)
    S32 = _s32(42, d)
    Sd = torch.from_numpy(S32).cuda()
    base = synth.normal_rows(98, 4, d).double()
    rows = [torch.zeros(d), torch.full((d,), 3.0), torch.eye(d)[5]]
    rows += [base[0] * 2.0 ** k for k in (-30, 0, 30)]
    x = torch.stack([r.float() for r in rows])
    pk, nm, rn = abi.tq_encode_qjl(plan, bits, Sd, x.cuda())
    torch.cuda.synchronize()
    pk, nm, rn = pk.cpu().numpy(), nm.cpu().numpy(), rn.cpu().numpy()
    _check_qjl_encode(O.signs(42, d), bits, x.double().numpy(), S32, pk, nm, rn)
    assert nm[0] == 0 and rn[0] == 0
    assert np.array_equal(pk[3], pk[4]) and np.array_equal(pk[4], pk[5])
    one = abi.tq_encode_qjl(plan, bits, Sd, x[3:4].cuda())
    assert np.array_equal(one[0].cpu().numpy()[0], pk[3])
    empty = abi.tq_encode_qjl(plan, bits, Sd, torch.empty(0, d, device="cuda"))
    assert empty[0].shape == (0, d * bits // 8)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_parity(d, bits, out_dtype):
    """Oracle-encoded rows and random codes (any bytes are a valid code) with
    random norms and gammas, 257 rows."""
    S32 = _s32(42, d)
    s = O.signs(42, d)
    x = synth.normal_rows(800 + d + bits, 129, d).double().numpy()
    pk, nm, rn = O.encode_qjl(s, bits, x, S32.astype(np.float64))
    rng = np.random.default_rng(900 + d + bits)
    pk = np.concatenate([pk, rng.integers(0, 256, (128, d * bits // 8), dtype=np.uint8)])
    nm = np.concatenate([nm, rng.uniform(0, 30, 128).astype(np.float32)])
    rn = np.concatenate([rn, rng.uniform(0, 10, 128).astype(np.float32)])
    y = abi.tq_decode_qjl(abi.Plan(d, 42), bits, torch.from_numpy(S32).cuda(), torch.from_numpy(pk).cuda(),
                          torch.from_numpy(nm).cuda(), torch.from_numpy(rn).cuda(), out_dtype)
    torch.cuda.synchronize()
    want = O.decode_qjl(s, bits, pk, nm, rn, S32.astype(np.float64))
    got = y.float().cpu().numpy().astype(np.float64)
    tol = DECODE_REL * np.linalg.norm(want, axis=1, keepdims=True) / math.sqrt(d)
    if out_dtype == torch.bfloat16:
        tol = tol + bf16_ulp(want)
    assert np.all(np.abs(got - want) <= tol), float((np.abs(got - want) / tol).max())


def _qjl_cache(seed, d, B, Hkv, cap, kb, vb, S32):
    s = O.signs(42, d)
    k = synth.normal_rows(seed, B * Hkv * cap, d).double().numpy()
    v = synth.normal_rows(seed + 1, B * Hkv * cap, d).double().numpy()
    kp, kn, kg = O.encode_qjl(s, kb, k, S32.astype(np.float64))
    vp, vn = O.encode(s, vb, v)
    shape = (B, Hkv, cap)
    return (kp.reshape(*shape, -1), kn.reshape(shape), kg.reshape(shape), vp.reshape(*shape, -1),
            vn.reshape(shape))


@pytest.mark.parametrize("d,B,Hq,Hkv,cap,ctx", [
    (128, 2, 32, 8, 1100, 1037),   # several splits and a ragged tail
    (128, 1, 8, 8, 64, 1),         # one position: the V row
    (128, 1, 16, 2, 900, 777),     # eight query heads per KV head
    (128, 3, 2, 1, 300, 211),      # six query rows: a part-filled block of the query kernel
    (64, 3, 16, 2, 700, 700),      # group of 8, the whole cache
    (32, 1, 4, 4, 300, 257),
])
@pytest.mark.parametrize("kb,vb", [(4, 3), (3, 2), (2, 4)])
def test_attention_parity(d, B, Hq, Hkv, cap, ctx, kb, vb):
    S32 = _s32(42, d)
    kp, kn, kg, vp, vn = _qjl_cache(1000 + d + kb, d, B, Hkv, cap, kb, vb, S32)
    q = synth.normal_rows(1100 + d, B * Hq, d, torch.bfloat16).reshape(B, Hq, d)
    scale = 1.0 / math.sqrt(d)
    want = O.attention_qjl(O.signs(42, d), q.double().numpy(), kp, kn, kg, S32.astype(np.float64), vp, vn, kb,
                           vb, ctx, scale)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    cache = abi.Cache(dev(kp), dev(kn), dev(vp), dev(vn), kb, vb)
    got = abi.tq_attn_decode_qjl(abi.Plan(d, 42), dev(S32), q.cuda(), cache, dev(kg), ctx, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status() == 0
    err = np.abs(got.cpu().numpy().astype(np.float64) - want)
    assert err.max() <= ATTN_ATOL, err.max()


def test_attention_two_sided_gaussian_plan():
    d, B, Hq, Hkv, cap, kb, vb = 128, 1, 16, 4, 600, 3, 3
    flags = abi.PLAN_GAUSSIAN_CODEBOOK | abi.PLAN_TWO_SIDED_SIGNS
    S32 = _s32(42, d)
    s, s2 = O.signs(42, d), O.signs2(42, d)
    k = synth.normal_rows(1201, B * Hkv * cap, d).double().numpy()
    v = synth.normal_rows(1202, B * Hkv * cap, d).double().numpy()
    kp, kn, kg = O.encode_qjl(s, kb, k, S32.astype(np.float64), s2=s2, kind="gauss")
    vp, vn = O.encode(s, vb, v, s2=s2, kind="gauss")
    shape = (B, Hkv, cap)
    kp, kn, kg = kp.reshape(*shape, -1), kn.reshape(shape), kg.reshape(shape)
    vp, vn = vp.reshape(*shape, -1), vn.reshape(shape)
    q = synth.normal_rows(1203, B * Hq, d, torch.bfloat16).reshape(B, Hq, d)
    want = O.attention_qjl(s, q.double().numpy(), kp, kn, kg, S32.astype(np.float64), vp, vn, kb, vb, 555,
                           0.125, s2=s2, kind="gauss")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    got = abi.tq_attn_decode_qjl(abi.Plan(d, 42, flags), dev(S32), q.cuda(),
                                 abi.Cache(dev(kp), dev(kn), dev(vp), dev(vn), kb, vb), dev(kg), 555, 0.125)
    torch.cuda.synchronize()
    assert np.abs(got.cpu().numpy() - want).max() <= ATTN_ATOL


def test_library_round_trip_is_unbiased():
    """Through the library alone (its own matrix, encode and decode), over 300
    plan seeds: <y, x_hat> - <y, x> averages to zero within four standard
    errors, while the library's MSE-only codec at b - 1 bits misses by more
    than ten (the shrinkage the second stage removes)."""
    d, bits = 128, 3
    x = synth.normal_rows(1300, 4, d).cuda()
    y = x + 0.5 * synth.normal_rows(1301, 4, d).cuda()
    truth = (x * y).sum(dim=1)
    eq, em = [], []
    for seed in range(300):
        plan = abi.Plan(d, 5000 + seed)
        S = abi.tq_qjl_matrix(plan)
        pk, nm, rn = abi.tq_encode_qjl(plan, bits, S, x)
        eq.append(((abi.tq_decode_qjl(plan, bits, S, pk, nm, rn) * y).sum(dim=1) - truth).double().cpu().numpy())
        mp, mn = abi.tq_encode(plan, bits - 1, x)
        em.append(((abi.tq_decode(plan, bits - 1, mp, mn) * y).sum(dim=1) - truth).double().cpu().numpy())
    for est, unbiased in ((np.array(eq), True), (np.array(em), False)):
        bias = est.mean(axis=0)
        se = est.std(axis=0, ddof=1) / math.sqrt(est.shape[0])
        if unbiased:
            assert np.all(np.abs(bias) < 4 * se), (bias, se)
        else:
            assert np.all(np.abs(bias) > 10 * se), (bias, se)
