"""GPU parity of tq_encode / tq_decode / tq_append against the CPU oracle,
called through the C ABI on the same seeded input bytes."""
import math

import numpy as np
import pytest
import torch

from kv_cache_vector_gb300 import abi, synth
from oracle import oracle as O
from parity import compare_decode, compare_encode

pytestmark = pytest.mark.gpu

DIMS = [8, 16, 32, 64, 128, 256]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kv_cache_vector_gb300 import build
    build.build()
    abi.lib()


def _encode(plan, bits, x):
    pk, nm = abi.tq_encode(plan, bits, x.cuda())
    torch.cuda.synchronize()
    return pk.cpu().numpy(), nm.cpu().numpy()


def test_codec_round_trip_4096x128_fp32():
    """4096 rows x d=128 fp32 N(0,1) from seed 0, signs from seed 42, 4 bits:
    encode parity, decode parity, per-row cosine and MSE."""
    d, bits = 128, 4
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    x = synth.normal_rows(0, 4096, d, torch.float32)
    pk, nm = _encode(plan, bits, x)
    st = compare_encode(s, bits, x.double().numpy(), pk, nm)
    y = abi.tq_decode(plan, bits, torch.from_numpy(pk).cuda(), torch.from_numpy(nm).cuda())
    y = y.cpu().numpy()
    compare_decode(s, bits, pk, nm, y, bf16=False)
    xn = x.double().numpy()
    cos = (xn * y).sum(1) / np.linalg.norm(xn, axis=1) / np.linalg.norm(y, axis=1)
    mse = ((xn - y) ** 2).mean(1) / (xn ** 2).mean(1)
    assert cos.min() > 0.98 and cos.mean() == pytest.approx(math.sqrt(1 - 0.009315), abs=2e-3)
    assert mse.mean() < 0.012
    print("config-1 encode", st, "cos mean %.5f min %.5f" % (cos.mean(), cos.min()))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("d", DIMS)
def test_encode_parity_ragged(d, bits, dtype):
    n = 333  # not a multiple of the 256-thread block, nor of 32
    plan = abi.Plan(d, 7)
    x = synth.normal_rows(d * 10 + bits, n, d, dtype)
    pk, nm = _encode(plan, bits, x)
    compare_encode(O.signs(7, d), bits, x.double().numpy(), pk, nm)


@pytest.mark.parametrize("d", [8, 128, 256])
def test_encode_edge_rows(d):
    """Zero rows, constant rows, one-hot rows, power-of-two scalings and
    extreme (but finite-norm) magnitudes (Foundry spec, Testing Strategy 6)."""
    bits = 4
    plan = abi.Plan(d, 42)
    base = synth.normal_rows(99, 8, d).double()
    rows = [torch.zeros(d), torch.full((d,), 3.0), torch.full((d,), -0.5)]
    rows += [torch.eye(d)[j] for j in (0, d // 2, d - 1)]
    rows += [base[0] * 2.0 ** k for k in (-40, -8, 0, 8, 40)]
    x = torch.stack([r.float() for r in rows])
    pk, nm = _encode(plan, bits, x)
    s = O.signs(42, d)
    compare_encode(s, bits, x.double().numpy(), pk, nm)
    idx = O.unpack(pk, d, bits)
    assert np.all(idx[0] == 8) and nm[0] == 0.0
    for k in range(6, 11):  # scalings by 2^k keep the indices
        assert np.array_equal(idx[k], idx[8])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [8, 64, 128, 256])
def test_encode_rows_beyond_fp32_squares(d, dtype):
    """Rows of finite norm whose sum of squares leaves fp32's range (scalings
    by 2^+-70 and 2^+-100 of seeded rows), beside in-range ones and a zero
    row: every encoder (thread per row, TMA-fed, tensor-core at d = 128 and
    256, bf16 and fp32 rows) gives the oracle's indices, the indices of the
    unscaled row, and the norm scaled by 2^k."""
    bits = 4
    plan = abi.Plan(d, 42)
    base = synth.normal_rows(123 + d, 6, d).double()
    ks = (-100, -70, 0, 70, 100)
    rows = [base[j] * 2.0 ** k for j in range(6) for k in ks] + [torch.zeros(d, dtype=torch.float64)]
    x = torch.stack(rows).to(dtype)
    pk, nm = _encode(plan, bits, x)
    s = O.signs(42, d)
    compare_encode(s, bits, x.double().numpy(), pk, nm)
    idx = O.unpack(pk, d, bits)
    for j in range(6):
        r0 = j * len(ks) + ks.index(0)
        for i, k in enumerate(ks):
            r = j * len(ks) + i
            assert np.array_equal(idx[r], idx[r0])
            assert abs(float(nm[r]) / 2.0 ** k / float(nm[r0]) - 1.0) < 1e-6
    assert nm[-1] == 0.0 and np.all(idx[-1] == 8)


def test_append_rows_beyond_fp32_squares():
    """The append's warp-per-row encoder on rows scaled by 2^+-100."""
    d, kb, vb, B, Hkv, cap = 128, 4, 2, 1, 2, 8
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    cache = abi.Cache.empty(B, Hkv, cap, d, kb, vb)
    base = synth.normal_rows(77, B * Hkv * 2, d).double()
    scale = torch.tensor([2.0 ** 100, 2.0 ** -100, 2.0 ** 100, 1.0], dtype=torch.float64)[:, None]
    k = (base * scale).to(torch.bfloat16).reshape(B, Hkv, 2, d)
    v = (base * scale.flip(0)).to(torch.bfloat16).reshape(B, Hkv, 2, d)
    abi.tq_append(plan, cache, k.cuda(), v.cuda(), 3)
    torch.cuda.synchronize()
    for x, bits, pk_t, nm_t in ((k, kb, cache.k_packed, cache.k_norm), (v, vb, cache.v_packed, cache.v_norm)):
        got_pk = pk_t.cpu().numpy()[:, :, 3:5].reshape(-1, d * bits // 8)
        got_nm = nm_t.cpu().numpy()[:, :, 3:5].reshape(-1)
        compare_encode(s, bits, x.double().numpy().reshape(-1, d), got_pk, got_nm)


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_encode_spiky_rotated_rows_bf16(d, bits):
    """bf16 rows whose rotated, normalised coordinates reach |u| = 1 or sit
    near |u| = 0.5: a sign-flipped column of the Hadamard matrix, scaled, plus
    seeded noise.  The d = 128 and d = 256 encoders bucket every finite row
    through their 1/64-cell table, cells -64 .. 64 included (they once had a
    window |u| < 0.5 and a binary-search fallback); all must agree with the
    oracle."""
    s = O.signs(42, d)
    noise = synth.normal_rows(4242 + d, 64, d).double().numpy()
    j = np.arange(d)
    rows = []
    for r in range(64):
        k = (r * 37) % d
        col = s * np.where([bin(int(i) & k).count("1") % 2 for i in j], -1.0, 1.0)
        a = (1.0, -1.0, 0.9, 0.6, 0.52, 0.5, 0.48, 0.3)[r % 8]
        b = 0.0 if r % 16 < 2 else 0.03 * (1 + r % 5)
        rows.append(a * col / math.sqrt(d) + b * noise[r])
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16)
    plan = abi.Plan(d, 42)
    pk, nm = _encode(plan, bits, x)
    compare_encode(s, bits, x.double().numpy(), pk, nm)
    u = O.encode(s, bits, x.double().numpy(), want_u=True)[2]
    m = np.abs(u).max(axis=1)
    assert m.max() > 0.99 and (m >= 0.5).sum() >= 16 and ((m > 0.4) & (m < 0.6)).sum() >= 8


def test_encode_single_row_and_empty():
    plan = abi.Plan(128, 3)
    x = synth.normal_rows(5, 1, 128)
    pk, nm = _encode(plan, 3, x)
    compare_encode(O.signs(3, 128), 3, x.double().numpy(), pk, nm)
    e = torch.empty(0, 128, device="cuda")
    pk, nm = abi.tq_encode(plan, 3, e)
    assert pk.shape == (0, 48)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("d", DIMS)
def test_decode_parity_random_codes(d, bits, out_dtype):
    """Any byte string is a valid code: seeded random bytes and norms (some
    zero) go through both decoders."""
    n = 333
    rng = np.random.default_rng(d * 7 + bits)
    packed = rng.integers(0, 256, size=(n, d * bits // 8), dtype=np.uint8)
    norms = (rng.random(n) * 20).astype(np.float32)
    norms[::17] = 0.0
    plan = abi.Plan(d, 11)
    y = abi.tq_decode(plan, bits, torch.from_numpy(packed).cuda(), torch.from_numpy(norms).cuda(),
                      out_dtype=out_dtype)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy()
    compare_decode(O.signs(11, d), bits, packed, norms, got, bf16=out_dtype == torch.bfloat16)
    assert np.all(got[::17] == 0.0)


@pytest.mark.parametrize("d,kb,vb", [(64, 4, 2), (128, 4, 3), (128, 3, 3), (256, 4, 4), (32, 2, 4)])
@pytest.mark.parametrize("n_new,pos", [(1, 0), (1, 13), (5, 7), (4, 16)])
def test_append_parity_and_untouched(d, kb, vb, n_new, pos):
    B, Hkv, cap = 2, 3, 20
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    cache = abi.Cache.empty(B, Hkv, cap, d, kb, vb)
    for t in (cache.k_packed, cache.v_packed):
        t.fill_(0xA5)
    cache.k_norm.fill_(-1.0)
    cache.v_norm.fill_(-1.0)
    k = synth.normal_rows(1, B * Hkv * n_new, d, torch.bfloat16).reshape(B, Hkv, n_new, d)
    v = synth.normal_rows(2, B * Hkv * n_new, d, torch.bfloat16).reshape(B, Hkv, n_new, d)
    abi.tq_append(plan, cache, k.cuda(), v.cuda(), pos)
    torch.cuda.synchronize()
    for side, x, bits, pk_t, nm_t in (("k", k, kb, cache.k_packed, cache.k_norm),
                                      ("v", v, vb, cache.v_packed, cache.v_norm)):
        pk = pk_t.cpu().numpy()
        nm = nm_t.cpu().numpy()
        got_pk = pk[:, :, pos:pos + n_new].reshape(-1, d * bits // 8)
        got_nm = nm[:, :, pos:pos + n_new].reshape(-1)
        compare_encode(s, bits, x.double().numpy().reshape(-1, d), got_pk, got_nm)
        mask = np.ones(cap, bool)
        mask[pos:pos + n_new] = False
        assert np.all(pk[:, :, mask] == 0xA5), f"{side}: bytes outside the appended rows changed"
        assert np.all(nm[:, :, mask] == -1.0), f"{side}: norms outside the appended rows changed"


def test_append_errors():
    plan = abi.Plan(128, 1)
    cache = abi.Cache.empty(1, 2, 8, 128, 4, 2)
    k = torch.zeros(1, 2, 3, 128, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(abi.TQError, match="RANGE"):
        abi.tq_append(plan, cache, k, k, 6)
    with pytest.raises(abi.TQError, match="RANGE"):
        abi.tq_append(plan, cache, k, k, -1)
