"""GPU parity of the prefill (multi-query, causal) attention over the packed
cache (tq_attn_prefill, tcgen05) against the oracle, through the C ABI.

Cases span several 128-row query tiles with a ragged last tile, KV ranges
that end inside a 128-position block, every supported group size (1, 2, 4,
8 query heads per KV head), start positions past zero, mixed K/V widths and
the plan's format variants."""
import math

import numpy as np
import pytest
import torch

from kv_cache_vector_gb300 import abi, synth
from oracle import oracle as O
from parity import compare_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kv_cache_vector_gb300 import build
    build.build()
    abi.lib()
    abi.tq_device_status(reset=True)


def _setup(seed, B, T, Hq, Hkv, cap, kb, vb, flags=0):
    d = 128
    plan = abi.Plan(d, 42, flags)
    s = O.signs(42, d)
    s2 = O.signs2(42, d) if flags & abi.PLAN_TWO_SIDED_SIGNS else None
    kind = "gauss" if flags & abi.PLAN_GAUSSIAN_CODEBOOK else "sphere"
    kx = synth.normal_rows(seed, B * Hkv * cap, d, torch.bfloat16, stream=1).double().numpy()
    vx = synth.normal_rows(seed, B * Hkv * cap, d, torch.bfloat16, stream=2).double().numpy()
    kp, kn = O.encode(s, kb, kx, s2=s2, kind=kind)
    vp, vn = O.encode(s, vb, vx, s2=s2, kind=kind)
    shp = (B, Hkv, cap)
    arrs = (kp.reshape(*shp, -1), kn.reshape(shp), vp.reshape(*shp, -1), vn.reshape(shp))
    cache = abi.Cache(*(torch.from_numpy(a).cuda() for a in arrs), kb, vb)
    q = synth.normal_rows(seed + 1, B * T * Hq, d, torch.bfloat16, stream=3).reshape(B, T, Hq, d)
    return plan, s, s2, kind, arrs, cache, q


CASES = [
    # B, T, Hq, Hkv, q_start, cap, kb, vb
    (1, 8, 8, 2, [0], 64, 4, 3),
    (2, 100, 8, 2, [0, 37], 256, 3, 2),
    (1, 64, 32, 8, [300], 512, 4, 4),
    (1, 50, 4, 4, [130], 256, 2, 2),
    (2, 33, 16, 2, [5, 200], 300, 4, 2),
    (1, 200, 8, 8, [0], 256, 2, 4),
    (2, 45, 8, 2, [3, 211], 257, 3, 3),  # a capacity that leaves norm rows 4-byte aligned only
]


@pytest.mark.parametrize("B,T,Hq,Hkv,q_start,cap,kb,vb", CASES)
def test_prefill_parity(B, T, Hq, Hkv, q_start, cap, kb, vb):
    plan, s, s2, kind, arrs, cache, q = _setup(5 + T, B, T, Hq, Hkv, cap, kb, vb)
    qs = torch.tensor(q_start, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(128)
    out = abi.tq_attn_prefill(plan, q.cuda(), cache, qs, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    want = O.attention_prefill(s, q.double().numpy(), *arrs, kb, vb, np.array(q_start, np.int32), scale)
    compare_attention(out.cpu().numpy(), want)


@pytest.mark.parametrize("flags", [abi.PLAN_GAUSSIAN_CODEBOOK | abi.PLAN_TWO_SIDED_SIGNS, abi.PLAN_TWO_SIDED_SIGNS])
def test_prefill_format_variants(flags):
    B, T, Hq, Hkv, cap, kb, vb = 1, 70, 8, 2, 200, 4, 3
    plan, s, s2, kind, arrs, cache, q = _setup(91, B, T, Hq, Hkv, cap, kb, vb, flags)
    qs = torch.tensor([60], dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(128)
    out = abi.tq_attn_prefill(plan, q.cuda(), cache, qs, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    want = O.attention_prefill(s, q.double().numpy(), *arrs, kb, vb, np.array([60], np.int32), scale, s2=s2,
                               kind=kind)
    compare_attention(out.cpu().numpy(), want)


def test_prefill_last_token_matches_decode():
    """The chunk's last token attends over the same rows as a decode call with
    ctx = q_start + T; both kernels agree within the attention tolerance."""
    B, T, Hq, Hkv, cap, kb, vb = 2, 40, 8, 2, 300, 4, 3
    plan, s, s2, kind, arrs, cache, q = _setup(93, B, T, Hq, Hkv, cap, kb, vb)
    start = 250
    qs = torch.full((B,), start, dtype=torch.int32, device="cuda")
    out = abi.tq_attn_prefill(plan, q.cuda(), cache, qs, 0.1)
    dec = abi.tq_attn_decode(plan, q[:, -1].contiguous().cuda(), cache, start + T, 0.1)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    assert float((out[:, -1] - dec).abs().max()) <= 2e-3


def test_prefill_out_of_range_start():
    """q_start[b] + T past the cache: that sequence gets zero rows and status
    52; the others are computed."""
    B, T, Hq, Hkv, cap, kb, vb = 2, 20, 8, 2, 64, 3, 3
    plan, s, s2, kind, arrs, cache, q = _setup(95, B, T, Hq, Hkv, cap, kb, vb)
    qs = torch.tensor([10, 50], dtype=torch.int32, device="cuda")  # 50 + 20 > 64
    out = abi.tq_attn_prefill(plan, q.cuda(), cache, qs, 0.09)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 52
    got = out.cpu().numpy()
    assert np.all(got[1] == 0)
    want = O.attention_prefill(s, q[:1].double().numpy(), *(a[:1] for a in arrs), kb, vb,
                               np.array([10], np.int32), 0.09)
    compare_attention(got[:1], want)


def _sweep_cases(n, seed):
    import random
    rng = random.Random(seed)
    cases = []
    for _ in range(n):
        B = rng.choice([1, 2, 3])
        G = rng.choice([1, 2, 4, 8])
        Hkv = rng.choice([1, 2]) if G == 8 else rng.choice([1, 2, 4])
        T = rng.choice([1, 7, 33, 128, 129, 255, 300])
        starts = [rng.choice([0, 1, 63, 127, 128, 200, 400]) for _ in range(B)]
        cap = max(starts) + T + rng.choice([0, 1, 5, 130])
        flags = rng.choice([0, 0, abi.PLAN_TWO_SIDED_SIGNS, abi.PLAN_GAUSSIAN_CODEBOOK | abi.PLAN_TWO_SIDED_SIGNS])
        cases.append((B, T, G * Hkv, Hkv, starts, cap, rng.choice([2, 3, 4]), rng.choice([2, 3, 4]), flags,
                      rng.random() < 0.5))
    return cases


@pytest.mark.parametrize("B,T,Hq,Hkv,q_start,cap,kb,vb,flags,lowrank", _sweep_cases(10, 1234))
def test_prefill_seeded_sweep(B, T, Hq, Hkv, q_start, cap, kb, vb, flags, lowrank):
    """Seeded draws over batch, chunk length, group size, start positions
    (including a last position at the capacity), bit widths, format variants,
    and N(0,1) or low-rank rows with x8 outlier channels."""
    d = 128
    plan = abi.Plan(d, 42, flags)
    s = O.signs(42, d)
    s2 = O.signs2(42, d) if flags & abi.PLAN_TWO_SIDED_SIGNS else None
    kind = "gauss" if flags & abi.PLAN_GAUSSIAN_CODEBOOK else "sphere"
    n = B * Hkv * cap
    seed = 700 + T + cap
    if lowrank:
        kx = synth.lowrank_rows(seed, n, d, stream=1).double().numpy()
        vx = synth.lowrank_rows(seed, n, d, stream=2).double().numpy()
    else:
        kx = synth.normal_rows(seed, n, d, torch.bfloat16, stream=1).double().numpy()
        vx = synth.normal_rows(seed, n, d, torch.bfloat16, stream=2).double().numpy()
    kp, kn = O.encode(s, kb, kx, s2=s2, kind=kind)
    vp, vn = O.encode(s, vb, vx, s2=s2, kind=kind)
    shp = (B, Hkv, cap)
    arrs = (kp.reshape(*shp, -1), kn.reshape(shp), vp.reshape(*shp, -1), vn.reshape(shp))
    cache = abi.Cache(*(torch.from_numpy(a).cuda() for a in arrs), kb, vb)
    q = synth.normal_rows(seed + 1, B * T * Hq, d, torch.bfloat16, stream=3).reshape(B, T, Hq, d)
    qs = torch.tensor(q_start, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    out = abi.tq_attn_prefill(plan, q.cuda(), cache, qs, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    want = O.attention_prefill(s, q.double().numpy(), *arrs, kb, vb, np.array(q_start, np.int32), scale, s2=s2,
                               kind=kind)
    compare_attention(out.cpu().numpy(), want)
