"""GPU parity of the plan's format variants ("CITATIONS", N(0, 1/d) codebook
replacement; Two-sided Rademacher signs in WHT) against the oracle, through
the C ABI, on every kernel path: encode (tcgen05 d=128 bf16, TMA d=64 bf16,
per-thread fp32 and d=256), decode (d=128 bf16 staged, d=128 fp32, d=256),
append (warp per row, and the per-thread path at d=16), the d=128
tensor-core attention and the CUDA-core attention (d=64), and the paged
attention with its fused append."""
import math

import numpy as np
import pytest
import torch

from kv_cache_vector_gb300 import abi, synth
from oracle import oracle as O
from parity import compare_attention, compare_decode, compare_encode

pytestmark = pytest.mark.gpu

FLAGS = [abi.PLAN_GAUSSIAN_CODEBOOK, abi.PLAN_TWO_SIDED_SIGNS,
         abi.PLAN_GAUSSIAN_CODEBOOK | abi.PLAN_TWO_SIDED_SIGNS]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kv_cache_vector_gb300 import build
    build.build()
    abi.lib()
    abi.tq_device_status(reset=True)


def variant(plan):
    s2 = O.signs2(plan.seed, plan.d) if plan.flags & abi.PLAN_TWO_SIDED_SIGNS else None
    kind = "gauss" if plan.flags & abi.PLAN_GAUSSIAN_CODEBOOK else "sphere"
    return O.signs(plan.seed, plan.d), s2, kind


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (128, torch.float32), (64, torch.bfloat16),
                                     (256, torch.bfloat16)])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_encode_decode_variants(flags, d, dtype, bits):
    plan = abi.Plan(d, 42, flags)
    s, s2, kind = variant(plan)
    n = 3000  # several tiles and a ragged tail
    x = synth.normal_rows(60 + bits, n, d, dtype)
    pk, nm = abi.tq_encode(plan, bits, x.cuda())
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    compare_encode(s, bits, x.double().numpy(), pk.cpu().numpy(), nm.cpu().numpy(), s2=s2, kind=kind)
    # decode the oracle's bytes, so decode is checked on its own
    opk, onm = O.encode(s, bits, x.double().numpy(), s2=s2, kind=kind)
    for out_dtype in (torch.bfloat16, torch.float32):
        y = abi.tq_decode(plan, bits, torch.from_numpy(opk).cuda(), torch.from_numpy(onm).cuda(), out_dtype)
        torch.cuda.synchronize()
        compare_decode(s, bits, opk, onm, y.float().cpu().numpy(), out_dtype == torch.bfloat16, s2=s2, kind=kind)


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("d", [16, 128])
def test_append_variants(flags, d):
    plan = abi.Plan(d, 7, flags)
    s, s2, kind = variant(plan)
    B, Hkv, cap, kb, vb, pos = 3, 2, 40, 4, 3, 17
    cache = abi.Cache.empty(B, Hkv, cap, d, kb, vb)
    k = synth.normal_rows(71, B * Hkv, d, torch.bfloat16, stream=1).reshape(B, Hkv, 1, d)
    v = synth.normal_rows(71, B * Hkv, d, torch.bfloat16, stream=2).reshape(B, Hkv, 1, d)
    abi.tq_append(plan, cache, k.cuda(), v.cuda(), pos)
    torch.cuda.synchronize()
    for bits, x, pk_t, nm_t in ((kb, k, cache.k_packed, cache.k_norm), (vb, v, cache.v_packed, cache.v_norm)):
        got_pk = pk_t[:, :, pos].reshape(B * Hkv, -1).cpu().numpy()
        got_nm = nm_t[:, :, pos].reshape(B * Hkv).cpu().numpy()
        compare_encode(s, bits, x.reshape(B * Hkv, d).double().numpy(), got_pk, got_nm, s2=s2, kind=kind)


def _filled_cache(plan, s, s2, kind, B, Hkv, ctx, kb, vb, seed):
    d = plan.d
    kx = synth.normal_rows(seed, B * Hkv * ctx, d, torch.bfloat16, stream=1).double().numpy()
    vx = synth.normal_rows(seed, B * Hkv * ctx, d, torch.bfloat16, stream=2).double().numpy()
    kp, kn = O.encode(s, kb, kx, s2=s2, kind=kind)
    vp, vn = O.encode(s, vb, vx, s2=s2, kind=kind)
    shape = (B, Hkv, ctx)
    return (kp.reshape(*shape, -1), kn.reshape(shape), vp.reshape(*shape, -1), vn.reshape(shape))


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("d,kb,vb", [(128, 4, 3), (128, 3, 2), (64, 4, 2)])
def test_attention_variants(flags, d, kb, vb):
    plan = abi.Plan(d, 42, flags)
    s, s2, kind = variant(plan)
    B, Hq, Hkv, ctx = 2, 8, 2, 700
    kp, kn, vp, vn = _filled_cache(plan, s, s2, kind, B, Hkv, ctx, kb, vb, 81)
    cache = abi.Cache(*(torch.from_numpy(a).cuda() for a in (kp, kn, vp, vn)), kb, vb)
    q = synth.normal_rows(82, B * Hq, d, torch.bfloat16).reshape(B, Hq, d)
    scale = 1.0 / math.sqrt(d)
    out = abi.tq_attn_decode(plan, q.cuda(), cache, ctx, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    want = O.attention(s, q.double().numpy(), kp, kn, vp, vn, kb, vb, ctx, scale, s2=s2, kind=kind)
    compare_attention(out.cpu().numpy(), want)


@pytest.mark.parametrize("flags", FLAGS)
def test_paged_fused_step_variants(flags):
    """Paged cache, one decode step through the fused call: the appended rows
    and the attention follow the variant."""
    d, kb, vb, page = 128, 4, 3, 32
    plan = abi.Plan(d, 42, flags)
    s, s2, kind = variant(plan)
    lens, Hq, Hkv = [40, 95, 1], 8, 2
    B = len(lens)
    max_pages = 4
    bt = torch.tensor([[0, 1, -1, -1], [2, 3, 4, -1], [5, -1, -1, -1]], dtype=torch.int32)
    cache = abi.PagedCache.empty(6, Hkv, page, d, kb, vb)
    seqs = []
    for b, L in enumerate(lens):
        kp, kn, vp, vn = _filled_cache(plan, s, s2, kind, 1, Hkv, L, kb, vb, 90 + b)
        for pos in range(L):
            pg, off = int(bt[b, pos // page]), pos % page
            cache.k_packed[pg, :, off] = torch.from_numpy(kp[0, :, pos]).cuda()
            cache.k_norm[pg, :, off] = torch.from_numpy(kn[0, :, pos]).cuda()
            cache.v_packed[pg, :, off] = torch.from_numpy(vp[0, :, pos]).cuda()
            cache.v_norm[pg, :, off] = torch.from_numpy(vn[0, :, pos]).cuda()
        seqs.append((kp[0], kn[0], vp[0], vn[0]))
    k_new = synth.normal_rows(97, B * Hkv, d, torch.float32, stream=1).reshape(B, Hkv, d)
    v_new = synth.normal_rows(97, B * Hkv, d, torch.float32, stream=2).reshape(B, Hkv, d)
    q = synth.normal_rows(98, B * Hq, d, torch.bfloat16).reshape(B, Hq, d)
    scale = 1.0 / math.sqrt(d)
    pos_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = abi.tq_attn_decode_append_paged(plan, q.cuda(), k_new.cuda(), v_new.cuda(), cache, bt.cuda(), pos_t,
                                          max(lens) + 1, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    got = out.cpu().numpy()
    for b, L in enumerate(lens):
        kpn, knn = O.encode(s, kb, k_new[b].double().numpy(), s2=s2, kind=kind)
        vpn, vnn = O.encode(s, vb, v_new[b].double().numpy(), s2=s2, kind=kind)
        pg, off = int(bt[b, L // page]), L % page
        compare_encode(s, kb, k_new[b].double().numpy(), cache.k_packed[pg, :, off].cpu().numpy(),
                       cache.k_norm[pg, :, off].cpu().numpy(), s2=s2, kind=kind)
        kp, kn, vp, vn = seqs[b]
        seq = [np.concatenate([a, n_[:, None]], 1) for a, n_ in ((kp, kpn), (kn, knn), (vp, vpn), (vn, vnn))]
        want = O.attention(s, q[b].double().numpy()[None], seq[0][None], seq[1][None], seq[2][None], seq[3][None],
                           kb, vb, L + 1, scale, s2=s2, kind=kind)
        compare_attention(got[b][None], want)
