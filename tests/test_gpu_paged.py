"""GPU parity of the paged-cache entry points (tq_attn_decode_paged,
tq_append_paged) against the CPU oracle, called through the C ABI.

The packed rows come from the oracle's encoder on seeded inputs and are
scattered into pages through a shuffled block table; each sequence attends
over its own length.  Every page slot that holds no row of a sequence is
filled with garbage bytes and NaN norms, and block-table entries past a
sequence's pages are -1, so a read outside a sequence shows up as a wrong or
non-finite result, or as a non-zero device status word."""
import math

import numpy as np
import pytest
import torch

from kv_cache_vector_gb300 import abi, synth
from oracle import oracle as O
from parity import compare_attention, compare_encode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kv_cache_vector_gb300 import build
    build.build()
    abi.lib()
    abi.tq_device_status(reset=True)


def make_paged(seed, lens, Hq, Hkv, d, page, kb, vb, spare_pages=3, extra_slot=False):
    """Pages for sequences of the given lengths (plus, with extra_slot, room
    for one more position per sequence).  Returns the oracle's per-sequence
    rows, the device cache, the block table and max_pages."""
    s = O.signs(42, d)
    B = len(lens)
    need = [-(-(l + (1 if extra_slot else 0)) // page) for l in lens]
    max_pages = max(max(need), 1)
    n_pages = sum(need) + spare_pages
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n_pages, generator=g).tolist()
    bt = np.full((B, max_pages), -1, np.int32)
    k = 0
    for b in range(B):
        for i in range(need[b]):
            bt[b, i] = perm[k]
            k += 1
    kp = torch.randint(0, 256, (n_pages, Hkv, page, d * kb // 8), generator=g, dtype=torch.uint8).numpy()
    vp = torch.randint(0, 256, (n_pages, Hkv, page, d * vb // 8), generator=g, dtype=torch.uint8).numpy()
    kn = np.full((n_pages, Hkv, page), np.nan, np.float32)
    vn = np.full((n_pages, Hkv, page), np.nan, np.float32)
    seqs = []
    for b, L in enumerate(lens):
        if L == 0:
            seqs.append(None)
            continue
        kx = synth.normal_rows(seed * 100 + b, Hkv * L, d, torch.bfloat16, stream=1).double().numpy()
        vx = synth.normal_rows(seed * 100 + b, Hkv * L, d, torch.bfloat16, stream=2).double().numpy()
        kpb, knb = O.encode(s, kb, kx)
        vpb, vnb = O.encode(s, vb, vx)
        kpb, knb = kpb.reshape(Hkv, L, -1), knb.reshape(Hkv, L)
        vpb, vnb = vpb.reshape(Hkv, L, -1), vnb.reshape(Hkv, L)
        pos = np.arange(L)
        pg, off = bt[b, pos // page], pos % page
        hh = np.arange(Hkv)
        kp[pg[:, None], hh[None, :], off[:, None]] = kpb.transpose(1, 0, 2)
        vp[pg[:, None], hh[None, :], off[:, None]] = vpb.transpose(1, 0, 2)
        kn[pg[:, None], hh[None, :], off[:, None]] = knb.T
        vn[pg[:, None], hh[None, :], off[:, None]] = vnb.T
        seqs.append((kpb, knb, vpb, vnb))
    q = synth.normal_rows(seed, B * Hq, d, torch.bfloat16, stream=3).reshape(B, Hq, d)
    cache = abi.PagedCache(*(torch.from_numpy(a).cuda() for a in (kp, kn, vp, vn)), kb, vb)
    return s, q, seqs, cache, torch.from_numpy(bt).cuda(), max_pages


def oracle_seq(s, q_b, seq, kb, vb, L, scale, thr=0.0):
    if seq is None or L == 0:
        return np.zeros((q_b.shape[0], q_b.shape[1]))
    kpb, knb, vpb, vnb = seq
    return O.attention(s, q_b.double().numpy()[None], kpb[None], knb[None], vpb[None], vnb[None],
                       kb, vb, L, scale, thr)[0]


CASES = [
    # lens, Hq, Hkv, page, kb, vb
    ([1, 31, 32, 33, 64, 65, 200, 1000], 8, 2, 64, 4, 3),
    ([0, 5, 4097, 300], 16, 2, 32, 3, 2),
    ([2048, 2047, 1, 777], 8, 8, 256, 4, 4),
]


@pytest.mark.parametrize("d", [128, 64, 256])
@pytest.mark.parametrize("lens,Hq,Hkv,page,kb,vb", CASES)
def test_paged_attention_parity(lens, Hq, Hkv, page, kb, vb, d):
    """The tensor-core kernel at d = 128, the generic one at 64 and 256."""
    plan = abi.Plan(d, 42)
    s, q, seqs, cache, bt, max_pages = make_paged(11, lens, Hq, Hkv, d, page, kb, vb)
    scale = 1.0 / math.sqrt(d)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for max_ctx in (max(max(lens), 1), max_pages * page):  # a tight and a loose bound
        out = abi.tq_attn_decode_paged(plan, q.cuda(), cache, bt, lens_t, max_ctx, scale)
        torch.cuda.synchronize()
        assert abi.tq_device_status(reset=True) == 0
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        for b, L in enumerate(lens):
            want = oracle_seq(s, q[b], seqs[b], kb, vb, L, scale)
            compare_attention(got[b][None], want[None])


def test_paged_sparse_v():
    """Sparse V on a paged cache.  The kernel gates on each chunk's running
    maximum, so it keeps a superset of the oracle's rows and lies between the
    dense and the sparse oracle; at the contexts used here (as in the
    contiguous sparse-V test) both are within the attention tolerance."""
    lens, Hq, Hkv, page, kb, vb = [1000, 17, 700], 8, 2, 64, 4, 2
    d = 128
    plan = abi.Plan(d, 42)
    s, q, seqs, cache, bt, _ = make_paged(12, lens, Hq, Hkv, d, page, kb, vb)
    q = q * 3  # sharper softmax: more rows fall below the threshold
    scale = 1.0 / math.sqrt(d)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = abi.tq_attn_decode_paged(plan, q.to(torch.bfloat16).cuda(), cache, bt, lens_t, max(lens), scale, 1e-4)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    got = out.cpu().numpy()
    qb = q.to(torch.bfloat16)
    for b, L in enumerate(lens):
        for thr in (0.0, 1e-4):
            compare_attention(got[b][None], oracle_seq(s, qb[b], seqs[b], kb, vb, L, scale, thr)[None])


def test_paged_matches_contiguous():
    """Uniform lengths: the paged call and tq_attn_decode on the same rows agree."""
    d, B, Hq, Hkv, ctx, page, kb, vb = 128, 3, 8, 2, 777, 32, 4, 3
    plan = abi.Plan(d, 42)
    s, q, seqs, cache, bt, _ = make_paged(13, [ctx] * B, Hq, Hkv, d, page, kb, vb)
    flat = abi.Cache.empty(B, Hkv, ctx, d, kb, vb)
    for b in range(B):
        kpb, knb, vpb, vnb = seqs[b]
        flat.k_packed[b] = torch.from_numpy(kpb).cuda()
        flat.k_norm[b] = torch.from_numpy(knb).cuda()
        flat.v_packed[b] = torch.from_numpy(vpb).cuda()
        flat.v_norm[b] = torch.from_numpy(vnb).cuda()
    scale = 1.0 / math.sqrt(d)
    lens_t = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
    a = abi.tq_attn_decode_paged(plan, q.cuda(), cache, bt, lens_t, ctx, scale)
    c = abi.tq_attn_decode(plan, q.cuda(), flat, ctx, scale)
    torch.cuda.synchronize()
    assert float((a - c).abs().max()) <= 1e-6


def test_paged_append_rows_and_range_checks():
    d, Hkv, page, kb, vb = 128, 2, 32, 4, 3
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    cache = abi.PagedCache.empty(8, Hkv, page, d, kb, vb)
    bt = torch.tensor([[3, 1, -1, -1], [0, 5, 6, 7], [2, 4, -1, -1]], dtype=torch.int32, device="cuda")
    pos = [33, 127, 5]
    B = len(pos)
    k_new = synth.normal_rows(21, B * Hkv, d, torch.bfloat16, stream=1).reshape(B, Hkv, d)
    v_new = synth.normal_rows(21, B * Hkv, d, torch.bfloat16, stream=2).reshape(B, Hkv, d)
    abi.tq_append_paged(plan, cache, k_new.cuda(), v_new.cuda(), bt,
                        torch.tensor(pos, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    btn = bt.cpu().numpy()
    written = np.zeros((8, Hkv, page), bool)
    for side, x, pk_t, nm_t, bits in (("k", k_new, cache.k_packed, cache.k_norm, kb),
                                      ("v", v_new, cache.v_packed, cache.v_norm, vb)):
        pkh, nmh = pk_t.cpu().numpy(), nm_t.cpu().numpy()
        for b, p in enumerate(pos):
            pg, off = btn[b, p // page], p % page
            compare_encode(s, bits, x[b].double().numpy(), pkh[pg, :, off], nmh[pg, :, off])
            written[pg, :, off] = True
        assert not pkh[~written].any() and not nmh[~written].any()  # nothing else was touched
    # out of range: a negative position, one past max_pages * page, and a -1 page
    before = [t.clone() for t in (cache.k_packed, cache.k_norm, cache.v_packed, cache.v_norm)]
    abi.tq_append_paged(plan, cache, k_new.cuda(), v_new.cuda(), bt,
                        torch.tensor([-1, 128, 70], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 42
    for t0, t1 in zip(before, (cache.k_packed, cache.k_norm, cache.v_packed, cache.v_norm)):
        assert torch.equal(t0, t1)


def test_paged_append_then_attend():
    """A decode step on a paged cache: append one token per sequence at its
    length, then attend over length + 1."""
    lens, Hq, Hkv, page, kb, vb = [63, 64, 10, 1], 8, 2, 64, 4, 3
    d = 128
    plan = abi.Plan(d, 42)
    s, q, seqs, cache, bt, max_pages = make_paged(14, lens, Hq, Hkv, d, page, kb, vb, extra_slot=True)
    B = len(lens)
    k_new = synth.normal_rows(31, B * Hkv, d, torch.bfloat16, stream=1).reshape(B, Hkv, d)
    v_new = synth.normal_rows(31, B * Hkv, d, torch.bfloat16, stream=2).reshape(B, Hkv, d)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    abi.tq_append_paged(plan, cache, k_new.cuda(), v_new.cuda(), bt, lens_t)
    scale = 1.0 / math.sqrt(d)
    out = abi.tq_attn_decode_paged(plan, q.cuda(), cache, bt, lens_t + 1, max(lens) + 1, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    got = out.cpu().numpy()
    for b, L in enumerate(lens):
        kpn, knn = O.encode(s, kb, k_new[b].double().numpy())
        vpn, vnn = O.encode(s, vb, v_new[b].double().numpy())
        kpb, knb, vpb, vnb = seqs[b]
        seq = (np.concatenate([kpb, kpn[:, None]], 1), np.concatenate([knb, knn[:, None]], 1),
               np.concatenate([vpb, vpn[:, None]], 1), np.concatenate([vnb, vnn[:, None]], 1))
        compare_attention(got[b][None], oracle_seq(s, q[b], seq, kb, vb, L + 1, scale)[None])


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("kv_dtype", [torch.bfloat16, torch.float32])
def test_fused_append_attend_matches_two_calls(kv_dtype, d):
    """tq_attn_decode_append_paged writes the same cache bytes as
    tq_append_paged and returns what tq_attn_decode_paged returns over the
    lengths + 1; both agree with the oracle over the grown sequences (one
    launch sequence at d = 128, the append and then the generic kernel at
    d = 256)."""
    lens, Hq, Hkv, page, kb, vb = [63, 64, 10, 1, 300], 8, 2, 64, 4, 3
    plan = abi.Plan(d, 42)
    s, q, seqs, cache, bt, max_pages = make_paged(15, lens, Hq, Hkv, d, page, kb, vb, extra_slot=True)
    B = len(lens)
    k_new = synth.normal_rows(41, B * Hkv, d, kv_dtype, stream=1).reshape(B, Hkv, d)
    v_new = synth.normal_rows(41, B * Hkv, d, kv_dtype, stream=2).reshape(B, Hkv, d)
    pos = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    max_ctx = max(lens) + 1
    twin = abi.PagedCache(*(t.clone() for t in (cache.k_packed, cache.k_norm, cache.v_packed, cache.v_norm)),
                          kb, vb)
    abi.tq_append_paged(plan, twin, k_new.cuda(), v_new.cuda(), bt, pos)
    want = abi.tq_attn_decode_paged(plan, q.cuda(), twin, bt, pos + 1, max_ctx, scale)
    got = abi.tq_attn_decode_append_paged(plan, q.cuda(), k_new.cuda(), v_new.cuda(), cache, bt, pos, max_ctx,
                                          scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    for a, b in zip((cache.k_packed, cache.k_norm, cache.v_packed, cache.v_norm),
                    (twin.k_packed, twin.k_norm, twin.v_packed, twin.v_norm)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert torch.equal(got, want)
    out = got.cpu().numpy()
    for b, L in enumerate(lens):
        kpn, knn = O.encode(s, kb, k_new[b].double().numpy())
        vpn, vnn = O.encode(s, vb, v_new[b].double().numpy())
        kpb, knb, vpb, vnb = seqs[b]
        seq = (np.concatenate([kpb, kpn[:, None]], 1), np.concatenate([knb, knn[:, None]], 1),
               np.concatenate([vpb, vpn[:, None]], 1), np.concatenate([vnb, vnn[:, None]], 1))
        compare_attention(out[b][None], oracle_seq(s, q[b], seq, kb, vb, L + 1, scale)[None])


def test_fused_append_attend_range_checks():
    """A position out of range (negative, or on a -1 page) writes nothing,
    sets status 42, and that sequence attends over min(position + 1, max_ctx)
    rows (none for a negative position); the other sequences are unaffected."""
    lens, Hq, Hkv, page, kb, vb = [40, 64, 5], 8, 2, 64, 3, 2
    d = 128
    plan = abi.Plan(d, 42)
    s, q, seqs, cache, bt, max_pages = make_paged(16, lens, Hq, Hkv, d, page, kb, vb)
    B = len(lens)
    k_new = synth.normal_rows(42, B * Hkv, d, torch.bfloat16, stream=1).reshape(B, Hkv, d)
    v_new = synth.normal_rows(42, B * Hkv, d, torch.bfloat16, stream=2).reshape(B, Hkv, d)
    # sequence 0: a negative position; sequence 1: position 64, past max_pages * page_size (one
    # page each here); sequence 2: a valid append at its length
    pos = torch.tensor([-1, 64, 5], dtype=torch.int32, device="cuda")
    before = [t.clone() for t in (cache.k_packed, cache.k_norm, cache.v_packed, cache.v_norm)]
    scale = 1.0 / math.sqrt(d)
    got = abi.tq_attn_decode_append_paged(plan, q.cuda(), k_new.cuda(), v_new.cuda(), cache, bt, pos, 64, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 42
    btn = bt.cpu().numpy()
    # bytes, not values: unused slots hold NaN norms
    changed = [(t0.view(torch.uint8) != t1.view(torch.uint8)).reshape(t0.shape[0], Hkv, page, -1)
               for t0, t1 in zip(before, (cache.k_packed, cache.k_norm, cache.v_packed, cache.v_norm))]
    # only sequence 2's slot at position 5 changed
    pg, off = btn[2, 0], 5
    for c in changed:
        c = c.cpu().numpy().copy()
        c[pg, :, off] = False
        assert not c.any()
    out = got.cpu().numpy()
    assert np.all(out[0] == 0)
    compare_attention(out[1][None], oracle_seq(s, q[1], seqs[1], kb, vb, 64, scale)[None])
    kpn, knn = O.encode(s, kb, k_new[2].double().numpy())
    vpn, vnn = O.encode(s, vb, v_new[2].double().numpy())
    kpb, knb, vpb, vnb = seqs[2]
    seq = (np.concatenate([kpb, kpn[:, None]], 1), np.concatenate([knb, knn[:, None]], 1),
           np.concatenate([vpb, vpn[:, None]], 1), np.concatenate([vnb, vnn[:, None]], 1))
    compare_attention(out[2][None], oracle_seq(s, q[2], seq, kb, vb, 6, scale)[None])
