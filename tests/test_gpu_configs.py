"""Parity at the full sizes of the five workloads, in the launch configuration
the bench times.  Inputs are drawn on the device (seeded); the oracle encodes
and attends over sampled raw input rows it reads back (inputs only), and the
library's outputs for those rows are compared with it."""
import math

import numpy as np
import pytest
import torch

from kv_cache_vector_gb300 import abi, synth
from oracle import oracle as O
from parity import compare_attention, compare_decode, compare_encode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kv_cache_vector_gb300 import build
    build.build()
    abi.lib()


def _sample_rows(n, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, n, (k,), generator=g).sort().values


def test_llama8b_prefill_codec_full_size():
    """32 layers x 8 KV heads x batch 16 x 8192 tokens x d 128, bf16, low-rank
    + diagonal with 4 outlier channels x8 per (layer, head); K 4 bits, V 2
    bits.  Encode and decode all 33,554,432 rows of each; check 4096 sampled
    rows of each against the oracle."""
    d, per = 128, 16 * 8192
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    stats = {}
    for side, bits, stream0 in (("k", 4, 0), ("v", 2, 1)):
        x = torch.empty(32 * 8 * per, d, dtype=torch.bfloat16, device="cuda")
        for lh in range(32 * 8):
            x[lh * per:(lh + 1) * per] = synth.lowrank_rows(1000, per, d, stream=2 * lh + stream0,
                                                            device="cuda")
        pk, nm = abi.tq_encode(plan, bits, x)
        y = abi.tq_decode(plan, bits, pk, nm, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        idx = _sample_rows(x.shape[0], 4096, 7 + bits).cuda()
        xs = x[idx].double().cpu().numpy()
        st = compare_encode(s, bits, xs, pk[idx].cpu().numpy(), nm[idx].cpu().numpy())
        opk, onm = O.encode(s, bits, xs)
        same = np.all(opk == pk[idx].cpu().numpy(), axis=1)
        compare_decode(s, bits, opk[same], onm[same], y[idx].float().cpu().numpy()[same], bf16=True)
        stats[side] = st
        del x, pk, nm, y
        torch.cuda.empty_cache()
    print("llama8b prefill", stats)


def _attention_case(B, Hq, Hkv, ctx, kb, vb, kgen, vgen, seed, groups, thr_list):
    d = 128
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    cache = abi.Cache.empty(B, Hkv, ctx, d, kb, vb)
    raw = {}
    for h in range(Hkv):
        for side, gen, bits, pk_t, nm_t in (("k", kgen, kb, cache.k_packed, cache.k_norm),
                                            ("v", vgen, vb, cache.v_packed, cache.v_norm)):
            r = gen(h, side).reshape(B, ctx, d)
            raw[(side, h)] = r
            p2, n2 = abi.tq_encode(plan, bits, r.reshape(-1, d))
            pk_t[:, h] = p2.view(B, ctx, -1)
            nm_t[:, h] = n2.view(B, ctx)
    q = synth.device_normal(seed, (B, Hq, d))
    G = Hq // Hkv
    results = {}
    for thr in thr_list:
        out = abi.tq_attn_decode(plan, q, cache, ctx, 1.0 / math.sqrt(d), thr)
        torch.cuda.synchronize()
        worst = 0.0
        for b, h in groups:
            kx = raw[("k", h)][b].double().cpu().numpy()
            vx = raw[("v", h)][b].double().cpu().numpy()
            kp, kn = O.encode(s, kb, kx)
            vp, vn = O.encode(s, vb, vx)
            qq = q[b, h * G:(h + 1) * G].double().cpu().numpy()[None]
            got = out[b, h * G:(h + 1) * G].cpu().numpy()[None]
            for othr in sorted({0.0, thr}):
                want = O.attention(s, qq, kp[None, None], kn[None, None], vp[None, None],
                                   vn[None, None], kb, vb, ctx, 1.0 / math.sqrt(d), othr)
                worst = max(worst, compare_attention(got, want)["max_abs_err"])
        results[thr] = worst
    return results


def test_gqa_decode_attention_full_size():
    """Batch 32, 32 query / 8 KV heads, d 128, context 32768, K4/V3, cache
    drawn like the prefill; two sampled (batch, KV head) groups checked."""
    B, Hq, Hkv, ctx = 32, 32, 8, 32768

    def gen(h, side):
        return synth.lowrank_rows(2000, B * ctx, 128, stream=(0 if side == "k" else 100) + h,
                                  device="cuda")

    res = _attention_case(B, Hq, Hkv, ctx, 4, 3, gen, gen, 3, [(0, 0), (B - 1, Hkv - 1)], [0.0])
    print("gqa decode", res)


def test_long_context_dense_and_sparse_full_size():
    """Batch 1, 32 query / 8 KV heads, d 128, context 131072, K3/V2, keys
    N(0,1) with 2 outlier channels x8, values N(0,1); dense and sparse-V at
    1e-4, both within 2e-3 of the dense and of the sparse oracle."""
    B, Hq, Hkv, ctx = 1, 32, 8, 131072

    def kgen(h, side):
        return synth.outlier_rows(3000, B * ctx, 128, 2, stream=h, device="cuda")

    def vgen(h, side):
        return synth.device_normal(3100 + h, (B * ctx, 128))

    res = _attention_case(B, Hq, Hkv, ctx, 3, 2, kgen, vgen, 5, [(0, 0), (0, 5)], [0.0, 1e-4])
    print("long context", res)


@pytest.mark.parametrize("B,T,q_start", [(1, 2048, 0), (4, 512, 4096)])
def test_prefill_attention_full_size(B, T, q_start):
    """Prefill attention at the sizes the bench times: 32 query / 8 KV heads,
    d 128, K4/V3, rows low-rank + diag drawn as the bench draws them; a fresh
    2048-token prompt, and 4 x 512 tokens after 4096 cached.  For two
    sampled (sequence, KV head) groups the oracle encodes the raw rows it
    reads back and computes every token of the chunk for the group's query
    heads."""
    d, Hq, Hkv, kb, vb = 128, 32, 8, 4, 3
    G = Hq // Hkv
    cap = q_start + T
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    cache = abi.Cache.empty(B, Hkv, cap, d, kb, vb)
    rows = B * Hkv * cap
    raw = {}
    for side, bits, pk, nm, stream in (("k", kb, cache.k_packed, cache.k_norm, 40000),
                                       ("v", vb, cache.v_packed, cache.v_norm, 41000)):
        x = synth.lowrank_rows(95, rows, d, stream=stream, device="cuda")
        raw[side] = x.view(B, Hkv, cap, d)
        abi.tq_encode(plan, bits, x, pk.view(-1, d * bits // 8), nm.view(-1))
    q = synth.device_normal(96, (B, T, Hq, d))
    qs = torch.full((B,), q_start, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    out = abi.tq_attn_prefill(plan, q, cache, qs, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status(reset=True) == 0
    worst = 0.0
    for b, h in [(0, 0), (B - 1, Hkv - 1)]:
        kp, kn = O.encode(s, kb, raw["k"][b, h].double().cpu().numpy())
        vp, vn = O.encode(s, vb, raw["v"][b, h].double().cpu().numpy())
        qq = q[b:b + 1, :, h * G:(h + 1) * G].double().cpu().numpy()
        want = O.attention_prefill(s, qq, kp[None, None], kn[None, None], vp[None, None], vn[None, None], kb, vb,
                                   np.array([q_start], np.int32), scale)
        got = out[b:b + 1, :, h * G:(h + 1) * G].cpu().numpy()
        worst = max(worst, compare_attention(got, want)["max_abs_err"])
    print("prefill", B, T, q_start, "max abs err", worst)


def test_decode_attention_moderate_context_outliers():
    """Decode attention (batch 1, 32 query / 8 KV heads, K4/V3) on the
    bench's low-rank rows with x8 outlier channels, at contexts from 17 to
    2048: few rows per softmax, so the outputs stay close to raw V values
    and the keys' fp16 rounding is least averaged.  Four queries per context,
    all eight groups, against the oracle's own encoding of the raw rows."""
    d, Hq, Hkv, kb, vb, cap = 128, 32, 8, 4, 3, 2048
    G = Hq // Hkv
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    cache = abi.Cache.empty(1, Hkv, cap, d, kb, vb)
    enc = {}
    for side, bits, pk, nm, stream in (("k", kb, cache.k_packed, cache.k_norm, 40000),
                                       ("v", vb, cache.v_packed, cache.v_norm, 41000)):
        x = synth.lowrank_rows(95, Hkv * cap, d, stream=stream, device="cuda")
        abi.tq_encode(plan, bits, x, pk.view(-1, d * bits // 8), nm.view(-1))
        xs = x.view(Hkv, cap, d)
        for h in range(Hkv):
            enc[(side, h)] = O.encode(s, bits, xs[h].double().cpu().numpy())
    worst = 0.0
    for ctx in (17, 100, 300, 700, 1184, 1600, 2048):
        for trial in range(4):
            q = synth.device_normal(500 + trial, (1, Hq, d))
            out = abi.tq_attn_decode(plan, q, cache, ctx, 1.0 / math.sqrt(d), 0.0)
            torch.cuda.synchronize()
            for h in range(Hkv):
                (kp, kn), (vp, vn) = enc[("k", h)], enc[("v", h)]
                qq = q[:, h * G:(h + 1) * G].double().cpu().numpy()
                want = O.attention(s, qq, kp[None, None], kn[None, None], vp[None, None], vn[None, None], kb, vb,
                                   ctx, 1.0 / math.sqrt(d), 0.0)
                got = out[:, h * G:(h + 1) * G].cpu().numpy()
                worst = max(worst, compare_attention(got, want)["max_abs_err"])
    print("decode moderate contexts, outliers: max abs err", worst)


def test_gemma_window_encode_and_append_loop():
    """34 layers x 4 KV heads x d 256: full 512-token window written with
    tq_append (512 new rows per head) and tq_encode, then 50 single-token
    appends per layer, the 34-layer step captured in a CUDA graph; sampled
    layers checked against the oracle."""
    L, Hkv, d, T, steps = 34, 4, 256, 512, 50
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    cap = T + steps
    caches = [abi.Cache.empty(1, Hkv, cap, d, 4, 4) for _ in range(L)]
    win_k = synth.device_normal(4000, (L, 1, Hkv, T, d))
    win_v = synth.device_normal(4001, (L, 1, Hkv, T, d))
    new_k = synth.device_normal(4002, (steps, L, 1, Hkv, 1, d))
    new_v = synth.device_normal(4003, (steps, L, 1, Hkv, 1, d))
    for l in range(L):
        abi.tq_append(plan, caches[l], win_k[l], win_v[l], 0)
    # flat encode of the same window agrees with the cache rows: the two
    # kernels sum the norm in different orders, so an index may differ only
    # where a coordinate sits on a boundary (both are checked against the
    # oracle below)
    pk, nm = abi.tq_encode(plan, 4, win_k.reshape(-1, d))
    torch.cuda.synchronize()
    flat = O.unpack(pk.cpu().numpy(), d, 4)
    app = O.unpack(torch.stack([c.k_packed[0, :, :T] for c in caches]).reshape(-1, d // 2).cpu().numpy(), d, 4)
    assert np.mean(flat != app) <= 1e-5
    napp = torch.stack([c.k_norm[0, :, :T] for c in caches]).reshape(-1)
    assert torch.allclose(nm, napp, rtol=1e-6, atol=0)
    # one decode step (34 appends) captured once per position
    stream = torch.cuda.Stream()
    for step in range(steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                abi.tq_append(plan, caches[l], new_k[step, l], new_v[step, l], T + step)
        g.replay()
    torch.cuda.synchronize()
    for l in (0, 17, 33):
        for side, win, new, pk_t, nm_t in (("k", win_k, new_k, caches[l].k_packed, caches[l].k_norm),
                                           ("v", win_v, new_v, caches[l].v_packed, caches[l].v_norm)):
            rows = torch.cat([win[l, 0], new[:, l, 0, :, 0].permute(1, 0, 2)], dim=1)  # [Hkv, cap, d]
            compare_encode(s, 4, rows.reshape(-1, d).double().cpu().numpy(),
                           pk_t[0].reshape(-1, d // 2).cpu().numpy(), nm_t[0].reshape(-1).cpu().numpy())


@pytest.mark.parametrize("d,bits,in_dtype,out_dtype", [(128, 4, torch.bfloat16, torch.bfloat16),
                                                       (128, 2, torch.bfloat16, torch.bfloat16),
                                                       (128, 3, torch.float32, torch.float32),
                                                       (256, 4, torch.bfloat16, torch.bfloat16),
                                                       (256, 3, torch.bfloat16, torch.float32)])
def test_codec_ragged_large(d, bits, in_dtype, out_dtype):
    """1,000,003 rows (a multiple of neither 128 nor 32): the persistent
    encoders and decoders take several tiles per CTA, so their stage and
    accumulator phases wrap, and the last tile is ragged (the tensor-map load
    past the end fills zeros, the tensor-map store clips).  Encode, then
    decode; 2048 sampled rows and the last 200 rows against the oracle."""
    n = 1_000_003
    plan = abi.Plan(d, 42)
    s = O.signs(42, d)
    x = synth.lowrank_rows(1234 + d, n, d, dtype=in_dtype, stream=bits, device="cuda")
    pk, nm = abi.tq_encode(plan, bits, x)
    y = abi.tq_decode(plan, bits, pk, nm, out_dtype=out_dtype)
    torch.cuda.synchronize()
    idx = torch.cat([_sample_rows(n - 200, 2048, 11 + bits), torch.arange(n - 200, n)]).cuda()
    xs = x[idx].double().cpu().numpy()
    st = compare_encode(s, bits, xs, pk[idx].cpu().numpy(), nm[idx].cpu().numpy())
    opk, onm = O.encode(s, bits, xs)
    same = np.all(opk == pk[idx].cpu().numpy(), axis=1)
    compare_decode(s, bits, opk[same], onm[same], y[idx].float().cpu().numpy()[same],
                   bf16=out_dtype == torch.bfloat16)
    print("ragged codec", d, bits, st)


def test_decode_attention_ragged_large_context():
    """Batch 3, 32 query / 8 KV heads, context 70,001 (not a multiple of a
    chunk, a warp slice or a split), K4/V3, rows drawn like the prefill; three
    sampled (batch, KV head) groups checked."""
    B, Hq, Hkv, ctx = 3, 32, 8, 70001

    def gen(h, side):
        return synth.lowrank_rows(2100, B * ctx, 128, stream=(0 if side == "k" else 100) + h, device="cuda")

    res = _attention_case(B, Hq, Hkv, ctx, 4, 3, gen, gen, 4, [(0, 0), (1, 3), (2, Hkv - 1)], [0.0])
    print("ragged decode attention", res)
