"""Seeded sweep of the d = 128 decode attention's error over moderate contexts.

Few positions per softmax leave the outputs close to raw V values, and the
low-rank rows with x8 outlier channels (the Llama-8B-shaped workload) reach
|o| of about 25 there, so this is where the kernel's fp16 operand roundings
are least averaged.  1000 context lengths drawn without replacement from
[17, 2048], each with its own bf16 query, all eight KV-head groups (32 query
heads), through the contiguous kernel (one call per context) and the paged
kernel (one call, one sequence per context, all sharing the same pages).

Expected values: the oracle's causal attention over the oracle's own encoding
of the raw rows; token t of that prefill is the decode attention over the
first t + 1 positions ("TurboQuant KV Cache Compression -- Spec",
fa_tq_attention_cached).  The packed bytes the GPU reads are the oracle's.
Bound: every element within 2e-3 (the method's tolerance) and the worst
context below 1.5e-3, a margin on the tolerance.
"""
import math

import numpy as np
import pytest
import torch

from kv_cache_vector_gb300 import abi, synth
from oracle import oracle as O
from parity import ATTN_ATOL

pytestmark = pytest.mark.gpu

D, HQ, HKV, CAP, PAGE = 128, 32, 8, 2048, 256
N_CTX = 1000
SWEEP_BOUND = 1.5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kv_cache_vector_gb300 import build
    build.build()
    abi.lib()
    abi.tq_device_status(reset=True)


@pytest.fixture(scope="module")
def raw_rows():
    """Host rows [HKV, CAP, D] of K and V: low-rank plus four x8 outlier channels per group."""
    k = np.stack([synth.lowrank_rows(95, CAP, D, stream=40000 + g).double().numpy() for g in range(HKV)])
    v = np.stack([synth.lowrank_rows(95, CAP, D, stream=41000 + g).double().numpy() for g in range(HKV)])
    return k, v


@pytest.mark.parametrize("kb,vb", [(4, 3), (4, 2), (3, 2)])
def test_decode_attention_context_sweep(raw_rows, kb, vb):
    k, v = raw_rows
    s = O.signs(42, D)
    scale = 1.0 / math.sqrt(D)
    kp, kn = O.encode(s, kb, k.reshape(-1, D))
    vp, vn = O.encode(s, vb, v.reshape(-1, D))
    kp, kn = kp.reshape(HKV, CAP, -1), kn.reshape(HKV, CAP)
    vp, vn = vp.reshape(HKV, CAP, -1), vn.reshape(HKV, CAP)
    # token t's query; the oracle gives every token's attention over [0, t]
    q = synth.normal_rows(600 + 10 * kb + vb, CAP * HQ, D, torch.bfloat16, stream=5).reshape(CAP, HQ, D)
    want = O.attention_prefill(s, q.double().numpy()[None], kp[None], kn[None], vp[None], vn[None], kb, vb,
                               np.zeros(1, np.int32), scale)[0]
    ctxs = np.sort(np.random.default_rng(7 + kb * 10 + vb).choice(np.arange(17, CAP + 1), N_CTX, replace=False))

    plan = abi.Plan(D, 42)
    dev = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (kp, kn, vp, vn)]
    cache = abi.Cache(*(a[None] for a in dev), kb, vb)
    qd = q.cuda()
    got = torch.empty(N_CTX, HQ, D, device="cuda")
    for i, L in enumerate(ctxs):
        abi.tq_attn_decode(plan, qd[L - 1:L], cache, int(L), scale, out=got[i:i + 1])
    # paged: page p of every sequence is page p of the cache, each sequence its own length
    npg = CAP // PAGE
    pages = [a.reshape(HKV, npg, PAGE, *a.shape[2:]).transpose(0, 1).contiguous() for a in dev]
    pcache = abi.PagedCache(*pages, kb, vb)
    bt = torch.arange(npg, dtype=torch.int32, device="cuda").repeat(N_CTX, 1)
    lens = torch.from_numpy(ctxs.astype(np.int32)).cuda()
    got_p = abi.tq_attn_decode_paged(plan, qd[lens.long() - 1].contiguous(), pcache, bt, lens, CAP, scale)
    torch.cuda.synchronize()
    assert abi.tq_device_status() == 0
    ref = want[ctxs - 1]
    for name, g in (("contiguous", got), ("paged", got_p)):
        err = np.abs(g.cpu().numpy().astype(np.float64) - ref).reshape(N_CTX, -1).max(axis=1)
        print(f"K{kb}/V{vb} {name}: {N_CTX} contexts, worst {err.max():.3e}, "
              f"99th percentile {np.quantile(err, 0.99):.3e}, median {np.median(err):.3e}")
        assert err.max() <= ATTN_ATOL
        assert err.max() < SWEEP_BOUND, f"{name}: worst context error {err.max():.3e}"
