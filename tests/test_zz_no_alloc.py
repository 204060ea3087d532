"""tq_attn_decode_noalloc: the decode-attention call for callers that may not
allocate device memory while they run (a plugin whose host framework owns all
device memory, a serving loop with a memory plan fixed up front).  It must
give what tq_attn_decode gives, call after call, from its fixed scratch array,
and refuse sizes whose partials do not fit that array."""
import math

import numpy as np
import pytest
import torch

from kv_cache_vector_gb300 import abi, synth
from parity import ATTN_ATOL

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kv_cache_vector_gb300 import build
    build.build()
    abi.lib()


def _filled_cache(plan, B, Hkv, cap, kb, vb, seed):
    d = plan.d
    cache = abi.Cache.empty(B, Hkv, cap, d, kb, vb)
    k = synth.device_normal(seed, (B, Hkv, cap, d))
    v = synth.device_normal(seed + 1, (B, Hkv, cap, d))
    abi.tq_append(plan, cache, k, v, 0)
    return cache


def _raw_noalloc(plan, q, cache, ctx, scale, thr, out):
    """The entry point called straight through the C ABI."""
    import ctypes
    B, Hq, _ = q.shape
    Hkv = cache.k_norm.shape[1]
    return abi.lib().tq_attn_decode_noalloc(
        plan.handle, q.data_ptr(), B, Hq, Hkv, cache.view(), ctx, cache.k_bits, cache.v_bits,
        ctypes.c_float(scale), ctypes.c_float(thr), out.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("B,Hq,Hkv,d,ctx,kb,vb,thr", [
    (2, 8, 2, 128, 3001, 4, 3, 0.0),
    (1, 32, 8, 128, 20000, 3, 2, 1e-4),
    (3, 4, 4, 64, 257, 4, 4, 0.0),
])
def test_noalloc_matches_workspace_call_twice(B, Hq, Hkv, d, ctx, kb, vb, thr):
    plan = abi.Plan(d, 42)
    cache = _filled_cache(plan, B, Hkv, ctx, kb, vb, seed=B * 1000 + ctx)
    q = synth.device_normal(7 + ctx, (B, Hq, d))
    scale = 1.0 / math.sqrt(d)
    assert abi.tq_attn_workspace_bytes(B, Hq, Hkv, d, ctx) <= SCRATCH_BYTES
    want = abi.tq_attn_decode(plan, q, cache, ctx, scale, thr).cpu().numpy()
    for _ in range(2):  # the scratch keeps the previous call's contents
        out = torch.full((B, Hq, d), float("nan"), device="cuda")
        assert _raw_noalloc(plan, q, cache, ctx, scale, thr, out) == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - want)) <= ATTN_ATOL


def test_noalloc_refuses_sizes_beyond_its_scratch():
    B, Hq, Hkv, d, ctx = 32, 64, 8, 128, 4096
    while abi.tq_attn_workspace_bytes(B, Hq, Hkv, d, ctx) <= SCRATCH_BYTES:
        ctx *= 2  # the split geometry decides the size: grow the context until it overflows
        assert ctx <= 1 << 20
    plan = abi.Plan(d, 42)
    cache = abi.Cache.empty(B, Hkv, ctx, d, 4, 3)
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(B, Hq, d, device="cuda")
    assert _raw_noalloc(plan, q, cache, ctx, 0.1, 0.0, out) == 5   # TQ_ERR_WORKSPACE
    with pytest.raises(abi.TQError, match="WORKSPACE"):
        abi.tq_attn_decode_noalloc(plan, q, cache, ctx, 0.1, out=out)
