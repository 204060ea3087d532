"""Decode steps captured in a CUDA graph and replayed.

The attention kernels are launched with programmatic stream serialization:
each may start while the previous kernel of the stream still runs, and waits
for it before reading what it wrote.  Here every layer's attention follows an
append into the same cache, so a kernel that read the cache before that wait
would miss the appended row.  Three layers of (tq_append, tq_attn_decode) are
captured in one graph and replayed twice; the outputs must equal the eager
calls bit for bit and the oracle's attention over the oracle's encoding of
the same rows (appended row included) within 2e-3 (the sparse-V call: within
2e-3 of the eager call too, since its gate depends on the order in which the
CTAs raise a shared running maximum) ("TurboQuant KV Cache
Compression -- Spec", fa_tq_attention_cached: quantise the new K/V into the
cache, then attend over it).
"""
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


@pytest.mark.parametrize("d,kb,vb,thr", [(128, 4, 3, 0.0), (128, 3, 2, 1e-4), (256, 4, 4, 0.0), (64, 4, 2, 0.0)])
def test_append_then_attend_in_a_graph(d, kb, vb, thr):
    L, B, Hq, Hkv, cap, ctx0 = 3, 2, 8, 2, 1024, 700
    s = O.signs(42, d)
    plan = abi.Plan(d, 42)
    scale = 1.0 / math.sqrt(d)
    layers = []
    for l in range(L):
        k = synth.normal_rows(3000 + 10 * l + d, B * Hkv * cap, d, torch.bfloat16, stream=1)
        v = synth.normal_rows(3000 + 10 * l + d, B * Hkv * cap, d, torch.bfloat16, stream=2)
        kp, kn = O.encode(s, kb, k.double().numpy())
        vp, vn = O.encode(s, vb, v.double().numpy())
        shape = (B, Hkv, cap)
        host = dict(k_packed=kp.reshape(*shape, -1).copy(), k_norm=kn.reshape(shape).copy(),
                    v_packed=vp.reshape(*shape, -1).copy(), v_norm=vn.reshape(shape).copy())
        # the rows the graph appends at position ctx0 are the raw rows there
        k_new = k.reshape(B, Hkv, cap, d)[:, :, ctx0:ctx0 + 1].contiguous()
        v_new = v.reshape(B, Hkv, cap, d)[:, :, ctx0:ctx0 + 1].contiguous()
        for f in ("k_packed", "k_norm", "v_packed", "v_norm"):  # the slot starts out zeroed
            host[f][:, :, ctx0] = 0
        cache = abi.Cache(*(torch.from_numpy(np.ascontiguousarray(host[f])).cuda()
                            for f in ("k_packed", "k_norm", "v_packed", "v_norm")), kb, vb)
        q = synth.normal_rows(3100 + l + d, B * Hq, d, torch.bfloat16, stream=3).reshape(B, Hq, d)
        want = O.attention(s, q.double().numpy(), kp.reshape(*shape, -1), kn.reshape(shape),
                           vp.reshape(*shape, -1), vn.reshape(shape), kb, vb, ctx0 + 1, scale)
        ws = torch.empty(max(16, abi.tq_attn_workspace_bytes(B, Hq, Hkv, d, ctx0 + 1)), dtype=torch.uint8,
                         device="cuda")
        layers.append(dict(cache=cache, k_new=k_new.cuda(), v_new=v_new.cuda(), q=q.cuda(), want=want, ws=ws,
                           out=torch.empty(B, Hq, d, device="cuda")))

    def step():
        for ly in layers:
            abi.tq_append(plan, ly["cache"], ly["k_new"], ly["v_new"], ctx0)
            abi.tq_attn_decode(plan, ly["q"], ly["cache"], ctx0 + 1, scale, thr, out=ly["out"], workspace=ly["ws"])

    step()  # eager
    torch.cuda.synchronize()
    eager = [ly["out"].clone() for ly in layers]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    for ly in layers:
        ly["out"].zero_()
    with torch.cuda.graph(g, stream=side):
        step()
    for _ in range(2):
        for ly in layers:
            ly["out"].zero_()
        g.replay()
        torch.cuda.synchronize()
        for ly, e in zip(layers, eager):
            if thr == 0.0:
                assert torch.equal(ly["out"], e)
            else:  # the gate reads a running maximum raised in a timing-dependent order
                compare_attention(ly["out"].cpu().numpy(), e.cpu().numpy().astype(np.float64))
    assert abi.tq_device_status() == 0
    for ly in layers:
        compare_attention(ly["out"].cpu().numpy(), ly["want"])
