"""GPU parity of tq_attn_decode against the CPU oracle.  The packed cache is
built by the oracle's encoder from seeded inputs and uploaded, so both sides
read the same bytes; the oracle attends in the unrotated domain."""
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


def make_case(seed, B, Hq, Hkv, d, cap, kb, vb, n_outliers=0):
    s = O.signs(42, d)
    n = B * Hkv * cap
    if n_outliers:
        k = synth.outlier_rows(seed, n, d, n_outliers, torch.bfloat16, stream=1)
    else:
        k = synth.normal_rows(seed, n, d, torch.bfloat16, stream=1)
    v = synth.normal_rows(seed, n, d, torch.bfloat16, stream=2)
    kp, kn = O.encode(s, kb, k.double().numpy())
    vp, vn = O.encode(s, vb, v.double().numpy())
    q = synth.normal_rows(seed, B * Hq, d, torch.bfloat16, stream=3).reshape(B, Hq, d)
    host = dict(k_packed=kp.reshape(B, Hkv, cap, -1), k_norm=kn.reshape(B, Hkv, cap),
                v_packed=vp.reshape(B, Hkv, cap, -1), v_norm=vn.reshape(B, Hkv, cap))
    cache = abi.Cache(*(torch.from_numpy(host[f]).cuda() for f in
                        ("k_packed", "k_norm", "v_packed", "v_norm")), kb, vb)
    return s, q, host, cache


def run(plan, q, cache, ctx, scale, thr=0.0):
    out = abi.tq_attn_decode(plan, q.cuda(), cache, ctx, scale, thr)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_out(s, q, host, kb, vb, ctx, scale, thr=0.0, kept=False):
    return O.attention(s, q.double().numpy(), host["k_packed"], host["k_norm"], host["v_packed"],
                       host["v_norm"], kb, vb, ctx, scale, thr, want_kept=kept)


CASES = [
    # B, Hq, Hkv, d, ctx, cap, kb, vb
    (1, 1, 1, 32, 1, 4, 4, 2),
    (2, 4, 2, 64, 33, 40, 4, 3),
    (1, 8, 2, 128, 257, 300, 4, 2),
    (2, 8, 8, 128, 31, 31, 2, 4),
    (3, 2, 2, 128, 2, 5, 3, 3),
    (1, 8, 1, 256, 513, 600, 3, 2),
    (2, 32, 8, 128, 1000, 1000, 4, 3),
    (1, 4, 1, 128, 5000, 5003, 4, 4),   # several splits and a ragged last split
    (1, 16, 2, 64, 3001, 3001, 3, 2),
    # d != 128 with at most 8 splits: merged inside a thread-block cluster
    (1, 8, 2, 64, 200, 210, 4, 2),      # 4 splits of 64
    (1, 4, 4, 256, 600, 600, 2, 3),     # 10 splits of 64 become 8 of 75
    (2, 8, 4, 256, 700, 700, 4, 4),     # 11 splits stay (split and combine launches)
]


@pytest.mark.parametrize("B,Hq,Hkv,d,ctx,cap,kb,vb", CASES)
def test_attention_parity(B, Hq, Hkv, d, ctx, cap, kb, vb):
    s, q, host, cache = make_case(B * 100 + ctx, B, Hq, Hkv, d, cap, kb, vb)
    plan = abi.Plan(d, 42)
    scale = 1.0 / math.sqrt(d)
    got = run(plan, q, cache, ctx, scale)
    want = oracle_out(s, q, host, kb, vb, ctx, scale)
    compare_attention(got, want)


@pytest.mark.parametrize("B,Hq,Hkv,d,ctx,cap,kb,vb", [CASES[2], CASES[6], CASES[7]])
def test_sparse_v(B, Hq, Hkv, d, ctx, cap, kb, vb):
    """Sparse-V at threshold 1e-4 matches both the sparse and the dense oracle;
    threshold 0 reproduces the dense GPU output bit for bit."""
    s, q, host, cache = make_case(7 + ctx, B, Hq, Hkv, d, cap, kb, vb, n_outliers=2)
    plan = abi.Plan(d, 42)
    scale = 1.0 / math.sqrt(d)
    q = (q.float() * 3).to(torch.bfloat16)  # sharper softmax: rows actually get skipped
    dense = run(plan, q, cache, ctx, scale)
    zero = run(plan, q, cache, ctx, scale, 0.0)
    assert np.array_equal(dense, zero)
    sparse = run(plan, q, cache, ctx, scale, 1e-4)
    want_sparse, kept = oracle_out(s, q, host, kb, vb, ctx, scale, 1e-4, kept=True)
    want_dense = oracle_out(s, q, host, kb, vb, ctx, scale)
    compare_attention(sparse, want_sparse)
    compare_attention(sparse, want_dense)
    assert kept.min() < ctx  # the oracle did drop rows


@pytest.mark.parametrize("B,Hq,Hkv,d,ctx,kb,vb", [(1, 32, 8, 128, 20000, 3, 2), (2, 8, 2, 128, 3001, 4, 3),
                                                  (1, 4, 1, 64, 3001, 3, 2)])
def test_sparse_v_skips_value_rows(B, Hq, Hkv, d, ctx, kb, vb):
    """A sharpened softmax (query x 6, keys with two x8 outlier channels): the
    sparse-V call reads the V rows of at most the context (at context 20000
    well under 80% of them), as tq_attn_decode_ex counts them per (batch, KV
    head), never fewer than any head of the group keeps in the oracle, and its
    output stays within the tolerance of both the sparse and the dense oracle.
    A dense call reads every row."""
    s, q, host, cache = make_case(11 + ctx, B, Hq, Hkv, d, ctx, kb, vb, n_outliers=2)
    plan = abi.Plan(d, 42)
    scale = 1.0 / math.sqrt(d)
    q = (q.float() * 6).to(torch.bfloat16)
    out_d, rows_d = abi.tq_attn_decode_ex(plan, q.cuda(), cache, ctx, scale, 0.0)
    out_s, rows_s = abi.tq_attn_decode_ex(plan, q.cuda(), cache, ctx, scale, 1e-4)
    torch.cuda.synchronize()
    rows_d, rows_s = rows_d.cpu().numpy(), rows_s.cpu().numpy()
    assert np.all(rows_d == ctx)
    assert np.all(rows_s <= ctx), rows_s
    if ctx >= 20000:  # enough chunks per CTA for the shared running maximum to settle
        assert rows_s.sum() < 0.8 * rows_s.size * ctx, rows_s
    want_sparse, kept = oracle_out(s, q, host, kb, vb, ctx, scale, 1e-4, kept=True)
    want_dense = oracle_out(s, q, host, kb, vb, ctx, scale)
    compare_attention(out_s.cpu().numpy(), want_sparse)
    compare_attention(out_s.cpu().numpy(), want_dense)
    compare_attention(out_d.cpu().numpy(), want_dense)
    G = Hq // Hkv
    assert np.all(kept.reshape(B, Hkv, G).max(axis=2) <= rows_s)
    print(f"sparse V, d {d} ctx {ctx}: V rows read {rows_s.tolist()} of {ctx}; oracle keeps per head "
          f"{kept.tolist()}")


def test_attention_errors():
    s, q, host, cache = make_case(3, 1, 4, 2, 128, 64, 4, 2)
    plan = abi.Plan(128, 42)
    with pytest.raises(abi.TQError, match="RANGE"):
        abi.tq_attn_decode(plan, q.cuda(), cache, 65, 0.1)
    need = abi.tq_attn_workspace_bytes(1, 4, 2, 128, 64)
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(abi.TQError, match="WORKSPACE"):
        abi.tq_attn_decode(plan, q.cuda(), cache, 64, 0.1, workspace=small)
