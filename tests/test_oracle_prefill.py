"""Pins of the oracle's prefill (multi-query, causal) attention against a
scipy restatement over the oracle's (separately pinned) row decode, closed
forms (one position gives the V row, scale 0 gives the mean of the rows
attended) and causality.  CPU only."""
import math

import numpy as np
import pytest
import scipy.special

from kv_cache_vector_gb300 import synth
from oracle import oracle as O


def _cache(seed, B, Hkv, cap, d, kb, vb, s, s2=None, kind="sphere"):
    kx = synth.normal_rows(seed, B * Hkv * cap, d, stream=1).double().numpy()
    vx = synth.normal_rows(seed, B * Hkv * cap, d, stream=2).double().numpy()
    kp, kn = O.encode(s, kb, kx, s2=s2, kind=kind)
    vp, vn = O.encode(s, vb, vx, s2=s2, kind=kind)
    return kp.reshape(B, Hkv, cap, -1), kn.reshape(B, Hkv, cap), vp.reshape(B, Hkv, cap, -1), vn.reshape(B, Hkv, cap)


@pytest.mark.parametrize("two_sided", [False, True])
def test_prefill_matches_scipy_restatement(two_sided):
    d, B, T, Hq, Hkv, cap, kb, vb = 32, 2, 5, 4, 2, 12, 4, 2
    s = O.signs(5, d)
    s2 = O.signs2(5, d) if two_sided else None
    kp, kn, vp, vn = _cache(3, B, Hkv, cap, d, kb, vb, s, s2)
    q = synth.normal_rows(4, B * T * Hq, d).double().numpy().reshape(B, T, Hq, d)
    q_start = np.array([0, 7], np.int32)
    scale = 1 / math.sqrt(d)
    got = O.attention_prefill(s, q, kp, kn, vp, vn, kb, vb, q_start, scale, s2=s2)
    G = Hq // Hkv
    for b in range(B):
        for g in range(Hkv):
            K = O.decode(s, kb, kp[b, g], kn[b, g], s2=s2)
            V = O.decode(s, vb, vp[b, g], vn[b, g], s2=s2)
            for t in range(T):
                n = q_start[b] + t + 1
                for hh in range(G):
                    h = g * G + hh
                    p = scipy.special.softmax(scale * (K[:n] @ q[b, t, h]))
                    assert np.allclose(got[b, t, h], p @ V[:n], atol=1e-12)


def test_prefill_closed_forms_and_causality():
    d, B, T, Hq, Hkv, cap, kb, vb = 16, 1, 4, 2, 1, 8, 3, 3
    s = O.signs(9, d)
    kp, kn, vp, vn = _cache(8, B, Hkv, cap, d, kb, vb, s)
    q = synth.normal_rows(10, B * T * Hq, d).double().numpy().reshape(B, T, Hq, d)
    V = O.decode(s, vb, vp[0, 0], vn[0, 0])
    # token 0 at position 0 attends over one row: the output is that V row
    out = O.attention_prefill(s, q, kp, kn, vp, vn, kb, vb, np.array([0], np.int32), 0.3)
    for h in range(Hq):
        assert np.allclose(out[0, 0, h], V[0], atol=1e-13)
    # scale 0: uniform weights, the mean of rows [0, q_start + t]
    out0 = O.attention_prefill(s, q, kp, kn, vp, vn, kb, vb, np.array([2], np.int32), 0.0)
    for t in range(T):
        assert np.allclose(out0[0, t, 0], V[:2 + t + 1].mean(0), atol=1e-13)
    # causality: rows after a token's position do not change its output
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[0, 0, 4:] ^= 0x5A
    vp2[0, 0, 4:] ^= 0xA5
    a = O.attention_prefill(s, q, kp, kn, vp, vn, kb, vb, np.array([1], np.int32), 0.25)
    c = O.attention_prefill(s, q, kp2, kn, vp2, vn, kb, vb, np.array([1], np.int32), 0.25)
    assert np.array_equal(a[0, :3], c[0, :3])      # positions 1..3 reach rows <= 3
    assert not np.allclose(a[0, 3], c[0, 3])       # position 4 reads the changed row
