"""Parity checks shared by the GPU tests and the bench: library output vs the
oracle on the same seeded input bytes, with the tolerances the method states.

* indices / bytes: bit-exact, except coordinates whose normalised value u (the
  oracle's, in double) lies within 1e-6 of a boundary; the fraction of such
  disagreements must stay below 1e-5.
* norms: relative 1e-5.
* decoded values: per row max |y - y_oracle| <= 1e-5 * ||y_oracle|| / sqrt(d)
  (plus one bf16 unit in the last place for bf16 output).
* attention outputs: 2e-3 absolute per element.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import oracle as O

NEAR_BOUNDARY = 1e-6
MAX_DISAGREE_FRACTION = 1e-5
NORM_RTOL = 1e-5
DECODE_REL = 1e-5
ATTN_ATOL = 2e-3


def compare_encode(s, bits, x64, gpu_packed, gpu_norms, s2=None, kind="sphere"):
    """Returns a dict of statistics; raises AssertionError on a violation.
    s2 / kind: the plan's format variant (second signs, codebook kind)."""
    n, d = x64.shape
    opk, onm, u = O.encode(s, bits, x64, want_u=True, s2=s2, kind=kind)
    gi = O.unpack(gpu_packed, d, bits)
    oi = O.unpack(opk, d, bits)
    diff = gi != oi
    ndiff = int(diff.sum())
    _, bnd = O.codebook_f32(d, bits, kind)
    dist = np.min(np.abs(u[..., None] - bnd.astype(np.float64)), axis=-1)
    near_pop = float((dist <= NEAR_BOUNDARY).mean())
    if ndiff:
        worst = float(dist[diff].max())
        assert worst <= NEAR_BOUNDARY, f"index differs {worst:.3g} away from any boundary"
        assert ndiff / diff.size < MAX_DISAGREE_FRACTION, f"{ndiff} of {diff.size} indices differ"
    same_rows = ~diff.any(axis=1)
    assert np.array_equal(gpu_packed[same_rows], opk[same_rows]), "packed bytes differ"
    assert np.allclose(gpu_norms, onm, rtol=NORM_RTOL, atol=0), \
        f"norms differ: max rel {np.max(np.abs(gpu_norms - onm) / np.maximum(onm, 1e-30)):.3g}"
    return {"coords": int(diff.size), "disagree": ndiff, "disagree_fraction": ndiff / diff.size,
            "near_boundary_population": near_pop}


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1e-38)))
    return np.where(ax > 0, 2.0 ** (e - 7), 2.0 ** -133)


def compare_decode(s, bits, packed, norms, gpu_out, bf16: bool, s2=None, kind="sphere"):
    n = norms.shape[0]
    want = O.decode(s, bits, packed, norms, s2=s2, kind=kind)
    d = want.shape[1]
    got = gpu_out.astype(np.float64)
    tol = DECODE_REL * np.linalg.norm(want, axis=1, keepdims=True) / math.sqrt(d)
    if bf16:
        tol = tol + bf16_ulp(want)
    err = np.abs(got - want)
    assert np.all(err <= tol), f"decode error {float((err / np.maximum(tol, 1e-300)).max()):.3g} x tolerance"
    return {"rows": n, "max_err_over_tol": float((err / np.maximum(tol, 1e-300)).max())}


def compare_attention(got, want):
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(err <= ATTN_ATOL), f"attention max abs error {err.max():.3g}"
    return {"max_abs_err": float(err.max())}
