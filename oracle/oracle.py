"""ctypes binding of the plain-C double-precision oracle (``tq_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` import this module.  The library package
``kv_cache_vector_gb300`` never imports it, and this module never imports the
library: the two share no code.  Inputs reach both sides from the seeded
generators in ``kv_cache_vector_gb300.synth``, which hold none of the method's
arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from functools import lru_cache

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")

_u8p = ctypes.POINTER(ctypes.c_uint8)
_i8p = ctypes.POINTER(ctypes.c_int8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE double, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "tq_oracle.h"))
    ):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", _SO, _SRC, "-lm"]
        subprocess.check_call(cmd)
    return _SO


@lru_cache(maxsize=1)
def _lib():
    build()
    L = ctypes.CDLL(_SO)
    L.orc_splitmix64_next.restype = ctypes.c_uint64
    L.orc_splitmix64_next.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    L.orc_signs.argtypes = [ctypes.c_uint64, ctypes.c_int, _i8p]
    L.orc_fwht.argtypes = [_f64p, ctypes.c_int]
    L.orc_rotate.argtypes = [_i8p, _i8p, ctypes.c_int, _f64p, _f64p]
    L.orc_unrotate.argtypes = [_i8p, _i8p, ctypes.c_int, _f64p, _f64p]
    L.orc_codebook.restype = ctypes.c_int
    L.orc_codebook.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p]
    L.orc_codebook_mse.restype = ctypes.c_double
    L.orc_codebook_mse.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p]
    L.orc_codebook_gauss.restype = ctypes.c_int
    L.orc_codebook_gauss.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p]
    L.orc_codebook_gauss_mse.restype = ctypes.c_double
    L.orc_codebook_gauss_mse.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p]
    L.orc_density_mass.restype = ctypes.c_double
    L.orc_density_mass.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double]
    L.orc_bucket.restype = ctypes.c_int
    L.orc_bucket.argtypes = [ctypes.c_float, ctypes.c_int, _f32p]
    L.orc_pack.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p]
    L.orc_unpack.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p]
    L.orc_encode.argtypes = [_i8p, _i8p, ctypes.c_int, ctypes.c_int, _f32p, _f64p,
                             ctypes.c_int64, _u8p, _f32p, _f64p]
    L.orc_decode.argtypes = [_i8p, _i8p, ctypes.c_int, ctypes.c_int, _f32p, _u8p, _f32p,
                             ctypes.c_int64, _f64p]
    L.orc_attention.argtypes = [
        _i8p, _i8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_int, _f32p, _u8p, _f32p, ctypes.c_int, _f32p, _u8p,
        _f32p, _f64p, ctypes.c_double, ctypes.c_double, _f64p, _i64p]
    L.orc_attention_prefill.argtypes = [
        _i8p, _i8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
        ctypes.POINTER(ctypes.c_int32), ctypes.c_int, _f32p, _u8p, _f32p, ctypes.c_int, _f32p, _u8p, _f32p,
        _f64p, ctypes.c_double, _f64p]
    L.orc_qjl_matrix.argtypes = [ctypes.c_uint64, ctypes.c_int, _f64p]
    L.orc_encode_qjl.argtypes = [_i8p, _i8p, ctypes.c_int, ctypes.c_int, _f32p, _f32p, _f64p, _f64p,
                                 ctypes.c_int64, _u8p, _f32p, _f32p, _f64p]
    L.orc_decode_qjl.argtypes = [_i8p, _i8p, ctypes.c_int, ctypes.c_int, _f32p, _f64p, _u8p, _f32p, _f32p,
                                 ctypes.c_int64, _f64p]
    L.orc_attention_qjl.argtypes = [
        _i8p, _i8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int, _f32p, _f64p, _u8p, _f32p, _f32p, ctypes.c_int, _f32p, _u8p, _f32p, _f64p,
        ctypes.c_double, _f64p]
    return L


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous arrays"
    return a.ctypes.data_as(t)


def splitmix64_stream(seed: int, n: int) -> np.ndarray:
    st = ctypes.c_uint64(seed)
    return np.array([_lib().orc_splitmix64_next(ctypes.byref(st)) for _ in range(n)],
                    dtype=np.uint64)


def signs(seed: int, d: int) -> np.ndarray:
    s = np.empty(d, np.int8)
    _lib().orc_signs(ctypes.c_uint64(seed), d, _p(s, _i8p))
    return s


def signs2(seed: int, d: int) -> np.ndarray:
    """Second sign vector of the two-sided rotation ("CITATIONS", Two-sided
    Rademacher signs in WHT): outputs d .. 2d - 1 of the same splitmix64
    stream, s2_i = -1 iff the top bit is set."""
    s = np.empty(2 * d, np.int8)
    _lib().orc_signs(ctypes.c_uint64(seed), 2 * d, _p(s, _i8p))
    return np.ascontiguousarray(s[d:])


def _s2p(s2):
    return None if s2 is None else _p(np.ascontiguousarray(s2, np.int8), _i8p)


def fwht(v: np.ndarray) -> np.ndarray:
    out = np.ascontiguousarray(v, dtype=np.float64).copy()
    for row in out.reshape(-1, out.shape[-1]):
        _lib().orc_fwht(_p(row, _f64p), row.shape[0])
    return out


def rotate(s: np.ndarray, x: np.ndarray, s2: np.ndarray | None = None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    d = x.shape[-1]
    for xr, yr in zip(x.reshape(-1, d), y.reshape(-1, d)):
        _lib().orc_rotate(_p(s, _i8p), _s2p(s2), d, _p(xr, _f64p), _p(yr, _f64p))
    return y


def unrotate(s: np.ndarray, y: np.ndarray, s2: np.ndarray | None = None) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float64)
    x = np.empty_like(y)
    d = y.shape[-1]
    for yr, xr in zip(y.reshape(-1, d), x.reshape(-1, d)):
        _lib().orc_unrotate(_p(s, _i8p), _s2p(s2), d, _p(yr, _f64p), _p(xr, _f64p))
    return x


@lru_cache(maxsize=None)
def codebook(d: int, bits: int, kind: str = "sphere"):
    """(centroids[2^b], boundaries[2^b - 1], iterations), double precision.
    kind "sphere": the exact coordinate density; "gauss": N(0, 1/d)."""
    L = 1 << bits
    c = np.empty(L, np.float64)
    b = np.empty(L - 1, np.float64)
    fn = {"sphere": _lib().orc_codebook, "gauss": _lib().orc_codebook_gauss}[kind]
    it = fn(d, bits, _p(c, _f64p), _p(b, _f64p))
    if it < 0:
        raise RuntimeError(f"oracle codebook failed for d={d} bits={bits}")
    c.setflags(write=False)
    b.setflags(write=False)
    return c, b, it


def codebook_f32(d: int, bits: int, kind: str = "sphere"):
    """The stored (fp32) form of the codebook."""
    c, b, _ = codebook(d, bits, kind)
    return c.astype(np.float32), b.astype(np.float32)


def codebook_mse(d: int, bits: int, c: np.ndarray, b: np.ndarray, kind: str = "sphere") -> float:
    c = np.ascontiguousarray(c, np.float64)
    b = np.ascontiguousarray(b, np.float64)
    fn = {"sphere": _lib().orc_codebook_mse, "gauss": _lib().orc_codebook_gauss_mse}[kind]
    return fn(d, bits, _p(c, _f64p), _p(b, _f64p))


def density_mass(d: int, a: float, b: float) -> float:
    return _lib().orc_density_mass(d, a, b)


def bucket(u: float, bits: int, boundaries: np.ndarray) -> int:
    bf = np.ascontiguousarray(boundaries, np.float32)
    return _lib().orc_bucket(ctypes.c_float(u), bits, _p(bf, _f32p))


def pack(idx: np.ndarray, bits: int) -> np.ndarray:
    idx = np.ascontiguousarray(idx, np.uint8)
    d = idx.shape[-1]
    out = np.empty(idx.shape[:-1] + (d * bits // 8,), np.uint8)
    for ir, orow in zip(idx.reshape(-1, d), out.reshape(-1, d * bits // 8)):
        _lib().orc_pack(_p(ir, _u8p), d, bits, _p(orow, _u8p))
    return out


def unpack(packed: np.ndarray, d: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8)
    rb = d * bits // 8
    out = np.empty(packed.shape[:-1] + (d,), np.uint8)
    for pr, orow in zip(packed.reshape(-1, rb), out.reshape(-1, d)):
        _lib().orc_unpack(_p(pr, _u8p), d, bits, _p(orow, _u8p))
    return out


def encode(s: np.ndarray, bits: int, x: np.ndarray, want_u: bool = False, s2: np.ndarray | None = None,
           kind: str = "sphere"):
    """x: [n, d] (any real dtype; converted exactly to double).
    Returns packed [n, d*bits/8] uint8, norms [n] float32 (and u [n, d]).
    s2: the second signs of a two-sided rotation; kind: the codebook."""
    x = np.ascontiguousarray(x, np.float64)
    n, d = x.shape
    _, bnd = codebook_f32(d, bits, kind)
    packed = np.empty((n, d * bits // 8), np.uint8)
    norms = np.empty(n, np.float32)
    u = np.empty((n, d), np.float64) if want_u else None
    _lib().orc_encode(_p(s, _i8p), _s2p(s2), d, bits, _p(bnd, _f32p), _p(x, _f64p), n,
                      _p(packed, _u8p), _p(norms, _f32p),
                      _p(u, _f64p) if want_u else None)
    return (packed, norms, u) if want_u else (packed, norms)


def decode(s: np.ndarray, bits: int, packed: np.ndarray, norms: np.ndarray, s2: np.ndarray | None = None,
           kind: str = "sphere") -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8)
    norms = np.ascontiguousarray(norms, np.float32)
    n = norms.shape[0]
    d = packed.shape[-1] * 8 // bits
    cen, _ = codebook_f32(d, bits, kind)
    out = np.empty((n, d), np.float64)
    _lib().orc_decode(_p(s, _i8p), _s2p(s2), d, bits, _p(cen, _f32p), _p(packed, _u8p),
                      _p(norms, _f32p), n, _p(out, _f64p))
    return out


def attention(s, q, k_packed, k_norm, v_packed, v_norm, k_bits, v_bits, ctx_len,
              scale, sparse_thr=0.0, want_kept=False, s2=None, kind="sphere"):
    """q: [B, Hq, d]; k_packed: [B, Hkv, cap, d*kb/8]; k_norm: [B, Hkv, cap]."""
    q = np.ascontiguousarray(q, np.float64)
    B, Hq, d = q.shape
    Hkv, cap = k_norm.shape[1], k_norm.shape[2]
    kc, _ = codebook_f32(d, k_bits, kind)
    vc, _ = codebook_f32(d, v_bits, kind)
    k_packed = np.ascontiguousarray(k_packed, np.uint8)
    v_packed = np.ascontiguousarray(v_packed, np.uint8)
    k_norm = np.ascontiguousarray(k_norm, np.float32)
    v_norm = np.ascontiguousarray(v_norm, np.float32)
    out = np.empty((B, Hq, d), np.float64)
    kept = np.empty((B, Hq), np.int64)
    _lib().orc_attention(_p(s, _i8p), _s2p(s2), d, B, Hq, Hkv, cap, ctx_len, k_bits,
                         _p(kc, _f32p), _p(k_packed, _u8p), _p(k_norm, _f32p),
                         v_bits, _p(vc, _f32p), _p(v_packed, _u8p), _p(v_norm, _f32p),
                         _p(q, _f64p), float(scale), float(sparse_thr), _p(out, _f64p),
                         _p(kept, _i64p))
    return (out, kept) if want_kept else out


def attention_prefill(s, q, k_packed, k_norm, v_packed, v_norm, k_bits, v_bits, q_start, scale, s2=None,
                      kind="sphere"):
    """Prefill attention, plain definition. q: [B, T, Hq, d]; k_packed:
    [B, Hkv, cap, d*kb/8]; q_start: [B] (token t of sequence b sits at
    q_start[b] + t and attends causally). Returns [B, T, Hq, d]."""
    q = np.ascontiguousarray(q, np.float64)
    B, T, Hq, d = q.shape
    Hkv, cap = k_norm.shape[1], k_norm.shape[2]
    kc, _ = codebook_f32(d, k_bits, kind)
    vc, _ = codebook_f32(d, v_bits, kind)
    qs = np.ascontiguousarray(q_start, np.int32)
    assert np.all(qs >= 0) and np.all(qs + T <= cap)
    k_packed = np.ascontiguousarray(k_packed, np.uint8)
    v_packed = np.ascontiguousarray(v_packed, np.uint8)
    k_norm = np.ascontiguousarray(k_norm, np.float32)
    v_norm = np.ascontiguousarray(v_norm, np.float32)
    out = np.empty((B, T, Hq, d), np.float64)
    _lib().orc_attention_prefill(_p(s, _i8p), _s2p(s2), d, B, T, Hq, Hkv, cap,
                                 qs.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), k_bits,
                                 _p(kc, _f32p), _p(k_packed, _u8p), _p(k_norm, _f32p),
                                 v_bits, _p(vc, _f32p), _p(v_packed, _u8p), _p(v_norm, _f32p),
                                 _p(q, _f64p), float(scale), _p(out, _f64p))
    return out


# ------------------------------------------------------------ QJL residual keys
# Reading ("CITATIONS", Google TurboQuant entry; "TurboQuant KV Cache
# Compression -- Spec", Why not QJL?): b bits = a (b - 1)-bit MSE index per
# coordinate plus one sign of a Gaussian projection of the rotated residual per
# coordinate; the residual norm gamma rides beside the row norm.  Full
# statement in tq_oracle.h.

def qjl_matrix(seed: int, d: int) -> np.ndarray:
    """The d x d Gaussian projection S drawn from the plan seed's stream."""
    S = np.empty((d, d), np.float64)
    _lib().orc_qjl_matrix(ctypes.c_uint64(seed), d, _p(S, _f64p))
    return S


def encode_qjl(s: np.ndarray, bits: int, x: np.ndarray, S: np.ndarray, s2: np.ndarray | None = None,
               kind: str = "sphere", want_proj: bool = False):
    """x: [n, d]. Returns packed [n, d*bits/8] uint8, norms [n] and gamma [n]
    (float32), and with want_proj the projections S r [n, d] in double."""
    x = np.ascontiguousarray(x, np.float64)
    n, d = x.shape
    assert 2 <= bits and (d * (bits - 1)) % 8 == 0
    cen, bnd = codebook_f32(d, bits - 1, kind)
    S = np.ascontiguousarray(S, np.float64)
    packed = np.empty((n, d * bits // 8), np.uint8)
    norms = np.empty(n, np.float32)
    rnorms = np.empty(n, np.float32)
    proj = np.empty((n, d), np.float64) if want_proj else None
    _lib().orc_encode_qjl(_p(s, _i8p), _s2p(s2), d, bits, _p(cen, _f32p), _p(bnd, _f32p), _p(S, _f64p),
                          _p(x, _f64p), n, _p(packed, _u8p), _p(norms, _f32p), _p(rnorms, _f32p),
                          _p(proj, _f64p) if want_proj else None)
    return (packed, norms, rnorms, proj) if want_proj else (packed, norms, rnorms)


def decode_qjl(s: np.ndarray, bits: int, packed: np.ndarray, norms: np.ndarray, rnorms: np.ndarray,
               S: np.ndarray, s2: np.ndarray | None = None, kind: str = "sphere") -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8)
    norms = np.ascontiguousarray(norms, np.float32)
    rnorms = np.ascontiguousarray(rnorms, np.float32)
    n = norms.shape[0]
    d = packed.shape[-1] * 8 // bits
    cen, _ = codebook_f32(d, bits - 1, kind)
    S = np.ascontiguousarray(S, np.float64)
    out = np.empty((n, d), np.float64)
    _lib().orc_decode_qjl(_p(s, _i8p), _s2p(s2), d, bits, _p(cen, _f32p), _p(S, _f64p), _p(packed, _u8p),
                          _p(norms, _f32p), _p(rnorms, _f32p), n, _p(out, _f64p))
    return out


def attention_qjl(s, q, k_packed, k_norm, k_rnorm, S, v_packed, v_norm, k_bits, v_bits, ctx_len, scale,
                  s2=None, kind="sphere"):
    """Dense decode attention with QJL keys. q: [B, Hq, d]; k_packed:
    [B, Hkv, cap, d*kb/8]; k_norm, k_rnorm: [B, Hkv, cap]; values plain."""
    q = np.ascontiguousarray(q, np.float64)
    B, Hq, d = q.shape
    Hkv, cap = k_norm.shape[1], k_norm.shape[2]
    kc, _ = codebook_f32(d, k_bits - 1, kind)
    vc, _ = codebook_f32(d, v_bits, kind)
    k_packed = np.ascontiguousarray(k_packed, np.uint8)
    v_packed = np.ascontiguousarray(v_packed, np.uint8)
    k_norm = np.ascontiguousarray(k_norm, np.float32)
    k_rnorm = np.ascontiguousarray(k_rnorm, np.float32)
    v_norm = np.ascontiguousarray(v_norm, np.float32)
    S = np.ascontiguousarray(S, np.float64)
    out = np.empty((B, Hq, d), np.float64)
    _lib().orc_attention_qjl(_p(s, _i8p), _s2p(s2), d, B, Hq, Hkv, cap, ctx_len, k_bits, _p(kc, _f32p),
                             _p(S, _f64p), _p(k_packed, _u8p), _p(k_norm, _f32p), _p(k_rnorm, _f32p),
                             v_bits, _p(vc, _f32p), _p(v_packed, _u8p), _p(v_norm, _f32p), _p(q, _f64p),
                             float(scale), _p(out, _f64p))
    return out
