"""CPU tests of the C ABI: the library loads and exports what include/tq.h
declares; its host-side parts (codebook, signs, argument validation, the
bucketing-table geometry) agree with the oracle and the header.  No kernel is
launched here."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from kv_cache_vector_gb300 import abi
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from kv_cache_vector_gb300 import build
    build.build()
    return abi.lib()


def test_exports_every_declared_symbol(L):
    hdr = open(os.path.join(ROOT, "include", "tq.h")).read()
    declared = set(re.findall(r"\b(tq_[a-z_0-9]+)\s*\(", hdr))
    assert declared == set(abi.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


@pytest.mark.parametrize("d", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_matches_oracle(L, d, bits):
    """The library's codebook (closed-form cell masses) and the oracle's
    (Gauss-Legendre) are independent computations of the same fixed point."""
    c, b = abi.tq_codebook_init(d, bits)
    oc, ob, _ = O.codebook(d, bits)
    scale = 1.0 / math.sqrt(d)
    assert np.max(np.abs(c - oc)) < 1e-12 * scale
    assert np.max(np.abs(b - ob)) < 1e-12 * scale
    assert np.array_equal(c.astype(np.float32), oc.astype(np.float32))
    assert np.array_equal(b.astype(np.float32), ob.astype(np.float32))


@pytest.mark.parametrize("seed", [0, 42, 2**63 + 5])
@pytest.mark.parametrize("d", [8, 128, 256])
def test_plan_signs_and_codebooks(L, seed, d):
    p = abi.Plan(d, seed)
    assert np.array_equal(p.signs(), O.signs(seed, d))
    for bits in (2, 3, 4):
        c, b = p.codebook(bits)
        oc, ob = O.codebook_f32(d, bits)
        assert np.array_equal(c, oc) and np.array_equal(b, ob)
    p.close()


@pytest.mark.parametrize("d", [1, 8, 64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_gaussian_codebook_matches_oracle(L, d, bits):
    """N(0, 1/d) codebooks: the library's (positive half, mirrored) and the
    oracle's (all cells) agree to rounding, and identically after fp32."""
    c, b = abi.tq_codebook_init_gaussian(d, bits)
    oc, ob, _ = O.codebook(d, bits, "gauss")
    scale = 1.0 / math.sqrt(d)
    assert np.max(np.abs(c - oc)) < 1e-12 * scale
    assert np.max(np.abs(b - ob)) < 1e-12 * scale
    assert np.array_equal(c.astype(np.float32), oc.astype(np.float32))
    assert np.array_equal(b.astype(np.float32), ob.astype(np.float32))


@pytest.mark.parametrize("flags", [1, 2, 3])
@pytest.mark.parametrize("d", [8, 128, 256])
def test_plan_format_variants(L, flags, d):
    """Plan flags: the codebook kind and the second sign vector follow the
    oracle's definitions; s1 does not change."""
    p = abi.Plan(d, 42, flags)
    kind = "gauss" if flags & abi.PLAN_GAUSSIAN_CODEBOOK else "sphere"
    assert np.array_equal(p.signs(), O.signs(42, d))
    want2 = O.signs2(42, d) if flags & abi.PLAN_TWO_SIDED_SIGNS else np.ones(d, np.int8)
    assert np.array_equal(p.signs2(), want2)
    for bits in (2, 3, 4):
        c, b = p.codebook(bits)
        oc, ob = O.codebook_f32(d, bits, kind)
        assert np.array_equal(c, oc) and np.array_equal(b, ob)
    p.close()


def test_codebook_and_plan_argument_errors(L):
    c = np.empty(16)
    b = np.empty(15)
    assert L.tq_codebook_init(2, 4, c.ctypes.data, b.ctypes.data) == 2
    assert L.tq_codebook_init(128, 5, c.ctypes.data, b.ctypes.data) == 2
    assert L.tq_codebook_init(128, 4, None, b.ctypes.data) == 1
    h = ctypes.c_void_p()
    for d in (0, 4, 96, 512):
        assert L.tq_plan_create(d, 1, ctypes.byref(h)) == 2
    assert L.tq_plan_create(128, 1, None) == 1
    assert L.tq_plan_create_ex(128, 1, 4, ctypes.byref(h)) == 2  # unknown flag bit
    assert L.tq_plan_create_ex(96, 1, 1, ctypes.byref(h)) == 2
    assert L.tq_codebook_init_gaussian(0, 2, c.ctypes.data, b.ctypes.data) == 2
    assert L.tq_codebook_init_gaussian(128, 5, c.ctypes.data, b.ctypes.data) == 2
    assert L.tq_plan_signs2(None, c.ctypes.data) == 1
    assert L.tq_status_string(0) == b"ok"


def test_hot_call_validation_before_launch(L):
    """Wrong arguments come back as status codes; none of these reaches CUDA."""
    p = abi.Plan(128, 42)
    h = p.handle
    A = 1 << 20  # a 16-byte aligned address (never dereferenced)
    s = None
    assert L.tq_encode(None, 4, A, 1, 8, A, A, s) == 1
    assert L.tq_encode(h, 5, A, 1, 8, A, A, s) == 2
    assert L.tq_encode(h, 4, A, 7, 8, A, A, s) == 2
    assert L.tq_encode(h, 4, A, 1, -1, A, A, s) == 1
    assert L.tq_encode(h, 4, A, 1, 0, None, None, s) == 0   # empty: no-op
    assert L.tq_encode(h, 4, None, 1, 8, A, A, s) == 1
    assert L.tq_encode(h, 4, A + 8, 1, 8, A, A, s) == 3
    assert L.tq_encode(h, 4, A, 1, 8, A + 4, A, s) == 3
    assert L.tq_decode(h, 1, A, A, 8, A, 0, s) == 2
    assert L.tq_decode(h, 4, A, A, 8, A + 2, 0, s) == 3
    cv = abi.CacheView(A, A, A, A, 16)
    assert L.tq_append(h, 4, 2, A, A, 1, 1, 2, 1, cv, 16, s) == 4      # pos == cap
    assert L.tq_append(h, 4, 2, A, A, 1, 1, 2, 4, cv, 13, s) == 4      # runs past cap
    assert L.tq_append(h, 4, 2, A, A, 1, 1, 2, 1, cv, -1, s) == 4
    assert L.tq_append(h, 4, 9, A, A, 1, 1, 2, 1, cv, 0, s) == 2
    f = ctypes.c_float
    assert L.tq_attn_decode(h, A, 1, 6, 4, cv, 8, 4, 2, f(1.0), f(0.0), A, A, 1 << 20, s) == 1
    assert L.tq_attn_decode(h, A, 1, 32, 2, cv, 8, 4, 2, f(1.0), f(0.0), A, A, 1 << 20, s) == 2
    assert L.tq_attn_decode(h, A, 1, 8, 2, cv, 0, 4, 2, f(1.0), f(0.0), A, A, 1 << 20, s) == 4
    assert L.tq_attn_decode(h, A, 1, 8, 2, cv, 17, 4, 2, f(1.0), f(0.0), A, A, 1 << 20, s) == 4
    assert L.tq_attn_decode(h, A, 1, 8, 2, cv, 8, 4, 2, f(1.0), f(-1.0), A, A, 1 << 20, s) == 1
    assert L.tq_attn_workspace_bytes(1, 6, 4, 128, 8) == 0
    assert L.tq_attn_paged_workspace_bytes(1, 6, 4, 128, 8) == 0
    assert L.tq_attn_paged_workspace_bytes(1, 8, 2, 64, 8) > 0    # d = 64: the generic kernel
    assert L.tq_attn_paged_workspace_bytes(1, 8, 2, 16, 8) == 0   # no attention below d = 32
    p.close()


def _emulate_table_bucket(bnd32: np.ndarray, w: np.ndarray, S: int = 256, C: int = 512,
                          N: int = 1024) -> np.ndarray:
    """numpy restatement of the kernels' bucketing table: cell = rint(w*S)
    (round half even, exact), lo = #{beta < cell_lo}, thr = the boundary in the
    closed cell, idx = lo + [w >= thr].  Defaults: the 1024-cell table; the
    d = 128 tensor-core encoder's is S = 64 with one byte of cell (C = 128,
    N = 256)."""
    g = np.arange(N)
    lo = ((g - C - 0.5) / S).astype(np.float32).astype(np.float64)
    hi = ((g - C + 0.5) / S).astype(np.float32).astype(np.float64)
    b = bnd32.astype(np.float64)
    cnt = (b[None, :] < lo[:, None]).sum(1)
    inside = (b[None, :] >= lo[:, None]) & (b[None, :] <= hi[:, None])
    assert inside.sum(1).max() <= 1
    thr = np.full(N, np.inf)
    rows, cols = np.nonzero(inside)
    thr[rows] = b[cols]
    cell = (np.rint(w.astype(np.float64) * S).astype(np.int64) + C) & (N - 1)
    return cnt[cell] + (w.astype(np.float64) >= thr[cell])


@pytest.mark.parametrize("d", [8, 32, 128, 256])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_bucketing_table_is_exact(L, d, bits):
    """The table the encode kernels build gives #{j : w >= beta_j} for every
    fp32 w a finite row can produce (|w| <= |y_i| / (sqrt(d) n) <= 1, plus
    rounding): checked on boundaries, their neighbours, cell edges and a dense
    random sweep."""
    p = abi.Plan(d, 1)
    _, bnd = p.codebook(bits)
    rng = np.random.default_rng(d + bits)
    edges = ((np.arange(-265, 265) + 0.5) / 256).astype(np.float32)
    w = np.concatenate([
        bnd, np.nextafter(bnd, np.float32(-9)), np.nextafter(bnd, np.float32(9)),
        edges, np.nextafter(edges, np.float32(-9)), np.nextafter(edges, np.float32(9)),
        rng.normal(0, 1 / math.sqrt(d), 200000).astype(np.float32),
        rng.uniform(-1, 1, 200000).astype(np.float32), np.array([0.0, -0.0, 1.0, -1.0], np.float32)])
    want = np.searchsorted(bnd, w, side="right")
    assert np.array_equal(_emulate_table_bucket(bnd, w), want)
    p.close()


@pytest.mark.parametrize("gauss", [False, True])
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("d", [128, 256])
def test_tensor_core_encoder_table_is_exact(L, d, bits, gauss):
    """The tensor-core encoders' table (d = 128 and 256: cells of width 1/64,
    one byte of cell index, no window) gives #{j : w >= beta_j} for every fp32
    w in [-1, 1] plus rounding, with no cell index outside 64 .. 192."""
    p = abi.Plan(d, 1, abi.PLAN_GAUSSIAN_CODEBOOK) if gauss else abi.Plan(d, 1)
    _, bnd = p.codebook(bits)
    rng = np.random.default_rng(d + bits + gauss)
    edges = ((np.arange(-64, 64) + 0.5) / 64).astype(np.float32)
    w = np.concatenate([
        bnd, np.nextafter(bnd, np.float32(-9)), np.nextafter(bnd, np.float32(9)),
        edges, np.nextafter(edges, np.float32(-9)), np.nextafter(edges, np.float32(9)),
        rng.normal(0, 1 / math.sqrt(d), 200000).astype(np.float32),
        rng.uniform(-1, 1, 200000).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, np.nextafter(np.float32(1), np.float32(2)),
                  np.nextafter(np.float32(-1), np.float32(-2))], np.float32)])
    cell = np.rint(w.astype(np.float64) * 64).astype(np.int64) + 128
    assert cell.min() >= 64 and cell.max() <= 192
    want = np.searchsorted(bnd, w, side="right")
    assert np.array_equal(_emulate_table_bucket(bnd, w, 64, 128, 256), want)
    p.close()


def test_paged_call_validation_before_launch(L):
    """The paged entry points check their arguments on the host and return
    status codes before any launch."""
    p128, p64, p16 = abi.Plan(128, 42), abi.Plan(64, 42), abi.Plan(16, 42)
    A = 1 << 20
    s = None
    f = ctypes.c_float

    def pc(n_pages=4, page_size=64):
        return abi.PagedCacheView(A, A, A, A, n_pages, page_size)

    h = p128.handle
    # tq_append_paged(plan, kb, vb, k_new, v_new, dtype, B, Hkv, cache, bt, max_pages, positions, s)
    assert L.tq_append_paged(None, 4, 2, A, A, 1, 2, 2, pc(), A, 4, A, s) == 1
    assert L.tq_append_paged(h, 5, 2, A, A, 1, 2, 2, pc(), A, 4, A, s) == 2
    assert L.tq_append_paged(h, 4, 2, A, A, 1, 2, 2, pc(page_size=48), A, 4, A, s) == 2
    assert L.tq_append_paged(h, 4, 2, A, A, 1, 2, 2, pc(page_size=16), A, 4, A, s) == 2
    assert L.tq_append_paged(p16.handle, 4, 2, A, A, 1, 2, 2, pc(), A, 4, A, s) == 2
    assert L.tq_append_paged(h, 4, 2, A, A, 1, 2, 2, pc(), A, 0, A, s) == 1
    assert L.tq_append_paged(h, 4, 2, A, A, 1, 2, 2, pc(n_pages=0), A, 4, A, s) == 1
    assert L.tq_append_paged(h, 4, 2, A, A, 1, 0, 2, pc(), None, 4, None, s) == 0  # B = 0: no-op
    assert L.tq_append_paged(h, 4, 2, A, A, 1, 2, 2, pc(), None, 4, A, s) == 1
    assert L.tq_append_paged(h, 4, 2, A + 8, A, 1, 2, 2, pc(), A, 4, A, s) == 3
    assert L.tq_append_paged(h, 4, 2, A, A, 1, 2, 2, pc(), A, 4, A + 2, s) == 3
    # tq_attn_decode_paged(plan, q, B, Hq, Hkv, cache, bt, max_pages, lens, max_ctx, kb, vb,
    #                      scale, thr, out, ws, ws_bytes, s)
    W = 1 << 24
    assert L.tq_attn_decode_paged(h, A, 1, 6, 4, pc(), A, 4, A, 100, 4, 3, f(1.0), f(0.0), A, A, W, s) == 1
    assert L.tq_attn_decode_paged(h, A, 1, 32, 2, pc(), A, 4, A, 100, 4, 3, f(1.0), f(0.0), A, A, W, s) == 2
    # d = 64 runs the generic kernel: its workspace check still comes before any launch
    assert L.tq_attn_decode_paged(p64.handle, A, 1, 8, 2, pc(), A, 4, A, 100, 4, 3, f(1.0), f(0.0), A, A, 16,
                                  s) == 5
    assert L.tq_attn_decode_paged(p16.handle, A, 1, 8, 2, pc(), A, 4, A, 100, 4, 3, f(1.0), f(0.0), A, A, W,
                                  s) == 2
    assert L.tq_attn_decode_paged(h, A, 1, 8, 2, pc(page_size=100), A, 4, A, 100, 4, 3, f(1.0), f(0.0), A,
                                  A, W, s) == 2
    assert L.tq_attn_decode_paged(h, A, 1, 8, 2, pc(), A, 4, A, 0, 4, 3, f(1.0), f(0.0), A, A, W, s) == 4
    assert L.tq_attn_decode_paged(h, A, 1, 8, 2, pc(), A, 4, A, 257, 4, 3, f(1.0), f(0.0), A, A, W, s) == 4
    assert L.tq_attn_decode_paged(h, A, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(-1.0), A, A, W, s) == 1
    assert L.tq_attn_decode_paged(h, A, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, 16, s) == 5
    assert L.tq_attn_decode_paged(h, A + 4, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, W,
                                  s) == 3
    assert L.tq_attn_decode_paged(h, A, 0, 8, 2, pc(), None, 4, None, 256, 4, 3, f(1.0), f(0.0), None,
                                  None, 0, s) == 0  # B = 0: no-op
    # tq_attn_decode_append_paged(plan, q, k_new, v_new, kv_dtype, B, Hq, Hkv, cache, bt, max_pages,
    #                             positions, max_ctx, kb, vb, scale, thr, out, ws, ws_bytes, s)
    fa = L.tq_attn_decode_append_paged
    assert fa(None, A, A, A, 1, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, W, s) == 1
    assert fa(h, A, A, A, 7, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, W, s) == 2  # dtype
    assert fa(h, A, A, A, 1, 1, 32, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, W, s) == 2  # GQA 16
    assert fa(p16.handle, A, A, A, 1, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, W, s) == 2
    assert fa(h, A, A, A, 1, 1, 8, 2, pc(), A, 4, A, 257, 4, 3, f(1.0), f(0.0), A, A, W, s) == 4
    assert fa(h, A, A, A, 1, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, 16, s) == 5
    assert fa(h, A, A + 8, A, 1, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, W, s) == 3
    assert fa(h, A, A, None, 1, 1, 8, 2, pc(), A, 4, A, 256, 4, 3, f(1.0), f(0.0), A, A, W, s) == 1
    assert fa(h, A, None, None, 1, 0, 8, 2, pc(), None, 4, None, 256, 4, 3, f(1.0), f(0.0), None, None, 0,
              s) == 0  # B = 0: no-op


def test_prefill_call_validation_before_launch(L):
    """tq_attn_prefill checks its arguments on the host before any launch."""
    p128, p64 = abi.Plan(128, 42), abi.Plan(64, 42)
    h = p128.handle
    A = 1 << 20
    f = ctypes.c_float
    cv = abi.CacheView(A, A, A, A, 256)
    W = 1 << 24
    # tq_attn_prefill(plan, q, B, T, Hq, Hkv, cache, q_start, kb, vb, scale, out, ws, ws_bytes, s)
    assert L.tq_attn_prefill(None, A, 1, 8, 8, 2, cv, A, 4, 3, f(1.0), A, A, W, None) == 1
    assert L.tq_attn_prefill(h, A, 1, 0, 8, 2, cv, A, 4, 3, f(1.0), A, A, W, None) == 1      # T = 0
    assert L.tq_attn_prefill(h, A, 1, 8, 12, 4, cv, A, 4, 3, f(1.0), A, A, W, None) == 2     # group of 3
    assert L.tq_attn_prefill(p64.handle, A, 1, 8, 8, 2, cv, A, 4, 3, f(1.0), A, A, W, None) == 2
    assert L.tq_attn_prefill(h, A, 1, 8, 8, 2, cv, A, 5, 3, f(1.0), A, A, W, None) == 2
    assert L.tq_attn_prefill(h, A, 1, 300, 8, 2, cv, A, 4, 3, f(1.0), A, A, W, None) == 4    # cap < T
    big = abi.CacheView(A, A, A, A, 1 << 23)
    assert L.tq_attn_prefill(h, A, 1, 2_100_000, 8, 2, big, A, 4, 3, f(1.0), A, A, W, None) == 2  # tiles > 65535
    assert L.tq_attn_prefill(h, A + 8, 1, 8, 8, 2, cv, A, 4, 3, f(1.0), A, A, W, None) == 3
    assert L.tq_attn_prefill(h, A, 1, 8, 8, 2, cv, A, 4, 3, f(1.0), A, A, 16, None) == 5
    assert L.tq_attn_prefill(h, A, 1, 8, 8, 2, cv, A, 4, 3, f(float("nan")), A, A, W, None) == 1
    assert L.tq_attn_prefill(h, None, 0, 8, 8, 2, cv, None, 4, 3, f(1.0), None, None, 0, None) == 0
    # the 32 KB rotation matrix, then a 99328-byte tile image and a float per 128 positions per
    # (sequence, KV head), 16-byte rounded
    assert L.tq_attn_prefill_workspace_bytes(2, 10, 8, 2, 300, 128) == 32768 + 2 * 2 * 3 * 99328 + 48
    assert L.tq_attn_prefill_workspace_bytes(2, 10, 8, 2, 256, 128) == 32768 + 2 * 2 * 2 * 99328 + 32
    assert L.tq_attn_prefill_workspace_bytes(2, 10, 8, 2, 300, 64) == 0
    assert L.tq_attn_prefill_workspace_bytes(2, 10, 8, 2, 9, 128) == 0   # cap < T


def test_qjl_call_validation_before_launch(L):
    """The QJL entry points check their arguments on the host before any
    launch: d outside {32, 64, 128}, bits outside 2..4, null and misaligned
    pointers, and the attention workspace size."""
    p128, p256, p16 = abi.Plan(128, 42), abi.Plan(256, 42), abi.Plan(16, 42)
    h = p128.handle
    A = 1 << 20
    f = ctypes.c_float
    assert L.tq_qjl_matrix(None, A, None) == 1
    assert L.tq_qjl_matrix(h, None, None) == 1
    assert L.tq_qjl_matrix(p256.handle, A, None) == 2
    assert L.tq_qjl_matrix(p16.handle, A, None) == 2
    assert L.tq_qjl_matrix(h, A + 4, None) == 3
    # tq_encode_qjl(plan, bits, S, x, dtype, n, packed, norms, rnorms, stream)
    assert L.tq_encode_qjl(h, 1, A, A, 0, 4, A, A, A, None) == 2
    assert L.tq_encode_qjl(h, 5, A, A, 0, 4, A, A, A, None) == 2
    assert L.tq_encode_qjl(h, 3, A, A, 7, 4, A, A, A, None) == 2
    assert L.tq_encode_qjl(p256.handle, 3, A, A, 0, 4, A, A, A, None) == 2
    assert L.tq_encode_qjl(h, 3, A, A, 0, -1, A, A, A, None) == 1
    assert L.tq_encode_qjl(h, 3, None, None, 0, 0, None, None, None, None) == 0
    assert L.tq_encode_qjl(h, 3, None, A, 0, 4, A, A, A, None) == 1
    assert L.tq_encode_qjl(h, 3, A, A, 0, 4, A, A, None, None) == 1
    assert L.tq_encode_qjl(h, 3, A + 4, A, 0, 4, A, A, A, None) == 3
    assert L.tq_encode_qjl(h, 3, A, A, 0, 4, A, A, A + 2, None) == 3
    # tq_decode_qjl(plan, bits, S, packed, norms, rnorms, n, y, dtype, stream)
    assert L.tq_decode_qjl(h, 1, A, A, A, A, 4, A, 0, None) == 2
    assert L.tq_decode_qjl(p16.handle, 3, A, A, A, A, 4, A, 0, None) == 2
    assert L.tq_decode_qjl(h, 3, A, A, A, None, 4, A, 0, None) == 1
    assert L.tq_decode_qjl(h, 3, A, A + 8, A, A, 4, A, 0, None) == 3
    assert L.tq_decode_qjl(h, 3, None, None, None, None, 0, None, 0, None) == 0
    # workspace of the CUDA-core kernel (d = 64): rotated and projected
    # queries (2 d floats per query head, in 64-float units) then (d + 2)
    # floats per query head and split; at d = 128 also the tensor-core
    # kernel's (two fp16 query prefixes, partials, work partition)
    assert L.tq_attn_qjl_workspace_bytes(1, 8, 2, 256, 1000) == 0
    assert L.tq_attn_qjl_workspace_bytes(1, 12, 8, 128, 1000) == 0  # Hq % Hkv
    n = L.tq_attn_qjl_workspace_bytes(1, 8, 2, 64, 1000)
    assert n >= 4 * (1024 + 8 * 66) and (n - 4 * 1024) % (4 * 8 * 66) == 0
    assert L.tq_attn_qjl_workspace_bytes(1, 8, 2, 128, 1000) >= 4 * (2048 + 8 * 130)
    cv = abi.CacheView(A, A, A, A, 256)
    W = 1 << 24
    # tq_attn_decode_qjl(plan, S, q, B, Hq, Hkv, cache, k_rnorm, ctx, kb, vb, scale, out, ws, ws_bytes, s)
    assert L.tq_attn_decode_qjl(None, A, A, 1, 8, 2, cv, A, 100, 3, 3, f(1.0), A, A, W, None) == 1
    assert L.tq_attn_decode_qjl(p256.handle, A, A, 1, 8, 2, cv, A, 100, 3, 3, f(1.0), A, A, W, None) == 2
    assert L.tq_attn_decode_qjl(h, A, A, 1, 8, 2, cv, A, 100, 5, 3, f(1.0), A, A, W, None) == 2
    assert L.tq_attn_decode_qjl(h, A, A, 1, 36, 2, cv, A, 100, 3, 3, f(1.0), A, A, W, None) == 2  # group 18
    assert L.tq_attn_decode_qjl(h, A, A, 1, 8, 2, cv, A, 300, 3, 3, f(1.0), A, A, W, None) == 4  # ctx > cap
    assert L.tq_attn_decode_qjl(h, A, A + 8, 1, 8, 2, cv, A, 100, 3, 3, f(1.0), A, A, W, None) == 3
    assert L.tq_attn_decode_qjl(h, A, A, 0, 8, 2, cv, A, 100, 3, 3, f(1.0), A, A, W, None) == 0  # B = 0
