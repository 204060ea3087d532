"""Thin ctypes binding of ``libtq.so`` (include/tq.h), same names as the C ABI.

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, turned into pointers, and the call is enqueued on torch's current
CUDA stream.  Every step of the codec and the attention runs in the library's
kernels.  There is no fallback: if ``libtq.so`` is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from functools import lru_cache

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtq.so")

TQ_F32, TQ_BF16 = 0, 1
STATUS = {0: "TQ_OK", 1: "TQ_ERR_INVALID_ARG", 2: "TQ_ERR_UNSUPPORTED", 3: "TQ_ERR_ALIGNMENT",
          4: "TQ_ERR_RANGE", 5: "TQ_ERR_WORKSPACE", 6: "TQ_ERR_CUDA", 7: "TQ_ERR_NOMEM"}

# every symbol include/tq.h declares
EXPORTS = ("tq_codebook_init", "tq_plan_create", "tq_plan_destroy", "tq_plan_signs",
           "tq_plan_codebook", "tq_encode", "tq_decode", "tq_append", "tq_attn_workspace_bytes", "tq_attn_paged_workspace_bytes",
           "tq_attn_decode", "tq_status_string", "tq_last_cuda_error", "tq_device_status",
           "tq_attn_decode_noalloc", "tq_attn_decode_ex", "tq_append_paged", "tq_attn_decode_paged",
           "tq_attn_decode_append_paged", "tq_plan_create_ex", "tq_plan_signs2", "tq_codebook_init_gaussian",
           "tq_attn_prefill_workspace_bytes", "tq_attn_prefill", "tq_qjl_matrix", "tq_encode_qjl",
           "tq_decode_qjl", "tq_attn_qjl_workspace_bytes", "tq_attn_decode_qjl")


class TQError(RuntimeError):
    def __init__(self, fn: str, code: int, lib=None):
        self.code = code
        name = STATUS.get(code, str(code))
        extra = ""
        if code == 6 and lib is not None:
            extra = f" (cudaError {lib.tq_last_cuda_error()})"
        super().__init__(f"{fn} failed: {name}{extra}")


class CacheView(ctypes.Structure):
    _fields_ = [("k_packed", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("v_packed", ctypes.c_void_p), ("v_norm", ctypes.c_void_p),
                ("cap", ctypes.c_int64)]


class PagedCacheView(ctypes.Structure):
    _fields_ = [("k_packed", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("v_packed", ctypes.c_void_p), ("v_norm", ctypes.c_void_p),
                ("n_pages", ctypes.c_int64), ("page_size", ctypes.c_int32)]


@lru_cache(maxsize=1)
def lib() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m kv_cache_vector_gb300.build` "
            "(needs nvcc); there is no CPU fallback")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
    for name, res, args in [
        ("tq_codebook_init", i32, [i32, i32, vp, vp]),
        ("tq_plan_create", i32, [i32, u64, ctypes.POINTER(vp)]),
        ("tq_plan_create_ex", i32, [i32, u64, ctypes.c_uint32, ctypes.POINTER(vp)]),
        ("tq_plan_signs2", i32, [vp, vp]),
        ("tq_codebook_init_gaussian", i32, [i32, i32, vp, vp]),
        ("tq_plan_destroy", i32, [vp]),
        ("tq_plan_signs", i32, [vp, vp]),
        ("tq_plan_codebook", i32, [vp, i32, vp, vp]),
        ("tq_encode", i32, [vp, i32, vp, i32, i64, vp, vp, vp]),
        ("tq_decode", i32, [vp, i32, vp, vp, i64, vp, i32, vp]),
        ("tq_append", i32, [vp, i32, i32, vp, vp, i32, i32, i32, i64, CacheView, i64, vp]),
        ("tq_attn_workspace_bytes", ctypes.c_size_t, [i32, i32, i32, i32, i64]),
        ("tq_attn_paged_workspace_bytes", ctypes.c_size_t, [i32, i32, i32, i32, i64]),
        ("tq_attn_decode", i32, [vp, vp, i32, i32, i32, CacheView, i64, i32, i32, f32, f32, vp, vp,
                                 ctypes.c_size_t, vp]),
        ("tq_attn_decode_noalloc", i32, [vp, vp, i32, i32, i32, CacheView, i64, i32, i32, f32, f32,
                                         vp, vp]),
        ("tq_qjl_matrix", i32, [vp, vp, vp]),
        ("tq_encode_qjl", i32, [vp, i32, vp, vp, i32, i64, vp, vp, vp, vp]),
        ("tq_decode_qjl", i32, [vp, i32, vp, vp, vp, vp, i64, vp, i32, vp]),
        ("tq_attn_qjl_workspace_bytes", ctypes.c_size_t, [i32, i32, i32, i32, i64]),
        ("tq_attn_decode_qjl", i32, [vp, vp, vp, i32, i32, i32, CacheView, vp, i64, i32, i32, f32, vp, vp,
                                     ctypes.c_size_t, vp]),
        ("tq_attn_decode_ex", i32, [vp, vp, i32, i32, i32, CacheView, i64, i32, i32, f32, f32, vp, vp, vp,
                                    ctypes.c_size_t, vp]),
        ("tq_append_paged", i32, [vp, i32, i32, vp, vp, i32, i32, i32, PagedCacheView, vp, i32, vp, vp]),
        ("tq_attn_decode_paged", i32, [vp, vp, i32, i32, i32, PagedCacheView, vp, i32, vp, i64, i32, i32,
                                       f32, f32, vp, vp, ctypes.c_size_t, vp]),
        ("tq_attn_decode_append_paged", i32, [vp, vp, vp, vp, i32, i32, i32, i32, PagedCacheView, vp, i32, vp,
                                              i64, i32, i32, f32, f32, vp, vp, ctypes.c_size_t, vp]),
        ("tq_attn_prefill_workspace_bytes", ctypes.c_size_t, [i32, i32, i32, i32, i64, i32]),
        ("tq_attn_prefill", i32, [vp, vp, i32, i32, i32, i32, CacheView, vp, i32, i32, f32, vp, vp,
                                  ctypes.c_size_t, vp]),
        ("tq_status_string", ctypes.c_char_p, [i32]),
        ("tq_last_cuda_error", i32, []),
        ("tq_device_status", i32, [i32, ctypes.POINTER(i32)]),
    ]:
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def _check(fn: str, code: int):
    if code != 0:
        raise TQError(fn, code, lib())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TQ_F32
    if t.dtype == torch.bfloat16:
        return TQ_BF16
    raise TypeError(f"dtype {t.dtype} not supported (fp32 or bf16)")


def _cuda(*ts):
    for t in ts:
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
            raise ValueError("expected contiguous CUDA tensors")


def tq_codebook_init(d: int, bits: int):
    """Lloyd-Max codebook (double): (centroids[2^b], boundaries[2^b - 1])."""
    c = np.empty(1 << bits, np.float64)
    b = np.empty((1 << bits) - 1, np.float64)
    _check("tq_codebook_init", lib().tq_codebook_init(d, bits, c.ctypes.data, b.ctypes.data))
    return c, b


PLAN_GAUSSIAN_CODEBOOK = 1  # TQ_PLAN_GAUSSIAN_CODEBOOK
PLAN_TWO_SIDED_SIGNS = 2    # TQ_PLAN_TWO_SIDED_SIGNS


class Plan:
    """Owns a tq_plan (host object: d, seed, format flags, signs, fp32 codebooks)."""

    def __init__(self, d: int, seed: int, flags: int = 0):
        h = ctypes.c_void_p()
        _check("tq_plan_create_ex", lib().tq_plan_create_ex(d, ctypes.c_uint64(seed), flags, ctypes.byref(h)))
        self.handle, self.d, self.seed, self.flags = h, d, seed, flags

    def signs(self) -> np.ndarray:
        s = np.empty(self.d, np.int8)
        _check("tq_plan_signs", lib().tq_plan_signs(self.handle, s.ctypes.data))
        return s

    def signs2(self) -> np.ndarray:
        s = np.empty(self.d, np.int8)
        _check("tq_plan_signs2", lib().tq_plan_signs2(self.handle, s.ctypes.data))
        return s

    def codebook(self, bits: int):
        c = np.empty(1 << bits, np.float32)
        b = np.empty((1 << bits) - 1, np.float32)
        _check("tq_plan_codebook", lib().tq_plan_codebook(self.handle, bits, c.ctypes.data, b.ctypes.data))
        return c, b

    def close(self):
        if getattr(self, "handle", None):
            lib().tq_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tq_plan_create(d: int, seed: int, flags: int = 0) -> Plan:
    return Plan(d, seed, flags)


def tq_codebook_init_gaussian(d: int, bits: int):
    """(centroids[2^b], boundaries[2^b - 1]) of N(0, 1/d), float64, on the host."""
    c = np.empty(1 << bits, np.float64)
    b = np.empty((1 << bits) - 1, np.float64)
    _check("tq_codebook_init_gaussian", lib().tq_codebook_init_gaussian(d, bits, c.ctypes.data, b.ctypes.data))
    return c, b


def tq_encode(plan: Plan, bits: int, x: torch.Tensor, packed: torch.Tensor | None = None,
              norms: torch.Tensor | None = None):
    """x: [n, d] fp32/bf16 CUDA -> (packed [n, d*bits/8] uint8, norms [n] fp32)."""
    x2 = x.reshape(-1, plan.d)
    n = x2.shape[0]
    if packed is None:
        packed = torch.empty(n, plan.d * bits // 8, dtype=torch.uint8, device=x.device)
    if norms is None:
        norms = torch.empty(n, dtype=torch.float32, device=x.device)
    _cuda(x2, packed, norms)
    _check("tq_encode", lib().tq_encode(plan.handle, bits, x2.data_ptr(), _dt(x2), n,
                                        packed.data_ptr(), norms.data_ptr(), _stream(x2)))
    return packed, norms


def tq_decode(plan: Plan, bits: int, packed: torch.Tensor, norms: torch.Tensor,
              out_dtype=torch.float32, out: torch.Tensor | None = None) -> torch.Tensor:
    n = norms.numel()
    if out is None:
        out = torch.empty(n, plan.d, dtype=out_dtype, device=packed.device)
    _cuda(packed, norms, out)
    _check("tq_decode", lib().tq_decode(plan.handle, bits, packed.data_ptr(), norms.data_ptr(), n,
                                        out.data_ptr(), _dt(out), _stream(out)))
    return out


@dataclass
class Cache:
    """One layer of a packed KV cache (caller-owned device tensors)."""
    k_packed: torch.Tensor  # [B, Hkv, cap, d*kb/8] uint8
    k_norm: torch.Tensor    # [B, Hkv, cap] fp32
    v_packed: torch.Tensor  # [B, Hkv, cap, d*vb/8] uint8
    v_norm: torch.Tensor    # [B, Hkv, cap] fp32
    k_bits: int
    v_bits: int

    @staticmethod
    def empty(B, Hkv, cap, d, k_bits, v_bits, device="cuda"):
        return Cache(torch.zeros(B, Hkv, cap, d * k_bits // 8, dtype=torch.uint8, device=device),
                     torch.zeros(B, Hkv, cap, dtype=torch.float32, device=device),
                     torch.zeros(B, Hkv, cap, d * v_bits // 8, dtype=torch.uint8, device=device),
                     torch.zeros(B, Hkv, cap, dtype=torch.float32, device=device), k_bits, v_bits)

    @property
    def cap(self) -> int:
        return self.k_norm.shape[2]

    def view(self) -> CacheView:
        _cuda(self.k_packed, self.k_norm, self.v_packed, self.v_norm)
        return CacheView(self.k_packed.data_ptr(), self.k_norm.data_ptr(), self.v_packed.data_ptr(),
                         self.v_norm.data_ptr(), self.cap)


def tq_append(plan: Plan, cache: Cache, k_new: torch.Tensor, v_new: torch.Tensor, pos: int):
    """k_new, v_new: [B, Hkv, n_new, d] fp32/bf16 -> written at positions pos..pos+n_new-1."""
    B, Hkv, n_new, d = k_new.shape
    if v_new.shape != k_new.shape or v_new.dtype != k_new.dtype or d != plan.d:
        raise ValueError("k_new / v_new must both be [B, Hkv, n_new, d] of one dtype")
    _cuda(k_new, v_new)
    _check("tq_append", lib().tq_append(plan.handle, cache.k_bits, cache.v_bits, k_new.data_ptr(),
                                        v_new.data_ptr(), _dt(k_new), B, Hkv, n_new, cache.view(),
                                        pos, _stream(k_new)))


def tq_attn_workspace_bytes(B: int, Hq: int, Hkv: int, d: int, ctx_len: int) -> int:
    return int(lib().tq_attn_workspace_bytes(B, Hq, Hkv, d, ctx_len))


def tq_attn_paged_workspace_bytes(B: int, Hq: int, Hkv: int, d: int, max_ctx: int) -> int:
    return int(lib().tq_attn_paged_workspace_bytes(B, Hq, Hkv, d, max_ctx))


def tq_attn_decode(plan: Plan, q: torch.Tensor, cache: Cache, ctx_len: int, scale: float,
                   sparse_v_threshold: float = 0.0, out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None) -> torch.Tensor:
    """q: [B, Hq, d] bf16 -> out [B, Hq, d] fp32."""
    B, Hq, d = q.shape
    Hkv = cache.k_norm.shape[1]
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    need = tq_attn_workspace_bytes(B, Hq, Hkv, d, ctx_len)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(q, out, workspace)
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bf16")
    _check("tq_attn_decode", lib().tq_attn_decode(
        plan.handle, q.data_ptr(), B, Hq, Hkv, cache.view(), ctx_len, cache.k_bits, cache.v_bits,
        ctypes.c_float(scale), ctypes.c_float(sparse_v_threshold), out.data_ptr(),
        workspace.data_ptr(), workspace.numel(), _stream(q)))
    return out


def tq_attn_decode_ex(plan: Plan, q: torch.Tensor, cache: Cache, ctx_len: int, scale: float,
                      sparse_v_threshold: float = 0.0, out: torch.Tensor | None = None,
                      v_rows_read: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None):
    """tq_attn_decode that also returns, per (batch, KV head), how many cached
    rows' V bytes the call read: (out [B, Hq, d] fp32, v_rows_read [B, Hkv] int32)."""
    B, Hq, d = q.shape
    Hkv = cache.k_norm.shape[1]
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    if v_rows_read is None:
        v_rows_read = torch.empty(B, Hkv, dtype=torch.int32, device=q.device)
    need = tq_attn_workspace_bytes(B, Hq, Hkv, d, ctx_len)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(q, out, workspace, v_rows_read)
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bf16")
    _i32(v_rows_read, "v_rows_read")
    _check("tq_attn_decode_ex", lib().tq_attn_decode_ex(
        plan.handle, q.data_ptr(), B, Hq, Hkv, cache.view(), ctx_len, cache.k_bits, cache.v_bits,
        ctypes.c_float(scale), ctypes.c_float(sparse_v_threshold), out.data_ptr(), v_rows_read.data_ptr(),
        workspace.data_ptr(), workspace.numel(), _stream(q)))
    return out, v_rows_read


def tq_attn_decode_noalloc(plan: Plan, q: torch.Tensor, cache: Cache, ctx_len: int, scale: float,
                           sparse_v_threshold: float = 0.0,
                           out: torch.Tensor | None = None) -> torch.Tensor:
    """As tq_attn_decode, without a workspace: for callers that may not
    allocate device memory while they run.  The library's fixed 8 MiB device
    array holds the split-K partials; sizes that need more raise TQError
    (TQ_ERR_WORKSPACE).  Calls that overlap on the GPU share that array and
    race.  (This wrapper allocates `out` only when none is passed.)"""
    B, Hq, d = q.shape
    Hkv = cache.k_norm.shape[1]
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    _cuda(q, out)
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bf16")
    _check("tq_attn_decode_noalloc", lib().tq_attn_decode_noalloc(
        plan.handle, q.data_ptr(), B, Hq, Hkv, cache.view(), ctx_len, cache.k_bits, cache.v_bits,
        ctypes.c_float(scale), ctypes.c_float(sparse_v_threshold), out.data_ptr(), _stream(q)))
    return out


@dataclass
class PagedCache:
    """One layer of a paged KV cache (caller-owned device tensors): pages of
    page_size positions, each holding every KV head."""
    k_packed: torch.Tensor  # [n_pages, Hkv, page_size, d*kb/8] uint8
    k_norm: torch.Tensor    # [n_pages, Hkv, page_size] fp32
    v_packed: torch.Tensor  # [n_pages, Hkv, page_size, d*vb/8] uint8
    v_norm: torch.Tensor    # [n_pages, Hkv, page_size] fp32
    k_bits: int
    v_bits: int

    @staticmethod
    def empty(n_pages, Hkv, page_size, d, k_bits, v_bits, device="cuda"):
        return PagedCache(
            torch.zeros(n_pages, Hkv, page_size, d * k_bits // 8, dtype=torch.uint8, device=device),
            torch.zeros(n_pages, Hkv, page_size, dtype=torch.float32, device=device),
            torch.zeros(n_pages, Hkv, page_size, d * v_bits // 8, dtype=torch.uint8, device=device),
            torch.zeros(n_pages, Hkv, page_size, dtype=torch.float32, device=device), k_bits, v_bits)

    @property
    def n_pages(self) -> int:
        return self.k_norm.shape[0]

    @property
    def Hkv(self) -> int:
        return self.k_norm.shape[1]

    @property
    def page_size(self) -> int:
        return self.k_norm.shape[2]

    def view(self) -> PagedCacheView:
        _cuda(self.k_packed, self.k_norm, self.v_packed, self.v_norm)
        return PagedCacheView(self.k_packed.data_ptr(), self.k_norm.data_ptr(), self.v_packed.data_ptr(),
                              self.v_norm.data_ptr(), self.n_pages, self.page_size)


def _i32(t: torch.Tensor, name: str):
    _cuda(t)
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")


def tq_append_paged(plan: Plan, cache: PagedCache, k_new: torch.Tensor, v_new: torch.Tensor,
                    block_table: torch.Tensor, positions: torch.Tensor):
    """k_new, v_new: [B, Hkv, d] fp32/bf16; block_table [B, max_pages] int32;
    positions [B] int32: row (b, h) goes to position positions[b] of sequence b."""
    B, Hkv, d = k_new.shape
    if v_new.shape != k_new.shape or v_new.dtype != k_new.dtype or d != plan.d or Hkv != cache.Hkv:
        raise ValueError("k_new / v_new must both be [B, Hkv, d] of one dtype")
    _cuda(k_new, v_new)
    _i32(block_table, "block_table")
    _i32(positions, "positions")
    _check("tq_append_paged", lib().tq_append_paged(
        plan.handle, cache.k_bits, cache.v_bits, k_new.data_ptr(), v_new.data_ptr(), _dt(k_new), B, Hkv,
        cache.view(), block_table.data_ptr(), block_table.shape[1], positions.data_ptr(), _stream(k_new)))


def tq_attn_decode_paged(plan: Plan, q: torch.Tensor, cache: PagedCache, block_table: torch.Tensor,
                         ctx_lens: torch.Tensor, max_ctx: int, scale: float,
                         sparse_v_threshold: float = 0.0, out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None) -> torch.Tensor:
    """q: [B, Hq, d] bf16; block_table [B, max_pages] int32; ctx_lens [B] int32
    (each at most max_ctx) -> out [B, Hq, d] fp32."""
    B, Hq, d = q.shape
    Hkv = cache.Hkv
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    need = tq_attn_paged_workspace_bytes(B, Hq, Hkv, d, max_ctx)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(q, out, workspace)
    _i32(block_table, "block_table")
    _i32(ctx_lens, "ctx_lens")
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bf16")
    _check("tq_attn_decode_paged", lib().tq_attn_decode_paged(
        plan.handle, q.data_ptr(), B, Hq, Hkv, cache.view(), block_table.data_ptr(), block_table.shape[1],
        ctx_lens.data_ptr(), max_ctx, cache.k_bits, cache.v_bits, ctypes.c_float(scale),
        ctypes.c_float(sparse_v_threshold), out.data_ptr(), workspace.data_ptr(), workspace.numel(),
        _stream(q)))
    return out


def tq_attn_decode_append_paged(plan: Plan, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                cache: PagedCache, block_table: torch.Tensor, positions: torch.Tensor,
                                max_ctx: int, scale: float, sparse_v_threshold: float = 0.0,
                                out: torch.Tensor | None = None,
                                workspace: torch.Tensor | None = None) -> torch.Tensor:
    """One decode step: append k_new/v_new [B, Hkv, d] (fp32 or bf16) at
    positions [B] int32, then attend q [B, Hq, d] bf16 over positions + 1
    (at most max_ctx) -> out [B, Hq, d] fp32."""
    B, Hq, d = q.shape
    Hkv = cache.Hkv
    if tuple(k_new.shape) != (B, Hkv, d) or tuple(v_new.shape) != (B, Hkv, d):
        raise ValueError("k_new and v_new must be [B, Hkv, d]")
    if k_new.dtype != v_new.dtype:
        raise TypeError("k_new and v_new must share a dtype")
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    need = tq_attn_paged_workspace_bytes(B, Hq, Hkv, d, max_ctx)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(q, k_new, v_new, out, workspace)
    _i32(block_table, "block_table")
    _i32(positions, "positions")
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bf16")
    k_new, v_new = k_new.contiguous(), v_new.contiguous()
    _check("tq_attn_decode_append_paged", lib().tq_attn_decode_append_paged(
        plan.handle, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), _dt(k_new), B, Hq, Hkv, cache.view(),
        block_table.data_ptr(), block_table.shape[1], positions.data_ptr(), max_ctx, cache.k_bits,
        cache.v_bits, ctypes.c_float(scale), ctypes.c_float(sparse_v_threshold), out.data_ptr(),
        workspace.data_ptr(), workspace.numel(), _stream(q)))
    return out


def tq_attn_prefill(plan: Plan, q: torch.Tensor, cache: Cache, q_start: torch.Tensor, scale: float,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """q: [B, T, Hq, d] bf16; q_start [B] int32 (token t of sequence b sits at
    q_start[b] + t and attends causally) -> out [B, T, Hq, d] fp32."""
    B, T, Hq, d = q.shape
    Hkv = cache.k_norm.shape[1]
    if out is None:
        out = torch.empty(B, T, Hq, d, dtype=torch.float32, device=q.device)
    need = int(lib().tq_attn_prefill_workspace_bytes(B, T, Hq, Hkv, cache.cap, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(q, out, workspace)
    _i32(q_start, "q_start")
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bf16")
    _check("tq_attn_prefill", lib().tq_attn_prefill(
        plan.handle, q.contiguous().data_ptr(), B, T, Hq, Hkv, cache.view(), q_start.data_ptr(), cache.k_bits,
        cache.v_bits, ctypes.c_float(scale), out.data_ptr(), workspace.data_ptr(), workspace.numel(),
        _stream(q)))
    return out


def tq_device_status(reset: bool = False) -> int:
    st = ctypes.c_int(0)
    _check("tq_device_status", lib().tq_device_status(int(reset), ctypes.byref(st)))
    return st.value


# ------------------------------------------------------------ QJL residual keys

def tq_qjl_matrix(plan: Plan, device="cuda", out: torch.Tensor | None = None) -> torch.Tensor:
    """The plan's QJL projection S [d, d] fp32, drawn on the device."""
    if out is None:
        out = torch.empty(plan.d, plan.d, dtype=torch.float32, device=device)
    _cuda(out)
    _check("tq_qjl_matrix", lib().tq_qjl_matrix(plan.handle, out.data_ptr(), _stream(out)))
    return out


def tq_encode_qjl(plan: Plan, bits: int, S: torch.Tensor, x: torch.Tensor):
    """x: [n, d] fp32/bf16 -> (packed [n, d*bits/8] uint8, norms [n], rnorms [n] fp32)."""
    x2 = x.reshape(-1, plan.d)
    n = x2.shape[0]
    packed = torch.empty(n, plan.d * bits // 8, dtype=torch.uint8, device=x.device)
    norms = torch.empty(n, dtype=torch.float32, device=x.device)
    rnorms = torch.empty(n, dtype=torch.float32, device=x.device)
    _cuda(S, x2, packed, norms, rnorms)
    _check("tq_encode_qjl", lib().tq_encode_qjl(plan.handle, bits, S.data_ptr(), x2.data_ptr(), _dt(x2), n,
                                                packed.data_ptr(), norms.data_ptr(), rnorms.data_ptr(),
                                                _stream(x2)))
    return packed, norms, rnorms


def tq_decode_qjl(plan: Plan, bits: int, S: torch.Tensor, packed: torch.Tensor, norms: torch.Tensor,
                  rnorms: torch.Tensor, out_dtype=torch.float32) -> torch.Tensor:
    n = norms.numel()
    out = torch.empty(n, plan.d, dtype=out_dtype, device=packed.device)
    _cuda(S, packed, norms, rnorms, out)
    _check("tq_decode_qjl", lib().tq_decode_qjl(plan.handle, bits, S.data_ptr(), packed.data_ptr(),
                                                norms.data_ptr(), rnorms.data_ptr(), n, out.data_ptr(),
                                                _dt(out), _stream(out)))
    return out


def tq_attn_qjl_workspace_bytes(B: int, Hq: int, Hkv: int, d: int, ctx_len: int) -> int:
    return int(lib().tq_attn_qjl_workspace_bytes(B, Hq, Hkv, d, ctx_len))


def tq_attn_decode_qjl(plan: Plan, S: torch.Tensor, q: torch.Tensor, cache: Cache, k_rnorm: torch.Tensor,
                       ctx_len: int, scale: float, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None) -> torch.Tensor:
    """q: [B, Hq, d] bf16; cache.k_* in the QJL format of cache.k_bits with
    k_rnorm [B, Hkv, cap] the gammas -> out [B, Hq, d] fp32."""
    B, Hq, d = q.shape
    Hkv = cache.k_norm.shape[1]
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    need = tq_attn_qjl_workspace_bytes(B, Hq, Hkv, d, ctx_len)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _cuda(S, q, k_rnorm, out, workspace)
    if q.dtype != torch.bfloat16:
        raise TypeError("q must be bf16")
    _check("tq_attn_decode_qjl", lib().tq_attn_decode_qjl(
        plan.handle, S.data_ptr(), q.data_ptr(), B, Hq, Hkv, cache.view(), k_rnorm.data_ptr(), ctx_len,
        cache.k_bits, cache.v_bits, ctypes.c_float(scale), out.data_ptr(), workspace.data_ptr(),
        workspace.numel(), _stream(q)))
    return out
