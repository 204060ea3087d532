"""TurboQuant KV-cache codec and packed decode attention for GB300 (sm_103a).

The compute lives in ``libtq.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/tq.h``); ``kv_cache_vector_gb300.abi`` is its thin
Python binding.  Importing the package does not load the library; the first
call does, and raises if it has not been built.
"""
from .abi import (Cache, PagedCache, Plan, TQError, tq_append, tq_append_paged,  # noqa: F401
                  tq_attn_decode, tq_attn_decode_append_paged, tq_attn_decode_paged, tq_attn_prefill,
                  tq_attn_paged_workspace_bytes, tq_attn_workspace_bytes, tq_codebook_init,
                  tq_codebook_init_gaussian, tq_decode, tq_device_status, tq_encode, tq_plan_create,
                  PLAN_GAUSSIAN_CODEBOOK, PLAN_TWO_SIDED_SIGNS)
