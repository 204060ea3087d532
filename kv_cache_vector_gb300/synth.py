"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds none of the codec's or the attention's arithmetic: only
random-number generation and the shaping of distributions.  Both the CUDA path
and the CPU oracle read the *same bytes* produced here.

Two generators:

* ``normal_host``: counter-based, splitmix64 (Vigna) over a counter, two
  53-bit uniforms per value, Box-Muller in double.  Any element can be
  regenerated on its own from (seed, stream, index), so the oracle can be fed
  a sample of a large input without the whole of it.
* ``torch`` generators on the device (Philox) for inputs of many GB, which the
  host cannot produce quickly; the oracle then reads back the sampled input
  rows from the device buffer (inputs only, never a result of the library).

Workload recipes (the shapes and distributions the pages' workloads have):

* i.i.d. N(0, 1) rows (codec round trip; Gemma-3-4B-like caches).
* ``lowrank_rows``: per (layer, head) ``x = A z + sqrt(delta) * eps`` with
  ``A`` in R^{d x r}, ``A_ij ~ N(0, 1/r)``, ``r = 16``, ``delta = 0.25``, plus
  ``n_outliers`` seeded channels scaled by 8 -- correlated K/V activations with
  a few outlier channels, as in the Llama-8B-like prefill.
"""
from __future__ import annotations

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_at(seed: int, counters: np.ndarray) -> np.ndarray:
    """The k-th output (k = counters, 0-based) of splitmix64 seeded with seed."""
    with np.errstate(over="ignore"):
        k = counters.astype(np.uint64) + np.uint64(1)
        return _mix(np.uint64(seed) + k * _GAMMA)


def _stream_seed(seed: int, stream: int) -> int:
    """Independent streams: hash (seed, stream) into one 64-bit seed."""
    with np.errstate(over="ignore"):
        z = _mix(np.array([np.uint64(seed) ^ (np.uint64(stream) * _M2)], np.uint64))
    return int(z[0])


def normal_host(seed: int, n: int, stream: int = 0, start: int = 0) -> np.ndarray:
    """n standard-normal doubles: elements [start, start + n) of stream `stream`."""
    s = _stream_seed(seed, stream) if stream else seed
    idx = np.arange(start, start + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        r1 = splitmix64_at(s, idx * np.uint64(2))
        r2 = splitmix64_at(s, idx * np.uint64(2) + np.uint64(1))
    u1 = (r1 >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    u2 = (r2 >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)


def normal_rows(seed: int, n_rows: int, d: int, dtype=torch.float32, stream: int = 0) -> torch.Tensor:
    """[n_rows, d] i.i.d. N(0, 1) on the host, rounded to `dtype` (RNE)."""
    x = normal_host(seed, n_rows * d, stream).reshape(n_rows, d)
    return torch.from_numpy(x).to(dtype)


def unit_rows(seed: int, n_rows: int, d: int, stream: int = 0) -> torch.Tensor:
    """[n_rows, d] fp32 rows with uniformly random direction and unit norm."""
    x = normal_host(seed, n_rows * d, stream).reshape(n_rows, d)
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    return torch.from_numpy(x).to(torch.float32)


def lowrank_rows(seed: int, n_rows: int, d: int, dtype=torch.bfloat16, rank: int = 16,
                 delta: float = 0.25, n_outliers: int = 4, stream: int = 0,
                 device="cpu") -> torch.Tensor:
    """[n_rows, d] rows x = A z + sqrt(delta) eps with `n_outliers` channels x8.

    One (A, outlier set) per call: callers pass a distinct `stream` per
    (layer, head).  On the host the draw is the counter-based generator; on a
    CUDA device it is torch's Philox seeded from (seed, stream).
    """
    s = _stream_seed(seed, stream + 1)
    A = torch.from_numpy(normal_host(s, d * rank, 1).reshape(d, rank) / np.sqrt(rank)).float()
    out_ch = np.random.default_rng(s & 0xFFFFFFFF).choice(d, size=n_outliers, replace=False)
    scale = torch.ones(d)
    scale[torch.from_numpy(out_ch)] = 8.0
    if str(device) == "cpu":
        z = torch.from_numpy(normal_host(s, n_rows * rank, 2).reshape(n_rows, rank)).float()
        e = torch.from_numpy(normal_host(s, n_rows * d, 3).reshape(n_rows, d)).float()
    else:
        g = torch.Generator(device=device)
        g.manual_seed(s & 0x7FFFFFFFFFFFFFFF)
        z = torch.randn(n_rows, rank, generator=g, device=device)
        e = torch.randn(n_rows, d, generator=g, device=device)
        A, scale = A.to(device), scale.to(device)
    x = (z @ A.T + np.sqrt(delta) * e) * scale
    return x.to(dtype)


def outlier_rows(seed: int, n_rows: int, d: int, n_outliers: int, dtype=torch.bfloat16,
                 stream: int = 0, device="cpu") -> torch.Tensor:
    """[n_rows, d] i.i.d. N(0, 1) with `n_outliers` seeded channels scaled x8."""
    s = _stream_seed(seed, stream + 1)
    out_ch = np.random.default_rng(s & 0xFFFFFFFF).choice(d, size=n_outliers, replace=False)
    scale = torch.ones(d)
    scale[torch.from_numpy(out_ch)] = 8.0
    if str(device) == "cpu":
        x = torch.from_numpy(normal_host(s, n_rows * d, 4).reshape(n_rows, d)).float()
    else:
        g = torch.Generator(device=device)
        g.manual_seed(s & 0x7FFFFFFFFFFFFFFF)
        x = torch.randn(n_rows, d, generator=g, device=device)
        scale = scale.to(device)
    return (x * scale).to(dtype)


def device_normal(seed: int, shape, dtype=torch.bfloat16, device="cuda") -> torch.Tensor:
    """Large i.i.d. N(0, 1) tensor drawn on the device (torch Philox)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed & 0x7FFFFFFFFFFFFFFF)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)
