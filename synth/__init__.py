"""Seeded synthetic inputs for the CSA/HCA attention layer.

This module is the one piece shared by the tests, the bench and the oracle
harness.  It draws random numbers and rounds them to the storage dtype; it
holds none of the layer's arithmetic (no compression, scoring, selection or
attention).  Every tensor is identified by (seed, tensor id) and is drawn in
fixed-size chunks, each chunk from its own Philox4x32-10 stream keyed by
(seed, tensor id, chunk), so values do not depend on the thread count.

Storage dtypes:
  "f32"  -> numpy float32
  "bf16" -> numpy uint16 holding bfloat16 bit patterns (round-to-nearest-even
            from the float32 draw)
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 22
_THREADS = max(1, min(32, os.cpu_count() or 1))


def _fill_normal(out: np.ndarray, seed: int, tid: int) -> None:
    flat = out.reshape(-1)
    nchunks = (flat.size + CHUNK - 1) // CHUNK

    def one(i):
        g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tid, i])))
        g.standard_normal(out=flat[i * CHUNK:(i + 1) * CHUNK], dtype=np.float32)

    if nchunks <= 1:
        for i in range(nchunks):
            one(i)
    else:
        with ThreadPoolExecutor(min(_THREADS, nchunks)) as ex:
            list(ex.map(one, range(nchunks)))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, np.uint16)
    flat_u, flat_o = u.reshape(-1), out.reshape(-1)
    step = 1 << 24

    def one(i):
        s = flat_u[i:i + step]
        r = s + (np.uint32(0x7FFF) + ((s >> np.uint32(16)) & np.uint32(1)))
        flat_o[i:i + step] = (r >> np.uint32(16)).astype(np.uint16)

    starts = range(0, flat_u.size, step)
    if flat_u.size > step:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(one, starts))
    else:
        for i in starts:
            one(i)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array -> float64 (exact)."""
    if dtype == "bf16":
        return bf16_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float array -> storage dtype (float32 RNE, or bf16 bits RNE via float32)."""
    x32 = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits(x32)
    return np.ascontiguousarray(x32)


def normal(seed: int, tid: int, shape, std: float = 1.0, dtype: str = "bf16") -> np.ndarray:
    """i.i.d. N(0, std^2) drawn in float32, then rounded to the storage dtype."""
    a = np.empty(tuple(int(s) for s in shape), np.float32)
    _fill_normal(a, seed, tid)
    if std != 1.0:
        a *= np.float32(std)
    return to_storage(a, dtype)


def softmax_normal(seed: int, tid: int, shape) -> np.ndarray:
    """float32 weights: softmax over the last axis of i.i.d. N(0,1) draws
    (the indexer head-weight distribution of the workloads)."""
    a = np.empty(tuple(int(s) for s in shape), np.float32)
    _fill_normal(a, seed, tid)
    a64 = a.astype(np.float64)
    a64 -= a64.max(axis=-1, keepdims=True)
    e = np.exp(a64)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


from .workloads import WORKLOADS, make_inputs  # noqa: E402,F401
