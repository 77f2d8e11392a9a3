"""Low-precision cache formats, fp64 reference (test infrastructure).

Only the tests may import this module; the product library shares no code
with it.  It states, from their definitions, the number formats the pages
give for the production caches, so that a kernel reading those caches can be
checked against it:

* main KV entries: the last r (rotary) dims in BF16, the other c - r dims in
  FP8 E4M3 ["DeepSeek-V4" book, ch.8 "The main compressed-entry payload";
  ch.16 "The two main FP4 targets"];
* indexer queries and keys: MXFP4, FP4 E2M1 elements with one shared
  power-of-two scale per 1 x 32 block [ch.16 "The two main FP4 targets",
  "Why use fine-grained scales?"];
* index scores: FP32 rounded to BF16 before the top-k [ch.16 "BF16 index
  scores"].

Readings where the pages leave a rule open (each is also listed in the
design notes):

* E4M3 is the finite variant (largest magnitude 448, no infinities); values
  round to nearest, ties to even, and saturate at +-448.
* The FP8 part of a KV entry carries one fp32 scale per group of `group`
  consecutive dims (default 128, the 1 x 128 activation tile of DeepSeek's
  FP8 recipe; the last group of the 448 non-rotary dims is 64 wide): scale =
  amax / 448, so the group's largest magnitude maps to the top of the range.
  An all-zero group gets scale 1.
* The entry is quantised as the fp32 values a kernel holds it in: the scale
  is rounded to fp32, and the quotient x / scale that the E4M3 rounding
  decides on is formed in fp32 (the precision of the FP8 conversion), so a
  quotient within an fp32 rounding of an E4M3 midpoint is decided as that
  arithmetic decides it.  The rotary dims are rounded to BF16 from fp32.
* MXFP4 follows the OCP microscaling rule: shared exponent =
  floor(log2(amax)) - 2 (2 is the largest E2M1 exponent), elements round to
  nearest, ties to even, and saturate at +-6; an all-zero block has scale 1.
* A BF16 score is the fp64 score rounded once, to nearest even.

Every function works on float64 numpy arrays and returns float64 arrays
holding exactly representable values of the format (dequantised).
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6       # smallest normal: 2^-6
E4M3_MANT_BITS = 3
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E2M1_MAX = 6.0
E2M1_EMAX = 2                  # 6 = 1.5 * 2^2


def _round_half_even(v: np.ndarray) -> np.ndarray:
    return np.round(v)         # numpy rounds halves to the even integer


def e4m3_round(x) -> np.ndarray:
    """x rounded to the nearest FP8 E4M3 value (ties to even), saturating at
    +-448.  Spacing is 2^(e-3) in the binade [2^e, 2^(e+1)) for e >= -6 and
    2^-9 below 2^-6 (subnormals)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, E4M3_MIN_NORMAL_EXP)
    step = np.exp2(e - E4M3_MANT_BITS)
    q = _round_half_even(a / step) * step
    q = np.minimum(q, E4M3_MAX)
    return np.where(a > 0, np.copysign(q, x), 0.0 * x)


def e2m1_round(x) -> np.ndarray:
    """x rounded to the nearest FP4 E2M1 value {0, .5, 1, 1.5, 2, 3, 4, 6}
    (ties to the value with even mantissa bit), saturating at +-6."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E2M1_MAX)
    # spacing: 0.5 below 2, 1 in [2, 4), 2 in [4, 6]
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    q = _round_half_even(a / step) * step
    q = np.minimum(q, E2M1_MAX)
    return np.copysign(q, x)


def mxfp4(x, block: int = 32) -> np.ndarray:
    """Blocks of `block` consecutive values along the last axis share one
    scale 2^(floor(log2(amax)) - 2); each value becomes scale * E2M1(x / scale).
    Returns the dequantised values."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    assert n % block == 0, "the last axis must be a whole number of blocks"
    xb = x.reshape(x.shape[:-1] + (n // block, block))
    amax = np.max(np.abs(xb), axis=-1, keepdims=True)
    exp = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - E2M1_EMAX
    exp = np.clip(exp, -127, 127)
    scale = np.where(amax > 0, np.exp2(exp), 1.0)
    return (e2m1_round(xb / scale) * scale).reshape(x.shape)


def bf16_round(x) -> np.ndarray:
    """x rounded once to the nearest bfloat16 value (ties to even)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    step = np.exp2(e - 7)
    q = _round_half_even(a / step) * step
    return np.where(a > 0, np.copysign(q, x), 0.0 * x)


def kv_entry_fp8(e, rope_dims: int = 64, group: int = 128) -> np.ndarray:
    """One stored KV entry (or rows of entries, last axis = c): the first
    c - rope_dims dims in FP8 E4M3 with one fp32 scale per `group` dims, the
    rotary dims in BF16.  Returns the dequantised entry."""
    e32 = np.asarray(e, dtype=np.float64).astype(np.float32)
    c = e32.shape[-1]
    nr = c - rope_dims
    out = np.empty(e32.shape, np.float64)
    for g0 in range(0, nr, group):
        g1 = min(g0 + group, nr)
        part = e32[..., g0:g1]
        amax = np.max(np.abs(part), axis=-1, keepdims=True).astype(np.float64)
        # the scale itself is stored in fp32
        scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)
        quot = (part / scale).astype(np.float64)          # formed in fp32
        out[..., g0:g1] = e4m3_round(quot) * scale.astype(np.float64)
    out[..., nr:] = bf16_round(e32[..., nr:].astype(np.float64))
    return out


def entry_payload_bytes(c: int = 512, rope_dims: int = 64, dI: int = 128) -> dict:
    """Scalar payload per stored entry, scales and padding excluded: the main
    KV entry (FP8 non-rotary + BF16 rotary dims) and one FP4 indexer key."""
    return {"kv": (c - rope_dims) * 1 + rope_dims * 2, "index_key": dI // 2}


def index_scores_lowp(qI, w, q_pos, kI, m) -> np.ndarray:
    """One sequence with MXFP4 indexer queries and keys and BF16 scores:
    I[t, j] = bf16( sum_h w[t, h] * max(0, q4[t, h] . k4[j]) ) for visible j,
    -inf otherwise, where q4 / k4 are the MXFP4-dequantised qI / kI (blocks of
    32 along the indexer dim)."""
    qI = mxfp4(np.asarray(qI, dtype=np.float64))
    kI = mxfp4(np.asarray(kI, dtype=np.float64))
    w = np.asarray(w, dtype=np.float64)
    T, E = qI.shape[0], kI.shape[0]
    out = np.full((T, E), -np.inf)
    for t in range(T):
        nv = min(max((int(q_pos[t]) + 1) // m, 0), E)
        if nv == 0:
            continue
        dots = qI[t] @ kI[:nv].T                    # [hI, nv]
        out[t, :nv] = bf16_round(w[t] @ np.maximum(dots, 0.0))
    return out


def e4m3_values() -> np.ndarray:
    """Every finite non-negative E4M3 value, from its bit fields (for tests)."""
    vals = []
    for ebits in range(16):
        for m in range(8):
            if ebits == 15 and m == 7:
                continue                               # the NaN encoding
            if ebits == 0:
                vals.append(m * 2.0 ** -9)
            else:
                vals.append((1 + m / 8.0) * 2.0 ** (ebits - 7))
    return np.array(sorted(set(vals)))


def nearest_even(x: float, grid: np.ndarray, mant_of) -> float:
    """Brute force: the grid value nearest to |x| (ties to the one whose
    mantissa bit `mant_of(v)` is even), with x's sign; beyond the grid's top,
    the top."""
    a = min(abs(x), float(grid[-1]))
    d = np.abs(grid - a)
    best = np.flatnonzero(d == d.min())
    if len(best) > 1:
        best = [b for b in best if mant_of(grid[b]) % 2 == 0]
    return math.copysign(float(grid[best[0]]), x)
