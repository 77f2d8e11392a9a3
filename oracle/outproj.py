"""Query / KV normalisation and the grouped output projection, fp64 reference
(test infrastructure).

Only the tests may import this module; the product library shares no code
with it.  It states the two steps on either side of the attention layer's
boundary ["DeepSeek-V4" book, ch.7 "Query and KV normalization"; ch.6 "Why
output projection is a large cost"]:

* RMSNorm, applied separately to each query head and to the shared
  compressed KV head before core attention: y = x / sqrt(mean(x^2) + eps) * g;
* the grouped output projection: the heads are split into groups of
  `heads_per_group`; each group's concatenated outputs (heads_per_group * c
  coordinates) are projected to d_g, the group results are concatenated and
  projected to the hidden width d.

Readings where the pages leave a rule open (also in the design notes):

* eps = 1e-6 and one learned gain per coordinate (shared by all query heads;
  a separate gain for the KV head);
* the norm acts on the vector as produced, before RoPE: q is normalised per
  head, then rotated at t; a compressed entry is normalised after pooling,
  then rotated at its block's last position;
* the projection reads the de-rotated attention output.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def rmsnorm(x, g, eps: float = EPS) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def grouped_out_proj(o, w_g, w_o, heads_per_group: int = 8) -> np.ndarray:
    """o [T, H, c] -> [T, d].  w_g [G, heads_per_group * c, d_g] holds one
    matrix per group, w_o [G * d_g, d] the final projection."""
    o = np.asarray(o, dtype=np.float64)
    T, H, c = o.shape
    G = H // heads_per_group
    assert G * heads_per_group == H and w_g.shape[0] == G
    y = [o[:, g * heads_per_group:(g + 1) * heads_per_group, :].reshape(T, -1) @ w_g[g]
         for g in range(G)]
    return np.concatenate(y, axis=1) @ w_o


def direct_weight(w_g, w_o) -> np.ndarray:
    """The single [H * c, d] matrix the grouped projection amounts to:
    blockdiag(w_g[0], ..., w_g[G-1]) @ w_o."""
    G, gin, dg = w_g.shape
    bd = np.zeros((G * gin, G * dg))
    for g in range(G):
        bd[g * gin:(g + 1) * gin, g * dg:(g + 1) * dg] = w_g[g]
    return bd @ w_o


def projection_weights(H: int, c: int, d: int, d_g: int = 1024, heads_per_group: int = 8) -> dict:
    """Principal weight counts of the output projection: direct (H c d) and
    grouped (G heads_per_group c d_g + G d_g d)."""
    G = H // heads_per_group
    return {"direct": H * c * d, "grouped": G * heads_per_group * c * d_g + G * d_g * d}
