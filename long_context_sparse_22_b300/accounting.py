"""Algorithmic work of the CSA / HCA layer: the FLOPs and HBM bytes the method
itself must spend, independent of any kernel.  Used for roofline fractions.

Counting rules (DeepSeek-V4 book ch.8 "A Cost Model for Long Context",
sections "Main-attention arithmetic" and "Indexer arithmetic"):
  - core attention: 4 * c * E * H FLOPs per query (2cE for the dot products,
    2cE for the weighted sum, per head) over the E entries it reads;
  - indexer: 2 * dI * hI FLOPs per (query, visible entry) pair.
Bytes count each tensor the step must read or write once, in its storage
dtype; gathered entries are counted once per query that reads them.  An
implementation's own intermediates (the fp32 score array between the
indexer and the selection) are not algorithmic and are not counted.
"""
from __future__ import annotations


def attn_flops_per_query(c: int, E: int, H: int) -> int:
    return 4 * c * E * H


def indexer_flops_per_query(dI: int, hI: int, entries: int) -> int:
    return 2 * dI * hI * entries


def visible(t: int, m: int, E: int) -> int:
    return max(0, min(E, (t + 1) // m))


def _floor_sum(N: int, m: int) -> int:
    """sum_{u=1}^{N} floor(u/m) in closed form."""
    if N <= 0:
        return 0
    q, r = divmod(N, m)
    return m * q * (q - 1) // 2 + q * (r + 1)


def sum_visible(n: int, m: int, E: int | None = None) -> int:
    """sum over t in [0, n) of min(E, floor((t+1)/m))."""
    E = n // m if E is None else E
    edge = E * m - 1                  # u <= edge is below the cap
    if n <= edge:
        return _floor_sum(n, m)
    return _floor_sum(edge, m) + E * (n - edge)


def _window(t: int, W: int) -> int:
    return min(W, t + 1) if W > 0 else 0


def sum_window(n: int, W: int) -> int:
    """sum over t in [0, n) of min(W, t+1)."""
    if W <= 0:
        return 0
    k = min(n, W)
    return k * (k + 1) // 2 + max(0, n - W) * W


def sum_selected(n: int, m: int, k: int) -> int:
    """sum over t of min(k, visible(t))."""
    return sum_visible(n, m, min(n // m, k))


def csa_layer_prefill(s: dict) -> dict:
    """Per-step work of one CSA layer's prefill (compression of KV and indexer
    keys, indexer, top-k, sparse attention)."""
    B, n, H, c, hI, dI, k, W = s["B"], s["n"], s["H"], s["c"], s["hI"], s["dI"], s["top_k"], s["n_win"]
    m = s["m"]
    es = 2 if s["dtype"] == "bf16" else 4
    E = n // m
    vis = sum_visible(n, m)
    sel = sum_selected(n, m, k)
    win = sum_window(n, W)
    q_bytes = B * n * H * c * es
    out = {"indexer_pairs": B * vis,
           "indexer_flops": B * 2 * dI * hI * vis,
           "csa_attn_flops": B * 4 * c * H * (sel + win),
           # compress reads C, Z (+ key C, Z), writes entries, keys and rotated raw rows
           "compress_bytes": B * n * (2 * c + 2 * dI) * es + B * (E * c + E * dI + n * c) * es,
           "indexer_bytes": B * (n * hI * dI * es + n * hI * 4 + E * dI * es),
           "topk_bytes": B * (vis * 4 + n * k * 4),
           "csa_attn_bytes": 2 * q_bytes + B * ((sel + win) * c * es + n * k * 4)}
    out["flops"] = out["indexer_flops"] + out["csa_attn_flops"]
    out["bytes"] = (out["compress_bytes"] + out["indexer_bytes"] + out["topk_bytes"]
                    + out["csa_attn_bytes"])
    out["query_tokens"] = B * n
    return out


def hca_layer_prefill(s: dict, m: int) -> dict:
    """Per-step work of one HCA layer's prefill with rate m (compression,
    dense attention over every visible entry)."""
    B, n, H, c, W = s["B"], s["n"], s["H"], s["c"], s["n_win"]
    es = 2 if s["dtype"] == "bf16" else 4
    E2 = n // m
    vis2 = sum_visible(n, m)
    win = sum_window(n, W)
    q_bytes = B * n * H * c * es
    out = {"hca_attn_flops": B * 4 * c * H * (vis2 + win),
           "compress_bytes": B * n * 2 * c * es + B * (E2 * c + n * c) * es,
           "hca_attn_bytes": 2 * q_bytes + B * (vis2 + win) * c * es}
    out["flops"] = out["hca_attn_flops"]
    out["bytes"] = out["compress_bytes"] + out["hca_attn_bytes"]
    out["query_tokens"] = B * n
    return out


def hybrid_prefill(s: dict) -> dict:
    """Per-step work of the interleaved CSA + HCA prefill (one CSA layer with
    rate m, one HCA layer with rate m2, over the same tokens)."""
    a = csa_layer_prefill(s)
    h = hca_layer_prefill(s, s.get("m2", s["m"]))
    out = dict(a)
    out["hca_attn_flops"] = h["hca_attn_flops"]
    out["hca_attn_bytes"] = h["hca_attn_bytes"]
    out["compress_bytes"] = a["compress_bytes"] + h["compress_bytes"]
    out["flops"] = a["flops"] + h["flops"]
    out["bytes"] = a["bytes"] + h["bytes"]
    return out


def decode(s: dict, hca: bool, lowp: bool = False) -> dict:
    """Per-step work of one decode step (one query per sequence).  lowp: the
    low-precision caches (an FP8 KV record of (c - 64) + 64 * 2 bytes plus
    four fp32 scales per entry, an MXFP4 key of dI / 2 bytes plus dI / 32
    scale bytes); window rows, queries and outputs stay in the dtype."""
    B, H, c, hI, dI, k, W, t = s["B"], s["H"], s["c"], s["hI"], s["dI"], s["top_k"], s["n_win"], s["t"]
    es = 2 if s["dtype"] == "bf16" else 4
    E = s.get("E", (t + 1) // s["m"])
    nv = visible(t, s["m"], E)
    sel = min(k, nv)
    win = _window(t, W)
    ent_b = (c - 64) + 64 * 2 + 16 if lowp else c * es        # bytes of one stored entry
    key_b = dI // 2 + dI // 32 if lowp else dI * es            # bytes of one indexer key
    out = {"indexer_flops": B * 2 * dI * hI * nv,
           "indexer_bytes": B * (nv * key_b + hI * dI * es + hI * 4),
           "csa_attn_flops": B * 4 * c * H * (sel + win),
           "csa_attn_bytes": B * (sel * ent_b + win * c * es + 2 * H * c * es + k * 4)}
    out["topk_bytes"] = B * (nv * 4 + k * 4)
    flops = out["indexer_flops"] + out["csa_attn_flops"]
    byts = out["indexer_bytes"] + out["csa_attn_bytes"]
    if hca:
        E2 = s.get("E2", (t + 1) // s["m2"])
        nv2 = visible(t, s["m2"], E2)
        out["hca_attn_flops"] = B * 4 * c * H * (nv2 + win)
        out["hca_attn_bytes"] = B * (nv2 * ent_b + win * c * es + 2 * H * c * es)
        flops += out["hca_attn_flops"]
        byts += out["hca_attn_bytes"]
    out["flops"] = flops
    out["bytes"] = byts
    out["query_tokens"] = B
    return out
