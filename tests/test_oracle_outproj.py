"""Pins for the query / KV RMSNorm and the grouped output projection of the
oracle (oracle/outproj.py): the weight counts the pages print, closed forms of
RMSNorm, the grouped projection against the single block-structured matrix it
amounts to, and the order of the norm and RoPE."""
import json
import os

import numpy as np

from oracle import outproj

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def test_projection_counts_match_pages():
    g = json.load(open(os.path.join(GOLD, "out_proj_counts.json")))
    assert g["heads_per_group"] * 512 == g["group_in"]
    f = g["flash"]
    assert f["H"] * f["c"] == f["coords"]
    w = outproj.projection_weights(f["H"], f["c"], f["d"], g["d_g"], g["heads_per_group"])
    assert w["grouped"] / w["direct"] == f["ratio"]
    p = g["pro"]
    assert p["H"] * p["c"] == p["coords"] and p["H"] // g["heads_per_group"] == p["groups"]
    w = outproj.projection_weights(p["H"], p["c"], p["d"], g["d_g"], g["heads_per_group"])
    r = w["grouped"] / w["direct"]
    assert abs(r - p["ratio_approx"]) < 5e-4 and abs((1 - r) - p["reduction_approx"]) < 5e-4


def test_rmsnorm_closed_forms():
    x = np.array([3.0, 4.0])
    y = outproj.rmsnorm(x, np.ones(2), eps=0.0)
    assert np.allclose(y, x / np.sqrt(12.5), rtol=0, atol=1e-15)
    r = rng(0)
    x = r.standard_normal((10, 64))
    g = r.uniform(0.5, 2.0, 64)
    # unit gain: mean square ms / (ms + eps)
    y = outproj.rmsnorm(x, np.ones(64))
    ms = np.mean(x * x, -1)
    assert np.allclose(np.mean(y * y, -1), ms / (ms + outproj.EPS), rtol=1e-12)
    # without eps, invariant to a positive scale of the input; the gain multiplies per coordinate
    assert np.allclose(outproj.rmsnorm(7.5 * x, g, 0.0), outproj.rmsnorm(x, g, 0.0), rtol=1e-13)
    assert np.allclose(outproj.rmsnorm(x, g), outproj.rmsnorm(x, np.ones(64)) * g, rtol=1e-15)


def test_grouped_projection_is_block_structured_direct_map():
    r = rng(1)
    T, H, c, hpg, dg, d = 5, 16, 8, 8, 4, 6
    o = r.standard_normal((T, H, c))
    w_g = r.standard_normal((H // hpg, hpg * c, dg))
    w_o = r.standard_normal((H // hpg * dg, d))
    z = outproj.grouped_out_proj(o, w_g, w_o, hpg)
    z_direct = o.reshape(T, H * c) @ outproj.direct_weight(w_g, w_o)
    assert np.allclose(z, z_direct, rtol=1e-12, atol=1e-12)
    # a group's heads only reach the output through its own matrix
    o2 = o.copy()
    o2[:, :hpg] = 0.0
    w_g2 = w_g.copy()
    w_g2[0] = r.standard_normal(w_g2[0].shape)
    assert np.allclose(outproj.grouped_out_proj(o2, w_g, w_o, hpg),
                       outproj.grouped_out_proj(o2, w_g2, w_o, hpg), rtol=1e-12, atol=1e-12)


def test_norm_before_rope(orc):
    """Rotation keeps each pair's length, so with a gain equal on both members of
    every rotary pair the norm and the rotation commute; with another gain the
    order matters and the oracle normalises first."""
    r = rng(2)
    c, rd = 64, 32
    x = r.standard_normal(c)
    g = r.uniform(0.5, 2.0, c)
    g[c - rd:] = np.repeat(r.uniform(0.5, 2.0, rd // 2), 2)
    a = orc.rope(outproj.rmsnorm(x, g), 123.0, rd)
    b = outproj.rmsnorm(orc.rope(x, 123.0, rd), g)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    g[c - rd:] = r.uniform(0.5, 2.0, rd)
    a = orc.rope(outproj.rmsnorm(x, g), 123.0, rd)
    b = outproj.rmsnorm(orc.rope(x, 123.0, rd), g)
    assert not np.allclose(a, b)
