"""Pins for the low-precision cache formats of the oracle (oracle/lowp.py):
the payload sizes the pages print, library casts of the same formats, every
grid value and tie of the FP8 / FP4 definitions, the OCP block-scale rule,
and a cross-check of the low-precision index scores against the full-precision
oracle routine on inputs that the formats hold exactly."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import lowp

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def test_payload_matches_pages():
    g = json.load(open(os.path.join(GOLD, "lowp_payload.json")))
    b = lowp.entry_payload_bytes(g["c"], g["rope_dims"], g["dI"])
    assert b["kv"] / g["m_csa"] == g["csa_main_bytes_per_token"]
    assert b["kv"] / g["m_hca"] == g["hca_main_bytes_per_token"]
    assert b["index_key"] == g["index_key_bytes"]
    assert b["index_key"] / g["m_csa"] == g["csa_index_bytes_per_token"]
    assert (b["kv"] + b["index_key"]) / g["m_csa"] == g["csa_total_bytes_per_token"]


# ------------------------------------------------------------------ FP8 E4M3

def test_e4m3_grid():
    v = lowp.e4m3_values()
    assert len(v) == 127 and v[0] == 0.0 and v[-1] == 448.0
    assert v[1] == 2.0 ** -9 and 2.0 ** -6 in v
    assert np.array_equal(lowp.e4m3_round(v), v)
    assert np.array_equal(lowp.e4m3_round(-v), -v)


def test_e4m3_hand_values():
    # ties go to the even mantissa; past the top the value saturates
    cases = {1.0625: 1.0, 1.1875: 1.25, 17.0: 16.0, 19.0: 20.0, 2.0 ** -10: 0.0,
             3 * 2.0 ** -10: 2.0 ** -8, 464.0: 448.0, 470.0: 448.0, 1e9: 448.0}
    for x, want in cases.items():
        assert lowp.e4m3_round(x) == want, x
        assert lowp.e4m3_round(-x) == -want, -x


def test_e4m3_matches_library_cast():
    v = lowp.e4m3_values()
    mids = (v[:-1] + v[1:]) / 2                       # exact ties
    r = rng(0)
    x = np.concatenate([mids, -mids, r.uniform(-448, 448, 20000),
                        r.standard_normal(20000) * 2.0 ** r.integers(-12, 8, 20000)])
    x = x.astype(np.float32).astype(np.float64)       # single rounding in the library cast
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(lowp.e4m3_round(x), ref)


# ------------------------------------------------------------- FP4 E2M1, MX

def _e2m1_mant(v):
    # mantissa bit of an E2M1 value: 0.5 (subnormal), 1.5, 3 and 6 have it set
    return 1 if v in (0.5, 1.5, 3.0, 6.0) else 0


def test_e2m1_ties():
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
             7.0: 6.0, 100.0: 6.0, 0.0: 0.0}
    for x, want in cases.items():
        assert lowp.e2m1_round(x) == want, x
        assert lowp.e2m1_round(-x) == -want, -x


def test_e2m1_brute_force():
    r = rng(1)
    x = np.concatenate([r.uniform(-8, 8, 5000), np.arange(-7, 7.25, 0.25)])
    got = lowp.e2m1_round(x)
    want = np.array([lowp.nearest_even(v, lowp.E2M1_GRID, _e2m1_mant) for v in x])
    assert np.array_equal(got, want)


def test_mxfp4_scale_rule():
    g = lowp.E2M1_GRID
    # a block whose largest magnitude is 6 has scale 1: grid values survive
    blk = np.concatenate([g, -g, g, -g])              # 32 values, amax 6
    assert np.array_equal(lowp.mxfp4(blk), blk)
    # amax 1 -> shared exponent floor(log2 1) - 2 = -2: scale 1/4
    blk = np.zeros(32)
    blk[0], blk[1], blk[2] = 1.0, 0.3, -0.05
    q = lowp.mxfp4(blk)
    assert q[0] == 1.0 and q[1] == 0.25 and q[2] == 0.0      # 0.3 / 0.25 = 1.2 -> 1; -0.2 -> -0
    # amax 7.5 -> scale 1 and 7.5 saturates at 6
    blk = np.zeros(32)
    blk[5] = 7.5
    assert lowp.mxfp4(blk)[5] == 6.0
    # zeros stay zero; blocks are independent
    two = np.concatenate([np.zeros(32), np.linspace(-3, 3, 32)])
    q2 = lowp.mxfp4(two)
    assert np.all(q2[:32] == 0.0)
    assert np.array_equal(q2[32:], lowp.mxfp4(two[32:]))


def test_mxfp4_error_bound():
    r = rng(2)
    x = r.standard_normal((64, 128)) * 2.0 ** r.integers(-6, 6, (64, 1))
    q = lowp.mxfp4(x)
    blocks = x.reshape(64, 4, 32)
    scale = np.exp2(np.floor(np.log2(np.abs(blocks).max(-1, keepdims=True))) - 2)
    err = np.abs(q.reshape(64, 4, 32) - blocks)
    # half a step of the top binade (step 2 * scale), or the saturation loss at the top
    sat = np.maximum(np.abs(blocks) - 6 * scale, 0)
    assert np.all(err <= scale + sat + 1e-300)


# ----------------------------------------------------------------- BF16

def test_bf16_round_matches_library_cast():
    r = rng(3)
    x = (r.standard_normal(50000) * 2.0 ** r.integers(-40, 40, 50000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(lowp.bf16_round(x.astype(np.float64)), ref)


# ---------------------------------------------------------------- KV entry

def test_kv_entry_fp8():
    r = rng(4)
    e = r.standard_normal((16, 512))
    q = lowp.kv_entry_fp8(e, rope_dims=64, group=128)
    # rotary dims: BF16
    assert np.array_equal(q[:, 448:], lowp.bf16_round(e[:, 448:].astype(np.float32)))
    # non-rotary dims: each group's largest magnitude maps onto the top of the E4M3 range,
    # every value within half a step (3 mantissa bits) of its scaled input
    for g0, g1 in ((0, 128), (128, 256), (256, 384), (384, 448)):
        p32 = e[:, g0:g1].astype(np.float32)
        s32 = (np.abs(p32).max(-1, keepdims=True) / np.float32(448.0)).astype(np.float32)
        part, scale = p32.astype(np.float64), s32.astype(np.float64)
        y = part / scale
        # the stored codes are those of the fp32 quotient; they differ from the exact
        # quotient's only where the two straddle an E4M3 midpoint
        y32 = (p32 / s32).astype(np.float64)
        assert np.array_equal(q[:, g0:g1], lowp.e4m3_round(y32) * scale)
        assert np.mean(lowp.e4m3_round(y32) != lowp.e4m3_round(y)) < 1e-3
        normal = np.abs(y) >= 2.0 ** -6
        assert np.all(np.abs(q[:, g0:g1] - part)[normal] <= (np.abs(part) * 2.0 ** -4)[normal] * (1 + 1e-12))
    # an all-zero group stays zero
    z = np.zeros((1, 512))
    assert np.all(lowp.kv_entry_fp8(z) == 0.0)


# ---------------------------------------------------------- index scores

def test_index_scores_lowp_cross_check(orc):
    """On inputs MXFP4 holds exactly, the low-precision scores are the oracle's
    full-precision scores rounded once to BF16."""
    r = rng(5)
    T, hI, dI, E, m = 6, 4, 64, 40, 4
    g = lowp.E2M1_GRID

    def exact_mx(shape):
        v = r.choice(np.concatenate([g, -g]), size=shape)
        v[..., ::32] = 6.0                              # every block's largest magnitude is 6
        return v * 2.0 ** r.integers(-3, 3, shape[:-1] + (1,))
    qI, kI = exact_mx((T, hI, dI)), exact_mx((E, dI))
    w = r.uniform(0, 1, (T, hI))
    q_pos = np.arange(T) * 30 + 7
    lo = lowp.index_scores_lowp(qI, w, q_pos, kI, m)
    hi = orc.index_scores(qI, w, q_pos, kI, m)
    vis = np.isfinite(hi)
    assert np.array_equal(np.isfinite(lo), vis)
    assert np.array_equal(lo[vis], lowp.bf16_round(hi[vis]))
    assert np.all(lo[vis] >= 0)                         # w >= 0


def test_bf16_scores_tie_to_lower_index(orc):
    """Scores that differ in fp32 but round to the same BF16 value tie, and the
    top-k keeps the lower index."""
    s = np.array([[1.0, 1.0 + 2.0 ** -10, 0.5, 1.0 + 2.0 ** -9]])
    b = lowp.bf16_round(s)
    assert b[0, 0] == b[0, 1] == b[0, 3] == 1.0
    idx, cnt = orc.topk(b, np.array([15]), 4, 2)
    assert cnt[0] == 2 and list(idx[0]) == [0, 1]
    idx, _ = orc.topk(s, np.array([15]), 4, 2)         # in full precision 3 and 1 win
    assert list(idx[0]) == [1, 3]
