"""Pins for the fp64 oracle: worked examples and counts printed on the pages,
closed forms, invariants, special cases that reduce to textbook routines, and
brute force on tiny inputs.  Each test is chosen so that a plausible mistake
in the oracle (a dropped term, a wrong sign or index, a transposed operand,
softmax along the wrong axis) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------ compression

def test_compress_worked_example(orc):
    """Book ch.5 'A scalar worked example': weights (0.4,0.2,0.2,0.2) -> 9.6."""
    g = gold("compress_worked_example.json")
    m = g["m"]
    # two blocks of m tokens; entry 1 reads block 1 (branch a) and block 0 (branch b)
    C = np.zeros((2 * m, 1)); Z = np.zeros((2 * m, 1))
    Cb = np.zeros((2 * m, 1)); Zb = np.zeros((2 * m, 1))
    C[m:, 0] = g["current_values"]
    Z[m:, 0] = np.log(g["current_exp_logits"])
    Cb[:m, 0] = g["previous_values"]
    Zb[:m, 0] = np.log(g["previous_exp_logits"])
    bias = np.zeros((m, 1)); biasb = np.zeros((m, 1))
    e = orc.compress(C, Z, bias, m, overlap=1, Cb=Cb, Zb=Zb, biasb=biasb)
    assert e.shape == (2, 1)
    assert abs(e[1, 0] - g["expected"]) < 1e-12
    # swapping which current value carries the weight-2 logit does not give 9.6
    Z2 = Z.copy(); Z2[m:, 0] = Z[m:, 0][::-1]
    e2 = orc.compress(C, Z2, bias, m, overlap=1, Cb=Cb, Zb=Zb, biasb=biasb)
    assert abs(e2[1, 0] - g["expected"]) > 0.5
    # the bias is added to the logit: moving log 2 from Z into the bias gives the same value
    Z3 = Z.copy(); Z3[m:, 0] = 0.0
    bias3 = np.log(np.array(g["current_exp_logits"]))[:, None]
    e3 = orc.compress(C, Z3, bias3, m, overlap=1, Cb=Cb, Zb=Zb, biasb=biasb)
    assert abs(e3[1, 0] - g["expected"]) < 1e-12


def test_compress_first_block_has_no_previous_branch(orc):
    """Book ch.5: at the start the missing b branch has zero content and -inf
    logits, so entry 0 of the two-branch form equals the one-branch entry."""
    r = rng(1)
    n, c, m = 16, 5, 4
    C, Z, Cb, Zb = (r.standard_normal((n, c)) for _ in range(4))
    bias, biasb = r.standard_normal((m, c)), r.standard_normal((m, c))
    e2 = orc.compress(C, Z, bias, m, overlap=1, Cb=Cb, Zb=Zb, biasb=biasb)
    e1 = orc.compress(C, Z, bias, m)
    np.testing.assert_allclose(e2[0], e1[0], atol=1e-14)
    assert np.abs(e2[1:] - e1[1:]).max() > 1e-3


@pytest.mark.parametrize("overlap", [0, 1])
def test_compress_identical_tokens(orc, overlap):
    """A block of identical tokens compresses to that token (any logits, bias)."""
    r = rng(2)
    n, c, m = 32, 7, 4
    row = r.standard_normal(c)
    C = np.tile(row, (n, 1))
    Z = r.standard_normal((n, c)) * 3
    bias = r.standard_normal((m, c))
    kw = dict(overlap=overlap)
    if overlap:
        kw.update(Cb=C.copy(), Zb=r.standard_normal((n, c)), biasb=r.standard_normal((m, c)))
    e = orc.compress(C, Z, bias, m, **kw)
    np.testing.assert_allclose(e, np.tile(row, (n // m, 1)), atol=1e-13)


def test_compress_m1_is_identity(orc):
    r = rng(3)
    C, Z = r.standard_normal((9, 6)), r.standard_normal((9, 6))
    e = orc.compress(C, Z, r.standard_normal((1, 6)), 1)
    np.testing.assert_allclose(e, C, atol=1e-15)


@pytest.mark.parametrize("m", [4, 128])
def test_compress_convex_per_channel(orc, m):
    """Per-channel softmax over slots: each coordinate lies between the block's
    min and max of that coordinate (fails for a softmax across channels)."""
    r = rng(4)
    n, c = 2 * m + 3, 16
    C = r.standard_normal((n, c)) * np.arange(1, c + 1)     # channel scales differ
    Z = r.standard_normal((n, c))
    e = orc.compress(C, Z, 0.1 * r.standard_normal((m, c)), m)
    assert e.shape == (n // m, c)
    blocks = C[: (n // m) * m].reshape(n // m, m, c)
    assert np.all(e <= blocks.max(1) + 1e-12) and np.all(e >= blocks.min(1) - 1e-12)


def test_compress_shift_invariance_and_uniform(orc):
    """Adding one constant per channel to every slot logit changes nothing;
    equal logits give the plain mean of the block."""
    r = rng(5)
    n, c, m = 24, 8, 4
    C, Z = r.standard_normal((n, c)), r.standard_normal((n, c))
    bias = r.standard_normal((m, c))
    shift = r.standard_normal(c) * 5
    e0 = orc.compress(C, Z, bias, m)
    e1 = orc.compress(C, Z + shift, bias, m)
    np.testing.assert_allclose(e0, e1, atol=1e-12)
    eu = orc.compress(C, np.zeros((n, c)), np.zeros((m, c)), m)
    np.testing.assert_allclose(eu, C.reshape(n // m, m, c).mean(1), atol=1e-14)


def test_compress_extreme_logit_picks_slot(orc):
    """A very large logit on one slot selects that slot's content exactly."""
    n, c, m = 8, 3, 4
    C = np.arange(n * c, dtype=float).reshape(n, c)
    Z = np.zeros((n, c)); Z[2, :] = 800.0; Z[5, 1] = 800.0
    e = orc.compress(C, Z, np.zeros((m, c)), m)
    np.testing.assert_allclose(e[0], C[2], atol=1e-12)
    assert abs(e[1, 1] - C[5, 1]) < 1e-12


def test_compress_rope_position_is_block_end(orc):
    """A stored entry is rotated at its block's last position (j+1)m-1."""
    r = rng(6)
    n, c, m, rd = 16, 8, 4, 4
    C, Z = r.standard_normal((n, c)), r.standard_normal((n, c))
    bias = r.standard_normal((m, c))
    plain = orc.compress(C, Z, bias, m)
    rot = orc.compress(C, Z, bias, m, rope_dims=rd, theta=10000.0)
    for j in range(n // m):
        np.testing.assert_allclose(rot[j], orc.rope(plain[j], (j + 1) * m - 1, rd), atol=1e-13)
    np.testing.assert_allclose(rot[:, : c - rd], plain[:, : c - rd], atol=0)


# ---------------------------------------------------------------- rounding

def test_round_matches_torch_bf16_and_float(orc):
    """The oracle's bf16/f32 rounding of float32-representable values agrees with
    torch's conversion (a library routine) and with the generator's bit trick."""
    import torch
    r = rng(7)
    x32 = (r.standard_normal(20000) * np.exp(r.uniform(-20, 20, 20000))).astype(np.float32)
    x32[:4] = [1.00390625, 1.01171875, -1.00390625, 3.0e-39]   # ties and a subnormal
    ob = orc.round_to(x32.astype(np.float64), "bf16")
    tb = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ob, tb)
    np.testing.assert_array_equal(ob, synth.widen(synth.bf16_bits(x32), "bf16"))
    x64 = r.standard_normal(1000) * 1e3
    np.testing.assert_array_equal(orc.round_to(x64, "f32"), x64.astype(np.float32).astype(np.float64))


# ---------------------------------------------------------------- visibility

def test_visible_counts(orc):
    g = gold("visible_counts.json")
    for cs in g["cases"]:
        tok, m = cs["tokens"], cs["m"]
        # the query at the last position t = tokens - 1 sees every complete block
        v = orc.visible(tok - 1, m, 1 << 40)
        assert v == cs["entries"], cs
        assert tok - v * m == cs["tail"], cs


def test_visible_rule_brute_force(orc):
    """Entry j (positions jm..jm+m-1) is visible at t iff its last position <= t."""
    for m in (1, 2, 4, 8):
        for t in range(0, 40):
            brute = sum(1 for j in range(100) if j * m + m - 1 <= t)
            assert orc.visible(t, m, 100) == brute
    assert orc.visible(1000, 4, 10) == 10


# ----------------------------------------------------------------- indexer

def _scores_brute(qI, w, kI, t_pos, m):
    T, hI, dI = qI.shape
    E = kI.shape[0]
    out = np.full((T, E), -np.inf)
    for t in range(T):
        for j in range(E):
            if (j + 1) * m <= t_pos[t] + 1:
                out[t, j] = sum(w[t, h] * max(0.0, float(qI[t, h] @ kI[j])) for h in range(hI))
    return out


def test_index_scores_hand_example(orc):
    """Two heads, two dims: head 0 matches +, head 1 is clipped by ReLU."""
    qI = np.array([[[1.0, 0.0], [0.0, -1.0]]])           # [T=1, hI=2, dI=2]
    w = np.array([[0.8, 0.2]])
    kI = np.array([[2.0, 1.0], [1.0, -3.0], [-1.0, 0.5]])
    s = orc.index_scores(qI, w, np.array([11]), kI, 4)   # t=11 sees 3 entries
    np.testing.assert_allclose(s[0], [0.8 * 2.0, 0.8 * 1.0 + 0.2 * 3.0, 0.0], atol=1e-15)
    s = orc.index_scores(qI, w, np.array([6]), kI, 4)    # t=6 sees 1 entry
    assert s[0, 0] == 1.6 and np.isneginf(s[0, 1:]).all()


def test_index_scores_brute_linear_nonneg(orc):
    r = rng(8)
    T, hI, dI, E, m = 9, 3, 5, 6, 2
    qI, kI = r.standard_normal((T, hI, dI)), r.standard_normal((E, dI))
    w = r.standard_normal((T, hI))
    pos = np.arange(T) + 3
    s = orc.index_scores(qI, w, pos, kI, m)
    np.testing.assert_allclose(s, _scores_brute(qI, w, kI, pos, m), atol=1e-12)
    # linear in w
    w2 = r.standard_normal((T, hI))
    s2 = orc.index_scores(qI, w2, pos, kI, m)
    s12 = orc.index_scores(qI, 2 * w - 3 * w2, pos, kI, m)
    fin = np.isfinite(s)
    with np.errstate(invalid="ignore"):
        lin = 2 * s - 3 * s2
    np.testing.assert_allclose(s12[fin], lin[fin], atol=1e-12)
    # nonnegative weights give nonnegative scores
    assert (orc.index_scores(qI, np.abs(w), pos, kI, m)[fin] >= 0).all()


# ------------------------------------------------------------------- top-k

def _topk_brute(s_row, nv, k):
    """Exhaustive: the unique k-subset S of the visible entries such that every
    member beats every non-member by (score desc, index asc)."""
    if nv <= k:
        return list(range(nv))
    def beats(i, j):
        return s_row[i] > s_row[j] or (s_row[i] == s_row[j] and i < j)
    found = []
    for S in itertools.combinations(range(nv), k):
        Sset = set(S)
        if all(beats(i, j) for i in S for j in range(nv) if j not in Sset):
            found.append(list(S))
    assert len(found) == 1
    return found[0]


def test_topk_exhaustive_small(orc):
    r = rng(9)
    m = 1
    for trial in range(40):
        E = int(r.integers(1, 12))
        k = int(r.integers(1, 6))
        T = 3
        s = np.round(r.standard_normal((T, E)) * 2) / 2       # many exact ties
        pos = r.integers(0, E + 2, T)
        idx, cnt = orc.topk(s, pos, m, k)
        for t in range(T):
            nv = min(E, pos[t] + 1)
            want = _topk_brute(s[t], nv, k)
            assert cnt[t] == len(want)
            assert list(idx[t, : cnt[t]]) == want
            assert (idx[t, cnt[t]:] == -1).all()


def test_topk_all_when_few_and_ties_to_lower_index(orc):
    s = np.array([[5.0, 1.0, 5.0, 5.0, 0.0, -0.0, 2.0]])
    idx, cnt = orc.topk(s, np.array([6]), 1, 2)
    assert list(idx[0]) == [0, 2] and cnt[0] == 2
    idx, cnt = orc.topk(s, np.array([6]), 1, 5)
    assert list(idx[0]) == [0, 1, 2, 3, 6]
    # -0.0 and +0.0 tie; the lower index wins
    s2 = np.array([[-0.0, 0.0, -1.0]])
    idx, _ = orc.topk(s2, np.array([2]), 1, 1)
    assert list(idx[0]) == [0]
    idx, cnt = orc.topk(s, np.array([6]), 1, 10)     # fewer visible than k: keep all
    assert cnt[0] == 7 and list(idx[0, :7]) == list(range(7)) and (idx[0, 7:] == -1).all()
    idx, cnt = orc.topk(s, np.array([2]), 4, 3)      # t=2, m=4: nothing visible
    assert cnt[0] == 0 and (idx[0] == -1).all()


# --------------------------------------------------------------- attention

def rope_complex(x, pos, r, theta=10000.0):
    """RoPE written as complex multiplication (independent of the oracle's
    real-pair form): pairs (c-r+2i, c-r+2i+1) times exp(i * pos * theta^(-2i/r))."""
    x = np.array(x, dtype=np.float64, copy=True)
    if r == 0:
        return x
    c = x.shape[-1]
    z = x[..., c - r::2] + 1j * x[..., c - r + 1::2]
    freqs = theta ** (-np.arange(0, r, 2) / r)
    z = z * np.exp(1j * np.asarray(pos, dtype=np.float64)[..., None] * freqs)
    x[..., c - r::2] = z.real
    x[..., c - r + 1::2] = z.imag
    return x


def test_rope_matches_complex_form_and_relative(orc):
    r = rng(10)
    c, rd = 12, 8
    x = r.standard_normal(c)
    for p in (0, 1, 7, 131072, 1048576):
        np.testing.assert_allclose(orc.rope(x, p, rd), rope_complex(x, p, rd), atol=1e-9)
    # q.k depends only on the position difference (Book ch.7, Partial RoPE)
    q, k = r.standard_normal(c), r.standard_normal(c)
    d0 = orc.rope(q, 100, rd) @ orc.rope(k, 37, rd)
    d1 = orc.rope(q, 100 + 5000, rd) @ orc.rope(k, 37 + 5000, rd)
    assert abs(d0 - d1) < 1e-10
    np.testing.assert_allclose(orc.rope(orc.rope(x, 123, rd), -123, rd), x, atol=1e-13)


@pytest.mark.parametrize("pos0", [0, 1, 127, 4093, (1 << 20) - 128])
def test_rope_rows_rotates_row_l_at_pos0_plus_l(orc, pos0):
    """Stored raw rows: row l of a block starting at pos0 is rotated at
    pos0 + l ([Book] ch.7 "Partial rotary position embeddings": a key is
    rotated at its own position).  Checked row by row against the complex
    form at the row's own position, so an off-by-one in the row position
    (pos0 + l + 1, or pos0 for every row) fails."""
    r = rng(pos0 % 1000 + 17)
    L, c, rd = 6, 16, 8
    x = r.standard_normal((L, c))
    got = orc.rope_rows(x, pos0, rd, 10000.0, "f64")
    for l in range(L):
        np.testing.assert_allclose(got[l], rope_complex(x[l], pos0 + l, rd), atol=1e-9)
    # a neighbouring position is distinguishable at these sizes
    assert np.abs(got[1] - rope_complex(x[1], pos0 + 2, rd)).max() > 1e-3
    # rounding to the storage dtype happens after the rotation, once
    gb = orc.rope_rows(x, pos0, rd, 10000.0, "bf16")
    for l in range(L):
        want = synth.widen(synth.to_storage(rope_complex(x[l], pos0 + l, rd), "bf16"), "bf16")
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(want), 1e-30))) - 7)
        assert np.all(np.abs(gb[l] - want) <= ulp)


def test_sink_mass_example(orc):
    """Book ch.7 'Attention sinks': real mass 4, sink mass 6 -> real weights 0.4."""
    g = gold("sink_mass_example.json")
    c = 4
    v = np.array([[1.0, -2.0, 3.0, 0.5]])                   # one real entry (no window)
    q = np.zeros((1, 1, c)); q[0, 0, 0] = np.log(g["real_mass"]) * np.sqrt(c) / v[0, 0]
    sink = np.array([np.log(g["sink_mass"])])
    out, lse = orc.attend(q, np.array([3]), v, 4, np.zeros((1, c)), 0, sink, idx=np.array([[0]]),
                          n_win=0, rope_dims=0, derotate=0, want_lse=True)
    np.testing.assert_allclose(out[0, 0], g["expected_real_weight_sum"] * v[0], atol=1e-14)
    assert abs(lse[0, 0] - np.log(g["real_mass"] + g["sink_mass"])) < 1e-13


def _dense_attention_brute(q, qpos, cols, col_ok, sink, scale, rd, derot):
    """Explicit masked matrix: q [T,H,c] (unrotated), cols [N,c] stored (rotated)
    rows, col_ok [T,N] bool mask; plain softmax with one extra sink column."""
    T, H, c = q.shape
    out = np.zeros((T, H, c))
    for t in range(T):
        qt = rope_complex(q[t], np.full(H, qpos[t]), rd)          # [H, c]
        logits = (qt @ cols.T) * scale                             # [H, N]
        logits = np.where(col_ok[t][None, :], logits, -np.inf)
        full = np.concatenate([logits, sink[:, None]], axis=1)
        mx = full.max(1, keepdims=True)
        p = np.exp(full - mx)
        p /= p.sum(1, keepdims=True)
        o = p[:, :-1] @ cols
        if derot:
            o = rope_complex(o, np.full(H, -qpos[t]), rd)
        out[t] = o
    return out


@pytest.mark.parametrize("m,k,n_win,derot", [(4, 3, 5, 1), (2, 2, 3, 0), (4, 100, 4, 1), (1, 1, 1, 1)])
def test_csa_prefill_brute_force(orc, m, k, n_win, derot):
    """Whole CSA prefill on tiny n against an explicit (T x (E + n)) mask with a
    dense softmax, the mask built from brute-force top-k and window rules."""
    r = rng(11 + m + k)
    n, H, c, rd, hI, dI = 13, 2, 6, 4, 2, 3
    C, Z = r.standard_normal((n, c)), r.standard_normal((n, c))
    bias = 0.1 * r.standard_normal((m, c))
    Ck, Zk = r.standard_normal((n, dI)), r.standard_normal((n, dI))
    biask = 0.1 * r.standard_normal((m, dI))
    q, qI = r.standard_normal((n, H, c)), r.standard_normal((n, hI, dI))
    w = r.standard_normal((n, hI))
    sink = r.standard_normal(H)
    pos = np.arange(n)
    kvc = orc.compress(C, Z, bias, m, rope_dims=rd)
    kIc = orc.compress(Ck, Zk, biask, m)
    raw = orc.rope_rows(C, 0, rd, 10000.0, "f64")
    sc = orc.index_scores(qI, w, pos, kIc, m)
    idx, cnt = orc.topk(sc, pos, m, k)
    out = orc.attend(q, pos, kvc, m, raw, 0, sink, idx=idx, n_win=n_win, rope_dims=rd, derotate=derot)
    # brute-force mask
    E = kvc.shape[0]
    cols = np.concatenate([kvc, raw])
    ok = np.zeros((n, E + n), bool)
    for t in range(n):
        nv = sum(1 for j in range(E) if (j + 1) * m <= t + 1)
        for j in _topk_brute(sc[t], nv, k):
            ok[t, j] = True
        for p in range(max(0, t - n_win + 1), t + 1):
            ok[t, E + p] = True
    ref = _dense_attention_brute(q, pos, cols, ok, sink, 1 / np.sqrt(c), rd, derot)
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_causal_attention_special_case(orc):
    """m = 1, no window, k >= t+1, sink -inf, no de-rotation: textbook causal
    attention softmax(QK^T/sqrt(c) + causal mask) V with K = V = RoPE'd rows."""
    r = rng(12)
    n, H, c, rd = 10, 3, 8, 4
    X = r.standard_normal((n, c))
    q = r.standard_normal((n, H, c))
    kvc = orc.compress(X, r.standard_normal((n, c)), np.zeros((1, c)), 1, rope_dims=rd)
    pos = np.arange(n)
    idx = np.tile(np.arange(n, dtype=np.int32), (n, 1))
    idx[np.arange(n)[:, None] < np.arange(n)[None, :]] = -1
    out = orc.attend(q, pos, kvc, 1, np.zeros((1, c)), 0, np.full(H, -np.inf), idx=idx,
                     n_win=0, rope_dims=rd, derotate=0)
    K = rope_complex(X, pos, rd)
    for h in range(H):
        Q = rope_complex(q[:, h], pos, rd)
        S = Q @ K.T / np.sqrt(c) + np.triu(np.full((n, n), -np.inf), 1)
        P = np.exp(S - S.max(1, keepdims=True)); P /= P.sum(1, keepdims=True)
        np.testing.assert_allclose(out[:, h], P @ K, atol=1e-12)


def test_csa_equals_dense_when_k_covers_all(orc):
    """k >= |visible| reduces CSA to HCA-style dense attention (two oracle routes:
    the selected-index path and the every-visible-entry path)."""
    r = rng(13)
    n, H, c, m, rd = 40, 2, 8, 4, 4
    kvc = r.standard_normal((n // m, c))
    raw = r.standard_normal((n, c))
    q = r.standard_normal((n, H, c))
    sink = r.standard_normal(H)
    pos = np.arange(n)
    sc = r.standard_normal((n, n // m))
    idx, _ = orc.topk(sc, pos, m, n)
    a = orc.attend(q, pos, kvc, m, raw, 0, sink, idx=idx, n_win=7, rope_dims=rd)
    b = orc.attend(q, pos, kvc, m, raw, 0, sink, idx=None, n_win=7, rope_dims=rd)
    np.testing.assert_allclose(a, b, atol=1e-13)
    # and a smaller k really does change the answer
    idx2, _ = orc.topk(sc, pos, m, 2)
    c2 = orc.attend(q, pos, kvc, m, raw, 0, sink, idx=idx2, n_win=7, rope_dims=rd)
    assert np.abs(c2 - b).max() > 1e-3


def test_sink_minus_inf_is_plain_softmax_and_weights_bounded(orc):
    r = rng(14)
    T, H, c = 3, 4, 6
    kv = r.standard_normal((5, c))
    q = r.standard_normal((T, H, c))
    pos = np.array([19, 20, 21])
    idx = np.tile(np.arange(5, dtype=np.int32), (T, 1))
    a = orc.attend(q, pos, kv, 4, np.zeros((1, c)), 0, np.full(H, -np.inf), idx=idx, n_win=0,
                   rope_dims=0, derotate=0)
    for t in range(T):
        for h in range(H):
            lg = kv @ q[t, h] / np.sqrt(c)
            p = np.exp(lg - lg.max()); p /= p.sum()
            np.testing.assert_allclose(a[t, h], p @ kv, atol=1e-13)
    # a finite sink shrinks every output toward 0 by the factor sum(e^l)/(e^z+sum(e^l))
    z = r.standard_normal(H)
    b = orc.attend(q, pos, kv, 4, np.zeros((1, c)), 0, z, idx=idx, n_win=0, rope_dims=0, derotate=0)
    for t in range(T):
        for h in range(H):
            lg = kv @ q[t, h] / np.sqrt(c)
            f = np.exp(lg).sum() / (np.exp(z[h]) + np.exp(lg).sum())
            np.testing.assert_allclose(b[t, h], f * a[t, h], atol=1e-13)


def test_derotation_gives_relative_rotation(orc):
    """Book ch.7 'Why the output is de-rotated': with de-rotation the rotary part
    of the output is sum_j a_j R_{p_j - t} v_j (v_j unrotated content)."""
    r = rng(15)
    c, rd, H = 8, 4, 1
    t = 50
    V = r.standard_normal((6, c))                     # unrotated content
    p_j = np.array([3, 7, 11, 15, 19, 23])            # entry positions (m=4 block ends)
    stored = np.stack([rope_complex(V[i], p_j[i], rd) for i in range(6)])
    q = r.standard_normal((1, H, c))
    idx = np.arange(6, dtype=np.int32)[None]
    o = orc.attend(q, np.array([t]), stored, 4, np.zeros((1, c)), 0, np.array([-np.inf]),
                   idx=idx, n_win=0, rope_dims=rd, derotate=1)
    qt = rope_complex(q[0, 0], t, rd)
    lg = stored @ qt / np.sqrt(c)
    a = np.exp(lg - lg.max()); a /= a.sum()
    want = sum(a[i] * rope_complex(V[i], p_j[i] - t, rd) for i in range(6))
    np.testing.assert_allclose(o[0, 0], want, atol=1e-12)


def test_empty_history_and_sink_only(orc):
    """t = 0 with m = 4: no compressed entry; the window holds the token itself."""
    c, rd = 4, 2
    raw = np.array([[1.0, 2.0, 3.0, 4.0]])
    q = np.ones((1, 1, c))
    o = orc.attend(q, np.array([0]), np.zeros((0, c)), 4, raw, 0, np.array([-np.inf]),
                   idx=np.full((1, 2), -1, np.int32), n_win=128, rope_dims=rd, derotate=0)
    np.testing.assert_allclose(o[0, 0], raw[0], atol=1e-15)
    # nothing at all to read: output is zero, lse = sink
    o, lse = orc.attend(q, np.array([0]), np.zeros((0, c)), 4, raw, 0, np.array([0.7]),
                        idx=np.full((1, 2), -1, np.int32), n_win=0, rope_dims=rd, want_lse=True)
    assert (o == 0).all() and abs(lse[0, 0] - 0.7) < 1e-15


def test_window_bounds(orc):
    """The window is positions t-n_win+1 .. t, the query's own row included."""
    r = rng(16)
    n, c = 20, 4
    raw = r.standard_normal((n, c))
    q = r.standard_normal((n, 1, c))
    pos = np.arange(n)
    o = orc.attend(q, pos, np.zeros((0, c)), 4, raw, 0, np.array([-np.inf]), idx=None,
                   n_win=3, rope_dims=0, derotate=0)
    for t in range(n):
        rows = raw[max(0, t - 2): t + 1]
        lg = rows @ q[t, 0] / 2.0
        p = np.exp(lg - lg.max()); p /= p.sum()
        np.testing.assert_allclose(o[t, 0], p @ rows, atol=1e-13)
    with pytest.raises(ValueError):
        orc.attend(q[:1], np.array([5]), np.zeros((0, c)), 4, raw[:2], 0, np.array([0.0]),
                   idx=None, n_win=3, rope_dims=0)


# --------------------------------------------------- workloads end to end

def test_workload_prefill_small_runs(orc):
    """The composed CSA + HCA prefill on a shrunken workload (f32 and bf16)."""
    s, x = synth.make_inputs("csa_prefill_f32", n=64)
    st = orc.csa_prefill_seq(s, x, 0, return_steps=True)
    assert st["out"].shape == (64, 4, 64) and np.isfinite(st["out"]).all()
    assert st["kvc"].shape == (16, 64)
    # stored entries are f32-representable, the raw rows too
    assert (st["kvc"] == st["kvc"].astype(np.float32)).all()
    s2, x2 = synth.make_inputs("hca_prefill_bf16", n=384)
    o2 = orc.hca_prefill_seq(s2, x2, 0)
    assert o2.shape == (384, 16, 128) and np.isfinite(o2).all()
