"""GPU parity: every C-ABI entry point against the fp64 oracle on the same
seeded inputs, at sizes that span several tiles and a ragged tail, plus the
five workloads (full size where the oracle can follow, sampled outputs where
it cannot), edge cases, the device status word, determinism and batch
invariance.  Tolerances are in tests/parity.py."""
import numpy as np
import pytest
import torch

import synth
from parity import (check_close, compare_topk, dev, gap_rows, host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_sparse_22_b300 as m
    m.lib()
    return m


def _np_rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------- compression

@pytest.mark.parametrize("dtype,n,c,m,r,overlap,sc", [
    ("f32", 2048, 64, 4, 32, 0, 1.0),
    ("f32", 2046, 64, 4, 32, 1, 1.0),         # ragged tail, two branches
    ("bf16", 1030, 512, 4, 64, 0, 1.0),
    ("bf16", 1024, 128, 4, 0, 1, 1.0),        # indexer-key form, two branches
    ("bf16", 8192 + 37, 128, 128, 64, 0, 128 ** -0.5),
    ("f32", 300, 64, 1, 32, 0, 1.0),          # m = 1
])
def test_compress(csa, orc, dtype, n, c, m, r, overlap, sc):
    B = 2
    seed = 100 + n + m
    C_ = synth.normal(seed, 1, (B, n, c), sc, dtype)
    Z = synth.normal(seed, 2, (B, n, c), sc, dtype)
    bias = synth.normal(seed, 3, (m, c), 0.1, "f32")
    kw = {}
    if overlap:
        kw = dict(Cb=synth.normal(seed, 4, (B, n, c), sc, dtype),
                  Zb=synth.normal(seed, 5, (B, n, c), sc, dtype),
                  biasb=synth.normal(seed, 6, (m, c), 0.1, "f32"))
    dkw = {k: dev(v) for k, v in kw.items()}
    out, raw = csa.csa_compress(dev(C_), dev(Z), dev(bias), m=m, overlap=overlap, rope_dims=r,
                                want_raw=True, **dkw)
    torch.cuda.synchronize()
    for b in range(B):
        ref = orc.compress(C_[b], Z[b], bias, m, overlap=overlap,
                           Cb=kw["Cb"][b] if overlap else None, Zb=kw["Zb"][b] if overlap else None,
                           biasb=kw.get("biasb"), rope_dims=r, out_dtype=dtype)
        g = host(out[b])
        if dtype == "f32":
            check_close(g, ref, "f32", "entries")
        else:   # stored bf16 entries: at most one bf16 step apart
            assert np.all(np.abs(g - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-5), "entries"
        rref = orc.rope_rows(C_[b], 0, r, 10000.0, dtype)
        gr = host(raw[b])
        if dtype == "f32":
            check_close(gr, rref, "f32", "raw rows")
        else:
            assert np.all(np.abs(gr - rref) <= 2.0 ** -7 * np.abs(rref) + 1e-5), "raw rows"


# ----------------------------------------------------------------- indexer

@pytest.mark.parametrize("dtype,B,T,hI,dI,E,m,pos0", [
    ("f32", 1, 2048, 4, 32, 512, 4, 0),
    ("bf16", 2, 40, 64, 128, 2100, 4, 8000),
    ("bf16", 2, 37, 64, 128, 1500, 4, 3000),      # a last query block with one token
    ("bf16", 3, 1, 64, 128, 5000, 4, 19999),      # decode shape
    ("bf16", 1, 33, 16, 64, 300, 2, 500),
])
def test_indexer_score(csa, orc, dtype, B, T, hI, dI, E, m, pos0):
    seed = 200 + T + E
    qI = synth.normal(seed, 1, (B, T, hI, dI), 1.0, dtype)
    kI = synth.normal(seed, 2, (B, E, dI), 1.0, dtype)
    w = synth.softmax_normal(seed, 3, (B, T, hI))
    w[..., ::3] *= -1.0                                # signs are unconstrained
    pos = np.tile(pos0 + np.arange(T, dtype=np.int64) * (1 if T > 1 else 0), (B, 1))
    if pos0 == 0:
        pos = np.tile(np.arange(T, dtype=np.int64), (B, 1))
    s = csa.indexer_score(dev(qI), dev(w), dev(kI), dev(pos), m)
    g = host(s)
    for b in range(B):
        ref = orc.index_scores(qI[b], w[b], pos[b], kI[b], m)
        fin = np.isfinite(ref)
        assert np.array_equal(np.isfinite(g[b]), fin)
        assert np.all(np.isneginf(g[b][~fin]))
        scale = np.abs(ref[fin]).max() if fin.any() else 1.0
        assert np.abs(g[b][fin] - ref[fin]).max() <= 2e-6 * scale


# ------------------------------------------------------------------- top-k

@pytest.mark.parametrize("B,T,E,k,m", [
    (1, 300, 512, 64, 4),
    (2, 5, 50000, 512, 1),        # beyond the shared-memory key cache
    (3, 4, 40000, 1024, 1),
    (1, 1, 262144, 1024, 4),
    (1, 2, 300000, 1024, 1),      # longer than the cluster kernel takes: two launches
])
def test_topk_exact(csa, orc, B, T, E, k, m):
    r = _np_rng(300 + E)
    sc = (np.round(r.standard_normal((B, T, E)) * 8) / 8).astype(np.float32)   # many ties
    sc[..., ::7] = 0.0
    sc[..., 3::7] = -0.0
    sc[..., 5::11] = np.float32(r.standard_normal()) * 1e-30
    if T > 3:
        pos = np.tile(np.linspace(0, (E - 1) * m + m - 1, T).astype(np.int64), (B, 1))
        pos[:, 0] = max(0, k * m - 1 - m)      # k-1 visible
        pos[:, 1] = k * m - 1                  # exactly k
        pos[:, 2] = k * m + m - 1              # k+1
        pos[:, 3] = 1 if m > 2 else 0          # nothing (m > 2) or 1 entry
    else:
        pos = np.full((B, T), E * m - 1, np.int64)
    idx, cnt = csa.topk_select(dev(sc), dev(pos), m, k)
    gi, gc = host(idx), host(cnt)
    for b in range(B):
        oi, oc = orc.topk(sc[b].astype(np.float64), pos[b], m, k)
        np.testing.assert_array_equal(gc[b], oc)
        np.testing.assert_array_equal(gi[b], oi)


def _topk_check(csa, orc, sc, pos, m, k):
    idx, cnt = csa.topk_select(dev(sc), dev(pos), m, k)
    gi, gc = host(idx), host(cnt)
    for b in range(sc.shape[0]):
        oi, oc = orc.topk(sc[b].astype(np.float64), pos[b], m, k)
        np.testing.assert_array_equal(gc[b], oc)
        np.testing.assert_array_equal(gi[b], oi)


@pytest.mark.parametrize("ties", [False, True])
def test_topk_prefill_rows(csa, orc, ties):
    """Many rows of up to 16384 visible entries (one CTA per row, keys in
    registers, sampled candidate bound); with heavy ties the candidates
    overflow and the exact whole-row selection runs."""
    r = _np_rng(311 + ties)
    T, E, k, m = 40, 16384, 512, 4
    sc = r.standard_normal((1, T, E)).astype(np.float32)
    if ties:
        sc = (np.round(sc * 2) / 2).astype(np.float32)
    pos = np.linspace(2 * k * m, E * m - 1, T).astype(np.int64).reshape(1, T)
    _topk_check(csa, orc, sc, pos, m, k)


def test_topk_sample_miss_prefill(csa, orc):
    """The largest keys sit exactly at the sampled positions, so the sampled
    bound admits fewer than k keys and the exact whole-row selection runs."""
    r = _np_rng(313)
    T, E, k, m = 4, 16384, 512, 4
    sc = r.standard_normal((1, T, E)).astype(np.float32)
    hot = (np.arange(E) % 8) == 0              # the 2048 evenly spaced sample positions
    sc[..., hot] = 100.0 + r.standard_normal((T, int(hot.sum()))).astype(np.float32)
    pos = np.full((1, T), E * m - 1, np.int64)
    _topk_check(csa, orc, sc, pos, m, k)


def test_topk_sample_miss_decode(csa, orc):
    """Decode rows whose largest keys sit exactly at the evenly spaced sample
    positions: the long-row path falls back to the exact selection."""
    r = _np_rng(317)
    B, E, k, m = 2, 262144, 1024, 4
    sc = r.standard_normal((B, 1, E)).astype(np.float32)
    sc[..., ::64] = 100.0 + r.standard_normal((B, 1, E // 64)).astype(np.float32)
    pos = np.full((B, 1), E * m - 1, np.int64)
    _topk_check(csa, orc, sc, pos, m, k)


def test_topk_decode_all_ties(csa, orc):
    """Decode rows whose visible keys are all equal: every CTA's candidates
    overflow and the exact selection over the whole row runs (ties go to the
    lowest indices)."""
    B, E, k, m = 2, 262144, 1024, 4
    sc = np.full((B, 1, E), 0.5, np.float32)
    pos = np.array([[E * m - 1], [E * m // 2 + 5]], np.int64)
    _topk_check(csa, orc, sc, pos, m, k)


# --------------------------------------------------------------- attention

def _nan_ws(csa, nbytes=1 << 26):
    """A workspace whose scratch bytes all hold NaN, so that a read of a split-KV
    partial that was never written shows in the output instead of passing on
    whatever an earlier call left there."""
    ws = csa.Workspace(nbytes)
    ws.buf[256:].fill_(0xFF)
    return ws


@pytest.mark.parametrize("dtype,B,T,H,c,E,k,m,n_win,r,derot", [
    ("f32", 1, 200, 4, 64, 60, 16, 4, 128, 32, 1),
    ("bf16", 2, 3, 64, 512, 3000, 512, 4, 128, 64, 1),
    ("bf16", 1, 17, 16, 128, 100, 8, 4, 5, 64, 0),
    ("bf16", 1, 300, 96, 512, 200, 64, 4, 128, 64, 1),    # two head groups, one partial
    ("bf16", 1, 40, 64, 512, 400, 128, 4, 128, 32, 1),    # 16 rotary pairs
    ("bf16", 1, 40, 64, 512, 400, 128, 4, 128, 192, 1),   # rotary dims across two chunks
    ("bf16", 1, 20, 64, 512, 100, 64, 4, 16, 0, 1),       # no rotary dims
])
def test_sparse_attn(csa, orc, dtype, B, T, H, c, E, k, m, n_win, r, derot):
    seed = 400 + E
    q = synth.normal(seed, 1, (B, T, H, c), 1.0, dtype)
    kvc = synth.normal(seed, 2, (B, E, c), 1.0, dtype)
    t_last = E * m + 7
    L = t_last + 1                                  # raw rows 0 .. t_last
    kv_raw = synth.normal(seed, 3, (B, L, c), 1.0, dtype)
    sink = synth.normal(seed, 4, (H,), 1.0, "f32")
    pos = np.tile(t_last - T + 1 + np.arange(T, dtype=np.int64), (B, 1))
    pos[:, 0] = 2                                   # an early query: few entries, short window
    raw_pos0 = np.zeros(B, np.int64)
    r_ = _np_rng(seed)
    idx = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        for t in range(T):
            nv = min(E, (pos[b, t] + 1) // m)
            kk = min(k, nv)
            sel = np.sort(r_.choice(nv, kk, replace=False)) if kk else np.zeros(0, int)
            idx[b, t, :kk] = sel
    p = csa.params(m=m, top_k=k, n_win=n_win, rope_dims=r, derotate=derot)
    lse = torch.empty((B, T, H), dtype=torch.float32, device="cuda")
    out = csa.sparse_attn(dev(q), dev(pos), dev(kvc), dev(idx), dev(kv_raw), dev(raw_pos0),
                          dev(sink), p, lse=lse, ws=_nan_ws(csa))
    g, gl = host(out), host(lse)
    for b in range(B):
        ro, rl = orc.attend(q[b], pos[b], kvc[b], m, kv_raw[b], int(raw_pos0[b]), sink, idx=idx[b],
                            n_win=n_win, rope_dims=r, derotate=derot, want_lse=True)
        check_close(g[b], ro, dtype, "sparse_attn out")
        # log-denominator: fp32 path to 1e-4; the bf16 path rounds the rotated
        # query to bf16 before the product, so its logits carry ~2^-9 relative error
        assert np.abs(gl[b] - rl).max() <= (1e-4 if dtype == "f32" else 1e-2)


# t0 > 0: the last query sits at position t0 (past 2^24, where the kernels'
# rotary angles take their double-precision reduction), with every entry visible
@pytest.mark.parametrize("dtype,B,T,H,c,E,m,n_win,r,t0", [
    ("bf16", 1, 70, 16, 128, 64, 128, 128, 64, 0),
    ("bf16", 2, 1, 128, 512, 700, 128, 128, 64, 0),
    ("f32", 1, 40, 4, 64, 30, 4, 16, 32, 0),
    ("bf16", 1, 3, 64, 512, 200, 128, 128, 64, (1 << 25) + 77),
    ("f32", 1, 5, 4, 64, 30, 4, 16, 32, (1 << 26) + 3),
    # c = 128 with 32, 64 and 128 heads: 4, 2 and 1 queries on an item's 128 rows
    # (37 queries leave a short last item)
    ("bf16", 2, 37, 32, 128, 40, 128, 128, 64, 0),
    ("bf16", 1, 9, 64, 128, 30, 4, 16, 32, 0),
    ("bf16", 1, 3, 128, 128, 20, 128, 128, 64, 0),
    # c = 512 with 64 heads: two sequences, consecutive queries straddling a
    # block boundary (visible counts E - 1 and E), a window shorter than a tile
    ("bf16", 2, 37, 64, 512, 300, 128, 128, 64, 300 * 128 + 5),
    ("bf16", 1, 8, 64, 512, 40, 4, 16, 32, 0),
])
def test_hca_attn(csa, orc, dtype, B, T, H, c, E, m, n_win, r, t0):
    seed = 500 + E
    q = synth.normal(seed, 1, (B, T, H, c), 1.0, dtype)
    kvc = synth.normal(seed, 2, (B, E, c), 1.0, dtype)
    t_last = t0 if t0 else E * m + m // 2
    L = n_win + T
    kv_raw = synth.normal(seed, 3, (B, L, c), 1.0, dtype)
    sink = synth.normal(seed, 4, (H,), 1.0, "f32")
    pos = np.tile(t_last - T + 1 + np.arange(T, dtype=np.int64), (B, 1))
    raw_pos0 = np.full(B, t_last - L + 1, np.int64)
    p = csa.params(m=m, n_win=n_win, rope_dims=r)
    out = csa.hca_attn(dev(q), dev(pos), dev(kvc), dev(kv_raw), dev(raw_pos0), dev(sink), p,
                       ws=_nan_ws(csa))
    g = host(out)
    for b in range(B):
        ro = orc.attend(q[b], pos[b], kvc[b], m, kv_raw[b], int(raw_pos0[b]), sink, idx=None,
                        n_win=n_win, rope_dims=r)
        check_close(g[b], ro, dtype, "hca_attn out")


def test_hca_attn_c128_no_derotate(csa, orc):
    """Dense attention at c = 128, 16 heads (eight queries per item), output
    left rotated, with the log-denominators."""
    dtype, B, T, H, c, E, m, n_win, r = "bf16", 1, 45, 16, 128, 50, 128, 128, 64
    seed = 650
    q = synth.normal(seed, 1, (B, T, H, c), 1.0, dtype)
    kvc = synth.normal(seed, 2, (B, E, c), 1.0, dtype)
    t_last = E * m + 3
    L = n_win + T
    kv_raw = synth.normal(seed, 3, (B, L, c), 1.0, dtype)
    sink = synth.normal(seed, 4, (H,), 1.0, "f32")
    pos = np.tile(t_last - T + 1 + np.arange(T, dtype=np.int64), (B, 1))
    raw_pos0 = np.full(B, t_last - L + 1, np.int64)
    p = csa.params(m=m, n_win=n_win, rope_dims=r, derotate=0)
    lse = torch.empty((B, T, H), dtype=torch.float32, device="cuda")
    out = csa.hca_attn(dev(q), dev(pos), dev(kvc), dev(kv_raw), dev(raw_pos0), dev(sink), p, lse=lse,
                       ws=_nan_ws(csa))
    ro, rl = orc.attend(q[0], pos[0], kvc[0], m, kv_raw[0], int(raw_pos0[0]), sink, idx=None, n_win=n_win,
                        rope_dims=r, derotate=0, want_lse=True)
    check_close(host(out)[0], ro, dtype, "hca_attn c128 no derotate")
    # log-denominator: the bf16 rounding of the rotated query leaves ~2^-9 relative
    # error in the logits
    assert np.abs(host(lse)[0] - rl).max() <= 1e-2


def test_hca_attn_c512_lse(csa, orc):
    """Dense attention at c = 512, 64 heads, output left rotated, with the
    log-denominators."""
    dtype, B, T, H, c, E, m, n_win, r = "bf16", 1, 6, 64, 512, 150, 128, 128, 64
    seed = 660
    q = synth.normal(seed, 1, (B, T, H, c), 1.0, dtype)
    kvc = synth.normal(seed, 2, (B, E, c), 1.0, dtype)
    t_last = E * m + 2
    L = n_win + T
    kv_raw = synth.normal(seed, 3, (B, L, c), 1.0, dtype)
    sink = synth.normal(seed, 4, (H,), 1.0, "f32")
    pos = np.tile(t_last - T + 1 + np.arange(T, dtype=np.int64), (B, 1))
    raw_pos0 = np.full(B, t_last - L + 1, np.int64)
    p = csa.params(m=m, n_win=n_win, rope_dims=r, derotate=0)
    lse = torch.empty((B, T, H), dtype=torch.float32, device="cuda")
    out = csa.hca_attn(dev(q), dev(pos), dev(kvc), dev(kv_raw), dev(raw_pos0), dev(sink), p, lse=lse,
                       ws=_nan_ws(csa))
    ro, rl = orc.attend(q[0], pos[0], kvc[0], m, kv_raw[0], int(raw_pos0[0]), sink, idx=None, n_win=n_win,
                        rope_dims=r, derotate=0, want_lse=True)
    check_close(host(out)[0], ro, dtype, "hca_attn c512 no derotate")
    assert np.abs(host(lse)[0] - rl).max() <= 1e-2


@pytest.mark.parametrize("B", [20, 80])
def test_hca_attn_decode_chunk_cap(csa, orc, B):
    """Split-KV decode whose chunk count is capped by the CTAs of one round:
    128 heads of B one-query sequences are 2 B items before the split, so at
    B = 20 the length rule's 4 chunks come down to 3, and at B = 80 (160
    units, more than the SMs) the list is not split at all.  NaN-filled
    scratch shows any partial the combine reads without an item writing it."""
    dtype, T, H, c, E, m, n_win, r = "bf16", 1, 128, 512, 700, 128, 128, 64
    seed = 670 + B
    q = synth.normal(seed, 1, (B, T, H, c), 1.0, dtype)
    kvc = synth.normal(seed, 2, (B, E, c), 1.0, dtype)
    t_last = E * m + 5
    L = n_win + T
    kv_raw = synth.normal(seed, 3, (B, L, c), 1.0, dtype)
    sink = synth.normal(seed, 4, (H,), 1.0, "f32")
    pos = np.full((B, T), t_last, np.int64)
    raw_pos0 = np.full(B, t_last - L + 1, np.int64)
    p = csa.params(m=m, n_win=n_win, rope_dims=r)
    out = csa.hca_attn(dev(q), dev(pos), dev(kvc), dev(kv_raw), dev(raw_pos0), dev(sink), p,
                       ws=_nan_ws(csa, 1 << 28))
    g = host(out)
    for b in (0, B // 2, B - 1):
        ro = orc.attend(q[b], pos[b], kvc[b], m, kv_raw[b], int(raw_pos0[b]), sink, idx=None,
                        n_win=n_win, rope_dims=r)
        check_close(g[b], ro, dtype, f"hca_attn decode chunk cap b={b}")


# ---------------------------------------------------------------- fused

def _prefill_csa_gpu(csa, s, x, idx_out=True):
    d = {k: dev(v) for k, v in x.items()}
    p = csa.params(m=s["m"], overlap=s.get("overlap", 0), top_k=s["top_k"], n_win=s["n_win"],
                   rope_dims=s["rope_dims"], rope_theta=s["theta"])
    io = torch.empty((s["B"], s["n"], s["top_k"]), dtype=torch.int32, device="cuda") if idx_out else None
    out = csa.csa_prefill(d["C"], d["Z"], d["bias"], d["Ck"], d["Zk"], d["biask"], d["q"], d["qI"],
                          d["w"], d["sink"], p, Cb=d.get("Cb"), Zb=d.get("Zb"), biasb=d.get("biasb"),
                          Ckb=d.get("Ckb"), Zkb=d.get("Zkb"), biaskb=d.get("biaskb"), idx_out=io)
    return out, io


def _check_csa_prefill(orc, s, x, out, io, q_sel=None):
    dt = s["dtype"]
    st = orc.csa_prefill_seq(s, x, 0, q_sel=q_sel, return_steps=True)
    qp = np.arange(s["n"]) if q_sel is None else np.asarray(q_sel)
    g_out = host(out[0])[qp]
    g_idx = host(io[0])[qp]
    differ = compare_topk(g_idx, st["idx"], st["scores"], qp, s["m"], s["top_k"])
    ref = st["out"].copy()
    if differ.size:       # below-gap rows: compare against the oracle on the GPU's set
        kvc_s = orc._storage(st["kvc"], dt)
        raw_s = orc._storage(st["raw"], dt)
        ref[differ] = orc.attend(x["q"][0][qp[differ]], qp[differ], kvc_s, s["m"], raw_s, 0,
                                 x["sink"], idx=g_idx[differ], n_win=s["n_win"],
                                 rope_dims=s["rope_dims"], theta=s["theta"])
    check_close(g_out, ref, dt, "csa_prefill out")
    return differ.size


def test_csa_prefill_cfg1_full(csa, orc):
    """CSA single-layer prefill in fp32, n = 2048 (the whole workload)."""
    s, x = synth.make_inputs("csa_prefill_f32")
    out, io = _prefill_csa_gpu(csa, s, x)
    _check_csa_prefill(orc, s, x, out, io)


def test_csa_prefill_cfg1_overlap(csa, orc):
    s, x = synth.make_inputs("csa_prefill_f32", n=1030, overlap=1)
    out, io = _prefill_csa_gpu(csa, s, x)
    _check_csa_prefill(orc, s, x, out, io)


def test_csa_prefill_bf16_sampled(csa, orc):
    """Flash-shaped CSA layer (H=64, c=512, hI=64, dI=128, k=512) at n=4100,
    where the top-k binds for t >= 2048; oracle on sampled rows."""
    s, x = synth.make_inputs("hybrid_prefill_flash", n=4100)
    out, io = _prefill_csa_gpu(csa, s, x)
    q_sel = np.unique(np.r_[0, 1, 2, 3, 4, 127, 128, 2043, 2047, 2048, 2051, 2052, 3000,
                            _np_rng(5).integers(0, 4100, 24), 4095, 4099])
    _check_csa_prefill(orc, s, x, out, io, q_sel)


def test_hca_prefill_cfg2_full(csa, orc):
    """HCA single-layer prefill in bf16, n = 8192 (the whole workload)."""
    s, x = synth.make_inputs("hca_prefill_bf16")
    d = {k: dev(v) for k, v in x.items()}
    p = csa.params(m=s["m"], n_win=s["n_win"], rope_dims=s["rope_dims"], rope_theta=s["theta"])
    out = csa.hca_prefill(d["C"], d["Z"], d["bias"], d["q"], d["sink"], p)
    ref = orc.hca_prefill_seq(s, x, 0)
    check_close(host(out[0]), ref, "bf16", "hca_prefill out")


def _decode_gpu(csa, s, x, hca, batch_invariant=0):
    d = {k: dev(v) for k, v in x.items()}
    p = csa.params(m=s["m"], top_k=s["top_k"], n_win=s["n_win"], rope_dims=s["rope_dims"],
                   rope_theta=s["theta"], batch_invariant=batch_invariant)
    p2 = csa.params(m=s.get("m2", 128), n_win=s["n_win"], rope_dims=s["rope_dims"],
                    rope_theta=s["theta"], batch_invariant=batch_invariant)
    io = torch.empty((s["B"], 1, s["top_k"]), dtype=torch.int32, device="cuda")
    kw = dict(q2=d["q2"], kvc2=d["kvc2"], kv_raw2=d["kv_raw2"], sink2=d["sink2"], p2=p2) if hca else {}
    res = csa.hybrid_decode(d["q"], d["qI"], d["w"], d["kvc"], d["kIc"], d["kv_raw"], d["sink"],
                            d["q_pos"], d["raw_pos0"], p, idx_out=io, **kw)
    return res, io


def _check_decode(orc, s, x, res, io, seqs, hca):
    out, out2 = (res if hca else (res, None))
    for b in seqs:
        st = orc.csa_decode_seq(s, x, b, return_steps=True)
        gi = host(io[b])
        differ = compare_topk(gi, st["idx"], st["scores"], x["q_pos"][b], s["m"], s["top_k"])
        ref = st["out"]
        if differ.size:
            ref = orc.attend(x["q"][b], x["q_pos"][b], x["kvc"][b], s["m"], x["kv_raw"][b],
                             int(x["raw_pos0"][b]), x["sink"], idx=gi, n_win=s["n_win"],
                             rope_dims=s["rope_dims"], theta=s["theta"])
        check_close(host(out[b]), ref, s["dtype"], f"decode out seq {b}")
        if hca:
            check_close(host(out2[b]), orc.hca_decode_seq(s, x, b), s["dtype"], f"hca out seq {b}")


def test_decode_cfg3_flash(csa, orc):
    """Flash-shaped CSA decode: B=32, 32768 entries each; oracle on 4 sequences."""
    s, x = synth.make_inputs("csa_decode_flash")
    res, io = _decode_gpu(csa, s, x, False)
    _check_decode(orc, s, x, res, io, [0, 7, 19, 31], False)


def test_decode_cfg5_pro(csa, orc):
    """Pro-shaped hybrid decode at 1,048,576 positions: B=8; oracle on 2 sequences."""
    s, x = synth.make_inputs("hybrid_decode_pro")
    res, io = _decode_gpu(csa, s, x, True)
    _check_decode(orc, s, x, res, io, [0, 5], True)


def _cfg4_rows(n):
    """Query rows checked at full size: the first and last query blocks of
    the indexer (4 queries each), every row around the top-k transition
    (|V| = k at t = 2047 .. 2050, k + 1 from t = 2051), and a stratified
    sample of 14 rows from each of the 16 bands of 4096 queries, so every
    region of the indexer's block schedule and of the attention work list is
    reached."""
    r = _np_rng(44)
    rows = [np.arange(0, 8), np.arange(n - 8, n), np.arange(2040, 2060)]
    for band in range(16):
        lo = band * (n // 16)
        rows.append(lo + r.choice(n // 16, 14, replace=False))
    rows.append(np.array([4095, 4096, 16383, 16384, 32767, 32768, 49151, 49152]))
    return np.unique(np.concatenate(rows))


def test_prefill_cfg4_flash_sampled(csa, orc):
    """Flash-shaped interleaved CSA + HCA prefill at the full n = 65536, in the
    launch configuration the bench times; oracle on sampled query rows."""
    s, x = synth.make_inputs("hybrid_prefill_flash")
    out, io = _prefill_csa_gpu(csa, s, x)
    q_sel = _cfg4_rows(s["n"])
    assert q_sel.size >= 256
    _check_csa_prefill(orc, s, x, out, io, q_sel)
    d = {k: dev(v) for k, v in x.items() if k.endswith("2")}
    p2 = csa.params(m=s["m2"], n_win=s["n_win"], rope_dims=s["rope_dims"], rope_theta=s["theta"])
    out2 = csa.hca_prefill(d["C2"], d["Z2"], d["bias2"], d["q2"], d["sink2"], p2)
    ref2 = orc.hca_prefill_seq(s, x, 0, q_sel=q_sel, suffix="2")
    check_close(host(out2[0])[q_sel], ref2, "bf16", "hca layer out")


# ------------------------------------------------- status word, determinism

def test_status_word_reports_missing_window(csa):
    B, T, H, c, E, m = 1, 1, 4, 64, 8, 4
    q = torch.randn(B, T, H, c, device="cuda")
    kvc = torch.randn(B, E, c, device="cuda")
    kv_raw = torch.randn(B, 4, c, device="cuda")
    pos = torch.tensor([[100]], device="cuda")
    rp0 = torch.tensor([90], device="cuda")          # rows hold 90..93: window 0..100 not covered
    sink = torch.zeros(H, device="cuda")
    ws = csa.Workspace(4096)
    p = csa.params(m=m, n_win=8, rope_dims=0)
    csa.hca_attn(q, pos, kvc, kv_raw, rp0, sink, p, ws=ws)
    with pytest.raises(csa.CsaError) as e:
        ws.status()
    assert e.value.status == 6
    ws.status()                                     # cleared
    idx = torch.tensor([[[0, 99, -1, -1]]], dtype=torch.int32, device="cuda")
    rp0 = torch.tensor([97], device="cuda")
    csa.sparse_attn(q, pos, kvc, idx, kv_raw, rp0, sink, csa.params(m=m, top_k=4, n_win=4, rope_dims=0), ws=ws)
    with pytest.raises(csa.CsaError):
        ws.status()


def test_prefill_deterministic(csa):
    s, x = synth.make_inputs("csa_prefill_f32", n=1024)
    a, ia = _prefill_csa_gpu(csa, s, x)
    b, ib = _prefill_csa_gpu(csa, s, x)
    assert torch.equal(a, b) and torch.equal(ia, ib)


def test_decode_batch_invariant_full_batch(csa, orc):
    """With batch_invariant set, a sequence decoded alone gives bitwise the same output as
    inside a batch that fills the GPU by itself (300 sequences of 640 entries, where the
    default would skip the split of each list into chunks)."""
    s, x = synth.make_inputs("csa_decode_flash", B=300, t=2047)
    res, io = _decode_gpu(csa, s, x, False, batch_invariant=1)
    _check_decode(orc, s, x, res, io, [0, 299], False)      # and the batch run is right
    for b in (0, 299):
        xb = {k: (v[b:b + 1] if k not in ("sink",) else v) for k, v in x.items()}
        rb, ib = _decode_gpu(csa, dict(s, B=1), xb, False, batch_invariant=1)
        assert torch.equal(rb[0], res[b]) and torch.equal(ib[0], io[b])


def test_decode_batch_invariant(csa):
    """A sequence decoded alone gives bitwise the same output as inside a batch."""
    s, x = synth.make_inputs("csa_decode_flash", B=6, t=8191)
    res, io = _decode_gpu(csa, s, x, False)
    for b in (0, 4):
        xb = {k: (v[b:b + 1] if k not in ("sink",) else v) for k, v in x.items()}
        sb = dict(s, B=1)
        rb, ib = _decode_gpu(csa, sb, xb, False)
        assert torch.equal(rb[0], res[b]) and torch.equal(ib[0], io[b])


def test_wait_probe_reports_timeout(csa):
    """A bounded wait that nothing completes gives up after spin_limit polls,
    sets the timeout bit, and the context stays usable for the next call."""
    ws = csa.Workspace(1 << 16)
    csa.wait_probe(2000, ws)
    with pytest.raises(csa.CsaError) as e:
        ws.status()
    assert e.value.status == 5
    ws.status()                                     # cleared
    s, x = synth.make_inputs("hybrid_decode_pro", B=1, t=1023)
    res, io = _decode_gpu(csa, s, x, True)
    torch.cuda.synchronize()
    assert torch.isfinite(res[0]).all() and torch.isfinite(res[1]).all()


def test_hybrid_decode_two_threads_two_streams(csa):
    """Two host threads, each on its own stream and workspace, issue 20
    Pro-shaped hybrid decode calls each (the HCA layer runs on an auxiliary
    stream inside every call); q2 is rewritten on the caller's stream right
    before each call.  Every output equals, bit for bit, the same call made
    serially afterwards."""
    import threading
    sets = []
    for j in range(4):
        s, x = synth.make_inputs("hybrid_decode_pro", B=2, t=4095 + 128 * j, seed=40 + j)
        sets.append((s, {k: dev(v) for k, v in x.items()}))
    s0 = sets[0][0]
    p = csa.params(m=4, top_k=s0["top_k"], n_win=128, rope_dims=64)
    p2 = csa.params(m=128, n_win=128, rope_dims=64)
    N = 20
    results = {}
    errors = []

    def one(d, q2buf, ws, out, out2):
        q2buf.copy_(d["q2"])
        csa.hybrid_decode(d["q"], d["qI"], d["w"], d["kvc"], d["kIc"], d["kv_raw"], d["sink"],
                          d["q_pos"], d["raw_pos0"], p, q2=q2buf, kvc2=d["kvc2"],
                          kv_raw2=d["kv_raw2"], sink2=d["sink2"], p2=p2, out=out, out2=out2, ws=ws)

    def worker(j):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                ws = csa.Workspace(1 << 26)
                q2buf = torch.empty_like(sets[0][1]["q2"])
                for i in range(N):
                    d = sets[(i + j) % 4][1]
                    out, out2 = torch.empty_like(d["q"]), torch.empty_like(d["q2"])
                    one(d, q2buf, ws, out, out2)
                    results[(j, i)] = (out, out2)
                st.synchronize()
        except Exception as e:  # surfaced below
            errors.append(e)

    th = [threading.Thread(target=worker, args=(j,)) for j in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    ws = csa.Workspace(1 << 26)
    q2buf = torch.empty_like(sets[0][1]["q2"])
    for (j, i), (out, out2) in sorted(results.items()):
        d = sets[(i + j) % 4][1]
        o, o2 = torch.empty_like(d["q"]), torch.empty_like(d["q2"])
        one(d, q2buf, ws, o, o2)
        torch.cuda.synchronize()
        assert torch.equal(o, out) and torch.equal(o2, out2), (j, i)
