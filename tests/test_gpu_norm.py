"""GPU parity of the q / KV RMSNorm (csa_params q_norm, kv_norm) against the
oracle's definition (oracle/outproj.rmsnorm) composed with the oracle's
steps in the order the pages give: a compressed entry is pooled, normalised,
rotated at its block's last position and rounded once; a stored raw row is
normalised, rotated at its position and rounded; each query head is
normalised and then rotated at t.  Covers the tensor-core attention (bf16,
c = 512 and 128), the fp32 CUDA-core path, the fused prefill entry points and
the incremental decode state (bitwise against the prefill compression)."""
import numpy as np
import pytest
import torch

import synth
from oracle import outproj
from parity import check_close, compare_topk, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_sparse_22_b300 as m
    m.lib()
    return m


def _gains(seed, c):
    g = 1.0 + 0.1 * synth.normal(seed, 90, (c,), 1.0, "f32").astype(np.float64)
    return g.astype(np.float32)


def _orc_stored(orc, Cx, Zx, bias, m, r, theta, dt, g, eps=1e-6):
    """Normalised, rotated, rounded entries and raw rows of one sequence."""
    pooled = orc.compress(Cx, Zx, bias, m, rope_dims=0, out_dtype="f64")
    normed = outproj.rmsnorm(pooled, g, eps)
    ent = np.stack([orc.rope(normed[j], (j + 1) * m - 1, r, theta) for j in range(normed.shape[0])]) \
        if normed.shape[0] else normed
    rawn = outproj.rmsnorm(synth.widen(Cx, dt), g, eps)
    raw = np.stack([orc.rope(rawn[p], p, r, theta) for p in range(rawn.shape[0])])
    return orc.round_to(ent, dt), orc.round_to(raw, dt)


def _storage(orc, a, dt):
    return orc._storage(a, dt)


@pytest.mark.parametrize("name,n", [("hybrid_prefill_flash", 1030), ("csa_prefill_f32", 700)])
def test_csa_prefill_with_norms(csa, orc, name, n):
    s, x = synth.make_inputs(name, n=n)
    dt, c, m, r, th = s["dtype"], s["c"], s["m"], s["rope_dims"], s["theta"]
    gq, gk = _gains(5, c), _gains(6, c)
    d = {k: dev(v) for k, v in x.items()}
    gq_d, gk_d = dev(gq), dev(gk)
    p = csa.params(m=m, top_k=s["top_k"], n_win=s["n_win"], rope_dims=r, rope_theta=th, q_norm=gq_d,
                   kv_norm=gk_d)
    io = torch.empty((1, n, s["top_k"]), dtype=torch.int32, device="cuda")
    out = csa.csa_prefill(d["C"], d["Z"], d["bias"], d["Ck"], d["Zk"], d["biask"], d["q"], d["qI"],
                          d["w"], d["sink"], p, idx_out=io)
    # oracle: keys as in the plain path (no norm); KV and q normalised
    ent, raw = _orc_stored(orc, x["C"][0], x["Z"][0], x["bias"], m, r, th, dt, gk)
    kIc = orc.compress(x["Ck"][0], x["Zk"][0], x["biask"], m, rope_dims=0, out_dtype=dt)
    q_sel = np.unique(np.r_[0, 3, 4, 127, 128, 255, 256, 257, n // 2, n - 2, n - 1])
    sc = orc.index_scores(x["qI"][0][q_sel], x["w"][0][q_sel], q_sel, _storage(orc, kIc, dt), m)
    oi, _ = orc.topk(sc, q_sel, m, s["top_k"])
    gi = host(io[0])[q_sel]
    compare_topk(gi, oi, sc, q_sel, m, s["top_k"])
    qn = outproj.rmsnorm(synth.widen(x["q"][0][q_sel], dt), gq)
    ref = orc.attend(qn, q_sel, _storage(orc, ent, dt), m, _storage(orc, raw, dt), 0, x["sink"], idx=gi,
                     n_win=s["n_win"], rope_dims=r, theta=th)
    check_close(host(out[0])[q_sel], ref, dt, "csa_prefill with norms")


@pytest.mark.parametrize("H,c", [(16, 128), (64, 512)])
def test_hca_prefill_with_norms(csa, orc, H, c):
    s, x = synth.make_inputs("hca_prefill_bf16", n=1000, H=H, c=c)
    dt, m, r, th = s["dtype"], s["m"], s["rope_dims"], s["theta"]
    gq, gk = _gains(7, c), _gains(8, c)
    d = {k: dev(v) for k, v in x.items()}
    gq_d, gk_d = dev(gq), dev(gk)
    p = csa.params(m=m, n_win=s["n_win"], rope_dims=r, rope_theta=th, q_norm=gq_d, kv_norm=gk_d)
    out = csa.hca_prefill(d["C"], d["Z"], d["bias"], d["q"], d["sink"], p)
    ent, raw = _orc_stored(orc, x["C"][0], x["Z"][0], x["bias"], m, r, th, dt, gk)
    q_sel = np.unique(np.r_[0, 1, 126, 127, 128, 300, 511, 512, 999])
    qn = outproj.rmsnorm(synth.widen(x["q"][0][q_sel], dt), gq)
    ref = orc.attend(qn, q_sel, _storage(orc, ent, dt), m, _storage(orc, raw, dt), 0, x["sink"],
                     idx=None, n_win=s["n_win"], rope_dims=r, theta=th)
    check_close(host(out[0])[q_sel], ref, dt, "hca_prefill with norms")


def test_decode_append_with_norm_matches_prefill(csa):
    """The incremental state with the KV norm stores bitwise the entries and
    ring rows of the prefill compression with the same norm."""
    B, n, c, dI = 2, 260, 512, 128
    for m, overlap in ((4, 0), (4, 1), (128, 0)):
        C_ = torch.randn(B, n, c, device="cuda").to(torch.bfloat16)
        Z = torch.randn(B, n, c, device="cuda").to(torch.bfloat16)
        bias = torch.randn(m, c, device="cuda") * 0.1
        g = (1 + 0.1 * torch.randn(c, device="cuda")).float()
        kw = {}
        if overlap:
            kw = dict(Cb=torch.randn(B, n, c, device="cuda").to(torch.bfloat16),
                      Zb=torch.randn(B, n, c, device="cuda").to(torch.bfloat16),
                      biasb=torch.randn(m, c, device="cuda") * 0.1)
        p = csa.params(m=m, overlap=overlap, n_win=128, rope_dims=64, kv_norm=g)
        ent, raw = csa.csa_compress(C_, Z, bias, m=m, overlap=overlap, rope_dims=64, want_raw=True,
                                    kv_norm=g, **kw)
        win = torch.zeros((B, 128, c), dtype=torch.bfloat16, device="cuda")
        tail = torch.empty(csa.decode_tail_bytes(1, B, c, 0, p), dtype=torch.uint8, device="cuda")
        kvc = torch.zeros((B, n // m + 1, c), dtype=torch.bfloat16, device="cuda")
        for t in range(n):
            tt = torch.full((B,), t, dtype=torch.int64, device="cuda")
            ekw = {}
            if overlap:
                ekw = dict(Cb=kw["Cb"][:, t].contiguous(), Zb=kw["Zb"][:, t].contiguous(),
                           biasb=kw["biasb"])
            csa.decode_append(tt, C_[:, t].contiguous(), Z[:, t].contiguous(), bias, win, tail, kvc, p,
                              **ekw)
        torch.cuda.synchronize()
        assert torch.equal(kvc[:, :n // m], ent), (m, overlap)
        slots = [q % 128 for q in range(n - 128, n)]
        assert torch.equal(win[:, slots], raw[:, n - 128:]), (m, overlap)
