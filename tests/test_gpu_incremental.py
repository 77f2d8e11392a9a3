"""GPU parity of the incremental decode state (decode_append + hybrid_decode)
against the oracle's token-by-token state (oracle/incremental.py):

* a hybrid stream (CSA layer with m = 4, one branch; HCA layer with m' = 128)
  of 700 tokens, and a two-branch CSA stream of 333 tokens, one token per
  step for two sequences at once;
* every step's selection and output against the oracle's query at that
  position (the gap rule and tolerances of tests/parity.py);
* at the end, the caches and the window ring bitwise against the prefill
  path's own compression of the whole sequence (csa_compress), and within
  one bf16 step of the oracle's entries.
"""
import numpy as np
import pytest
import torch

import synth
from parity import check_close, compare_topk, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_sparse_22_b300 as m
    m.lib()
    return m


SPEC = dict(dtype="bf16", c=128, H=16, hI=64, dI=128, top_k=32, n_win=128, rope_dims=64,
            theta=10000.0, derotate=1)


def _inputs(seed, B, n, overlap, hca):
    c, dI, H, hI = SPEC["c"], SPEC["dI"], SPEC["H"], SPEC["hI"]
    x = {}
    for i, name in enumerate(["C", "Z", "Cb", "Zb", "C2", "Z2"]):
        if name in ("Cb", "Zb") and not overlap or name in ("C2", "Z2") and not hca:
            continue
        x[name] = synth.normal(seed, 1 + i, (B, n, c), 1.0, "bf16")
    for i, name in enumerate(["Ck", "Zk", "Ckb", "Zkb"]):
        if name in ("Ckb", "Zkb") and not overlap:
            continue
        x[name] = synth.normal(seed, 10 + i, (B, n, dI), 1.0, "bf16")
    x["bias"] = synth.normal(seed, 20, (4, c), 0.1, "f32")
    x["biask"] = synth.normal(seed, 21, (4, dI), 0.1, "f32")
    if overlap:
        x["biasb"] = synth.normal(seed, 22, (4, c), 0.1, "f32")
        x["biaskb"] = synth.normal(seed, 23, (4, dI), 0.1, "f32")
    if hca:
        x["bias2"] = synth.normal(seed, 24, (128, c), 0.1, "f32")
        x["q2"] = synth.normal(seed, 25, (B, n, H, c), 1.0, "bf16")
        x["sink2"] = synth.normal(seed, 26, (H,), 1.0, "f32")
    x["q"] = synth.normal(seed, 30, (B, n, H, c), 1.0, "bf16")
    x["qI"] = synth.normal(seed, 31, (B, n, hI, dI), 1.0, "bf16")
    x["w"] = synth.softmax_normal(seed, 32, (B, n, hI))
    x["sink"] = synth.normal(seed, 33, (H,), 1.0, "f32")
    return x


def _steps_major(a):
    """[B, n, ...] -> device [n, B, ...] so that step t's slice is contiguous."""
    return dev(np.ascontiguousarray(np.swapaxes(a, 0, 1)))


def _stream(csa, x, B, n, overlap, hca):
    """Run n decode steps on the GPU; return the per-step outputs, selections
    and the final state."""
    c, dI, H, k, W = SPEC["c"], SPEC["dI"], SPEC["H"], SPEC["top_k"], SPEC["n_win"]
    E_cap, E2_cap = n // 4 + 1, n // 128 + 1
    p = csa.params(m=4, overlap=overlap, top_k=k, n_win=W, rope_dims=SPEC["rope_dims"])
    p2 = csa.params(m=128, n_win=W, rope_dims=SPEC["rope_dims"])
    d = {key: _steps_major(v) for key, v in x.items() if v.ndim >= 2 and v.shape[1] == n}
    bias = {key: dev(x[key]) for key in ("bias", "biask", "biasb", "biaskb", "bias2") if key in x}
    sink, sink2 = dev(x["sink"]), dev(x["sink2"]) if hca else None
    bf = torch.bfloat16
    win = torch.zeros((B, W, c), dtype=bf, device="cuda")
    tail = torch.empty(csa.decode_tail_bytes(1, B, c, dI, p), dtype=torch.uint8, device="cuda")
    kvc = torch.zeros((B, E_cap, c), dtype=bf, device="cuda")
    kIc = torch.zeros((B, E_cap, dI), dtype=bf, device="cuda")
    if hca:
        win2 = torch.zeros((B, W, c), dtype=bf, device="cuda")
        tail2 = torch.empty(csa.decode_tail_bytes(1, B, c, 0, p2), dtype=torch.uint8, device="cuda")
        kvc2 = torch.zeros((B, E2_cap, c), dtype=bf, device="cuda")
    pos = torch.arange(n, device="cuda", dtype=torch.int64).view(n, 1).repeat(1, B).contiguous()
    rp0 = (pos - (W - 1)).clamp(min=0).contiguous()
    out = torch.empty((n, B, 1, H, c), dtype=bf, device="cuda")
    out2 = torch.empty_like(out) if hca else None
    idx = torch.empty((n, B, 1, k), dtype=torch.int32, device="cuda")
    ws = csa.Workspace(1 << 24)
    ws_a = csa.Workspace(4096)
    for t in range(n):
        kw = {}
        if overlap:
            kw = dict(Cb=d["Cb"][t], Zb=d["Zb"][t], biasb=bias["biasb"], Ckb=d["Ckb"][t],
                      Zkb=d["Zkb"][t], biaskb=bias["biaskb"])
        csa.decode_append(pos[t], d["C"][t], d["Z"][t], bias["bias"], win, tail, kvc, p,
                          Ck=d["Ck"][t], Zk=d["Zk"][t], biask=bias["biask"], kIc=kIc, ws=ws_a, **kw)
        hk = {}
        if hca:
            csa.decode_append(pos[t], d["C2"][t], d["Z2"][t], bias["bias2"], win2, tail2, kvc2, p2,
                              ws=ws_a)
            hk = dict(q2=d["q2"][t].unsqueeze(1), kvc2=kvc2, kv_raw2=win2, sink2=sink2, p2=p2,
                      out2=out2[t])
        csa.hybrid_decode(d["q"][t].unsqueeze(1), d["qI"][t].unsqueeze(1), d["w"][t].unsqueeze(1),
                          kvc, kIc, win, sink, pos[t].view(B, 1), rp0[t], p, out=out[t],
                          idx_out=idx[t], ws=ws, **hk)
    ws_a.status()
    ws.status()
    state = dict(win=win, kvc=kvc, kIc=kIc)
    if hca:
        state.update(win2=win2, kvc2=kvc2)
    return out, out2, idx, state


def _oracle_check(orc, x, b, n, overlap, hca, out, out2, idx):
    from oracle.incremental import LayerState
    s = dict(SPEC)
    L1 = LayerState(s, m=4, csa=True, overlap=overlap)
    L2 = LayerState(s, m=128, csa=False) if hca else None
    bias1 = {key: x[key] for key in ("bias", "biask", "biasb", "biaskb") if key in x}
    g_out, g_idx = host(out[:, b, 0]), host(idx[:, b, 0])
    g_out2 = host(out2[:, b, 0]) if hca else None
    differ = 0
    for t in range(n):
        row = {key: x[key][b, t] for key in ("C", "Z", "Ck", "Zk", "Cb", "Zb", "Ckb", "Zkb") if key in x}
        L1.push(row, bias1)
        r1 = L1.query(x["q"][b, t], x["sink"], qI=x["qI"][b, t], w=x["w"][b, t])
        d = compare_topk(g_idx[t][None], r1["idx"][None], r1["scores"][None], np.array([t]), 4,
                         SPEC["top_k"])
        ref = r1["out"]
        if d.size:                   # below the gap: the oracle on the GPU's selection
            differ += 1
            raw = orc._storage(np.stack([rr for _, rr in L1.win]), "bf16")
            kv = orc._storage(np.stack(L1.entries), "bf16")
            ref = orc.attend(x["q"][b, t][None], np.array([t]), kv, 4, raw, L1.win[0][0], x["sink"],
                             idx=g_idx[t][None], n_win=SPEC["n_win"], rope_dims=SPEC["rope_dims"])[0]
        check_close(g_out[t], ref, "bf16", f"csa step {t}")
        if hca:
            L2.push({"C": x["C2"][b, t], "Z": x["Z2"][b, t]}, {"bias": x["bias2"]})
            r2 = L2.query(x["q2"][b, t], x["sink2"])
            check_close(g_out2[t], r2["out"], "bf16", f"hca step {t}")
    return L1, L2, differ


def _check_caches(csa, orc, x, B, n, overlap, hca, state, L1s, L2s):
    c, W = SPEC["c"], SPEC["n_win"]
    E = n // 4
    kw = {}
    if overlap:
        kw = dict(Cb=dev(x["Cb"]), Zb=dev(x["Zb"]), biasb=dev(x["biasb"]))
    ent, raw = csa.csa_compress(dev(x["C"]), dev(x["Z"]), dev(x["bias"]), m=4, overlap=overlap,
                                rope_dims=SPEC["rope_dims"], want_raw=True, **kw)
    kkw = dict(Cb=dev(x["Ckb"]), Zb=dev(x["Zkb"]), biasb=dev(x["biaskb"])) if overlap else {}
    keys = csa.csa_compress(dev(x["Ck"]), dev(x["Zk"]), dev(x["biask"]), m=4, overlap=overlap, **kkw)
    torch.cuda.synchronize()
    assert torch.equal(state["kvc"][:, :E], ent), "entries differ from the prefill compression"
    assert torch.equal(state["kIc"][:, :E], keys), "keys differ from the prefill compression"
    slots = [p % W for p in range(n - W, n)]
    assert torch.equal(state["win"][:, slots], raw[:, n - W:]), "window ring differs from the raw rows"
    for b in range(B):
        g = host(state["kvc"][b, :E])
        ref = np.stack(L1s[b].entries)
        assert np.all(np.abs(g - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-6), "entries vs oracle"
    if hca:
        E2 = n // 128
        ent2, raw2 = csa.csa_compress(dev(x["C2"]), dev(x["Z2"]), dev(x["bias2"]), m=128,
                                      rope_dims=SPEC["rope_dims"], want_raw=True)
        torch.cuda.synchronize()
        assert torch.equal(state["kvc2"][:, :E2], ent2), "HCA entries differ from the prefill compression"
        assert torch.equal(state["win2"][:, slots], raw2[:, n - W:])
        for b in range(B):
            ref = np.stack(L2s[b].entries)
            g = host(state["kvc2"][b, :E2])
            assert np.all(np.abs(g - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-6), "HCA entries vs oracle"


@pytest.mark.parametrize("overlap,hca,n", [(0, True, 700), (1, False, 333)])
def test_incremental_decode_stream(csa, orc, overlap, hca, n):
    B = 2
    x = _inputs(70 + overlap, B, n, overlap, hca)
    out, out2, idx, state = _stream(csa, x, B, n, overlap, hca)
    L1s, L2s = [], []
    for b in range(B):
        L1, L2, differ = _oracle_check(orc, x, b, n, overlap, hca, out, out2, idx)
        assert differ <= n // 20, f"{differ} steps below the top-k gap"
        assert L1.state_rows()["window"] == SPEC["n_win"] and L1.state_rows()["tail"] < 4
        L1s.append(L1)
        L2s.append(L2)
    _check_caches(csa, orc, x, B, n, overlap, hca, state, L1s, L2s)


def test_decode_append_full_cache_sets_status(csa):
    """A completed block past the cache's capacity is not stored; the range bit
    of the status word reports it."""
    B, c, dI = 1, 128, 128
    p = csa.params(m=4, n_win=128, rope_dims=64)
    C_ = torch.randn(B, c, device="cuda").to(torch.bfloat16)
    bias = torch.zeros(4, c, device="cuda")
    win = torch.zeros(B, 128, c, dtype=torch.bfloat16, device="cuda")
    tail = torch.empty(csa.decode_tail_bytes(1, B, c, 0, p), dtype=torch.uint8, device="cuda")
    kvc = torch.zeros(B, 1, c, dtype=torch.bfloat16, device="cuda")
    ws = csa.Workspace(4096)
    for t in range(8):                          # blocks 0 and 1 complete; capacity 1
        csa.decode_append(torch.tensor([t], device="cuda"), C_, C_, bias, win, tail, kvc, p, ws=ws)
    with pytest.raises(csa.CsaError) as e:
        ws.status()
    assert e.value.status == 6
