"""Pins for the incremental decode state of the oracle (oracle/incremental.py):
streaming a sequence token by token must leave exactly the caches the prefill
path builds, keep the per-request state bounded (the window and one block's
tail), and give every query the output and selection the prefill oracle gives
it ("DeepSeek-V4" book, ch.5 "What is retained during decode", ch.13
"Bounded state per request")."""
import numpy as np
import pytest

import synth
from oracle import incremental

CSA_KEYS = ("C", "Z", "Ck", "Zk", "Cb", "Zb", "Ckb", "Zkb")


def _stream(s, x, layer, keys, q, sink, qI=None, w=None, b=0):
    bias = {k: x[k] for k in ("bias", "biask", "biasb", "biaskb") if k in x}
    bias = {k.replace("2", ""): v for k, v in bias.items()}
    outs, idxs = [], []
    for t in range(s["n"]):
        layer.push({k.rstrip("2"): x[k][b][t] for k in keys}, bias)
        r = layer.query(q[b][t], sink, None if qI is None else qI[b][t], None if w is None else w[b][t])
        outs.append(r["out"])
        if "idx" in r:
            idxs.append(r["idx"])
        st = layer.state_rows()
        # bounded state: the window, this block's tail and (two-branch) one previous block
        assert st["window"] == min(t + 1, s["n_win"])
        assert st["tail"] == (t + 1) % layer.m
        assert st["prev"] <= layer.m and st["entries"] == (t + 1) // layer.m
    return np.stack(outs), (np.stack(idxs) if idxs else None)


@pytest.mark.parametrize("overlap", [0, 1])
def test_csa_stream_matches_prefill(orc, overlap):
    s, x = synth.make_inputs("csa_prefill_f32", n=333, overlap=overlap)
    full = orc.csa_prefill_seq(s, x, 0, return_steps=True)
    layer = incremental.LayerState(s, m=s["m"], csa=True, overlap=overlap)
    keys = [k for k in CSA_KEYS if k in x]
    out, idx = _stream(s, x, layer, keys, x["q"], x["sink"], x["qI"], x["w"])
    assert np.array_equal(np.stack(layer.entries), full["kvc"])
    assert np.array_equal(np.stack(layer.keys), full["kIc"])
    win = np.stack([r for _, r in layer.win])
    assert np.array_equal(win, full["raw"][s["n"] - s["n_win"]:])
    assert np.array_equal(idx, full["idx"])
    assert np.array_equal(out, full["out"])


def test_hca_stream_matches_prefill(orc):
    s, x = synth.make_inputs("hca_prefill_bf16", n=700)
    full = orc.hca_prefill_seq(s, x, 0, return_steps=True)
    layer = incremental.LayerState(s, m=s["m"], csa=False)
    out, _ = _stream(s, x, layer, ("C", "Z"), x["q"], x["sink"])
    assert np.array_equal(np.stack(layer.entries), full["kvc"])
    assert np.array_equal(out, full["out"])


def test_entry_moves_to_cache_when_block_completes(orc):
    """Before its block completes a token reaches later queries only through the
    window; the entry appears at the block's last position."""
    s, x = synth.make_inputs("csa_prefill_f32", n=12)
    layer = incremental.LayerState(s, m=s["m"], csa=True)
    keys = [k for k in CSA_KEYS if k in x]
    bias = {k: x[k] for k in ("bias", "biask")}
    seen = []
    for t in range(12):
        layer.push({k: x[k][0][t] for k in keys}, bias)
        seen.append(len(layer.entries))
    assert seen == [0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 2, 3]
