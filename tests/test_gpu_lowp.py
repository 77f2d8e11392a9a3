"""GPU parity of the low-precision caches against the oracle's format
definitions (oracle/lowp.py):

* the FP8 KV records and the MXFP4 rows the quantisers write, decoded and
  compared bit for bit with the oracle's dequantised values (these are byte
  work: exact), on inputs that include all-zero groups, exact E4M3 / E2M1
  ties, subnormal quotients and wide magnitude ranges;
* the decode scores over MXFP4 keys: BF16 values, each equal to the oracle's
  BF16 score or one BF16 step from it (the GPU rounds an fp32 score, the
  oracle an fp64 one), almost all equal;
* the whole low-precision decode step at the Flash-decode and Pro-decode
  shapes: selections against the oracle's top-k of its own BF16 scores
  wherever the k-th and (k+1)-th of them are more than two BF16 steps apart
  (no one-step difference can reorder them there), outputs within the bf16
  tolerance against the oracle's attention over the dequantised entries.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import lowp
from parity import check_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_sparse_22_b300 as m
    m.lib()
    return m


def _rng(seed):
    return np.random.default_rng(seed)


def decode_fp8_records(rec: np.ndarray) -> np.ndarray:
    """[rows, 592] uint8 records -> [rows, 512] float64 values (from the stated layout)."""
    rows = rec.shape[0]
    codes = rec[:, :448].astype(np.int64)
    s = np.where(codes & 0x80, -1.0, 1.0)
    E = (codes >> 3) & 15
    m = codes & 7
    val = np.where(E == 0, m * 2.0 ** -9, (8 + m) * np.exp2(E - 10.0)) * s
    scales = rec[:, 576:592].copy().view(np.float32).astype(np.float64)   # [rows, 4]
    grp = np.minimum(np.arange(448) // 128, 3)
    out = np.empty((rows, 512))
    out[:, :448] = val * scales[:, grp]
    rot = rec[:, 448:576].copy().view(np.uint16)
    out[:, 448:] = synth.widen(rot, "bf16")
    return out


E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def decode_fp4_rows(buf: np.ndarray, rows: int) -> np.ndarray:
    """MXFP4 planar buffer -> [rows, 128] float64 values (from the stated layout)."""
    codes = buf[:rows * 64].reshape(rows, 64)
    nib = np.empty((rows, 128), np.int64)
    nib[:, 0::2] = codes & 15
    nib[:, 1::2] = codes >> 4
    val = E2M1_MAG[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    sc = buf[rows * 64: rows * 64 + rows * 4].reshape(rows, 4).astype(np.int64) - 127
    return val * np.exp2(np.repeat(sc, 32, axis=1).astype(np.float64))


def _hard_entries(rows, seed):
    """bf16 entries with zero groups, exact ties after scaling, tiny and huge values."""
    r = _rng(seed)
    x = r.standard_normal((rows, 512)) * np.exp2(r.integers(-12, 12, (rows, 1)))
    x[0, :128] = 0.0                                   # an all-zero group
    x[1, 128:256] = 1e-30                              # quotients at the top of the range
    x[2, 256:384] *= 1e-3
    x[2, 256] = 448.0                                  # scale 1: codes are the values themselves
    x[2, 257:300] = np.array([0.5 + 0.0625 * k for k in range(43)])   # midpoints of the 2^-1 binade
    x[3, 384:448] = np.exp2(r.integers(-20, 8, 64)).astype(np.float64)
    x[3, 384] = 448.0 * 2 ** 7
    return synth.to_storage(x, "bf16")


def test_quantize_kv_fp8_exact(csa):
    rows = 777
    xs = _hard_entries(rows, 11)
    rec = host(csa.quantize_kv_fp8(dev(xs)))
    got = decode_fp8_records(rec.astype(np.uint8))
    want = lowp.kv_entry_fp8(synth.widen(xs, "bf16"), rope_dims=64, group=128)
    assert np.array_equal(got, want)
    # the scales are the fp32 amax / 448 of each group (1 for the zero group)
    sc = rec[:, 576:592].astype(np.uint8).copy().view(np.float32)
    x32 = synth.widen(xs, "bf16").astype(np.float32)
    for gi, (g0, g1) in enumerate(((0, 128), (128, 256), (256, 384), (384, 448))):
        am = np.abs(x32[:, g0:g1]).max(1)
        ref = np.where(am > 0, (am.astype(np.float64) / 448.0).astype(np.float32), np.float32(1.0))
        assert np.array_equal(sc[:, gi], ref)


def _hard_rows(rows, seed):
    r = _rng(seed)
    x = r.standard_normal((rows, 128)) * np.exp2(r.integers(-30, 30, (rows, 4)).repeat(32, axis=1))
    x[0, :32] = 0.0                                    # an all-zero block
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 0.0625])
    x[1, 32:42] = ties                                 # amax 7 -> scale 1: ties to even, saturation
    x[1, 42:64] = 0.1
    x[2, 64:74] = -ties * 2.0 ** -10
    x[2, 74:96] = 1e-6 * 2.0 ** -10
    return synth.to_storage(x, "bf16")


def test_quantize_index_fp4_exact(csa):
    rows = 1001                                        # not a multiple of 4
    xs = _hard_rows(rows, 12)
    buf = host(csa.quantize_index_fp4(dev(xs))).astype(np.uint8)
    assert buf.size == csa.lib().index_fp4_bytes(rows)
    got = decode_fp4_rows(buf, rows)
    want = lowp.mxfp4(synth.widen(xs, "bf16"))
    assert np.array_equal(got, want)


def _bf16_step(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.exp2(np.maximum(e, -126) - 7)


@pytest.mark.parametrize("B,E,t", [(3, 5001, 20003), (2, 700, 1500), (1, 262144, 1048575)])
def test_indexer_score_fp4(csa, B, E, t):
    seed = 600 + E
    qI = synth.normal(seed, 1, (B, 1, 64, 128), 1.0, "bf16")
    kI = synth.normal(seed, 2, (B, E, 128), 1.0, "bf16")
    w = synth.softmax_normal(seed, 3, (B, 1, 64))
    w[..., ::5] *= -1.0
    pos = np.array([[t - 97 * b] for b in range(B)], np.int64)
    kI4 = csa.quantize_index_fp4(dev(kI))
    sc = host(csa.indexer_score_fp4(dev(qI), dev(w), kI4, dev(pos), E, 4))
    same = total = 0
    for b in range(B):
        ref = lowp.index_scores_lowp(synth.widen(qI[b, 0], "bf16")[None], w[b], pos[b],
                                     synth.widen(kI[b], "bf16"), 4)[0]
        g = sc[b, 0]
        fin = np.isfinite(ref)
        assert np.array_equal(np.isfinite(g), fin)
        assert np.all(np.isneginf(g[~fin]))
        d = np.abs(g[fin] - ref[fin])
        assert np.all(d <= _bf16_step(ref[fin]) * 1.0000001), "a score more than one BF16 step away"
        assert np.array_equal(g[fin], lowp.bf16_round(g[fin])), "scores are not BF16 values"
        same += int((d == 0).sum())
        total += int(fin.sum())
    assert same >= 0.99 * total, f"only {same} of {total} BF16 scores equal"


def _lowp_decode(csa, s, x, hca):
    d = {k: dev(v) for k, v in x.items()}
    kv8 = csa.quantize_kv_fp8(d["kvc"])
    kI4 = csa.quantize_index_fp4(d["kIc"])
    p = csa.params(m=s["m"], top_k=s["top_k"], n_win=s["n_win"], rope_dims=s["rope_dims"],
                   rope_theta=s["theta"], cache_format=1)
    p2 = csa.params(m=s.get("m2", 128), n_win=s["n_win"], rope_dims=s["rope_dims"],
                    rope_theta=s["theta"], cache_format=1)
    io = torch.empty((s["B"], 1, s["top_k"]), dtype=torch.int32, device="cuda")
    kw = {}
    if hca:
        kw = dict(q2=d["q2"], kvc2=csa.quantize_kv_fp8(d["kvc2"]), kv_raw2=d["kv_raw2"],
                  sink2=d["sink2"], p2=p2)
    res = csa.hybrid_decode(d["q"], d["qI"], d["w"], kv8, kI4, d["kv_raw"], d["sink"], d["q_pos"],
                            d["raw_pos0"], p, idx_out=io, **kw)
    # the same scores through the standalone entry point (same kernel, same grid)
    sc = csa.indexer_score_fp4(d["qI"], d["w"], kI4, d["q_pos"], x["kIc"].shape[1], s["m"])
    torch.cuda.synchronize()
    return res, io, host(sc)


def _orc_attend_entries(orc, s, q, pos, ent, m, raw, rp0, sink, idx):
    """Attention over the listed entries: the listed rows are dequantised from
    their FP8 records' definition and renumbered (stored entries carry their
    rotation, so only the set matters)."""
    sel = idx[idx >= 0]
    kv = lowp.kv_entry_fp8(synth.widen(ent[sel], "bf16"), rope_dims=64, group=128)
    if kv.shape[0] == 0:
        kv = np.zeros((1, ent.shape[1]))
    ridx = np.full_like(idx, -1)
    ridx[0, :sel.size] = np.arange(sel.size)
    return orc.attend(q, pos, kv, m, synth.widen(raw, "bf16"), rp0, sink, idx=ridx, n_win=s["n_win"],
                      rope_dims=s["rope_dims"], theta=s["theta"])


def _check_lowp(orc, s, x, res, io, gsc, seqs, hca):
    out, out2 = (res if hca else (res, None))
    k, m = s["top_k"], s["m"]
    differ = 0
    for b in seqs:
        qp = x["q_pos"][b]
        # selection over the GPU's own BF16 scores: integer work, exact (ties to the lower index)
        np.testing.assert_array_equal(host(io[b]), orc.topk(gsc[b], qp, m, k)[0])
        sc = lowp.index_scores_lowp(synth.widen(x["qI"][b], "bf16"), x["w"][b], qp,
                                    synth.widen(x["kIc"][b], "bf16"), m)
        oi, oc = orc.topk(sc, qp, m, k)
        gi = host(io[b])
        row = np.sort(sc[0][np.isfinite(sc[0])])[::-1]
        if row.size > k:
            gap = row[k - 1] - row[k]
            fixed = gap > 2 * _bf16_step(np.array([row[k - 1]]))[0]
        else:
            fixed = True
        if fixed:
            np.testing.assert_array_equal(gi, oi)
        elif not np.array_equal(gi, oi):
            differ += 1
        ref = _orc_attend_entries(orc, s, x["q"][b], qp, x["kvc"][b], m, x["kv_raw"][b],
                                  int(x["raw_pos0"][b]), x["sink"], gi)
        check_close(host(out[b]), ref, "bf16", f"low-precision decode out seq {b}")
        if hca:
            E2 = x["kvc2"].shape[1]
            allidx = np.arange(E2, dtype=np.int32)[None]
            nv2 = min(E2, (int(qp[0]) + 1) // s["m2"])
            allidx[0, nv2:] = -1
            ref2 = _orc_attend_entries(orc, s, x["q2"][b], qp, x["kvc2"][b], s["m2"], x["kv_raw2"][b],
                                       int(x["raw_pos0"][b]), x["sink2"], allidx)
            check_close(host(out2[b]), ref2, "bf16", f"low-precision hca out seq {b}")
    return differ


def test_lowp_decode_cfg3_flash(csa, orc):
    """Flash-shaped CSA decode (B=32, 32768 entries) on FP8 / MXFP4 caches."""
    s, x = synth.make_inputs("csa_decode_flash")
    res, io, gsc = _lowp_decode(csa, s, x, False)
    _check_lowp(orc, s, x, res, io, gsc, [0, 13, 31], False)


def test_lowp_decode_cfg5_pro(csa, orc):
    """Pro-shaped hybrid decode at 1,048,576 positions (B=8) on FP8 / MXFP4 caches."""
    s, x = synth.make_inputs("hybrid_decode_pro")
    res, io, gsc = _lowp_decode(csa, s, x, True)
    _check_lowp(orc, s, x, res, io, gsc, [0, 5], True)


def test_lowp_decode_small_and_split(csa, orc):
    """A short history (fewer visible entries than k, the split-KV path with
    FP8 tiles) and exact BF16 ties broken toward the lower index."""
    s, x = synth.make_inputs("hybrid_decode_pro", B=3, t=8191)
    s3, x3 = synth.make_inputs("hybrid_decode_pro", B=3, t=3000)
    x["kIc"][1, 300:1800] = x["kIc"][1, 5]              # 1501 equal keys straddle the k-th place
    for xx, ss in ((x, s), (x3, s3)):
        res, io, gsc = _lowp_decode(csa, ss, xx, True)
        _check_lowp(orc, ss, xx, res, io, gsc, [0, 1, 2], True)
    # the tie group is cut at the lower indices
    sel = host(io[1, 0])
    grp = set(range(300, 1800)) | {5}
    chosen = sorted(j for j in sel if j in grp)
    assert chosen == sorted(grp)[:len(chosen)]
