"""The five synthetic CSA/HCA workloads and their input recipes.

Each workload is a dict of sizes plus a recipe (which tensors, which
distribution).  `make_inputs(name, **overrides)` draws the host arrays in
their storage dtype; overrides shrink a workload (e.g. n=1024) for parity
tests while keeping its structure.  Shapes are row-major, batch outermost.
"""
from __future__ import annotations

import math

import numpy as np

from . import normal, softmax_normal

# tensor ids: stable across workloads so that a tensor keeps its stream
TID = {name: i + 1 for i, name in enumerate([
    "C", "Z", "bias", "Cb", "Zb", "biasb", "Ck", "Zk", "biask", "Ckb", "Zkb", "biaskb",
    "q", "qI", "w", "sink",
    "C2", "Z2", "bias2", "q2", "sink2",
    "kvc", "kIc", "kv_raw", "kvc2", "kv_raw2",
])}

WORKLOADS = {
    # CSA single-layer prefill, fp32
    "csa_prefill_f32": dict(kind="csa_prefill", dtype="f32", seed=0, B=1, n=2048, H=4, c=64,
                            rope_dims=32, theta=10000.0, m=4, hI=4, dI=32, top_k=64,
                            n_win=128, overlap=0, in_scale=1.0),
    # HCA single-layer prefill, bf16, inputs scaled by 1/sqrt(d)
    "hca_prefill_bf16": dict(kind="hca_prefill", dtype="bf16", seed=1, B=1, n=8192, H=16, c=128,
                             rope_dims=64, theta=10000.0, m=128, n_win=128,
                             in_scale=1.0 / math.sqrt(128.0)),
    # Flash-shaped CSA decode, bf16
    "csa_decode_flash": dict(kind="csa_decode", dtype="bf16", seed=2, B=32, t=131072, H=64,
                             c=512, rope_dims=64, theta=10000.0, m=4, hI=64, dI=128,
                             top_k=512, n_win=128),
    # Flash-shaped interleaved CSA + HCA prefill, bf16
    "hybrid_prefill_flash": dict(kind="hybrid_prefill", dtype="bf16", seed=3, B=1, n=65536,
                                 H=64, c=512, rope_dims=64, theta=10000.0, m=4, m2=128,
                                 hI=64, dI=128, top_k=512, n_win=128, overlap=0,
                                 in_scale=1.0),
    # Pro-shaped hybrid decode at 1,048,576 positions, bf16
    "hybrid_decode_pro": dict(kind="hybrid_decode", dtype="bf16", seed=4, B=8, t=1048576,
                              H=128, c=512, rope_dims=64, theta=10000.0, m=4, m2=128,
                              hI=64, dI=128, top_k=1024, n_win=128),
}

BIAS_STD = 0.1


def spec(name: str, **overrides) -> dict:
    s = dict(WORKLOADS[name])
    s.update(overrides)
    s["name"] = name
    return s


def _csa_layer(s, out, prefix=""):
    seed, dt, B, n, c = s["seed"], s["dtype"], s["B"], s["n"], s["c"]
    m, hI, dI, H = s["m"], s["hI"], s["dI"], s["H"]
    sc = s.get("in_scale", 1.0)
    out["C"] = normal(seed, TID["C"], (B, n, c), sc, dt)
    out["Z"] = normal(seed, TID["Z"], (B, n, c), sc, dt)
    out["bias"] = normal(seed, TID["bias"], (m, c), BIAS_STD, "f32")
    out["Ck"] = normal(seed, TID["Ck"], (B, n, dI), sc, dt)
    out["Zk"] = normal(seed, TID["Zk"], (B, n, dI), sc, dt)
    out["biask"] = normal(seed, TID["biask"], (m, dI), BIAS_STD, "f32")
    if s.get("overlap", 0):
        out["Cb"] = normal(seed, TID["Cb"], (B, n, c), sc, dt)
        out["Zb"] = normal(seed, TID["Zb"], (B, n, c), sc, dt)
        out["biasb"] = normal(seed, TID["biasb"], (m, c), BIAS_STD, "f32")
        out["Ckb"] = normal(seed, TID["Ckb"], (B, n, dI), sc, dt)
        out["Zkb"] = normal(seed, TID["Zkb"], (B, n, dI), sc, dt)
        out["biaskb"] = normal(seed, TID["biaskb"], (m, dI), BIAS_STD, "f32")
    out["q"] = normal(seed, TID["q"], (B, n, H, c), sc, dt)
    out["qI"] = normal(seed, TID["qI"], (B, n, hI, dI), sc, dt)
    out["w"] = softmax_normal(seed, TID["w"], (B, n, hI))
    out["sink"] = normal(seed, TID["sink"], (H,), 1.0, "f32")


def _hca_layer(s, out, suffix=""):
    seed, dt, B, n, c, H = s["seed"], s["dtype"], s["B"], s["n"], s["c"], s["H"]
    m = s["m2"] if suffix else s["m"]
    sc = s.get("in_scale", 1.0)
    out["C" + suffix] = normal(seed, TID["C" + suffix], (B, n, c), sc, dt)
    out["Z" + suffix] = normal(seed, TID["Z" + suffix], (B, n, c), sc, dt)
    out["bias" + suffix] = normal(seed, TID["bias" + suffix], (m, c), BIAS_STD, "f32")
    out["q" + suffix] = normal(seed, TID["q" + suffix], (B, n, H, c), sc, dt)
    out["sink" + suffix] = normal(seed, TID["sink" + suffix], (H,), 1.0, "f32")


def make_inputs(name: str, **overrides) -> tuple[dict, dict]:
    """Return (spec, arrays) for a workload, arrays in storage dtype."""
    s = spec(name, **overrides)
    kind, seed, dt = s["kind"], s["seed"], s["dtype"]
    out: dict[str, np.ndarray] = {}
    if kind == "csa_prefill":
        _csa_layer(s, out)
    elif kind == "hca_prefill":
        _hca_layer(s, out)
    elif kind == "hybrid_prefill":
        _csa_layer(s, out)
        _hca_layer(s, out, "2")
    elif kind in ("csa_decode", "hybrid_decode"):
        B, t, H, c, m = s["B"], s["t"], s["H"], s["c"], s["m"]
        hI, dI, W = s["hI"], s["dI"], s["n_win"]
        E = s.get("E", (t + 1) // m)
        s["E"] = E
        out["kvc"] = normal(seed, TID["kvc"], (B, E, c), 1.0, dt)
        out["kIc"] = normal(seed, TID["kIc"], (B, E, dI), 1.0, dt)
        out["kv_raw"] = normal(seed, TID["kv_raw"], (B, W, c), 1.0, dt)
        out["q"] = normal(seed, TID["q"], (B, 1, H, c), 1.0, dt)
        out["qI"] = normal(seed, TID["qI"], (B, 1, hI, dI), 1.0, dt)
        out["w"] = softmax_normal(seed, TID["w"], (B, 1, hI))
        out["sink"] = normal(seed, TID["sink"], (H,), 1.0, "f32")
        if kind == "hybrid_decode":
            m2 = s["m2"]
            E2 = s.get("E2", (t + 1) // m2)
            s["E2"] = E2
            out["kvc2"] = normal(seed, TID["kvc2"], (B, E2, c), 1.0, dt)
            out["kv_raw2"] = normal(seed, TID["kv_raw2"], (B, W, c), 1.0, dt)
            out["q2"] = normal(seed, TID["q2"], (B, 1, H, c), 1.0, dt)
            out["sink2"] = normal(seed, TID["sink2"], (H,), 1.0, "f32")
        # decode query position = number of cached tokens; the window rows hold
        # positions t-W+1 .. t (the new token's row last)
        out["q_pos"] = np.full((B, 1), t, np.int64)
        out["raw_pos0"] = np.full((B,), t - W + 1, np.int64)
    else:
        raise ValueError(kind)
    if kind in ("csa_prefill", "hca_prefill", "hybrid_prefill"):
        out["q_pos"] = np.broadcast_to(np.arange(s["n"], dtype=np.int64), (s["B"], s["n"])).copy()
        out["raw_pos0"] = np.zeros((s["B"],), np.int64)
    return s, out
