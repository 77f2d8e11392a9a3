"""fp64 CPU oracle for the CSA/HCA attention layer (test infrastructure).

Only the tests, the smoke check and the bench's CPU-baseline leg may import
this package.  The product library never loads it and shares no code with
it.  The arithmetic lives in `csa_oracle.c` (plain C, OpenMP over queries or
entries); this module is ctypes marshalling plus the composition of the
layer's steps in the order the pages give them:

  CSA prefill:  compress KV (RoPE at each block's last position) and the
                indexer keys (no RoPE) -> index scores -> top-k ->
                attention over the selected entries + window + sink.
  HCA prefill:  compress KV with m' -> attention over all visible entries +
                window + sink.
  decode:       the caches are inputs; scores -> top-k -> attention.

Inputs are numpy arrays in storage dtype (float64, float32, or uint16
bfloat16 bits), widened exactly to double inside the C code.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

DT = {"f64": 0, "f32": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile the oracle's C source into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
               "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        P, I64, I32, D = C.c_void_p, C.c_int64, C.c_int, C.c_double
        L.orc_rope.argtypes = [P, I32, I32, D, D]
        L.orc_rope_rows.argtypes = [I32, P, I64, I32, I32, D, I64, I32, P]
        L.orc_compress.argtypes = [I32, P, P, P, I32, P, P, P, I64, I32, I32, I32, I32, D, I32, P]
        L.orc_visible.argtypes = [I64, I32, I64]
        L.orc_visible.restype = I64
        L.orc_index_scores.argtypes = [I32, P, I32, P, P, I64, I32, I32, I32, P, I64, I32, P]
        L.orc_topk.argtypes = [P, P, I64, I64, I32, I32, P, P]
        L.orc_attend.argtypes = [I32, P, P, I64, I32, I32, I32, P, I64, I32, P, I32,
                                 P, I64, I64, I32, I32, P, I32, D, D, I32, P, P]
        L.orc_attend.restype = I64
        L.orc_round.argtypes = [P, I64, I32]
        _lib = L
    return _lib


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float64:
        return 0
    if a.dtype == np.float32:
        return 1
    if a.dtype == np.uint16:
        return 2
    raise TypeError(a.dtype)


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a):
    return None if a is None else np.ascontiguousarray(a)


# ------------------------------------------------------------------ steps

def visible(t: int, m: int, E: int) -> int:
    """Number of compressed entries visible at query position t."""
    return int(lib().orc_visible(int(t), int(m), int(E)))


def rope(x: np.ndarray, p: float, r: int, theta: float = 10000.0) -> np.ndarray:
    """RoPE on the last r dims of a 1-D float64 vector at position p."""
    y = np.array(x, dtype=np.float64, copy=True)
    lib().orc_rope(_p(y), y.shape[-1], int(r), float(theta), float(p))
    return y


def rope_rows(x: np.ndarray, pos0: int, r: int, theta: float, out_dtype: str) -> np.ndarray:
    """Rows x[l] rotated at position pos0 + l, rounded to out_dtype."""
    x = _c(x)
    L, c = x.shape
    out = np.empty((L, c), np.float64)
    lib().orc_rope_rows(_dt(x), _p(x), L, c, int(r), float(theta), int(pos0), DT[out_dtype], _p(out))
    return out


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    y = np.array(x, dtype=np.float64, copy=True)
    lib().orc_round(_p(y), y.size, DT[dtype])
    return y


def compress(Cc, Zc, bias, m, *, overlap=0, Cb=None, Zb=None, biasb=None,
             rope_dims=0, theta=10000.0, out_dtype="f64") -> np.ndarray:
    """One sequence: C, Z [n, c], bias [m, c] -> entries [n // m, c] (float64
    holding values rounded to out_dtype)."""
    Cc, Zc, bias = _c(Cc), _c(Zc), _c(bias)
    n, c = Cc.shape
    if overlap:
        Cb, Zb, biasb = _c(Cb), _c(Zb), _c(biasb)
        assert Cb.dtype == Cc.dtype and Zb.dtype == Cc.dtype and biasb.dtype == bias.dtype
    assert Zc.dtype == Cc.dtype
    out = np.empty((n // m, c), np.float64)
    lib().orc_compress(_dt(Cc), _p(Cc), _p(Zc), _p(bias), _dt(bias),
                       _p(Cb), _p(Zb), _p(biasb), n, c, int(m), int(overlap),
                       int(rope_dims), float(theta), DT[out_dtype], _p(out))
    return out


def index_scores(qI, w, q_pos, kI, m) -> np.ndarray:
    """One sequence: qI [T, hI, dI], w [T, hI], q_pos [T], kI [E, dI] ->
    scores [T, E] (float64, -inf where not visible)."""
    qI, w, kI = _c(qI), _c(w), _c(kI)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int64)
    T, hI, dI = qI.shape
    E = kI.shape[0]
    out = np.empty((T, E), np.float64)
    lib().orc_index_scores(_dt(qI), _p(qI), _dt(w), _p(w), _p(q_pos), T, hI, dI,
                           _dt(kI), _p(kI), E, int(m), _p(out))
    return out


def topk(scores, q_pos, m, k):
    """One sequence: scores [T, E] -> (idx [T, k] int32 ascending, -1 padded, cnt [T])."""
    scores = np.ascontiguousarray(scores, dtype=np.float64)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int64)
    T, E = scores.shape
    idx = np.empty((T, k), np.int32)
    cnt = np.empty((T,), np.int32)
    lib().orc_topk(_p(scores), _p(q_pos), T, E, int(m), int(k), _p(idx), _p(cnt))
    return idx, cnt


def attend(q, q_pos, kvc, m, kv_raw, raw_pos0, sink, *, idx=None, n_win=128,
           rope_dims=64, theta=10000.0, scale=0.0, derotate=1, want_lse=False):
    """One sequence: q [T, H, c]; kvc [E, c] stored entries; idx [T, k] or None
    (None = every visible entry, the HCA path); kv_raw [L, c] stored raw rows
    (row l at position raw_pos0 + l); sink [H] -> out [T, H, c] (and lse)."""
    q, kvc, kv_raw, sink = _c(q), _c(kvc), _c(kv_raw), _c(sink)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int64)
    T, H, c = q.shape
    E = kvc.shape[0]
    L = kv_raw.shape[0]
    assert kvc.dtype == kv_raw.dtype
    k = 0
    if idx is not None:
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        k = idx.shape[1]
    out = np.empty((T, H, c), np.float64)
    lse = np.empty((T, H), np.float64) if want_lse else None
    missing = lib().orc_attend(_dt(q), _p(q), _p(q_pos), T, H, c, _dt(kvc), _p(kvc), E, int(m),
                               _p(idx), int(k), _p(kv_raw), L, int(raw_pos0), int(n_win),
                               _dt(sink), _p(sink), int(rope_dims), float(theta), float(scale),
                               int(derotate), _p(out), _p(lse))
    if missing:
        raise ValueError(f"kv_raw does not cover {missing} window positions")
    return (out, lse) if want_lse else out


# ------------------------------------------------------------ compositions

def _storage(a_f64: np.ndarray, dtype: str) -> np.ndarray:
    """Values already rounded to dtype, as the storage array the next step reads."""
    return a_f64.astype(np.float32) if dtype == "f32" else _bf16_bits_exact(a_f64)


def _bf16_bits_exact(a: np.ndarray) -> np.ndarray:
    f = a.astype(np.float32)              # exact: values are bf16-representable
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def csa_prefill_prepare(s: dict, x: dict, b: int = 0) -> dict:
    """CSA layer, the per-sequence part: compressed KV (rotated at each block's
    last position), compressed indexer keys (no RoPE) and the stored raw rows
    (rotated at their positions), each rounded to the storage dtype."""
    dt, m, r, th = s["dtype"], s["m"], s["rope_dims"], s["theta"]
    ov = s.get("overlap", 0)
    kvc = compress(x["C"][b], x["Z"][b], x["bias"], m, overlap=ov,
                   Cb=x["Cb"][b] if ov else None, Zb=x["Zb"][b] if ov else None,
                   biasb=x.get("biasb"), rope_dims=r, theta=th, out_dtype=dt)
    kIc = compress(x["Ck"][b], x["Zk"][b], x["biask"], m, overlap=ov,
                   Cb=x["Ckb"][b] if ov else None, Zb=x["Zkb"][b] if ov else None,
                   biasb=x.get("biaskb"), rope_dims=0, out_dtype=dt)
    raw = rope_rows(x["C"][b], 0, r, th, dt)
    return dict(kvc=kvc, kIc=kIc, raw=raw, kvc_s=_storage(kvc, dt), kIc_s=_storage(kIc, dt),
                raw_s=_storage(raw, dt))


def csa_prefill_queries(s: dict, x: dict, prep: dict, b: int = 0, q_sel=None) -> dict:
    """CSA layer, per query: index scores -> top-k -> attention."""
    m, r, th = s["m"], s["rope_dims"], s["theta"]
    qp = x["q_pos"][b] if q_sel is None else np.asarray(q_sel, np.int64)
    sel = qp if q_sel is not None else slice(None)
    sc = index_scores(x["qI"][b][sel], x["w"][b][sel], qp, prep["kIc_s"], m)
    idx, cnt = topk(sc, qp, m, s["top_k"])
    out = attend(x["q"][b][sel], qp, prep["kvc_s"], m, prep["raw_s"], 0, x["sink"], idx=idx,
                 n_win=s["n_win"], rope_dims=r, theta=th, derotate=s.get("derotate", 1))
    return dict(scores=sc, idx=idx, cnt=cnt, out=out)


def csa_prefill_seq(s: dict, x: dict, b: int = 0, q_sel=None, return_steps=False):
    """CSA layer prefill for batch row b of a workload (spec s, inputs x).
    q_sel: optional array of query positions to evaluate (default all)."""
    prep = csa_prefill_prepare(s, x, b)
    res = csa_prefill_queries(s, x, prep, b, q_sel)
    if return_steps:
        return dict(kvc=prep["kvc"], kIc=prep["kIc"], raw=prep["raw"], **res)
    return res["out"]


def hca_prefill_prepare(s: dict, x: dict, b: int = 0, suffix="") -> dict:
    dt, r, th = s["dtype"], s["rope_dims"], s["theta"]
    m = s["m2"] if suffix else s["m"]
    kvc = compress(x["C" + suffix][b], x["Z" + suffix][b], x["bias" + suffix], m,
                   rope_dims=r, theta=th, out_dtype=dt)
    raw = rope_rows(x["C" + suffix][b], 0, r, th, dt)
    return dict(kvc=kvc, raw=raw, kvc_s=_storage(kvc, dt), raw_s=_storage(raw, dt))


def hca_prefill_queries(s: dict, x: dict, prep: dict, b: int = 0, q_sel=None, suffix=""):
    r, th = s["rope_dims"], s["theta"]
    m = s["m2"] if suffix else s["m"]
    qp = x["q_pos"][b] if q_sel is None else np.asarray(q_sel, np.int64)
    sel = qp if q_sel is not None else slice(None)
    return attend(x["q" + suffix][b][sel], qp, prep["kvc_s"], m, prep["raw_s"], 0,
                  x["sink" + suffix], idx=None, n_win=s["n_win"], rope_dims=r, theta=th,
                  derotate=s.get("derotate", 1))


def hca_prefill_seq(s: dict, x: dict, b: int = 0, q_sel=None, suffix="", return_steps=False):
    """HCA layer prefill for batch row b (suffix "2" = the HCA layer of a hybrid)."""
    prep = hca_prefill_prepare(s, x, b, suffix)
    out = hca_prefill_queries(s, x, prep, b, q_sel, suffix)
    if return_steps:
        return dict(kvc=prep["kvc"], raw=prep["raw"], out=out)
    return out


def csa_decode_seq(s: dict, x: dict, b: int, return_steps=False):
    """CSA decode for sequence b: caches are inputs (stored, rotated)."""
    m, r, th = s["m"], s["rope_dims"], s["theta"]
    qp = x["q_pos"][b]
    sc = index_scores(x["qI"][b], x["w"][b], qp, x["kIc"][b], m)
    idx, cnt = topk(sc, qp, m, s["top_k"])
    out = attend(x["q"][b], qp, x["kvc"][b], m, x["kv_raw"][b], int(x["raw_pos0"][b]),
                 x["sink"], idx=idx, n_win=s["n_win"], rope_dims=r, theta=th,
                 derotate=s.get("derotate", 1))
    if return_steps:
        return dict(scores=sc, idx=idx, cnt=cnt, out=out)
    return out


def hca_decode_seq(s: dict, x: dict, b: int):
    """HCA decode for sequence b over every visible entry of kvc2."""
    r, th = s["rope_dims"], s["theta"]
    qp = x["q_pos"][b]
    return attend(x["q2"][b], qp, x["kvc2"][b], s["m2"], x["kv_raw2"][b], int(x["raw_pos0"][b]),
                  x["sink2"], idx=None, n_win=s["n_win"], rope_dims=r, theta=th,
                  derotate=s.get("derotate", 1))
