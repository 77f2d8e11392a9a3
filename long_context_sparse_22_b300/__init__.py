"""Python binding of libcsa, the B300 (sm_103a) CSA / HCA attention library.

Argument marshalling only: every step runs in the CUDA kernels of
`libcsa.so`; PyTorch supplies device memory and the current stream.  The
entry points carry the C ABI's names (include/csa.h).  There is no CPU
path: if the library is missing or no CUDA device is present, the calls
raise.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")
_lib = None

CSA_F32, CSA_BF16 = 0, 1
STATUS_NAMES = {0: "CSA_OK", 1: "CSA_ERR_INVALID_ARG", 2: "CSA_ERR_UNSUPPORTED",
                3: "CSA_ERR_WORKSPACE", 4: "CSA_ERR_CUDA", 5: "CSA_ERR_TIMEOUT", 6: "CSA_ERR_DEVICE"}


class CsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class CsaParams(C.Structure):
    _fields_ = [("m", C.c_int32), ("overlap", C.c_int32), ("top_k", C.c_int32),
                ("n_win", C.c_int32), ("rope_dims", C.c_int32), ("derotate", C.c_int32),
                ("rope_theta", C.c_double), ("scale", C.c_float), ("batch_invariant", C.c_int32),
                ("spin_limit", C.c_int64), ("cache_format", C.c_int32),
                ("q_norm", C.c_void_p), ("kv_norm", C.c_void_p), ("norm_eps", C.c_float)]

CACHE_DTYPE, CACHE_LOWP = 0, 1
KV_FP8_BYTES = 592


def params(m=4, overlap=0, top_k=512, n_win=128, rope_dims=64, derotate=1, rope_theta=10000.0,
           scale=0.0, batch_invariant=0, spin_limit=0, cache_format=0, q_norm=None, kv_norm=None,
           norm_eps=0.0) -> CsaParams:
    """Layer parameters; q_norm / kv_norm are float32 device tensors of c gains
    (kept alive by the caller while the parameters are in use) or None."""
    return CsaParams(int(m), int(overlap), int(top_k), int(n_win), int(rope_dims), int(derotate),
                     float(rope_theta), float(scale), int(batch_invariant), int(spin_limit),
                     int(cache_format), _p(q_norm), _p(kv_norm), float(norm_eps))


_SIGS = {
    "csa_last_error": ([], C.c_char_p),
    "csa_version": ([], C.c_char_p),
    "csa_launch_count": ([], C.c_int64),
    "csa_stream_status": ([C.c_void_p, C.c_void_p], C.c_int),
    "csa_workspace_init": ([C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "csa_wait_probe": ([C.c_int64, C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "csa_timing_enable": ([C.c_int32], C.c_int),
    "csa_timing_read": ([C.POINTER(C.c_double), C.POINTER(C.c_int64), C.c_int32], C.c_int),
    "csa_compress": ([C.c_int, C.c_int64, C.c_int64, C.c_int32] + [C.c_void_p] * 8
                     + [C.POINTER(CsaParams), C.c_void_p], C.c_int),
    "indexer_score_ws_size": ([], C.c_size_t),
    "indexer_score": ([C.c_int, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int64, C.c_int32]
                      + [C.c_void_p] * 5 + [C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "topk_select_ws_size": ([C.c_int64, C.c_int64, C.c_int64, C.c_int32], C.c_size_t),
    "topk_select": ([C.c_int64, C.c_int64, C.c_int64, C.c_int32, C.c_int32] + [C.c_void_p] * 4
                    + [C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "topk_select_noalloc": ([C.c_int64, C.c_int64, C.c_int64, C.c_int32, C.c_int32] + [C.c_void_p] * 4
                            + [C.c_void_p], C.c_int),
    "attn_ws_size": ([C.c_int, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int64, C.c_int32,
                      C.POINTER(CsaParams)], C.c_size_t),
    "sparse_attn": ([C.c_int, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int64, C.c_int32,
                     C.c_int64] + [C.c_void_p] * 9 + [C.POINTER(CsaParams), C.c_void_p, C.c_size_t,
                                                      C.c_void_p], C.c_int),
    "hca_attn": ([C.c_int, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int64, C.c_int64]
                 + [C.c_void_p] * 8 + [C.POINTER(CsaParams), C.c_void_p, C.c_size_t,
                                       C.c_void_p], C.c_int),
    "csa_prefill_ws_size": ([C.c_int, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int32,
                             C.c_int32, C.POINTER(CsaParams)], C.c_size_t),
    "csa_prefill": ([C.c_int, C.c_int64, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32]
                    + [C.c_void_p] * 18 + [C.POINTER(CsaParams), C.c_void_p, C.c_size_t,
                                           C.c_void_p], C.c_int),
    "hca_prefill_ws_size": ([C.c_int, C.c_int64, C.c_int64, C.c_int32, C.c_int32,
                             C.POINTER(CsaParams)], C.c_size_t),
    "hca_prefill": ([C.c_int, C.c_int64, C.c_int64, C.c_int32, C.c_int32] + [C.c_void_p] * 6
                    + [C.POINTER(CsaParams), C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "hybrid_decode_ws_size": ([C.c_int, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                               C.c_int64, C.c_int64, C.POINTER(CsaParams), C.POINTER(CsaParams)],
                              C.c_size_t),
    "hybrid_decode": ([C.c_int, C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int64,
                       C.c_int64, C.c_int64] + [C.c_void_p] * 16
                      + [C.POINTER(CsaParams), C.POINTER(CsaParams), C.c_void_p, C.c_size_t,
                         C.c_void_p], C.c_int),
    "index_fp4_bytes": ([C.c_int64], C.c_size_t),
    "quantize_kv_fp8": ([C.c_int, C.c_int64, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p],
                        C.c_int),
    "quantize_index_fp4": ([C.c_int, C.c_int64, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p], C.c_int),
    "indexer_score_fp4": ([C.c_int64, C.c_int64, C.c_int32] + [C.c_void_p] * 5
                          + [C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "out_proj_ws_size": ([C.c_int64, C.c_int32, C.c_int32, C.c_int32], C.c_size_t),
    "out_proj": ([C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32] + [C.c_void_p] * 4
                 + [C.c_void_p, C.c_size_t, C.c_void_p], C.c_int),
    "decode_tail_bytes": ([C.c_int, C.c_int64, C.c_int32, C.c_int32, C.POINTER(CsaParams)],
                          C.c_size_t),
    "decode_append": ([C.c_int, C.c_int64, C.c_int32, C.c_int32] + [C.c_void_p] * 17
                      + [C.c_int64, C.POINTER(CsaParams), C.c_void_p, C.c_size_t, C.c_void_p],
                      C.c_int),
}


def lib():
    """Load libcsa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libcsa.so not built at {LIB_PATH}; run "
                              "`python -m long_context_sparse_22_b300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _check(status: int, what: str):
    if status != 0:
        msg = lib().csa_last_error().decode(errors="replace")
        raise CsaError(status, f"{what}: {msg}")


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CSA_BF16
    if t.dtype == torch.float32:
        return CSA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libcsa takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libcsa takes contiguous tensors")
    return t.data_ptr()


def _stream():
    if not torch.cuda.is_available():
        raise RuntimeError("libcsa needs a CUDA device; there is no CPU path")
    return torch.cuda.current_stream().cuda_stream


class Workspace:
    """A caller-owned device workspace; its first bytes hold the status word."""

    def __init__(self, nbytes: int, device=None):
        nbytes = max(int(nbytes), 256)
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
        _check(lib().csa_workspace_init(self.ptr, self.nbytes, _stream()), "workspace init")

    @property
    def ptr(self):
        return self.buf.data_ptr()

    @property
    def nbytes(self):
        return self.buf.numel()

    def status(self):
        """Synchronise the current stream and raise on a device-side error bit."""
        _check(lib().csa_stream_status(self.ptr, _stream()), "device status")


_ws_cache: dict = {}


def _ws(nbytes: int, ws: Workspace | None):
    if ws is not None:
        return ws
    dev = torch.cuda.current_device()
    cur = _ws_cache.get(dev)
    if cur is None or cur.nbytes < nbytes:
        cur = Workspace(nbytes)
        _ws_cache[dev] = cur
    return cur


def wait_probe(spin_limit: int, ws: Workspace):
    """Enqueue the bounded-wait check: a kernel waits on a barrier nothing
    completes for at most spin_limit polls and records a timeout in ws."""
    _check(lib().csa_wait_probe(int(spin_limit), ws.ptr, ws.nbytes, _stream()), "csa_wait_probe")


# ------------------------------------------------------------------ steps

def csa_compress(C_, Z, bias, *, m, overlap=0, Cb=None, Zb=None, biasb=None, rope_dims=0,
                 rope_theta=10000.0, want_raw=False, out=None, raw_out=None, kv_norm=None,
                 norm_eps=0.0):
    """[B, n, c] content and logits -> entries [B, n // m, c] (and the raw rows
    rotated at their positions when want_raw); kv_norm: RMSNorm gains [c]."""
    B, n, c = C_.shape
    p = params(m=m, overlap=overlap, rope_dims=rope_dims, rope_theta=rope_theta, kv_norm=kv_norm,
               norm_eps=norm_eps)
    if out is None:
        out = torch.empty((B, n // m, c), dtype=C_.dtype, device=C_.device)
    if want_raw and raw_out is None:
        raw_out = torch.empty_like(C_)
    _check(lib().csa_compress(_dt(C_), B, n, c, _p(C_), _p(Z), _p(bias), _p(Cb), _p(Zb), _p(biasb),
                              _p(out), _p(raw_out), C.byref(p), _stream()), "csa_compress")
    return (out, raw_out) if want_raw else out


def indexer_score(qI, w, kI, q_pos, m, scores=None, ws=None):
    """qI [B,T,hI,dI], w [B,T,hI] f32, kI [B,E,dI], q_pos [B,T] -> scores [B,T,E] f32."""
    B, T, hI, dI = qI.shape
    E = kI.shape[1]
    if scores is None:
        scores = torch.empty((B, T, E), dtype=torch.float32, device=qI.device)
    ws = _ws(lib().indexer_score_ws_size(), ws)
    _check(lib().indexer_score(_dt(qI), B, T, hI, dI, E, m, _p(qI), _p(w), _p(kI), _p(q_pos),
                               _p(scores), ws.ptr, ws.nbytes, _stream()), "indexer_score")
    return scores


def topk_select(scores, q_pos, m, k, idx=None, cnt=None, ws=None):
    """scores [B,T,E] f32 -> idx [B,T,k] int32 (ascending, -1 padded), cnt [B,T] int32."""
    B, T, E = scores.shape
    if idx is None:
        idx = torch.empty((B, T, k), dtype=torch.int32, device=scores.device)
    if cnt is None:
        cnt = torch.empty((B, T), dtype=torch.int32, device=scores.device)
    ws = _ws(lib().topk_select_ws_size(B, T, E, k), ws)
    _check(lib().topk_select(B, T, E, k, m, _p(scores), _p(q_pos), _p(idx), _p(cnt), ws.ptr,
                             ws.nbytes, _stream()), "topk_select")
    return idx, cnt


def topk_select_noalloc(scores, q_pos, m, k, idx=None, cnt=None):
    """topk_select that takes no workspace (its scratch is a fixed array inside
    the library); for callers that cannot allocate device memory."""
    B, T, E = scores.shape
    if idx is None:
        idx = torch.empty((B, T, k), dtype=torch.int32, device=scores.device)
    if cnt is None:
        cnt = torch.empty((B, T), dtype=torch.int32, device=scores.device)
    _check(lib().topk_select_noalloc(B, T, E, k, m, _p(scores), _p(q_pos), _p(idx), _p(cnt),
                                     _stream()), "topk_select_noalloc")
    return idx, cnt


def _attn_common(q, kvc, p):
    B, T, H, c = q.shape
    E = kvc.shape[1] if kvc is not None else 0
    return B, T, H, c, E


def sparse_attn(q, q_pos, kvc, idx, kv_raw, raw_pos0, sink, p: CsaParams, out=None, lse=None,
                ws=None):
    B, T, H, c, E = _attn_common(q, kvc, p)
    k = idx.shape[-1]
    L = kv_raw.shape[1]
    if out is None:
        out = torch.empty_like(q)
    ws = _ws(lib().attn_ws_size(_dt(q), B, T, H, c, E, k, C.byref(p)), ws)
    _check(lib().sparse_attn(_dt(q), B, T, H, c, E, k, L, _p(q), _p(q_pos), _p(kvc), _p(idx),
                             _p(kv_raw), _p(raw_pos0), _p(sink), _p(out), _p(lse), C.byref(p),
                             ws.ptr, ws.nbytes, _stream()), "sparse_attn")
    return out


def hca_attn(q, q_pos, kvc, kv_raw, raw_pos0, sink, p: CsaParams, out=None, lse=None, ws=None):
    B, T, H, c, E = _attn_common(q, kvc, p)
    L = kv_raw.shape[1]
    if out is None:
        out = torch.empty_like(q)
    ws = _ws(lib().attn_ws_size(_dt(q), B, T, H, c, E, 0, C.byref(p)), ws)
    _check(lib().hca_attn(_dt(q), B, T, H, c, E, L, _p(q), _p(q_pos), _p(kvc), _p(kv_raw),
                          _p(raw_pos0), _p(sink), _p(out), _p(lse), C.byref(p), ws.ptr, ws.nbytes,
                          _stream()), "hca_attn")
    return out


# ------------------------------------------------------------------ fused

def csa_prefill_ws_size(dtype, B, n, H, c, hI, dI, p: CsaParams) -> int:
    return lib().csa_prefill_ws_size(dtype, B, n, H, c, hI, dI, C.byref(p))


def csa_prefill(C_, Z, bias, Ck, Zk, biask, q, qI, w, sink, p: CsaParams, *, Cb=None, Zb=None,
                biasb=None, Ckb=None, Zkb=None, biaskb=None, out=None, idx_out=None, ws=None):
    B, n, c = C_.shape
    H = q.shape[2]
    hI, dI = qI.shape[2], qI.shape[3]
    if out is None:
        out = torch.empty_like(q)
    ws = _ws(csa_prefill_ws_size(_dt(q), B, n, H, c, hI, dI, p), ws)
    _check(lib().csa_prefill(_dt(q), B, n, H, c, hI, dI, _p(C_), _p(Z), _p(bias), _p(Cb), _p(Zb),
                             _p(biasb), _p(Ck), _p(Zk), _p(biask), _p(Ckb), _p(Zkb), _p(biaskb),
                             _p(q), _p(qI), _p(w), _p(sink), _p(out), _p(idx_out), C.byref(p),
                             ws.ptr, ws.nbytes, _stream()), "csa_prefill")
    return out


def hca_prefill_ws_size(dtype, B, n, H, c, p: CsaParams) -> int:
    return lib().hca_prefill_ws_size(dtype, B, n, H, c, C.byref(p))


def hca_prefill(C_, Z, bias, q, sink, p: CsaParams, *, out=None, ws=None):
    B, n, c = C_.shape
    H = q.shape[2]
    if out is None:
        out = torch.empty_like(q)
    ws = _ws(hca_prefill_ws_size(_dt(q), B, n, H, c, p), ws)
    _check(lib().hca_prefill(_dt(q), B, n, H, c, _p(C_), _p(Z), _p(bias), _p(q), _p(sink),
                             _p(out), C.byref(p), ws.ptr, ws.nbytes, _stream()), "hca_prefill")
    return out


def hybrid_decode_ws_size(dtype, B, H, c, hI, dI, E, E2, p: CsaParams, p2: CsaParams) -> int:
    return lib().hybrid_decode_ws_size(dtype, B, H, c, hI, dI, E, E2, C.byref(p), C.byref(p2))


def hybrid_decode(q, qI, w, kvc, kIc, kv_raw, sink, q_pos, raw_pos0, p: CsaParams, *, q2=None,
                  kvc2=None, kv_raw2=None, sink2=None, p2: CsaParams | None = None, out=None,
                  out2=None, idx_out=None, ws=None):
    B, _, H, c = q.shape
    hI, dI = qI.shape[2], qI.shape[3]
    E = kvc.shape[1]
    E2 = kvc2.shape[1] if kvc2 is not None else 0
    L = kv_raw.shape[1]
    p2 = p2 if p2 is not None else p
    if out is None:
        out = torch.empty_like(q)
    if q2 is not None and out2 is None:
        out2 = torch.empty_like(q2)
    ws = _ws(hybrid_decode_ws_size(_dt(q), B, H, c, hI, dI, E, E2, p, p2), ws)
    _check(lib().hybrid_decode(_dt(q), B, H, c, hI, dI, E, E2, L, _p(q), _p(qI), _p(w), _p(kvc),
                               _p(kIc), _p(kv_raw), _p(sink), _p(q2), _p(kvc2), _p(kv_raw2),
                               _p(sink2), _p(q_pos), _p(raw_pos0), _p(out), _p(out2),
                               _p(idx_out), C.byref(p), C.byref(p2), ws.ptr, ws.nbytes,
                               _stream()), "hybrid_decode")
    return (out, out2) if q2 is not None else out


# -------------------------------------------------------- low precision

def quantize_kv_fp8(x, out=None):
    """[..., 512] entries (64 rotary dims) -> [..., KV_FP8_BYTES] uint8 FP8 records."""
    rows = x.numel() // x.shape[-1]
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (KV_FP8_BYTES,), dtype=torch.uint8, device=x.device)
    _check(lib().quantize_kv_fp8(_dt(x), rows, x.shape[-1], 64, _p(x), _p(out), _stream()),
           "quantize_kv_fp8")
    return out


def quantize_index_fp4(x, out=None):
    """[..., 128] rows -> uint8 buffer of index_fp4_bytes(rows): codes, then scale bytes."""
    rows = x.numel() // x.shape[-1]
    if out is None:
        out = torch.empty(lib().index_fp4_bytes(rows), dtype=torch.uint8, device=x.device)
    _check(lib().quantize_index_fp4(_dt(x), rows, x.shape[-1], _p(x), _p(out), _stream()),
           "quantize_index_fp4")
    return out


def indexer_score_fp4(qI, w, kI4, q_pos, E, m, scores=None, ws=None):
    """Decode scores over MXFP4 keys: qI [B,1,64,128] bf16, w [B,1,64], kI4 the
    MXFP4 cache of B*E keys -> scores [B,1,E] (BF16 values; -inf past the
    visible prefix)."""
    B = qI.shape[0]
    if scores is None:
        scores = torch.empty((B, 1, E), dtype=torch.float32, device=qI.device)
    ws = _ws(256, ws)
    _check(lib().indexer_score_fp4(B, E, m, _p(qI), _p(w), _p(kI4), _p(q_pos), _p(scores), ws.ptr,
                                   ws.nbytes, _stream()), "indexer_score_fp4")
    return scores


# ------------------------------------------------- grouped output projection

def out_proj(o, w_g, w_o, heads_per_group=8, y=None, ws=None):
    """o [T, H, c] bf16; w_g [G, d_g, hg*c]; w_o [d, G*d_g] -> y [T, d] bf16."""
    T, H, c = o.shape[0], o.shape[-2], o.shape[-1]
    T = o.numel() // (H * c)
    d_g, d = w_g.shape[1], w_o.shape[0]
    if y is None:
        y = torch.empty((T, d), dtype=torch.bfloat16, device=o.device)
    ws = _ws(lib().out_proj_ws_size(T, H, heads_per_group, d_g), ws)
    _check(lib().out_proj(T, H, c, heads_per_group, d_g, d, _p(o), _p(w_g), _p(w_o), _p(y), ws.ptr,
                          ws.nbytes, _stream()), "out_proj")
    return y


# ------------------------------------------------------- incremental decode

def decode_tail_bytes(dtype, B, c, dI, p: CsaParams) -> int:
    return lib().decode_tail_bytes(dtype, B, c, dI, C.byref(p))


def decode_append(t, C_, Z, bias, win, tail, kvc, p: CsaParams, *, Cb=None, Zb=None, biasb=None,
                  Ck=None, Zk=None, biask=None, Ckb=None, Zkb=None, biaskb=None, kIc=None, ws=None):
    """One new token per sequence at positions t [B] (int64): C, Z [B, c]
    (Ck, Zk [B, dI] for a CSA layer's indexer keys) into the window ring win
    [B, n_win, c] and the tail; a completed block is compressed into kvc
    [B, E_cap, c] (and kIc [B, E_cap, dI])."""
    B, c = C_.shape
    dI = Ck.shape[1] if Ck is not None else 0
    E_cap = kvc.shape[1]
    ws = _ws(256, ws)
    _check(lib().decode_append(_dt(C_), B, c, dI, _p(t), _p(C_), _p(Z), _p(bias), _p(Cb), _p(Zb),
                               _p(biasb), _p(Ck), _p(Zk), _p(biask), _p(Ckb), _p(Zkb), _p(biaskb),
                               _p(win), _p(tail), _p(kvc), _p(kIc), E_cap, C.byref(p), ws.ptr,
                               ws.nbytes, _stream()), "decode_append")


STAGES = ["compress", "indexer", "topk", "sparse_attn", "hca_attn"]


def launch_count() -> int:
    """Kernels launched by libcsa in this process so far."""
    return int(lib().csa_launch_count())


def timing_enable(on: bool = True):
    _check(lib().csa_timing_enable(1 if on else 0), "timing enable")


def timing_read() -> dict:
    """{stage: (total device ms, launches)} since the last read."""
    n = len(STAGES)
    ms = (C.c_double * n)()
    cnt = (C.c_int64 * n)()
    _check(lib().csa_timing_read(ms, cnt, n), "timing read")
    return {STAGES[i]: (ms[i], cnt[i]) for i in range(n)}

