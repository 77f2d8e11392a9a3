"""Small, self-contained launches of one stage each, sized for an ncu capture
(inputs larger than L2 so DRAM counters mean something, a few GB at most).

    python profile_cases.py CASE [--reps R]

Cases:
  indexer_prefill   indexer_score, 16384 queries x 4096 entries, 64 x 128 (bf16)
  indexer_decode    indexer_score, 8 sequences x 262144 entries, 1 query each (bf16)
  indexer_decode_flash  indexer_score, 32 sequences x 32768 entries, 1 query each (bf16)
  topk_prefill      topk_select over [16384, 4096] fp32 scores, k = 512
  topk_decode       topk_select over [8, 262144] fp32 scores, k = 1024
  compress          csa_compress, n = 65536, c = 512, m = 4 (bf16, with raw rows)
  compress_hca      csa_compress, n = 65536, c = 512, m' = 128 (bf16, with raw rows)
  hca_prefill_c128  hca_attn, 8192 queries, 16 heads x 128, m' = 128 + window
  sparse_attn       sparse_attn, 4096 queries, 64 heads x 512, k = 512 + window
  hca_decode        hca_attn, 8 sequences x 8192 entries, 128 heads x 512
  hca_prefill       hca_attn, 8192 queries over 64 entries (m' = 128) + window, 64 heads x 512
  csa_prefill       csa_prefill, n = 16384, Flash shapes
  sparse_attn_decode  sparse_attn, 8 sequences x 1 query, 128 heads x 512, k = 1024 +
                    window (lists split over CTAs: the split-KV combine runs)
  attn_simt         sparse_attn in fp32, 2048 queries, 4 heads x 64, k = 64 + window
  indexer_simt      indexer_score in fp32, 2048 queries x 512 entries, 4 x 32
  indexer_fp4       indexer_score_fp4, 8 sequences x 262144 MXFP4 keys, 1 query each
  hca_decode_fp8    hca_attn on FP8 entries, 8 sequences x 8192 entries, 128 heads x 512
  out_proj          out_proj, 4096 tokens, 64 heads x 512 in 8 groups -> 1024 -> 4096
  decode_append     decode_append, 64 sequences, c = 512, dI = 128, m = 4 (one step)
  compress_norm     csa_compress with the KV RMSNorm, n = 65536, c = 512, m = 4 (bf16, raw rows)
  quantize          quantize_kv_fp8 of 262144 entries and quantize_index_fp4 of 2097152 keys
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import long_context_sparse_22_b300 as csa  # noqa: E402


def _bf16(*shape, scale=1.0):
    return (torch.randn(*shape, device="cuda") * scale).to(torch.bfloat16)


def case_indexer(T, E, B, m=4):
    qI = _bf16(B, T, 64, 128)
    w = torch.softmax(torch.randn(B, T, 64, device="cuda"), -1)
    kI = _bf16(B, E, 128)
    if T == 1:
        pos = torch.full((B, 1), E * m - 1, dtype=torch.int64, device="cuda")
    else:
        pos = (torch.arange(T, device="cuda") + (E * m - T)).repeat(B, 1)
    scores = torch.empty(B, T, E, device="cuda")
    return lambda: csa.indexer_score(qI, w, kI, pos, m, scores=scores)


def case_indexer_f32(T=2048, E=512, hI=4, dI=32, m=4):
    qI = torch.randn(1, T, hI, dI, device="cuda")
    w = torch.softmax(torch.randn(1, T, hI, device="cuda"), -1)
    kI = torch.randn(1, E, dI, device="cuda")
    pos = torch.arange(T, device="cuda").view(1, T)
    scores = torch.empty(1, T, E, device="cuda")
    return lambda: csa.indexer_score(qI, w, kI, pos, m, scores=scores)


def case_topk(T, E, B, k, m=4):
    sc = torch.randn(B, T, E, device="cuda")
    if T == 1:
        pos = torch.full((B, 1), E * m - 1, dtype=torch.int64, device="cuda")
    else:
        pos = (torch.arange(T, device="cuda") + (E * m - T)).repeat(B, 1)
    idx = torch.empty(B, T, k, dtype=torch.int32, device="cuda")
    cnt = torch.empty(B, T, dtype=torch.int32, device="cuda")
    return lambda: csa.topk_select(sc, pos, m, k, idx=idx, cnt=cnt)


def case_compress(m=4):
    n, c = 65536, 512
    C, Z = _bf16(1, n, c), _bf16(1, n, c)
    bias = torch.randn(m, c, device="cuda") * 0.1
    out = torch.empty(1, n // m, c, device="cuda", dtype=torch.bfloat16)
    raw = torch.empty_like(C)
    return lambda: csa.csa_compress(C, Z, bias, m=m, rope_dims=64, want_raw=True, out=out, raw_out=raw)


def case_sparse_attn():
    T, H, c, E, k, m = 4096, 64, 512, 16384, 512, 4
    q = _bf16(1, T, H, c)
    kvc = _bf16(1, E, c)
    L = E * m
    raw = _bf16(1, L, c)
    pos = (torch.arange(T, device="cuda") + (L - T)).view(1, T)
    idx = torch.sort(torch.stack([torch.randperm(E, device="cuda")[:k] for _ in range(T)]), -1)[0]
    idx = idx.to(torch.int32).view(1, T, k).contiguous()
    rp0 = torch.zeros(1, dtype=torch.int64, device="cuda")
    sink = torch.randn(H, device="cuda")
    out = torch.empty_like(q)
    p = csa.params(m=m, top_k=k, n_win=128, rope_dims=64)
    return lambda: csa.sparse_attn(q, pos, kvc, idx, raw, rp0, sink, p, out=out)


def case_sparse_attn_decode():
    B, H, c, E, k, m = 8, 128, 512, 262144, 1024, 4
    t = E * m - 1
    q = _bf16(B, 1, H, c)
    kvc = _bf16(B, E, c)
    raw = _bf16(B, 128, c)
    pos = torch.full((B, 1), t, dtype=torch.int64, device="cuda")
    rp0 = torch.full((B,), t - 127, dtype=torch.int64, device="cuda")
    idx = torch.sort(torch.stack([torch.randperm(E, device="cuda")[:k] for _ in range(B)]), -1)[0]
    idx = idx.to(torch.int32).view(B, 1, k).contiguous()
    sink = torch.randn(H, device="cuda")
    out = torch.empty_like(q)
    p = csa.params(m=m, top_k=k, n_win=128, rope_dims=64)
    return lambda: csa.sparse_attn(q, pos, kvc, idx, raw, rp0, sink, p, out=out)


def case_attn_simt():
    T, H, c, E, k, m = 2048, 4, 64, 512, 64, 4
    q = torch.randn(1, T, H, c, device="cuda")
    kvc = torch.randn(1, E, c, device="cuda")
    raw = torch.randn(1, T, c, device="cuda")
    pos = torch.arange(T, device="cuda").view(1, T)
    nv = ((pos + 1) // m).clamp(max=E)                   # visible entries per query
    j = torch.arange(E, device="cuda").view(1, 1, E)
    r = torch.where(j < nv.view(1, T, 1), torch.rand(1, T, E, device="cuda"), -1.0)
    top = torch.topk(r, k, -1)                           # invisible entries never win
    sel = torch.sort(torch.where(top.values >= 0, top.indices, E), -1).values
    idx = torch.where(sel == E, -1, sel).to(torch.int32).contiguous()   # ascending, -1 padded
    rp0 = torch.zeros(1, dtype=torch.int64, device="cuda")
    sink = torch.randn(H, device="cuda")
    out = torch.empty_like(q)
    p = csa.params(m=m, top_k=k, n_win=128, rope_dims=32)
    return lambda: csa.sparse_attn(q, pos, kvc, idx, raw, rp0, sink, p, out=out)


def case_indexer_fp4(B=8, E=262144, m=4):
    qI = _bf16(B, 1, 64, 128)
    w = torch.softmax(torch.randn(B, 1, 64, device="cuda"), -1)
    kI4 = csa.quantize_index_fp4(_bf16(B, E, 128))
    pos = torch.full((B, 1), E * m - 1, dtype=torch.int64, device="cuda")
    scores = torch.empty(B, 1, E, device="cuda")
    return lambda: csa.indexer_score_fp4(qI, w, kI4, pos, E, m, scores=scores)


def case_hca_decode_fp8():
    B, H, c, E, m = 8, 128, 512, 8192, 128
    t = E * m
    q = _bf16(B, 1, H, c)
    kv8 = csa.quantize_kv_fp8(_bf16(B, E, c))
    raw = _bf16(B, 128, c)
    pos = torch.full((B, 1), t, dtype=torch.int64, device="cuda")
    rp0 = torch.full((B,), t - 127, dtype=torch.int64, device="cuda")
    sink = torch.randn(H, device="cuda")
    out = torch.empty_like(q)
    p = csa.params(m=m, n_win=128, rope_dims=64, cache_format=1)
    return lambda: csa.hca_attn(q, pos, kv8, raw, rp0, sink, p, out=out)


def case_out_proj(T=4096, H=64, c=512, hg=8, d_g=1024, d=4096):
    G = H // hg
    o = _bf16(T, H, c)
    w_g = _bf16(G, d_g, hg * c, scale=(hg * c) ** -0.5)
    w_o = _bf16(d, G * d_g, scale=(G * d_g) ** -0.5)
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    return lambda: csa.out_proj(o, w_g, w_o, heads_per_group=hg, y=y)


def case_decode_append(B=64, c=512, dI=128, m=4):
    p = csa.params(m=m, n_win=128, rope_dims=64)
    C_, Z = _bf16(B, c), _bf16(B, c)
    Ck, Zk = _bf16(B, dI), _bf16(B, dI)
    bias = torch.randn(m, c, device="cuda") * 0.1
    biask = torch.randn(m, dI, device="cuda") * 0.1
    win = _bf16(B, 128, c)
    tail = torch.zeros(csa.decode_tail_bytes(1, B, c, dI, p), dtype=torch.uint8, device="cuda")
    kvc, kIc = _bf16(B, 4096, c), _bf16(B, 4096, dI)
    t = torch.full((B,), 4 * 1000 + 3, dtype=torch.int64, device="cuda")   # completes block 1000
    return lambda: csa.decode_append(t, C_, Z, bias, win, tail, kvc, p, Ck=Ck, Zk=Zk, biask=biask, kIc=kIc)


def case_compress_norm(m=4):
    n, c = 65536, 512
    C, Z = _bf16(1, n, c), _bf16(1, n, c)
    bias = torch.randn(m, c, device="cuda") * 0.1
    g = 1 + 0.1 * torch.randn(c, device="cuda")
    out = torch.empty(1, n // m, c, device="cuda", dtype=torch.bfloat16)
    raw = torch.empty_like(C)
    return lambda: csa.csa_compress(C, Z, bias, m=m, rope_dims=64, want_raw=True, out=out, raw_out=raw,
                                    kv_norm=g)


def case_quantize():
    kv = _bf16(262144, 512)
    ki = _bf16(2097152, 128)
    kv8 = torch.empty(262144, csa.KV_FP8_BYTES, dtype=torch.uint8, device="cuda")
    ki4 = torch.empty(csa.lib().index_fp4_bytes(2097152), dtype=torch.uint8, device="cuda")

    def run():
        csa.quantize_kv_fp8(kv, out=kv8)
        csa.quantize_index_fp4(ki, out=ki4)
    return run


def case_hca_decode():
    B, H, c, E, m = 8, 128, 512, 8192, 128
    t = E * m
    q = _bf16(B, 1, H, c)
    kvc = _bf16(B, E, c)
    raw = _bf16(B, 128, c)
    pos = torch.full((B, 1), t, dtype=torch.int64, device="cuda")
    rp0 = torch.full((B,), t - 127, dtype=torch.int64, device="cuda")
    sink = torch.randn(H, device="cuda")
    out = torch.empty_like(q)
    p = csa.params(m=m, n_win=128, rope_dims=64)
    return lambda: csa.hca_attn(q, pos, kvc, raw, rp0, sink, p, out=out)


def case_hca_prefill(H=64, c=512, q_norm=False):
    T, m = 8192, 128
    q = _bf16(1, T, H, c)
    E = T // m
    kvc = _bf16(1, E, c)
    raw = _bf16(1, T, c)
    pos = torch.arange(T, device="cuda").view(1, T)
    rp0 = torch.zeros(1, dtype=torch.int64, device="cuda")
    sink = torch.randn(H, device="cuda")
    out = torch.empty_like(q)
    gain = (1 + 0.1 * torch.randn(c, device="cuda")) if q_norm else None
    p = csa.params(m=m, n_win=128, rope_dims=64, q_norm=gain)
    return lambda: csa.hca_attn(q, pos, kvc, raw, rp0, sink, p, out=out)


def case_csa_prefill():
    n, H, c = 16384, 64, 512
    C, Z = _bf16(1, n, c), _bf16(1, n, c)
    Ck, Zk = _bf16(1, n, 128), _bf16(1, n, 128)
    bias = torch.randn(4, c, device="cuda") * 0.1
    biask = torch.randn(4, 128, device="cuda") * 0.1
    q, qI = _bf16(1, n, H, c), _bf16(1, n, 64, 128)
    w = torch.softmax(torch.randn(1, n, 64, device="cuda"), -1)
    sink = torch.randn(H, device="cuda")
    out = torch.empty_like(q)
    p = csa.params(m=4, top_k=512, n_win=128, rope_dims=64)
    return lambda: csa.csa_prefill(C, Z, bias, Ck, Zk, biask, q, qI, w, sink, p, out=out)


CASES = {
    "indexer_prefill": lambda: case_indexer(16384, 4096, 1),
    "indexer_decode": lambda: case_indexer(1, 262144, 8),
    "indexer_decode_flash": lambda: case_indexer(1, 32768, 32),
    "topk_prefill": lambda: case_topk(16384, 4096, 1, 512),
    "topk_decode": lambda: case_topk(1, 262144, 8, 1024),
    "compress": case_compress,
    "compress_hca": lambda: case_compress(128),
    "hca_prefill_c128": lambda: case_hca_prefill(16, 128),
    "sparse_attn": case_sparse_attn,
    "hca_decode": case_hca_decode,
    "hca_prefill": case_hca_prefill,
    "csa_prefill": case_csa_prefill,
    "sparse_attn_decode": case_sparse_attn_decode,
    "attn_simt": case_attn_simt,
    "indexer_simt": case_indexer_f32,
    "indexer_fp4": case_indexer_fp4,
    "hca_decode_fp8": case_hca_decode_fp8,
    "out_proj": case_out_proj,
    "decode_append": case_decode_append,
    "compress_norm": case_compress_norm,
    "quantize": case_quantize,
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    torch.manual_seed(0)
    fn = CASES[args.case]()
    for _ in range(args.reps):
        fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(args.reps):
        fn()
    ev[1].record()
    torch.cuda.synchronize()
    print(f"{args.case}: {ev[0].elapsed_time(ev[1]) / args.reps:.3f} ms per call")


if __name__ == "__main__":
    main()
