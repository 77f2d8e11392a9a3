"""Throughput of the CSA / HCA layer on one B300, in query-tokens/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic input.
Default workload: the Flash-shaped interleaved CSA + HCA prefill (n = 65536,
64 heads of dim 512, indexer 64 x 128, top-k 512, m = 4 / m' = 128): the
one workload whose step runs every step of the path (compression of both
layers, indexer, top-k, sparse attention, dense HCA attention).
Other workloads: csa_prefill_f32, hca_prefill_bf16, csa_decode_flash,
hybrid_decode_pro.

Under torchrun each rank runs its own replica of the workload (the layer
does not shard for one sequence); value = all ranks' query-tokens / the
slowest rank's time.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload (rank 0 only).

The line also carries `workloads`: every one of the five workloads timed in
the same run (the headline's numbers, then the other four), each with its
per-stage roofline, its SM clocks and the whole step's algorithmic bytes
against HBM (8 TB/s and the measured copy rate).  `--no-all` skips them.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402
from long_context_sparse_22_b300 import accounting  # noqa: E402

METRIC = "CSA/HCA query-tokens/s (decode & prefill), % of HBM/tensor roofline, 1xB300"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# DRAM bytes (read + write) per unit of the stage's work, from one ncu capture
# of the same kernel on a smaller case of the same shape (files in profiles/):
# attention per query token (attn_tc_sparse_attn_4096q.md,
# attn_tc_hca_prefill_8192q.md), decode indexer per visible entry
# (indexer_tc_decode_8x262144.md, and indexer_fp4_decode_8x262144.md on the
# low-precision caches).  Traffic per launch = this x the launch's units.
TRAFFIC_PER_UNIT = {
    ("sparse_attn", "prefill"): (301.270016e6 + 236.418304e6) / 4096,
    ("hca_attn", "prefill"): (545.577728e6 + 491.951872e6) / 8192,
    ("indexer", "decode"): (537.052928e6 + 3.294976e6) / (8 * 262144),
    # the MXFP4 decode indexer (indexer_fp4_decode_8x262144.md)
    ("indexer", "decode_lowp"): (142.865152e6 + 3.076096e6) / (8 * 262144),
}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def samples(self) -> int:
        """Rows nvidia-smi has written so far."""
        if self.proc is None:
            return 0
        try:
            with open(self.file.name) as f:
                return sum(1 for line in f if line.count(",") >= 8)
        except OSError:
            return 0

    def keep_busy(self, step, rows: int, limit_s: float = 5.0):
        """Run untimed steps until `rows` more samples have arrived, so that
        the samples taken right before and after a short timed region are
        taken under the same load."""
        if self.proc is None:
            return
        import torch
        want = self.samples() + rows
        t0 = time.time()
        while self.samples() < want and time.time() - t0 < limit_s:
            for _ in range(4):
                step()
            torch.cuda.synchronize()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ multi-rank

def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (x itself on one process)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, ms_step: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (ms_step / 1e3)


# --------------------------------------------------------------- workloads

# decode workloads on the low-precision caches (FP8 KV records, MXFP4 indexer
# keys, BF16 scores): the same inputs, caches quantised on the device once
LOWP = {"csa_decode_flash_lowp": "csa_decode_flash", "hybrid_decode_pro_lowp": "hybrid_decode_pro"}
ALL_WORKLOADS = sorted(synth.WORKLOADS) + sorted(LOWP)


class Workload:
    """Device buffers and the step of one workload through the public API."""

    def __init__(self, name: str, csa, torch):
        self.name, self.csa, self.torch = name, csa, torch
        self.lowp = name in LOWP
        t0 = time.time()
        self.s, self.x = synth.make_inputs(LOWP.get(name, name))
        self.gen_s = time.time() - t0
        self.kind = self.s["kind"]
        s = self.s
        if self.kind == "hybrid_prefill":
            self.work = accounting.hybrid_prefill(s)
        elif self.kind in ("csa_decode", "hybrid_decode"):
            self.work = accounting.decode(s, self.kind == "hybrid_decode", lowp=self.lowp)
        elif self.kind == "csa_prefill":
            self.work = accounting.csa_layer_prefill(s)
        else:
            self.work = accounting.hca_layer_prefill(s, s["m"])
        self.units = self.work["query_tokens"]
        self.in_keys = [k for k in self.x]
        self.d = {k: self._dev(v) for k, v in self.x.items()}
        self.h2d_bytes = sum(v.nbytes for v in self.x.values())
        p = csa.params
        cf = 1 if self.lowp else 0
        self.p = p(m=s["m"], overlap=s.get("overlap", 0), top_k=s.get("top_k", 1),
                   n_win=s["n_win"], rope_dims=s["rope_dims"], rope_theta=s["theta"], cache_format=cf)
        self.p2 = p(m=s.get("m2", s["m"]), n_win=s["n_win"], rope_dims=s["rope_dims"],
                    rope_theta=s["theta"], cache_format=cf)
        if self.lowp:
            # the stored caches in their low-precision formats (resident state, as in serving)
            self.d["kvc"] = csa.quantize_kv_fp8(self.d["kvc"])
            self.d["kIc"] = csa.quantize_index_fp4(self.d["kIc"])
            if "kvc2" in self.d:
                self.d["kvc2"] = csa.quantize_kv_fp8(self.d["kvc2"])
            torch.cuda.synchronize()
        self._alloc()

    def _dev(self, a):
        t = self.torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
        return t.view(self.torch.bfloat16) if a.dtype == np.uint16 else t

    def _alloc(self):
        csa, d, s = self.csa, self.d, self.s
        T = self.torch
        if self.kind in ("hybrid_prefill", "csa_prefill"):
            B, n, H, c = s["B"], s["n"], s["H"], s["c"]
            dt = 1 if s["dtype"] == "bf16" else 0
            self.out = T.empty_like(d["q"])
            self.ws = csa.Workspace(csa.csa_prefill_ws_size(dt, B, n, H, c, s["hI"], s["dI"], self.p))
            if self.kind == "hybrid_prefill":
                self.out2 = T.empty_like(d["q2"])
                self.ws2 = csa.Workspace(csa.hca_prefill_ws_size(dt, B, n, H, c, self.p2))
        elif self.kind == "hca_prefill":
            B, n, H, c = s["B"], s["n"], s["H"], s["c"]
            self.out = T.empty_like(d["q"])
            self.ws = csa.Workspace(csa.hca_prefill_ws_size(1, B, n, H, c, self.p))
        else:
            B, H, c = s["B"], s["H"], s["c"]
            self.out = T.empty_like(d["q"])
            self.out2 = T.empty_like(d["q2"]) if self.kind == "hybrid_decode" else None
            self.ws = csa.Workspace(csa.hybrid_decode_ws_size(1, B, H, c, s["hI"], s["dI"],
                                                              s["E"], s.get("E2", 0), self.p,
                                                              self.p2))

    def outputs(self):
        return [o for o in (self.out, getattr(self, "out2", None)) if o is not None]

    def step(self, d=None, outs=None):
        csa, d = self.csa, d or self.d
        out, out2 = outs if outs is not None else (self.out, getattr(self, "out2", None))
        if self.kind in ("hybrid_prefill", "csa_prefill"):
            csa.csa_prefill(d["C"], d["Z"], d["bias"], d["Ck"], d["Zk"], d["biask"], d["q"], d["qI"],
                            d["w"], d["sink"], self.p, Cb=d.get("Cb"), Zb=d.get("Zb"),
                            biasb=d.get("biasb"), Ckb=d.get("Ckb"), Zkb=d.get("Zkb"),
                            biaskb=d.get("biaskb"), out=out, ws=self.ws)
            if self.kind == "hybrid_prefill":
                csa.hca_prefill(d["C2"], d["Z2"], d["bias2"], d["q2"], d["sink2"], self.p2,
                                out=out2, ws=self.ws2)
        elif self.kind == "hca_prefill":
            csa.hca_prefill(d["C"], d["Z"], d["bias"], d["q"], d["sink"], self.p, out=out,
                            ws=self.ws)
        else:
            kw = {}
            if self.kind == "hybrid_decode":
                kw = dict(q2=d["q2"], kvc2=d["kvc2"], kv_raw2=d["kv_raw2"], sink2=d["sink2"],
                          p2=self.p2, out2=out2)
            csa.hybrid_decode(d["q"], d["qI"], d["w"], d["kvc"], d["kIc"], d["kv_raw"], d["sink"],
                              d["q_pos"], d["raw_pos0"], self.p, out=out, ws=self.ws, **kw)

    # end-to-end: per step, the step's inputs go host -> device from pinned
    # memory and the outputs come back.  For decode the compressed caches are
    # resident state (as a KV cache is in serving) and stay on the device; the
    # per-step inputs are the query-side tensors and the window rows.  Steps
    # are pipelined as a serving loop would run them: two device sets of the
    # per-step inputs and outputs, the inputs of step i + 1 copied in on one
    # copy stream and the outputs of step i copied out on another while step
    # i + 1 computes; every step still moves all of its bytes.
    def e2e_setup(self):
        T = self.torch
        if self.kind in ("csa_decode", "hybrid_decode"):
            keys = [k for k in self.x if k not in ("kvc", "kIc", "kvc2", "sink", "sink2")]
        else:
            keys = list(self.x)
        self.e2e_keys = keys
        self.h_in = {}
        for k in keys:
            t = self.torch.from_numpy(self.x[k].view(np.int16) if self.x[k].dtype == np.uint16 else self.x[k])
            self.h_in[k] = t.pin_memory()
        self.d_e2e = [dict(self.d), dict(self.d)]
        for k in keys:
            self.d_e2e[1][k] = T.empty_like(self.d[k])
        outs = self.outputs()
        self.o_e2e = [outs, [T.empty_like(o) for o in outs]]
        self.h_out = [T.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        self.e2e_h2d = sum(self.x[k].nbytes for k in keys)
        self.e2e_d2h = sum(o.numel() * o.element_size() for o in outs)
        self.s_in, self.s_out = T.cuda.Stream(), T.cuda.Stream()
        self.ev = {n: [T.cuda.Event(), T.cuda.Event()] for n in ("in", "comp", "out")}
        self.e2e_i = 0

    def e2e_step(self):
        T = self.torch
        b = self.e2e_i & 1
        main = T.cuda.current_stream()
        first = self.e2e_i < 2
        with T.cuda.stream(self.s_in):
            if not first:
                self.s_in.wait_event(self.ev["comp"][b])        # step i - 2 is done reading set b
            for k in self.e2e_keys:
                dst, src = self.d_e2e[b][k], self.h_in[k]
                if dst.dtype == T.bfloat16:
                    dst.view(T.int16).copy_(src, non_blocking=True)
                else:
                    dst.copy_(src, non_blocking=True)
            self.ev["in"][b].record(self.s_in)
        main.wait_event(self.ev["in"][b])
        if not first:
            main.wait_event(self.ev["out"][b])                   # step i - 2's outputs are on the host
        outs = self.o_e2e[b]
        self.step(self.d_e2e[b], (outs[0], outs[1] if len(outs) > 1 else None))
        self.ev["comp"][b].record(main)
        with T.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev["comp"][b])
            for h, o in zip(self.h_out, outs):
                h.copy_(o, non_blocking=True)
            self.ev["out"][b].record(self.s_out)
        self.e2e_i += 1

    def e2e_sync(self):
        self.torch.cuda.synchronize()


# ------------------------------------------------------------- CPU oracle

def oracle_sample(name: str, budget_s: float = 15.0, x=None, s=None):
    """Time the fp64 oracle on a bounded sample of the workload; returns
    (query-tokens/s, threads, description)."""
    import oracle
    oracle.lib()
    if x is None:
        s, x = synth.make_inputs(name)
    kind = s["kind"]
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    if kind in ("csa_decode", "hybrid_decode"):
        t0 = time.time()
        done = 0
        for b in range(s["B"]):
            oracle.csa_decode_seq(s, x, b)
            if kind == "hybrid_decode":
                oracle.hca_decode_seq(s, x, b)
            done += 1
            if time.time() - t0 > budget_s:
                break
        dt = time.time() - t0
        return done / dt, threads, f"{done} of {s['B']} sequences, full decode step each"
    # prefill: full compression of the layer(s), then a sample of query rows
    n = s["n"]
    rng = np.random.default_rng(0)
    csa_l = kind in ("csa_prefill", "hybrid_prefill")
    hca_l = kind in ("hca_prefill", "hybrid_prefill")
    suf = "2" if kind == "hybrid_prefill" else ""
    t0 = time.time()
    prep = oracle.csa_prefill_prepare(s, x, 0) if csa_l else None
    prep2 = oracle.hca_prefill_prepare(s, x, 0, suf) if hca_l else None
    t_comp = time.time() - t0
    S, t_q, batch = 0, 0.0, 8
    while t_q < budget_s and S < n:
        sel = np.sort(rng.integers(0, n, batch))
        t1 = time.time()
        if csa_l:
            oracle.csa_prefill_queries(s, x, prep, 0, sel)
        if hca_l:
            oracle.hca_prefill_queries(s, x, prep2, 0, sel, suf)
        t_q += time.time() - t1
        S += batch
        batch = min(batch * 2, 256)
    total_s = t_comp + (t_q / S) * n
    return n / total_s, threads, (f"full compression of every layer ({t_comp:.1f} s, once per "
                                  f"step) plus {S} uniformly drawn query rows ({t_q:.1f} s), the "
                                  f"per-row time extrapolated to all n={n} rows")


# -------------------------------------------------------------------- arms

def run_reference(args, rank, world):
    if rank != 0:
        return
    # the low-precision decode variants share their inputs with the dtype workloads
    s, x = synth.make_inputs(LOWP.get(args.workload, args.workload))
    vals = []
    for _ in range(args.warmup):
        oracle_sample(s["name"], budget_s=2.0, x=x, s=s)
    desc = threads = None
    for _ in range(args.steps):
        v, threads, desc = oracle_sample(s["name"], budget_s=args.ref_budget, x=x, s=s)
        vals.append(v)
    value = float(statistics.median(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "query-tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * s.get("n", s["B"]) / value if "n" in s else 1e3 * s["B"] / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload},
            "cpu_baseline": {"value": value, "unit": "query-tokens/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "query-tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure(wl, steps, warmup, local, dist, torch):
    """Device time of `steps` steps of a workload (CUDA events on the launching
    stream, barrier and synchronise on both sides) with the SM clocks sampled
    during the timed region; then the library's per-stage times from the same
    number of steps run again with its event hooks on (kept out of the timed
    region, where the extra events would lengthen short decode steps)."""
    csa = wl.csa
    dev_stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    clocks.keep_busy(wl.step, 2)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_launch0 = csa.launch_count()
    ev0.record(dev_stream)
    for _ in range(steps):
        wl.step()
    ev1.record(dev_stream)
    n_launches = csa.launch_count() - n_launch0
    torch.cuda.synchronize()
    barrier()
    clocks.keep_busy(wl.step, 2)
    clk = clocks.stop()
    ms_step = max_over_ranks(ev0.elapsed_time(ev1) / steps, dist, "cuda")
    csa.timing_enable(True)
    csa.timing_read()
    for _ in range(steps):
        wl.step()
    torch.cuda.synchronize()
    csa.timing_enable(False)
    stages = csa.timing_read()
    return {"ms_step": ms_step, "stages": stages, "clocks": clk, "launches": n_launches}


def roofline(wl, stages, steps):
    """The dominant stage against its roofline: achieved = the stage's
    algorithmic FLOPs or bytes per launch / its average launch time."""
    pk, pk_kind = peaks()
    stage_ms = {k: v[0] / max(1, steps) for k, v in stages.items()}
    launches = {k: v[1] for k, v in stages.items()}
    dom = max(stage_ms, key=lambda k: stage_ms[k])
    per_launch_ms = stages[dom][0] / max(1, stages[dom][1])
    launches_per_step = max(1, stages[dom][1] // max(1, steps))
    w = wl.work
    flop_key = {"indexer": "indexer_flops", "sparse_attn": "csa_attn_flops",
                "hca_attn": "hca_attn_flops"}.get(dom)
    byte_key = {"compress": "compress_bytes", "topk": "topk_bytes", "indexer": "indexer_bytes",
                "sparse_attn": "csa_attn_bytes", "hca_attn": "hca_attn_bytes"}.get(dom)
    decode = wl.kind in ("csa_decode", "hybrid_decode")
    if flop_key and not (decode and dom in ("indexer",)):
        bound, unit = "tensor", "TFLOP/s"
        achieved = w.get(flop_key, 0) / launches_per_step / (per_launch_ms / 1e3) / 1e12
        peak = pk["bf16_tflops"]
    else:
        bound, unit = "hbm", "GB/s"
        achieved = w.get(byte_key, 0) / launches_per_step / (per_launch_ms / 1e3) / 1e9
        peak = pk["hbm_gbs"]
    phase = ("decode_lowp" if wl.lowp else "decode") if decode else "prefill"
    # the captures are of the tensor-core kernels (bf16, c = 512)
    tc_path = wl.s["dtype"] == "bf16" and wl.s["c"] == 512
    per_unit = TRAFFIC_PER_UNIT.get((dom, phase)) if tc_path else None
    traffic = None
    if per_unit is not None:
        if decode:
            launch_units = wl.s["B"] * wl.s["E"]                 # visible entries per launch
        else:
            launch_units = wl.s["B"] * wl.s["n"] / launches_per_step   # query tokens per launch
        traffic = per_unit * launch_units
    return {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": pk_kind, "traffic": traffic,
            "traffic_unit": "bytes per launch",
            "stage_ms_per_step": {k: round(v, 4) for k, v in stage_ms.items()},
            "stage_launches": launches}


def step_hbm(wl, ms_step):
    """The whole step's algorithmic bytes against HBM: against the nominal
    8 TB/s and against the measured copy rate."""
    pk, pk_kind = peaks()
    gbs = wl.work["bytes"] / (ms_step / 1e3) / 1e9
    return {"bytes": wl.work["bytes"], "achieved_gbs": gbs, "frac_of_8tbs": gbs / 8000.0,
            "frac_of_measured": gbs / pk["hbm_gbs"], "measured_gbs": pk["hbm_gbs"],
            "peak_source": pk_kind}


def run_ours(args, rank, world, dist):
    import torch

    import long_context_sparse_22_b300 as csa
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    csa.lib()
    wl = Workload(args.workload, csa, torch)
    m = measure(wl, args.steps, args.warmup, local, dist, torch)
    ms_step = m["ms_step"]
    value = job_value(wl.units, world, ms_step)

    # end to end through the public API with host buffers
    def barrier():
        if dist is not None:
            dist.barrier()

    wl.e2e_setup()
    wl.e2e_step()
    torch.cuda.synchronize()
    k_e2e = max(1, min(args.steps, 8))
    barrier()
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        wl.e2e_step()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / k_e2e, dist, "cuda")
    e2e_value = job_value(wl.units, world, e2e_ms)
    roof = roofline(wl, m["stages"], args.steps)

    line = {"metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.s["dtype"], "data": "synthetic",
            "config": {"workload": args.workload, "global_batch": world * wl.s["B"],
                       "seq_len": wl.s.get("n", wl.s.get("t")),
                       "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (126 MB) each step, no flush needed"},
            "gpu_launches": int(m["launches"]),
            "e2e": {"value": e2e_value, "unit": "query-tokens/s", "h2d_bytes_per_step": wl.e2e_h2d,
                    "d2h_bytes_per_step": wl.e2e_d2h, "ms_per_step": e2e_ms},
            "roofline": roof, "clocks": m["clocks"]}
    if rank == 0 and world == 1 and not args.no_cpu:
        v, thr, desc = oracle_sample(wl.s["name"], budget_s=args.ref_budget, x=wl.x, s=wl.s)
        line["cpu_baseline"] = {"value": v, "unit": "query-tokens/s", "cores": thr, "kind": "oracle",
                                "sample": desc}

    # every workload in the same run, each with its own clocks: the headline's
    # numbers again, then the other four (decode included)
    if not args.no_all:
        allw = {args.workload: {"ms_per_step": ms_step, "value": value, "roofline": roof,
                                "clocks": m["clocks"], "steps": args.steps,
                                "step_hbm": step_hbm(wl, ms_step)}}
        del wl
        torch.cuda.empty_cache()
        for name in ALL_WORKLOADS:
            if name == args.workload:
                continue
            w2 = Workload(name, csa, torch)
            k2 = args.all_steps if w2.kind in ("csa_decode", "hybrid_decode") else max(3, min(args.steps, 10))
            m2 = measure(w2, k2, args.warmup, local, dist, torch)
            allw[name] = {"ms_per_step": m2["ms_step"],
                          "value": job_value(w2.units, world, m2["ms_step"]),
                          "roofline": roofline(w2, m2["stages"], k2), "clocks": m2["clocks"],
                          "steps": k2, "dtype": w2.s["dtype"],
                          "step_hbm": step_hbm(w2, m2["ms_step"])}
            del w2
            torch.cuda.empty_cache()
        line["workloads"] = allw
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="hybrid_prefill_flash", choices=ALL_WORKLOADS)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-all", action="store_true", help="time only the selected workload")
    ap.add_argument("--all-steps", type=int, default=200,
                    help="timed steps of each decode workload in the all-workloads record")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
