"""Pins of the algorithmic-work counting that every roofline fraction uses.

The pages print three per-query counts for one layer ([Book] ch.8 "A Cost
Model for Long Context", sections "Main-attention arithmetic" and "Indexer
arithmetic"); the fixture tests/golden/flop_accounting.json holds them with
their citation.  They are reproduced here through the same counting
functions the bench calls, both directly and through the per-step totals of
the decode workloads (a Pro decode step at 2^20 - 1 reads top-k 1024 + 128
window rows in the CSA layer), so a wrong factor or a dropped window term in
the accounting fails.
"""
import json
import os

import pytest

import synth
from long_context_sparse_22_b300 import accounting

GOLD = os.path.join(os.path.dirname(__file__), "golden", "flop_accounting.json")


def cases():
    with open(GOLD) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", cases(), ids=lambda c: c["name"])
def test_pages_counts(case):
    if case["kind"] == "attn":
        got = accounting.attn_flops_per_query(case["c"], case["E"], case["H"])
    else:
        got = accounting.indexer_flops_per_query(case["dI"], case["hI"], case["entries"])
    if "expected" in case:
        assert got == case["expected"]
    else:
        assert abs(got - case["expected_approx"]) <= case["rel_tol"] * case["expected_approx"]


def test_decode_step_totals_match_pages():
    # Pro CSA layer: top-k 1024 + 128 window rows, 128 heads of dim 512 (~302 M per query)
    s = synth.workloads.spec("hybrid_decode_pro")
    s["E"], s["E2"] = (s["t"] + 1) // s["m"], (s["t"] + 1) // s["m2"]
    w = accounting.decode(s, True)
    per_q = cases()[0]["expected"]
    assert w["csa_attn_flops"] == s["B"] * per_q
    # HCA at the pages' one million tokens: 7,812 visible + 128 window (~2.08 G)
    s2 = dict(s, t=10 ** 6 - 1)
    s2["E"], s2["E2"] = (s2["t"] + 1) // s2["m"], (s2["t"] + 1) // s2["m2"]
    w2 = accounting.decode(s2, True)
    hca = cases()[1]
    assert abs(w2["hca_attn_flops"] / s2["B"] - hca["expected_approx"]) <= hca["rel_tol"] * hca["expected_approx"]
    # indexer at N = 10^6 tokens: 250,000 visible entries, 64 heads x 128 (~4.096 G)
    assert w2["indexer_flops"] / s2["B"] == cases()[2]["expected"]


def test_prefill_sums_brute_force():
    # the closed forms of the prefill totals against direct summation
    for n, m, k, W in [(1000, 4, 64, 128), (4100, 4, 512, 128), (777, 128, 1, 16), (300, 1, 50, 0)]:
        E = n // m
        assert accounting.sum_visible(n, m) == sum(min(E, (t + 1) // m) for t in range(n))
        assert accounting.sum_selected(n, m, k) == sum(min(k, E, (t + 1) // m) for t in range(n))
        assert accounting.sum_window(n, W) == sum(min(W, t + 1) if W else 0 for t in range(n))
