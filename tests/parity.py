"""Helpers shared by the GPU parity tests: device transfer of the generator's
storage arrays, and the tolerances the CUDA path must meet against the
oracle:

  float32 outputs: max |gpu - oracle| <= 1e-4;
  bf16 outputs:    max |gpu - oracle| <= 2e-2 and
                   ||gpu - oracle||_2 / ||oracle||_2 <= 1e-2;
  top-k sets:      identical wherever the oracle's gap between its k-th and
                   (k+1)-th score exceeds 1e-3 relative; where the gap is
                   smaller either set is accepted and the output is compared
                   against the oracle run on the GPU's set.
"""
from __future__ import annotations

import numpy as np
import torch

import synth

F32_ATOL = 1e-4
BF16_ATOL = 2e-2
BF16_RTOL = 1e-2
TOPK_GAP = 1e-3


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64) if t.is_floating_point() else t.cpu().numpy()


def check_close(gpu: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite GPU output"
    d = np.abs(gpu - ref)
    mx = float(d.max()) if d.size else 0.0
    if dtype == "f32":
        assert mx <= F32_ATOL, f"{what}: max abs err {mx:.3e} > {F32_ATOL}"
    else:
        rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30))
        assert mx <= BF16_ATOL, f"{what}: max abs err {mx:.3e} > {BF16_ATOL}"
        assert rel <= BF16_RTOL, f"{what}: relative err {rel:.3e} > {BF16_RTOL}"
    return mx


def gap_rows(scores: np.ndarray, q_pos: np.ndarray, m: int, k: int) -> np.ndarray:
    """True for rows whose top-k set is fixed to within the gap criterion
    (at most k visible entries, or the k-th/(k+1)-th gap > 1e-3 relative)."""
    T, E = scores.shape
    ok = np.ones(T, bool)
    for t in range(T):
        nv = min(E, (int(q_pos[t]) + 1) // m)
        if nv <= k:
            continue
        row = np.sort(scores[t, :nv])[::-1]
        a, b = row[k - 1], row[k]
        ok[t] = (a - b) > TOPK_GAP * max(abs(a), 1e-30)
    return ok


def compare_topk(gpu_idx: np.ndarray, orc_idx: np.ndarray, scores: np.ndarray, q_pos, m, k):
    """Assert identical sets on rows the gap criterion fixes; return the rows
    where the sets differ (allowed only below the gap)."""
    fixed = gap_rows(scores, q_pos, m, k)
    differ = np.array([not np.array_equal(gpu_idx[t], orc_idx[t]) for t in range(len(orc_idx))])
    bad = np.nonzero(differ & fixed)[0]
    assert bad.size == 0, f"top-k mismatch on {bad.size} rows with a clear gap, e.g. t={bad[:5]}"
    return np.nonzero(differ)[0]


def storage(x: np.ndarray, dtype: str) -> np.ndarray:
    return synth.to_storage(x, dtype)
