"""topk_select_noalloc: selection for callers that cannot allocate device
memory.

Some callers of this library cannot call cudaMalloc: code that runs where the
allocator is unavailable or forbidden and only receives ready-made input and
output buffers.  topk_select_noalloc serves them by keeping its scratch in a
fixed array inside the library.  These tests call it through the C ABI and
check that it returns exactly what the workspace entry point topk_select
returns (indices are integers, so the comparison is bit-exact), on two calls
in a row, so the second call must not see the first call's leftovers.  The
file is named to be collected last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_sparse_22_b300 as m
    m.lib()
    return m


def _scores(seed, B, T, E):
    g = torch.Generator(device="cpu").manual_seed(seed)
    s = torch.round(torch.randn(B, T, E, generator=g) * 8) / 8      # many exact ties
    return s.cuda()


def _noalloc_via_abi(csa, scores, q_pos, m, k):
    B, T, E = scores.shape
    idx = torch.full((B, T, k), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, T), -7, dtype=torch.int32, device="cuda")
    st = csa.lib().topk_select_noalloc(B, T, E, k, m, C.c_void_p(scores.data_ptr()),
                                       C.c_void_p(q_pos.data_ptr()), C.c_void_p(idx.data_ptr()),
                                       C.c_void_p(cnt.data_ptr()),
                                       C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, csa.lib().csa_last_error()
    return idx, cnt


@pytest.mark.parametrize("B,T,E,k,m", [
    (8, 1, 262144, 1024, 4),     # long rows: the path that uses the fixed scratch
    (32, 1, 32768, 512, 4),
    (1, 300, 512, 64, 4),        # short rows: no scratch needed
])
def test_noalloc_matches_workspace_entry_point(csa, B, T, E, k, m):
    for call, seed in enumerate((11, 12)):           # two calls in a row
        sc = _scores(seed + E, B, T, E)
        if T == 1:
            pos = torch.full((B, 1), E * m - 1, dtype=torch.int64, device="cuda")
            pos[0, 0] = (k - 1) * m + m - 1           # one row with exactly k visible
        else:
            pos = torch.arange(T, dtype=torch.int64, device="cuda").view(1, T) * (E * m // T)
        idx_n, cnt_n = _noalloc_via_abi(csa, sc, pos, m, k)
        idx_w, cnt_w = csa.topk_select(sc, pos, m, k)
        torch.cuda.synchronize()
        assert torch.equal(cnt_n, cnt_w), f"call {call}: counts differ"
        assert torch.equal(idx_n, idx_w), f"call {call}: indices differ"
        # and the selection is a valid top-k: ascending, -1 padded
        i = idx_n.cpu().numpy()
        c = cnt_n.cpu().numpy()
        for b in range(B):
            for t in range(T):
                row = i[b, t, : c[b, t]]
                assert np.all(np.diff(row) > 0) and np.all(i[b, t, c[b, t]:] == -1)


def test_noalloc_rejects_beyond_its_scratch(csa):
    """More than 2^21 row x entry products on the long-row path: refused on
    the host with nothing enqueued."""
    B, T, E = 16, 1, 262144
    st = csa.lib().topk_select_noalloc(B, T, E, 1024, 4, C.c_void_p(1 << 20), C.c_void_p(1 << 20),
                                       C.c_void_p(1 << 20), C.c_void_p(1 << 20), None)
    assert st == 2
    assert b"static scratch" in csa.lib().csa_last_error()
