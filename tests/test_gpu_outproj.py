"""GPU parity of the grouped output projection (out_proj, two tcgen05 GEMMs)
against the oracle's definition (oracle/outproj.py), at the Flash shape
(64 heads of 512 in 8 groups, d_g = 1024, d = 4096) and the Pro shape (128
heads in 16 groups, d = 7168), with token counts that leave a ragged last
row tile.  The oracle's weights are in-features-major; the library's are the
out-features-major transpose (a linear layer's layout)."""
import numpy as np
import pytest
import torch

import synth
from oracle import outproj
from parity import check_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import long_context_sparse_22_b300 as m
    m.lib()
    return m


@pytest.mark.parametrize("T,H,c,hg,d_g,d", [
    (300, 64, 512, 8, 1024, 4096),
    (130, 128, 512, 8, 1024, 7168),
    (1, 16, 128, 4, 256, 512),
])
def test_out_proj(csa, T, H, c, hg, d_g, d):
    seed = 800 + T
    G = H // hg
    o = synth.normal(seed, 1, (T, H, c), 1.0, "bf16")
    w_g = synth.normal(seed, 2, (G, d_g, hg * c), (hg * c) ** -0.5, "bf16")     # [G, out, in]
    w_o = synth.normal(seed, 3, (d, G * d_g), (G * d_g) ** -0.5, "bf16")        # [out, in]
    y = csa.out_proj(dev(o), dev(w_g), dev(w_o), heads_per_group=hg)
    ref = outproj.grouped_out_proj(synth.widen(o, "bf16"),
                                   np.transpose(synth.widen(w_g, "bf16"), (0, 2, 1)),
                                   synth.widen(w_o, "bf16").T, heads_per_group=hg)
    check_close(host(y), ref, "bf16", "out_proj")
    # the grouped form against the single block-diagonal matrix it amounts to
    direct = synth.widen(o, "bf16").reshape(T, H * c) @ outproj.direct_weight(
        np.transpose(synth.widen(w_g, "bf16"), (0, 2, 1)), synth.widen(w_o, "bf16").T)
    check_close(host(y), direct, "bf16", "out_proj vs direct")
