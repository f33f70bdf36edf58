"""Phase clocks of the decode path's tensor-core kernels (hc_debug_phase_clocks).

The timed variants must compute exactly what the plain kernels compute (they
only add stamps), and every CTA must leave a complete, ordered record: each
point stamped, SM clocks non-decreasing from point to point.
"""
import numpy as np
import pytest
import torch

from _parity import KEYS
from hyper_connection_rank_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import hyper_connection_rank_gb300 as m
    yield m
    m._binding.lib().hc_debug_phase_clocks(None, 0)


@pytest.mark.parametrize("rows", [1, 8])
def test_timed_kernels_same_bits_and_complete_records(hc, rows):
    C, H, R = 4, 2560, 320
    L = hc._binding.lib()
    d = I.make_block(rows, C, H, R, "bf16", seed=51, prologue=True)
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    plain = hc.lowrank_mix(*[g[k] for k in KEYS], num_branches=C, **I.QWEN_ATTRS)
    torch.cuda.synchronize()
    slot = L.hc_debug_phase_clocks(None, 0)
    buf = torch.zeros(2 * slot // 8, dtype=torch.int64, device="cuda")
    assert L.hc_debug_phase_clocks(buf.data_ptr(), 2 * slot) == slot
    try:
        timed = hc.lowrank_mix(*[g[k] for k in KEYS], num_branches=C, **I.QWEN_ATTRS)
        torch.cuda.synchronize()
    finally:
        L.hc_debug_phase_clocks(None, 0)
    for a, b in zip(plain, timed):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    st = buf.view(2, 2, 256, 10, 2).cpu().numpy()
    assert not st[1].any(), "one call wrote more than one slot"
    for k, n, last in ((0, C * H // 80, 9), (1, (H // 128) * C, 7)):
        rec = st[0, k]
        assert (rec[:n, :last + 1, :] != 0).all(), "a point of a CTA was not stamped"
        assert not rec[n:].any() and not rec[:, last + 1:].any(), "stamps outside the grid or the points"
        assert (np.diff(rec[:n, :last + 1, 1].astype(np.int64), axis=1) >= 0).all(), "SM clocks out of order"
