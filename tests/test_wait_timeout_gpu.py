"""The bounded device waits give up cleanly (failure detection without a GPU
fault).

Every wait of the library's kernels on an mbarrier (a copy landing, a peer's
store, an MMA completing) is bounded: after its limit it counts itself, the
kernel writes NaN where its result would go and exits, and the host learns of
it from hc_debug_wait_timeouts. Here one CTA waits on an mbarrier that nothing
arrives on and no copy completes, with a limit of about a millisecond, so the
give-up path runs for real; nothing is in flight when it gives up, and the
context must stay usable (a decode block run afterwards still matches the
oracle).
"""
import pytest
import torch

from _parity import compare, run_gpu, run_oracle
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
    m.debug_wait_timeouts(reset=True)


def test_wait_that_nothing_completes_gives_up_and_reports(hc):
    hc.debug_wait_timeouts(reset=True)
    out = hc.debug_wait_timeout(limit_cycles=2_000_000)
    torch.cuda.synchronize()
    assert torch.isnan(out).all(), "the probe's wait did not give up"
    assert hc.debug_wait_timeouts() == 1
    out = hc.debug_wait_timeout(limit_cycles=4_000_000)
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and hc.debug_wait_timeouts(reset=True) == 2
    # the context is still healthy: a real block runs and matches the oracle,
    # and its own waits do not give up
    C, H, R = 4, 2560, 320
    d = I.make_block(2, C, H, R, "bf16", seed=44, prologue=True)
    compare(run_gpu(hc, d, C, I.QWEN_ATTRS), run_oracle(d, C, "bf16", I.QWEN_ATTRS), "bf16", C, H, R, I.QWEN_ATTRS,
            inputs=d)
    assert hc.debug_wait_timeouts() == 0


def test_limit_is_validated_on_the_host(hc):
    out = torch.zeros(32, device="cuda")
    L = hc._binding.lib()
    assert L.hc_debug_wait_timeout(out.data_ptr(), 10, None) == hc._binding.HC_ERR_INVALID_ARG
    assert L.hc_debug_wait_timeout(None, 2_000_000, None) == hc._binding.HC_ERR_INVALID_ARG
