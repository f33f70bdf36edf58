"""The synchronisation-cost probe (hc_debug_sync_probe) runs every mode to the
end with no bounded poll giving up, and refuses bad arguments on the host."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from hyper_connection_rank_gb300 import _binding as B
    return B.lib()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("ctas", [1, 128])
def test_every_mode_completes(L, mode, ctas):
    scratch = torch.zeros(32 + ctas, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    assert L.hc_debug_sync_probe(mode, ctas, 50, 100 * 1024, scratch.data_ptr(), scratch.numel() * 4,
                                 s.cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(scratch[0].item()) == 0, "a bounded poll gave up"
    if mode == 1:
        assert int(scratch[1].item()) == 50 * ctas      # every CTA added once per round
    if mode == 2:
        assert torch.all(scratch[32:32 + ctas] == 50)   # every CTA published its last round


def test_arguments_checked_on_the_host(L):
    scratch = torch.zeros(64, dtype=torch.int32, device="cuda")
    p, n = scratch.data_ptr(), scratch.numel() * 4
    assert L.hc_debug_sync_probe(3, 8, 1, 0, p, n, None) == 1
    assert L.hc_debug_sync_probe(0, 0, 1, 0, p, n, None) == 1
    assert L.hc_debug_sync_probe(0, 8, 0, 0, p, n, None) == 1
    assert L.hc_debug_sync_probe(0, 64, 1, 0, p, n, None) == 3      # scratch too small for 64 CTAs
    assert L.hc_debug_sync_probe(0, 8, 1, 300 * 1024, p, n, None) == 1
