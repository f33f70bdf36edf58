"""The allocation-free decode entry point, through the C ABI.

Some callers of this library cannot allocate device memory when they run a
block: a host whose memory pool owns the whole GPU, a plug-in interface that
hands over tensors and a stream but no allocator, or code inside a strict
stream capture. hc_lowrank_mix_decode_noalloc serves them by keeping its
scratch in a fixed array inside the library. These tests call it twice in a
row and check both results bit for bit against hc_lowrank_mix (which takes a
workspace from the caller and runs the same kernels in the same order) and
against the CPU oracle within the tolerance of the parity tests, and check
that problems too large for the array are refused with a clear error.
"""
import ctypes

import numpy as np
import pytest
import torch

from _parity import compare, run_oracle
from _util import to_codes
from hyper_connection_rank_gb300 import inputs as I

pytestmark = pytest.mark.gpu

KEYS = ("streams", "norm_scale", "down_w", "up_w", "inject_w", "prev_out", "prev_gate")


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import hyper_connection_rank_gb300 as hc
    from hyper_connection_rank_gb300 import _binding as B
    L = B.load_library()
    f = L.hc_lowrank_mix_decode_noalloc
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.argtypes = [vp] * 7 + [i64, ci, ci, ci, ctypes.POINTER(B.HcAttrs), ci, vp, vp, vp, vp]
    f.restype = ci
    return hc, B, f


def call_noalloc(B, f, g, rows, C, H, R, out, attrs):
    ptr = lambda t: None if t is None else t.data_ptr()
    a = B.make_attrs(**attrs)
    code = B.DTYPE_CODES[g["streams"].dtype]
    return f(*[ptr(g[k]) for k in KEYS], rows, C, H, R, ctypes.byref(a), code, ptr(out[0]), ptr(out[1]), ptr(out[2]),
             torch.cuda.current_stream().cuda_stream)


def test_two_calls_in_a_row_match_the_workspace_entry_point(api):
    hc, B, f = api
    C, H, R = 4, 2560, 320
    cases = [(8, 31), (1, 32)]          # a larger call, then a smaller one over the same scratch
    blocks, outs, hosts = [], [], []
    for rows, seed in cases:
        d = I.make_block(rows, C, H, R, "bf16", seed=seed, prologue=True)
        hosts.append(d)
        g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
        out = (torch.empty(rows, H, dtype=torch.bfloat16, device="cuda"),
               torch.empty(rows, C, dtype=torch.bfloat16, device="cuda"),
               torch.empty(rows, C * H, dtype=torch.bfloat16, device="cuda"))
        blocks.append(g)
        outs.append(out)
    for (rows, _), g, out in zip(cases, blocks, outs):   # back to back, no synchronisation between
        status = call_noalloc(B, f, g, rows, C, H, R, out, I.QWEN_ATTRS)
        assert status == 0, B.lib().hc_last_error().decode()
    torch.cuda.synchronize()
    for (rows, _), g, out, d in zip(cases, blocks, outs, hosts):
        ref = hc.lowrank_mix(*[g[k] for k in KEYS], num_branches=C, **I.QWEN_ATTRS)
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        compare(tuple(to_codes(t) for t in out), run_oracle(d, C, "bf16", I.QWEN_ATTRS), "bf16", C, H, R,
                I.QWEN_ATTRS, inputs=d)


def test_refuses_problems_beyond_the_static_scratch(api):
    hc, B, f = api
    # rows=2, C=8, H=16384, R=512 is a decode-path shape whose partial sums
    # (about 1.06 MB) exceed the 1 MiB array; buffers are real but never read.
    rows, C, H, R = 2, 8, 16384, 512
    t = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    g = dict(streams=t(rows, C * H), norm_scale=t(C * H), down_w=t(C * H, R), up_w=t(R, C * H),
             inject_w=t(C * H, C), prev_out=t(rows, H), prev_gate=t(rows, C))
    out = (t(rows, H), t(rows, C), t(rows, C * H))
    assert call_noalloc(B, f, g, rows, C, H, R, out, I.QWEN_ATTRS) == 2   # HC_ERR_UNSUPPORTED
    assert b"scratch" in B.lib().hc_last_error()
    # more than 16 rows is not a decode-path problem
    rows = 17
    C, H, R = 4, 256, 32
    g = dict(streams=t(rows, C * H), norm_scale=t(C * H), down_w=t(C * H, R), up_w=t(R, C * H),
             inject_w=t(C * H, C), prev_out=t(rows, H), prev_gate=t(rows, C))
    out = (t(rows, H), t(rows, C), t(rows, C * H))
    assert call_noalloc(B, f, g, rows, C, H, R, out, I.QWEN_ATTRS) == 2
    assert b"decode" in B.lib().hc_last_error()
