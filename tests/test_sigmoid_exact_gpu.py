"""The fast rounded sigmoid of the fp16/bf16 kernels, checked on every input.

Where the numerics contract (ONNX Runtime PR #33384, "HyperConnectionLowRankMix",
section "Numerics contract") rounds sigmoid(z) to T and z is itself a value of
T (the ScaledSiLU gate SG = rT(sigmoid(Z)) with Z = rT(alpha x), and
g = rT(sigmoid(rT(up)))), the kernels evaluate a fast sigmoid that must give
the same T value as the accurate 1 / (1 + expf(-z)). A 16-bit type has 65536
codes, so the claim is checked exhaustively: the library evaluates both forms
on every code (hc_debug_sigmoid_exact) and they must agree bit for bit. The
accurate form is also compared with the oracle's own sigmoid (host libm expf),
which may differ from CUDA's expf by an ulp of fp32 and so, very rarely, round
to a neighbouring value of T.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DT = {"bf16": (torch.bfloat16, 2), "f16": (torch.float16, 1)}


@pytest.fixture(scope="module")
def hc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import hyper_connection_rank_gb300 as m
    return m


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_fast_sigmoid_equals_accurate_on_every_code(hc, dt):
    tdt, code = DT[dt]
    fast, acc = hc.debug_sigmoid_exact(tdt)
    torch.cuda.synchronize()
    f = fast.cpu().numpy().view(np.uint16)
    a = acc.cpu().numpy().view(np.uint16)
    bad = np.nonzero(f != a)[0]
    assert bad.size == 0, f"{bad.size} codes differ, e.g. input codes {bad[:8].tolist()}"


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_accurate_sigmoid_matches_oracle_rounding(hc, dt):
    tdt, code = DT[dt]
    _, acc = hc.debug_sigmoid_exact(tdt)
    torch.cuda.synchronize()
    a = acc.cpu().numpy().view(np.uint16)
    xs = oracle.to_float(np.arange(65536, dtype=np.uint16), code)
    ref = oracle.from_float(np.array([oracle.sigmoid(float(x)) for x in xs], np.float32), code).view(np.uint16)
    finite = np.isfinite(xs)
    mism = np.count_nonzero((a != ref) & finite)
    assert mism <= 16, f"{mism} finite codes round differently from the oracle's sigmoid"
    # NaN inputs give NaN
    nan_out = oracle.to_float(a[~finite & np.isnan(xs)], code)
    assert np.isnan(nan_out).all()


def test_prefill_table_gate_equals_accurate_on_every_code(hc):
    """The bf16 prefill epilogue's gate (table, packed clamps, mixed-precision
    multiply-add) on every bf16 code of up against the accurate rounded
    sigmoid evaluated by the library, code for code; NaN gives NaN."""
    g = hc.debug_sigmoid_table()
    _, acc = hc.debug_sigmoid_exact(torch.bfloat16)
    torch.cuda.synchronize()
    g = g.cpu().numpy()
    a = acc.cpu().numpy().view(np.uint16)
    xs = oracle.to_float(np.arange(65536, dtype=np.uint16), 2)
    nan_in = np.isnan(xs)
    assert np.isnan(g[nan_in]).all()
    # g is a bf16 value carried in fp32: its top half is the bf16 code
    gb = (g[~nan_in].view(np.uint32) >> 16).astype(np.uint16)
    low = g[~nan_in].view(np.uint32) & 0xFFFF
    assert not low.any(), "gate is not a bf16 value"
    bad = np.nonzero(gb != a[~nan_in])[0]
    assert bad.size == 0, f"{bad.size} codes differ, e.g. {np.arange(65536)[~nan_in][bad[:8]].tolist()}"


def test_prefill_fp16_table_gate_equals_accurate_on_every_code(hc):
    """The fp16 prefill epilogue's gate (the table built per call, packed
    clamps, mixed-precision multiply-add) on every fp16 code of up against
    the accurate rounded sigmoid evaluated by the library, code for code;
    NaN gives NaN."""
    g = hc.debug_sigmoid_table_f16()
    _, acc = hc.debug_sigmoid_exact(torch.float16)
    torch.cuda.synchronize()
    g = g.cpu().numpy()
    a = acc.cpu().numpy().view(np.uint16)
    xs = oracle.to_float(np.arange(65536, dtype=np.uint16), 1)
    nan_in = np.isnan(xs)
    assert np.isnan(g[nan_in]).all()
    # g is an fp16 value carried in fp32: converting it to fp16 is exact
    gh = g[~nan_in].astype(np.float16)
    assert np.array_equal(gh.astype(np.float32), g[~nan_in]), "gate is not an fp16 value"
    bad = np.nonzero(gh.view(np.uint16) != a[~nan_in])[0]
    assert bad.size == 0, f"{bad.size} codes differ, e.g. {np.arange(65536)[~nan_in][bad[:8]].tolist()}"
