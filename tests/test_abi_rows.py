"""hc_inv_rms and hc_engram_gate (include/hc_row_ops.h) reject bad arguments on
the host before any launch (CPU only; no compute calls)."""
import ctypes

import pytest

from hyper_connection_rank_gb300 import _binding as B
from hyper_connection_rank_gb300 import build as gpu_build


@pytest.fixture(scope="module")
def L():
    gpu_build.build()
    return B.load_library()


X, OUT = 0x100000, 0x900000


@pytest.mark.parametrize("over", [dict(rows=-1), dict(dim=0), dict(dt=7), dict(x=None), dict(out=None),
                                  dict(out=X + 64)], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_inv_rms_rejects(L, over):
    a = dict(x=X, rows=4, dim=64, dt=B.HC_BF16, out=OUT)
    a.update(over)
    assert L.hc_inv_rms(a["x"], a["rows"], a["dim"], 1e-6, a["dt"], a["out"], None) == B.HC_ERR_INVALID_ARG
    assert len(L.hc_last_error()) > 0


def test_inv_rms_zero_rows_is_ok(L):
    assert L.hc_inv_rms(None, 0, 64, 1e-6, B.HC_BF16, None, None) == B.HC_OK


ENG = dict(key=0x100000, query=0x200000, value=0x300000, ks=0x400000, qs=0x500000, out=0x600000)


@pytest.mark.parametrize("over", [dict(rows=-1), dict(M=0), dict(D=0), dict(dt=9), dict(key=None),
                                  dict(value=None), dict(qs=None), dict(out=None),
                                  dict(out=ENG["query"] + 32), dict(out=ENG["ks"] - 16)],
                         ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_engram_gate_rejects(L, over):
    a = dict(ENG, rows=2, M=4, D=64, dt=B.HC_F16)
    a.update(over)
    rc = L.hc_engram_gate(a["key"], a["query"], a["value"], a["ks"], a["qs"], a["rows"], a["M"], a["D"], 1e-5,
                          a["dt"], a["out"], None)
    assert rc == B.HC_ERR_INVALID_ARG
    assert len(L.hc_last_error()) > 0


def test_engram_gate_zero_rows_is_ok(L):
    assert L.hc_engram_gate(None, None, None, None, None, 0, 4, 64, 1e-5, B.HC_F16, None, None) == B.HC_OK
