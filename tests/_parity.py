"""Helpers for GPU-vs-oracle parity tests.

Tolerance (stated with the block's target): float32 within 1e-5 relative,
float16 / bfloat16 within 2 ulp of T, at every output element. pre_output is a
signed sum over the branches and can cancel, where a per-element relative
bound is ill-posed; an element that misses the plain bound is re-judged
against the same bound at the condition-aware magnitude
max(|pre|, |rho| * sum_c |hn * g|) (hn and g from the oracle's trace), and the
number of such elements is reported. streams_out must match bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from _util import DT_CODE, codes_to_f64, to_codes, ulp_diff

KEYS = ("streams", "norm_scale", "down_w", "up_w", "inject_w", "prev_out", "prev_gate")
SIG_BITS = {"f32": 24, "f16": 11, "bf16": 8}
DT_OF = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def spacing(x, dt):
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 2.0 ** (e - (SIG_BITS[dt] - 1))


def run_oracle(d, C, dt, attrs, rows_idx=None):
    """Oracle on the whole batch, or on the selected rows only (rows are
    independent by construction, so this equals those rows of a full run)."""
    dd = dict(d)
    if rows_idx is not None:
        for k in ("streams", "prev_out", "prev_gate"):
            if dd[k] is not None:
                dd[k] = dd[k][rows_idx]
    return oracle.lowrank_mix(*[to_codes(dd[k]) for k in KEYS], num_branches=C, dtype=DT_CODE[dt],
                              trace=True, **attrs)


def run_gpu(hc, d, C, attrs, flags=0, want_streams_out=True, device="cuda"):
    g = {k: (v.to(device) if v is not None else None) for k, v in d.items()}
    pre, post, sout = hc.lowrank_mix(g["streams"], g["norm_scale"], g["down_w"], g["up_w"], g["inject_w"],
                                     g["prev_out"], g["prev_gate"], num_branches=C, flags=flags,
                                     want_streams_out=want_streams_out, **attrs)
    torch.cuda.synchronize()
    return to_codes(pre), to_codes(post), (to_codes(sout) if sout is not None else None)


def compare(gpu, ref, dt, C, H, R, attrs, check_streams_out=True):
    """Assert parity; return a dict of statistics."""
    gpre, gpost, gsout = gpu
    opre, opost, osout, tr = ref
    rows = opre.shape[0]
    stats = {}
    if check_streams_out and gsout is not None:
        assert np.array_equal(gsout, osout), "streams_out is not bit-identical to the oracle"
    t = oracle.split_trace(tr, C, H, R)
    cond = abs(attrs["reduction_scale"]) * np.abs(
        t["hn"].reshape(rows, C, H).astype(np.float64) * t["g"].reshape(rows, C, H)).sum(1)
    gp, op = codes_to_f64(gpre, dt), codes_to_f64(opre, dt)
    nan_ok = np.isnan(gp) == np.isnan(op)
    assert nan_ok.all(), "NaN pattern of pre_output differs"
    if dt == "f32":
        plain = np.abs(gp - op) <= 1e-5 * np.abs(op)
        aware = np.abs(gp - op) <= 1e-5 * np.maximum(np.abs(op), cond)
    else:
        plain = ulp_diff(gpre, opre, dt) <= 2
        aware = np.abs(gp - op) <= 2 * spacing(np.maximum(np.abs(op), cond), dt)
    ok = plain | aware | np.isnan(op)
    stats["pre_bit_identical"] = float((gpre == opre).mean()) if gpre.size else 1.0
    stats["pre_cond_rescued"] = int((~plain & aware).sum())
    bad = np.argwhere(~ok)
    assert ok.all(), (f"pre_output outside tolerance at {len(bad)} elements, e.g. {bad[:5].tolist()}: "
                      f"gpu {gp[tuple(bad[0])]} oracle {op[tuple(bad[0])]} cond {cond[tuple(bad[0])]}")
    gq, oq = codes_to_f64(gpost, dt), codes_to_f64(opost, dt)
    if dt == "f32":
        okq = np.abs(gq - oq) <= 1e-5 * np.abs(oq)
    else:
        okq = ulp_diff(gpost, opost, dt) <= 2
    assert (okq | (np.isnan(gq) & np.isnan(oq))).all(), f"post_gate outside tolerance: {gq[~okq][:4]} vs {oq[~okq][:4]}"
    stats["post_bit_identical"] = float((gpost == opost).mean()) if gpost.size else 1.0
    return stats
