"""Helpers for GPU-vs-oracle parity tests.

Tolerance (stated with the block's target): float32 within 1e-5 relative,
float16 / bfloat16 within 2 ulp of T, at every output element. Two situations
make a per-element bound on pre_output ill-posed, and elements that miss the
plain bound are re-judged for them, each count reported:
  1. cancellation: pre_output is a signed sum over the branches, so the bound
     is applied at the condition-aware magnitude max(|pre|, |rho| sum_c |hn g|);
  2. intermediate rounding flips: the contract ("Numerics contract") fixes
     where values are rounded to T (down, d, up, hn, g among them) but not the
     order of the fp32 sums before them; any order other than the oracle's
     sequential one (the tensor cores' fp32 accumulation in particular) moves
     an fp32 value that lies next to a rounding midpoint of T to the other
     side, so the rounded value differs by one ulp, and the flip propagates.
     At C = 1 nothing cancels it: a flip of up flips g, and rho * hn * g moves
     by up to 2 ulp more (seen: 3 and 4 ulp). The element then passes if it is
     within 2 ulp of the condition-aware magnitude plus the first-order effect
     of ONE flip at each rounding site of its own chain (its up and g, its
     branches' hn) and of one flip among the d values feeding it, propagated
     with the oracle's values:
       dd   = 2 ulp(d) + (SG + |alpha down| SG (1 - SG)) ulp(down)
       dup  = ulp(up) + max_r dd_r * max_r |W_u[r, n]|
       dg   = ulp(g) + g (1 - g) dup
       dpre = |rho| sum_c (|hn| dg + ulp(hn) |g|).
     Such elements must stay rare and close: at most FLIP_CAP_FRAC of a call's
     elements (at least FLIP_CAP_MIN) and each within FLIP_CAP_ULP ulp; more
     means something other than isolated flips (a wrong site or order).
Every element outside the plain bound is counted per tier with its largest
ulp distance (``compare`` returns them and appends them to HC_PARITY_LOG). For
float16 / bfloat16 at least 85% of pre_output elements must be bit-identical
to the oracle (a missing rounding site or a wrong order shows up as a far lower
figure). streams_out must match bit for bit.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from _util import DT_CODE, codes_to_f64, to_codes, ulp_diff

KEYS = ("streams", "norm_scale", "down_w", "up_w", "inject_w", "prev_out", "prev_gate")
FLIP_CAP_FRAC, FLIP_CAP_MIN, FLIP_CAP_ULP = 1e-4, 2, 6
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


def flip_bound(t, inputs, dt, rows, C, H, R, attrs):
    """First-order bound on |pre - oracle pre| from single one-ulp flips at
    the contract's rounding sites along each element's chain (see the module
    docstring)."""
    u = lambda x: spacing(x, dt)
    down, sg, d = (t[k].astype(np.float64) for k in ("down", "SG", "hidden"))
    up, g, hn = (t[k].astype(np.float64) for k in ("up", "g", "hn"))
    dd = 2 * u(d) + (np.abs(sg) + np.abs(attrs["silu_alpha"] * down) * sg * (1 - sg)) * u(down)
    wu_max = np.abs(inputs["up_w"].to(torch.float64).numpy()).max(0)
    dup = u(up) + dd.max(1, keepdims=True) * wu_max[None, :]
    dg = u(g) + g * (1 - g) * dup
    hn3, g3, dg3 = hn.reshape(rows, C, H), g.reshape(rows, C, H), dg.reshape(rows, C, H)
    return abs(attrs["reduction_scale"]) * (np.abs(hn3) * dg3 + u(hn3) * np.abs(g3)).sum(1)


def compare(gpu, ref, dt, C, H, R, attrs, check_streams_out=True, inputs=None):
    """Assert parity; return a dict of statistics. ``inputs`` (the block's
    input tensors) enables the rounding-flip re-judgement for fp16/bf16."""
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
        flips = aware
    else:
        plain = ulp_diff(gpre, opre, dt) <= 2
        aware = np.abs(gp - op) <= 2 * spacing(np.maximum(np.abs(op), cond), dt)
        flips = aware
        if inputs is not None and not (plain | aware).all():
            flip_mag = flip_bound(t, inputs, dt, rows, C, H, R, attrs)
            flips = np.abs(gp - op) <= 2 * spacing(np.maximum(np.abs(op), cond), dt) + flip_mag
    ok = plain | aware | flips | np.isnan(op)
    ud = ulp_diff(gpre, opre, dt)
    fin = ~np.isnan(op)
    cond_only, flip_only = ~plain & aware & fin, ~plain & ~aware & flips & fin
    stats["elements"] = int(gpre.size)
    stats["pre_bit_identical"] = float((gpre == opre).mean()) if gpre.size else 1.0
    stats["pre_max_ulp"] = int(ud[fin].max()) if fin.any() else 0
    stats["pre_cond_rescued"] = int(cond_only.sum())
    stats["pre_cond_max_ulp"] = int(ud[cond_only].max()) if cond_only.any() else 0
    stats["pre_flip_rescued"] = int(flip_only.sum())
    stats["pre_flip_max_ulp"] = int(ud[flip_only].max()) if flip_only.any() else 0
    gq, oq = codes_to_f64(gpost, dt), codes_to_f64(opost, dt)
    if dt == "f32":
        okq = np.abs(gq - oq) <= 1e-5 * np.abs(oq)
    else:
        okq = ulp_diff(gpost, opost, dt) <= 2
    finq = ~np.isnan(oq)
    stats["post_bit_identical"] = float((gpost == opost).mean()) if gpost.size else 1.0
    stats["post_max_ulp"] = int(ulp_diff(gpost, opost, dt)[finq].max()) if finq.any() else 0
    stats["fail"] = int((~ok).sum())
    log_stats(stats, dt)
    cap = max(FLIP_CAP_MIN, int(FLIP_CAP_FRAC * gpre.size))
    assert stats["pre_flip_rescued"] <= cap, (f"{stats['pre_flip_rescued']} elements need the rounding-flip tier "
                                              f"(cap {cap})")
    assert stats["pre_flip_max_ulp"] <= FLIP_CAP_ULP, f"a flip-tier element is {stats['pre_flip_max_ulp']} ulp off"
    if dt != "f32" and gpre.size >= 1000:
        assert stats["pre_bit_identical"] >= 0.85, f"only {stats['pre_bit_identical']:.3f} of pre_output bit-identical"
    bad = np.argwhere(~ok)
    assert ok.all(), (f"pre_output outside tolerance at {len(bad)} elements, e.g. {bad[:5].tolist()}: "
                      f"gpu {gp[tuple(bad[0])]} oracle {op[tuple(bad[0])]} cond {cond[tuple(bad[0])]}")
    assert (okq | (np.isnan(gq) & np.isnan(oq))).all(), f"post_gate outside tolerance: {gq[~okq][:4]} vs {oq[~okq][:4]}"
    return stats


def log_stats(stats, dt):
    """Append the statistics of one comparison, with the test that made it, to
    the file named by HC_PARITY_LOG (if set): the record of which elements
    needed a tier beyond the plain bound."""
    path = os.environ.get("HC_PARITY_LOG")
    if not path:
        return
    rec = dict(stats, dtype=dt, test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0])
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")
