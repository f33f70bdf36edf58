"""CPU oracle of the hyper-connection low-rank mix block, the row inverse RMS
and the Engram gate -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The GPU library never uses it.

The arithmetic lives in ``hc_oracle.cpp`` (plain C++17, built with
``-O2 -ffp-contract=off``, no fast-math). This module builds it with g++ on
first use and wraps it with ctypes; it adds no arithmetic of its own.
Definition followed: ONNX Runtime PR #33384 "HyperConnectionLowRankMix",
sections "Schema summary" and "Numerics contract".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hc_oracle.cpp")
_HDR = os.path.join(_HERE, "hc_oracle.h")
_LIB = os.path.join(_HERE, "libhc_oracle.so")

DT_F32, DT_F16, DT_BF16 = 0, 1, 2
_NP_STORAGE = {DT_F32: np.float32, DT_F16: np.uint16, DT_BF16: np.uint16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libhc_oracle.so`` (idempotent)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i64, f32, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
            L.hc_oracle_abi_version.restype = ci
            L.hc_oracle_trace_floats_per_row.argtypes = [ci, ci, ci]
            L.hc_oracle_trace_floats_per_row.restype = i64
            L.hc_oracle_lowrank_mix.argtypes = [vp] * 7 + [i64, ci, ci, ci] + [f32] * 5 + [ci, vp, vp, vp, vp, ci]
            L.hc_oracle_lowrank_mix.restype = ci
            L.hc_oracle_round.argtypes = [f32, ci]
            L.hc_oracle_round.restype = f32
            L.hc_oracle_sigmoid.argtypes = [f32]
            L.hc_oracle_sigmoid.restype = f32
            f64 = ctypes.c_double
            L.hc_oracle_inv_rms.argtypes = [vp, i64, i64, f64, ci, vp]
            L.hc_oracle_inv_rms.restype = ci
            L.hc_oracle_engram_gate.argtypes = [vp] * 5 + [i64, ci, i64, f64, ci, vp, vp]
            L.hc_oracle_engram_gate.restype = ci
            L.hc_oracle_to_float.argtypes = [vp, ci, i64, vp]
            L.hc_oracle_from_float.argtypes = [vp, ci, i64, vp]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _as_storage(a, dtype_code, name):
    want = _NP_STORAGE[dtype_code]
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError(f"{name}: expected storage dtype {np.dtype(want).name}, got {a.dtype}")
    return a


def lowrank_mix(streams, norm_scale, down_w, up_w, inject_w, prev_out=None, prev_gate=None, *,
                num_branches, dtype, epsilon=1e-5, reduction_scale=1.0, silu_alpha=1.0,
                gate_div=1.0, gate_mul=1.0, trace=False, nthreads=0):
    """Run the oracle on host arrays holding T codes (float32, or uint16 codes
    for float16 / bfloat16). Returns ``(pre_output, post_gate, streams_out[, trace])``
    as arrays of the same storage type; ``trace`` is a float32 array of shape
    (rows, trace_floats_per_row) when requested."""
    C = int(num_branches)
    streams = _as_storage(streams, dtype, "streams")
    rows, CH = streams.shape
    if CH % C:
        raise ValueError("streams width is not a multiple of num_branches")
    H = CH // C
    R = down_w.shape[1]
    args = [_as_storage(x, dtype, n) for x, n in ((norm_scale, "norm_scale"), (down_w, "down_w"), (up_w, "up_w"),
                                                 (inject_w, "inject_w"), (prev_out, "prev_out"),
                                                 (prev_gate, "prev_gate"))]
    st = _NP_STORAGE[dtype]
    pre = np.empty((rows, H), st)
    post = np.empty((rows, C), st)
    sout = np.empty((rows, CH), st)
    L = lib()
    tr = None
    if trace:
        tr = np.empty((rows, L.hc_oracle_trace_floats_per_row(C, H, R)), np.float32)
    rc = L.hc_oracle_lowrank_mix(_ptr(streams), *[_ptr(a) for a in args], rows, C, H, R,
                                 epsilon, reduction_scale, silu_alpha, gate_div, gate_mul, dtype,
                                 _ptr(pre), _ptr(post), _ptr(sout), _ptr(tr), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return (pre, post, sout, tr) if trace else (pre, post, sout)


def split_trace(tr, C, H, R):
    """Split a per-row trace into named float32 arrays (rows, n)."""
    CH = C * H
    names = [("S", CH), ("inv", C), ("hn", CH), ("down", R), ("inject", C), ("Z", R), ("SG", R),
             ("hidden", R), ("up", CH), ("g", CH)]
    out, o = {}, 0
    for n, w in names:
        out[n] = tr[:, o:o + w]
        o += w
    return out


def inv_rms(x, *, dtype, epsilon):
    """Row inverse RMS of FreeToken PR #101 ("The problem"): float64 array
    (rows,) of 1/sqrt(mean(x^2) + eps) for x (rows, dim) holding T codes."""
    x = _as_storage(x, dtype, "x")
    rows, dim = x.shape
    out = np.empty(rows, np.float64)
    if lib().hc_oracle_inv_rms(_ptr(x), rows, dim, float(epsilon), dtype, _ptr(out)) != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def engram_gate(key, query, value, key_scale, query_scale, *, dtype, epsilon=1e-5):
    """com.microsoft.EngramGate (its README, "Description"): key, query (rows, M, D),
    value (rows, D), key_scale, query_scale (M, D), all T codes. Returns
    (output (rows, M, D) T codes, gate (rows, M) float64)."""
    key = _as_storage(key, dtype, "key")
    rows, M, D = key.shape
    args = [_as_storage(a, dtype, n) for a, n in ((query, "query"), (value, "value"), (key_scale, "key_scale"),
                                                 (query_scale, "query_scale"))]
    if args[0].shape != key.shape or args[1].shape != (rows, D) or args[2].shape != (M, D) \
            or args[3].shape != (M, D):
        raise ValueError("shape mismatch")
    out = np.empty(key.shape, _NP_STORAGE[dtype])
    gate = np.empty((rows, M), np.float64)
    if lib().hc_oracle_engram_gate(_ptr(key), *[_ptr(a) for a in args], rows, M, D, float(epsilon), dtype,
                                   _ptr(out), _ptr(gate)) != 0:
        raise ValueError("oracle rejected the arguments")
    return out, gate


def round_t(x: float, dtype: int) -> float:
    return lib().hc_oracle_round(float(x), int(dtype))


def sigmoid(x: float) -> float:
    return lib().hc_oracle_sigmoid(float(x))


def to_float(codes, dtype):
    codes = _as_storage(codes, dtype, "codes")
    out = np.empty(codes.shape, np.float32)
    lib().hc_oracle_to_float(_ptr(codes), dtype, codes.size, _ptr(out))
    return out


def from_float(x, dtype):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, _NP_STORAGE[dtype])
    lib().hc_oracle_from_float(_ptr(x), dtype, x.size, _ptr(out))
    return out
