"""ctypes binding of the C ABI in include/hc_lowrank_mix.h.

Argument marshalling only: every step of the block runs in the CUDA kernels
of libhc_lowrank_mix.so. PyTorch provides device memory and the current
stream. There is no CPU fallback: if the library is missing or the device is
not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhc_lowrank_mix.so")

HC_OK, HC_ERR_INVALID_ARG, HC_ERR_UNSUPPORTED, HC_ERR_WORKSPACE, HC_ERR_CUDA = range(5)
HC_F32, HC_F16, HC_BF16 = 0, 1, 2
HC_FLAG_WEIGHTS_STATIC = 1
HC_FLAG_FORCE_GENERAL = 2
HC_PATH_NONE, HC_PATH_DECODE, HC_PATH_PREFILL, HC_PATH_GENERAL = 0, 1, 2, 3
PATH_NAMES = {0: "none", 1: "decode", 2: "prefill", 3: "general"}

DTYPE_CODES = {torch.float32: HC_F32, torch.float16: HC_F16, torch.bfloat16: HC_BF16}

# Every symbol include/hc_lowrank_mix.h declares.
EXPORTS = ("hc_attrs_default", "hc_lowrank_mix_path", "hc_lowrank_mix_workspace_size", "hc_lowrank_mix",
           "hc_status_string", "hc_last_error", "hc_debug_wait_timeouts", "hc_debug_sigmoid_exact",
           "hc_debug_sigmoid_table", "hc_debug_sigmoid_table_f16", "hc_debug_sigmoid_table_f16_bytes", "hc_debug_wait_timeout", "hc_debug_phase_clocks", "hc_debug_sync_probe", "hc_lowrank_mix_decode_noalloc", "hc_inv_rms",
           "hc_engram_gate")


class HcAttrs(ctypes.Structure):
    _fields_ = [("epsilon", ctypes.c_float), ("reduction_scale", ctypes.c_float), ("silu_alpha", ctypes.c_float),
                ("gate_div", ctypes.c_float), ("gate_mul", ctypes.c_float), ("flags", ctypes.c_uint32)]


class HcError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load the GPU library (no build). Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"GPU library {path} is not built; run hyper_connection_rank_gb300.build.build()")
        L = ctypes.CDLL(path)
        vp, i64, ci, u32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t
        L.hc_attrs_default.restype = HcAttrs
        L.hc_lowrank_mix_path.argtypes = [i64, ci, ci, ci, ci, u32]
        L.hc_lowrank_mix_path.restype = ci
        L.hc_lowrank_mix_workspace_size.argtypes = [i64, ci, ci, ci, ci, u32]
        L.hc_lowrank_mix_workspace_size.restype = sz
        L.hc_lowrank_mix.argtypes = [vp] * 7 + [i64, ci, ci, ci, ctypes.POINTER(HcAttrs), ci, vp, vp, vp, vp, sz, vp]
        L.hc_lowrank_mix.restype = ci
        L.hc_status_string.argtypes = [ci]
        L.hc_status_string.restype = ctypes.c_char_p
        L.hc_last_error.restype = ctypes.c_char_p
        L.hc_debug_wait_timeouts.argtypes = [ci]
        L.hc_debug_wait_timeouts.restype = ctypes.c_uint
        L.hc_debug_sigmoid_exact.argtypes = [ci, vp, vp, vp]
        L.hc_debug_sigmoid_exact.restype = ci
        L.hc_debug_sigmoid_table.argtypes = [vp, vp]
        L.hc_debug_sigmoid_table.restype = ci
        L.hc_debug_sigmoid_table_f16_bytes.restype = sz
        L.hc_debug_sigmoid_table_f16.argtypes = [vp, vp, sz, vp]
        L.hc_debug_sigmoid_table_f16.restype = ci
        L.hc_debug_wait_timeout.argtypes = [vp, ctypes.c_longlong, vp]
        L.hc_debug_wait_timeout.restype = ci
        L.hc_debug_phase_clocks.argtypes = [vp, sz]
        L.hc_debug_phase_clocks.restype = sz
        L.hc_debug_sync_probe.argtypes = [ci, ci, ci, sz, vp, sz, vp]
        L.hc_debug_sync_probe.restype = ci
        f32 = ctypes.c_float
        L.hc_inv_rms.argtypes = [vp, i64, i64, f32, ci, vp, vp]
        L.hc_inv_rms.restype = ci
        L.hc_engram_gate.argtypes = [vp] * 5 + [i64, ci, i64, f32, ci, vp, vp]
        L.hc_engram_gate.restype = ci
        _lib = L
        return L


def lib():
    return _lib if _lib is not None else load_library()


def attrs_default() -> HcAttrs:
    return lib().hc_attrs_default()


def make_attrs(epsilon=1e-5, reduction_scale=1.0, silu_alpha=1.0, gate_div=1.0, gate_mul=1.0, flags=0) -> HcAttrs:
    return HcAttrs(epsilon, reduction_scale, silu_alpha, gate_div, gate_mul, flags)


def path(rows: int, C: int, H: int, R: int, dtype: torch.dtype, flags: int = 0) -> int:
    return lib().hc_lowrank_mix_path(rows, C, H, R, DTYPE_CODES[dtype], flags)


def workspace_size(rows: int, C: int, H: int, R: int, dtype: torch.dtype, flags: int = 0) -> int:
    return lib().hc_lowrank_mix_workspace_size(rows, C, H, R, DTYPE_CODES[dtype], flags)


def check(status: int):
    if status != HC_OK:
        L = lib()
        raise HcError(status, f"{L.hc_status_string(status).decode()}: {L.hc_last_error().decode()}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def raw_call(streams, norm_scale, down_w, up_w, inject_w, prev_out, prev_gate, rows, C, H, R, attrs: HcAttrs,
             dtype_code, pre_output, post_gate, streams_out, workspace, workspace_bytes, stream) -> int:
    """The C call with raw device addresses (ints or None); returns the status."""
    return lib().hc_lowrank_mix(streams, norm_scale, down_w, up_w, inject_w, prev_out, prev_gate, rows, C, H, R,
                                ctypes.byref(attrs), dtype_code, pre_output, post_gate, streams_out, workspace,
                                workspace_bytes, stream)


def lowrank_mix(streams, norm_scale, down_w, up_w, inject_w, prev_out=None, prev_gate=None, *, num_branches,
                epsilon=1e-5, reduction_scale=1.0, silu_alpha=1.0, gate_div=1.0, gate_mul=1.0, flags=0,
                want_streams_out=True, out=None, workspace=None, stream=None):
    """One hyper-connection low-rank mix block on the GPU.

    streams (..., C*H), norm_scale (C*H), down_w (C*H, R), up_w (R, C*H),
    inject_w (C*H, C), optional prev_out (..., H) and prev_gate (..., C); all
    CUDA tensors of one dtype. Returns (pre_output (..., H), post_gate (..., C),
    streams_out (..., C*H) or None). ``out`` may supply the three output
    tensors; ``workspace`` a uint8 CUDA tensor of at least workspace_size()
    bytes (allocated here when omitted).
    """
    C = int(num_branches)
    if streams.shape[-1] % C:
        raise ValueError("streams width is not a multiple of num_branches")
    lead = streams.shape[:-1]
    CH = streams.shape[-1]
    H = CH // C
    R = down_w.shape[-1]
    rows = 1
    for s in lead:
        rows *= int(s)
    dt = streams.dtype
    if dt not in DTYPE_CODES:
        raise TypeError(f"unsupported dtype {dt}")
    tensors = dict(streams=streams, norm_scale=norm_scale, down_w=down_w, up_w=up_w, inject_w=inject_w,
                   prev_out=prev_out, prev_gate=prev_gate)
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor of dtype {dt}")
    if tuple(down_w.shape) != (CH, R) or tuple(up_w.shape) != (R, CH) or tuple(inject_w.shape) != (CH, C) \
            or norm_scale.numel() != CH:
        raise ValueError("weight shapes do not match streams / num_branches")
    if out is None:
        pre = torch.empty(*lead, H, dtype=dt, device=streams.device)
        post = torch.empty(*lead, C, dtype=dt, device=streams.device)
        sout = torch.empty_like(streams) if want_streams_out else None
    else:
        pre, post, sout = out
    if workspace is None:  # (a caller's workspace is checked against the requirement by the library)
        need = workspace_size(rows, C, H, R, dt, flags)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=streams.device)
    attrs = make_attrs(epsilon, reduction_scale, silu_alpha, gate_div, gate_mul, flags)
    s = torch.cuda.current_stream(streams.device) if stream is None else stream
    status = raw_call(_ptr(streams), _ptr(norm_scale), _ptr(down_w), _ptr(up_w), _ptr(inject_w), _ptr(prev_out),
                      _ptr(prev_gate), rows, C, H, R, attrs, DTYPE_CODES[dt], _ptr(pre), _ptr(post), _ptr(sout),
                      _ptr(workspace), workspace.numel(), s.cuda_stream)
    check(status)
    return pre, post, sout


def debug_wait_timeouts(reset: bool = False) -> int:
    return lib().hc_debug_wait_timeouts(1 if reset else 0)


def debug_wait_timeout(limit_cycles: int = 2_000_000, device="cuda"):
    """Run the bounded-wait give-up check (hc_debug_wait_timeout): returns the
    32 floats the probe kernel wrote (NaN where its wait gave up)."""
    out = torch.zeros(32, dtype=torch.float32, device=device)
    s = torch.cuda.current_stream(out.device)
    check(lib().hc_debug_wait_timeout(_ptr(out), int(limit_cycles), s.cuda_stream))
    return out


def debug_sigmoid_exact(dt: torch.dtype, device="cuda"):
    """(fast, accurate) T codes of rT(sigmoid(x)) for all 65536 codes x of dt
    (float16 or bfloat16), as int16 tensors on `device` (see
    hc_debug_sigmoid_exact)."""
    fast = torch.empty(65536, dtype=torch.int16, device=device)
    acc = torch.empty(65536, dtype=torch.int16, device=device)
    s = torch.cuda.current_stream(fast.device)
    check(lib().hc_debug_sigmoid_exact(DTYPE_CODES[dt], _ptr(fast), _ptr(acc), s.cuda_stream))
    return fast, acc


def debug_sigmoid_table_f16(device="cuda"):
    """g for every fp16 code through the fp16 prefill epilogue's table lookup,
    as a float32 tensor on `device` (see hc_debug_sigmoid_table_f16)."""
    L = lib()
    g = torch.empty(65536, dtype=torch.float32, device=device)
    n = L.hc_debug_sigmoid_table_f16_bytes()
    table = torch.empty(n, dtype=torch.uint8, device=device)
    s = torch.cuda.current_stream(g.device)
    check(L.hc_debug_sigmoid_table_f16(_ptr(g), _ptr(table), n, s.cuda_stream))
    return g


def debug_sigmoid_table(device="cuda"):
    """g for all 65536 bf16 codes of up as the bf16 prefill epilogue forms it,
    as a float32 tensor on `device` (see hc_debug_sigmoid_table)."""
    g = torch.empty(65536, dtype=torch.float32, device=device)
    s = torch.cuda.current_stream(g.device)
    check(lib().hc_debug_sigmoid_table(_ptr(g), s.cuda_stream))
    return g


def _check_cuda(name, t, dt):
    if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of dtype {dt}")


def inv_rms(x, epsilon=1e-6, *, out=None, stream=None):
    """Row inverse RMS (hc_inv_rms): 1/sqrt(mean(x^2, -1) + epsilon) as float32,
    shape x.shape[:-1]. x: contiguous CUDA tensor (float32, float16 or bfloat16)."""
    dt = x.dtype
    if dt not in DTYPE_CODES:
        raise TypeError(f"unsupported dtype {dt}")
    _check_cuda("x", x, dt)
    dim = x.shape[-1]
    rows = x.numel() // max(dim, 1)
    if out is None:
        out = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    s = torch.cuda.current_stream(x.device) if stream is None else stream
    check(lib().hc_inv_rms(_ptr(x), rows, dim, float(epsilon), DTYPE_CODES[dt], _ptr(out), s.cuda_stream))
    return out


def engram_gate(key, query, value, key_norm_scale, query_norm_scale, epsilon=1e-5, *, out=None, stream=None):
    """com.microsoft.EngramGate (hc_engram_gate). key, query: (B, S, M, D);
    value: (B, S, D); scales: (M, D); all one dtype on the GPU. Returns the gated
    value (B, S, M, D)."""
    dt = key.dtype
    if dt not in DTYPE_CODES:
        raise TypeError(f"unsupported dtype {dt}")
    for n, t in (("key", key), ("query", query), ("value", value), ("key_norm_scale", key_norm_scale),
                 ("query_norm_scale", query_norm_scale)):
        _check_cuda(n, t, dt)
    if key.dim() < 2 or query.shape != key.shape:
        raise ValueError("query must have the shape of key (..., M, D)")
    M, D = key.shape[-2], key.shape[-1]
    rows = key.numel() // max(M * D, 1)
    if tuple(value.shape) != tuple(key.shape[:-2]) + (D,) or tuple(key_norm_scale.shape) != (M, D) \
            or tuple(query_norm_scale.shape) != (M, D):
        raise ValueError("value must be (..., D) and the scales (M, D)")
    if out is None:
        out = torch.empty_like(key)
    s = torch.cuda.current_stream(key.device) if stream is None else stream
    check(lib().hc_engram_gate(_ptr(key), _ptr(query), _ptr(value), _ptr(key_norm_scale), _ptr(query_norm_scale),
                               rows, M, D, float(epsilon), DTYPE_CODES[dt], _ptr(out), s.cuda_stream))
    return out
