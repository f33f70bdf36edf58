"""Seeded synthetic inputs for the hyper-connection low-rank mix block (and the
row inverse RMS and Engram gate workloads).

This module holds no arithmetic of the block itself: it only draws random
tensors. Both the oracle-side tests and the GPU benchmark use it, so that the
two sides see identical input codes.

Generator (counter-based, stateless):
  * splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): output i of stream ``key`` is
    ``mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` with the published finaliser
    ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31``.
  * stream key of a tensor: ``mix(mix(mix(seed) + block) + tensor_id)``.
  * uniform in (0, 1): ``((top 24 bits) + 0.5) / 2**24``.
  * normal: Box-Muller on consecutive pairs, in float64, then cast to float32.
  * every value is drawn in float32 and then rounded to nearest even into T.

Distributions (synthetic, shaped like the Qwen3.8-Flash-Next block: 4 streams
x 2560, rank 320; no trained weights are used or needed):
  streams ~ N(0, 1), prev_block_output ~ N(0, 1), prev_post_gate ~ U(0, 2),
  norm_scale = 1 + 0.1 N(0, 1), down_weight and inject_weight ~ N(0, 1/sqrt(C*H))
  (standard deviation = 1/sqrt(fan-in)), up_weight ~ N(0, 1/sqrt(R)).

All tensors are generated with torch on the requested device (CPU for the
tests; CUDA for the large benchmark weight sets). CPU and CUDA share the
integer stream exactly; the float64 log/cos may differ in the last bit between
devices, which never matters because each side of a comparison uses one device.
"""
from __future__ import annotations

import math

import torch

GOLDEN = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

TENSOR_IDS = {"streams": 1, "prev_out": 2, "prev_gate": 3, "norm_scale": 4,
              "down_w": 5, "up_w": 6, "inject_w": 7,
              # row inverse RMS and Engram gate workloads
              "x": 8, "key": 9, "query": 10, "value": 11, "key_scale": 12, "query_scale": 13}

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# Attribute set of the Qwen-shaped configurations (epsilon, reduction_scale,
# silu_alpha, gate_div, gate_mul) as listed for the operator's Qwen3.8 use.
QWEN_ATTRS = dict(epsilon=1e-6, reduction_scale=0.25, silu_alpha=0.25, gate_div=4.0, gate_mul=2.0)


def _s64(u: int) -> int:
    """Unsigned 64-bit constant as the signed int64 with the same bits."""
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def mix64_int(x: int) -> int:
    """splitmix64 finaliser on a Python int (mod 2**64)."""
    z = (x + GOLDEN) & MASK64
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, block: int, tensor_id: int) -> int:
    return mix64_int((mix64_int((mix64_int(seed) + block) & MASK64) + tensor_id) & MASK64)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bits."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def raw64(key: int, start: int, n: int, device) -> torch.Tensor:
    """Outputs start..start+n-1 of the splitmix64 stream ``key`` as int64 bits."""
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    z = i * _s64(GOLDEN) + _s64(key)            # state after i+1 steps; wraps mod 2**64
    z = (z ^ _lsr(z, 30)) * _s64(M1)
    z = (z ^ _lsr(z, 27)) * _s64(M2)
    return z ^ _lsr(z, 31)


def uniform01(key: int, start: int, n: int, device) -> torch.Tensor:
    top24 = _lsr(raw64(key, start, n, device), 40)
    return (top24.to(torch.float64) + 0.5) * (1.0 / (1 << 24))


def normal(key: int, n: int, device, chunk: int = 1 << 24) -> torch.Tensor:
    """n standard normal draws (float32) from stream ``key``."""
    out = torch.empty(n, dtype=torch.float32, device=device)
    pairs = (n + 1) // 2
    for p0 in range(0, pairs, chunk // 2):
        p1 = min(pairs, p0 + chunk // 2)
        u = uniform01(key, 2 * p0, 2 * (p1 - p0), device).view(-1, 2)
        rad = torch.sqrt(-2.0 * torch.log(u[:, 0]))
        ang = (2.0 * math.pi) * u[:, 1]
        z = torch.stack((rad * torch.cos(ang), rad * torch.sin(ang)), dim=1).reshape(-1)
        lo, hi = 2 * p0, min(n, 2 * p1)
        out[lo:hi] = z[: hi - lo].to(torch.float32)
    return out


def uniform(key: int, n: int, lo: float, hi: float, device) -> torch.Tensor:
    u = uniform01(key, 0, n, device)
    return (lo + (hi - lo) * u).to(torch.float32)


def draw(name: str, shape, dtype: str, seed: int = 0, block: int = 0, device="cpu", C=None, H=None, R=None):
    """One named tensor of the block, drawn per the recipe above, in dtype T."""
    n = 1
    for s in shape:
        n *= int(s)
    key = stream_key(seed, block, TENSOR_IDS[name])
    if name in ("streams", "prev_out", "x", "key", "query", "value"):
        x = normal(key, n, device)
    elif name in ("key_scale", "query_scale"):
        x = 1.0 + 0.1 * normal(key, n, device)
    elif name == "prev_gate":
        x = uniform(key, n, 0.0, 2.0, device)
    elif name == "norm_scale":
        x = 1.0 + 0.1 * normal(key, n, device)
    elif name in ("down_w", "inject_w"):
        x = normal(key, n, device) * (1.0 / math.sqrt(C * H))
    elif name == "up_w":
        x = normal(key, n, device) * (1.0 / math.sqrt(R))
    else:
        raise KeyError(name)
    return x.to(torch.float32).reshape(*shape).to(TORCH_DTYPES[dtype])


def make_weights(C: int, H: int, R: int, dtype: str, seed: int = 0, block: int = 0, device="cpu"):
    CH = C * H
    kw = dict(dtype=dtype, seed=seed, block=block, device=device, C=C, H=H, R=R)
    return dict(norm_scale=draw("norm_scale", (CH,), **kw),
                down_w=draw("down_w", (CH, R), **kw),
                up_w=draw("up_w", (R, CH), **kw),
                inject_w=draw("inject_w", (CH, C), **kw))


def make_activations(rows: int, C: int, H: int, dtype: str, seed: int = 0, block: int = 0,
                     prologue: bool = True, device="cpu"):
    kw = dict(dtype=dtype, seed=seed, block=block, device=device, C=C, H=H)
    out = dict(streams=draw("streams", (rows, C * H), **kw))
    if prologue:
        out["prev_out"] = draw("prev_out", (rows, H), **kw)
        out["prev_gate"] = draw("prev_gate", (rows, C), **kw)
    else:
        out["prev_out"] = None
        out["prev_gate"] = None
    return out


def make_block(rows: int, C: int, H: int, R: int, dtype: str, seed: int = 0, block: int = 0,
               prologue: bool = True, device="cpu"):
    d = make_weights(C, H, R, dtype, seed, block, device)
    d.update(make_activations(rows, C, H, dtype, seed, block, prologue, device))
    return d


def make_inv_rms_input(rows: int, dim: int, dtype: str, seed: int = 0, device="cpu"):
    """Hidden state of the row inverse RMS workload (FreeToken PR #101: rows x
    hc_dim, bf16 in the page's measurements): x ~ N(0, 1)."""
    return draw("x", (rows, dim), dtype, seed=seed, device=device)


def make_engram_inputs(rows: int, M: int, D: int, dtype: str, seed: int = 0, device="cpu"):
    """Engram gate workload (com.microsoft.EngramGate README): key, query
    (rows, M, D) ~ N(0, 1); value (rows, D) ~ N(0, 1); per-stream scales (M, D)
    = 1 + 0.1 N(0, 1). rows = batch * sequence."""
    kw = dict(dtype=dtype, seed=seed, device=device)
    return dict(key=draw("key", (rows, M, D), **kw), query=draw("query", (rows, M, D), **kw),
                value=draw("value", (rows, D), **kw), key_scale=draw("key_scale", (M, D), **kw),
                query_scale=draw("query_scale", (M, D), **kw))
