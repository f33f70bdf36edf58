"""Test helpers: moving T codes between torch and numpy, and ulp distances.

These helpers carry no arithmetic of the block; they only reinterpret bits.
"""
from __future__ import annotations

import numpy as np
import torch

DT_CODE = {"f32": 0, "f16": 1, "bf16": 2}
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_codes(t):
    """torch tensor in T -> numpy array of codes (float32 or uint16)."""
    if t is None:
        return None
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def from_codes(a, dt: str):
    """numpy codes -> torch tensor in T (CPU)."""
    if dt == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(TORCH_DT[dt])


def codes_to_f64(a, dt: str):
    return from_codes(a, dt).to(torch.float64).numpy()


def ordered(a, dt: str):
    """Map T codes to integers whose difference counts representable steps (ulps)."""
    if dt == "f32":
        i = np.ascontiguousarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)
    i = np.ascontiguousarray(a).view(np.uint16).astype(np.int64)
    mag = i & 0x7FFF
    return np.where(i & 0x8000, -mag, mag)


def ulp_diff(a, b, dt: str):
    return np.abs(ordered(a, dt) - ordered(b, dt))


def is_nan(a, dt: str):
    return np.isnan(codes_to_f64(a, dt))
