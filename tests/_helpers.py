"""Shared test helpers: golden fixtures, ulp distances, tensor conversion.

Nothing here computes a norm or a clip; the oracle and the library do that.
"""
from __future__ import annotations

import os

import numpy as np
import torch

from oracle import OracleTensor

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    """Parse a `key = numbers...` fixture; `#` lines are the citation."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals = [float(x) for x in v.split()]
            out[k] = vals if len(vals) > 1 else vals[0]
    return out


def to_oracle(t: torch.Tensor) -> OracleTensor:
    """Host copy of a torch tensor as oracle storage (bit-exact)."""
    t = t.detach().contiguous().cpu().reshape(-1)
    if t.dtype == torch.float32:
        return OracleTensor(t.numpy().copy(), "f32")
    if t.dtype == torch.float16:
        return OracleTensor(t.numpy().copy(), "f16")
    if t.dtype == torch.bfloat16:
        return OracleTensor(t.view(torch.int16).numpy().view(np.uint16).copy(), "bf16")
    raise TypeError(t.dtype)


def storage_bits(t: OracleTensor) -> np.ndarray:
    """Raw bit patterns as signed integers of the storage width."""
    if t.dtype == "f32":
        return t.data.view(np.int32).astype(np.int64)
    return t.data.view(np.int16).astype(np.int64)


def ordered(bits: np.ndarray, width: int) -> np.ndarray:
    """Map IEEE bit patterns to integers whose order is the numeric order, so
    that the difference of two values is their distance in ulps."""
    sign_bit = 1 << (width - 1)
    u = bits & ((1 << width) - 1)
    neg = (u & sign_bit) != 0
    return np.where(neg, -(u & (sign_bit - 1)), u)


def ulp_distance(a: OracleTensor, b: OracleTensor) -> np.ndarray:
    assert a.dtype == b.dtype and a.data.size == b.data.size
    width = 32 if a.dtype == "f32" else 16
    return np.abs(ordered(storage_bits(a), width) - ordered(storage_bits(b), width))


def as_float64(t: OracleTensor) -> np.ndarray:
    if t.dtype == "f32":
        return t.data.astype(np.float64)
    if t.dtype == "f16":
        return t.data.astype(np.float64)
    return (t.data.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def make(values, dtype: str) -> OracleTensor:
    """Storage for exactly representable values (rounded by numpy / torch,
    which the conversion pins check independently)."""
    v = np.asarray(values, dtype=np.float64).reshape(-1)
    if dtype == "f32":
        return OracleTensor(v.astype(np.float32), "f32")
    if dtype == "f16":
        return OracleTensor(v.astype(np.float16), "f16")
    tb = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    return OracleTensor(tb.view(torch.int16).numpy().view(np.uint16).copy(), "bf16")
