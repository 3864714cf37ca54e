"""Rounding helpers for the CPU oracle (16-bit activation types).

Test infrastructure: see the package docstring for who may import this.

numpy has no bfloat16, so bf16 values are carried in float32 arrays whose low
16 bits are zero. Rounding to bf16 is round-to-nearest-even on the upper half
of the float32 bit pattern.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bf16 (ties to even), returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("NaN/Inf reached the bf16 rounding")
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return u.astype(np.uint32).view(np.float32)


def round_f16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest fp16 (ties to even), returned as float32."""
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)


def round_act(x: np.ndarray, act_dtype: str) -> np.ndarray:
    if act_dtype == "f16":
        return round_f16(x)
    if act_dtype == "bf16":
        return round_bf16(x)
    raise ValueError(act_dtype)


def is_representable(x: np.ndarray, act_dtype: str) -> bool:
    x = np.asarray(x, np.float32)
    return bool(np.array_equal(round_act(x, act_dtype), x))
