"""Vanilla RoPE baked into K at absolute positions (CPU oracle).

Test infrastructure: see the package docstring for who may import this.

Source: posttrainllm "StreamingLLM + KIVI" doc, section "RoPE caveat - the
'vanilla' StreamingLLM choice": keys keep the rotation of their ORIGINAL
absolute position, and the query at generation step T uses its own absolute
position.

Readings where the page is silent:
  * Pairing is the half-split one: channel i rotates with channel i + D/2.
  * theta_i = base^(-2i/D); angle = pos * theta_i, all in double; cos and
    sin are evaluated in double (the C library's cos/sin through Python's
    math module) and rounded once to float32. The table depends only on
    (base, D, pos).
  * The rotation is x' = x c - y s, y' = x s + y c in float32 with every
    product and sum rounded separately, then the rotated key is rounded to
    the activation dtype before it is stored or quantised.
  * The query is rotated at position L - 1 (the newest token) in float32 and
    is not rounded to the activation dtype.
"""
from __future__ import annotations

import math

import numpy as np

from .numerics import round_act


def cos_sin(positions, head_dim: int, base: float) -> np.ndarray:
    """float32 [len(positions), D/2, 2] table of (cos, sin)."""
    half = head_dim // 2
    positions = [int(p) for p in np.atleast_1d(positions)]
    tab = np.empty((len(positions), half, 2), np.float32)
    for i in range(half):
        inv = base ** (-(2.0 * i) / head_dim)
        for r, p in enumerate(positions):
            ang = p * inv
            tab[r, i, 0] = math.cos(ang)
            tab[r, i, 1] = math.sin(ang)
    return tab


def rotate64(x: np.ndarray, positions, base: float) -> np.ndarray:
    """Rotate float64 rows x [..., T, D] at positions [T] (any integers,
    negative ones un-rotate), angles, cos and sin all in double."""
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    half = D // 2
    pos = np.asarray(positions, np.float64)[:, None]
    inv = np.array([base ** (-(2.0 * i) / D) for i in range(half)], np.float64)[None, :]
    c = np.cos(pos * inv)
    s = np.sin(pos * inv)
    a = x[..., :half]
    b = x[..., half:]
    out = np.empty_like(x)
    out[..., :half] = a * c - b * s
    out[..., half:] = a * s + b * c
    return out


def rotate(x: np.ndarray, positions, base: float) -> np.ndarray:
    """Rotate float32 rows x [..., T, D] at absolute positions [T] (float32)."""
    x = np.asarray(x, np.float32)
    D = x.shape[-1]
    half = D // 2
    tab = cos_sin(positions, D, base)            # [T, D/2, 2]
    c = tab[..., 0]
    s = tab[..., 1]
    a = x[..., :half]
    b = x[..., half:]
    out = np.empty_like(x)
    out[..., :half] = a * c - b * s
    out[..., half:] = a * s + b * c
    return out


def rotate_keys(k: np.ndarray, first_pos: int, base: float, act_dtype: str) -> np.ndarray:
    """Keys [..., T, D] at positions first_pos.., rounded back to the act dtype."""
    T = k.shape[-2]
    return round_act(rotate(k, np.arange(first_pos, first_pos + T), base), act_dtype)
