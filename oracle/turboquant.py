"""TurboQuant rotated Lloyd-Max code (CPU oracle).

Test infrastructure: see the package docstring for who may import this.

Source: Foundry "TurboQuant KV Cache Compression - Spec":
  * "As-Built Notes" 1: the random +-1 sign diagonal D is applied BEFORE the
    Walsh-Hadamard transform, y = H (D x) / sqrt(d).
  * "As-Built Notes" 2: normalise by the vector L2 norm, so each rotated
    coordinate lands on the unit sphere; (u + 1) / 2 then follows
    Beta(d/2, d/2) on [0, 1] (the page's statement of the law).
  * "Step 2: Lloyd-Max Scalar Quantization": the level index of a coordinate
    comes from the decision boundaries, the reconstruction from the centroids.
  * "Codebook Generation": uniform boundaries on [0, 1] to start, centroids
    as conditional means E[X | cell] under Beta(d/2, d/2), boundaries as the
    midpoints of adjacent centroids, repeated until converged.
  * "Hadamard Transform Detail": the in-place butterfly with the stage length
    growing 1, 2, 4, ... and (u + v, u - v) per pair.
  * "Optimization: Fused dequant-dot": dot(Q, R^T k_rot) = dot(R Q, k_rot);
    the output accumulates in the rotated domain and is rotated back once.

Readings where the page is silent or contradicts itself:
  * The spec text writes rotate(x) = D H x / sqrt(d); the as-built note puts
    the signs first. The as-built order is used: R = H D / sqrt(d).
  * The page calls the inverse "the same operation". For R = H D / sqrt(d)
    the inverse is R^T = D H / sqrt(d): FWHT first, then the signs. The
    mathematics is followed.
  * Signs: SplitMix64 (Vigna's published generator) from the seed; sign j is
    -1 when the top bit of the j-th output is set, else +1.
  * 1/sqrt(d) is computed in double and rounded once to float32.
  * The norm is sqrt of a fixed pairwise tree sum of x_j^2 (stride d/2, then
    d/4, ..., 1) in float32; sqrt is the correctly rounded float32 sqrt.
  * u = y / n and w = (u + 1) * 0.5, each rounded to float32; the code is the
    number of boundaries b_i with w >= b_i (ties go up). A zero vector keeps
    n = 0 and takes u = 0, so its code is the one for w = 0.5 and it
    dequantises to exactly 0.
  * One float32 norm is stored per (token, head) for K and one for V, in place
    of the page's two range floats.
  * Dequantisation: y_hat_j = n * (2 c[code_j] - 1) in float32; x_hat =
    D (FWHT(y_hat) * r).
  * The codebook iteration stops when no boundary moves by more than 1e-14;
    its fixed point is unique because the Beta(a, a) density is log-concave
    for a >= 1, so the start only changes the iteration count.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import betainc, betaincc

_MASK64 = (1 << 64) - 1


def splitmix64(seed: int, n: int) -> list[int]:
    """The first n outputs of SplitMix64 started from `seed`."""
    state = seed & _MASK64
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        out.append(z ^ (z >> 31))
    return out


def signs(seed: int, d: int) -> np.ndarray:
    """The +-1 diagonal D as float32 [d]."""
    return np.array([-1.0 if (z >> 63) else 1.0 for z in splitmix64(seed, d)], np.float32)


def fwht(x: np.ndarray) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform along the last axis (float32).

    Stage lengths 1, 2, 4, ...; each pair (u, v) becomes (u + v, u - v).
    """
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("FWHT needs a power-of-two length")
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(*lead, d // (2 * h), 2, h)
        u = y[..., 0, :].copy()
        v = y[..., 1, :].copy()
        y[..., 0, :] = u + v
        y[..., 1, :] = u - v
        y = y.reshape(*lead, d)
        h *= 2
    return y


def inv_sqrt(d: int) -> np.float32:
    return np.float32(1.0 / math.sqrt(d))


def rotate(x: np.ndarray, sgn: np.ndarray) -> np.ndarray:
    """y = FWHT(D x) / sqrt(d), float32."""
    d = x.shape[-1]
    return fwht(np.asarray(x, np.float32) * sgn) * inv_sqrt(d)


def unrotate(y: np.ndarray, sgn: np.ndarray) -> np.ndarray:
    """x = D FWHT(y) / sqrt(d), the inverse (transpose) of `rotate`."""
    d = y.shape[-1]
    return (fwht(np.asarray(y, np.float32)) * inv_sqrt(d)) * sgn


def tree_sum(a: np.ndarray) -> np.ndarray:
    """Pairwise float32 sum along the last axis: stride d/2, d/4, ..., 1."""
    a = np.asarray(a, np.float32)
    while a.shape[-1] > 1:
        h = a.shape[-1] // 2
        a = a[..., :h] + a[..., h:]
    return a[..., 0]


def l2norm(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float32)
    return np.sqrt(tree_sum(x * x))


# ---------------------------------------------------------------- codebooks

def _cell_mass(al: float, be: float, lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    """P(lo < X < hi) for X ~ Beta(al, be), taken from the nearer tail so that
    tiny tail masses keep their relative precision."""
    out = np.empty(len(lo))
    for i, (l, h) in enumerate(zip(lo, hi)):
        if h <= 0.5:
            out[i] = betainc(al, be, h) - betainc(al, be, l)
        elif l >= 0.5:
            out[i] = betaincc(al, be, l) - betaincc(al, be, h)
        else:
            out[i] = 1.0 - betainc(al, be, l) - betaincc(al, be, h)
    return out


def conditional_means(a: float, edges: np.ndarray) -> np.ndarray:
    """E[X | edges[i] < X < edges[i+1]] for X ~ Beta(a, a).

    With x f_{a,a}(x) = (a / 2a) f_{a+1,a}(x), the conditional mean is
    (1/2) * mass_{a+1,a}(cell) / mass_{a,a}(cell). A cell with no mass in
    double keeps its midpoint.
    """
    lo, hi = edges[:-1], edges[1:]
    m0 = _cell_mass(a, a, lo, hi)
    m1 = _cell_mass(a + 1.0, a, lo, hi)
    safe = np.where(m0 > 0, m0, 1.0)
    return np.where(m0 > 0, 0.5 * m1 / safe, 0.5 * (lo + hi))


def lloyd_max_beta(a: float, bits: int, tol: float = 1e-14, max_iter: int = 200000):
    """Lloyd-Max quantiser of Beta(a, a) on [0, 1] with 2^bits levels.

    Returns (boundaries float64 [2^bits - 1], centroids float64 [2^bits],
    iterations).
    """
    n_lev = 1 << bits
    b = np.arange(1, n_lev, dtype=np.float64) / n_lev
    c = conditional_means(a, np.concatenate([[0.0], b, [1.0]]))
    it = 0
    for it in range(1, max_iter + 1):
        nb = 0.5 * (c[:-1] + c[1:])
        moved = float(np.max(np.abs(nb - b))) if len(b) else 0.0
        b = nb
        c = conditional_means(a, np.concatenate([[0.0], b, [1.0]]))
        if moved < tol:
            break
    return b, c, it


_CODEBOOKS: dict = {}


def codebook(head_dim: int, bits: int):
    """float32 (boundaries, centroids) for Beta(d/2, d/2) with 2^bits levels."""
    key = (head_dim, bits)
    if key not in _CODEBOOKS:
        b, c, _ = lloyd_max_beta(head_dim / 2.0, bits)
        _CODEBOOKS[key] = (b.astype(np.float32), c.astype(np.float32))
    return _CODEBOOKS[key]


# ---------------------------------------------------------------- quantise

def quantize(x: np.ndarray, sgn: np.ndarray, boundaries: np.ndarray):
    """Quantise rows x [..., d] (float32). Returns (codes uint8 [..., d],
    norms float32 [...])."""
    x = np.asarray(x, np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("NaN/Inf input")
    y = rotate(x, sgn)
    n = l2norm(x)
    nz = n > 0
    u = np.zeros_like(y)
    u[nz] = y[nz] / n[nz][..., None]
    w = (u + np.float32(1.0)) * np.float32(0.5)
    codes = (w[..., None] >= boundaries).sum(axis=-1).astype(np.uint8)
    return codes, n


def dequantize_rotated(codes: np.ndarray, norms: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """y_hat = n * (2 c[code] - 1) in the rotated domain (float32)."""
    t = np.float32(2.0) * centroids[codes] - np.float32(1.0)
    return np.asarray(norms, np.float32)[..., None] * t


def dequantize(codes, norms, sgn, centroids) -> np.ndarray:
    """x_hat = D FWHT(y_hat) / sqrt(d) in the original domain (float32)."""
    return unrotate(dequantize_rotated(codes, norms, centroids), sgn)
