"""KVSink-style dynamic sink selection and calibration exclusion (CPU oracle).

Test infrastructure: see the package docstring for who may import this.

Source: VeloxQuant-MLX "KVSink-Adapted Sink Protection", section "How it
works": (1) per-token key L2 norm, mean over KV heads, folded into a top-k of
the highest-norm positions; (2) sink tokens are stored fp16 and never
quantised; (3) calibration exclusion - before a group's min/max is taken,
sink rows are replaced by the nearest non-sink row; (4) byte accounting keeps
sink bytes apart from residual bytes. "Known v1 limitation": selection is
prefill-dominant; a token quantised earlier is never restored later.

Readings where the page is silent:
  * The norm of one head's key is the float32 sqrt of the fixed pairwise tree
    sum of k_c^2 (stride D/2, D/4, ..., 1); the per-token value is the sum of
    the Hkv head norms in head order, divided by Hkv (float32 division).
  * The top-k is per batch element (per sequence), ordered by norm
    descending, ties to the lower position.
  * The running top-k is folded call by call (every append and prefill, the
    page's "on every update_and_fetch"): the candidates are the call's tokens
    and the sinks whose group was not yet quantised when the call began; a
    sink whose group is already quantised is locked (its codes hold a
    substitute's values, its fp16 row is its only faithful copy, and the
    page never restores a quantised token), so it neither leaves the set nor
    yields its place. The set is the locked sinks plus the best
    min(k, L) - locked candidates. On an empty cache one call is the plain
    top-k over its tokens.
  * Sink K AND V rows are kept exact and replaced, in their group, by the
    nearest non-sink row of the SAME group (nearest by position, ties to the
    earlier row). A group with no non-sink row is left as it is.
"""
from __future__ import annotations

import numpy as np

from .turboquant import tree_sum


def key_norms(k: np.ndarray) -> np.ndarray:
    """k: float32 [B, Hkv, T, D] -> m float32 [B, T] (mean over heads of ||k||)."""
    k = np.asarray(k, np.float32)
    per_head = np.sqrt(tree_sum(k * k))          # [B, H, T]
    acc = per_head[:, 0, :].copy()
    for h in range(1, per_head.shape[1]):
        acc = acc + per_head[:, h, :]
    return acc / np.float32(per_head.shape[1])


def top_k(m: np.ndarray, k: int, first_pos: int = 0) -> np.ndarray:
    """Top-k absolute positions per row of m [B, T]: norm descending, ties to
    the lower position. Returned sorted by position, int64 [B, min(k, T)]."""
    B, T = m.shape
    kk = min(k, T)
    out = np.empty((B, kk), np.int64)
    for b in range(B):
        # primary key: norm descending; secondary key: position ascending
        order = np.lexsort((np.arange(T), -m[b].astype(np.float32)))
        out[b] = np.sort(order[:kk].astype(np.int64)) + first_pos
    return out


def admit(members: list, m_call: np.ndarray, first_pos: int, q0: int, k: int) -> list:
    """One call's fold of one sequence into the running top-k.

    members: [(pos, m)] of the set before the call; m_call: float32 [n] norms
    of the call's tokens at positions first_pos .. first_pos + n - 1; q0: the
    end of the quantised groups when the call began (members below it are
    locked). Returns the new set [(pos, m)] sorted by position, of size
    min(k, first_pos + n).
    """
    n = len(m_call)
    locked = [(p, m) for p, m in members if p < q0]
    cand = [(p, m) for p, m in members if p >= q0]
    cand += [(first_pos + i, np.float32(m_call[i])) for i in range(n)]
    budget = min(k, first_pos + n) - len(locked)
    # norm descending, ties to the lower position
    cand.sort(key=lambda pm: (-float(pm[1]), pm[0]))
    return sorted(locked + cand[:max(budget, 0)])


def substitutes(sink_rows: set, n: int = 32) -> dict:
    """For each sink row r of a group of n rows: the nearest non-sink row
    (ties to the earlier one). Empty when every row is a sink."""
    free = [r for r in range(n) if r not in sink_rows]
    if not free:
        return {}
    return {r: min(free, key=lambda f: (abs(f - r), f)) for r in sink_rows}


def exclude(rows: np.ndarray, sink_rows: set) -> np.ndarray:
    """Copy of one group's rows [..., 32, D] with every sink row replaced by
    its substitute row."""
    out = np.array(rows, copy=True)
    for r, f in substitutes(sink_rows, rows.shape[-2]).items():
        out[..., r, :] = rows[..., f, :]
    return out
