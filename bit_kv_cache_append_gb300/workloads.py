"""Seeded synthetic workloads for the quantised KV-cache path.

This module only draws random numbers and shapes them like the workloads the
pages describe. It holds none of the method's arithmetic (no quantisation, no
rotation, no norms): the CUDA path and the CPU oracle both take their inputs
from here and from nowhere else.

Every generator returns float32 numpy arrays whose values are exactly
representable in the workload's activation dtype (fp16 or bf16), so the same
bits reach both sides.

The five shapes follow the workloads named for this method:
  * ``tiny``      - KIVI K2/V4, B1, Hkv2, Hq4, D64, 512 tokens, fp16, 4 of 64 K
                    channels per KV head scaled x10 (channel outliers).
  * ``llama8b``   - Llama-3-8B-shaped decode: B16, Hq32, Hkv8, D128, 32768
                    tokens, bf16, K channel (h, c) scaled by exp(U(0, ln 75)).
  * ``ring``      - StreamingLLM ring: 12 layers, B64, H8 (MHA), D64, fp16,
                    each (layer, h, c) K channel x20 with probability 0.02.
  * ``turboquant``- D128, Hkv8, Hq32, B32, 16384 tokens, fp16 AR(1) over
                    channels with rho = 0.6.
  * ``kvsink``    - B4, Hkv8, Hq32, D128, 131072 tokens, fp16, five planted
                    sink positions whose K rows are x25 in every KV head.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    context: int
    act_dtype: str          # "f16" or "bf16"
    mode: str               # "kivi" or "turboquant"
    k_bits: int
    v_bits: int
    n_layers: int = 1
    n_sink: int = 0
    window: int = 0
    evict_window: int = 0
    n_dyn_sinks: int = 0
    rope_base: float = 0.0

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 4, 64, 512, "f16", "kivi", 2, 4,
                     n_sink=4, window=64),
    "llama8b": Workload("llama8b", 16, 8, 32, 128, 32768, "bf16", "kivi", 2, 4,
                        n_sink=4, window=128),
    "ring_int8": Workload("ring_int8", 64, 8, 8, 64, 65536, "f16", "kivi", 8, 8,
                          n_layers=12, n_sink=4, evict_window=4096,
                          rope_base=10000.0),
    "ring_int4": Workload("ring_int4", 64, 8, 8, 64, 65536, "f16", "kivi", 4, 4,
                          n_layers=12, n_sink=4, evict_window=4096,
                          rope_base=10000.0),
    "turboquant_k4v2": Workload("turboquant_k4v2", 32, 8, 32, 128, 16384, "f16",
                                "turboquant", 4, 2),
    "turboquant_k4v4": Workload("turboquant_k4v4", 32, 8, 32, 128, 16384, "f16",
                                "turboquant", 4, 4),
    "kvsink": Workload("kvsink", 4, 8, 32, 128, 131072, "f16", "kivi", 2, 2,
                       n_dyn_sinks=5),
}


def round_to_act(x: np.ndarray, act_dtype: str) -> np.ndarray:
    """Round float32 values to the activation dtype and return them as float32.

    fp16 uses numpy's round-to-nearest-even cast; bf16 uses torch's CPU cast
    (also round-to-nearest-even). Values beyond the fp16 range are clipped
    first so every generated value is finite in either dtype.
    """
    x = np.asarray(x, dtype=np.float32)
    if act_dtype == "f16":
        return np.clip(x, -65504.0, 65504.0).astype(np.float16).astype(np.float32)
    if act_dtype == "bf16":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
        return t.to(torch.float32).numpy()
    raise ValueError(f"unknown activation dtype {act_dtype!r}")


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def normal(seed: int, stream: int, shape) -> np.ndarray:
    return _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)


def k_channel_factors(w: Workload, seed: int, layer: int = 0) -> np.ndarray:
    """Per-(KV head, channel) K multipliers, shape [Hkv, D] (float32)."""
    H, D = w.n_kv_heads, w.head_dim
    r = _rng(seed, 1000 + layer)
    f = np.ones((H, D), np.float32)
    if w.name == "tiny":
        for h in range(H):
            ch = r.choice(D, size=4, replace=False)
            f[h, ch] = 10.0
    elif w.name == "llama8b":
        f[:] = np.exp(r.uniform(0.0, math.log(75.0), size=(H, D))).astype(np.float32)
    elif w.name.startswith("ring"):
        f[r.random((H, D)) < 0.02] = 20.0
    return f


def ar1_channels(seed: int, stream: int, shape, rho: float = 0.6) -> np.ndarray:
    """AR(1) over the last axis: x0 = z0, xi = rho x(i-1) + sqrt(1 - rho^2) zi."""
    z = normal(seed, stream, shape)
    x = np.empty_like(z)
    x[..., 0] = z[..., 0]
    c = np.float32(math.sqrt(1.0 - rho * rho))
    for i in range(1, z.shape[-1]):
        x[..., i] = np.float32(rho) * x[..., i - 1] + c * z[..., i]
    return x


def sink_positions(seed: int, batch: int, context: int, k: int = 5) -> np.ndarray:
    """Distinct planted positions per batch element, sorted, int64 [B, k]."""
    r = _rng(seed, 2000)
    return np.stack([np.sort(r.choice(context, size=k, replace=False))
                     for _ in range(batch)]).astype(np.int64)


def kv_tokens(w: Workload, seed: int, n_tokens: int, layer: int = 0,
              first_pos: int = 0, batch_slice=None, head_slice=None):
    """K, V float32 [B, Hkv, n_tokens, D] for absolute positions first_pos... .

    The draw depends on (seed, layer, first_pos, n_tokens): a streaming
    caller that draws one token per step gets an independent row per step.
    """
    B, H, D = w.batch, w.n_kv_heads, w.head_dim
    shape = (B, H, n_tokens, D)
    s_k = 10 * layer + 1 + 100000 * first_pos
    s_v = 10 * layer + 2 + 100000 * first_pos
    if w.mode == "turboquant":
        k = ar1_channels(seed, s_k, shape)
        v = ar1_channels(seed, s_v, shape)
    else:
        k = normal(seed, s_k, shape)
        v = normal(seed, s_v, shape)
    k = k * k_channel_factors(w, seed, layer)[None, :, None, :]
    if w.name == "kvsink":
        pos = sink_positions(seed, B, w.context)
        for b in range(B):
            for p in pos[b]:
                if first_pos <= p < first_pos + n_tokens:
                    k[b, :, p - first_pos, :] *= np.float32(25.0)
    if batch_slice is not None:
        k, v = k[batch_slice], v[batch_slice]
    if head_slice is not None:
        k, v = k[:, head_slice], v[:, head_slice]
    return round_to_act(k, w.act_dtype), round_to_act(v, w.act_dtype)


def queries(w: Workload, seed: int, step: int = 0) -> np.ndarray:
    """q float32 [B, Hq, D] ~ N(0,1) (AR(1) over channels for turboquant)."""
    shape = (w.batch, w.n_q_heads, w.head_dim)
    if w.mode == "turboquant":
        q = ar1_channels(seed, 3000 + step, shape)
    else:
        q = normal(seed, 3000 + step, shape)
    return round_to_act(q, w.act_dtype)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some fields changed (smaller parity cases)."""
    return dataclasses.replace(w, **changes)
