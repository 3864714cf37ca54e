"""Helpers shared by the GPU parity tests: run the same seeded inputs through
the CUDA library (via the C-ABI binding) and the CPU oracle, and compare.

Codes, scales, zeros, norms, sink positions, sink rows, tail rows and
eviction ranges must match bit for bit; decode attention must agree within
relative L2 <= 1e-3 and max-abs <= 5e-3 (fp32 output against the oracle's
double computation from the same dequantised values).
"""
from __future__ import annotations

import numpy as np

REL_L2 = 1e-3
MAX_ABS = 5e-3

# (rel_l2, max_abs, test) of every attention comparison of the session, for
# the summary the test session prints at its end
ERRORS: list = []

KIVI_ARRAYS = ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero")
TQ_ARRAYS = ("k_codes", "k_norm", "v_codes", "v_norm")


def torch_act(x: np.ndarray, act: str):
    import torch
    dt = torch.bfloat16 if act == "bf16" else torch.float16
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dt).cuda()


def cache_kwargs(w, max_tokens, n_layers=None, **over):
    kw = dict(n_layers=n_layers or w.n_layers, batch=w.batch, n_kv_heads=w.n_kv_heads,
              n_q_heads=w.n_q_heads, head_dim=w.head_dim, max_tokens=max_tokens,
              mode=w.mode, k_bits=w.k_bits, v_bits=w.v_bits, n_sink=w.n_sink, window=w.window,
              evict_window=w.evict_window, n_dyn_sinks=w.n_dyn_sinks, act_dtype=w.act_dtype,
              seed=over.pop("seed", 0), rope_base=w.rope_base,
              rope_max_pos=over.pop("rope_max_pos", max_tokens if w.rope_base else 0))
    kw.update(over)
    return kw


def oracle_config(kw):
    from oracle import CacheConfig
    return CacheConfig(n_layers=kw["n_layers"], batch=kw["batch"], n_kv_heads=kw["n_kv_heads"],
                       n_q_heads=kw["n_q_heads"], head_dim=kw["head_dim"],
                       max_tokens=kw["max_tokens"], mode=kw["mode"], k_bits=kw["k_bits"],
                       v_bits=kw["v_bits"], n_sink=kw["n_sink"], window=kw["window"],
                       evict_window=kw["evict_window"], n_dyn_sinks=kw["n_dyn_sinks"],
                       act_dtype=kw["act_dtype"], seed=kw["seed"], rope_base=kw["rope_base"],
                       rope_reposition=bool(kw.get("rope_reposition", False)),
                       v_q4_0=bool(kw.get("v_q4_0", False)), k_pre_rope=bool(kw.get("k_pre_rope", False)))


def compare_exports(gpu_cache, oc, layer: int) -> None:
    """Bit-exact comparison of every stored array of one layer."""
    ref = oc.export(layer)
    names = TQ_ARRAYS if oc.cfg.mode == "turboquant" else KIVI_ARRAYS
    for name in names:
        got = gpu_cache.export(layer, name)
        if name not in ref:
            assert got.size == 0, name
            continue
        want = ref[name]
        if name.endswith(("scale", "zero")):
            got, want = got.view(np.uint16), want.view(np.uint16)
        elif name.endswith("norm"):
            got, want = got.view(np.uint32), want.astype(np.float32).view(np.uint32)
        assert got.shape == want.shape, (name, got.shape, want.shape)
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{name}: {len(bad)} mismatches, first at {bad[:5].tolist()}"
    sp = gpu_cache.export(layer, "sink_pos")
    assert np.array_equal(sp, ref["sink_pos"]), (sp, ref["sink_pos"])
    for name in ("sink_k", "sink_v"):
        assert np.array_equal(gpu_cache.export(layer, name), ref[name]), name
    if "tail_k" in ref:
        for name in ("tail_k", "tail_v"):
            assert np.array_equal(gpu_cache.export(layer, name), ref[name]), name
    if oc.cfg.mode == "kivi" and "sink_mask" in ref:
        assert np.array_equal(gpu_cache.export(layer, "sink_mask"), ref["sink_mask"])
    s_gpu, s_ref = gpu_cache.stats(layer), oc.stats(layer)
    for key, val in s_ref.items():
        assert s_gpu[key] == val, (key, s_gpu[key], val)


def compare_attention(out_gpu: np.ndarray, out_ref: np.ndarray, heads=None) -> dict:
    """Tolerance check; returns the measured errors."""
    if heads is not None:
        idx = tuple(np.array(heads).T)
        out_gpu, out_ref = out_gpu[idx], out_ref[idx]
    d = out_gpu.astype(np.float64) - out_ref.astype(np.float64)
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(out_ref.astype(np.float64)), 1e-30))
    mx = float(np.max(np.abs(d))) if d.size else 0.0
    assert np.all(np.isfinite(out_gpu)), "non-finite output"
    import os
    ERRORS.append((rel, mx, os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]))
    assert rel <= REL_L2 and mx <= MAX_ABS, dict(rel_l2=rel, max_abs=mx)
    return dict(rel_l2=rel, max_abs=mx)
