"""Pins of the oracle cache: segments, eviction, byte accounting, RoPE and
decode attention (no GPU)."""
import math

import numpy as np
import pytest
import torch

from oracle import CacheConfig, OracleCache, kivi, rope
from oracle.numerics import round_bf16
from tests.conftest import read_golden


def _f16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16).astype(np.float32)


def _cfg(**kw):
    base = dict(n_layers=1, batch=2, n_kv_heads=2, n_q_heads=4, head_dim=64,
                max_tokens=1024, k_bits=2, v_bits=4)
    base.update(kw)
    return CacheConfig(**base)


def _sdpa64(q, K, V):
    """Reference attention by torch's SDPA in float64 (a different routine)."""
    qt = torch.from_numpy(q.astype(np.float64))[None, None, None]
    Kt = torch.from_numpy(K.astype(np.float64))[None, None]
    Vt = torch.from_numpy(V.astype(np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)[0, 0, 0].numpy()


def _partition_ok(c, layer=0):
    s = c.stats(layer)
    B = c.cfg.batch
    return s["n_quant"] + s["n_sink"] + s["n_tail"] + s["n_evicted"] == B * s["length"]


@pytest.mark.parametrize("kw", [dict(n_sink=4, window=64), dict(), dict(window=40),
                                dict(n_sink=4, evict_window=96),
                                dict(mode="turboquant", k_bits=4, v_bits=2, n_sink=2, window=8)])
def test_pool_partition_every_step(kw):
    rng = np.random.default_rng(0)
    c = OracleCache(_cfg(**kw))
    for step in range(230):
        n = 1 if step % 7 else 5
        c.append(0, _f16(rng, (2, 2, n, 64)), _f16(rng, (2, 2, n, 64)))
        c.evict(0)
        assert _partition_ok(c)
        pos, _, _, _ = c.read_set(0, 1, 1)
        s = c.stats(0)
        # every retained position is read exactly once
        assert len(pos) == len(set(pos.tolist()))
        assert len(pos) == s["length"] - s["n_evicted"] // c.cfg.batch


def test_streaming_cap_matches_smoke_test():
    """P1 smoke test: sink 4 + window 256 caps the stored count at 260."""
    g = {r[0]: int(r[1]) for r in read_golden("streaming_llm_smoke.txt")}
    rng = np.random.default_rng(1)
    c = OracleCache(_cfg(batch=1, n_kv_heads=1, n_q_heads=1, k_bits=8, v_bits=8,
                         n_sink=g["sink"], evict_window=g["window"], max_tokens=400))
    ranges = []
    for L in range(1, g["tokens"] + 1):
        c.append(0, _f16(rng, (1, 1, 1, 64)), _f16(rng, (1, 1, 1, 64)))
        b, e = c.evict(0)
        if e > b:
            ranges.append((b, e))
        s = c.stats(0)
        stored = s["length"] - s["n_evicted"]
        assert stored == min(L, g["stored_cap"])
    # evicted ranges are contiguous, disjoint and cover [sink, L - window)
    assert ranges[0][0] == g["sink"]
    assert all(ranges[i][1] == ranges[i + 1][0] for i in range(len(ranges) - 1))
    assert ranges[-1][1] == g["tokens"] - g["window"]


def test_window_covering_context_is_exact_attention():
    """A window covering the whole context gives exact fp16 attention."""
    rng = np.random.default_rng(2)
    c = OracleCache(_cfg(n_sink=4, window=10_000))
    k, v = _f16(rng, (2, 2, 300, 64), 3.0), _f16(rng, (2, 2, 300, 64))
    c.prefill_quantize(0, k, v)
    q = _f16(rng, (2, 4, 64))
    out, _ = c.decode_attn(0, q)
    for b in range(2):
        for j in range(4):
            ref = _sdpa64(q[b, j], k[b, j // 2], v[b, j // 2])
            assert np.allclose(out[b, j], ref, rtol=1e-6, atol=1e-7)


def test_zero_query_gives_mean_of_values():
    """q = 0 makes every score equal: out = mean of the retained values. V on
    an exact 2-bit grid per 32-channel group dequantises exactly."""
    rng = np.random.default_rng(3)
    T = 200
    v = ((np.arange(64) % 4) * 0.25 - 0.5).astype(np.float32)
    v = np.broadcast_to(v, (2, 2, T, 64)).copy()
    v *= (1 + rng.integers(0, 3, size=(2, 2, T, 1))).astype(np.float32)
    c = OracleCache(_cfg(v_bits=2))
    c.prefill_quantize(0, _f16(rng, (2, 2, T, 64)), v)
    out, lse = c.decode_attn(0, np.zeros((2, 4, 64), np.float32))
    for b in range(2):
        for j in range(4):
            assert np.allclose(out[b, j], v[b, j // 2].mean(0), atol=1e-6)
            assert abs(lse[b, j] - math.log(T)) < 1e-6


def test_gqa_head_mapping():
    """Query head j reads KV head j // (Hq / Hkv): KV head h holds the
    constant h + 1, so out[b, j] = j // g + 1 exactly."""
    rng = np.random.default_rng(4)
    H, Hq, T = 4, 8, 96
    v = np.zeros((1, H, T, 64), np.float32)
    for h in range(H):
        v[0, h] = h + 1
    c = OracleCache(_cfg(batch=1, n_kv_heads=H, n_q_heads=Hq))
    c.prefill_quantize(0, _f16(rng, (1, H, T, 64)), v)
    out, _ = c.decode_attn(0, _f16(rng, (1, Hq, 64)))
    for j in range(Hq):
        assert np.allclose(out[0, j], j // 2 + 1, atol=1e-6)


def test_one_at_a_time_equals_prefill():
    rng = np.random.default_rng(5)
    cfg = _cfg(n_sink=4, window=64)
    k, v = _f16(rng, (2, 2, 333, 64)), _f16(rng, (2, 2, 333, 64))
    a, b = OracleCache(cfg), OracleCache(cfg)
    a.prefill_quantize(0, k, v)
    for t in range(333):
        b.append(0, k[:, :, t:t + 1], v[:, :, t:t + 1])
    ea, eb = a.export(0), b.export(0)
    assert ea.keys() == eb.keys()
    for key in ea:
        assert np.array_equal(ea[key], eb[key]), key


def test_plain_kivi_when_no_overlay():
    """n_sink = window = 0: every position below Q_end is read from codes,
    the residual from the tail; attention equals SDPA over those rows
    (dequantised here from the exported packed codes)."""
    rng = np.random.default_rng(6)
    T = 250
    k, v = _f16(rng, (1, 2, T, 64)), _f16(rng, (1, 2, T, 64))
    c = OracleCache(_cfg(batch=1))
    c.prefill_quantize(0, k, v)
    s = c.stats(0)
    assert s["n_quant"] == 224 and s["n_tail"] == 26 and s["n_sink"] == 0
    ex = c.export(0)
    q = _f16(rng, (1, 4, 64))
    out, _ = c.decode_attn(0, q)
    for h in range(2):
        kc = kivi.unpack_codes(ex["k_codes"][0, h], 2).astype(np.float32)     # [224, 64]
        ks = np.repeat(ex["k_scale"][0, h].astype(np.float32), 32, axis=0)
        kz = np.repeat(ex["k_zero"][0, h].astype(np.float32), 32, axis=0)
        vc = kivi.unpack_codes(ex["v_codes"][0, h], 4).astype(np.float32)
        vs = np.repeat(ex["v_scale"][0, h].astype(np.float32), 32, axis=1)
        vz = np.repeat(ex["v_zero"][0, h].astype(np.float32), 32, axis=1)
        K = np.concatenate([kc * ks + kz, k[0, h, 224:]])
        V = np.concatenate([vc * vs + vz, v[0, h, 224:]])
        for j in (2 * h, 2 * h + 1):
            assert np.allclose(out[0, j], _sdpa64(q[0, j], K, V), rtol=1e-5, atol=1e-6)


def test_segments_config_tiny():
    """Tiny workload (N_s 4, W 64, L 512): quantised [4, 448), tail [448, 512)."""
    rng = np.random.default_rng(7)
    c = OracleCache(_cfg(batch=1, n_sink=4, window=64, max_tokens=512))
    c.prefill_quantize(0, _f16(rng, (1, 2, 512, 64)), _f16(rng, (1, 2, 512, 64)))
    s = c.stats(0)
    assert (s["fp16_begin"], s["quant_end"], s["n_quant"], s["n_sink"], s["n_tail"]) == (448, 512, 2 * 0 + 444, 4, 64)


def test_byte_accounting_matches_pages():
    """Code and fp16 bytes per token against the pages' arithmetic."""
    rng = np.random.default_rng(8)
    # P2 table: TQ K4/V2 codes for 16 heads x D128 = 1024 + 512 B per token.
    fo = {r[0]: [int(x) for x in r[1:]] for r in read_golden("foundry_turboquant_bytes.txt")}
    for name in ("K4V2_16H", "K4V2_32H"):
        H, D, kb, vb, keys, values, meta, total = fo[name]
        c = OracleCache(_cfg(batch=1, n_kv_heads=H, n_q_heads=H, head_dim=D,
                             mode="turboquant", k_bits=kb, v_bits=vb))
        c.append(0, _f16(rng, (1, H, 1, D)), _f16(rng, (1, H, 1, D)))
        s = c.stats(0)
        assert s["code_bytes"] == keys + values
        assert s["kmeta_bytes"] + s["vmeta_bytes"] == meta // 2   # one float per vector, not two
    # K3/V2 with 3-bit codes packed tight (eight in three bytes), the count
    # the memory table prints
    H, D, kb, vb, keys, values, meta, total = fo["K3V2_16H_tight"]
    c = OracleCache(_cfg(batch=1, n_kv_heads=H, n_q_heads=H, head_dim=D,
                         mode="turboquant", k_bits=kb, v_bits=vb))
    c.append(0, _f16(rng, (1, H, 1, D)), _f16(rng, (1, H, 1, D)))
    assert c.stats(0)["code_bytes"] == keys + values
    # P3: FP16 2048 B/cell and q2k code bits 384 B/cell for 2 x 256 dims (= 4 x 128 here).
    pr = {r[0]: int(r[1]) for r in read_golden("pr2318_memory_math.txt")}
    c = OracleCache(_cfg(batch=1, n_kv_heads=4, n_q_heads=4, head_dim=128, k_bits=2, v_bits=4,
                         window=10_000))
    c.append(0, _f16(rng, (1, 4, 1, 128)), _f16(rng, (1, 4, 1, 128)))
    assert c.stats(0)["tail_bytes"] == pr["FP16"]
    c = OracleCache(_cfg(batch=1, n_kv_heads=4, n_q_heads=4, head_dim=128, k_bits=2, v_bits=4))
    c.append(0, _f16(rng, (1, 4, 32, 128)), _f16(rng, (1, 4, 32, 128)))
    assert c.stats(0)["code_bytes"] == 32 * 384
    # P1: 12 L x 8 H x D32 at T = 500 (8 x 32 = 256 dims per token = 2 x 128 here).
    p1 = {r[0]: int(r[1]) for r in read_golden("streaming_llm_kivi_bytes.txt")}
    T, Lyr = p1["tokens"], p1["layers"]
    assert p1["heads"] * p1["head_dim"] == 2 * 128
    c = OracleCache(_cfg(batch=1, n_kv_heads=2, n_q_heads=2, head_dim=128, window=10_000))
    c.append(0, _f16(rng, (1, 2, T, 128)), _f16(rng, (1, 2, T, 128)))
    assert Lyr * c.stats(0)["tail_bytes"] == p1["bf16_bytes"]
    for bits, key in ((8, "int8_code_bytes"), (4, "int4_packed_code_bytes")):
        c = OracleCache(_cfg(batch=1, n_kv_heads=2, n_q_heads=2, head_dim=128, k_bits=bits,
                             v_bits=bits, max_tokens=512))
        c.append(0, _f16(rng, (1, 2, 512, 128)), _f16(rng, (1, 2, 512, 128)))
        assert Lyr * c.stats(0)["code_bytes"] * T // 512 == p1[key]


def test_capacity_and_config_errors():
    rng = np.random.default_rng(9)
    c = OracleCache(_cfg(max_tokens=64))
    c.append(0, _f16(rng, (2, 2, 60, 64)), _f16(rng, (2, 2, 60, 64)))
    with pytest.raises(OverflowError):
        c.append(0, _f16(rng, (2, 2, 5, 64)), _f16(rng, (2, 2, 5, 64)))
    assert c.stats(0)["length"] == 60
    for bad in (dict(head_dim=96), dict(n_q_heads=3), dict(k_bits=5), dict(evict_window=16),
                dict(n_dyn_sinks=5, n_sink=4), dict(mode="turboquant", k_bits=8)):
        with pytest.raises(ValueError):
            OracleCache(_cfg(**bad))


# ------------------------------------------------------------------ RoPE

def test_rope_identity_at_zero_and_norm():
    rng = np.random.default_rng(10)
    x = _f16(rng, (3, 1, 64))
    assert np.array_equal(rope.rotate(x, [0], 10000.0), x)
    for p in (1, 17, 4095, 65000):
        y = rope.rotate(x, [p], 10000.0)
        assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-6)


def test_rope_matches_complex_rotation_and_relative_position():
    """Half-split pairs (x_i, x_{i+D/2}) rotate like x_i + i x_{i+D/2} times
    exp(i pos theta_i), theta_i = base^(-2i/D); scores depend on m - n only."""
    rng = np.random.default_rng(11)
    D, base = 64, 10000.0
    x = _f16(rng, (1, D))
    for p in (3, 1000):
        th = base ** (-(2.0 * np.arange(D // 2)) / D)
        z = (x[0, :D // 2] + 1j * x[0, D // 2:]) * np.exp(1j * p * th)
        want = np.concatenate([z.real, z.imag])
        assert np.allclose(rope.rotate(x, [p], base)[0], want, atol=1e-5)
    q, k = _f16(rng, (1, D)), _f16(rng, (1, D))
    s1 = np.dot(rope.rotate(q, [5], base)[0], rope.rotate(k, [2], base)[0])
    s2 = np.dot(rope.rotate(q, [1003], base)[0], rope.rotate(k, [1000], base)[0])
    assert abs(s1 - s2) < 1e-4


def test_rope_keys_rounded_to_act_dtype():
    rng = np.random.default_rng(12)
    k = _f16(rng, (1, 1, 8, 64))
    y = rope.rotate_keys(k, 100, 10000.0, "bf16")
    assert np.array_equal(round_bf16(y), y)
    assert np.array_equal(round_bf16(np.array([1.0 + 2 ** -8], np.float32)), np.array([1.0], np.float32))
    assert np.array_equal(round_bf16(np.array([1.0 + 3 * 2 ** -8], np.float32)),
                          np.array([1.0 + 2 ** -6], np.float32))
    t = torch.from_numpy(y.ravel()).to(torch.bfloat16).float().numpy()
    assert np.array_equal(t, y.ravel())


def test_rope_bf16_rounding_agrees_with_torch():
    x = np.random.default_rng(13).standard_normal(100000).astype(np.float32) * 7
    assert np.array_equal(round_bf16(x), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_ring_with_rope_reads_keys_at_absolute_positions():
    """Window covering the retained tokens after eviction: attention equals
    SDPA over keys rotated at their ORIGINAL positions (vanilla scheme)."""
    rng = np.random.default_rng(14)
    base = 10000.0
    c = OracleCache(_cfg(batch=1, n_kv_heads=1, n_q_heads=1, n_sink=4, window=64,
                         evict_window=64, rope_base=base, max_tokens=160))
    ks, vs = [], []
    for t in range(300):
        k, v = _f16(rng, (1, 1, 1, 64)), _f16(rng, (1, 1, 1, 64))
        ks.append(k)
        vs.append(v)
        c.append(0, k, v)
        c.evict(0)
    q = _f16(rng, (1, 1, 64))
    out, _ = c.decode_attn(0, q)
    keep = list(range(4)) + list(range(300 - 64, 300))
    K = np.concatenate([rope.rotate_keys(ks[p], p, base, "f16")[0, 0] for p in keep])
    V = np.concatenate([vs[p][0, 0] for p in keep])
    qr = rope.rotate(q[:, :, None, :], [299], base)[0, 0, 0]
    assert np.allclose(out[0, 0], _sdpa64(qr, K, V), rtol=1e-6, atol=1e-7)


def test_turboquant_cache_attention_quality():
    """TQ attention tracks exact attention (cosine near the page's figures)."""
    from bit_kv_cache_append_gb300 import workloads as W
    w = W.scaled(W.WORKLOADS["turboquant_k4v4"], batch=1, n_kv_heads=2, n_q_heads=8, context=1024)
    k, v = W.kv_tokens(w, 5, 1024)
    q = W.queries(w, 5)
    c = OracleCache(_cfg(batch=1, n_kv_heads=2, n_q_heads=8, head_dim=128, mode="turboquant",
                         k_bits=4, v_bits=4, seed=5))
    c.prefill_quantize(0, k, v)
    out, _ = c.decode_attn(0, q)
    cos = []
    for j in range(8):
        ref = _sdpa64(q[0, j], k[0, j // 4], v[0, j // 4])
        cos.append(np.dot(out[0, j], ref) / (np.linalg.norm(out[0, j]) * np.linalg.norm(ref)))
    assert np.mean(cos) > 0.97


# ------------------------------------------------------------------ RoPE re-positioning

def _ring_stream(reposition, n_sink, T=300, keep=96, D=128, seed=0, zero_rows=False):
    """One sequence streamed token by token with eviction after each append
    (StreamingLLM ring), RoPE base 10000, K8/V8."""
    c = OracleCache(_cfg(batch=1, n_kv_heads=1, n_q_heads=1, head_dim=D, k_bits=8, v_bits=8,
                         n_sink=n_sink, evict_window=keep, rope_base=10000.0, rope_reposition=reposition,
                         max_tokens=keep + 64))
    rng = np.random.default_rng(seed)
    for t in range(T):
        if zero_rows:
            k = np.zeros((1, 1, 1, D), np.float32)
            v = np.zeros((1, 1, 1, D), np.float32)
            if t == 0:
                k[0, 0, 0, 0] = 1.0      # the one sink: e_0 (unchanged by RoPE at position 0)
                v[0, 0, 0, 1] = 1.0
        else:
            k, v = _f16(rng, (1, 1, 1, D)), _f16(rng, (1, 1, 1, D))
        c.append(0, k, v)
        c.evict(0)
    return c


def test_reposition_closed_form_single_sink():
    """StreamingLLM "RoPE caveat": with re-positioning the query sits at its
    cache slot N_s + (L - 1 - E) = keep instead of L - 1. One sink key e_0,
    every other key and value zero, q = 8 e_0: the sink score is
    8 cos(pos * theta_0) / sqrt(D) with theta_0 = 1, the others 0, so
    out[1] = e^s / (e^s + n - 1) and every other channel is 0."""
    import math
    T, keep, D = 300, 96, 128
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 8.0
    for reposition, qpos in ((False, T - 1), (True, keep)):
        c = _ring_stream(reposition, 1, T, keep, D, zero_rows=True)
        assert c.layers[0].E == T - keep
        n = 1 + keep                       # the sink and the kept window
        s = 8.0 * math.cos(qpos) / math.sqrt(D)
        out, _ = c.decode_attn(0, q)
        assert abs(float(out[0, 0, 1]) - math.exp(s) / (math.exp(s) + n - 1)) < 1e-6
        assert np.all(np.delete(out[0, 0], 1) == 0.0)


def test_reposition_is_vanilla_without_eviction_or_sinks():
    """Until something is evicted every cache slot is the absolute position,
    and with no sinks every kept key and the query move by the same offset:
    both give the vanilla output (relative rotations are all that attention
    sees)."""
    rng = np.random.default_rng(5)
    q = _f16(rng, (1, 1, 128))
    for n_sink, T in ((4, 80), (0, 300)):
        a = _ring_stream(False, n_sink, T, seed=7)
        b = _ring_stream(True, n_sink, T, seed=7)
        assert (a.layers[0].E > n_sink) == (T > 96)
        oa, _ = a.decode_attn(0, q)
        ob, _ = b.decode_attn(0, q)
        assert np.allclose(oa, ob, rtol=1e-5, atol=1e-6)
    # with sinks and eviction the sinks' distance changes, and so does the output
    a = _ring_stream(False, 4, 300, seed=7)
    b = _ring_stream(True, 4, 300, seed=7)
    assert not np.allclose(a.decode_attn(0, q)[0], b.decode_attn(0, q)[0], rtol=1e-3)


# ------------------------------------------------------------------ K before RoPE

def test_pre_rope_codes_do_not_turn_with_the_position():
    """posttrainllm "StreamingLLM + KIVI", "Caveats": K quantised before RoPE
    sees a per-channel basis that does not turn with the position. The same
    rows appended at position 0 or at 1024 get identical codes, scales and
    zeros with k_pre_rope, and different ones with RoPE baked in."""
    rng = np.random.default_rng(3)
    xk, xv = _f16(rng, (1, 2, 64, 64)), _f16(rng, (1, 2, 64, 64))
    filler = _f16(rng, (1, 2, 1024, 64))
    for pre in (True, False):
        kw = dict(batch=1, n_kv_heads=2, n_q_heads=2, head_dim=64, rope_base=10000.0, k_pre_rope=pre,
                  max_tokens=2048)
        a, b = OracleCache(_cfg(**kw)), OracleCache(_cfg(**kw))
        a.append(0, xk, xv)
        b.append(0, filler, filler)
        b.append(0, xk, xv)
        ea, eb = a.export(0), b.export(0)
        same_codes = np.array_equal(ea["k_codes"], eb["k_codes"][:, :, 1024:])
        same_scales = np.array_equal(ea["k_scale"].view(np.uint16), eb["k_scale"][:, :, 32:].view(np.uint16))
        assert same_codes == pre and same_scales == pre
        assert np.array_equal(ea["v_codes"], eb["v_codes"][:, :, 1024:])   # V never rotates


def _one_pair_cache(pre, reposition, n_sink, keep, T, a_q=6.0, b_k=1.0, D=64):
    """T tokens whose keys are b e_0 (the first RoPE pair, theta_0 = 1) and
    whose values are zero except the first token's (e_1), streamed one by one
    with eviction (every kept row exact: the window is the kept span);
    returns the cache and q = a e_0."""
    c = OracleCache(_cfg(batch=1, n_kv_heads=1, n_q_heads=1, head_dim=D, k_bits=8, v_bits=8,
                         n_sink=n_sink, window=keep or 4096, evict_window=keep, rope_base=10000.0,
                         rope_reposition=reposition, k_pre_rope=pre, max_tokens=4096 + 64))
    for t in range(T):
        k = np.zeros((1, 1, 1, D), np.float32)
        v = np.zeros((1, 1, 1, D), np.float32)
        k[0, 0, 0, 0] = b_k
        if t == 0:
            v[0, 0, 0, 1] = 1.0
        c.append(0, k, v)
        c.evict(0)
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = a_q
    return c, q


def test_pre_rope_scores_follow_the_relative_rotation():
    """Keys rotated on read: a key d positions behind the query meets it
    rotated by d theta_0 in the first pair, so with q = a e_0 and every key
    b e_0 its score is a b cos(d) / sqrt(D), whatever the absolute position
    (all rows exact: the window covers them). The first token's value is e_1,
    so out[1] is its softmax weight: e^s0 / sum_p e^sp."""
    D, T, a, b = 64, 40, 6.0, 1.0
    c, q = _one_pair_cache(True, False, 0, 0, T, a, b, D)
    s = [a * b * math.cos(T - 1 - p) / math.sqrt(D) for p in range(T)]
    w0 = math.exp(s[0]) / sum(math.exp(x) for x in s)
    out, _ = c.decode_attn(0, q)
    assert abs(float(out[0, 0, 1]) - w0) < 1e-6
    assert np.all(np.delete(out[0, 0], 1) == 0.0)


def test_pre_rope_reposition_closed_form_after_eviction():
    """"True" re-positioning (posttrainllm "RoPE caveat": store K pre-RoPE and
    rotate at the compressed index): after eviction the sink keeps slot 0,
    the kept tokens slots 1 .. keep and the query slot keep; each score is
    a b cos(slot_q - slot) / sqrt(D). The first token is the sink (value
    e_1). Without re-positioning the sink sits T - 1 back."""
    D, T, keep, a, b = 64, 200, 48, 6.0, 1.0
    for reposition in (True, False):
        c, q = _one_pair_cache(True, reposition, 1, keep, T, a, b, D)
        assert c.layers[0].E == T - keep
        kept = [0] + list(range(T - keep, T))            # absolute positions still read
        if reposition:
            slots = [0] + list(range(1, keep + 1))
            qslot = keep
        else:
            slots, qslot = kept, T - 1
        s = [a * b * math.cos(qslot - sl) / math.sqrt(D) for sl in slots]
        w0 = math.exp(s[0]) / sum(math.exp(x) for x in s)
        out, _ = c.decode_attn(0, q)
        assert abs(float(out[0, 0, 1]) - w0) < 1e-6


def test_pre_rope_rules():
    with pytest.raises(ValueError):
        OracleCache(_cfg(k_pre_rope=True))                                   # needs RoPE in the cache
    with pytest.raises(ValueError):
        OracleCache(_cfg(k_pre_rope=True, rope_base=10000.0, mode="turboquant"))
    with pytest.raises(ValueError):
        OracleCache(_cfg(k_pre_rope=True, rope_base=10000.0, n_dyn_sinks=3))
