"""GPU parity of the StreamingLLM ring (eviction + RoPE), TurboQuant and
KVSink modes against the oracle, through the C ABI."""
import numpy as np
import pytest

from bit_kv_cache_append_gb300 import workloads as W
from tests.parity import cache_kwargs, compare_attention, compare_exports, oracle_config, torch_act

pytestmark = pytest.mark.gpu


def _pair(kw):
    from bit_kv_cache_append_gb300.binding import KVCache
    from oracle import OracleCache
    return KVCache(**kw), OracleCache(oracle_config(kw))


def _decode_both(gc, oc, layer, q, act, heads=None):
    import torch
    out = gc.decode_attn(layer, torch_act(q, act))
    torch.cuda.synchronize()
    gc.check_device_error()
    o_ref, _ = oc.decode_attn(layer, q, heads=heads)
    return compare_attention(out.cpu().numpy(), o_ref, heads)


# ------------------------------------------------------------------ ring

@pytest.mark.parametrize("pre_rope", [False, True])
@pytest.mark.parametrize("reposition", [False, True])
@pytest.mark.parametrize("name", ["ring_int8", "ring_int4"])
def test_ring_stream_with_rope_and_eviction(name, reposition, pre_rope):
    """Shortened StreamingLLM stream: 2 layers, per step append 1 -> evict ->
    decode; identical eviction ranges, codes and attention, with keys read
    at their absolute positions or re-positioned at their cache slots, and
    keys rotated before they are stored or stored before RoPE and rotated
    when read."""
    w = W.scaled(W.WORKLOADS[name], batch=4, n_kv_heads=4, n_q_heads=4, evict_window=96, n_layers=2)
    steps = 400
    kw = cache_kwargs(w, 96 + 64, rope_max_pos=steps, rope_reposition=reposition, k_pre_rope=pre_rope)
    gc, oc = _pair(kw)
    ranges_g, ranges_o = [], []
    for t in range(steps):
        for layer in range(2):
            k, v = W.kv_tokens(w, 3, 1, layer=layer, first_pos=t)
            gc.append(layer, torch_act(k, "f16"), torch_act(v, "f16"))
            oc.append(layer, k, v)
            ranges_g.append(gc.evict(layer))
            ranges_o.append(oc.evict(layer))
            if t % 37 == 5 or t == steps - 1:
                _decode_both(gc, oc, layer, W.queries(w, 3, t), "f16")
    assert ranges_g == ranges_o
    for layer in range(2):
        compare_exports(gc, oc, layer)


def test_rope_table_matches_oracle():
    from oracle import rope
    w = W.scaled(W.WORKLOADS["ring_int8"], batch=1, n_layers=1)
    gc, _ = _pair(cache_kwargs(w, 4096, rope_max_pos=70000))
    tab = gc.export(0, "rope")
    pos = [0, 1, 2, 3, 100, 4095, 4096, 65535, 69999]
    assert np.array_equal(tab[pos], rope.cos_sin(pos, 64, 10000.0))


def test_ring_capacity_requires_eviction():
    from bit_kv_cache_append_gb300.binding import KVError, KV_ERR_CAPACITY
    w = W.scaled(W.WORKLOADS["ring_int4"], batch=1, n_kv_heads=1, n_q_heads=1, evict_window=64, n_layers=1)
    gc, _ = _pair(cache_kwargs(w, 128, rope_max_pos=1000))
    for t in range(128):
        k, v = W.kv_tokens(w, 4, 1, first_pos=t)
        gc.append(0, torch_act(k, "f16"), torch_act(v, "f16"))
    with pytest.raises(KVError) as e:
        gc.append(0, torch_act(k, "f16"), torch_act(v, "f16"))
    assert e.value.status == KV_ERR_CAPACITY
    gc.evict(0)
    gc.append(0, torch_act(k, "f16"), torch_act(v, "f16"))


# ------------------------------------------------------------------ TurboQuant

@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("kb,vb", [(4, 2), (4, 4), (2, 2), (2, 4), (3, 2), (4, 3), (3, 3), (2, 3), (3, 4)])
def test_turboquant_codes_and_attention(kb, vb, D, act):
    w = W.scaled(W.WORKLOADS["turboquant_k4v2"], batch=2, n_kv_heads=2, n_q_heads=8, head_dim=D,
                 k_bits=kb, v_bits=vb, act_dtype=act)
    kw = cache_kwargs(w, 1024, seed=1234)
    gc, oc = _pair(kw)
    assert np.array_equal(gc.export(0, "tq_signs"), oc.sgn)
    for which, bits in (("codebook_k", kb), ("codebook_v", vb)):
        cb = gc.export(0, which)
        bnd, cen = oc.cb_k if which == "codebook_k" else oc.cb_v
        assert np.array_equal(cb[: (1 << bits) - 1], bnd), which
        assert np.array_equal(cb[(1 << bits) - 1:], cen), which
    k, v = W.kv_tokens(w, 6, 700)
    gc.prefill_quantize(0, torch_act(k, act), torch_act(v, act))
    oc.prefill_quantize(0, k, v)
    for i in range(5):
        k, v = W.kv_tokens(w, 6, 1 + 10 * i, first_pos=700 + i)
        gc.append(0, torch_act(k, act), torch_act(v, act))
        oc.append(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 6), act)


@pytest.mark.parametrize("D", [128, 64])
def test_turboquant_with_sinks_and_window(D):
    """TurboQuant with the exact overlay: sinks and the recent window are read
    exact (original domain) while the quantised middle is decoded in the
    rotated domain; the two parts meet in the merge."""
    w = W.scaled(W.WORKLOADS["turboquant_k4v2"], batch=2, n_kv_heads=2, n_q_heads=8, head_dim=D,
                 n_sink=4, window=40)
    gc, oc = _pair(cache_kwargs(w, 1024, seed=77))
    k, v = W.kv_tokens(w, 9, 300)
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    for i in range(6):
        k, v = W.kv_tokens(w, 9, 1 + 7 * i, first_pos=300 + i)
        gc.append(0, torch_act(k, "f16"), torch_act(v, "f16"))
        oc.append(0, k, v)
        _decode_both(gc, oc, 0, W.queries(w, 9, i), "f16")
    compare_exports(gc, oc, 0)


def test_turboquant_zero_rows():
    w = W.scaled(W.WORKLOADS["turboquant_k4v4"], batch=1, n_kv_heads=2, n_q_heads=2)
    gc, oc = _pair(cache_kwargs(w, 256))
    k, v = W.kv_tokens(w, 2, 64)
    k[:, :, 10] = 0.0
    v[:, :, 11] = 0.0
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 2), "f16")


@pytest.mark.parametrize("kb,vb,act", [(4, 2, "f16"), (3, 3, "bf16"), (2, 4, "bf16")])
@pytest.mark.parametrize("D", [128, 64])
def test_turboquant_rope_at_append(kb, vb, act, D):
    """TurboQuant with the cache applying RoPE: each key is rotated at its
    absolute position and rounded back to the activation dtype before the
    Walsh-Hadamard rotation and coding (posttrainllm "RoPE caveat"), the
    query at L - 1 before its own rotation; a prefill of 600 tokens, then
    appends of mixed sizes that start and end inside token pairs. Codes and
    norms bit-exact, attention within tolerance."""
    w = W.scaled(W.WORKLOADS["turboquant_k4v2"], batch=2, n_kv_heads=2, n_q_heads=8, head_dim=D,
                 k_bits=kb, v_bits=vb, act_dtype=act, rope_base=10000.0)
    gc, oc = _pair(cache_kwargs(w, 1024, seed=91, rope_max_pos=1024))
    k, v = W.kv_tokens(w, 15, 600)
    gc.prefill_quantize(0, torch_act(k, act), torch_act(v, act))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 15, 0), act)
    pos = 600
    for i, n in enumerate([1, 3, 31, 1, 32, 7]):
        k, v = W.kv_tokens(w, 15, n, first_pos=pos)
        gc.append(0, torch_act(k, act), torch_act(v, act))
        oc.append(0, k, v)
        pos += n
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 15, 7), act)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("kb,vb", [(4, 2), (3, 3), (2, 4)])
def test_turboquant_one_hot_rotations(kb, vb, D):
    """Rows that the rotation sends to one coordinate: x = a signs * H_r (a
    row of the Sylvester-Hadamard matrix), so y = a d e_r and u = y / n is
    +-1 up to rounding; w = (u + 1) / 2 sits at or just past 0 and 1, where
    the code is 0 or the top level. Mixed with ordinary rows; codes, norms
    and attention match the oracle."""
    w = W.scaled(W.WORKLOADS["turboquant_k4v2"], batch=2, n_kv_heads=2, n_q_heads=8, head_dim=D,
                 k_bits=kb, v_bits=vb)
    gc, oc = _pair(cache_kwargs(w, 512, seed=31))
    sgn = gc.export(0, "tq_signs").astype(np.float32)
    rng = np.random.default_rng(5)
    j = np.arange(D)
    k, v = W.kv_tokens(w, 12, 96)
    amps = np.array([1.0, 0.375, 0.8125, 0.0625], np.float32)  # the unit scale the tolerances assume
    for x in (k, v):
        for b in range(2):
            for h in range(2):
                for t in rng.choice(96, size=40, replace=False):
                    r = int(rng.integers(D))
                    hrow = np.array([1.0 if bin(r & c).count("1") % 2 == 0 else -1.0 for c in j], np.float32)
                    x[b, h, t] = rng.choice(amps) * rng.choice([-1.0, 1.0]) * sgn * hrow
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 12), "f16")


# ------------------------------------------------------------------ KVSink

@pytest.mark.parametrize("T", [4096, 1000, 37])
def test_kvsink_selection_exclusion_and_attention(T):
    w = W.scaled(W.WORKLOADS["kvsink"], batch=2, context=T)
    kw = cache_kwargs(w, 8192)
    gc, oc = _pair(kw)
    k, v = W.kv_tokens(w, 12, T)
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    if T >= 5:
        assert np.array_equal(gc.export(0, "sink_pos"), W.sink_positions(12, 2, T))
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 12), "f16")
    for i in range(40):   # decode-time appends flush groups that may hold sinks
        k, v = W.kv_tokens(w, 12, 1, first_pos=T + i)
        gc.append(0, torch_act(k, "f16"), torch_act(v, "f16"))
        oc.append(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 13), "f16")


def test_kvsink_ties_and_residual_sinks():
    """Equal key norms go to the lower position; a sink still in the residual
    is read from the tail until its group is quantised."""
    w = W.scaled(W.WORKLOADS["kvsink"], batch=1, n_kv_heads=2, n_q_heads=8, context=100)
    kw = cache_kwargs(w, 512, n_dyn_sinks=3)
    gc, oc = _pair(kw)
    rng = np.random.default_rng(0)
    k = rng.standard_normal((1, 2, 100, 128)).astype(np.float16).astype(np.float32)
    v = rng.standard_normal((1, 2, 100, 128)).astype(np.float16).astype(np.float32)
    for p in (7, 40, 70, 97):            # equal rows -> equal norms
        k[:, :, p] = 30.0
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    assert list(gc.export(0, "sink_pos")[0]) == [7, 40, 70]
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 1), "f16")


def _sink_rows_with_norms(norms, B, H, D=128, seed=0):
    """N(0,1) K/V rows (fp16 values) whose listed positions get their K row
    scaled so that its norm dominates: {pos: factor}."""
    rng = np.random.default_rng(seed)
    T = max(norms) + 1 if isinstance(norms, dict) else len(norms)
    k = rng.standard_normal((B, H, T, D)).astype(np.float16).astype(np.float32)
    v = rng.standard_normal((B, H, T, D)).astype(np.float16).astype(np.float32)
    for p, f in norms.items():
        k[:, :, p] = (k[:, :, p] * f).astype(np.float16).astype(np.float32)
    return k, v


@pytest.mark.parametrize("rope", [0.0, 10000.0])
def test_kvsink_running_admission_one_token_per_call(rope):
    """A prefill of 50 tokens leaves two of its three sinks in the open group
    (35, 45) and locks 5. Single-token calls then displace the weakest open
    sink when they beat it (55 displaces 45; 60 loses to 35); once group 1 is
    quantised every sink is locked and 70, the largest key of all, stays out.
    The set, rows, masks and codes equal the oracle's after every call, and
    attention along the way. With RoPE the key norms are taken on the keys
    rotated at their absolute positions (those of each call's tokens)."""
    import torch
    w = W.scaled(W.WORKLOADS["kvsink"], batch=2, n_kv_heads=2, n_q_heads=8, context=160, rope_base=rope)
    kw = cache_kwargs(w, 512, n_dyn_sinks=3)
    gc, oc = _pair(kw)
    k, v = _sink_rows_with_norms({5: 25.0, 35: 20.0, 45: 15.0, 55: 30.0, 60: 18.0, 70: 40.0, 159: 1.0},
                                 2, 2, seed=4)
    gc.prefill_quantize(0, torch_act(k[:, :, :50], "f16"), torch_act(v[:, :, :50], "f16"))
    oc.prefill_quantize(0, k[:, :, :50], v[:, :, :50])
    assert gc.export(0, "sink_pos").tolist() == [[5, 35, 45]] * 2
    compare_exports(gc, oc, 0)
    for t in range(50, 160):
        gc.append(0, torch_act(k[:, :, t:t + 1], "f16"), torch_act(v[:, :, t:t + 1], "f16"))
        oc.append(0, k[:, :, t:t + 1], v[:, :, t:t + 1])
        assert np.array_equal(gc.export(0, "sink_pos"), oc.export(0)["sink_pos"]), t
        if t % 23 == 0 or t in (55, 63, 64, 159):
            compare_exports(gc, oc, 0)
            _decode_both(gc, oc, 0, W.queries(w, t), "f16")
    assert gc.export(0, "sink_pos").tolist() == [[5, 35, 55]] * 2
    torch.cuda.synchronize()


@pytest.mark.parametrize("k_dyn", [1, 5])
def test_kvsink_running_admission_calls_across_groups(k_dyn):
    """Calls of random sizes (many spanning a group boundary, prefills among
    them) over planted high-norm rows whose norm grows with the position, so
    that later calls keep displacing the sinks still in an open group: sink
    sets, rows, masks and codes equal the oracle's after every call;
    attention at the end."""
    w = W.scaled(W.WORKLOADS["kvsink"], batch=2, n_kv_heads=2, n_q_heads=8, context=1200)
    kw = cache_kwargs(w, 2048, n_dyn_sinks=k_dyn)
    gc, oc = _pair(kw)
    rng = np.random.default_rng(11 + k_dyn)
    planted = {int(p): 3.0 + 27.0 * p / 1200 for p in rng.choice(1200, 60, replace=False)}
    planted[1199] = 1.0
    k, v = _sink_rows_with_norms(planted, 2, 2, seed=k_dyn)
    t = 0
    while t < 1200:
        n = int(rng.choice([1, 2, 7, 33, 45, 70, 300]))
        n = min(n, 1200 - t)
        if n >= 300:
            gc.prefill_quantize(0, torch_act(k[:, :, t:t + n], "f16"), torch_act(v[:, :, t:t + n], "f16"))
            oc.prefill_quantize(0, k[:, :, t:t + n], v[:, :, t:t + n])
        else:
            gc.append(0, torch_act(k[:, :, t:t + n], "f16"), torch_act(v[:, :, t:t + n], "f16"))
            oc.append(0, k[:, :, t:t + n], v[:, :, t:t + n])
        t += n
        compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 5), "f16")


def test_kvsink_group_of_only_sinks():
    """k = 32 with the 32 largest keys exactly filling group 0: the group is
    left as is (no non-sink row to substitute), its mask is full and every
    row of it is read exact from the sinks; then appends with larger keys
    find every sink locked."""
    import torch
    w = W.scaled(W.WORKLOADS["kvsink"], batch=2, n_kv_heads=2, n_q_heads=8, context=120)
    kw = cache_kwargs(w, 512, n_dyn_sinks=32)
    gc, oc = _pair(kw)
    k, v = _sink_rows_with_norms({p: 10.0 + p for p in range(32)} | {100: 80.0, 119: 1.0}, 2, 2, seed=6)
    gc.prefill_quantize(0, torch_act(k[:, :, :70], "f16"), torch_act(v[:, :, :70], "f16"))
    oc.prefill_quantize(0, k[:, :, :70], v[:, :, :70])
    assert gc.export(0, "sink_pos").tolist() == [list(range(32))] * 2
    assert gc.export(0, "sink_mask")[:, 0].tolist() == [0xFFFFFFFF] * 2
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 2), "f16")
    for t in range(70, 120):
        gc.append(0, torch_act(k[:, :, t:t + 1], "f16"), torch_act(v[:, :, t:t + 1], "f16"))
        oc.append(0, k[:, :, t:t + 1], v[:, :, t:t + 1])
    assert gc.export(0, "sink_pos").tolist() == [list(range(32))] * 2
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 3), "f16")
    torch.cuda.synchronize()


@pytest.mark.parametrize("kb,vb,act", [(2, 4, "bf16"), (4, 4, "f16"), (3, 8, "bf16"), (8, 2, "f16")])
@pytest.mark.parametrize("D", [128, 64])
def test_pre_rope_prefill_then_appends(kb, vb, act, D):
    """Keys stored before RoPE (posttrainllm "RoPE caveat"): prefill 1000
    tokens, then appends of mixed sizes, with a sink overlay and a window;
    codes, scales and zeros (the stored, un-rotated keys) bit-exact and
    attention, with every key rotated on read, within tolerance."""
    w = W.scaled(W.WORKLOADS["llama8b"], batch=2, n_kv_heads=2, n_q_heads=8, head_dim=D, context=2048,
                 k_bits=kb, v_bits=vb, act_dtype=act, n_sink=4, window=40, rope_base=10000.0)
    kw = cache_kwargs(w, 2048, rope_max_pos=2048, k_pre_rope=True)
    gc, oc = _pair(kw)
    k, v = W.kv_tokens(w, 12, 1000)
    gc.prefill_quantize(0, torch_act(k, act), torch_act(v, act))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 12, 0), act)
    pos = 1000
    for i, n in enumerate([1, 3, 31, 1, 32, 7, 64, 1]):
        k, v = W.kv_tokens(w, 12, n, first_pos=pos)
        gc.append(0, torch_act(k, act), torch_act(v, act))
        oc.append(0, k, v)
        pos += n
        if i % 3 == 2:
            _decode_both(gc, oc, 0, W.queries(w, 12, pos), act)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 12, 99), act)


@pytest.mark.parametrize("kb,vb,act", [(2, 4, "bf16"), (3, 3, "f16"), (8, 8, "bf16"), (4, 2, "bf16"), (2, 3, "f16")])
@pytest.mark.parametrize("D", [128, 64])
def test_rope_at_append_prefill_then_appends(kb, vb, act, D):
    """Keys rotated when appended (posttrainllm "RoPE caveat": each key keeps
    the rotation of its absolute position, rounded back to the activation
    dtype): a prefill of 1000 tokens, whose groups are quantised from the
    rotated rows in one pass, then appends of mixed sizes whose groups are
    completed from the tail ring; codes, scales and zeros bit-exact,
    attention within tolerance."""
    w = W.scaled(W.WORKLOADS["llama8b"], batch=2, n_kv_heads=2, n_q_heads=8, head_dim=D, context=2048,
                 k_bits=kb, v_bits=vb, act_dtype=act, n_sink=4, window=40, rope_base=10000.0)
    kw = cache_kwargs(w, 2048, rope_max_pos=2048)
    gc, oc = _pair(kw)
    k, v = W.kv_tokens(w, 14, 1000)
    gc.prefill_quantize(0, torch_act(k, act), torch_act(v, act))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 14, 0), act)
    pos = 1000
    for i, n in enumerate([1, 3, 31, 1, 32, 7, 64, 1]):
        k, v = W.kv_tokens(w, 14, n, first_pos=pos)
        gc.append(0, torch_act(k, act), torch_act(v, act))
        oc.append(0, k, v)
        pos += n
        if i % 3 == 2:
            _decode_both(gc, oc, 0, W.queries(w, 14, pos), act)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 14, 99), act)
