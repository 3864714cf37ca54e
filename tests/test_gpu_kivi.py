"""GPU parity of the KIVI path (append, prefill, overlay, decode) against the
oracle, through the C ABI."""
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
    lse = torch.empty(out.shape[:2], dtype=torch.float32, device=out.device)
    out2 = gc.decode_attn(layer, torch_act(q, act), lse=lse)
    torch.cuda.synchronize()
    gc.check_device_error()
    o_ref, l_ref = oc.decode_attn(layer, q, heads=heads)
    res = compare_attention(out.cpu().numpy(), o_ref, heads)
    assert np.array_equal(out.cpu().numpy(), out2.cpu().numpy())   # deterministic
    lg = lse.cpu().numpy()
    if heads is None:
        assert np.allclose(lg, l_ref, atol=2e-4, rtol=1e-5)
    return res


def test_tiny_one_at_a_time_and_prefill():
    """Tiny workload: 512 appends one at a time, decode; then the same tokens
    as one prefill give identical codes."""
    w = W.WORKLOADS["tiny"]
    k, v = W.kv_tokens(w, 11, 512)
    kw = cache_kwargs(w, 512)
    gc, oc = _pair(kw)
    for t in range(512):
        gc.append(0, torch_act(k[:, :, t:t + 1], w.act_dtype), torch_act(v[:, :, t:t + 1], w.act_dtype))
        oc.append(0, k[:, :, t:t + 1], v[:, :, t:t + 1])
        if t in (0, 3, 4, 31, 32, 63, 100, 447, 448, 511):
            _decode_both(gc, oc, 0, W.queries(w, 11, t), w.act_dtype)
    compare_exports(gc, oc, 0)
    gp, _ = _pair(kw)
    gp.prefill_quantize(0, torch_act(k, w.act_dtype), torch_act(v, w.act_dtype))
    compare_exports(gp, oc, 0)


@pytest.mark.parametrize("kb,vb,act", [(2, 4, "bf16"), (2, 2, "f16"), (4, 4, "f16"), (8, 8, "bf16"),
                                       (4, 2, "bf16"), (2, 8, "f16"), (8, 4, "f16"),
                                       (3, 3, "f16"), (3, 2, "bf16"), (2, 3, "f16"), (8, 3, "bf16"),
                                       (3, 4, "bf16"), (4, 3, "f16"), (3, 8, "f16")])
@pytest.mark.parametrize("D,H,Hq", [(128, 8, 32), (64, 4, 8), (128, 2, 2)])
def test_prefill_then_appends(kb, vb, act, D, H, Hq):
    """Several tiles and a ragged tail: prefill 1000 tokens, then 45 appends
    of mixed sizes; codes bit-exact, attention within tolerance."""
    w = W.scaled(W.WORKLOADS["llama8b"], batch=2, n_kv_heads=H, n_q_heads=Hq, head_dim=D, context=2048,
                 k_bits=kb, v_bits=vb, act_dtype=act)
    kw = cache_kwargs(w, 2048)
    gc, oc = _pair(kw)
    k, v = W.kv_tokens(w, 5, 1000)
    gc.prefill_quantize(0, torch_act(k, act), torch_act(v, act))
    oc.prefill_quantize(0, k, v)
    _decode_both(gc, oc, 0, W.queries(w, 5, 0), act)
    pos = 1000
    for i, n in enumerate([1, 1, 3, 31, 1, 32, 1, 7, 64, 1] * 4 + [1] * 5):
        k, v = W.kv_tokens(w, 5, n, first_pos=pos)
        gc.append(0, torch_act(k, act), torch_act(v, act))
        oc.append(0, k, v)
        pos += n
        if i % 9 == 0:
            _decode_both(gc, oc, 0, W.queries(w, 5, i), act)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 5, 99), act)


@pytest.mark.parametrize("L", [1, 3, 4, 5, 31, 32, 33, 64, 100, 131])
def test_short_contexts_and_overlay_edges(L):
    """Contexts shorter than the sinks, the window, one group: every pool
    boundary."""
    w = W.scaled(W.WORKLOADS["tiny"], batch=2)
    kw = cache_kwargs(w, 256)
    gc, oc = _pair(kw)
    k, v = W.kv_tokens(w, 7, L)
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 7), "f16")


@pytest.mark.parametrize("n_sink,window", [(0, 0), (0, 1000), (32, 0), (1, 33), (7, 200)])
def test_overlay_variants(n_sink, window):
    w = W.scaled(W.WORKLOADS["tiny"], batch=2, n_sink=n_sink, window=window)
    kw = cache_kwargs(w, 512)
    gc, oc = _pair(kw)
    k, v = W.kv_tokens(w, 8, 333)
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 8), "f16")


def test_split_count_invariance():
    """The LSE merge makes the result independent of the partition count."""
    import torch
    w = W.scaled(W.WORKLOADS["llama8b"], batch=2, context=4096)
    outs = []
    k, v = W.kv_tokens(w, 9, 3000)
    q = torch_act(W.queries(w, 9), "bf16")
    for ms in (1, 3, 64):
        kw = cache_kwargs(w, 4096, max_splits=ms)
        gc, _ = _pair(kw)
        gc.prefill_quantize(0, torch_act(k, "bf16"), torch_act(v, "bf16"))
        outs.append(gc.decode_attn(0, q).cpu().numpy())
    torch.cuda.synchronize()
    # the weights enter the value products as f16 (11 significant bits) taken
    # relative to each partition's own running max, so partitionings agree
    # to a few 1e-4 (relative rounding of at most 2^-11 twice per term); a
    # wrong log-sum-exp merge shows as an O(1) difference
    for o in outs[1:]:
        d = np.linalg.norm(o - outs[0]) / np.linalg.norm(outs[0])
        assert d < 5e-4


def test_constant_and_extreme_groups():
    """Constant channels (eps scale), tiny ranges and outliers: codes exact."""
    w = W.scaled(W.WORKLOADS["tiny"], batch=1, n_sink=0, window=0)
    kw = cache_kwargs(w, 256)
    gc, oc = _pair(kw)
    k, v = W.kv_tokens(w, 10, 128)
    k[:, :, :, 3] = 0.5
    k[:, :, 32:64, 7] = np.float32(np.float16(1.0 + 2 ** -10))
    k[:, :, 70, :] *= 300.0
    v[:, :, 5, :] = -2.0
    v[:, :, 9, 32:] = np.float32(np.float16(1e-4))
    k = k.astype(np.float16).astype(np.float32)
    v = v.astype(np.float16).astype(np.float32)
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 10), "f16")


def test_errors_leave_state_unchanged():
    import torch
    from bit_kv_cache_append_gb300.binding import KVCache, KVError, KV_ERR_CAPACITY, KV_ERR_STATE
    w = W.WORKLOADS["tiny"]
    gc = KVCache(**cache_kwargs(w, 64))
    q = torch_act(W.queries(w, 1), "f16")
    with pytest.raises(KVError) as e:
        gc.decode_attn(0, q)
    assert e.value.status == KV_ERR_STATE
    k, v = W.kv_tokens(w, 1, 60)
    gc.append(0, torch_act(k, "f16"), torch_act(v, "f16"))
    k, v = W.kv_tokens(w, 1, 5)
    with pytest.raises(KVError) as e:
        gc.append(0, torch_act(k, "f16"), torch_act(v, "f16"))
    assert e.value.status == KV_ERR_CAPACITY
    assert gc.stats(0)["length"] == 60
    torch.cuda.synchronize()


@pytest.mark.parametrize("n_layers", [3])
def test_layers_are_independent(n_layers):
    w = W.scaled(W.WORKLOADS["tiny"], batch=2)
    kw = cache_kwargs(w, 512, n_layers=n_layers)
    gc, oc = _pair(kw)
    for layer in range(n_layers):
        k, v = W.kv_tokens(w, 20 + layer, 100 + 37 * layer, layer=layer)
        gc.prefill_quantize(layer, torch_act(k, "f16"), torch_act(v, "f16"))
        oc.prefill_quantize(layer, k, v)
    for layer in range(n_layers):
        compare_exports(gc, oc, layer)
        _decode_both(gc, oc, layer, W.queries(w, 30 + layer), "f16")


@pytest.mark.parametrize("kb,act", [(2, "bf16"), (4, "f16")])
@pytest.mark.parametrize("D,H,Hq", [(128, 8, 32), (64, 4, 8)])
def test_v_q4_0_prefill_then_appends(kb, act, D, H, Hq):
    """V in the symmetric q4_0 form: prefill 1000 tokens (with a few rows of
    zeros and of equal-magnitude values of both signs), then appends; codes,
    scales and zeros bit-exact, attention within tolerance (the decode reads
    it as scale d, zero -8 d)."""
    w = W.scaled(W.WORKLOADS["llama8b"], batch=2, n_kv_heads=H, n_q_heads=Hq, head_dim=D, context=2048,
                 k_bits=kb, v_bits=4, act_dtype=act)
    kw = cache_kwargs(w, 2048, v_q4_0=True)
    gc, oc = _pair(kw)
    k, v = W.kv_tokens(w, 8, 1000)
    v[:, :, 10, :] = 0.0                          # d = 0: every code 8
    v[:, :, 11, :32] = 0.0
    v[:, :, 11, 3], v[:, :, 11, 7] = -2.0, 2.0    # the first extreme sets the sign; 2.0 clamps at 15
    # small nonzero slices: |m| about 1e-4 makes d an fp16 subnormal, about
    # 1e-7 rounds d to a few subnormal steps or to 0 while the values are not 0
    v[:, :, 12, :] = W.round_to_act(v[:, :, 12, :] * np.float32(1e-4), act)
    v[:, :, 13, :] = W.round_to_act(v[:, :, 13, :] * np.float32(1e-7), act)
    gc.prefill_quantize(0, torch_act(k, act), torch_act(v, act))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 8, 0), act)
    pos = 1000
    for i, n in enumerate([1, 3, 31, 1, 32, 7, 64, 1] * 2):
        k, v = W.kv_tokens(w, 8, n, first_pos=pos)
        gc.append(0, torch_act(k, act), torch_act(v, act))
        oc.append(0, k, v)
        pos += n
    compare_exports(gc, oc, 0)
    _decode_both(gc, oc, 0, W.queries(w, 8, 1), act)


@pytest.mark.parametrize("kb,vb", [(2, 2), (3, 3), (4, 4), (8, 8)])
@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_quotients_on_half_integers(kb, vb, act):
    """Values on the half-integer grid of their slice (j / 2 for j = 0 ..
    2 LB, scale 1 where the slice spans 0 .. LB), so that many quotients are
    exact half-integers and round half to even, plus values one step of the
    activation dtype on either side of a half-integer: codes bit-exact (no
    RoPE, sinks or window, so every value is quantised as given)."""
    w = W.scaled(W.WORKLOADS["tiny"], batch=2, n_kv_heads=2, n_q_heads=4, head_dim=128, n_sink=0, window=0,
                 k_bits=kb, v_bits=vb, act_dtype=act)
    kw = cache_kwargs(w, 256, rope_base=0.0)
    gc, oc = _pair(kw)
    lb = (1 << kb) - 1
    B, H, T, D = 2, 2, 96, 128
    t = np.arange(T)[:, None]
    c = np.arange(D)[None, :]
    k = ((t * 7 + c * 3) % (2 * lb + 1)).astype(np.float32) * 0.5
    k[0, :], k[1, :] = 0.0, float(lb)                     # every channel of group 0 spans 0 .. LB
    k[32, :], k[33, :] = 0.0, float(lb)
    k[64, :], k[65, :] = 0.0, float(lb)
    lv = (1 << vb) - 1
    v = ((t * 5 + c) % (2 * lv + 1)).astype(np.float32) * 0.5
    v[:, 0::32], v[:, 1::32] = 0.0, float(lv)             # every 32-channel slice spans 0 .. LB
    # one activation step either side of a half-integer on some rows
    step = np.float32(2.0 ** -7 if act == "bf16" else 2.0 ** -10)
    k[10::7, 5::11] += step * np.maximum(k[10::7, 5::11], 1.0)
    v[12::9, 7::13] -= step * np.maximum(v[12::9, 7::13], 1.0)
    k = W.round_to_act(np.broadcast_to(k, (B, H, T, D)).copy(), act)
    v = W.round_to_act(np.broadcast_to(v, (B, H, T, D)).copy(), act)
    gc.prefill_quantize(0, torch_act(k, act), torch_act(v, act))
    oc.prefill_quantize(0, k, v)
    compare_exports(gc, oc, 0)
