"""Full-size workloads in the launch configuration bench.py times: every
code, scale and zero bit-exact against the oracle, and attention checked on
sampled (sequence, query head) pairs the oracle computes one by one."""
import numpy as np
import pytest

from bit_kv_cache_append_gb300 import workloads as W
from tests.parity import cache_kwargs, compare_attention, compare_exports, oracle_config, torch_act

pytestmark = pytest.mark.gpu


def _sample_heads(B, Hq, n, seed):
    r = np.random.default_rng(seed)
    return sorted({(int(r.integers(B)), int(r.integers(Hq))) for _ in range(n)})


def test_llama8b_full_size():
    """Llama-3-8B-shaped decode at 32K: prefill 32767 tokens, append 1,
    decode (the bench's workload and launch configuration)."""
    import torch
    from bit_kv_cache_append_gb300.binding import KVCache
    from oracle import OracleCache
    w = W.WORKLOADS["llama8b"]
    kw = cache_kwargs(w, w.context + 64)
    gc, oc = KVCache(**kw), OracleCache(oracle_config(kw))
    k, v = W.kv_tokens(w, 2024, w.context - 1)
    gc.prefill_quantize(0, torch_act(k, "bf16"), torch_act(v, "bf16"))
    oc.prefill_quantize(0, k, v)
    del k, v
    k1, v1 = W.kv_tokens(w, 2024, 1, first_pos=w.context - 1)
    gc.append(0, torch_act(k1, "bf16"), torch_act(v1, "bf16"))
    oc.append(0, k1, v1)
    compare_exports(gc, oc, 0)
    q = W.queries(w, 2024)
    out = gc.decode_attn(0, torch_act(q, "bf16"))
    torch.cuda.synchronize()
    gc.check_device_error()
    heads = _sample_heads(w.batch, w.n_q_heads, 12, 1)
    o_ref, _ = oc.decode_attn(0, q, heads=heads)
    compare_attention(out.cpu().numpy(), o_ref, heads)


def test_kvsink_full_size_selection():
    """131072-token prefill with five planted 25x sinks per sequence: the
    selected set, the sink rows, the masks and all codes bit-exact."""
    import torch
    from bit_kv_cache_append_gb300.binding import KVCache
    from oracle import OracleCache
    w = W.WORKLOADS["kvsink"]
    kw = cache_kwargs(w, w.context + 64)
    gc, oc = KVCache(**kw), OracleCache(oracle_config(kw))
    k, v = W.kv_tokens(w, 77, w.context)
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k, v)
    del k, v
    assert np.array_equal(gc.export(0, "sink_pos"), W.sink_positions(77, w.batch, w.context))
    compare_exports(gc, oc, 0)
    q = W.queries(w, 77)
    out = gc.decode_attn(0, torch_act(q, "f16"))
    torch.cuda.synchronize()
    heads = _sample_heads(w.batch, w.n_q_heads, 4, 2)
    o_ref, _ = oc.decode_attn(0, q, heads=heads)
    compare_attention(out.cpu().numpy(), o_ref, heads)


def test_turboquant_full_size_sampled_sequences():
    """TurboQuant K4/V2 at full size (batch 32, 8 KV heads, 16384 tokens,
    AR(1) channels): the GPU holds every sequence; the oracle takes three
    sampled sequences (the sequences are independent), whose codes and
    norms must match bit for bit and whose attention is compared."""
    import torch
    from bit_kv_cache_append_gb300.binding import KVCache
    from oracle import OracleCache
    w = W.WORKLOADS["turboquant_k4v2"]
    bs = [0, 13, 31]
    kw = cache_kwargs(w, w.context + 64, seed=99)
    gc = KVCache(**kw)
    oc = OracleCache(oracle_config(dict(kw, batch=len(bs))))
    k, v = W.kv_tokens(w, 31, w.context - 1)
    gc.prefill_quantize(0, torch_act(k, "f16"), torch_act(v, "f16"))
    oc.prefill_quantize(0, k[bs], v[bs])
    del k, v
    k1, v1 = W.kv_tokens(w, 31, 1, first_pos=w.context - 1)
    gc.append(0, torch_act(k1, "f16"), torch_act(v1, "f16"))
    oc.append(0, k1[bs], v1[bs])
    ref = oc.export(0)
    for name in ("k_codes", "k_norm", "v_codes", "v_norm"):
        got = gc.export(0, name)[bs]
        want = ref[name]
        if name.endswith("norm"):
            got, want = got.view(np.uint32), want.astype(np.float32).view(np.uint32)
        assert got.shape == want.shape, (name, got.shape, want.shape)
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{name}: {len(bad)} mismatches, first at {bad[:5].tolist()}"
    q = W.queries(w, 31)
    out = gc.decode_attn(0, torch_act(q, "f16"))
    torch.cuda.synchronize()
    gc.check_device_error()
    heads = [(i, hq) for i in range(len(bs)) for hq in (0, 9, 22, 31)]
    o_ref, _ = oc.decode_attn(0, q[bs], heads=heads)
    got = out.cpu().numpy()[bs]
    compare_attention(got, o_ref, heads)
