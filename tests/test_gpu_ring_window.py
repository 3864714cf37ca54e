"""GPU parity of the StreamingLLM ring at its real retention window.

The ring workload keeps sink 4 + a 4096-token window (posttrainllm
"StreamingLLM + KIVI", "StreamingLLM - Implementation": after each per-layer
append drop [sink, len - window)). Eviction is logical: quantised groups live
in a ring of group slots, so once the stream passes the ring's capacity the
stored groups wrap from the last slot to the first. The decode kernel stages
runs of two consecutive groups with one bulk copy when their slots are
adjacent and with one copy per group when the run crosses the wrap; these
tests stream far enough past the wrap, with a stream-K grid small enough that
every CTA walks long runs, that the second form is taken, and check codes,
eviction ranges and attention against the oracle.
"""
import os

import numpy as np
import pytest

from bit_kv_cache_append_gb300 import workloads as W
from tests.parity import cache_kwargs, compare_attention, compare_exports, oracle_config, torch_act

GROUP = 32
PAIRS = 4        # warp pairs of a decode CTA
RUN = 2          # groups per staged run (chunks up to 6 KB)
FEW_CTAS = 4     # stream-K CTAs of the second cache


def _cache_with_ctas(kw, n_ctas):
    """A library cache whose decode uses `n_ctas` stream-K CTAs (read from
    the environment when the cache is created)."""
    from bit_kv_cache_append_gb300.binding import KVCache
    old = os.environ.get("KVQ_STREAM_CTAS")
    os.environ["KVQ_STREAM_CTAS"] = str(n_ctas)
    try:
        return KVCache(**kw)
    finally:
        if old is None:
            del os.environ["KVQ_STREAM_CTAS"]
        else:
            os.environ["KVQ_STREAM_CTAS"] = old


def wrapped_runs(units, n_groups, g_begin, n_slots, n_ctas):
    """Runs of two groups whose first chunk sits in the ring's last slot (so
    the run's chunks are not adjacent), under the decode's stream-K walk:
    the units' groups form one flat list cut into n_ctas equal ranges; inside
    a range, per unit, warp pair p takes the runs starting at the unit's first
    item in the range + RUN p + RUN PAIRS k."""
    work = units * n_groups
    hits = 0
    for c in range(n_ctas):
        i0, i1 = c * work // n_ctas, (c + 1) * work // n_ctas
        s = i0
        while s < i1:
            u = s // n_groups
            e = min((u + 1) * n_groups, i1)
            for item in range(s, e, RUN):
                grp = g_begin + item - u * n_groups
                if e - item >= RUN and grp % n_slots == n_slots - 1:
                    hits += 1
            s = e
    return hits


@pytest.mark.gpu
@pytest.mark.parametrize("reposition", [False, True])
@pytest.mark.parametrize("name", ["ring_int8", "ring_int4"])
def test_ring_full_window_across_the_slot_wrap(name, reposition):
    """head_dim 64, MHA 8 heads, sink 4, evict_window 4096, RoPE base 10000,
    2 layers, batch 2: prefill 4000 tokens, then per step append one token ->
    evict -> decode (every 23 steps) up to 4420 tokens. The group-slot ring
    holds 130 groups, so the stored groups wrap from about 4160 tokens on.
    Two library caches take the same stream: one with the default grid and
    one with 4 stream-K CTAs, whose runs cross the wrap."""
    from oracle import OracleCache
    w = W.scaled(W.WORKLOADS[name], batch=2, n_layers=2)
    n_pre, n_end = 4000, 4420
    kw = cache_kwargs(w, 4096 + 64, rope_max_pos=n_end, rope_reposition=reposition)
    caches = [_cache_with_ctas(kw, 0), _cache_with_ctas(kw, FEW_CTAS)]
    oc = OracleCache(oracle_config(kw))
    n_slots = (kw["max_tokens"] + GROUP - 1) // GROUP
    units = w.batch * w.n_kv_heads
    hits = 0
    for layer in range(2):
        k, v = W.kv_tokens(w, 21, n_pre, layer=layer)
        for gc in caches:
            gc.prefill_quantize(layer, torch_act(k, "f16"), torch_act(v, "f16"))
        oc.prefill_quantize(layer, k, v)
    ranges_g, ranges_o = [[], []], []
    for t in range(n_pre, n_end):
        for layer in range(2):
            k, v = W.kv_tokens(w, 21, 1, layer=layer, first_pos=t)
            for i, gc in enumerate(caches):
                gc.append(layer, torch_act(k, "f16"), torch_act(v, "f16"))
                ranges_g[i].append(gc.evict(layer))
            oc.append(layer, k, v)
            ranges_o.append(oc.evict(layer))
            if (t - n_pre) % 23 == 22 or t == n_end - 1:
                q = W.queries(w, 21, t)
                ref, _ = oc.decode_attn(layer, q)
                for gc in caches:
                    out = gc.decode_attn(layer, torch_act(q, "f16"))
                    gc.check_device_error()
                    compare_attention(out.cpu().numpy(), ref)
                st = oc.layers[layer]
                lo, F = max(w.n_sink, st.E), oc.fp16_begin(layer)
                g_begin = lo // GROUP
                hits += wrapped_runs(units, (F + GROUP - 1) // GROUP - g_begin, g_begin, n_slots, FEW_CTAS)
    assert hits > 0, "no decode staged a run across the slot wrap"
    assert ranges_g[0] == ranges_o and ranges_g[1] == ranges_o
    for layer in range(2):
        for gc in caches:
            compare_exports(gc, oc, layer)


def test_wrapped_runs_counts_a_known_case():
    """The coverage count itself, on a hand-checked case: one unit of 6
    groups starting at group 3 in a ring of 5 slots, one CTA: runs start at
    items 0, 2, 4 (groups 3, 5, 7; slots 3, 0, 2); none starts in slot 4.
    Starting at group 4 instead: runs at groups 4, 6, 8 (slots 4, 1, 3): one."""
    assert wrapped_runs(1, 6, 3, 5, 1) == 0
    assert wrapped_runs(1, 6, 4, 5, 1) == 1
    # a run cut short by the end of the unit is a single group: not counted
    assert wrapped_runs(1, 5, 0, 5, 1) == 0
