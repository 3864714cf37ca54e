"""The failure path of the device waits, made to run out on purpose.

Every wait of the decode kernels (a staged copy landing, a hand-off between
warps) is bounded: after its cycle budget it gives up, raises the CTA's abort
flag so the other warps give up too, and sets the cache's device error flag,
which kv_cache_check_device_error reports as KV_ERR_TIMEOUT. No GPU fault or
hang is involved: the hook waits on mbarriers that nothing arrives at and on
which no copy is pending, with a short budget, and returns.
"""
import numpy as np
import pytest

from bit_kv_cache_append_gb300 import workloads as W
from tests.parity import cache_kwargs, compare_attention, torch_act

pytestmark = pytest.mark.gpu


def test_bounded_waits_give_up_and_the_cache_stays_usable():
    import torch
    from bit_kv_cache_append_gb300.binding import KV_ERR_TIMEOUT, KVCache, KVError
    from oracle import OracleCache
    from tests.parity import oracle_config
    w = W.WORKLOADS["tiny"]
    kw = cache_kwargs(w, w.context)
    gc, oc = KVCache(**kw), OracleCache(oracle_config(kw))
    k, v = W.kv_tokens(w, 31, 300)
    gc.prefill_quantize(0, torch_act(k, w.act_dtype), torch_act(v, w.act_dtype))
    oc.prefill_quantize(0, k, v)
    q = W.queries(w, 31)
    before = gc.decode_attn(0, torch_act(q, w.act_dtype)).cpu().numpy()
    gc.check_device_error()

    budget = 2_000_000  # SM clock cycles, about a millisecond
    res = gc.test_bounded_wait(budget)
    assert res[:4] == [0, 0, 0, 0], res        # every wait gave up
    # the second warp (default budget, about 2^31 cycles) left through the
    # abort flag shortly after the first warp's budget ran out
    assert budget // 2 < res[4] < 64 * budget, res
    with pytest.raises(KVError) as e:
        gc.check_device_error()
    assert e.value.status == KV_ERR_TIMEOUT
    gc.check_device_error()                     # reading the flag cleared it

    after = gc.decode_attn(0, torch_act(q, w.act_dtype)).cpu().numpy()
    gc.check_device_error()
    assert np.array_equal(before.view(np.uint32), after.view(np.uint32))
    ref, _ = oc.decode_attn(0, q)
    compare_attention(after, ref)
    torch.cuda.synchronize()


def test_bounded_wait_rejects_budgets_out_of_range():
    from bit_kv_cache_append_gb300.binding import KV_ERR_INVALID_ARG, KVCache, KVError
    w = W.WORKLOADS["tiny"]
    gc = KVCache(**cache_kwargs(w, w.context))
    for bad in (0, 999, (1 << 31) + 1):
        with pytest.raises(KVError) as e:
            gc.test_bounded_wait(bad)
        assert e.value.status == KV_ERR_INVALID_ARG
