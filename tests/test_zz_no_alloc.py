"""kv_decode_attn_noalloc, the decode entry point that allocates nothing.

It serves callers that may not allocate device memory while decoding (a
serving loop whose memory pool already holds the whole GPU, a plug-in whose
host framework hands it no allocator, a loop that cannot take the device-wide
synchronisation of cudaMalloc / cudaFree): its split partials sit in a fixed
32 MiB block that the library declares. These tests check, through the C ABI,
that two calls in a row give exactly what kv_decode_attn gives on the same
cache (the same kernels run the same deterministic schedule; only the
address of the partials differs, so the outputs must be equal bit for bit),
and that a cache whose partials exceed the block is refused before any
launch.
The file is named to be collected last.
"""
import numpy as np
import pytest

from bit_kv_cache_append_gb300 import workloads as W
from tests.parity import cache_kwargs, torch_act

pytestmark = pytest.mark.gpu


def _same(a, b):
    """Bit-for-bit equality of two float32 arrays."""
    assert a.shape == b.shape
    bad = np.argwhere(a.view(np.uint32) != b.view(np.uint32))
    assert bad.size == 0, f"{len(bad)} elements differ, first at {bad[:5].tolist()}"


def _both(gc, q, act):
    """Output and lse of kv_decode_attn, then of kv_decode_attn_noalloc into
    freshly poisoned buffers."""
    import torch
    c = gc.cfg
    lse_ref = torch.empty((c.batch, c.n_q_heads), dtype=torch.float32, device="cuda")
    ref = gc.decode_attn(0, torch_act(q, act), lse=lse_ref)
    out = torch.full_like(ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    gc.decode_attn_noalloc(0, torch_act(q, act), out, lse=lse)
    torch.cuda.synchronize()
    gc.check_device_error()
    return ref.cpu().numpy(), lse_ref.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("name,n0", [("llama8b", 3000), ("turboquant_k4v4", 1500)])
def test_noalloc_matches_decode_twice(name, n0):
    """Two calls in a row, with an append between them, give output and lse
    identical to kv_decode_attn's."""
    from bit_kv_cache_append_gb300.binding import KVCache
    w = W.scaled(W.WORKLOADS[name], batch=4, context=4096)
    k, v = W.kv_tokens(w, 5, n0 + 40)
    gc = KVCache(**cache_kwargs(w, 4096))
    gc.prefill_quantize(0, torch_act(k[:, :, :n0], w.act_dtype), torch_act(v[:, :, :n0], w.act_dtype))
    for call, t in enumerate((n0, n0 + 40)):
        if call:
            gc.append(0, torch_act(k[:, :, n0:t], w.act_dtype), torch_act(v[:, :, n0:t], w.act_dtype))
        ref, lse_ref, out, lse = _both(gc, W.queries(w, 7 + call, t), w.act_dtype)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        _same(out, ref)
        _same(lse, lse_ref)


def test_noalloc_rejects_oversized_partials():
    """batch 64 x 32 query heads x 65 slots x 130 floats is about 69 MB of
    partials: refused with KV_ERR_CAPACITY, the output left untouched, and
    the next in-limit call still works."""
    import torch
    from bit_kv_cache_append_gb300.binding import KV_ERR_CAPACITY, KVCache, KVError
    w = W.scaled(W.WORKLOADS["llama8b"], batch=64, context=64)
    k, v = W.kv_tokens(w, 3, 40)
    gc = KVCache(**cache_kwargs(w, 64))
    gc.append(0, torch_act(k, w.act_dtype), torch_act(v, w.act_dtype))
    q = torch_act(W.queries(w, 3, 40), w.act_dtype)
    out = torch.full((64, w.n_q_heads, w.head_dim), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(KVError) as e:
        gc.decode_attn_noalloc(0, q, out)
    assert e.value.status == KV_ERR_CAPACITY and "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    small = W.scaled(W.WORKLOADS["llama8b"], batch=2, context=256)
    ks, vs = W.kv_tokens(small, 4, 200)
    gs = KVCache(**cache_kwargs(small, 256))
    gs.append(0, torch_act(ks, small.act_dtype), torch_act(vs, small.act_dtype))
    ref, lse_ref, o2, l2 = _both(gs, W.queries(small, 4, 200), small.act_dtype)
    _same(o2, ref)
    _same(l2, lse_ref)
