"""Pins of the oracle's KVSink selection and calibration exclusion (no GPU).

The claims follow VeloxQuant-MLX "KVSink-Adapted Sink Protection", section
"Evidence": planted sinks are found and kept bit-exact; protection lowers key
MSE; dynamic selection beats first-N at equal budget when sinks are not at
the front; n_sink_tokens = 0 is plain KIVI bit for bit; byte accounting
partitions the tokens; and (section "How it works" 3) leaving the exclusion
out inflates the neighbours' error.
"""
import numpy as np
import pytest

from oracle import CacheConfig, OracleCache, kivi, kvsink


def _setup(seed=0, T=1024, B=2, H=8, D=128, n_planted=5, front=False):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((B, H, T, D))).astype(np.float16).astype(np.float32)
    v = (rng.standard_normal((B, H, T, D))).astype(np.float16).astype(np.float32)
    planted = []
    for b in range(B):
        pos = np.sort(rng.choice(np.arange(5, T) if not front else np.arange(5), n_planted, replace=False))
        planted.append(pos)
        for p in pos:
            k[b, :, p] = (k[b, :, p] * 25.0).astype(np.float16).astype(np.float32)
    return k, v, np.array(planted)


def _cache(n_dyn=5, B=2, H=8, **kw):
    cfg = dict(n_layers=1, batch=B, n_kv_heads=H, n_q_heads=4 * H, head_dim=128,
               max_tokens=4096, k_bits=2, v_bits=2, n_dyn_sinks=n_dyn)
    cfg.update(kw)
    return OracleCache(CacheConfig(**cfg))


def _read_error(c, k, v):
    """Squared error of the K and V rows attention reads, over all positions."""
    ek = ev = 0.0
    for b in range(c.cfg.batch):
        for h in range(c.cfg.n_kv_heads):
            pos, K, V, _ = c.read_set(0, b, h)
            ek += float(np.sum((K - k[b, h, pos]) ** 2))
            ev += float(np.sum((V - v[b, h, pos]) ** 2))
    return ek, ev


def test_planted_sinks_selected_and_exact():
    k, v, planted = _setup()
    c = _cache()
    c.prefill_quantize(0, k, v)
    ex = c.export(0)
    assert np.array_equal(ex["sink_pos"], planted)
    for b in range(2):
        assert np.array_equal(ex["sink_k"][b], k[b][:, planted[b]])
        assert np.array_equal(ex["sink_v"][b], v[b][:, planted[b]])
    # the per-group mask marks exactly the planted rows
    for b in range(2):
        bits = [(g, r) for g in range(ex["sink_mask"].shape[1]) for r in range(32)
                if ex["sink_mask"][b, g] >> r & 1]
        assert sorted(32 * g + r for g, r in bits) == list(planted[b])


def test_protection_lowers_key_error():
    k, v, _ = _setup(1)
    prot, plain = _cache(5), _cache(0)
    prot.prefill_quantize(0, k, v)
    plain.prefill_quantize(0, k, v)
    assert _read_error(prot, k, v)[0] < 0.5 * _read_error(plain, k, v)[0]


def test_dynamic_beats_first_n_when_sinks_not_in_front():
    k, v, _ = _setup(2)
    dyn = _cache(5)
    first = _cache(0, n_sink=5)
    dyn.prefill_quantize(0, k, v)
    first.prefill_quantize(0, k, v)
    assert dyn.stats(0)["n_sink"] == first.stats(0)["n_sink"] == 2 * 5
    assert _read_error(dyn, k, v)[0] < _read_error(first, k, v)[0]


def test_no_sinks_is_plain_kivi_bit_for_bit():
    k, v, _ = _setup(3)
    a = _cache(0)
    a.prefill_quantize(0, k, v)
    ex = a.export(0)
    # plain KIVI straight from the quantiser, group by group
    for g in range(0, 1024 // 32, 7):
        kq, ks, kz = kivi.quantize_k_group(k[:, :, 32 * g:32 * g + 32], 2)
        assert np.array_equal(ex["k_codes"][:, :, 32 * g:32 * g + 32], kivi.pack_codes(kq, 2))
        assert np.array_equal(ex["k_scale"][:, :, g], ks) and np.array_equal(ex["k_zero"][:, :, g], kz)
    assert not np.any(ex["sink_mask"])


def test_exclusion_omitted_inflates_neighbours(monkeypatch):
    """Plant the mistake in the oracle: skip the substitution and the group
    scales of the sinks' groups blow up, ruining the neighbours."""
    k, v, planted = _setup(4)
    good = _cache(5)
    good.prefill_quantize(0, k, v)
    monkeypatch.setattr(kvsink, "exclude", lambda rows, sink_rows: np.array(rows, copy=True))
    bad = _cache(5)
    bad.prefill_quantize(0, k, v)

    def neighbour_error(c):
        e = 0.0
        for b in range(2):
            groups = {int(p) // 32 for p in planted[b]}
            for h in range(8):
                pos, K, _, pool = c.read_set(0, b, h)
                sel = np.array([int(p) // 32 in groups for p in pos]) & (pool == 1)
                e += float(np.sum((K[sel] - k[b, h, pos[sel]]) ** 2))
        return e

    assert neighbour_error(bad) > 10 * neighbour_error(good)


def test_byte_partition_exact():
    k, v, _ = _setup(5, T=1000)
    c = _cache(5)
    c.prefill_quantize(0, k, v)
    s = c.stats(0)
    assert s["n_quant"] + s["n_sink"] + s["n_tail"] + s["n_evicted"] == 2 * 1000
    H, D = 8, 128
    assert s["sink_bytes"] == s["n_sink"] * H * 4 * D
    assert s["tail_bytes"] == s["n_tail"] * H * 4 * D == 2 * 8 * H * 4 * D
    assert s["code_bytes"] == s["n_quant"] * H * D * 4 // 8


def test_substitute_rule():
    assert kvsink.substitutes({3}) == {3: 2}                 # tie 2 vs 4 -> earlier
    assert kvsink.substitutes({0}) == {0: 1}
    assert kvsink.substitutes({31}) == {31: 30}
    assert kvsink.substitutes({2, 3}) == {2: 1, 3: 4}
    assert kvsink.substitutes({1, 2, 3}) == {1: 0, 2: 0, 3: 4}
    assert kvsink.substitutes(set(range(32))) == {}


def test_top_k_ties_go_to_lower_position():
    m = np.array([[1.0, 3.0, 2.0, 3.0, 3.0, 0.5]], np.float32)
    assert list(kvsink.top_k(m, 2)[0]) == [1, 3]
    assert list(kvsink.top_k(m, 4)[0]) == [1, 2, 3, 4]


def test_key_norm_is_mean_over_heads():
    k = np.zeros((1, 2, 3, 128), np.float32)
    k[0, 0, 1, 0] = 3.0
    k[0, 0, 1, 1] = 4.0          # head 0 norm 5
    k[0, 1, 1, 7] = 1.0          # head 1 norm 1
    assert np.array_equal(kvsink.key_norms(k)[0], np.array([0.0, 3.0, 0.0], np.float32))


def test_selection_only_on_empty_cache():
    k, v, _ = _setup(6, T=64)
    c = _cache(5)
    c.prefill_quantize(0, k, v)
    with pytest.raises(RuntimeError):
        c.prefill_quantize(0, k, v)
