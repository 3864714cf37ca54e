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


def _normed_rows(norms, B=1, H=2, D=128, seed=0):
    """K rows whose key norm (every head) is exactly the given value (one
    nonzero channel), and N(0,1) V rows: float32 [B, H, T, D]."""
    T = len(norms)
    k = np.zeros((B, H, T, D), np.float32)
    k[:, :, :, 0] = np.asarray(norms, np.float32)[None, None, :]
    v = np.random.default_rng(seed).standard_normal((B, H, T, D)).astype(np.float16).astype(np.float32)
    return k, v


def _masks(c):
    ex = c.export(0)
    return [int(x) for x in ex["sink_mask"][0]] if "sink_mask" in ex else []


def test_running_admission_one_token_per_call():
    """k = 2, one token per call. While group 0 is open every member can be
    displaced: 3 (norm 5) displaces 1, 10 (9) displaces 0, 20 (7) displaces
    3; a later token of equal norm never displaces (ties to the lower
    position). Group 0 is quantised when token 31 arrives: from then on 10 and
    20 are locked and 33 (norm 8) is not admitted."""
    norms = [1.0] * 40
    norms[3], norms[10], norms[20], norms[33] = 5.0, 9.0, 7.0, 8.0
    k, v = _normed_rows(norms)
    c = _cache(2, B=1, H=2)
    want = {0: [0], 1: [0, 1], 2: [0, 1], 3: [0, 3], 9: [0, 3], 10: [3, 10], 19: [3, 10],
            20: [10, 20], 31: [10, 20], 32: [10, 20], 33: [10, 20], 39: [10, 20]}
    for t in range(40):
        c.append(0, k[:, :, t:t + 1], v[:, :, t:t + 1])
        if t in want:
            assert c.sink_positions(0)[0].tolist() == want[t], t
    ex = c.export(0)
    assert _masks(c) == [(1 << 10) | (1 << 20)]
    assert np.array_equal(ex["sink_k"][0], k[0][:, [10, 20]])
    assert np.array_equal(ex["sink_v"][0], v[0][:, [10, 20]])


def test_running_admission_calls_across_groups():
    """k = 2 with calls of several tokens. The prefill of 40 tokens takes 35
    (norm 7) and 5 (6); group 0 is quantised in that call, locking 5. Token
    40 (9) displaces 35, which is still in the residual and is later
    quantised as an ordinary row. The call of 41..64 holds 60 (9), which ties
    40 and loses to the lower position; its group 1 is quantised with 40 as
    its sink. Token 65 (20) finds both members locked."""
    norms = [1.0] * 66
    norms[5], norms[35], norms[40], norms[50], norms[60], norms[65] = 6.0, 7.0, 9.0, 8.0, 9.0, 20.0
    k, v = _normed_rows(norms, seed=1)
    c = _cache(2, B=1, H=2)
    c.prefill_quantize(0, k[:, :, :40], v[:, :, :40])
    assert c.sink_positions(0)[0].tolist() == [5, 35]
    assert _masks(c) == [1 << 5]
    c.append(0, k[:, :, 40:41], v[:, :, 40:41])
    assert c.sink_positions(0)[0].tolist() == [5, 40]
    c.append(0, k[:, :, 41:65], v[:, :, 41:65])
    assert c.sink_positions(0)[0].tolist() == [5, 40]
    assert _masks(c) == [1 << 5, 1 << 8]
    c.append(0, k[:, :, 65:66], v[:, :, 65:66])
    assert c.sink_positions(0)[0].tolist() == [5, 40]
    # the displaced 35 reads back from its quantised group like any other row
    pos, K, V, pool = c.read_set(0, 0, 0)
    i35 = int(np.nonzero(pos == 35)[0][0])
    assert pool[i35] == 1


def test_running_admission_is_plain_top_k_while_nothing_is_locked():
    """Brute force: calls of random sizes inside the first group (no group is
    quantised, so nothing is locked) leave exactly the top-k of every token so
    far."""
    rng = np.random.default_rng(7)
    for trial in range(20):
        kk = int(rng.integers(1, 6))
        norms = rng.integers(1, 9, 31).astype(np.float32)   # many ties
        k, v = _normed_rows(norms, seed=trial)
        c = _cache(kk, B=1, H=2)
        t = 0
        while t < 31:
            n = int(rng.integers(1, 6))
            c.append(0, k[:, :, t:t + n], v[:, :, t:t + n])
            t = min(31, t + n)
            want = kvsink.top_k(kvsink.key_norms(k[:, :, :t]), kk)[0].tolist()
            assert c.sink_positions(0)[0].tolist() == want, (trial, t)


def test_running_admission_invariants():
    """Over many groups with random calls: the set holds min(k, L) members,
    a member below the quantised end never leaves, and every member's rows
    are its own."""
    rng = np.random.default_rng(3)
    norms = rng.integers(1, 50, 300).astype(np.float32)
    k, v = _normed_rows(norms, seed=3)
    c = _cache(4, B=1, H=2)
    t, prev_locked = 0, set()
    while t < 300:
        n = int(rng.integers(1, 40))
        c.append(0, k[:, :, t:t + n], v[:, :, t:t + n])
        t = min(300, t + n)
        sp = c.sink_positions(0)[0].tolist()
        assert len(sp) == min(4, t)
        assert prev_locked <= set(sp)
        prev_locked = {p for p in sp if p < c.q_end(0)}
        ex = c.export(0)
        assert np.array_equal(ex["sink_k"][0], k[0][:, sp])


def test_group_of_only_sinks_is_left_as_is():
    """k = 32 with the 32 largest keys exactly filling group 0: no row of the
    group is left to substitute, so the group is quantised as plain KIVI
    would ("How it works" 3 needs a non-sink row), its mask is full, and
    attention reads all 32 rows exact from the sinks."""
    norms = [1.0] * 70
    for p in range(32):
        norms[p] = 10.0 + p
    k, v = _normed_rows(norms, seed=9)
    c = _cache(32, B=1, H=2)
    c.prefill_quantize(0, k, v)
    assert c.sink_positions(0)[0].tolist() == list(range(32))
    plain = _cache(0, B=1, H=2)
    plain.prefill_quantize(0, k, v)
    a, b = c.export(0), plain.export(0)
    for name in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero"):
        n = 1 if name in ("k_scale", "k_zero") else 32     # group 0: per group, or its 32 token rows
        assert np.array_equal(a[name][:, :, :n], b[name][:, :, :n]), name
    assert int(a["sink_mask"][0, 0]) == 0xFFFFFFFF
    pos, K, V, pool = c.read_set(0, 0, 0)
    assert np.array_equal(pool[pos < 32], np.zeros(32, np.int64))
