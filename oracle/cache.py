"""The quantised KV cache as a plain state machine, and decode attention by
its definition (CPU oracle).

Test infrastructure: see the package docstring for who may import this.

Sources (page title, section):
  * posttrainllm "StreamingLLM + KIVI" doc, "StreamingLLM - Implementation":
    after each per-layer append, when the cache holds more than sink + window
    tokens, drop [sink, len - window).
  * same doc, "KIVI": K per channel, V per token; "Caveats": freeze scales per
    token group (KIVI's group idea).
  * PR #2318 "KV cache: FP16 sliding window + attention sinks", "Summary":
    an FP16 overlay over the sink cells and the most recent N cells of the
    quantised bulk; recent context and sinks read exact, older context reads
    quantised.
  * VeloxQuant-MLX "KVSink-Adapted Sink Protection": KIVI's fp16 residual
    window holds tokens until a group fills; dynamic top-k sinks.
  * Foundry "TurboQuant KV Cache Compression - Spec": per-token quantisation,
    attention over dequantised keys and values.
  * posttrainllm "StreamingLLM + KIVI", "RoPE caveat": the "true"
    re-positioning stores K before RoPE and rotates on read; "Caveats": per-
    channel K quantisation then sees a basis that does not turn with the
    position. With k_pre_rope the stored keys (codes, sinks, tail) are the
    un-rotated inputs; attention rotates each retained key (dequantised, in
    double) at its absolute position, or at its cache slot when
    re-positioning, and the query as usual.

Segments of one layer after L appended tokens (absolute positions), with
N_s overlay sinks, W overlay window, E the eviction end ([N_s, E) evicted):
  * Q_end = 32 floor(L / 32) in KIVI mode (whole groups only; the rest sits in
    the fp16 residual), Q_end = L in TurboQuant mode (per-token codes).
  * F = min(Q_end, max(L - W, N_s)); the fp16 tail is [F, L).
  * The sink set P_s is [0, min(N_s, L)) (StreamingLLM overlay) or the KVSink
    top-k positions; sinks in [0, F) are read from the sink buffer, sinks at
    or after F are read from the tail.
  * The quantised segment is [max(N_s, E), F) minus P_s.
Every retained position is read exactly once; the four pools (sink,
quantised, tail, evicted) partition [0, L).

The overlay changes only where a position is READ from: quantisation is
plain KIVI over all tokens, so a group that holds overlay sinks is calibrated
with them, and n_sink = window = 0 is plain KIVI.

Attention: scale 1/sqrt(D); decode attends to every retained position (no
causal mask); query head j reads KV head floor(j / (Hq / Hkv)); dequantised
keys and values are float32 and every product, sum and the softmax are done
in double; the output is rounded once to float32. lse is the natural log of
the softmax denominator of the scaled scores.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import kivi, kvsink, rope
from . import turboquant as tq
from .numerics import is_representable

GROUP = 32


@dataclasses.dataclass
class CacheConfig:
    n_layers: int
    batch: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    max_tokens: int
    mode: str = "kivi"          # "kivi" | "turboquant"
    k_bits: int = 2
    v_bits: int = 4
    n_sink: int = 0
    window: int = 0
    evict_window: int = 0
    n_dyn_sinks: int = 0
    act_dtype: str = "f16"      # "f16" | "bf16"
    seed: int = 0
    rope_base: float = 0.0
    rope_reposition: bool = False   # StreamingLLM position re-encoding at read
    v_q4_0: bool = False            # V in the symmetric q4_0 form (KIVI, 4-bit V)
    k_pre_rope: bool = False        # keys stored before RoPE, rotated at read


def validate(cfg: CacheConfig) -> None:
    """The configuration rules shared by both implementations (restated
    independently in the library's host code)."""
    if cfg.n_layers < 1 or cfg.batch < 1 or cfg.n_kv_heads < 1 or cfg.n_q_heads < 1:
        raise ValueError("sizes must be positive")
    if cfg.n_q_heads % cfg.n_kv_heads:
        raise ValueError("n_q_heads must be a multiple of n_kv_heads")
    if cfg.head_dim not in (64, 128):
        raise ValueError("head_dim must be 64 or 128")
    if cfg.mode == "kivi":
        for b in (cfg.k_bits, cfg.v_bits):
            if b not in (2, 3, 4, 8):
                raise ValueError("KIVI bits must be 2, 3, 4 or 8")
    elif cfg.mode == "turboquant":
        for b in (cfg.k_bits, cfg.v_bits):
            if b not in (2, 3, 4):
                raise ValueError("TurboQuant bits must be 2, 3 or 4")
        if cfg.n_dyn_sinks:
            raise ValueError("KVSink sinks are defined on KIVI groups only")
    else:
        raise ValueError(f"unknown mode {cfg.mode!r}")
    if min(cfg.n_sink, cfg.window, cfg.evict_window, cfg.n_dyn_sinks) < 0:
        raise ValueError("negative size")
    if cfg.v_q4_0 and (cfg.mode != "kivi" or cfg.v_bits != 4):
        raise ValueError("the q4_0 V form is a 4-bit KIVI V format")
    if cfg.rope_reposition and not cfg.rope_base:
        raise ValueError("re-positioning needs the cache to apply RoPE")
    if cfg.k_pre_rope and (not cfg.rope_base or cfg.mode != "kivi" or cfg.n_dyn_sinks):
        raise ValueError("pre-RoPE keys need RoPE in the cache, KIVI mode and no KVSink sinks")
    if cfg.n_dyn_sinks and (cfg.n_sink or cfg.window or cfg.evict_window):
        raise ValueError("KVSink sinks exclude the StreamingLLM overlay and eviction")
    if cfg.n_dyn_sinks > 32:
        raise ValueError("at most 32 dynamic sinks")
    if cfg.evict_window and cfg.evict_window < max(cfg.window, GROUP):
        raise ValueError("evict_window must be >= max(window, 32)")
    if cfg.n_sink > GROUP:
        raise ValueError("at most 32 overlay sinks")
    if cfg.act_dtype not in ("f16", "bf16"):
        raise ValueError("act_dtype must be f16 or bf16")


class _Layer:
    def __init__(self, cfg: CacheConfig):
        self.L = 0
        self.E = cfg.n_sink
        self.rows = {}       # pos -> (k [B,H,D], v [B,H,D]) fp values still needed
        self.groups = {}     # KIVI: g -> dict of codes / fp16 scales and zeros
        self.tokens = {}     # TurboQuant: pos -> (kc [B,H,D], kn [B,H], vc, vn)
        B, H, D = cfg.batch, cfg.n_kv_heads, cfg.head_dim
        ns = max(cfg.n_sink, cfg.n_dyn_sinks)
        self.sink_k = np.zeros((B, H, ns, D), np.float32)
        self.sink_v = np.zeros((B, H, ns, D), np.float32)
        self.sink_pos = None  # KVSink: int64 [B, n] by position (n = min(k, L))
        self.sink_m = None    # KVSink: float32 [B, n] their key norms


class OracleCache:
    def __init__(self, cfg: CacheConfig):
        validate(cfg)
        self.cfg = cfg
        self.g = cfg.n_q_heads // cfg.n_kv_heads
        self.layers = [_Layer(cfg) for _ in range(cfg.n_layers)]
        if cfg.mode == "turboquant":
            self.sgn = tq.signs(cfg.seed, cfg.head_dim)
            self.cb_k = tq.codebook(cfg.head_dim, cfg.k_bits)
            self.cb_v = tq.codebook(cfg.head_dim, cfg.v_bits)

    # ------------------------------------------------------------ segments
    def q_end(self, layer: int) -> int:
        L = self.layers[layer].L
        return L if self.cfg.mode == "turboquant" else GROUP * (L // GROUP)

    def fp16_begin(self, layer: int) -> int:
        L = self.layers[layer].L
        return min(self.q_end(layer), max(L - self.cfg.window, self.cfg.n_sink))

    def sink_positions(self, layer: int) -> np.ndarray:
        """int64 [B, n]: the sink set P_s per batch element (all of it)."""
        st, cfg = self.layers[layer], self.cfg
        if cfg.n_dyn_sinks:
            if st.sink_pos is None:
                return np.zeros((cfg.batch, 0), np.int64)
            return st.sink_pos.copy()
        n = min(cfg.n_sink, st.L)
        return np.tile(np.arange(n, dtype=np.int64), (cfg.batch, 1))

    # ------------------------------------------------------------- appends
    def _check_input(self, k, v):
        cfg = self.cfg
        k = np.asarray(k, np.float32)
        v = np.asarray(v, np.float32)
        shape = (cfg.batch, cfg.n_kv_heads, k.shape[2], cfg.head_dim)
        if k.shape != shape or v.shape != shape:
            raise ValueError(f"expected K/V of shape {shape}")
        if not (is_representable(k, cfg.act_dtype) and is_representable(v, cfg.act_dtype)):
            raise ValueError("K/V values must be exact in the activation dtype")
        return k, v

    def _capacity_ok(self, st: _Layer, n: int) -> bool:
        first = GROUP * (st.E // GROUP)
        return st.L + n - first <= self.cfg.max_tokens

    def append(self, layer: int, k, v) -> None:
        """kv_append: new tokens take absolute positions L .. L+n-1."""
        k, v = self._check_input(k, v)
        st = self.layers[layer]
        if not self._capacity_ok(st, k.shape[2]):
            raise OverflowError("capacity")
        if self.cfg.rope_base and not self.cfg.k_pre_rope:
            k = rope.rotate_keys(k, st.L, self.cfg.rope_base, self.cfg.act_dtype)
        self._fold_sinks(layer, k, v)
        self._append_rotated(layer, k, v)

    def prefill_quantize(self, layer: int, k, v) -> None:
        """kv_prefill_quantize: the same state change as kv_append of the
        same tokens (the library runs it with a bulk quantiser)."""
        self.append(layer, k, v)

    def _fold_sinks(self, layer: int, k, v) -> None:
        """KVSink: fold the call's tokens (keys rotated like every stored key)
        into each sequence's running top-k before any of its groups is
        quantised (kvsink.admit); new members' K/V rows go to the sink rows."""
        st, cfg = self.layers[layer], self.cfg
        if not cfg.n_dyn_sinks:
            return
        L0 = st.L
        q0 = self.q_end(layer)
        m = kvsink.key_norms(k)
        old_pos = st.sink_pos if st.sink_pos is not None else np.zeros((cfg.batch, 0), np.int64)
        old_m = st.sink_m if st.sink_m is not None else np.zeros((cfg.batch, 0), np.float32)
        new = [kvsink.admit(list(zip(old_pos[b].tolist(), old_m[b].tolist())), m[b], L0, q0,
                            cfg.n_dyn_sinks) for b in range(cfg.batch)]
        n = len(new[0])
        pos = np.array([[p for p, _ in nb] for nb in new], np.int64).reshape(cfg.batch, n)
        sk = np.zeros_like(st.sink_k)
        sv = np.zeros_like(st.sink_v)
        for b in range(cfg.batch):
            for j, p in enumerate(pos[b]):
                if p >= L0:   # a token of this call
                    sk[b, :, j] = k[b, :, p - L0]
                    sv[b, :, j] = v[b, :, p - L0]
                else:         # a member kept from before
                    i = int(np.nonzero(old_pos[b] == p)[0][0])
                    sk[b, :, j] = st.sink_k[b, :, i]
                    sv[b, :, j] = st.sink_v[b, :, i]
        st.sink_k, st.sink_v = sk, sv
        st.sink_pos = pos
        st.sink_m = np.array([[mm for _, mm in nb] for nb in new], np.float32).reshape(cfg.batch, n)

    def _append_rotated(self, layer: int, k, v) -> None:
        st, cfg = self.layers[layer], self.cfg
        n = k.shape[2]
        L0, L1 = st.L, st.L + n
        for pos in range(L0, min(L1, cfg.n_sink)):
            st.sink_k[:, :, pos] = k[:, :, pos - L0]
            st.sink_v[:, :, pos] = v[:, :, pos - L0]
        q0 = self.q_end(layer)
        st.L = L1
        q1 = self.q_end(layer)

        def rows(p0, p1):
            """K, V rows [B, H, p1-p0, D] of positions p0..p1-1 (stored or new)."""
            if p0 >= L0:
                return k[:, :, p0 - L0:p1 - L0], v[:, :, p0 - L0:p1 - L0]
            ks = [st.rows[p][0] if p < L0 else k[:, :, p - L0] for p in range(p0, p1)]
            vs = [st.rows[p][1] if p < L0 else v[:, :, p - L0] for p in range(p0, p1)]
            return np.stack(ks, axis=2), np.stack(vs, axis=2)

        if cfg.mode == "kivi":
            g0, g1 = q0 // GROUP, q1 // GROUP
            if g1 > g0:
                kr, vr = rows(GROUP * g0, GROUP * g1)
                self._quantize_groups(layer, g0, kr, vr)
        elif q1 > q0:
            kr, vr = rows(q0, q1)
            kc, kn = tq.quantize(kr, self.sgn, self.cb_k[0])
            vc, vn = tq.quantize(vr, self.sgn, self.cb_v[0])
            for i, pos in enumerate(range(q0, q1)):
                st.tokens[pos] = (kc[:, :, i], kn[:, :, i], vc[:, :, i], vn[:, :, i])
        # keep the exact rows still read from the tail or waiting for a group
        F = self.fp16_begin(layer)
        for pos in [p for p in st.rows if p < F]:
            del st.rows[pos]
        for pos in range(max(F, L0), L1):
            st.rows[pos] = (k[:, :, pos - L0].copy(), v[:, :, pos - L0].copy())

    def _quantize_groups(self, layer: int, g0: int, kr: np.ndarray, vr: np.ndarray) -> None:
        """Quantise consecutive groups g0.. from rows [B, H, 32 * ng, D]."""
        st, cfg = self.layers[layer], self.cfg
        B, H, T, D = kr.shape
        ng = T // GROUP
        kr = kr.reshape(B, H, ng, GROUP, D)
        vr = vr.reshape(B, H, ng, GROUP, D)
        masks = np.zeros((ng, B), np.uint32)
        if cfg.n_dyn_sinks and st.sink_pos is not None:
            hit = sorted({int(p) // GROUP - g0 for p in st.sink_pos.ravel()
                          if 0 <= int(p) // GROUP - g0 < ng})
            if hit:
                kr = kr.copy()
                vr = vr.copy()
            for i in hit:
                g = g0 + i
                for b in range(B):
                    sink_rows = {int(p) - GROUP * g for p in st.sink_pos[b]
                                 if GROUP * g <= p < GROUP * (g + 1)}
                    for r in sink_rows:
                        masks[i, b] |= np.uint32(1 << r)
                    if sink_rows:
                        kr[b, :, i] = kvsink.exclude(kr[b, :, i], sink_rows)
                        vr[b, :, i] = kvsink.exclude(vr[b, :, i], sink_rows)
        kq, ks, kz = kivi.quantize_k_group(kr, cfg.k_bits)      # [B,H,ng,32,D], [B,H,ng,D]
        if cfg.v_q4_0:
            vq, vs, vz = kivi.quantize_v_rows_q4_0(vr)
        else:
            vq, vs, vz = kivi.quantize_v_rows(vr, cfg.v_bits)   # [B,H,ng,32,D], [B,H,ng,32,D/32]
        for i in range(ng):
            st.groups[g0 + i] = dict(kq=kq[:, :, i], ks=ks[:, :, i], kz=kz[:, :, i],
                                     vq=vq[:, :, i], vs=vs[:, :, i], vz=vz[:, :, i],
                                     mask=masks[i])

    # ------------------------------------------------------------ eviction
    def evict(self, layer: int):
        """kv_evict: drop [max(N_s, E), L - evict_window) when the retained
        count exceeds N_s + evict_window. Returns the absolute range dropped
        (begin == end when nothing is)."""
        st, cfg = self.layers[layer], self.cfg
        if not cfg.evict_window or st.L - cfg.evict_window <= st.E:
            return st.E, st.E
        begin, end = st.E, st.L - cfg.evict_window
        st.E = end
        for g in [g for g in st.groups if GROUP * (g + 1) <= end]:
            del st.groups[g]
        for p in [p for p in st.tokens if p < end]:
            del st.tokens[p]
        return begin, end

    # ------------------------------------------------------------ dequantise
    def _quant_rows(self, layer: int, b: int, h: int, positions: np.ndarray):
        """Dequantised float32 K, V rows [len(positions), D] of one (b, h)."""
        st, cfg = self.layers[layer], self.cfg
        D = cfg.head_dim
        K = np.empty((len(positions), D), np.float32)
        V = np.empty((len(positions), D), np.float32)
        if cfg.mode == "kivi":
            cache = {}
            for i, p in enumerate(positions):
                g, r = divmod(int(p), GROUP)
                if g not in cache:
                    gr = st.groups[g]
                    cache[g] = (kivi.dequantize_k_group(gr["kq"][b, h], gr["ks"][b, h], gr["kz"][b, h]),
                                kivi.dequantize_v_rows(gr["vq"][b, h], gr["vs"][b, h], gr["vz"][b, h]))
                K[i] = cache[g][0][r]
                V[i] = cache[g][1][r]
        else:
            for i, p in enumerate(positions):
                kc, kn, vc, vn = st.tokens[int(p)]
                K[i] = tq.dequantize(kc[b, h], kn[b, h], self.sgn, self.cb_k[1])
                V[i] = tq.dequantize(vc[b, h], vn[b, h], self.sgn, self.cb_v[1])
        return K, V

    def read_set(self, layer: int, b: int, h: int):
        """Positions and float32 K, V rows that attention reads for (b, h),
        as (positions, K, V, pool) with pool 0 = sink, 1 = quantised, 2 = tail."""
        st, cfg = self.layers[layer], self.cfg
        L, F = st.L, self.fp16_begin(layer)
        sp = self.sink_positions(layer)[b]
        pos_list, K_list, V_list, pool = [], [], [], []
        for j, p in enumerate(sp):
            if p < F:
                pos_list.append(np.array([p]))
                K_list.append(st.sink_k[b, h, j][None])
                V_list.append(st.sink_v[b, h, j][None])
                pool.append(np.array([0]))
        lo = max(cfg.n_sink, st.E)
        qpos = np.array([p for p in range(lo, F) if p not in set(int(x) for x in sp)], np.int64)
        if len(qpos):
            Kq, Vq = self._quant_rows(layer, b, h, qpos)
            pos_list.append(qpos)
            K_list.append(Kq)
            V_list.append(Vq)
            pool.append(np.ones(len(qpos), np.int64))
        tpos = np.arange(F, L, dtype=np.int64)
        if len(tpos):
            pos_list.append(tpos)
            K_list.append(np.stack([st.rows[int(p)][0][b, h] for p in tpos]))
            V_list.append(np.stack([st.rows[int(p)][1][b, h] for p in tpos]))
            pool.append(np.full(len(tpos), 2, np.int64))
        if not pos_list:
            D = cfg.head_dim
            return (np.zeros(0, np.int64), np.zeros((0, D), np.float32),
                    np.zeros((0, D), np.float32), np.zeros(0, np.int64))
        return (np.concatenate(pos_list), np.concatenate(K_list),
                np.concatenate(V_list), np.concatenate(pool))

    # ------------------------------------------------------------ attention
    def cache_position(self, layer: int, p):
        """Slot index of absolute position p inside the cache (StreamingLLM
        "RoPE caveat": the sinks keep 0 .. N_s - 1, the kept tokens follow
        without the evicted gap). Equal to p until something is evicted."""
        n_s, E = self.cfg.n_sink, self.layers[layer].E
        p = np.asarray(p, np.int64)
        return np.where(p < n_s, p, n_s + (p - E))

    def query_rotated(self, layer: int, q: np.ndarray) -> np.ndarray:
        """The query as attention uses it: RoPE'd at position L - 1 when the
        cache applies RoPE, at its cache slot when it re-positions (float32,
        not rounded to the activation dtype)."""
        q = np.asarray(q, np.float32)
        if self.cfg.rope_base:
            L = self.layers[layer].L
            pos = int(self.cache_position(layer, L - 1)) if self.cfg.rope_reposition else L - 1
            q = rope.rotate(q[..., None, :], [pos], self.cfg.rope_base)[..., 0, :]
        return q

    def decode_attn(self, layer: int, q: np.ndarray, heads=None):
        """kv_decode_attn by its definition. q: float32 [B, Hq, D] (act-exact).

        Returns (out float32 [B, Hq, D], lse float32 [B, Hq]); with `heads`
        (a list of (b, hq)) only those entries are computed (others are NaN).
        """
        cfg = self.cfg
        B, Hq, D = cfg.batch, cfg.n_q_heads, cfg.head_dim
        if self.layers[layer].L == 0:
            raise RuntimeError("decode on an empty cache")
        qr = self.query_rotated(layer, q).astype(np.float64)
        out = np.full((B, Hq, D), np.nan, np.float32)
        lse = np.full((B, Hq), np.nan, np.float32)
        todo = heads if heads is not None else [(b, j) for b in range(B) for j in range(Hq)]
        by_kv = {}
        for b, j in todo:
            by_kv.setdefault((b, j // self.g), []).append(j)
        for (b, h), js in by_kv.items():
            pos, K, V, _ = self.read_set(layer, b, h)
            K64 = K.astype(np.float64)
            if cfg.k_pre_rope:
                # keys stored before RoPE: rotated here, at their cache slot
                # when re-positioning, else at their absolute position
                kpos = self.cache_position(layer, pos) if cfg.rope_reposition else pos
                K64 = rope.rotate64(K64, kpos, cfg.rope_base)
            elif cfg.rope_reposition:
                # StreamingLLM re-positioning: un-rotate each stored key at
                # its absolute position, rotate it at its cache slot
                K64 = rope.rotate64(rope.rotate64(K64, -pos, cfg.rope_base),
                                    self.cache_position(layer, pos), cfg.rope_base)
            V64 = V.astype(np.float64)
            for j in js:
                s = (K64 @ qr[b, j]) / math.sqrt(D)
                m = s.max()
                p = np.exp(s - m)
                l = p.sum()
                out[b, j] = ((p @ V64) / l).astype(np.float32)
                lse[b, j] = np.float32(m + math.log(l))
        return out, lse

    # ------------------------------------------------------------ accounting
    def stats(self, layer: int) -> dict:
        """Token counts per read pool (summed over the batch) and the bytes
        each pool holds (the KV heads and the batch included)."""
        st, cfg = self.layers[layer], self.cfg
        B, H, D = cfg.batch, cfg.n_kv_heads, cfg.head_dim
        L, E, F, Q = st.L, st.E, self.fp16_begin(layer), self.q_end(layer)
        sp = self.sink_positions(layer)
        lo = max(cfg.n_sink, E)
        n_sink = int(np.sum(sp < F))
        n_sink_in_quant = int(np.sum((sp >= lo) & (sp < F)))
        n_quant = B * max(0, F - lo) - n_sink_in_quant
        n_tail = B * (L - F)
        n_evicted = B * (E - cfg.n_sink)
        row16 = 2 * D * 2                     # K + V row of a 16-bit dtype
        # stored bytes: D * bits / 8 per row (3-bit codes eight to three bytes)
        code = D * cfg.k_bits // 8 + D * cfg.v_bits // 8
        if cfg.mode == "kivi":
            g_lo, g_hi = lo // GROUP, (F + GROUP - 1) // GROUP
            n_kgroups = max(0, g_hi - g_lo) if F > lo else 0
            kmeta = n_kgroups * B * H * 4 * D
            vmeta = n_quant * H * (D // GROUP) * 4
        else:
            kmeta = n_quant * H * 4
            vmeta = n_quant * H * 4
        return dict(length=L, evict_end=E, quant_end=Q, fp16_begin=F,
                    n_quant=n_quant, n_sink=n_sink, n_tail=n_tail, n_evicted=n_evicted,
                    code_bytes=n_quant * H * code, kmeta_bytes=kmeta, vmeta_bytes=vmeta,
                    sink_bytes=n_sink * H * row16, tail_bytes=n_tail * H * row16)

    # ------------------------------------------------------------ export
    def token_range(self, layer: int):
        """[first, end) of the quantised tokens still stored (whole groups)."""
        st = self.layers[layer]
        return GROUP * (st.E // GROUP), self.q_end(layer)

    def export(self, layer: int) -> dict:
        """Canonical arrays over the stored quantised range, the sinks and the
        tail: the layout the library's export produces."""
        st, cfg = self.layers[layer], self.cfg
        first, end = self.token_range(layer)
        out = {}
        if cfg.mode == "kivi":
            gs = range(first // GROUP, end // GROUP)
            if len(gs):
                cat = lambda key, ax: np.concatenate([st.groups[g][key] for g in gs], axis=ax)
                out["k_codes"] = kivi.pack_codes(cat("kq", 2), cfg.k_bits)
                out["k_scale"] = np.stack([st.groups[g]["ks"] for g in gs], axis=2)
                out["k_zero"] = np.stack([st.groups[g]["kz"] for g in gs], axis=2)
                out["v_codes"] = kivi.pack_codes(cat("vq", 2), cfg.v_bits)
                out["v_scale"] = cat("vs", 2)
                out["v_zero"] = cat("vz", 2)
                out["sink_mask"] = np.stack([st.groups[g]["mask"] for g in gs], axis=1)
        else:
            ts = range(first, end)
            if len(ts):
                out["k_codes"] = kivi.pack_codes(np.stack([st.tokens[p][0] for p in ts], 2), cfg.k_bits)
                out["k_norm"] = np.stack([st.tokens[p][1] for p in ts], 2)
                out["v_codes"] = kivi.pack_codes(np.stack([st.tokens[p][2] for p in ts], 2), cfg.v_bits)
                out["v_norm"] = np.stack([st.tokens[p][3] for p in ts], 2)
        sp = self.sink_positions(layer)
        out["sink_pos"] = sp
        out["sink_k"] = st.sink_k[:, :, :sp.shape[1]].copy()
        out["sink_v"] = st.sink_v[:, :, :sp.shape[1]].copy()
        F = self.fp16_begin(layer)
        tp = range(F, st.L)
        if len(tp):
            out["tail_k"] = np.stack([st.rows[p][0] for p in tp], 2)
            out["tail_v"] = np.stack([st.rows[p][1] for p in tp], 2)
        return out
