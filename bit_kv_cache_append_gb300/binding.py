"""Thin Python binding of the C ABI in ``include/kvq.h`` (ctypes).

Argument marshalling only: every step of the cache runs in the CUDA
library ``libkvq.so``. PyTorch supplies device memory (the arena, inputs and
outputs) and streams. Importing this module loads the library and raises if
it is missing; there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_CAPACITY, KV_ERR_UNSUPPORTED, KV_ERR_CUDA, KV_ERR_TIMEOUT, KV_ERR_STATE = range(7)
KV_MODE_KIVI, KV_MODE_TURBOQUANT = 0, 1
KV_DT_F16, KV_DT_BF16 = 0, 1

EXPORT = dict(k_codes=0, k_scale=1, k_zero=2, v_codes=3, v_scale=4, v_zero=5, k_norm=6, v_norm=7,
              sink_pos=8, sink_k=9, sink_v=10, tail_k=11, tail_v=12, sink_mask=13,
              codebook_k=14, codebook_v=15, tq_signs=16, rope=17)

SYMBOLS = ("kv_cache_required_bytes", "kv_cache_create", "kv_cache_destroy", "kv_cache_reset",
           "kv_append", "kv_prefill_quantize", "kv_evict", "kv_decode_attn", "kv_cache_stats",
           "kv_cache_export_bytes", "kv_cache_export", "kv_cache_check_device_error",
           "kv_cache_set_timing_events", "kv_launch_count", "kv_copy_bandwidth_kernel",
           "kv_last_error", "kv_decode_attn_noalloc", "kv_cache_test_bounded_wait")


class KVError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kv_status {status}: {msg}")
        self.status = status


class CacheConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("batch", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("n_q_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("max_tokens", ctypes.c_int64),
                ("mode", ctypes.c_int), ("k_bits", ctypes.c_int), ("v_bits", ctypes.c_int),
                ("group_size", ctypes.c_int), ("residual", ctypes.c_int), ("n_sink", ctypes.c_int),
                ("window", ctypes.c_int), ("evict_window", ctypes.c_int), ("n_dyn_sinks", ctypes.c_int),
                ("act_dtype", ctypes.c_int), ("seed", ctypes.c_uint64), ("rope_base", ctypes.c_double),
                ("rope_max_pos", ctypes.c_int64), ("max_splits", ctypes.c_int),
                ("rope_reposition", ctypes.c_int), ("v_q4_0", ctypes.c_int), ("k_pre_rope", ctypes.c_int)]


class CacheStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "length", "evict_end", "quant_end", "fp16_begin", "n_quant", "n_sink", "n_tail", "n_evicted",
        "code_bytes", "kmeta_bytes", "vmeta_bytes", "sink_bytes", "tail_bytes")]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with bit_kv_cache_append_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(CacheConfig)
    sig = {
        "kv_cache_required_bytes": [cfgp, ctypes.POINTER(sz)],
        "kv_cache_create": [cfgp, vp, sz, ctypes.POINTER(vp)],
        "kv_cache_destroy": [vp],
        "kv_cache_reset": [vp],
        "kv_append": [vp, i32, vp, vp, i32, vp],
        "kv_prefill_quantize": [vp, i32, vp, vp, i32, vp],
        "kv_evict": [vp, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)],
        "kv_decode_attn": [vp, i32, vp, vp, vp, vp],
        "kv_decode_attn_noalloc": [vp, i32, vp, vp, vp, vp],
        "kv_cache_stats": [vp, i32, ctypes.POINTER(CacheStats)],
        "kv_cache_export_bytes": [vp, i32, i32, ctypes.POINTER(sz)],
        "kv_cache_export": [vp, i32, i32, vp, sz, vp],
        "kv_cache_check_device_error": [vp, vp],
        "kv_cache_test_bounded_wait": [vp, i64, ctypes.POINTER(i64), vp],
        "kv_cache_set_timing_events": [vp, vp, vp],
        "kv_copy_bandwidth_kernel": [vp, vp, sz, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.kv_launch_count.argtypes = []
    lib.kv_launch_count.restype = ctypes.c_int64
    lib.kv_last_error.argtypes = []
    lib.kv_last_error.restype = ctypes.c_char_p
    return lib


_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load_library()
    return _LIB


def check(status: int) -> None:
    if status != KV_OK:
        raise KVError(status, lib().kv_last_error().decode())


def make_config(*, n_layers, batch, n_kv_heads, n_q_heads, head_dim, max_tokens, mode="kivi", k_bits=2,
                v_bits=4, n_sink=0, window=0, evict_window=0, n_dyn_sinks=0, act_dtype="f16", seed=0,
                rope_base=0.0, rope_max_pos=0, max_splits=0, rope_reposition=False,
                v_q4_0=False, k_pre_rope=False) -> CacheConfig:
    tq = mode == "turboquant"
    return CacheConfig(n_layers, batch, n_kv_heads, n_q_heads, head_dim, max_tokens,
                       KV_MODE_TURBOQUANT if tq else KV_MODE_KIVI, k_bits, v_bits, 32, 0 if tq else 32,
                       n_sink, window, evict_window, n_dyn_sinks,
                       KV_DT_BF16 if act_dtype == "bf16" else KV_DT_F16, seed, float(rope_base),
                       rope_max_pos, max_splits, int(bool(rope_reposition)), int(bool(v_q4_0)),
                       int(bool(k_pre_rope)))


def required_bytes(cfg: CacheConfig) -> int:
    n = ctypes.c_size_t()
    check(lib().kv_cache_required_bytes(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def launch_count() -> int:
    return int(lib().kv_launch_count())


def _stream_ptr(stream) -> ctypes.c_void_p:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dptr(t) -> ctypes.c_void_p:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("device tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _check_f32_out(t, shape, device, name):
    """An output tensor the library writes: float32, contiguous, on the
    cache's device and of the exact shape (the C side sees only a pointer)."""
    import torch
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be float32 of shape {list(shape)}")
    if not t.is_cuda or t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor on {device}")


class KVCache:
    """One quantised KV cache in a torch-allocated device arena."""

    def __init__(self, device=None, **cfg_kwargs):
        import torch
        self.cfg = make_config(**cfg_kwargs)
        self.kwargs = dict(cfg_kwargs)
        self.act_dtype = torch.bfloat16 if cfg_kwargs.get("act_dtype", "f16") == "bf16" else torch.float16
        self.device = torch.device(device or "cuda")
        nbytes = required_bytes(self.cfg)
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.device = self.arena.device  # with its index ("cuda" alone has none)
        h = ctypes.c_void_p()
        check(lib().kv_cache_create(ctypes.byref(self.cfg), _dptr(self.arena), nbytes, ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib().kv_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        check(lib().kv_cache_reset(self.handle))

    def _kv(self, k, v):
        if k.dtype != self.act_dtype or v.dtype != self.act_dtype:
            raise TypeError(f"K/V must be {self.act_dtype}")
        c = self.cfg
        if k.dim() != 4 or k.shape != v.shape or tuple(k.shape[:2]) != (c.batch, c.n_kv_heads) or k.shape[3] != c.head_dim:
            raise ValueError("K/V must be [B, Hkv, n, D]")
        return k.shape[2]

    def append(self, layer, k, v, stream=None):
        n = self._kv(k, v)
        check(lib().kv_append(self.handle, layer, _dptr(k), _dptr(v), n, _stream_ptr(stream)))

    def prefill_quantize(self, layer, k, v, stream=None):
        n = self._kv(k, v)
        check(lib().kv_prefill_quantize(self.handle, layer, _dptr(k), _dptr(v), n, _stream_ptr(stream)))

    def evict(self, layer):
        b, e = ctypes.c_int64(), ctypes.c_int64()
        check(lib().kv_evict(self.handle, layer, ctypes.byref(b), ctypes.byref(e)))
        return b.value, e.value

    def _decode_args(self, q, out, lse):
        c = self.cfg
        if q.dtype != self.act_dtype or tuple(q.shape) != (c.batch, c.n_q_heads, c.head_dim):
            raise ValueError("q must be [B, Hq, D] in the activation dtype")
        if not q.is_cuda or q.device != self.device:
            raise ValueError(f"q must be on {self.device}")
        _check_f32_out(out, (c.batch, c.n_q_heads, c.head_dim), self.device, "out")
        if lse is not None:
            _check_f32_out(lse, (c.batch, c.n_q_heads), self.device, "lse")
        return _dptr(lse) if lse is not None else None

    def decode_attn(self, layer, q, out=None, lse=None, stream=None):
        import torch
        c = self.cfg
        if out is None:
            out = torch.empty((c.batch, c.n_q_heads, c.head_dim), dtype=torch.float32, device=self.device)
        lp = self._decode_args(q, out, lse)
        check(lib().kv_decode_attn(self.handle, layer, _dptr(q), _dptr(out), lp, _stream_ptr(stream)))
        return out

    def decode_attn_noalloc(self, layer, q, out, lse=None, stream=None):
        """kv_decode_attn_noalloc: decode into caller-given `out` (and `lse`)
        with the partials in the library's fixed device block; allocates
        nothing."""
        lp = self._decode_args(q, out, lse)
        check(lib().kv_decode_attn_noalloc(self.handle, layer, _dptr(q), _dptr(out), lp, _stream_ptr(stream)))
        return out

    def stats(self, layer) -> dict:
        s = CacheStats()
        check(lib().kv_cache_stats(self.handle, layer, ctypes.byref(s)))
        return {n: getattr(s, n) for n, _ in CacheStats._fields_}

    def export(self, layer, what, stream=None) -> np.ndarray:
        """One array in canonical layout as numpy (shape per kvq.h)."""
        wid = EXPORT[what]
        n = ctypes.c_size_t()
        check(lib().kv_cache_export_bytes(self.handle, layer, wid, ctypes.byref(n)))
        buf = np.zeros(n.value, np.uint8)
        check(lib().kv_cache_export(self.handle, layer, wid, buf.ctypes.data_as(ctypes.c_void_p), n.value,
                                    _stream_ptr(stream)))
        return self._shape(layer, what, buf)

    def _shape(self, layer, what, buf):
        c = self.cfg
        B, H, D = c.batch, c.n_kv_heads, c.head_dim
        st = self.stats(layer)
        T0 = 32 * (st["evict_end"] // 32)
        n = max(0, st["quant_end"] - T0)
        G = n // 32
        R = st["length"] - st["fp16_begin"]
        if what in ("k_codes", "v_codes"):
            bits = c.k_bits if what == "k_codes" else c.v_bits
            return buf.reshape(B, H, n, D * bits // 8)      # rows packed tight
        if what in ("k_scale", "k_zero"):
            return buf.view(np.float16).reshape(B, H, G, D)
        if what in ("v_scale", "v_zero"):
            return buf.view(np.float16).reshape(B, H, n, D // 32)
        if what in ("k_norm", "v_norm"):
            return buf.view(np.float32).reshape(B, H, n)
        if what == "sink_pos":
            return buf.view(np.int64).reshape(B, -1)
        if what in ("sink_k", "sink_v", "tail_k", "tail_v"):
            rows = buf.view(np.uint16).reshape(B, H, -1, D)
            return _act_to_f32(rows, self.kwargs.get("act_dtype", "f16"))
        if what == "sink_mask":
            return buf.view(np.uint32).reshape(B, G)
        if what in ("codebook_k", "codebook_v", "tq_signs"):
            return buf.view(np.float32)
        if what == "rope":
            return buf.view(np.float32).reshape(-1, D // 2, 2)
        raise KeyError(what)

    def check_device_error(self, stream=None):
        check(lib().kv_cache_check_device_error(self.handle, _stream_ptr(stream)))

    def test_bounded_wait(self, budget_cycles, stream=None):
        """kv_cache_test_bounded_wait: the device waits run out on purpose;
        returns the 5 result words (see kvq.h)."""
        res = (ctypes.c_int64 * 5)()
        check(lib().kv_cache_test_bounded_wait(self.handle, int(budget_cycles), res, _stream_ptr(stream)))
        return [int(x) for x in res]

    def set_timing_events(self, ev_begin, ev_end):
        if ev_begin is None:
            check(lib().kv_cache_set_timing_events(self.handle, None, None))
        else:
            check(lib().kv_cache_set_timing_events(self.handle, ctypes.c_void_p(ev_begin.cuda_event),
                                                   ctypes.c_void_p(ev_end.cuda_event)))


def _act_to_f32(bits: np.ndarray, act: str) -> np.ndarray:
    if act == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


def copy_bandwidth(src, dst, stream=None) -> None:
    """The 16-byte vectorised copy kernel (bandwidth reference)."""
    check(lib().kv_copy_bandwidth_kernel(_dptr(src), _dptr(dst), src.numel() * src.element_size(),
                                         _stream_ptr(stream)))
