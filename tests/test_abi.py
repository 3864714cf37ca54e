"""The C-ABI library loads, exports every symbol the header declares, has
the struct layout the binding assumes, and validates configurations on the
host (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    from bit_kv_cache_append_gb300 import build, binding
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:kv_status|int64_t|const char\*)\s+(kv_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 16
    from bit_kv_cache_append_gb300 import binding
    assert set(names) == set(binding.SYMBOLS)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", os.path.join(ROOT, "bit_kv_cache_append_gb300", "libkvq.so")],
                         capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}\b", out), n


def test_struct_layout_matches_c(tmp_path):
    from bit_kv_cache_append_gb300 import binding
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "kvq.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(kv_cache_config),'
                   ' offsetof(kv_cache_config, max_tokens), offsetof(kv_cache_config, seed),'
                   ' offsetof(kv_cache_config, rope_base), offsetof(kv_cache_config, max_splits),'
                   ' sizeof(kv_cache_stats_t)); return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    C = binding.CacheConfig
    assert got == [ctypes.sizeof(C), C.max_tokens.offset, C.seed.offset, C.rope_base.offset,
                   C.max_splits.offset, ctypes.sizeof(binding.CacheStats)]


def _status(lib, **kw):
    from bit_kv_cache_append_gb300 import binding
    base = dict(n_layers=1, batch=2, n_kv_heads=2, n_q_heads=4, head_dim=64, max_tokens=512)
    base.update(kw)
    cfg = binding.make_config(**base)
    n = ctypes.c_size_t()
    return lib.kv_cache_required_bytes(ctypes.byref(cfg), ctypes.byref(n)), n.value


def test_config_validation_on_host(lib):
    from bit_kv_cache_append_gb300 import binding as B
    ok, n = _status(lib)
    assert ok == B.KV_OK and n > 0
    bad = [dict(head_dim=96), dict(n_q_heads=3), dict(n_q_heads=16), dict(k_bits=5),
           dict(evict_window=16), dict(n_dyn_sinks=5, n_sink=4), dict(mode="turboquant", k_bits=8),
           dict(max_tokens=8), dict(n_sink=33), dict(n_dyn_sinks=40), dict(mode="turboquant", n_dyn_sinks=2),
           dict(rope_reposition=True), dict(v_q4_0=True, v_bits=2), dict(mode="turboquant", v_q4_0=True)]
    for kw in bad:
        st, _ = _status(lib, **kw)
        assert st in (B.KV_ERR_INVALID_ARG, B.KV_ERR_UNSUPPORTED), kw
        assert lib.kv_last_error()


def test_required_bytes_grow_with_capacity(lib):
    _, a = _status(lib, max_tokens=512)
    _, b = _status(lib, max_tokens=4096)
    assert b > a
    _, c = _status(lib, max_tokens=512, rope_base=10000.0, rope_max_pos=65536)
    assert c - a >= 65536 * 64 * 4


def test_null_arguments_rejected(lib):
    from bit_kv_cache_append_gb300 import binding as B
    assert lib.kv_cache_required_bytes(None, None) == B.KV_ERR_INVALID_ARG
    assert lib.kv_append(None, 0, None, None, 1, None) == B.KV_ERR_INVALID_ARG
    assert lib.kv_decode_attn(None, 0, None, None, None, None) == B.KV_ERR_INVALID_ARG
    b, e = ctypes.c_int64(), ctypes.c_int64()
    assert lib.kv_evict(None, 0, ctypes.byref(b), ctypes.byref(e)) == B.KV_ERR_INVALID_ARG


def test_product_path_has_no_oracle_import():
    """The library sources and the binding never reach the oracle."""
    pkg = os.path.join(ROOT, "bit_kv_cache_append_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "oracle/" not in text and "oracle." not in text, f
