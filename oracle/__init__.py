"""CPU oracle for the quantised KV-cache append and decode-attention path.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only the tests under ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import, call or execute anything in it. The
product path (the CUDA library and its Python binding) never does, and it
shares no code, header, table or constant generator with this package: the
only thing the two sides share is the seeded input generator module
``bit_kv_cache_append_gb300.workloads``, which holds none of the method's
arithmetic.

The oracle is plain, slow and written to be checked by eye against the pages
it follows (each module names its sources by page title and section):

  * ``kivi``       - KIVI min/max quantisation, dequantisation and packing.
  * ``rope``       - vanilla RoPE baked into keys at absolute positions.
  * ``turboquant`` - signs, FWHT, norms, the Beta Lloyd-Max codebook and the
                     rotated scalar code.
  * ``kvsink``     - key-norm top-k sink selection and calibration exclusion.
  * ``cache``      - the cache state machine (segments, eviction, append,
                     prefill) and decode attention by its definition.

Floating-point steps that decide an integer (a code, a sink choice) run in
float32 with every operation rounded on its own, the same precision the
kernels take those decisions in; attention itself is computed in double from
the float32 dequantised values.

Parity pins: every function is pinned by ``tests/test_oracle_*.py`` to values
the pages print, closed forms, invariants or independent library routines.
Parity unpinned: the exact float32 codebook values (pinned only through the
Lloyd-Max conditions, the closed forms at a = 1 and 1 bit, and symmetry; the
pages print no codebook numbers).
"""
from .cache import CacheConfig, OracleCache, validate  # noqa: F401
from . import kivi, kvsink, rope, turboquant, numerics  # noqa: F401
